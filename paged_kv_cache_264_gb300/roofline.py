"""Algorithmic bytes and flops of one decode step, for the HBM roofline.

Decode reads every cached token's K and V once per kv head (GQA groups share the read;
"LLM/MLLM inference optimisation", 2.2-2.3: the cache holds 2 x n_kv x head_dim x
seq_len x bytes per layer), plus q, the output and the page table.  Tokens actually
attended are counted, not whole 16-token blocks.  A decode step also appends one new
token per sequence (reads its bf16 K/V row, writes the cached row and, for INT8, the
scales).

A multi-query step (k draft tokens per sequence, verified in one call) reads the same
cached K/V once, k times the q and output rows, and appends k tokens per sequence; its
flops count each query over the tokens up to its own position.  With a sliding window of W
tokens a sequence's K/V read covers the union of its queries' windows, min(T, W + k - 1)
tokens, and each query attends to min(its position + 1, W).
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

BLOCK = 16


@dataclass(frozen=True)
class StepBytes:
    kv_read: int        # cached K and V (and INT8 scales) read by decode
    q_out: int          # q read + output written (bf16)
    tables: int         # block-table entries + context lengths read
    append: int         # the appended tokens: bf16 rows read, cached rows (+ scales) and slots
    flops: int          # 4 * (tokens attended, summed over queries) * Hq * d  (QK and PV)

    @property
    def decode(self) -> int:
        return self.kv_read + self.q_out + self.tables

    @property
    def step(self) -> int:
        return self.decode + self.append


def step_bytes(context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: str,
               append: bool = True, num_queries: int = 1, window: int = 0) -> StepBytes:
    lens = torch.as_tensor(context_lens, dtype=torch.int64)
    b = int(lens.numel())
    k = int(num_queries)
    if window > 0:
        read = torch.minimum(lens, torch.full_like(lens, window + k - 1))
        first_blk = torch.clamp(lens - (k - 1) - window, min=0) // BLOCK
    else:
        read = lens
        first_blk = torch.zeros_like(lens)
    sum_t = int(read.sum())
    sum_nb = int(((lens + BLOCK - 1) // BLOCK - first_blk).sum())
    esz = 2 if kv_dtype == "bf16" else 1
    kv = 2 * sum_t * num_kv_heads * head_dim * esz
    if kv_dtype in ("int8", "fp8"):
        kv += 2 * sum_t * num_kv_heads * 4
    q_out = 2 * b * k * num_q_heads * head_dim * 2
    tables = 4 * (sum_nb + b)
    app = 0
    if append:
        n_new = b * k
        app = 2 * n_new * num_kv_heads * head_dim * 2          # new K and V rows (bf16) read
        app += 2 * n_new * num_kv_heads * head_dim * esz       # cached rows written
        if kv_dtype in ("int8", "fp8"):
            app += 2 * n_new * num_kv_heads * 4                # scales written
        app += 4 * n_new                                       # slot_mapping read
    pos1 = lens[:, None] - (k - 1) + torch.arange(k)[None, :]  # query i sees pos_i + 1 tokens
    if window > 0:
        pos1 = torch.clamp(pos1, max=window)
    attended = int(pos1.sum())
    flops = 4 * attended * num_q_heads * head_dim
    return StepBytes(kv, q_out, tables, app, flops)
