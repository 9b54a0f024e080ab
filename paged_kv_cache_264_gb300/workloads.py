"""Seeded synthetic inputs for paged decode: context lengths, block pools, page tables,
slot mappings and N(0, 1) bf16 values.

This module builds inputs only.  It holds none of the attention or quantisation
arithmetic, so both the CUDA path and the CPU oracle can be fed from it without
sharing any of the method.

The five named workloads follow the shapes that the pages' decode discussion implies
(16-token blocks and a per-request page table over a shuffled, pre-allocated pool:
"Lesson 4: Model deployment and inference acceleration", section 4.2; LLaMA-2-7B and
Llama-3-8B head shapes; a long 32k context; INT8 continuous batching, section 5.3):

===============  ====  ===============================  =======  ====  =====  ================
name             B     context lengths                  Hq/Hkv   d     KV     extra
===============  ====  ===============================  =======  ====  =====  ================
tiny             2     {17, 40}                         4/4      64    bf16   16-block pool
llama2_7b        64    uniform [128, 2048]              32/32    128   bf16
llama3_8b_gqa    128   uniform [512, 8192]              32/8     128   bf16
long_32k         8     32768 each                       32/32    128   bf16   1% key chans x8
int8_cb          256   lognormal(ln 1024, 1) in         32/8     128   int8
                       [16, 16384]
fp8_cb           256   as int8_cb                       32/8     128   fp8
llama2_7b_       64    as llama2_7b                     32/32    128   bf16   k = 4 queries
verify4
llama3_8b_gqa_   128   as llama3_8b_gqa                 32/8     128   bf16   k = 4 queries
verify4
long_32k_       8     as long_32k                      32/32    128   bf16   window 4096
window4k
int8_cb_d64      256   as int8_cb                       32/8     64    int8
===============  ====  ===============================  =======  ====  =====  ================

The two ``verify4`` workloads are multi-query decode batches for speculative decoding
("Lesson 4", 5.2: the target model checks k draft tokens in one pass): each sequence's
last 4 cached tokens are the drafts, and q holds 4 query tokens per sequence
([B, 4, Hq, d]), query i attending causally to the tokens up to its own position.  They
reuse their base workload's context lengths and block pool (its seed), so a verify step
and a decode step over the same cache compare directly.  ``long_32k_window4k`` is the
long_32k cache decoded with a sliding window of 4096 tokens ("LLM/MLLM inference
optimisation", 2.3: keep only the most recent window): each query reads its last 4096
tokens.  ``int8_cb_d64`` is the int8_cb batch at head_dim 64 (two 64-byte token rows to each
128-byte swizzled row on the tensor-core path).

Pools other than ``tiny`` hold ``ceil(1.25 * sum_b ceil(T_b / 16))`` blocks; the blocks
that sequences use are drawn from a seeded permutation of the pool.  Everything is drawn
from ``torch.Generator`` seeded with ``1000 + index`` of the workload (1 .. 6).  Values
are drawn per sequence from a generator seeded by (workload seed, sequence), so any
subset of sequences can be regenerated alone.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 16


@dataclass(frozen=True)
class Spec:
    name: str
    index: int
    description: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str  # "bf16" | "int8" | "fp8"
    lens: tuple  # ("fixed", [..]) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi) | ("const", n)
    pool_blocks: int | None = None  # None: ceil(1.25 * blocks needed)
    outlier_key_channel_frac: float = 0.0
    outlier_key_scale: float = 8.0
    num_queries: int = 1  # query tokens per sequence (k > 1: draft verification)
    base_index: int | None = None  # draw lengths, pool and values as workload base_index does
    window: int = 0  # sliding window of the decode (0: none)

    @property
    def seed(self) -> int:
        return 1000 + (self.index if self.base_index is None else self.base_index)


SPECS: dict[str, Spec] = {
    s.name: s
    for s in (
        Spec("tiny", 1, "tiny paged decode: 2 sequences, context_lens {17, 40}, 4/4 heads, "
             "head_dim 64, 16-block pool", 2, 4, 4, 64, "bf16", ("fixed", [17, 40]), pool_blocks=16),
        Spec("llama2_7b", 2, "LLaMA-2-7B-shaped single layer: 64 sequences, context_lens uniform "
             "in [128, 2048], 32/32 heads, head_dim 128, bf16 KV", 64, 32, 32, 128, "bf16",
             ("uniform", 128, 2048)),
        Spec("llama3_8b_gqa", 3, "Llama-3-8B-shaped GQA single layer: 128 sequences, context_lens "
             "uniform in [512, 8192], 32/8 heads, head_dim 128, bf16 KV", 128, 32, 8, 128, "bf16",
             ("uniform", 512, 8192)),
        Spec("long_32k", 4, "long-context split-K: 8 sequences of 32768 tokens, 32/32 heads, "
             "head_dim 128, bf16 KV, 1% of key channels x8", 8, 32, 32, 128, "bf16",
             ("const", 32768), outlier_key_channel_frac=0.01),
        Spec("int8_cb", 5, "continuous-batching decode step with INT8 KV: 256 sequences, "
             "context_lens lognormal (median 1024, sigma 1) clipped to [16, 16384], 32/8 heads, "
             "head_dim 128", 256, 32, 8, 128, "int8", ("lognormal", 1024.0, 1.0, 16, 16384)),
        Spec("fp8_cb", 6, "continuous-batching decode step with FP8 (E4M3) KV: the int8_cb batch "
             "shape with E4M3 codes and per-(token, head) scales", 256, 32, 8, 128, "fp8",
             ("lognormal", 1024.0, 1.0, 16, 16384)),
        Spec("llama2_7b_verify4", 7, "LLaMA-2-7B-shaped draft verification: the llama2_7b batch "
             "shape with 4 query tokens per sequence (the last 4 cached tokens, causal)", 64, 32, 32,
             128, "bf16", ("uniform", 128, 2048), num_queries=4, base_index=2),
        Spec("llama3_8b_gqa_verify4", 8, "Llama-3-8B-shaped GQA draft verification: the "
             "llama3_8b_gqa batch shape with 4 query tokens per sequence (causal)", 128, 32, 8, 128,
             "bf16", ("uniform", 512, 8192), num_queries=4, base_index=3),
        Spec("long_32k_window4k", 9, "long-context sliding window: the long_32k cache (8 x 32768 "
             "tokens, 32/32 heads, head_dim 128, bf16) decoded with a 4096-token window", 8, 32, 32, 128,
             "bf16", ("const", 32768), outlier_key_channel_frac=0.01, base_index=4, window=4096),
        Spec("int8_cb_d64", 10, "INT8 continuous batching at head_dim 64: the int8_cb lengths "
             "with 32/8 heads of 64 dims", 256, 32, 8, 64,
             "int8", ("lognormal", 1024.0, 1.0, 16, 16384), base_index=5),
    )
}


@dataclass
class Workload:
    """Host-side description of one decode batch plus its bf16 values.

    ``key``/``value`` hold every cached token's rows in (sequence, position) order:
    rows ``seq_offsets[b] .. seq_offsets[b+1]-1`` are sequence ``b``'s tokens
    ``0 .. T_b-1``.  ``slot_mapping[r]`` is the pool slot of row ``r``.
    """

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str
    num_blocks: int
    context_lens: torch.Tensor  # int32 [B] (cpu)
    block_tables: torch.Tensor  # int32 [B, max_blocks_per_seq] (cpu), -1 past the end
    slot_mapping: torch.Tensor  # int32 [N] (cpu)
    seq_offsets: torch.Tensor  # int64 [B+1] (cpu)
    q: torch.Tensor  # bf16 [B, Hq, d], or [B, k, Hq, d] with k = num_queries > 1
    key: torch.Tensor  # bf16 [N, Hkv, d]
    value: torch.Tensor  # bf16 [N, Hkv, d]
    scale: float
    seed: int
    outlier_channels: list = field(default_factory=list)
    num_queries: int = 1

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0

    @property
    def num_tokens(self) -> int:
        return int(self.seq_offsets[-1].item())

    def last_token_rows(self) -> torch.Tensor:
        """Row indices of each sequence's newest k = num_queries tokens (the tokens a decode
        step appends: one new token, or k drafts), sequence by sequence."""
        k = self.num_queries
        ends = self.seq_offsets[1:].to(torch.int64)
        return (ends[:, None] - k + torch.arange(k, dtype=torch.int64)[None, :]).flatten()

    def history_rows(self) -> torch.Tensor:
        """Row indices of every token except each sequence's newest k."""
        keep = torch.ones(self.num_tokens, dtype=torch.bool)
        keep[self.last_token_rows()] = False
        return torch.nonzero(keep).flatten()


def _draw_context_lens(spec_lens: tuple, num_seqs: int, gen: torch.Generator) -> torch.Tensor:
    kind = spec_lens[0]
    if kind == "fixed":
        lens = torch.tensor(spec_lens[1], dtype=torch.int64)
        assert lens.numel() == num_seqs
    elif kind == "const":
        lens = torch.full((num_seqs,), int(spec_lens[1]), dtype=torch.int64)
    elif kind == "uniform":
        lo, hi = spec_lens[1], spec_lens[2]
        lens = torch.randint(lo, hi + 1, (num_seqs,), generator=gen, dtype=torch.int64)
    elif kind == "lognormal":
        median, sigma, lo, hi = spec_lens[1:]
        z = torch.randn(num_seqs, generator=gen, dtype=torch.float64)
        lens = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi).to(torch.int64)
    else:
        raise ValueError(kind)
    return lens


def _value_gen(seed: int, stream: int, seq: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919 + seq) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def build(
    *,
    name: str,
    context_lens,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    kv_dtype: str = "bf16",
    seed: int = 0,
    num_blocks: int | None = None,
    pool_factor: float = 1.25,
    max_blocks_per_seq: int | None = None,
    outlier_key_channel_frac: float = 0.0,
    outlier_key_scale: float = 8.0,
    device="cpu",
    seqs: list | None = None,
    num_queries: int = 1,
) -> Workload:
    """Build a workload from explicit context lengths.

    ``seqs`` (optional) restricts the generated q/key/value rows to a subset of the
    sequences; the page table and pool are still those of the whole batch, so a subset
    is an exact slice of the full workload.
    """
    gen = torch.Generator().manual_seed(2 * seed + 1)
    lens = torch.as_tensor(context_lens, dtype=torch.int64).flatten()
    b_all = lens.numel()
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    need = int(nblk.sum().item())
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * need))
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    width = int(nblk.max().item()) if b_all else 1
    if max_blocks_per_seq is not None:
        width = max(width, max_blocks_per_seq)
    perm = torch.randperm(num_blocks, generator=gen)[:need].to(torch.int32)
    tables = torch.full((b_all, max(width, 1)), -1, dtype=torch.int32)
    cursor = 0
    for b in range(b_all):
        n = int(nblk[b])
        tables[b, :n] = perm[cursor:cursor + n]
        cursor += n

    outlier = []
    if outlier_key_channel_frac > 0:
        n_out = max(1, round(outlier_key_channel_frac * head_dim))
        outlier = torch.randperm(head_dim, generator=gen)[:n_out].tolist()

    sel = list(range(b_all)) if seqs is None else list(seqs)
    sub_lens = lens[sel]
    offsets = torch.zeros(len(sel) + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(sub_lens, 0)
    n_tok = int(offsets[-1])

    # Slot of token t of sequence b: physical block table[b][t // 16], offset t % 16.
    slot_mapping = torch.empty(n_tok, dtype=torch.int32)
    for i, b in enumerate(sel):
        t = torch.arange(int(lens[b]), dtype=torch.int64)
        phys = tables[b].to(torch.int64)[t // BLOCK_SIZE]
        slot_mapping[offsets[i]:offsets[i + 1]] = (phys * BLOCK_SIZE + t % BLOCK_SIZE).to(torch.int32)

    if num_queries > 1 and int(lens.min()) < num_queries:
        raise ValueError("every context must hold the k query tokens")
    qshape = (num_q_heads, head_dim) if num_queries == 1 else (num_queries, num_q_heads, head_dim)
    q = torch.empty((len(sel),) + qshape, dtype=torch.bfloat16, device=device)
    key = torch.empty((n_tok, num_kv_heads, head_dim), dtype=torch.bfloat16, device=device)
    value = torch.empty_like(key)
    for i, b in enumerate(sel):
        q[i] = torch.randn(qshape, generator=_value_gen(seed, 0, b, device),
                           device=device, dtype=torch.float32).to(torch.bfloat16)
        lo, hi = int(offsets[i]), int(offsets[i + 1])
        kf = torch.randn((hi - lo, num_kv_heads, head_dim), generator=_value_gen(seed, 1, b, device),
                         device=device, dtype=torch.float32)
        if outlier:
            kf[:, :, outlier] *= outlier_key_scale
        key[lo:hi] = kf.to(torch.bfloat16)
        del kf
        value[lo:hi] = torch.randn((hi - lo, num_kv_heads, head_dim),
                                   generator=_value_gen(seed, 2, b, device), device=device,
                                   dtype=torch.float32).to(torch.bfloat16)

    return Workload(
        name=name, num_seqs=len(sel), num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, kv_dtype=kv_dtype, num_blocks=num_blocks,
        context_lens=sub_lens.to(torch.int32), block_tables=tables[sel].contiguous(),
        slot_mapping=slot_mapping, seq_offsets=offsets, q=q, key=key, value=value,
        scale=1.0 / math.sqrt(head_dim), seed=seed, outlier_channels=outlier,
        num_queries=num_queries,
    )


def context_lens_of(name: str) -> torch.Tensor:
    spec = SPECS[name]
    gen = torch.Generator().manual_seed(spec.seed)
    return _draw_context_lens(spec.lens, spec.num_seqs, gen)


def make(name: str, device="cpu", seqs: list | None = None) -> Workload:
    """One of the five named workloads (optionally only some of its sequences' values)."""
    spec = SPECS[name]
    lens = context_lens_of(name)
    return build(
        name=name, context_lens=lens, num_q_heads=spec.num_q_heads,
        num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim, kv_dtype=spec.kv_dtype,
        seed=spec.seed, num_blocks=spec.pool_blocks,
        outlier_key_channel_frac=spec.outlier_key_channel_frac,
        outlier_key_scale=spec.outlier_key_scale, device=device, seqs=seqs,
        num_queries=spec.num_queries,
    )


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bit patterns (copied to host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
