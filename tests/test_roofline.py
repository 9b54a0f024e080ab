"""The roofline numerator (algorithmic bytes and flops of a decode step) against a
brute-force count: every (sequence, query) pair's visible tokens enumerated as sets, the
K/V read as their union per sequence, and the page-table entries as the blocks from the
first one any query sees to the last.  The model reads each cached token's K and V once
per kv head ("LLM/MLLM inference optimisation", 2.2: the cache holds
2 x n_kv x head_dim x seq_len x bytes per layer)."""

import random

import pytest
import torch

from paged_kv_cache_264_gb300 import roofline


def brute(lens, hq, hkv, d, kv, k, window, append):
    esz = 2 if kv == "bf16" else 1
    quant = kv != "bf16"
    kv_read = q_out = tables = app = attended = 0
    for t_len in lens:
        union = set()
        for i in range(k):
            pos = t_len - k + i                       # query i's own position
            lo = 0 if window == 0 else max(0, pos - window + 1)
            seen = set(range(lo, pos + 1))
            attended += len(seen)
            union |= seen
        kv_read += len(union) * hkv * (2 * d * esz + (8 if quant else 0))
        first_blk = min(union) // 16
        tables += 4 * ((t_len + 15) // 16 - first_blk) + 4
        q_out += 2 * k * hq * d * 2
        if append:
            app += k * (2 * hkv * d * 2 + 2 * hkv * d * esz + (8 * hkv if quant else 0) + 4)
    return kv_read, q_out, tables, app, 4 * attended * hq * d


@pytest.mark.parametrize("seed", range(40))
def test_step_bytes_match_brute_force(seed):
    r = random.Random(seed)
    k = r.choice([1, 1, 2, 4, 7])
    window = r.choice([0, 0, 1, 5, 16, 33, 200])
    lens = [r.randint(k, 300) for _ in range(r.randint(1, 6))]
    hkv = r.choice([1, 2, 8])
    hq = hkv * r.choice([1, 4])
    d = r.choice([64, 128])
    kv = r.choice(["bf16", "int8", "fp8"])
    append = r.random() < 0.5
    sb = roofline.step_bytes(torch.tensor(lens), hq, hkv, d, kv, append=append, num_queries=k,
                             window=window)
    assert (sb.kv_read, sb.q_out, sb.tables, sb.append, sb.flops) == brute(
        lens, hq, hkv, d, kv, k, window, append)
    assert sb.decode == sb.kv_read + sb.q_out + sb.tables
    assert sb.step == sb.decode + sb.append


def test_long_context_step_closed_form():
    """8 sequences of 32768 tokens, 32/32 heads, d = 128, bf16, one appended token each:
    2 * 262144 * 32 * 128 * 2 B of K/V, plus q/out, 16392 table words and the append."""
    sb = roofline.step_bytes(torch.full((8,), 32768), 32, 32, 128, "bf16")
    assert sb.kv_read == 2 * 262144 * 32 * 128 * 2 == 4294967296
    assert sb.q_out == 2 * 8 * 32 * 128 * 2
    assert sb.tables == 4 * (8 * 2048 + 8)
    assert sb.step == 4295426112  # about 4.295 GB per step
    assert sb.flops == 4 * 262144 * 32 * 128


def test_window_wider_than_context_is_full_attention():
    lens = torch.tensor([5, 17, 300])
    full = roofline.step_bytes(lens, 8, 2, 128, "int8", num_queries=3)
    wide = roofline.step_bytes(lens, 8, 2, 128, "int8", num_queries=3, window=10_000)
    assert full == wide
