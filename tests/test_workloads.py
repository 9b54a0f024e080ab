"""The seeded input recipe: context-length distributions of the named workloads, the pool
size rule, page tables drawn from a permutation of the pool (no block used twice), slot
mappings that follow the tables ("Lesson 4: Model deployment and inference acceleration",
4.2: 16-token blocks of a pre-allocated pool, a page table per request), and values that
a subset of sequences regenerates bit for bit."""

import math

import pytest
import torch

from paged_kv_cache_264_gb300 import workloads as W


@pytest.mark.parametrize("name,lo,hi,count", [
    ("llama2_7b", 128, 2048, 64),
    ("llama3_8b_gqa", 512, 8192, 128),
    ("int8_cb", 16, 16384, 256),
    ("fp8_cb", 16, 16384, 256),
])
def test_context_length_ranges(name, lo, hi, count):
    lens = W.context_lens_of(name)
    assert lens.numel() == count
    assert int(lens.min()) >= lo and int(lens.max()) <= hi
    assert torch.equal(lens, W.context_lens_of(name))  # seeded


def test_lognormal_lengths_centre_on_1024():
    lens = W.context_lens_of("int8_cb").double()
    med = float(lens.median())
    assert 700 < med < 1500  # median 1024 with sigma 1 on 256 draws


def test_variants_share_their_base_lengths():
    assert torch.equal(W.context_lens_of("llama2_7b_verify4"), W.context_lens_of("llama2_7b"))
    assert torch.equal(W.context_lens_of("llama3_8b_gqa_verify4"), W.context_lens_of("llama3_8b_gqa"))
    assert torch.equal(W.context_lens_of("long_32k_window4k"), W.context_lens_of("long_32k"))
    assert (W.context_lens_of("long_32k") == 32768).all()
    assert W.SPECS["long_32k_window4k"].window == 4096
    assert W.SPECS["llama2_7b_verify4"].num_queries == 4
    assert torch.equal(W.context_lens_of("int8_cb_d64"), W.context_lens_of("int8_cb"))
    assert W.SPECS["int8_cb_d64"].head_dim == 64


@pytest.mark.parametrize("lens,k", [([17, 40], 1), ([1, 16, 33, 100, 257], 1), ([4, 20, 65], 4)])
def test_tables_slots_and_pool(lens, k):
    w = W.build(name="t", context_lens=lens, num_q_heads=8, num_kv_heads=2, head_dim=64,
                kv_dtype="bf16", seed=77, num_queries=k)
    nblk = [(t + 15) // 16 for t in lens]
    assert w.num_blocks == max(1, math.ceil(1.25 * sum(nblk)))
    used = []
    for b, t in enumerate(lens):
        row = w.block_tables[b, :nblk[b]].tolist()
        assert all(0 <= x < w.num_blocks for x in row)
        used += row
        lo = int(w.seq_offsets[b])
        slots = w.slot_mapping[lo:lo + t].tolist()
        assert slots == [row[i // 16] * 16 + i % 16 for i in range(t)]
    assert len(used) == len(set(used))  # every physical block belongs to one sequence
    assert w.key.shape == (sum(lens), 2, 64) and w.key.dtype == torch.bfloat16
    assert w.q.shape == ((len(lens), 8, 64) if k == 1 else (len(lens), k, 8, 64))


def test_subset_regenerates_the_same_values():
    lens = [30, 70, 5, 120]
    full = W.build(name="t", context_lens=lens, num_q_heads=4, num_kv_heads=4, head_dim=64,
                   kv_dtype="bf16", seed=5)
    part = W.build(name="t", context_lens=lens, num_q_heads=4, num_kv_heads=4, head_dim=64,
                   kv_dtype="bf16", seed=5, seqs=[1, 3])
    for i, b in enumerate([1, 3]):
        lo_f, lo_p = int(full.seq_offsets[b]), int(part.seq_offsets[i])
        t = lens[b]
        assert torch.equal(full.key[lo_f:lo_f + t], part.key[lo_p:lo_p + t])
        assert torch.equal(full.value[lo_f:lo_f + t], part.value[lo_p:lo_p + t])
        assert torch.equal(full.q[b], part.q[i])
