"""The decode entry point that allocates nothing, for callers that cannot allocate
device memory where they decode (for example a plugin hosted by a runtime that owns the
whole memory budget, or a serving loop that must not call cudaMalloc).

It is called here through the C ABI and checked against the regular entry point (which
takes a caller-allocated workspace) on the same inputs: both run the same kernels with
the same plan, so the outputs must agree bit for bit.  The library's fixed scratch array
keeps the previous call's contents, so before each compared call another batch of the
same shape (other values, same partition layout) fills it with different partials: a
partial that were read without being rewritten would then show.  Around the compared
calls neither torch's allocator nor the device's free memory may move.  This file is
collected last so that a run stopping at the first failure has already run every other
test; it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import _lib, build, workloads as W
from gpu_helpers import compare, oracle_decode

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _pool_with(w, kv):
    pool = pkv.PagedKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, kv, fill=0)
    pool.reshape_and_cache(w.key.cuda(), w.value.cuda(), w.slot_mapping.cuda())
    return pool


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


# Batches that split on the tensor cores: (lengths, Hq, Hkv, pool type).  The second batch
# of each pair has the same lengths (so the same plan and partial layout) and other values.
CASES = {
    "long_mha": ([8192] * 8, 32, 32, "bf16"),
    "gqa_split": (torch.randint(4000, 4097, (16,), generator=torch.Generator().manual_seed(5)).tolist(),
                  32, 8, "bf16"),
    "int8_gqa": (torch.randint(300, 3000, (24,), generator=torch.Generator().manual_seed(6)).tolist(),
                 32, 8, "int8"),
}


def _batch(name, seed):
    lens, hq, hkv, kv = CASES[name]
    return W.build(name=name, context_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                   kv_dtype=kv, seed=seed), kv


def _static_call(lib, pool, w, q, tab, lens, out, stream):
    st = lib.pkv_paged_attention_decode_static_scratch(
        pool.handle, _ptr(q), _ptr(tab), tab.shape[1], _ptr(lens), w.num_seqs, w.num_q_heads,
        w.max_context_len, ctypes.c_float(w.scale), _ptr(out), stream)
    assert st == 0, (lib.pkv_status_string(st), lib.pkv_static_scratch_error())


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_scratch_matches_workspace_entry_point(name):
    build.build()
    oracle.build()
    lib = _lib.load()
    w, kv = _batch(name, seed=101)
    other, _ = _batch(name, seed=202)
    pool, pool_other = _pool_with(w, kv), _pool_with(other, kv)
    q, tab, lens = w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda()
    oq, otab, olens = other.q.cuda(), other.block_tables.cuda(), other.context_lens.cuda()
    need = pkv.decode_workspace_bytes(pool, w.num_seqs, w.num_q_heads, w.max_context_len)
    assert 0 < need <= _lib.STATIC_SCRATCH_BYTES  # this shape uses scratch, and it fits
    assert pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len) == \
        pkv.decode_plan(pool_other, other.num_seqs, other.num_q_heads, other.max_context_len)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ref = pool.decode(q, tab, lens, w.scale, w.max_context_len)  # caller-allocated workspace
    ref_other = pool_other.decode(oq, otab, olens, other.scale, other.max_context_len)
    out = torch.empty_like(q)
    out_other = torch.empty_like(oq)
    for _ in range(2):  # two calls in a row, each after the other batch filled the scratch
        _static_call(lib, pool_other, other, oq, otab, olens, out_other, stream)
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        _static_call(lib, pool, w, q, tab, lens, out, stream)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
        assert torch.cuda.memory_allocated() == allocated0
        assert np.array_equal(_bits(out), _bits(ref))
        assert np.array_equal(_bits(out_other), _bits(ref_other))
    assert pool.device_error() == 0 and pool_other.device_error() == 0

    # and one sampled sequence against the oracle
    b = w.num_seqs // 2
    expect, _, _ = oracle_decode(w, kv, [b])
    compare(out[b:b + 1], expect, f"{name} static scratch, sequence {b}")
    pool.close()
    pool_other.close()


def test_static_scratch_rejects_shapes_beyond_its_size():
    build.build()
    lib = _lib.load()
    pool = pkv.PagedKVPool(64, 8, 128, "bf16", fill=0)
    b, hq, max_ctx = 128, 32, 8192
    need = pkv.decode_workspace_bytes(pool, b, hq, max_ctx)
    if need <= _lib.STATIC_SCRATCH_BYTES:
        pytest.skip("the automatic plan for this shape fits the static scratch")
    # Real, correctly sized inputs, so that nothing could read out of bounds even if the
    # call did launch.
    q = torch.zeros(b, hq, 128, dtype=torch.bfloat16, device="cuda")
    tab = (torch.arange(b * (max_ctx // 16), device="cuda") % 64).to(torch.int32).view(b, -1)
    lens = torch.full((b,), max_ctx, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    before = pkv.launch_count()
    st = lib.pkv_paged_attention_decode_static_scratch(
        pool.handle, _ptr(q), _ptr(tab), tab.shape[1], _ptr(lens), b, hq, max_ctx,
        ctypes.c_float(0.1), _ptr(out), None)
    assert st == _lib.PKV_ERR_WORKSPACE
    assert b"static scratch" in lib.pkv_static_scratch_error()
    assert pkv.launch_count() == before  # nothing launched
    torch.cuda.synchronize()
    pool.close()


def test_static_scratch_checks_shapes_before_launching():
    """The Python wrapper refuses mis-shaped tensors before calling the library."""
    build.build()
    pool = pkv.PagedKVPool(8, 2, 64, "bf16", fill=0)
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    tab = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    lens = torch.ones(2, dtype=torch.int32, device="cuda")
    before = pkv.launch_count()
    bad = [
        dict(block_tables=torch.zeros(1, 4, dtype=torch.int32, device="cuda")),  # fewer table rows
        dict(context_lens=torch.ones(3, dtype=torch.int32, device="cuda")),       # more lengths
        dict(q=torch.zeros(2, 4, 128, dtype=torch.bfloat16, device="cuda")),     # head_dim of another pool
        dict(out=torch.zeros(2, 2, 64, dtype=torch.bfloat16, device="cuda")),    # out not q's shape
    ]
    for change in bad:
        args = dict(q=q, block_tables=tab, context_lens=lens, out=None) | change
        with pytest.raises(ValueError):
            pkv.api.paged_attention_decode_static_scratch(pool, args["q"], args["block_tables"],
                                                          args["context_lens"], 0.125, 16, out=args["out"])
    torch.cuda.synchronize()
    assert pkv.launch_count() == before
    pool.close()


def test_static_scratch_without_split_needs_none():
    """A batch that fits one partition per sequence uses no scratch at all."""
    build.build()
    w = W.make("tiny", device="cuda")
    pool = _pool_with(w, "bf16")
    assert pkv.decode_workspace_bytes(pool, w.num_seqs, w.num_q_heads, w.max_context_len) == 0
    ref = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len)
    out = pkv.api.paged_attention_decode_static_scratch(pool, w.q.cuda(), w.block_tables.cuda(),
                                                         w.context_lens.cuda(), w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _bits(ref))
    pool.close()
