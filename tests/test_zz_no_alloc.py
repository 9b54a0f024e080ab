"""The decode entry point that allocates nothing, for callers that cannot allocate
device memory where they decode (for example a plugin hosted by a runtime that owns the
whole memory budget, or a serving loop that must not call cudaMalloc).

It is called here through the C ABI and checked against the regular entry point (which
takes a caller-allocated workspace) on the same inputs, twice in a row: the library's
fixed scratch array keeps the previous call's contents, and the second call must not be
affected by them.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import _lib, build, workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _pool_with(w, kv):
    pool = pkv.PagedKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, kv, fill=0)
    pool.reshape_and_cache(w.key.cuda(), w.value.cuda(), w.slot_mapping.cuda())
    return pool


def _close(a, b):
    err = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (err.max().item(), err.mean().item())


def _workload(name):
    if name == "gqa_split":  # 16 sequences of 4000-4096 tokens, 32/8 heads: split on the tensor cores
        lens = torch.randint(4000, 4097, (16,), generator=torch.Generator().manual_seed(5))
        return W.build(name=name, context_lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       seed=17, device="cuda"), "bf16"
    return W.make(name, device="cuda"), W.SPECS[name].kv_dtype


@pytest.mark.parametrize("name", ["long_32k", "gqa_split"])
def test_static_scratch_matches_workspace_entry_point(name):
    build.build()
    lib = _lib.load()
    w, kv = _workload(name)
    pool = _pool_with(w, kv)
    q, tab, lens = w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda()
    need = pkv.decode_workspace_bytes(pool, w.num_seqs, w.num_q_heads, w.max_context_len)
    assert 0 < need <= _lib.STATIC_SCRATCH_BYTES  # this shape uses scratch, and it fits
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ref = pool.decode(q, tab, lens, w.scale, w.max_context_len)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        st = lib.pkv_paged_attention_decode_static_scratch(
            pool.handle, _ptr(q), _ptr(tab), tab.shape[1], _ptr(lens), w.num_seqs, w.num_q_heads,
            w.max_context_len, ctypes.c_float(w.scale), _ptr(out), stream)
        assert st == 0, lib.pkv_status_string(st)
        torch.cuda.synchronize()
        _close(out, ref)
    assert pool.device_error() == 0
    pool.close()


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
    assert np.array_equal(out.view(torch.int16).cpu().numpy(), ref.view(torch.int16).cpu().numpy())
    pool.close()
