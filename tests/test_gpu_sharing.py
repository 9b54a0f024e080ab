"""Block sharing on the GPU: copy_blocks, and decode over page tables that alias shared
prefix blocks after fork and copy on write ("Efficient AI Lecture 13", section
"PagedAttention": shared prompt prefixes reuse physical blocks for parallel sampling and
beam search)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import build, workloads as W
from gpu_helpers import compare, fill_pool_garbage

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_copy_blocks_bit_exact(kv):
    nb, hkv, d = 40, 4, 128
    pool = pkv.PagedKVPool(nb, hkv, d, kv)
    g = torch.Generator(device="cuda").manual_seed(3)
    for t in (pool.k_cache, pool.v_cache):
        t.view(torch.uint8).copy_(torch.randint(0, 256, t.view(torch.uint8).shape, generator=g,
                                                device="cuda", dtype=torch.uint8))
    if pool.k_scale is not None:
        pool.k_scale.copy_(torch.rand(pool.k_scale.shape, generator=g, device="cuda"))
        pool.v_scale.copy_(torch.rand(pool.v_scale.shape, generator=g, device="cuda"))
    before = [t.clone() for t in (pool.k_cache, pool.v_cache, pool.k_scale, pool.v_scale) if t is not None]
    pairs = torch.tensor([[3, 10], [11, 0], [39, 20], [5, 6]], dtype=torch.int32, device="cuda")
    pkv.copy_blocks(pool, pairs)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    after = [t for t in (pool.k_cache, pool.v_cache, pool.k_scale, pool.v_scale) if t is not None]
    for b, a in zip(before, after):
        expect = b.clone()
        for src, dst in pairs.tolist():
            expect[dst] = b[src]
        assert torch.equal(a.view(torch.uint8), expect.view(torch.uint8))
    bad = torch.tensor([[0, nb]], dtype=torch.int32, device="cuda")
    pkv.copy_blocks(pool, bad)
    torch.cuda.synchronize()
    assert pool.device_error() == pkv.DEVERR_BLOCK_ID
    pool.close()


def _oracle_for(seq_rows, q_bits, kv, hkv, d, scale):
    """fp64 oracle over each sequence's own logical tokens, laid out contiguously."""
    o = oracle.load()
    lens = [len(r) for r in seq_rows]
    nblk = [(t + 15) // 16 for t in lens]
    tables = np.full((len(lens), max(nblk)), -1, np.int32)
    c = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = np.arange(c, c + n)
        c += n
    slots = np.concatenate([tables[i, np.arange(t) // 16] * 16 + np.arange(t) % 16 for i, t in enumerate(lens)]).astype(np.int32)
    key = np.concatenate([np.stack([r[0] for r in rows]) for rows in seq_rows])
    value = np.concatenate([np.stack([r[1] for r in rows]) for rows in seq_rows])
    shape = (c, hkv, 16, d)
    if kv == "bf16":
        kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
        o.reshape_and_cache_bf16(key, value, slots, kc, vc)
        return o.paged_decode(q_bits, kc, vc, tables, np.array(lens, np.int32), scale)
    cdt = np.int8 if kv == "int8" else np.uint8
    kc, vc = np.zeros(shape, cdt), np.zeros(shape, cdt)
    ks, vs = np.zeros(shape[:3], np.float32), np.zeros(shape[:3], np.float32)
    (o.reshape_and_cache_int8 if kv == "int8" else o.reshape_and_cache_fp8)(key, value, slots, kc, vc, ks, vs)
    return o.paged_decode(q_bits, kc, vc, tables, np.array(lens, np.int32), scale, ks, vs)


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_beams_share_prompt_blocks(kv, kernel):
    """A 37-token prompt forked into 3 beams: the beams share the prompt's blocks, the
    first append copies the shared partial block, and every beam then grows on its own.
    Decoding all four sequences over aliased tables equals the oracle over each one's own
    tokens; pool usage is far below four separate copies."""
    hq, hkv, d, prompt, steps = 16, 4, 128, 37, 21
    gen = torch.Generator().manual_seed(11)

    def rows(n):
        k = torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16)
        v = torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16)
        return k, v

    nb = 64
    m = pkv.BlockManager(nb, max_seqs=8, max_blocks_per_seq=8)
    pool = pkv.PagedKVPool(nb, hkv, d, kv)
    fill_pool_garbage(pool)

    p = m.add_sequence()
    k, v = rows(prompt)
    slots, pairs = m.append([p], [prompt])
    assert len(pairs) == 0
    pool.reshape_and_cache(k.cuda(), v.cuda(), slots.cuda())
    base = [(W.bf16_bits(k[i]), W.bf16_bits(v[i])) for i in range(prompt)]
    seqs = [p] + [m.fork(p) for _ in range(3)]
    logical = {s: list(base) for s in seqs}
    used_after_fork = nb - m.stats()[0]
    total_copies = 0
    for step in range(steps):
        k, v = rows(len(seqs))
        slots, pairs = m.append(seqs, [1] * len(seqs))
        if len(pairs):
            total_copies += len(pairs)
            pkv.copy_blocks(pool, pairs.cuda())
        pool.reshape_and_cache(k.cuda(), v.cuda(), slots.cuda())
        for i, s in enumerate(seqs):
            logical[s].append((W.bf16_bits(k[i]), W.bf16_bits(v[i])))
    assert total_copies == 3  # three of the four sharers copy the partial block; the last keeps it
    bt, cl = m.tables(seqs)
    assert cl.tolist() == [prompt + steps] * 4
    # the two full prompt blocks are shared by all four sequences
    assert all(m.refcount(b) == 4 for b in bt[0, :prompt // 16].tolist())
    used = nb - m.stats()[0]
    assert used < 4 * ((prompt + steps + 15) // 16) and used > used_after_fork

    q = torch.randn(len(seqs), hq, d, generator=gen).to(torch.bfloat16)
    scale = d ** -0.5
    out = pool.decode(q.cuda(), bt.cuda(), cl.cuda(), scale, int(cl.max()), kernel=kernel)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    ref = _oracle_for([logical[s] for s in seqs], W.bf16_bits(q), kv, hkv, d, scale)
    compare(out, ref, f"beams {kv} {kernel}")
    for s in seqs:
        m.free_sequence(s)
    assert m.stats() == (nb, 0)
    pool.close()
