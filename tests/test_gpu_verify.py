"""GPU parity for multi-query decode (verifying k draft tokens in one pass; "Lesson 4",
5.2 "Speculative Decoding": the target model scores every draft at once).  The k queries
of a sequence are its last k cached tokens, and query i attends causally to the tokens up
to its own position.  The CUDA path runs through the C ABI; the fp64 oracle's
paged_decode_multi gives the reference on the same seeded inputs.  Pools are pre-filled
with NaN so that a read past the context, or past a query's causal cut into a slot never
written, would show."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import compare, fill_pool_garbage, gpu_pool_from, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def verify_case(lens, hq, hkv, d, k, kv="bf16", seed=21):
    return W.build(name="verify", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                   kv_dtype=kv, seed=seed, num_queries=k)


def plan_or_skip(w, kv, kernel, partition_blocks=0):
    pool = pkv.PagedKVPool(1, w.num_kv_heads, w.head_dim, kv, fill=0)
    try:
        return pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len,
                               partition_blocks=partition_blocks, kernel=kernel,
                               num_queries=w.num_queries)
    except pkv.PagedKVError as e:
        assert "unsupported" in str(e)
        pytest.skip(f"{kernel} kernel not built for {w.num_q_heads // w.num_kv_heads} x {w.num_queries} columns")
    finally:
        pool.close()


def check_verify(w, kv, kernel=0, partition_blocks=0, seqs=None):
    plan = plan_or_skip(w, kv, kernel, partition_blocks)
    pool = gpu_pool_from(w, kv)
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale,
                      w.max_context_len, partition_blocks=partition_blocks, kernel=kernel)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    assert out.shape == w.q.shape
    ref, _, _ = oracle_decode(w, kv, seqs)
    sel = list(range(w.num_seqs)) if seqs is None else list(seqs)
    res = compare(out[torch.tensor(sel, device=out.device)], ref,
                  f"verify k={w.num_queries} {kv} P={partition_blocks} {kernel} ({plan['kernel']})")
    pool.close()
    return out, res


VERIFY_SHAPES = [
    # lens (each >= k), Hq, Hkv, d, k
    ([4, 5, 17, 33, 100, 250], 4, 4, 128, 4),     # MHA: 4 columns
    ([3, 16, 18, 47, 300], 8, 4, 64, 3),          # GQA 2 x 3 = 6 columns (8 slots)
    ([5, 17, 64, 129, 700], 32, 8, 128, 4),       # GQA 4 x 4 = 16 columns
    ([2, 31, 200], 16, 2, 128, 2),                # GQA 8 x 2 = 16 columns
    ([8, 40, 511], 8, 8, 128, 8),                 # MHA: 8 columns
    ([16, 33, 100], 4, 4, 64, 16),                # MHA: 16 columns, the most queries
    ([7, 20, 90], 8, 4, 128, 5),                  # GQA 2 x 5 = 10 columns (16 slots)
    ([2, 15, 16, 17, 32, 33], 4, 2, 128, 2),      # causal cut on block boundaries
    ([4, 33, 150], 16, 2, 128, 4),                # GQA 8 x 4 = 32 columns: two chunks
    ([16, 40, 200], 16, 2, 64, 16),               # GQA 8 x 16 = 128 columns: eight chunks
]
SHAPE_IDS = [f"Hq{s[1]}_Hkv{s[2]}_d{s[3]}_k{s[4]}" for s in VERIFY_SHAPES]


@pytest.mark.parametrize("kernel", ["auto", "cuda_core", "tensor_core"])
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("shape", VERIFY_SHAPES, ids=SHAPE_IDS)
def test_verify_shapes(shape, kv, kernel):
    lens, hq, hkv, d, k = shape
    check_verify(verify_case(lens, hq, hkv, d, k, kv), kv, kernel)


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("partition_blocks", [1, 2, 3, 64])
@pytest.mark.parametrize("heads", [(4, 4), (16, 8)], ids=["mha", "gqa2"])
def test_verify_partition_sweep(heads, partition_blocks, kv, kernel):
    """Split-K with causal cuts: with one block per partition the last partition of a
    sequence can hold tokens that only some queries see (its other columns end with an
    empty softmax state that the merge must ignore)."""
    hq, hkv = heads
    w = verify_case([4, 17, 18, 33, 95, 300], hq, hkv, 128, 4, kv, seed=23)
    check_verify(w, kv, kernel, partition_blocks)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_one_query_equals_plain_decode(kv):
    """k = 1 through a 4-D q is the plain decode, bit for bit."""
    w = W.build(name="k1", context_lens=[1, 17, 90, 400], num_q_heads=16, num_kv_heads=4, head_dim=128,
                kv_dtype=kv, seed=25)
    pool = gpu_pool_from(w, kv)
    args = (w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len)
    a = pool.decode(w.q.cuda(), *args)
    b = pool.decode(w.q.cuda()[:, None].contiguous(), *args)
    torch.cuda.synchronize()
    assert b.shape == (4, 1, 16, 128)
    assert torch.equal(a.view(torch.int16), b[:, 0].view(torch.int16))
    pool.close()


def test_context_shorter_than_k_is_flagged():
    """A sequence with T_b < k is out of range: zero output and the context-length bit; the
    other sequences are unaffected."""
    w = verify_case([20, 40, 9], 8, 4, 128, 4, seed=27)
    pool = gpu_pool_from(w, "bf16")
    lens = w.context_lens.clone()
    lens[2] = 3
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), lens.cuda(), w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert pool.device_error() & pkv.DEVERR_CONTEXT_LEN
    assert (out[2].float() == 0).all()
    ref, _, _ = oracle_decode(w, "bf16", [0, 1])
    compare(out[:2], ref, "verify neighbours of a short sequence")
    pool.close()


def test_plan_limits():
    pool = pkv.PagedKVPool(4, 8, 128, "bf16", fill=0)
    assert pkv.decode_plan(pool, 2, 32, 64, num_queries=4)["kernel"] == "tensor_core"   # 16 columns
    assert pkv.decode_plan(pool, 2, 8, 64, num_queries=4)["kernel"] == "tensor_core"    # MHA, 4 columns
    assert pkv.decode_plan(pool, 2, 8, 64, num_queries=1)["kernel"] == "tensor_core"    # MHA decode
    assert pkv.decode_plan(pool, 2, 8, 64, kernel="cuda_core")["kernel"] == "cuda_core"
    assert pkv.decode_plan(pool, 2, 64, 64, num_queries=4)["kernel"] == "tensor_core"   # 32 columns, 2 chunks
    assert pkv.decode_plan(pool, 2, 32, 64, num_queries=4, kernel="cuda_core")["kernel"] == "cuda_core"
    for bad_k in (17, -1):
        with pytest.raises(pkv.PagedKVError, match="invalid"):
            pkv.decode_plan(pool, 2, 8, 64, num_queries=bad_k)
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        pkv.decode_plan(pool, 2, 8, 3, num_queries=4)                  # max_context_len < k
    pool.close()
    for kv in ("int8", "fp8"):
        pool = pkv.PagedKVPool(4, 4, 64, kv, fill=0)                   # quantised pools at d = 64
        assert pkv.decode_plan(pool, 2, 8, 64, num_queries=4)["kernel"] == "tensor_core"
        assert pkv.decode_plan(pool, 2, 16, 64, num_queries=4)["kernel"] == "tensor_core"  # 16 columns
        assert pkv.decode_plan(pool, 2, 16, 64, num_queries=4, kernel="cuda_core")["kernel"] == "cuda_core"
        pool.close()


@pytest.mark.parametrize("name", ["llama2_7b_verify4", "llama3_8b_gqa_verify4"])
def test_named_verify_workload_full_size(name):
    """The full-size verification workloads in the benchmark's launch configuration; the
    oracle checks sampled sequences (shortest, longest, median, random)."""
    w = W.make(name, device="cuda")
    lens = w.context_lens.numpy()
    order = np.argsort(lens)
    rng = np.random.default_rng(0)
    seqs = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])} |
                  {int(x) for x in rng.choice(w.num_seqs, size=4, replace=False)})
    check_verify(w, "bf16", 0, 0, seqs)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_speculative_rounds_with_block_manager(kv):
    """Several draft-and-verify rounds over a block-managed pool: append k drafts per
    sequence (reshape_and_cache through the manager's slots), verify them in one call, keep
    a random accepted prefix (truncate), repeat.  Every verify output equals the oracle over
    each sequence's current tokens."""
    hq, hkv, d, k = 16, 4, 128, 4
    gen = torch.Generator().manual_seed(29)
    nb = 96
    m = pkv.BlockManager(nb, max_seqs=8, max_blocks_per_seq=16)
    pool = pkv.PagedKVPool(nb, hkv, d, kv)
    fill_pool_garbage(pool)
    seqs = [m.add_sequence() for _ in range(3)]
    tokens = {s: [] for s in seqs}

    def append(counts):
        kk = torch.randn(sum(counts), hkv, d, generator=gen).to(torch.bfloat16)
        vv = torch.randn(sum(counts), hkv, d, generator=gen).to(torch.bfloat16)
        slots, pairs = m.append(seqs, counts)
        if len(pairs):
            pkv.copy_blocks(pool, pairs.cuda())
        pool.reshape_and_cache(kk.cuda(), vv.cuda(), slots.cuda())
        r = 0
        for s, c in zip(seqs, counts):
            tokens[s].extend((kk[r + i], vv[r + i]) for i in range(c))
            r += c

    append([5, 19, 40])  # prompts
    rng = np.random.default_rng(3)
    for _ in range(4):
        append([k] * len(seqs))
        bt, cl = m.tables(seqs)
        q = torch.randn(len(seqs), k, hq, d, generator=gen).to(torch.bfloat16)
        out = pool.decode(q.cuda(), bt.cuda(), cl.cuda(), d ** -0.5, int(cl.max()))
        torch.cuda.synchronize()
        assert pool.device_error() == 0
        lens = [len(tokens[s]) for s in seqs]
        assert cl.tolist() == lens
        w = W.Workload(name="spec", num_seqs=len(seqs), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       kv_dtype=kv, num_blocks=nb, context_lens=cl, block_tables=bt,
                       slot_mapping=torch.zeros(0, dtype=torch.int32),
                       seq_offsets=torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64),
                       q=q, key=torch.stack([t[0] for s in seqs for t in tokens[s]]),
                       value=torch.stack([t[1] for s in seqs for t in tokens[s]]), scale=d ** -0.5,
                       seed=0, num_queries=k)
        ref, _, _ = oracle_decode(w, kv)
        compare(out, ref, f"speculative round {kv}")
        for s in seqs:  # accept a prefix of the drafts
            keep = len(tokens[s]) - k + int(rng.integers(0, k + 1))
            m.truncate(s, keep)
            del tokens[s][keep:]
    pool.close()
