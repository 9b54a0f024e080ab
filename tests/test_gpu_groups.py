"""GPU parity for every query-head grouping: MHA, GQA with any group size G = Hq / Hkv
(powers of two or not) and MQA (one kv head for all query heads).  "LLM/MLLM inference
optimisation" 2.2 defines MQA as n_kv = 1 and GQA as 1 <= n_kv < n_head query heads
sharing each K/V head, and the 2.3 table lists both.  Query head h reads kv head h / G
(contiguous groups).  The CUDA path runs through the C ABI against the fp64 oracle on the
same seeded inputs; pools are pre-filled with NaN."""

import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import compare, gpu_pool_from, oracle_decode

pytestmark = pytest.mark.gpu

KERNELS = ["cuda_core", "tensor_core"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def case(lens, hq, hkv, d, kv, seed, k=1):
    return W.build(name="groups", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                   kv_dtype=kv, seed=seed, num_queries=k)


def plan_or_skip(w, kv, kernel, partition_blocks=0, window=0):
    pool = pkv.PagedKVPool(1, w.num_kv_heads, w.head_dim, kv, fill=0)
    try:
        return pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len, partition_blocks,
                               kernel=kernel, num_queries=w.num_queries, window=window)
    except pkv.PagedKVError as e:
        assert "unsupported" in str(e)
        pytest.skip(f"{kernel} kernel not built for {kv} head_dim {w.head_dim}")
    finally:
        pool.close()


def run(w, kv, kernel=0, partition_blocks=0, window=0, seqs=None):
    plan = plan_or_skip(w, kv, kernel, partition_blocks, window)
    pool = gpu_pool_from(w, kv)
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len,
                      partition_blocks=partition_blocks, kernel=kernel, window=window)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    ref, _, _ = oracle_decode(w, kv, seqs, window=window)
    sel = list(range(w.num_seqs)) if seqs is None else list(seqs)
    compare(out[torch.tensor(sel, device=out.device)], ref,
            f"G={w.num_q_heads // w.num_kv_heads} Hkv={w.num_kv_heads} {kv} {kernel} P={partition_blocks} "
            f"W={window} k={w.num_queries} ({plan['kernel']})")
    pool.close()
    return out


# (Hq, Hkv): groups 3, 5, 6, 7 (not powers of two), 12 (two n-tiles of a 16-column tile),
# 16 (a full 16-column tile), 24 and 32 (column chunks), MQA with 8 and 32 query heads.
GROUPS = [(3, 1), (6, 2), (10, 2), (14, 2), (24, 2), (16, 1), (48, 2), (32, 1), (8, 1)]
LENS = [1, 15, 16, 17, 70, 333]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("heads", GROUPS, ids=lambda h: f"Hq{h[0]}_Hkv{h[1]}")
def test_group_sizes_each_kernel(heads, kv, kernel):
    hq, hkv = heads
    run(case(LENS, hq, hkv, 128, kv, seed=hq * 7 + hkv), kv, kernel=kernel)


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("heads", [(3, 1), (12, 2), (32, 1)], ids=lambda h: f"Hq{h[0]}_Hkv{h[1]}")
def test_group_sizes_head_dim_64(heads, kv):
    hq, hkv = heads
    run(case(LENS, hq, hkv, 64, kv, seed=hq * 5 + hkv), kv)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("partition_blocks", [1, 3, 8])
@pytest.mark.parametrize("heads", [(6, 2), (32, 1)], ids=lambda h: f"Hq{h[0]}_Hkv{h[1]}")
def test_group_sizes_split(heads, partition_blocks, kernel):
    """Split-K partials and the reduce for odd and chunked groups."""
    hq, hkv = heads
    run(case([5, 100, 257, 600], hq, hkv, 128, "bf16", seed=31), "bf16", kernel=kernel,
        partition_blocks=partition_blocks)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", [(3, 1, 3), (6, 2, 4), (7, 1, 2), (32, 1, 2)], ids=lambda s: f"Hq{s[0]}_Hkv{s[1]}_k{s[2]}")
def test_group_sizes_multi_query(shape, kernel, kv):
    """Several query tokens per sequence: columns = G x k, each query with its causal cut."""
    hq, hkv, k = shape
    run(case([k, 16 + k, 90, 301], hq, hkv, 128, kv, seed=41, k=k), kv, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("heads", [(6, 2), (32, 1)], ids=lambda h: f"Hq{h[0]}_Hkv{h[1]}")
def test_group_sizes_window(heads, kernel):
    hq, hkv = heads
    run(case([9, 64, 250, 777], hq, hkv, 128, "bf16", seed=51), "bf16", kernel=kernel, window=100)


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_mqa_full_size(kv):
    """A full-size MQA batch: the LLaMA-2-7B-shaped lengths (64 sequences, uniform in
    [128, 2048]) with 32 query heads over one kv head, every sequence against the oracle."""
    lens = W.context_lens_of("llama2_7b")
    w = W.build(name="mqa", context_lens=lens, num_q_heads=32, num_kv_heads=1, head_dim=128, kv_dtype=kv,
                seed=77)
    out = run(w, kv)
    assert out.shape == (64, 32, 128)


def test_group_not_dividing_is_rejected():
    pool = pkv.PagedKVPool(4, 2, 64, "bf16", fill=0)
    q = torch.zeros(1, 5, 64, dtype=torch.bfloat16, device="cuda")  # 5 heads over 2 kv heads
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        pool.decode(q, torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                    torch.ones(1, dtype=torch.int32, device="cuda"), 1.0, 16)
    pool.close()
