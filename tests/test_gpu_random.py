"""Seeded random parity sweep: every feature of the decode at once -- GQA group, head_dim,
pool type, kernel family, query tokens per sequence, sliding window, partition size and
ragged lengths (T = k, block boundaries, one-block windows) -- drawn at random per case and
compared with the fp64 oracle through the C ABI.  Pools are pre-filled with NaN."""

import random

import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import compare, few_token_queries, gpu_pool_from, oracle_decode

pytestmark = pytest.mark.gpu

N_CASES = 400


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def draw(seed):
    r = random.Random(seed)
    d = r.choice([64, 128])
    kv = r.choice(["bf16", "int8", "fp8"])
    group = r.choice([1, 2, 3, 4, 6, 8, 12, 16])
    hkv = r.choice([1, 2, 4])
    k = r.choice([1, 1, 2, 3, 4, 5, 8, 16])
    window = r.choice([0, 0, 1, 7, 16, 17, 50, 300])
    kernel = r.choice(["auto", "cuda_core", "tensor_core"])
    pb = r.choice([0, 0, 1, 2, 3, 7])
    b = r.randint(1, 6)
    lens = []
    for _ in range(b):
        kind = r.random()
        if kind < 0.15:
            lens.append(k)                                   # every token is a query
        elif kind < 0.35:
            lens.append(max(k, 16 * r.randint(1, 8) + r.choice([-1, 0, 1])))  # block edges
        else:
            lens.append(r.randint(k, 400))
    return dict(d=d, kv=kv, hq=group * hkv, hkv=hkv, k=k, window=window, kernel=kernel, pb=pb, lens=lens)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    c = draw(1000 + seed)
    w = W.build(name="random", context_lens=c["lens"], num_q_heads=c["hq"], num_kv_heads=c["hkv"],
                head_dim=c["d"], kv_dtype=c["kv"], seed=seed, num_queries=c["k"])
    probe = pkv.PagedKVPool(1, c["hkv"], c["d"], c["kv"], fill=0)
    try:
        pkv.decode_plan(probe, w.num_seqs, c["hq"], w.max_context_len, c["pb"], kernel=c["kernel"],
                        num_queries=c["k"], window=c["window"])
    except pkv.PagedKVError as e:
        assert "unsupported" in str(e)
        pytest.skip(f"not built: {c}")
    finally:
        probe.close()
    pool = gpu_pool_from(w, c["kv"])
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len,
                      partition_blocks=c["pb"], kernel=c["kernel"], window=c["window"])
    torch.cuda.synchronize()
    assert pool.device_error() == 0, c
    ref, _, _ = oracle_decode(w, c["kv"], window=c["window"])
    # Queries that attend to only a few tokens return (nearly) single V values: only their
    # outputs get the slack of their own bf16 rounding, as for other single-value outputs.
    few = few_token_queries(c["lens"], c["k"], c["window"])  # [B, k]
    mask = few[:, 0, None, None] if ref.ndim == 3 else few[:, :, None, None]
    compare(out, ref, str(c), output_rounding=mask)
    pool.close()
