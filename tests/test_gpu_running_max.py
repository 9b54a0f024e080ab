"""GPU parity on logit and V-scale patterns that move the softmax's running max, and the
quantised pools' V exponent, in the middle of a sequence ("LLM/MLLM inference
optimisation", section 3.2: the online softmax keeps a running max and a running sum over
the tiles).  The tensor-core kernel keeps its max until a logit passes it by a fixed
headroom, so probabilities above 1 meet the PV product and the sums between two moves;
the patterns below make it move often (a steady ramp), in jumps (a sawtooth) and on
isolated tokens (spikes), upwards for some heads and downwards for the others.  The fp64
oracle gives the reference on the same inputs."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import MAX_ABS, MEAN_ABS, gpu_pool_from, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def logit_pattern(kind: str, n: int, gen: torch.Generator) -> torch.Tensor:
    """Target logits (natural units) of a sequence's n tokens."""
    t = torch.arange(n, dtype=torch.float64)
    if kind == "ramp":        # +0.46 log2 units per block: the max moves every ~17 blocks
        return 0.02 * t
    if kind == "sawtooth":    # plateaus 100 tokens long, jumps of 6 (8.7 log2 units)
        return 6.0 * ((t // 100) % 3)
    spikes = torch.zeros(n, dtype=torch.float64)  # N(0,1) with runs of +12 on a few tokens
    spikes += torch.randn(n, generator=gen, dtype=torch.float64)
    for start in torch.randint(0, max(1, n - 4), (3,), generator=gen).tolist():
        spikes[start:start + 4] += 12.0
    return spikes


def patterned(lens, hq, hkv, d, kv, k=1, seed=31):
    """A workload whose logits follow logit_pattern: q is +1 on every dim for even heads
    and -1 for odd heads (so odd heads see the pattern upside down), and key token t is
    a_t / (scale * d) on every dim plus small noise.  V rows are N(0,1) clipped to
    [-3, 3] and scaled by a factor growing from 1/4 to 1 along the sequence, so that the
    quantised pools' V scales cross two binades."""
    w = W.build(name="running_max", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                kv_dtype=kv, seed=seed, num_queries=k)
    gen = torch.Generator().manual_seed(seed)
    kinds = ["ramp", "sawtooth", "spikes"]
    key = torch.empty(w.key.shape, dtype=torch.float64)
    value = torch.empty(w.value.shape, dtype=torch.float64)
    for b, n in enumerate(lens):
        lo = int(w.seq_offsets[b])
        a = logit_pattern(kinds[b % 3], n, gen)
        noise = 0.3 * torch.randn(n, hkv, d, generator=gen, dtype=torch.float64)
        key[lo:lo + n] = (a / (w.scale * d))[:, None, None] + noise
        grow = 0.25 + 0.75 * torch.arange(n, dtype=torch.float64) / max(1, n - 1)
        v = torch.randn(n, hkv, d, generator=gen, dtype=torch.float64).clamp(-3.0, 3.0)
        value[lo:lo + n] = v * grow[:, None, None]
    w.key = key.to(torch.bfloat16)
    w.value = value.to(torch.bfloat16)
    sign = torch.where(torch.arange(hq) % 2 == 0, 1.0, -1.0)
    w.q = (torch.ones(w.q.shape, dtype=torch.float32) * sign[:, None]).to(torch.bfloat16)
    return w


def plan_or_skip(w, kv, kernel):
    pool = pkv.PagedKVPool(1, w.num_kv_heads, w.head_dim, kv, fill=0)
    try:
        return pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len, kernel=kernel,
                               num_queries=w.num_queries)
    except pkv.PagedKVError as e:
        assert "unsupported" in str(e)
        pytest.skip(f"{kernel} kernel not built for this shape")
    finally:
        pool.close()


def check(w, kv, kernel, partition_blocks=0):
    plan_or_skip(w, kv, kernel)
    pool = gpu_pool_from(w, kv)
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale,
                      w.max_context_len, partition_blocks=partition_blocks, kernel=kernel)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    ref, _, _ = oracle_decode(w, kv)
    got = out.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    # Spiky softmaxes put single V values (|v| < 3) in the output, whose own bf16 rounding
    # (2^-9 relative) is allowed on top of the absolute bars.
    assert np.all(err <= MAX_ABS + 2.0 ** -8 * np.abs(ref)), f"max err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS + 2.0 ** -8 * np.abs(ref).mean(), f"mean err {err.mean():.3e}"
    pool.close()


SHAPES = [
    # lens, Hq, Hkv, d
    ([1500, 900, 700, 333, 1200, 17], 8, 2, 128),   # GQA 4
    ([1000, 640, 1100], 4, 4, 128),                  # MHA
    ([800, 260, 999], 8, 4, 64),                     # GQA 2, head_dim 64
]


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"Hq{s[1]}_Hkv{s[2]}_d{s[3]}")
def test_running_max_patterns(shape, kv, kernel):
    lens, hq, hkv, d = shape
    check(patterned(lens, hq, hkv, d, kv), kv, kernel)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("partition_blocks", [3, 16])
def test_running_max_patterns_split(kv, partition_blocks):
    """The same patterns cut into context partitions: each partition keeps its own lazy
    max and the merge brings them to a common one."""
    check(patterned([1500, 900, 700], 8, 2, 128, kv), kv, "tensor_core", partition_blocks)


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("k", [2, 4])
def test_running_max_patterns_multi_query(kv, k):
    """Several query tokens per sequence: every column keeps its own max behind its own
    causal cut."""
    check(patterned([1500, 900, 701, 64], 8, 2, 128, kv, k=k), kv, "tensor_core")
