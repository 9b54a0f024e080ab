"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle on the
same seeded inputs.

Bars: slot writes and INT8 codes/scales bit-exact; attention outputs within max-abs
1e-2 and mean-abs 1e-3 (bf16 output, fp32 accumulation; the INT8 oracle runs on the
same dequantised values).  Pools are pre-filled with NaN so that any read of a slot that
was never written (the tail of a last block, unused blocks) would show.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import (compare, gpu_decode, gpu_pool_blocks, gpu_pool_from, oracle_decode,
                         valid_slot_bytes_equal)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def custom(lens, hq, hkv, d, kv="bf16", seed=7, **kw):
    return W.build(name="custom", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                   kv_dtype=kv, seed=seed, **kw)


KERNELS = ["cuda_core", "tensor_core"]


def supported(w, kv, kernel):
    """Whether the kernel family is built for this shape (the plan call says so)."""
    pool = pkv.PagedKVPool(1, w.num_kv_heads, w.head_dim, kv, fill=0)
    try:
        pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, 16, kernel=kernel)
        return True
    except pkv.PagedKVError as e:
        assert "unsupported" in str(e)
        return False
    finally:
        pool.close()


def check_all(w, kv, partition_blocks=0, seqs=None, kernel=0, output_rounding=False):
    if kernel and not supported(w, kv, kernel):
        pytest.skip(f"{kernel} kernel not built for this shape")
    pool = gpu_pool_from(w, kv)
    out = gpu_decode(pool, w, partition_blocks, kernel=kernel)
    assert pool.device_error() == 0
    ref, ref_pool, c = oracle_decode(w, kv, seqs)
    sel = list(range(w.num_seqs)) if seqs is None else list(seqs)
    valid_slot_bytes_equal(gpu_pool_blocks(pool, c["orig_tables"], c["lens"]), ref_pool, c["lens"])
    res = compare(out[torch.tensor(sel, device=out.device)], ref, f"{w.name}/{kv}/P={partition_blocks}/{kernel}",
                  output_rounding=output_rounding)
    pool.close()
    return out, res


# ------------------------------------------------------------ small shapes

@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_tiny_workload(kv):
    w = W.make("tiny")
    check_all(w, kv)


SHAPES = [
    # lens, Hq, Hkv, d
    ([1, 15, 16, 17, 33, 100], 4, 4, 64),
    ([1, 2, 31, 48, 257], 8, 4, 64),
    ([5, 16, 63, 200], 16, 4, 128),
    ([17, 40, 129, 511, 700], 8, 1, 128),
    ([3, 64, 65, 300], 32, 32, 128),
    ([1, 16, 18, 99, 1000], 8, 2, 128),
    ([7, 250, 33], 16, 2, 64),
]


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{len(s[0])}_Hq{s[1]}_Hkv{s[2]}_d{s[3]}")
def test_shapes_auto_plan(shape, kv):
    lens, hq, hkv, d = shape
    check_all(custom(lens, hq, hkv, d, kv), kv)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{len(s[0])}_Hq{s[1]}_Hkv{s[2]}_d{s[3]}")
def test_shapes_each_kernel(shape, kv, kernel):
    lens, hq, hkv, d = shape
    check_all(custom(lens, hq, hkv, d, kv), kv, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("partition_blocks", [1, 2, 3, 5, 8, 64])
def test_partition_sweep(partition_blocks, kv, kernel):
    """Split-K: any partition size gives the oracle's result (log-sum-exp merge)."""
    w = custom([1, 16, 17, 95, 300, 613], 16, 4, 128, kv, seed=9)
    check_all(w, kv, partition_blocks, kernel=kernel)


@pytest.mark.parametrize("kv", ["int8", "fp8"])
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("qscale", [3e4, 1e-5])
def test_int8_extreme_query_magnitudes(qscale, kernel, kv):
    """Very large and very small queries: the tensor-core path brings q into fp16 range
    with a power of two, which must not change the result.  Large queries make the
    softmax one-hot, so each output is a single O(1) value of V and its own bf16 rounding
    is counted in the mean bound."""
    w = custom([40, 333], 16, 4, 128, kv, seed=12)
    w.q = (w.q.float() * qscale).to(torch.bfloat16)
    check_all(w, kv, kernel=kernel, output_rounding=qscale > 1)


@pytest.mark.parametrize("kv", ["int8", "fp8"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_int8_value_scales_spanning_binades(kernel, kv):
    """V rows whose scales differ by up to 2^14 across and within blocks (the tensor-core
    path keeps P in fp16 with a growing block exponent).  Values stay below 4x N(0,1) so
    that the absolute tolerance still applies to the bf16 output."""
    w = custom([500, 70], 16, 4, 128, kv, seed=13)
    g = torch.Generator().manual_seed(3)
    mult = torch.pow(2.0, torch.randint(-12, 3, (w.value.shape[0], 1, 1), generator=g).float())
    w.value = (w.value.float() * mult).to(torch.bfloat16)
    check_all(w, kv, kernel=kernel)


def test_partitions_agree_with_each_other():
    w = custom([700, 1000, 33], 8, 2, 128, "bf16", seed=10)
    pool = gpu_pool_from(w, "bf16")
    outs = [gpu_decode(pool, w, pb).float() for pb in (1, 4, 16, 64)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-2
    pool.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_permutation_gives_identical_bits(kernel):
    """Two different shuffles of the same tokens into the pool give bit-identical output:
    the kernel's reduction order depends only on logical token positions."""
    outs = []
    for seed_shift in (0, 1):
        w = custom([5, 40, 333, 1024], 16, 4, 128, "bf16", seed=21)
        gen = torch.Generator().manual_seed(99 + seed_shift)
        perm = torch.randperm(w.num_blocks, generator=gen).to(torch.int32)
        tab = w.block_tables.clone()
        m = tab >= 0
        tab[m] = perm[tab[m].long()]
        t = torch.arange(w.num_tokens)
        seq = torch.repeat_interleave(torch.arange(w.num_seqs), w.context_lens.long())
        pos = t - w.seq_offsets[seq]
        w.block_tables = tab
        w.slot_mapping = (tab[seq, pos // 16].long() * 16 + pos % 16).to(torch.int32)
        pool = gpu_pool_from(w, "bf16")
        outs.append(gpu_decode(pool, w, kernel=kernel).cpu())
        pool.close()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_long_single_sequence():
    """The longest context these tests build: one sequence of 65536 tokens, GQA group 4."""
    w = custom([65536], 32, 8, 128, "bf16", seed=31)
    check_all(w, "bf16")


@pytest.mark.parametrize("kv", ["int8", "fp8"])
def test_quantised_zero_rows(kv):
    """An all-zero row quantises to scale 0 and zero codes, and decodes without NaN."""
    w = custom([20, 33], 8, 4, 64, kv, seed=41)
    w.key[3].zero_()
    w.value[7].zero_()
    w.value[20:30].zero_()
    check_all(w, kv)


@pytest.mark.parametrize("kv", ["int8", "fp8"])
def test_quantiser_bit_exact_many_rows(kv):
    """Codes and scales of 64k token-head rows equal the oracle's bit for bit."""
    n, hkv, d = 8192, 8, 128
    gen = torch.Generator().manual_seed(5)
    key = (torch.randn(n, hkv, d, generator=gen) * torch.rand(n, hkv, 1, generator=gen) * 10).to(torch.bfloat16)
    value = torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16)
    nb = n // 16 + 3
    slots = torch.randperm(nb * 16, generator=gen)[:n].to(torch.int32)
    pool = pkv.PagedKVPool(nb, hkv, d, kv, fill=0)
    pool.reshape_and_cache(key.cuda(), value.cuda(), slots.cuda())
    torch.cuda.synchronize()
    o = oracle.load()
    kc = np.zeros((nb, hkv, 16, d), np.int8 if kv == "int8" else np.uint8)
    vc, ks, vs = kc.copy(), np.zeros((nb, hkv, 16), np.float32), np.zeros((nb, hkv, 16), np.float32)
    write = o.reshape_and_cache_int8 if kv == "int8" else o.reshape_and_cache_fp8
    write(W.bf16_bits(key), W.bf16_bits(value), slots.numpy(), kc, vc, ks, vs)
    assert np.array_equal(pool.k_cache.cpu().numpy(), kc)
    assert np.array_equal(pool.v_cache.cpu().numpy(), vc)
    assert np.array_equal(pool.k_scale.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(pool.v_scale.cpu().numpy().view(np.uint32), vs.view(np.uint32))
    pool.close()


def test_bf16_cache_write_bit_exact_and_skips_negative_slots():
    n, hkv, d = 3000, 4, 64
    gen = torch.Generator().manual_seed(6)
    key = torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16)
    value = torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16)
    nb = n // 16 + 5
    slots = torch.randperm(nb * 16, generator=gen)[:n].to(torch.int32)
    slots[::5] = -1
    pool = pkv.PagedKVPool(nb, hkv, d, "bf16", fill=0)
    pool.k_cache.view(torch.int16).fill_(0x1234)
    pool.v_cache.view(torch.int16).fill_(0x1234)
    pool.reshape_and_cache(key.cuda(), value.cuda(), slots.cuda())
    torch.cuda.synchronize()
    o = oracle.load()
    kc = np.full((nb, hkv, 16, d), 0x1234, np.uint16)
    vc = kc.copy()
    o.reshape_and_cache_bf16(W.bf16_bits(key), W.bf16_bits(value), slots.numpy(), kc, vc)
    assert np.array_equal(W.bf16_bits(pool.k_cache), kc)
    assert np.array_equal(W.bf16_bits(pool.v_cache), vc)
    pool.close()


# ------------------------------------------------------------ named workloads

def _sample(w, k=6):
    lens = w.context_lens.numpy()
    order = np.argsort(lens)
    picks = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    rng = np.random.default_rng(0)
    picks.update(int(x) for x in rng.choice(w.num_seqs, size=min(k, w.num_seqs), replace=False))
    return sorted(picks)


@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "long_32k", "int8_cb", "fp8_cb", "int8_cb_d64"])
def test_named_workload_full_size(name):
    """Full-size workloads in the launch configuration the benchmark times (automatic
    plan); the oracle checks sampled sequences (shortest, longest, median, random)."""
    w = W.make(name, device="cuda")
    kv = W.SPECS[name].kv_dtype
    seqs = _sample(w)
    check_all(w, kv, 0, seqs)


@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "long_32k", "int8_cb", "fp8_cb", "int8_cb_d64"])
def test_named_workload_cuda_core_kernel(name):
    """The full-size workloads through the CUDA-core kernel too (auto picks the tensor
    cores wherever they are built)."""
    w = W.make(name, device="cuda")
    check_all(w, W.SPECS[name].kv_dtype, 0, _sample(w, 3), kernel="cuda_core")


def test_tiny_named_partitions():
    w = W.make("tiny")
    for pb in (1, 2, 3):
        check_all(w, "bf16", pb)


# ------------------------------------------------------------ errors and edges

def test_device_error_bits():
    w = custom([40, 20], 4, 4, 64, "bf16", seed=51)
    pool = gpu_pool_from(w, "bf16", garbage=False)
    bt = w.block_tables.clone()
    bt[0, 1] = w.num_blocks + 5  # out of range
    out = pool.decode(w.q.cuda(), bt.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert pool.device_error() & pkv.DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()

    lens = w.context_lens.clone()
    lens[1] = 0
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), lens.cuda(), w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert pool.device_error() & pkv.DEVERR_CONTEXT_LEN
    assert (out[1].float() == 0).all()

    lens[1] = w.max_context_len + 1  # beyond the declared maximum
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), lens.cuda(), w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert pool.device_error() & pkv.DEVERR_CONTEXT_LEN

    bad_slots = torch.tensor([w.num_blocks * 16, -1], dtype=torch.int32, device="cuda")
    kv = torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    pool.reshape_and_cache(kv, kv, bad_slots)
    torch.cuda.synchronize()
    assert pool.device_error() == pkv.DEVERR_SLOT
    assert pool.device_error() == 0  # reading clears it
    pool.close()


def test_empty_calls_are_noops():
    pool = pkv.PagedKVPool(4, 2, 64, "bf16", fill=0)
    before = pkv.launch_count()
    q = torch.empty(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    pool.decode(q, torch.empty(0, 1, dtype=torch.int32, device="cuda"),
                torch.empty(0, dtype=torch.int32, device="cuda"), 0.125, 16)
    e = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    pool.reshape_and_cache(e, e, torch.empty(0, dtype=torch.int32, device="cuda"))
    assert pkv.launch_count() == before
    pool.close()


def test_host_validation_errors():
    pool = pkv.PagedKVPool(4, 2, 64, "bf16", fill=0)
    q = torch.zeros(1, 3, 64, dtype=torch.bfloat16, device="cuda")  # 3 heads over 2 kv heads
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        pool.decode(q, torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                    torch.ones(1, dtype=torch.int32, device="cuda"), 1.0, 16)
    q = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PagedKVError, match="invalid"):  # max_context_len beyond the table
        pool.decode(q, torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                    torch.ones(1, dtype=torch.int32, device="cuda"), 1.0, 17)
    with pytest.raises(pkv.PagedKVError, match="workspace"):
        pkv.paged_attention_decode(pool, q, torch.zeros(1, 4, dtype=torch.int32, device="cuda"),
                                   torch.ones(1, dtype=torch.int32, device="cuda"), 1.0, 64,
                                   workspace=torch.empty(16, dtype=torch.uint8, device="cuda"),
                                   partition_blocks=1)
    pool.close()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_small_remainder_joins_last_partition(kv, kernel):
    """With partition size P, a remainder of at most P / 4 blocks is taken by a sequence's
    last partition (which then holds up to P + P / 4 blocks) instead of an item of its own.
    P = 16: 20 blocks are one item; 21 blocks two (16 + 5); 36 blocks two (16 + 20); 37
    blocks three (16 + 16 + 5); 15.4 blocks one; a one-token tail past 20 blocks two."""
    blocks = [20, 21, 36, 37]
    lens = [16 * n for n in blocks] + [15 * 16 + 7, 20 * 16 + 1, 20 * 16 - 9]
    w = custom(lens, 8, 2, 128, kv, seed=67)
    pool = pkv.PagedKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, kv, fill=0)
    for nblk, parts in ((20, 1), (21, 2), (36, 2), (37, 3)):
        plan = pkv.decode_plan(pool, 1, 8, 16 * nblk, partition_blocks=16, kernel=kernel)
        assert plan["max_partitions"] == parts, (nblk, plan)
        assert plan["kernels_per_call"] == (1 if parts == 1 else 2)
    pool.close()
    check_all(w, kv, 16, kernel=kernel)


def test_launch_count_and_plan():
    w = custom([300, 40], 8, 2, 128, "bf16", seed=61)
    pool = gpu_pool_from(w, "bf16", garbage=False)
    plan = pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len, partition_blocks=4)
    assert plan == {"partition_blocks": 4, "max_partitions": math.ceil(19 / 4), "kernels_per_call": 2,
                    "kernel": "tensor_core"}
    assert pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len,
                           kernel="cuda_core")["kernel"] == "cuda_core"
    before = pkv.launch_count()
    gpu_decode(pool, w, 4)
    assert pkv.launch_count() - before == 2
    plan1 = pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len, partition_blocks=64)
    assert plan1["kernels_per_call"] == 1
    before = pkv.launch_count()
    gpu_decode(pool, w, 64)
    assert pkv.launch_count() - before == 1
    pool.close()


def test_side_stream():
    w = custom([77, 150], 8, 8, 128, "bf16", seed=71)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pool = gpu_pool_from(w, "bf16")
        out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale,
                          w.max_context_len, stream=s)
    s.synchronize()
    ref, _, _ = oracle_decode(w, "bf16")
    compare(out, ref, "side stream")
    pool.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_repeated_calls_identical(kernel):
    """The persistent grid takes items from counters that the last CTA of each call resets;
    consecutive calls (and a split and an unsplit plan in between) give identical bits."""
    w = custom([5, 700, 40, 1500, 16, 333], 16, 4, 128, "bf16", seed=81)
    pool = gpu_pool_from(w, "bf16")
    outs = []
    for pb in (0, 0, 64, 0, 3, 0):
        out = torch.full_like(w.q.cuda(), float("nan"))
        pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len,
                    out=out, partition_blocks=pb, kernel=kernel)
        torch.cuda.synchronize()
        if pb == 0:
            outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert pool.device_error() == 0
    pool.close()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("partition_blocks", [0, 2])
def test_large_batch_classic_grid(kernel, partition_blocks):
    """More sequences than the persistent scheduler holds (4096): one CTA per item slot,
    with and without split sequences."""
    g = torch.Generator().manual_seed(91)
    lens = torch.randint(1, 70, (4200,), generator=g)
    w = custom(lens, 8, 2, 64, "bf16", seed=92)
    if partition_blocks:
        pool = pkv.PagedKVPool(1, 2, 64, "bf16", fill=0)
        assert pkv.decode_plan(pool, 4200, 8, int(lens.max()), partition_blocks)["kernels_per_call"] == 2
        pool.close()
    check_all(w, "bf16", partition_blocks, kernel=kernel, seqs=list(range(0, 4200, 97)))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("kv", ["bf16", "int8"])
@pytest.mark.parametrize("partition_blocks", [1, 2, 3])
@pytest.mark.parametrize("d", [64, 128])
def test_reduce_over_many_partitions(kv, kernel, partition_blocks, d):
    """More than 32 partitions per row: the reduce kernel's lanes then hold several
    partitions each and its accumulator loop runs past its look-ahead (125 blocks in 125, 63
    or 42 partitions), next to short sequences that do not split; both head sizes (the
    reduce reads 4 or 2 floats per lane)."""
    w = custom([2000, 33, 1999, 700], 8, 2, d, kv, seed=97)
    pool = pkv.PagedKVPool(1, 2, d, kv, fill=0)
    plan = pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, w.max_context_len, partition_blocks, kernel=kernel)
    pool.close()
    assert plan["max_partitions"] > 32
    check_all(w, kv, partition_blocks, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_batch_at_the_persistent_scheduler_limit(kernel):
    """Exactly 4096 sequences, the largest batch the persistent scheduler serves: its prefix
    sum then takes 16 KiB of shared memory per CTA.  Split sequences make the plan take it."""
    g = torch.Generator().manual_seed(93)
    lens = torch.randint(1, 200, (4096,), generator=g)
    w = custom(lens, 8, 2, 64, "int8", seed=94)
    pool = pkv.PagedKVPool(1, 2, 64, "int8", fill=0)
    plan = pkv.decode_plan(pool, 4096, 8, int(lens.max()), 4, kernel=kernel)
    pool.close()
    assert plan["kernels_per_call"] == 2
    check_all(w, "int8", 4, kernel=kernel, seqs=list(range(0, 4096, 61)) + [4095])


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_scheduler_counters_reset_between_calls(kv):
    """The persistent scheduler's counters live in the pool's device memory and reset
    themselves: alternating batches of different shapes and partition sizes on one pool
    give the oracle's result every time."""
    wa = custom([1, 40, 300, 613, 17], 16, 4, 128, kv, seed=95)
    wb = custom([700, 5, 129, 64, 33, 250, 90, 1000], 16, 4, 128, kv, seed=96)
    ref_a, _, _ = oracle_decode(wa, kv)
    ref_b, _, _ = oracle_decode(wb, kv)
    pa, pb = gpu_pool_from(wa, kv), gpu_pool_from(wb, kv)
    for rep in range(3):
        for w, pool, ref in ((wa, pa, ref_a), (wb, pb, ref_b)):
            for P in (1, 3, 0):
                out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale,
                                  w.max_context_len, partition_blocks=P)
                torch.cuda.synchronize()
                compare(out, ref, f"merge counters rep {rep} P={P}")
    assert pa.device_error() == 0 and pb.device_error() == 0
    pa.close()
    pb.close()


RING_SHAPES = [("bf16", 128, 2, 1), ("bf16", 128, 3, 1), ("bf16", 64, 3, 1), ("bf16", 64, 2, 2),
               ("int8", 128, 3, 1), ("int8", 128, 2, 2), ("int8", 128, 3, 2), ("int8", 128, 2, 1),
               ("fp8", 128, 3, 1), ("fp8", 128, 2, 2), ("fp8", 128, 3, 2), ("fp8", 128, 2, 1),
               ("int8", 64, 2, 2), ("int8", 64, 3, 1), ("fp8", 64, 2, 2), ("fp8", 64, 3, 1)]


@pytest.mark.parametrize("partition_blocks", [0, 3, 5])
@pytest.mark.parametrize("shape", RING_SHAPES, ids=lambda s: f"{s[0]}_d{s[1]}_S{s[2]}_B{s[3]}")
def test_tensor_core_ring_shapes(shape, partition_blocks):
    """Every built ring shape of the tensor-core kernel, with odd block counts per item so
    that a two-block stage is sometimes half empty."""
    kv, d, stages, bps = shape
    w = custom([1, 16, 17, 49, 95, 300, 613], 16, 4, d, kv, seed=101 + d)
    pool = gpu_pool_from(w, kv)
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len,
                      partition_blocks=partition_blocks, kernel="tensor_core", stages=stages,
                      blocks_per_stage=bps)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    ref, _, _ = oracle_decode(w, kv)
    compare(out, ref, f"ring {shape} P={partition_blocks}")
    pool.close()


def test_misaligned_out_rejected():
    """out must be 16-byte aligned (the merge writes vectors); a view 2 bytes into a buffer
    is refused before any launch."""
    w = custom([40, 17], 8, 2, 128, "bf16", seed=3)
    pool = gpu_pool_from(w, "bf16")
    buf = torch.empty(w.q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[1:1 + w.q.numel()].view(w.q.shape)
    with pytest.raises(pkv.PagedKVError):
        pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale,
                    w.max_context_len, out=out)
    assert pool.device_error() == 0
    pool.close()
