"""GPU parity for sliding-window decode ("LLM/MLLM inference optimisation", 2.3: keep only
the most recent window of the KV cache): each query attends to its last W tokens.  The CUDA
path runs through the C ABI against the fp64 oracle's windowed decode.  Pools are filled
with NaN first, and in several tests the blocks behind the window are released (-1 table
entries, NaN contents), so any read outside the window would show."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import BF16_NAN, compare, fill_pool_garbage, gpu_pool_from, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


def case(lens, hq, hkv, d, k=1, kv="bf16", seed=41):
    return W.build(name="window", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                   kv_dtype=kv, seed=seed, num_queries=k)


def poison(pool, phys, lo=0, hi=16):
    """Slots lo..hi-1 of a block (every kv head) -> NaN values / NaN scales / E4M3 NaN codes."""
    if pool.dtype == "bf16":
        pool.k_cache[phys, :, lo:hi].view(torch.int16).fill_(BF16_NAN)
        pool.v_cache[phys, :, lo:hi].view(torch.int16).fill_(BF16_NAN)
    else:
        if pool.dtype == "fp8":
            pool.k_cache[phys, :, lo:hi].fill_(0x7F)
            pool.v_cache[phys, :, lo:hi].fill_(0x7F)
        pool.k_scale[phys, :, lo:hi].fill_(float("nan"))
        pool.v_scale[phys, :, lo:hi].fill_(float("nan"))


def release_behind(pool, w, window):
    """Table with -1 for every block before the first one any query sees, those blocks
    poisoned in the pool, and the first block's slots before every window poisoned too."""
    tab = w.block_tables.clone()
    k = w.num_queries
    for b, t_len in enumerate(w.context_lens.tolist()):
        lo = max(0, t_len - (k - 1) - window)  # first token any query sees
        first = lo // 16
        for j in range(first):
            poison(pool, int(tab[b, j]))
            tab[b, j] = -1
        if lo % 16:
            poison(pool, int(tab[b, first]), 0, lo % 16)
    return tab


def check_window(w, kv, window, kernel=0, partition_blocks=0, release=True):
    try:
        pkv.decode_plan(pkv.PagedKVPool(1, w.num_kv_heads, w.head_dim, kv, fill=0), w.num_seqs,
                        w.num_q_heads, w.max_context_len, kernel=kernel, num_queries=w.num_queries,
                        window=window)
    except pkv.PagedKVError as e:
        assert "unsupported" in str(e)
        pytest.skip(f"{kernel} kernel not built for this shape")
    pool = gpu_pool_from(w, kv)
    tab = release_behind(pool, w, window) if release else w.block_tables
    out = pool.decode(w.q.cuda(), tab.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len,
                      partition_blocks=partition_blocks, kernel=kernel, window=window)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    ref, _, _ = oracle_decode(w, kv, window=window)
    # A window of a few tokens makes each output an average of a few V values (one, for
    # W = 1: s * code for INT8), so the bf16 rounding of the output itself is counted in
    # the mean bound, as for other single-value outputs.
    res = compare(out, ref, f"window {window} k={w.num_queries} {kv} P={partition_blocks} {kernel}",
                  output_rounding=window < 16)
    pool.close()
    return res


SHAPES = [
    # lens, Hq, Hkv, d, k
    ([1, 15, 16, 17, 40, 100, 333], 8, 8, 128, 1),   # MHA
    ([5, 31, 64, 129, 300], 16, 4, 128, 1),          # GQA 4
    ([4, 20, 90, 260], 8, 4, 64, 3),                 # GQA 2 x 3 queries, d 64
    ([8, 70, 200], 32, 8, 128, 4),                   # GQA 4 x 4 queries (16 columns)
]


@pytest.mark.parametrize("kernel", ["auto", "cuda_core", "tensor_core"])
@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("window", [1, 7, 16, 33, 128, 5000])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"Hq{s[1]}_Hkv{s[2]}_d{s[3]}_k{s[4]}" for s in SHAPES])
def test_window_shapes(shape, window, kv, kernel):
    lens, hq, hkv, d, k = shape
    check_window(case(lens, hq, hkv, d, k, kv), kv, window, kernel)


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("partition_blocks", [1, 2, 3, 8])
@pytest.mark.parametrize("window", [16, 50, 200])
def test_window_partitions(window, partition_blocks, kernel):
    """Split-K over the window's blocks only: partitions start at the first visible block."""
    w = case([3, 17, 95, 300, 613], 16, 4, 128, 2, "bf16", seed=43)
    check_window(w, "bf16", window, kernel, partition_blocks)


def test_window_longer_than_context_is_full_attention():
    w = case([5, 40, 300], 16, 4, 128, 1, "bf16", seed=45)
    pool = gpu_pool_from(w, "bf16")
    args = (w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len)
    a = pool.decode(*args)
    b = pool.decode(*args, window=300)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    pool.close()


def test_window_plan_reads_fewer_blocks():
    pool = pkv.PagedKVPool(4, 32, 128, "bf16", fill=0)
    full = pkv.decode_plan(pool, 8, 32, 32768, partition_blocks=64)
    win = pkv.decode_plan(pool, 8, 32, 32768, partition_blocks=64, window=4096)
    # 2048 blocks: 32 partitions of 64; the window's 257 blocks: 4, the last taking the
    # 1-block remainder (a remainder of at most P / 4 joins the last partition)
    assert full["max_partitions"] == 32 and win["max_partitions"] == 4
    assert pkv.decode_workspace_bytes(pool, 8, 32, 32768, 64, window=4096) < \
        pkv.decode_workspace_bytes(pool, 8, 32, 32768, 64)
    with pytest.raises(pkv.PagedKVError, match="invalid"):
        pkv.decode_plan(pool, 8, 32, 32768, window=-1)
    pool.close()


def test_window_bound_plan_runs_one_wave():
    """When the window, not the lengths, bounds every unit's blocks and the units fit on the
    GPU at once, the automatic plan splits each unit into equal items that run in one wave
    on the grid; with more units than fit, the general rule applies."""
    pool = pkv.PagedKVPool(4, 32, 128, "bf16", fill=0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one = pkv.decode_plan(pool, 8, 32, 32768, window=4096)      # 256 units, 257-block bound
    parts = one["max_partitions"]
    assert parts >= 1 and 256 * parts <= 4 * sms                 # one wave (at most 4 CTAs per SM)
    assert one["partition_blocks"] == -(-257 // parts)             # equal items, no short tail
    if parts == 1:
        assert one["kernels_per_call"] == 1                        # no partials, no merge kernel
    many = pkv.decode_plan(pool, 256, 32, 32768, window=4096)   # 8192 units: more than one wave
    assert many["max_partitions"] > 1 and many["partition_blocks"] <= 128
    nowin = pkv.decode_plan(pool, 8, 32, 32768)                   # no window: lengths unknown
    assert nowin["max_partitions"] > parts
    pool.close()


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_sliding_window_generation_with_block_manager(kv):
    """A generation loop under a 40-token window: each step appends one token per sequence,
    decodes with the window, then releases the blocks the next step no longer needs.  Blocks
    in use stay bounded by the window, and every step equals the oracle."""
    hq, hkv, d, win = 8, 4, 128, 40
    gen = torch.Generator().manual_seed(47)
    nb = 64
    m = pkv.BlockManager(nb, max_seqs=4, max_blocks_per_seq=32)
    pool = pkv.PagedKVPool(nb, hkv, d, kv)
    fill_pool_garbage(pool)
    seqs = [m.add_sequence() for _ in range(3)]
    tokens = {s: [] for s in seqs}

    def append(counts):
        kk = torch.randn(sum(counts), hkv, d, generator=gen).to(torch.bfloat16)
        vv = torch.randn(sum(counts), hkv, d, generator=gen).to(torch.bfloat16)
        slots, pairs = m.append(seqs, counts)
        assert len(pairs) == 0
        pool.reshape_and_cache(kk.cuda(), vv.cuda(), slots.cuda())
        r = 0
        for s, c in zip(seqs, counts):
            tokens[s].extend((kk[r + i], vv[r + i]) for i in range(c))
            r += c

    append([30, 55, 90])
    for step in range(12):
        append([1, 1, 1])
        bt, cl = m.tables(seqs)
        q = torch.randn(len(seqs), hq, d, generator=gen).to(torch.bfloat16)
        out = pool.decode(q.cuda(), bt.cuda(), cl.cuda(), d ** -0.5, int(cl.max()), window=win)
        torch.cuda.synchronize()
        assert pool.device_error() == 0
        if step % 4 == 3:  # check against the oracle on every fourth step
            lens = [len(tokens[s]) for s in seqs]
            full_bt = torch.tensor(np.arange(len(seqs) * 32, dtype=np.int32).reshape(len(seqs), 32))
            wk = W.Workload(name="win", num_seqs=len(seqs), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                            kv_dtype=kv, num_blocks=nb, context_lens=cl, block_tables=full_bt,
                            slot_mapping=torch.zeros(0, dtype=torch.int32),
                            seq_offsets=torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64),
                            q=q, key=torch.stack([t[0] for s in seqs for t in tokens[s]]),
                            value=torch.stack([t[1] for s in seqs for t in tokens[s]]), scale=d ** -0.5, seed=0)
            ref, _, _ = oracle_decode(wk, kv, window=win)
            compare(out, ref, f"sliding window step {step} {kv}")
        for s, t_len in zip(seqs, cl.tolist()):
            m.release_before(s, max(0, t_len + 1 - win))  # what the next step's window needs
        used = nb - m.stats()[0]
        assert used <= len(seqs) * ((win + 15) // 16 + 1)
    pool.close()


def test_named_window_workload_full_size():
    """long_32k_window4k in the benchmark's launch configuration, sampled sequences."""
    w = W.make("long_32k_window4k", device="cuda")
    pool = gpu_pool_from(w, "bf16")
    out = pool.decode(w.q, w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len,
                      window=4096)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    seqs = [0, 5]
    ref, _, _ = oracle_decode(w, "bf16", seqs, window=4096)
    compare(out[torch.tensor(seqs, device=out.device)], ref, "long_32k_window4k")
    pool.close()
