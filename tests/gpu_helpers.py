"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the oracle
on the same seeded inputs, and compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W

MAX_ABS = 1e-2   # attention output tolerance (bf16 output, fp32 accumulation)
MEAN_ABS = 1e-3
BF16_NAN = 0x7FC0


def fill_pool_garbage(pool: pkv.PagedKVPool) -> None:
    """Fill every pool byte with NaN (bf16 / fp32) or 0x7f codes so that reading a slot
    that was never written shows up in the output."""
    if pool.dtype == "bf16":
        pool.k_cache.view(torch.int16).fill_(BF16_NAN)
        pool.v_cache.view(torch.int16).fill_(BF16_NAN)
    else:
        code = 127 if pool.dtype == "int8" else 0x7F  # 0x7F is an E4M3 NaN
        pool.k_cache.fill_(code)
        pool.v_cache.fill_(code)
        pool.k_scale.fill_(float("nan"))
        pool.v_scale.fill_(float("nan"))


def gpu_pool_from(w: W.Workload, kv: str, device="cuda", garbage=True, split_last=True) -> pkv.PagedKVPool:
    """Write the workload's tokens into a fresh pool with the library's cache write:
    first every token but each sequence's newest, then the newest tokens (a decode-step
    append)."""
    pool = pkv.PagedKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, kv, device=device)
    if garbage:
        fill_pool_garbage(pool)
    key, value = w.key.to(device), w.value.to(device)
    slots = w.slot_mapping.to(device)
    if split_last:
        for rows in (w.history_rows(), w.last_token_rows()):
            r = rows.to(device)
            if r.numel():
                pool.reshape_and_cache(key[r].contiguous(), value[r].contiguous(), slots[r].contiguous())
    else:
        pool.reshape_and_cache(key, value, slots)
    return pool


def gpu_decode(pool: pkv.PagedKVPool, w: W.Workload, partition_blocks=0, device="cuda",
               max_context_len=None, kernel=0) -> torch.Tensor:
    out = pool.decode(w.q.to(device), w.block_tables.to(device), w.context_lens.to(device), w.scale,
                      max_context_len or w.max_context_len, partition_blocks=partition_blocks,
                      kernel=kernel)
    torch.cuda.synchronize()
    return out


def compact_for_oracle(w: W.Workload, seqs):
    """Host inputs for the oracle restricted to sequences `seqs`: their blocks renumbered
    0..n-1 in table order (a relabelling of physical blocks, which the oracle's
    permutation-invariance pin shows does not change the result)."""
    seqs = list(seqs)
    tables = w.block_tables[seqs].numpy()
    lens = w.context_lens[seqs].numpy()
    nblk = (lens + 15) // 16
    new_tab = np.full((len(seqs), tables.shape[1]), -1, np.int32)
    cursor = 0
    for i, n in enumerate(nblk):
        new_tab[i, :n] = np.arange(cursor, cursor + n, dtype=np.int32)
        cursor += n
    rows, slots = [], []
    for i, b in enumerate(seqs):
        lo = int(w.seq_offsets[b])
        t = np.arange(int(lens[i]))
        rows.append(np.arange(lo, lo + int(lens[i])))
        slots.append(new_tab[i, t // 16] * 16 + t % 16)
    rows = np.concatenate(rows)
    slots = np.concatenate(slots).astype(np.int32)
    ridx = torch.from_numpy(rows)
    key = W.bf16_bits(w.key[ridx.to(w.key.device)])
    value = W.bf16_bits(w.value[ridx.to(w.value.device)])
    q = W.bf16_bits(w.q[torch.tensor(seqs, device=w.q.device)])
    return dict(q=q, key=key, value=value, slots=slots, tables=new_tab, lens=lens.astype(np.int32),
                num_blocks=max(cursor, 1), orig_tables=tables)


def oracle_decode(w: W.Workload, kv: str, seqs=None, o=None, q=None, window=0):
    """fp64 oracle output [len(seqs), Hq, d] (or [len(seqs), k, Hq, d] for a multi-query
    workload or a 4-D ``q``) plus its own pool (compacted).  ``window`` > 0: sliding-window
    attention over each query's last ``window`` tokens."""
    o = o or oracle.load()
    seqs = list(range(w.num_seqs)) if seqs is None else list(seqs)
    c = compact_for_oracle(w, seqs)
    if q is not None:
        c["q"] = W.bf16_bits(q[torch.tensor(seqs, device=q.device)])
    if window:
        single = c["q"].ndim == 3

        def decode(qb, *rest):
            out = o.paged_decode_multi(qb[:, None] if single else qb, *rest, window=window)
            return out[:, 0] if single else out
    else:
        decode = o.paged_decode_multi if c["q"].ndim == 4 else o.paged_decode
    shape = (c["num_blocks"], w.num_kv_heads, 16, w.head_dim)
    if kv == "bf16":
        kc, vc = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
        o.reshape_and_cache_bf16(c["key"], c["value"], c["slots"], kc, vc)
        out = decode(c["q"], kc, vc, c["tables"], c["lens"], w.scale)
        pool = dict(k_cache=kc, v_cache=vc)
    else:
        cdt = np.int8 if kv == "int8" else np.uint8
        kc, vc = np.zeros(shape, cdt), np.zeros(shape, cdt)
        ks, vs = np.zeros(shape[:3], np.float32), np.zeros(shape[:3], np.float32)
        write = o.reshape_and_cache_int8 if kv == "int8" else o.reshape_and_cache_fp8
        write(c["key"], c["value"], c["slots"], kc, vc, ks, vs)
        out = decode(c["q"], kc, vc, c["tables"], c["lens"], w.scale, ks, vs)
        pool = dict(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs)
    return out, pool, c


def gpu_pool_blocks(pool: pkv.PagedKVPool, tables: np.ndarray, lens: np.ndarray):
    """The GPU pool's blocks in the same compacted order as `compact_for_oracle`."""
    ids = []
    for i, t in enumerate(lens):
        n = (int(t) + 15) // 16
        ids.extend(tables[i, :n].tolist())
    idx = torch.tensor(ids, dtype=torch.long, device=pool.k_cache.device)

    def host(t):
        t = t[idx].cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    res = dict(k_cache=host(pool.k_cache), v_cache=host(pool.v_cache))
    if pool.dtype != "bf16":
        res.update(k_scale=host(pool.k_scale), v_scale=host(pool.v_scale))
    return res


def compare(out_gpu: torch.Tensor, ref: np.ndarray, what="", output_rounding=False):
    """Element-wise comparison with the fp64 oracle.

    ``output_rounding`` widens both bounds by the bf16 rounding of the output itself (bf16
    keeps 8 significant bits, so rounding moves x by at most 2^-8 |x|); it is used where
    the outputs are single values of V rather than averages over many tokens.  Such a
    value of magnitude 4 or more is 2^-5 apart from its bf16 neighbours, so even the
    correctly rounded output can miss the exact one by more than the 1e-2 bound.  It is
    either a bool (every element) or a boolean array broadcastable to ``ref`` that marks
    the elements which get the slack; the mean bound then grows by the slack of the marked
    elements only, averaged over all elements."""
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mask = np.broadcast_to(np.asarray(output_rounding, dtype=bool), ref.shape)
    slack = np.where(mask, 2.0 ** -8 * np.abs(ref), 0.0)
    mean_bound = MEAN_ABS + slack.mean()
    assert np.all(err <= MAX_ABS + slack), f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= mean_bound, f"{what}: mean abs err {err.mean():.3e} > {mean_bound:.3e}"
    return float(err.max()), float(err.mean())


def few_token_queries(lens, num_queries: int, window: int = 0, fewer_than: int = 16) -> np.ndarray:
    """Boolean [B, k]: query i of sequence b attends to fewer than ``fewer_than`` tokens
    (its causal prefix T_b - (k - 1 - i), cut to the window)."""
    lens = np.asarray(lens, dtype=np.int64)
    seen = lens[:, None] - (num_queries - 1 - np.arange(num_queries))[None, :]
    if window:
        seen = np.minimum(seen, window)
    return seen < fewer_than


def valid_slot_bytes_equal(pool_gpu: dict, pool_ref: dict, lens: np.ndarray):
    """Bit-exact comparison of the written slots (token t < T_b of each sequence)."""
    blk = 0
    for t_len in lens:
        n = (int(t_len) + 15) // 16
        for j in range(n):
            valid = min(16, int(t_len) - 16 * j)
            for key in pool_ref:
                g = pool_gpu[key][blk]
                r = pool_ref[key][blk]
                if key.endswith("scale"):
                    assert np.array_equal(g[:, :valid].view(np.uint32), r[:, :valid].view(np.uint32)), key
                else:
                    assert np.array_equal(g[:, :valid], r[:, :valid]), key
            blk += 1
