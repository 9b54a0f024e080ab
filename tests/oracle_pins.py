"""Pins for the CPU oracle: checks against facts the pages and mathematics fix, not
against the oracle itself.

Every pin takes an ``oracle.Oracle`` so that the mutation tests can run the same pins
against deliberately broken copies of the oracle and show that each planted mistake is
caught.  A pin fails by raising (AssertionError or OracleError).

Sources (page title, section):
  * "Lesson 4: Model deployment and inference acceleration", 4.2 -- attention formula and
    the statement that PagedAttention changes only the layout, 16-token blocks, page table.
  * "Lesson 4", 5.3 -- INT8 symmetric KV quantisation, s = max|K| / 127.
  * "LLM Engineer's Handbook -- inference optimisation", quantisation introduction --
    the absmax worked example (fixture tests/golden/absmax_worked_example.json).
  * "LLM/MLLM inference optimisation", 2.2 -- KV size closed form (fixture
    tests/golden/kv_cache_sizes.json); 2.3 -- MQA/GQA head sharing.
  * "Lesson 4", 5.2 "Speculative Decoding" -- the target model verifies k draft tokens in
    one pass: k queries per sequence, each causal over the prefix up to itself.
  * "LLM/MLLM inference optimisation", 2.3 (KV-cache table) -- a sliding window keeps only
    the most recent tokens: each query attends to its last W tokens.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle as oracle_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BS = 16


# ----------------------------------------------------------------- helpers

def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def rand_bf16(gen, *shape, scale=1.0):
    return (torch.randn(*shape, generator=gen, dtype=torch.float32) * scale).to(torch.bfloat16)


def paged_case(o, lens, hq, hkv, d, gen, *, num_blocks=None, perm=None, kv="bf16",
               k=None, v=None, q=None, fill_nan=True, table_width=None):
    """Lay the tokens of each sequence into a pool through a page table.

    Returns (q_bits, pool dict, tables, lens, dense K/V lists).  Unused pool slots are
    filled with NaN so that reading one shows up in the output.
    """
    lens = [int(x) for x in lens]
    nblk = [(t + BS - 1) // BS for t in lens]
    need = sum(nblk)
    if num_blocks is None:
        num_blocks = need + 3
    if perm is None:
        perm = torch.randperm(num_blocks, generator=gen)
    width = max(nblk) if table_width is None else table_width
    tables = np.full((len(lens), width), -1, np.int32)
    c = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[c:c + n].numpy()
        c += n
    if q is None:
        q = rand_bf16(gen, len(lens), hq, d)
    if k is None:
        k = [rand_bf16(gen, t, hkv, d) for t in lens]
    if v is None:
        v = [rand_bf16(gen, t, hkv, d) for t in lens]
    key = torch.cat(k, 0)
    value = torch.cat(v, 0)
    slots = []
    for b, t in enumerate(lens):
        for i in range(t):
            slots.append(tables[b, i // BS] * BS + i % BS)
    slots = np.array(slots, np.int32)
    pool = {}
    if kv == "bf16":
        nan = np.uint16(0x7FC0)
        kc = np.full((num_blocks, hkv, BS, d), nan if fill_nan else 0, np.uint16)
        vc = kc.copy()
        o.reshape_and_cache_bf16(bits(key), bits(value), slots, kc, vc)
        pool.update(k_cache=kc, v_cache=vc)
    else:
        cdt = np.int8 if kv == "int8" else np.uint8
        kc = np.zeros((num_blocks, hkv, BS, d), cdt)
        vc = kc.copy()
        ks = np.full((num_blocks, hkv, BS), np.nan if fill_nan else 0, np.float32)
        vs = ks.copy()
        write = o.reshape_and_cache_int8 if kv == "int8" else o.reshape_and_cache_fp8
        write(bits(key), bits(value), slots, kc, vc, ks, vs)
        pool.update(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs)
    return bits(q), pool, tables, np.array(lens, np.int32), k, v


def decode(o, qb, pool, tables, lens, scale):
    return o.paged_decode(qb, pool["k_cache"], pool["v_cache"], tables, lens, scale,
                          pool.get("k_scale"), pool.get("v_scale"))


def sdpa_fp64(q, k, v, scale):
    """torch's scaled_dot_product_attention in fp64 for one sequence.
    q [H, d]; k, v [T, H, d] (K/V already one per query head)."""
    qq = q.to(torch.float64)[:, None, :]                 # [H, 1, d]
    kk = k.to(torch.float64).permute(1, 0, 2)            # [H, T, d]
    vv = v.to(torch.float64).permute(1, 0, 2)
    out = torch.nn.functional.scaled_dot_product_attention(qq[None], kk[None], vv[None], scale=scale)
    return out[0, :, 0, :].numpy()


# ------------------------------------------------------------------- pins

def pin_permutation_invariance(o):
    """PagedAttention changes only the layout ("Lesson 4", 4.2): two different shuffles of
    the pool and an identity (contiguous) layout give bit-identical fp64 results."""
    gen = torch.Generator().manual_seed(11)
    lens, hq, hkv, d = [1, 15, 16, 17, 33, 70], 4, 2, 32
    q = rand_bf16(gen, len(lens), hq, d)
    k = [rand_bf16(gen, t, hkv, d) for t in lens]
    v = [rand_bf16(gen, t, hkv, d) for t in lens]
    outs = []
    for p in (torch.randperm(40, generator=gen), torch.randperm(40, generator=gen), torch.arange(40)):
        qb, pool, tab, ln, _, _ = paged_case(o, lens, hq, hkv, d, gen, num_blocks=40, perm=p, q=q, k=k, v=v)
        outs.append(decode(o, qb, pool, tab, ln, 0.25))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_library_sdpa(o):
    """Paged attention equals torch's fp64 scaled_dot_product_attention over the same
    tokens laid out contiguously (MHA and GQA with K/V heads repeated per group)."""
    gen = torch.Generator().manual_seed(12)
    for lens, hq, hkv, d in (([5, 16, 31, 50], 6, 6, 64), ([3, 17, 48], 8, 2, 128), ([20, 9], 3, 1, 16)):
        qb, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen)
        scale = 1.0 / math.sqrt(d)
        out = decode(o, qb, pool, tab, ln, scale)
        q = from_bits(qb)
        g = hq // hkv
        for b in range(len(lens)):
            ref = sdpa_fp64(q[b], k[b].repeat_interleave(g, dim=1), v[b].repeat_interleave(g, dim=1), scale)
            np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def pin_bruteforce_softmax(o):
    """exp(l_i) / sum_j exp(l_j) written as plain Python loops, no max shift, T <= 40."""
    gen = torch.Generator().manual_seed(13)
    lens, hq, hkv, d = [1, 2, 7, 16, 17, 40], 2, 1, 8
    qb, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen)
    scale = 0.3
    out = decode(o, qb, pool, tab, ln, scale)
    q = from_bits(qb).double().tolist()
    for b, t_len in enumerate(lens):
        kb, vb = k[b].double().tolist(), v[b].double().tolist()
        for h in range(hq):
            kvh = h // (hq // hkv)
            logits = [scale * sum(q[b][h][c] * kb[t][kvh][c] for c in range(d)) for t in range(t_len)]
            e = [math.exp(x) for x in logits]
            z = sum(e)
            ref = [sum(e[t] / z * vb[t][kvh][c] for t in range(t_len)) for c in range(d)]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-14)


def pin_single_token_returns_v(o):
    """T = 1: the softmax weight is exactly 1, so the output is that token's V exactly."""
    gen = torch.Generator().manual_seed(14)
    qb, pool, tab, ln, k, v = paged_case(o, [1, 1, 1], 4, 2, 64, gen)
    out = decode(o, qb, pool, tab, ln, 0.125)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(out[b, h], v[b][0, h // 2].double().numpy())


def pin_identical_keys_give_mean_v(o):
    """All keys equal => all logits equal => uniform weights => out = mean of V."""
    gen = torch.Generator().manual_seed(15)
    lens = [3, 16, 37]
    k = [rand_bf16(gen, 1, 2, 32).expand(t, 2, 32).contiguous() for t in lens]
    qb, pool, tab, ln, _, v = paged_case(o, lens, 2, 2, 32, gen, k=k)
    out = decode(o, qb, pool, tab, ln, 0.7)
    for b in range(3):
        np.testing.assert_allclose(out[b], v[b].double().mean(0).numpy(), rtol=1e-13, atol=1e-15)


def pin_zero_scale_gives_mean_v(o):
    """scale = 0 => every logit is 0 => out = mean of V, whatever the keys."""
    gen = torch.Generator().manual_seed(16)
    qb, pool, tab, ln, _, v = paged_case(o, [4, 29], 4, 4, 16, gen)
    out = decode(o, qb, pool, tab, ln, 0.0)
    for b in range(2):
        np.testing.assert_allclose(out[b], v[b].double().mean(0).numpy(), rtol=1e-13, atol=1e-15)


def pin_dominant_key(o):
    """One key aligned with q and a huge scale: the softmax is one-hot on that token, and
    the max-shifted evaluation must not overflow."""
    gen = torch.Generator().manual_seed(17)
    d, t_len, hot = 16, 45, 33
    q = torch.zeros(1, 1, d, dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    kk = torch.zeros(t_len, 1, d)
    kk[:, 0, 0] = torch.linspace(-1.0, 0.5, t_len)
    kk[hot, 0, 0] = 1.0
    k = [kk.to(torch.bfloat16)]
    qb, pool, tab, ln, _, v = paged_case(o, [t_len], 1, 1, d, gen, q=q, k=k)
    out = decode(o, qb, pool, tab, ln, 1.0e4)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], v[0][hot, 0].double().numpy(), rtol=0, atol=1e-12)


def pin_gqa_contiguous_groups(o):
    """GQA ("LLM/MLLM inference optimisation", 2.3): q head h reads kv head h // (Hq/Hkv).
    With V of kv head j set to the constant j, head h's output is exactly h // G."""
    gen = torch.Generator().manual_seed(18)
    hq, hkv, d, lens = 8, 2, 16, [9, 21]
    v = [torch.arange(hkv, dtype=torch.float32)[None, :, None].expand(t, hkv, d).to(torch.bfloat16) for t in lens]
    qb, pool, tab, ln, _, _ = paged_case(o, lens, hq, hkv, d, gen, v=v)
    out = decode(o, qb, pool, tab, ln, 0.5)
    for h in range(hq):
        np.testing.assert_allclose(out[:, h, :], h // (hq // hkv), rtol=0, atol=1e-13)


def pin_tail_and_padding_never_read(o):
    """Slots past T_b in the last block, unused pool blocks (all NaN) and -1 table
    entries past the last block are never read: the result is finite and equal to the
    one from a pool without that garbage."""
    gen = torch.Generator().manual_seed(19)
    lens = [17, 1, 31]
    q = rand_bf16(gen, 3, 2, 16)
    k = [rand_bf16(gen, t, 2, 16) for t in lens]
    v = [rand_bf16(gen, t, 2, 16) for t in lens]
    perm = torch.randperm(12, generator=gen)
    a = paged_case(o, lens, 2, 2, 16, gen, num_blocks=12, perm=perm, q=q, k=k, v=v, fill_nan=True, table_width=6)
    b = paged_case(o, lens, 2, 2, 16, gen, num_blocks=12, perm=perm, q=q, k=k, v=v, fill_nan=False, table_width=6)
    oa = decode(o, *a[:4], 0.25)
    ob = decode(o, *b[:4], 0.25)
    assert np.all(np.isfinite(oa))
    assert np.array_equal(oa, ob)


def pin_reshape_and_cache_layout(o):
    """The bf16 write puts token row r at slot s = slot_mapping[r]: seen through a
    [num_blocks, 16, Hkv, d] view of the [num_blocks, Hkv, 16, d] pool, flattened to
    [num_blocks * 16, Hkv, d], row s equals the token's K (and V).  Negative slots write
    nothing; every other slot keeps its old contents."""
    gen = torch.Generator().manual_seed(20)
    nb, hkv, d, n = 9, 3, 8, 40
    key = rand_bf16(gen, n, hkv, d)
    val = rand_bf16(gen, n, hkv, d)
    slots = torch.randperm(nb * BS, generator=gen)[:n].to(torch.int32).numpy().copy()
    slots[::7] = -1
    kc = np.full((nb, hkv, BS, d), 0x1234, np.uint16)
    vc = kc.copy()
    o.reshape_and_cache_bf16(bits(key), bits(val), slots, kc, vc)
    kview = kc.transpose(0, 2, 1, 3).reshape(nb * BS, hkv, d)
    vview = vc.transpose(0, 2, 1, 3).reshape(nb * BS, hkv, d)
    written = np.zeros(nb * BS, bool)
    for r, s in enumerate(slots):
        if s < 0:
            continue
        written[s] = True
        assert np.array_equal(kview[s], bits(key)[r]) and np.array_equal(vview[s], bits(val)[r])
    assert np.all(kview[~written] == 0x1234) and np.all(vview[~written] == 0x1234)


def pin_absmax_worked_example(o):
    """The pages' worked example: absmax 3.2, x = 0.1 -> 3.97 -> code 4 -> 0.1008,
    error 0.0008 (fixture absmax_worked_example.json)."""
    with open(os.path.join(GOLDEN, "absmax_worked_example.json")) as f:
        g = json.load(f)
    codes, s = o.quantize_row_f32(np.array([g["absmax"], g["x"], -g["absmax"]], np.float32))
    ratio = np.float32(g["x"]) / s
    assert round(float(ratio), 2) == g["ratio_approx"]
    assert int(codes[1]) == g["code"]
    deq = float(np.float32(codes[1]) * s)
    nd = g["printed_decimals"]
    assert round(deq, nd) == g["dequantised_approx"]
    assert round(abs(deq - g["x"]), nd) == g["rounding_error_approx"]
    assert int(codes[0]) == g["range"][1] and int(codes[2]) == -g["range"][1]


def pin_quantiser_roundtrip_bound(o):
    """|x - s * code| <= s / 2, widened by the fp32 rounding of y = x / s, codes in
    [-127, 127], and the element of largest magnitude maps to +-127 ("Lesson 4", 5.3).

    y = fl(x / s) is within 2^-24 |y| <= 2^-24 * 127 < 2^-17 of x / s, so
    |x / s - round(y)| <= 1/2 + 2^-17 and |x - s * code| <= s / 2 * (1 + 2^-16)."""
    gen = torch.Generator().manual_seed(21)
    for rows in (rand_bf16(gen, 500, 128), rand_bf16(gen, 200, 64, scale=1e-3),
                 rand_bf16(gen, 100, 128, scale=300.0)):
        codes, scales = o.quantize_rows(bits(rows))
        xf = rows.float().numpy().astype(np.float64)
        s = scales.astype(np.float64)[:, None]
        assert codes.min() >= -127 and codes.max() <= 127
        err = np.abs(xf - s * codes.astype(np.float64))
        assert np.all(err <= s / 2 * (1 + 2.0 ** -16))
        arg = np.abs(xf).argmax(1)
        picked = codes[np.arange(len(arg)), arg]
        assert np.all(np.abs(picked) == 127)
        np.testing.assert_array_equal(scales, (np.abs(rows.float().numpy()).max(1) / np.float32(127)).astype(np.float32))


def pin_quantiser_matches_torch_fp32(o):
    """Bit-exact against torch's fp32 `round(x / s)` (round half to even) with
    s = amax / 127 computed in fp32, on many random rows: the division form, not a
    multiply by a reciprocal."""
    gen = torch.Generator().manual_seed(22)
    x = rand_bf16(gen, 8192, 128)
    codes, scales = o.quantize_rows(bits(x))
    xf = x.float()
    s = xf.abs().amax(1) / 127.0
    ref = torch.round(xf / s[:, None]).clamp(-127, 127).to(torch.int8)
    assert torch.equal(torch.from_numpy(scales), s)
    assert torch.equal(torch.from_numpy(codes), ref)


def pin_quantiser_ties_half_even(o):
    """Ties go to the even code (the pages round with torch.round): with amax = 127 the
    scale is exactly 1, so x = 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, -0.5 -> 0."""
    codes, s = o.quantize_row_f32(np.array([127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5], np.float32))
    assert s == np.float32(1.0)
    assert codes.tolist() == [127, 2, 4, -2, 0, 0, 2]


def pin_quantiser_zero_row(o):
    """A row of zeros has scale 0 and codes 0, so it dequantises to exact zeros."""
    codes, s = o.quantize_row_f32(np.zeros(64, np.float32))
    assert s == 0.0 and not codes.any()


def pin_int8_cache_and_decode(o):
    """The INT8 write stores, at each slot, the row's own codes and scale; the INT8 decode
    equals fp64 SDPA over the dequantised values s * code."""
    gen = torch.Generator().manual_seed(23)
    lens, hq, hkv, d = [7, 16, 45], 8, 2, 64
    qb, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen, kv="int8")
    kc, vc, ks, vs = pool["k_cache"], pool["v_cache"], pool["k_scale"], pool["v_scale"]
    scale = 1.0 / math.sqrt(d)
    out = decode(o, qb, pool, tab, ln, scale)
    q = from_bits(qb)
    for b, t_len in enumerate(lens):
        kcodes, kscales = o.quantize_rows(bits(k[b]))
        vcodes, vscales = o.quantize_rows(bits(v[b]))
        blocks = tab[b, (np.arange(t_len) // BS)]
        offs = np.arange(t_len) % BS
        for h in range(hkv):
            assert np.array_equal(kc[blocks, h, offs], kcodes[:, h])
            assert np.array_equal(vs[blocks, h, offs], vscales[:, h])
        kd = torch.from_numpy(kcodes.astype(np.float64) * kscales.astype(np.float64)[..., None])
        vd = torch.from_numpy(vcodes.astype(np.float64) * vscales.astype(np.float64)[..., None])
        g = hq // hkv
        ref = sdpa_fp64(q[b], kd.repeat_interleave(g, 1), vd.repeat_interleave(g, 1), scale)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def pin_e4m3_decode_matches_torch(o):
    """Every E4M3 byte decodes to torch's float8_e4m3fn value of the same bits (NaN codes
    S.1111.111 included)."""
    codes = np.arange(256, dtype=np.uint8)
    mine = o.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(ref)], ref[~np.isnan(ref)])


def pin_e4m3_format_values(o):
    """Values the E4M3 definition fixes (bias 7, 3 mantissa bits, no infinities): the
    largest finite 448, 1.0, the smallest normal 2^-6 and subnormal 2^-9, ties to the even
    mantissa, saturation of out-of-range values at +-448."""
    cases = {448.0: 0x7E, 1.0: 0x38, 2.0 ** -6: 0x08, 2.0 ** -9: 0x01, -1.5: 0xBC, 0.0: 0x00,
             1.0625: 0x38, 1.1875: 0x3A, 3.0 * 2.0 ** -10: 0x02, 500.0: 0x7E, -1e6: 0xFE,
             464.0: 0x7E, 2.0 ** -11: 0x00}
    for y, code in cases.items():
        assert int(o.float_to_e4m3(np.float32(y))) == code, (y, hex(code))
    assert o.e4m3_to_float(np.uint8(0x7E)) == 448.0 and np.isnan(o.e4m3_to_float(np.uint8(0x7F)))


def pin_e4m3_encode_matches_torch(o):
    """Nearest E4M3 (ties to even) agrees with torch's float8_e4m3fn cast on in-range
    values spanning the subnormal and normal ranges, and on exact midpoints."""
    gen = torch.Generator().manual_seed(25)
    y = (torch.randn(20000, generator=gen) * torch.exp(torch.randn(20000, generator=gen) * 3)).clamp(-447.9, 447.9)
    grid = torch.from_numpy(np.arange(0, 0x7E, dtype=np.uint8)).view(torch.float8_e4m3fn).float()
    mids = (grid[1:] + grid[:-1]) / 2
    y = torch.cat([y, mids, -mids]).float()
    assert np.array_equal(o.float_to_e4m3(y.numpy()), y.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def pin_fp8_quantiser(o):
    """FP8 rows: s = max|x| / 448, the largest element maps to +-448, and every element is
    within half an E4M3 spacing of s * value(code): 2^-4 relative for normals, s * 2^-10
    absolute below the normal range."""
    gen = torch.Generator().manual_seed(26)
    for rows in (rand_bf16(gen, 300, 128), rand_bf16(gen, 100, 64, scale=1e-3)):
        codes, scales = o.quantize_rows_fp8(bits(rows))
        xf = rows.float().numpy().astype(np.float64)
        s = scales.astype(np.float64)[:, None]
        np.testing.assert_array_equal(scales, (np.abs(rows.float().numpy()).max(1) / np.float32(448)).astype(np.float32))
        deq = s * o.e4m3_to_float(codes)
        bound = np.maximum(np.abs(xf) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -10)
        assert np.all(np.abs(xf - deq) <= bound)
        arg = np.abs(xf).argmax(1)
        assert np.all(np.abs(o.e4m3_to_float(codes[np.arange(len(arg)), arg])) == 448.0)


def pin_fp8_cache_and_decode(o):
    """The FP8 write stores each row's own codes and scale at its slot; the FP8 decode
    equals fp64 SDPA over the dequantised values s * value(code)."""
    gen = torch.Generator().manual_seed(27)
    lens, hq, hkv, d = [9, 16, 40], 8, 2, 64
    qb, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen, kv="fp8")
    scale = 1.0 / math.sqrt(d)
    out = decode(o, qb, pool, tab, ln, scale)
    q = from_bits(qb)
    for b, t_len in enumerate(lens):
        kcodes, kscales = o.quantize_rows_fp8(bits(k[b]))
        vcodes, vscales = o.quantize_rows_fp8(bits(v[b]))
        blocks = tab[b, (np.arange(t_len) // BS)]
        offs = np.arange(t_len) % BS
        for h in range(hkv):
            assert np.array_equal(pool["k_cache"][blocks, h, offs], kcodes[:, h])
            assert np.array_equal(pool["v_scale"][blocks, h, offs], vscales[:, h])
        kd = torch.from_numpy(o.e4m3_to_float(kcodes) * kscales.astype(np.float64)[..., None])
        vd = torch.from_numpy(o.e4m3_to_float(vcodes) * vscales.astype(np.float64)[..., None])
        g = hq // hkv
        ref = sdpa_fp64(q[b], kd.repeat_interleave(g, 1), vd.repeat_interleave(g, 1), scale)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def sdpa_causal_fp64(q, k, v, scale):
    """torch's fp64 scaled_dot_product_attention for the last n positions of a sequence:
    q [n, H, d]; k, v [T, H, d]; query i (position T - n + i) may attend to t <= T - n + i,
    given to torch as an explicit boolean mask."""
    n, t_len = q.shape[0], k.shape[0]
    allowed = torch.arange(t_len)[None, :] <= (t_len - n + torch.arange(n))[:, None]
    qq = q.to(torch.float64).permute(1, 0, 2)[None]      # [1, H, n, d]
    kk = k.to(torch.float64).permute(1, 0, 2)[None]      # [1, H, T, d]
    vv = v.to(torch.float64).permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=allowed, scale=scale)
    return out[0].permute(1, 0, 2).numpy()                # [n, H, d]


def pin_multi_query_causal_sdpa(o):
    """Verifying k draft tokens in one pass ("Lesson 4", 5.2): each of the k queries of a
    sequence equals torch's fp64 SDPA under the causal mask over the sequence's last k
    positions, for bf16, INT8 (over s * code) and MHA/GQA."""
    gen = torch.Generator().manual_seed(31)
    for lens, nq, hq, hkv, d, kv in (([4, 17, 33, 48], 4, 4, 2, 32, "bf16"), ([5, 16], 5, 3, 3, 16, "bf16"),
                                     ([40], 1, 2, 1, 8, "bf16"), ([8, 19, 36], 3, 8, 2, 64, "int8")):
        _, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen, kv=kv)
        q = rand_bf16(gen, len(lens), nq, hq, d)
        scale = 1.0 / math.sqrt(d)
        out = o.paged_decode_multi(bits(q), pool["k_cache"], pool["v_cache"], tab, ln, scale,
                                   pool.get("k_scale"), pool.get("v_scale"))
        g = hq // hkv
        for b in range(len(lens)):
            kb, vb = k[b].double(), v[b].double()
            if kv == "int8":
                kcodes, kscales = o.quantize_rows(bits(k[b]))
                vcodes, vscales = o.quantize_rows(bits(v[b]))
                kb = torch.from_numpy(kcodes.astype(np.float64) * kscales.astype(np.float64)[..., None])
                vb = torch.from_numpy(vcodes.astype(np.float64) * vscales.astype(np.float64)[..., None])
            ref = sdpa_causal_fp64(q[b], kb.repeat_interleave(g, 1), vb.repeat_interleave(g, 1), scale)
            np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def pin_multi_query_first_draft(o):
    """With T == k the first query sees only token 0 (its output is v_0 exactly, in every
    head of the group) and the second sees tokens 0 and 1: a two-term softmax written out."""
    gen = torch.Generator().manual_seed(32)
    nq, hq, hkv, d = 3, 4, 2, 16
    _, pool, tab, ln, k, v = paged_case(o, [nq], hq, hkv, d, gen)
    q = rand_bf16(gen, 1, nq, hq, d)
    out = o.paged_decode_multi(bits(q), pool["k_cache"], pool["v_cache"], tab, ln, 0.5)
    kk, vv, qq = k[0].double(), v[0].double(), q[0].double()
    for h in range(hq):
        kvh = h // (hq // hkv)
        assert np.array_equal(out[0, 0, h], vv[0, kvh].numpy())
        l0 = 0.5 * float(qq[1, h] @ kk[0, kvh])
        l1 = 0.5 * float(qq[1, h] @ kk[1, kvh])
        w1 = 1.0 / (1.0 + math.exp(l0 - l1))
        np.testing.assert_allclose(out[0, 1, h], (1 - w1) * vv[0, kvh].numpy() + w1 * vv[1, kvh].numpy(),
                                   rtol=1e-12, atol=1e-14)
    try:
        o.paged_decode_multi(bits(rand_bf16(gen, 1, nq + 1, hq, d)), pool["k_cache"], pool["v_cache"],
                             tab, ln, 0.5)
    except oracle_mod.OracleError:
        return
    raise AssertionError("more queries than cached tokens accepted")


def sdpa_band_fp64(q, k, v, scale, window):
    """torch fp64 SDPA for the last n positions of a sequence under an explicit boolean
    band mask: query i at position p_i = T - n + i may attend to p_i - W < t <= p_i."""
    n, t_len = q.shape[0], k.shape[0]
    pos = (t_len - n + torch.arange(n))[:, None]
    t = torch.arange(t_len)[None, :]
    allowed = (t <= pos) & (t > pos - window)
    qq = q.to(torch.float64).permute(1, 0, 2)[None]
    kk = k.to(torch.float64).permute(1, 0, 2)[None]
    vv = v.to(torch.float64).permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=allowed, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


def pin_sliding_window_band_sdpa(o):
    """A sliding window of W tokens ("LLM/MLLM inference optimisation", 2.3) equals torch's
    fp64 SDPA under a band mask, for one and several queries per sequence, windows inside a
    block, on block boundaries and longer than the context, bf16 and INT8."""
    gen = torch.Generator().manual_seed(33)
    cases = (([1, 16, 17, 40, 70], 1, 4, 2, 32, 5, "bf16"), ([3, 20, 48, 90], 3, 4, 4, 16, 16, "bf16"),
             ([5, 33, 64], 4, 8, 2, 64, 17, "int8"), ([9, 30], 2, 2, 1, 8, 1, "bf16"),
             ([12, 50], 3, 3, 3, 16, 200, "bf16"))
    for lens, nq, hq, hkv, d, win, kv in cases:
        _, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen, kv=kv)
        q = rand_bf16(gen, len(lens), nq, hq, d)
        scale = 1.0 / math.sqrt(d)
        out = o.paged_decode_multi(bits(q), pool["k_cache"], pool["v_cache"], tab, ln, scale,
                                   pool.get("k_scale"), pool.get("v_scale"), window=win)
        g = hq // hkv
        for b in range(len(lens)):
            kb, vb = k[b].double(), v[b].double()
            if kv == "int8":
                kcodes, kscales = o.quantize_rows(bits(k[b]))
                vcodes, vscales = o.quantize_rows(bits(v[b]))
                kb = torch.from_numpy(kcodes.astype(np.float64) * kscales.astype(np.float64)[..., None])
                vb = torch.from_numpy(vcodes.astype(np.float64) * vscales.astype(np.float64)[..., None])
            ref = sdpa_band_fp64(q[b], kb.repeat_interleave(g, 1), vb.repeat_interleave(g, 1), scale, win)
            np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def pin_sliding_window_special_cases(o):
    """W = 1: each query returns its own token's V exactly.  W >= T: the full result, bit
    for bit.  Blocks wholly before the window may be released: their table entries (-1) and
    contents (NaN) are never read."""
    gen = torch.Generator().manual_seed(34)
    lens, nq, hq, hkv, d = [3, 18, 35, 64], 3, 4, 2, 16
    _, pool, tab, ln, k, v = paged_case(o, lens, hq, hkv, d, gen)
    q = rand_bf16(gen, len(lens), nq, hq, d)
    run = lambda t, w: o.paged_decode_multi(bits(q), pool["k_cache"], pool["v_cache"], t, ln, 0.25, window=w)
    one = run(tab, 1)
    for b, t_len in enumerate(lens):
        for i in range(nq):
            own = v[b][t_len - nq + i].double().numpy()  # [Hkv, d]
            assert np.array_equal(one[b, i], own.repeat(hq // hkv, axis=0))
    assert np.array_equal(run(tab, 64), run(tab, 0))
    win = 20
    full = run(tab, win)
    released = tab.copy()
    kc = pool["k_cache"].copy()
    for b, t_len in enumerate(lens):
        first = max(0, t_len - (nq - 1) - win) // BS  # first block any query sees
        for j in range(first):
            kc[released[b, j]] = np.uint16(0x7FC0)
            released[b, j] = -1
    out = o.paged_decode_multi(bits(q), kc, pool["v_cache"], released, ln, 0.25, window=win)
    assert np.array_equal(out, full)


def pin_kv_cache_size_closed_forms(o):
    """The size model reproduces the pages' printed figures (kv_cache_sizes.json)."""
    with open(os.path.join(GOLDEN, "kv_cache_sizes.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        n = oracle_mod.kv_cache_bytes(c["layers"], c["n_kv"], c["head_dim"], c["seq_len"], c["elem_bytes"])
        if "bytes" in c:
            assert n == c["bytes"], c
        else:
            assert n >= c["bytes_at_least"], c


def pin_rejects_bad_tables(o):
    """Out-of-range block ids, context lengths < 1 or beyond the table, and slots past
    the pool are errors, not reads."""
    gen = torch.Generator().manual_seed(24)
    qb, pool, tab, ln, _, _ = paged_case(o, [20], 2, 2, 8, gen, num_blocks=4)
    bad = tab.copy()
    bad[0, 1] = 4
    for t, l in ((bad, ln), (tab, np.array([0], np.int32)), (tab, np.array([33], np.int32))):
        try:
            decode(o, qb, pool, t, l, 1.0)
        except oracle_mod.OracleError:
            continue
        raise AssertionError("bad input accepted")
    kc = np.zeros((4, 2, BS, 8), np.uint16)
    try:
        o.reshape_and_cache_bf16(np.zeros((1, 2, 8), np.uint16), np.zeros((1, 2, 8), np.uint16),
                                 np.array([64], np.int32), kc, kc.copy())
    except oracle_mod.OracleError:
        return
    raise AssertionError("slot past the pool accepted")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
