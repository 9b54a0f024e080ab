"""fp64 CPU oracle for PagedAttention decode and the KV-cache write.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline and reference legs may import this package.  The CUDA
library never loads it, and this package never loads the CUDA library: the two meet only
through the seeded inputs that both are handed.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over (sequence, query head));
this module compiles it with gcc and wraps it for numpy arrays.  bf16 tensors are passed
as ``numpy.uint16`` arrays of their bit patterns.

What each function follows (page title, section):

* ``paged_decode`` -- ``out = softmax(q K^T * scale) V`` walked through the page table in
  logical order; "Lesson 4: Model deployment and inference acceleration", section 4.2
  (PagedAttention changes only the memory layout, not the formula).  GQA groups are
  contiguous ("LLM/MLLM inference optimisation", section 2.3).
* ``reshape_and_cache_bf16`` -- write each new token's K/V row into slot
  ``slot_mapping[t]`` (block ``slot // 16``, offset ``slot % 16``); "Lesson 4", 4.2.
* ``quantize_rows`` / ``reshape_and_cache_int8`` -- INT8 symmetric quantisation
  ``round(x / s)``, ``s = max|x| / 127``, one scale per (token, kv head) row, fp32
  arithmetic, round half to even, codes in [-127, 127]; "Lesson 4", section 5.3.
* ``e4m3_to_float`` / ``float_to_e4m3`` / ``quantize_rows_fp8`` / ``reshape_and_cache_fp8``
  -- the FP8 (E4M3) KV cache read as the INT8 scheme with E4M3 codes: ``s = max|x| / 448``,
  code = nearest E4M3 of ``x / s`` (ties to even, saturating); "Lesson 4", section 5.3
  names FP8 KV caches without a scaling rule.
* ``paged_decode_multi`` -- k query tokens per sequence for speculative verification (the
  target model checks k drafts in one pass; "Lesson 4", 5.2): the drafts are the last k
  cached tokens, query i attends causally to tokens ``0 .. T - k + i``.
* ``paged_decode_multi(..., window=W)`` -- a sliding window ("LLM/MLLM inference
  optimisation", 2.3: keep only the most recent window of the cache): each query attends to
  its last W tokens.
* ``kv_cache_bytes`` -- the KV-cache size closed form
  ``2 * layers * n_kv * head_dim * seq_len * bytes``; "LLM/MLLM inference
  optimisation", section 2.2.
"""

from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from pathlib import Path

import numpy as np

BLOCK_SIZE = 16
KV_BF16 = 0
KV_INT8 = 1
KV_FP8 = 2

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "oracle.c"

_ERRORS = {
    -1: "invalid argument",
    -2: "context length < 1 or beyond the block table",
    -3: "block-table entry out of range",
    -4: "slot_mapping entry out of range",
    -5: "out of memory",
}


class OracleError(RuntimeError):
    pass


def default_library_path() -> Path:
    return _HERE / "_build" / platform.machine() / "liboracle.so"


def build(source: Path | str = SOURCE, out: Path | str | None = None, force: bool = False) -> Path:
    """Compile ``oracle.c`` (or a given copy of it) into a shared library with gcc.

    IEEE semantics matter for the INT8 quantiser, so no fast-math and no FMA
    contraction.
    """
    source = Path(source)
    out = Path(out) if out is not None else default_library_path()
    if not force and out.exists() and out.stat().st_mtime >= source.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = [
        "gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
        "-fno-fast-math", "-ffp-contract=off", "-Wall",
        str(source), "-o", str(tmp), "-lm",
    ]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(f"oracle error {rc}: {_ERRORS.get(rc, 'unknown')}")


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


class Oracle:
    """A loaded copy of the oracle library (a patched copy can be loaded too)."""

    def __init__(self, lib_path: Path | str | None = None):
        if lib_path is None:
            lib_path = build()
        self.path = Path(lib_path)
        lib = ctypes.CDLL(str(self.path))
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_max_threads.restype = i32
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_float.restype = ctypes.c_float
        lib.oracle_reshape_and_cache_bf16.argtypes = [vp, vp, vp, i64, i32, i32, i64, vp, vp]
        lib.oracle_reshape_and_cache_bf16.restype = i32
        lib.oracle_quantize_row_f32.argtypes = [vp, i32, vp, vp]
        lib.oracle_quantize_rows_bf16.argtypes = [vp, i64, i32, vp, vp]
        lib.oracle_quantize_rows_bf16.restype = i32
        lib.oracle_reshape_and_cache_int8.argtypes = [vp, vp, vp, i64, i32, i32, i64, vp, vp, vp, vp]
        lib.oracle_reshape_and_cache_int8.restype = i32
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_float_to_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_float_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_quantize_row_fp8_f32.argtypes = [vp, i32, vp, vp]
        lib.oracle_quantize_rows_fp8_bf16.argtypes = [vp, i64, i32, vp, vp]
        lib.oracle_quantize_rows_fp8_bf16.restype = i32
        lib.oracle_reshape_and_cache_fp8.argtypes = [vp, vp, vp, i64, i32, i32, i64, vp, vp, vp, vp]
        lib.oracle_reshape_and_cache_fp8.restype = i32
        lib.oracle_paged_decode.argtypes = [
            vp, vp, vp, vp, vp, i32, i64, i32, i32, vp, i32, vp, i32, i32, ctypes.c_double, vp]
        lib.oracle_paged_decode.restype = i32
        lib.oracle_paged_decode_multi.argtypes = [
            vp, vp, vp, vp, vp, i32, i64, i32, i32, vp, i32, vp, i32, i32, i32, ctypes.c_double, vp]
        lib.oracle_paged_decode_multi.restype = i32
        lib.oracle_paged_decode_window.argtypes = [
            vp, vp, vp, vp, vp, i32, i64, i32, i32, vp, i32, vp, i32, i32, i32, i32, ctypes.c_double, vp]
        lib.oracle_paged_decode_window.restype = i32
        self.lib = lib

    # -- threads
    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def set_threads(self, n: int) -> None:
        self.lib.oracle_set_threads(int(n))

    # -- conversions
    def bf16_to_float(self, bits: int) -> float:
        return float(self.lib.oracle_bf16_to_float(int(bits)))

    # -- cache write
    def reshape_and_cache_bf16(self, key, value, slot_mapping, k_cache, v_cache) -> None:
        """In place: k_cache/v_cache uint16 [num_blocks, Hkv, 16, d]; key/value uint16 [N, Hkv, d]."""
        key, value = _c(key, np.uint16), _c(value, np.uint16)
        slots = _c(slot_mapping, np.int32)
        assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
        assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
        n, hkv, d = key.shape
        _check(self.lib.oracle_reshape_and_cache_bf16(
            _ptr(key), _ptr(value), _ptr(slots), n, hkv, d, k_cache.shape[0],
            _ptr(k_cache), _ptr(v_cache)))

    def quantize_row_f32(self, x) -> tuple[np.ndarray, np.float32]:
        x = _c(x, np.float32)
        codes = np.zeros(x.shape[0], np.int8)
        scale = np.zeros(1, np.float32)
        self.lib.oracle_quantize_row_f32(_ptr(x), x.shape[0], _ptr(codes), _ptr(scale))
        return codes, scale[0]

    def quantize_rows(self, x_bf16_bits) -> tuple[np.ndarray, np.ndarray]:
        """Quantise rows of bf16 bits [..., d] -> (int8 codes [..., d], fp32 scales [...])."""
        x = _c(x_bf16_bits, np.uint16)
        d = x.shape[-1]
        rows = x.size // d
        codes = np.zeros(x.shape, np.int8)
        scales = np.zeros(x.shape[:-1], np.float32)
        _check(self.lib.oracle_quantize_rows_bf16(_ptr(x), rows, d, _ptr(codes), _ptr(scales)))
        return codes, scales

    def reshape_and_cache_int8(self, key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> None:
        key, value = _c(key, np.uint16), _c(value, np.uint16)
        slots = _c(slot_mapping, np.int32)
        for a, dt in ((k_cache, np.int8), (v_cache, np.int8), (k_scale, np.float32), (v_scale, np.float32)):
            assert a.dtype == dt and a.flags.c_contiguous
        n, hkv, d = key.shape
        _check(self.lib.oracle_reshape_and_cache_int8(
            _ptr(key), _ptr(value), _ptr(slots), n, hkv, d, k_cache.shape[0],
            _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale)))

    # -- FP8 (E4M3)
    def e4m3_to_float(self, codes) -> np.ndarray:
        codes = np.asarray(codes, np.uint8)
        return np.array([self.lib.oracle_e4m3_to_double(int(c)) for c in codes.ravel()]).reshape(codes.shape)

    def float_to_e4m3(self, y) -> np.ndarray:
        y = np.asarray(y, np.float32)
        return np.array([self.lib.oracle_float_to_e4m3(float(v)) for v in y.ravel()], np.uint8).reshape(y.shape)

    def quantize_row_fp8_f32(self, x) -> tuple[np.ndarray, np.float32]:
        x = _c(x, np.float32)
        codes = np.zeros(x.shape[0], np.uint8)
        scale = np.zeros(1, np.float32)
        self.lib.oracle_quantize_row_fp8_f32(_ptr(x), x.shape[0], _ptr(codes), _ptr(scale))
        return codes, scale[0]

    def quantize_rows_fp8(self, x_bf16_bits) -> tuple[np.ndarray, np.ndarray]:
        x = _c(x_bf16_bits, np.uint16)
        d = x.shape[-1]
        codes = np.zeros(x.shape, np.uint8)
        scales = np.zeros(x.shape[:-1], np.float32)
        _check(self.lib.oracle_quantize_rows_fp8_bf16(_ptr(x), x.size // d, d, _ptr(codes), _ptr(scales)))
        return codes, scales

    def reshape_and_cache_fp8(self, key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> None:
        key, value = _c(key, np.uint16), _c(value, np.uint16)
        slots = _c(slot_mapping, np.int32)
        for a, dt in ((k_cache, np.uint8), (v_cache, np.uint8), (k_scale, np.float32), (v_scale, np.float32)):
            assert a.dtype == dt and a.flags.c_contiguous
        n, hkv, d = key.shape
        _check(self.lib.oracle_reshape_and_cache_fp8(
            _ptr(key), _ptr(value), _ptr(slots), n, hkv, d, k_cache.shape[0],
            _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale)))

    # -- decode
    def paged_decode(self, q, k_cache, v_cache, block_tables, context_lens, scale,
                     k_scale=None, v_scale=None) -> np.ndarray:
        """fp64 [B, Hq, d] attention output.

        q: uint16 bf16 bits [B, Hq, d]; k_cache/v_cache: uint16 (bf16), int8 (INT8) or uint8
        (FP8 E4M3 codes) [num_blocks, Hkv, 16, d]; k_scale/v_scale: fp32 [num_blocks, Hkv, 16]
        for INT8 and FP8.
        """
        q = _c(q, np.uint16)
        kdt = k_cache.dtype
        kv_dtype = {np.dtype(np.int8): KV_INT8, np.dtype(np.uint8): KV_FP8}.get(np.dtype(kdt), KV_BF16)
        if kv_dtype == KV_BF16:
            kdt = np.uint16
        k_cache, v_cache = _c(k_cache, kdt), _c(v_cache, kdt)
        if kv_dtype != KV_BF16:
            k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        b, hq, d = q.shape
        nb, hkv, bs, d2 = k_cache.shape
        assert bs == BLOCK_SIZE and d2 == d and bt.shape[0] == b and cl.shape[0] == b
        out = np.zeros((b, hq, d), np.float64)
        _check(self.lib.oracle_paged_decode(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype,
            nb, hkv, d, _ptr(bt), bt.shape[1], _ptr(cl), b, hq, float(scale), _ptr(out)))
        return out


    def paged_decode_multi(self, q, k_cache, v_cache, block_tables, context_lens, scale,
                           k_scale=None, v_scale=None, window: int = 0) -> np.ndarray:
        """fp64 [B, k, Hq, d]: q bf16 bits [B, k, Hq, d]; the k queries of sequence b are its
        last k cached tokens, query i attending causally to tokens 0 .. T_b - k + i (with
        ``window`` W > 0, only to its last W: T_b - k + i - W + 1 .. T_b - k + i)."""
        q = _c(q, np.uint16)
        kdt = k_cache.dtype
        kv_dtype = {np.dtype(np.int8): KV_INT8, np.dtype(np.uint8): KV_FP8}.get(np.dtype(kdt), KV_BF16)
        if kv_dtype == KV_BF16:
            kdt = np.uint16
        k_cache, v_cache = _c(k_cache, kdt), _c(v_cache, kdt)
        if kv_dtype != KV_BF16:
            k_scale, v_scale = _c(k_scale, np.float32), _c(v_scale, np.float32)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        b, nq, hq, d = q.shape
        nb, hkv, bs, d2 = k_cache.shape
        assert bs == BLOCK_SIZE and d2 == d and bt.shape[0] == b and cl.shape[0] == b
        out = np.zeros((b, nq, hq, d), np.float64)
        _check(self.lib.oracle_paged_decode_window(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype,
            nb, hkv, d, _ptr(bt), bt.shape[1], _ptr(cl), b, nq, int(window), hq, float(scale), _ptr(out)))
        return out


_DEFAULT: Oracle | None = None


def load() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def kv_cache_bytes(layers: int, n_kv: int, head_dim: int, seq_len: int, elem_bytes: int) -> int:
    """KV-cache size: 2 (K and V) x layers x n_kv x head_dim x seq_len x bytes per element."""
    return 2 * layers * n_kv * head_dim * seq_len * elem_bytes
