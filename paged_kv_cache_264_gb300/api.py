"""Thin Python binding of the C ABI (``include/pagedkv.h``).

Argument marshalling only: the functions check torch dtypes, devices and contiguity and
pass ``data_ptr()``s and the current CUDA stream to the library; every step of the
computation runs in the library's kernels.  Names follow the C calls without the
``pkv_`` prefix.  ``PagedKVPool`` bundles a pool's tensors with its descriptor.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import BLOCK_SIZE, DecodeOptions, PKV_KV_BF16, PKV_KV_FP8_E4M3, PKV_KV_INT8, check

_DTYPES = {"bf16": PKV_KV_BF16, "int8": PKV_KV_INT8, "fp8": PKV_KV_FP8_E4M3}
_CODE_DTYPES = {"bf16": torch.bfloat16, "int8": torch.int8, "fp8": torch.uint8}


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str, ndim: int | None = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


_KERNELS = {0: 0, "auto": 0, 1: 1, "cuda_core": 1, 2: 2, "tensor_core": 2}
_SCHEDULES = {0: 0, "auto": 0, 1: 1, "grid": 1, 2: 2, "persistent": 2}


def _options(partition_blocks: int = 0, kernel=0, schedule=0, stages=0,
             blocks_per_stage=0, num_queries=1, window=0) -> ctypes.POINTER(DecodeOptions) | None:
    if not (partition_blocks or _KERNELS[kernel] or _SCHEDULES[schedule] or stages or blocks_per_stage
            or num_queries != 1 or window):
        return None
    o = DecodeOptions()
    o.partition_blocks = int(partition_blocks)
    o.kernel = _KERNELS[kernel]
    o.schedule = _SCHEDULES[schedule]
    o.stages = int(stages)
    o.blocks_per_stage = int(blocks_per_stage)
    o.num_queries = int(num_queries)
    o.window = int(window)
    return ctypes.pointer(o)


def version() -> str:
    return _lib.load().pkv_version().decode()


def launch_count() -> int:
    return int(_lib.load().pkv_launch_count())


def pool_bytes(num_blocks: int, kv_heads: int, head_dim: int, dtype: str = "bf16") -> tuple[int, int]:
    kv, sc = ctypes.c_size_t(), ctypes.c_size_t()
    check(_lib.load().pkv_pool_bytes(num_blocks, kv_heads, head_dim, _DTYPES[dtype],
                                     ctypes.byref(kv), ctypes.byref(sc)), "pool_bytes")
    return kv.value, sc.value


def pool_create(num_blocks: int, kv_heads: int, head_dim: int, dtype: str, k_cache: torch.Tensor,
                v_cache: torch.Tensor, k_scale: torch.Tensor | None = None,
                v_scale: torch.Tensor | None = None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    check(_lib.load().pkv_pool_create(num_blocks, kv_heads, head_dim, BLOCK_SIZE, _DTYPES[dtype],
                                      _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                      ctypes.byref(h)), "pool_create")
    return h


def pool_destroy(handle) -> None:
    check(_lib.load().pkv_pool_destroy(handle), "pool_destroy")


class PagedKVPool:
    """A block pool ([num_blocks, kv_heads, 16, head_dim] K and V, plus fp32 scales for
    INT8 and FP8) allocated with torch on the current CUDA device, and its library
    descriptor.  FP8 codes are held as uint8 (E4M3 bit patterns)."""

    def __init__(self, num_blocks: int, kv_heads: int, head_dim: int, dtype: str = "bf16",
                 device=None, fill=None):
        if dtype not in _DTYPES:
            raise ValueError(f"dtype must be one of {list(_DTYPES)}")
        device = torch.device(device or "cuda")
        self.num_blocks, self.kv_heads, self.head_dim, self.dtype = num_blocks, kv_heads, head_dim, dtype
        shape = (num_blocks, kv_heads, BLOCK_SIZE, head_dim)
        tdt = _CODE_DTYPES[dtype]
        self.k_cache = torch.empty(shape, dtype=tdt, device=device)
        self.v_cache = torch.empty(shape, dtype=tdt, device=device)
        self.k_scale = self.v_scale = None
        if dtype != "bf16":
            self.k_scale = torch.empty(shape[:3], dtype=torch.float32, device=device)
            self.v_scale = torch.empty(shape[:3], dtype=torch.float32, device=device)
        if fill is not None:
            for t in (self.k_cache, self.v_cache, self.k_scale, self.v_scale):
                if t is not None:
                    t.fill_(fill)
        with torch.cuda.device(device):
            self.handle = pool_create(num_blocks, kv_heads, head_dim, dtype, self.k_cache,
                                      self.v_cache, self.k_scale, self.v_scale)

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass

    # convenience wrappers
    def reshape_and_cache(self, key, value, slot_mapping, stream=None):
        reshape_and_cache(self, key, value, slot_mapping, stream)

    def decode(self, q, block_tables, context_lens, scale, max_context_len, out=None,
               workspace=None, partition_blocks=0, kernel=0, schedule=0, stages=0,
               blocks_per_stage=0, window=0, stream=None):
        return paged_attention_decode(self, q, block_tables, context_lens, scale, max_context_len,
                                      out=out, workspace=workspace, partition_blocks=partition_blocks,
                                      kernel=kernel, schedule=schedule, stages=stages,
                                      blocks_per_stage=blocks_per_stage, window=window, stream=stream)

    def device_error(self, stream=None) -> int:
        return get_device_error(self, stream)


def _handle(pool) -> ctypes.c_void_p:
    return pool.handle if isinstance(pool, PagedKVPool) else pool


def reshape_and_cache(pool: PagedKVPool, key: torch.Tensor, value: torch.Tensor,
                      slot_mapping: torch.Tensor, stream=None) -> None:
    """Write key/value bf16 [N, Hkv, d] rows into the pool slots slot_mapping (int32 [N])."""
    _need(key, torch.bfloat16, "key", 3)
    _need(value, torch.bfloat16, "value", 3)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    if key.shape != value.shape or key.shape[0] != slot_mapping.shape[0]:
        raise ValueError("key, value and slot_mapping disagree in shape")
    if key.shape[1:] != (pool.kv_heads, pool.head_dim):
        raise ValueError(f"key rows must be [{pool.kv_heads}, {pool.head_dim}]")
    check(_lib.load().pkv_reshape_and_cache(_handle(pool), _ptr(key), _ptr(value), _ptr(slot_mapping),
                                            key.shape[0], _stream(stream)), "reshape_and_cache")


def decode_workspace_bytes(pool: PagedKVPool, num_seqs: int, num_q_heads: int, max_context_len: int,
                           partition_blocks: int = 0, kernel=0, num_queries: int = 1, window: int = 0) -> int:
    n = ctypes.c_size_t()
    check(_lib.load().pkv_decode_workspace_bytes(_handle(pool), num_seqs, num_q_heads, max_context_len,
                                                 _options(partition_blocks, kernel, num_queries=num_queries,
                                                          window=window),
                                                 ctypes.byref(n)),
          "decode_workspace_bytes")
    return n.value


def decode_plan(pool: PagedKVPool, num_seqs: int, num_q_heads: int, max_context_len: int,
                partition_blocks: int = 0, kernel=0, num_queries: int = 1, window: int = 0) -> dict:
    pb, mp, kc, kf = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    check(_lib.load().pkv_decode_plan(_handle(pool), num_seqs, num_q_heads, max_context_len,
                                      _options(partition_blocks, kernel, num_queries=num_queries, window=window),
                                      ctypes.byref(pb), ctypes.byref(mp),
                                      ctypes.byref(kc), ctypes.byref(kf)), "decode_plan")
    return {"partition_blocks": pb.value, "max_partitions": mp.value, "kernels_per_call": kc.value,
            "kernel": {1: "cuda_core", 2: "tensor_core"}.get(kf.value, str(kf.value))}


def check_decode_shapes(head_dim: int, q_shape, tables_shape, lens_shape, out_shape=None):
    """Shape agreement of a decode call's tensors, checked on the host before anything is
    launched: q [B, Hq, d] or [B, k, Hq, d] with d the pool's head_dim, block_tables
    [B, max_blocks], context_lens [B], out (if given) q's shape.  Returns (B, k, Hq);
    raises ValueError otherwise."""
    q_shape = tuple(q_shape)
    if len(q_shape) == 4:
        b, nq, hq, d = q_shape
    elif len(q_shape) == 3:
        (b, hq, d), nq = q_shape, 1
    else:
        raise ValueError(f"q must be [B, Hq, d] or [B, k, Hq, d], got {q_shape}")
    if d != head_dim:
        raise ValueError(f"q's head_dim {d} is not the pool's {head_dim}")
    if len(tables_shape) != 2 or tables_shape[0] != b or tuple(lens_shape) != (b,):
        raise ValueError("q, block_tables and context_lens disagree in shape")
    if out_shape is not None and tuple(out_shape) != q_shape:
        raise ValueError("out must have q's shape")
    return b, nq, hq


def paged_attention_decode(pool: PagedKVPool, q: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float, max_context_len: int,
                           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           partition_blocks: int = 0, kernel=0, schedule=0, stages=0,
                           blocks_per_stage=0, window: int = 0, stream=None) -> torch.Tensor:
    """Decode attention for q bf16 [B, Hq, d] over the pool; returns out bf16 [B, Hq, d].

    ``window`` W > 0: sliding window, each query attends to its last W tokens only (table
    entries of blocks before the first one any query sees are not read and may be -1).

    A 4-D q [B, k, Hq, d] holds k query tokens per sequence -- its last k cached positions,
    query i attending causally to tokens t < T_b - (k - 1 - i) -- for verifying k draft
    tokens in one pass; out is then [B, k, Hq, d].
    ``workspace`` (a uint8 CUDA tensor) is allocated here when not given and needed."""
    if q.dim() == 4:
        _need(q, torch.bfloat16, "q", 4)
    else:
        _need(q, torch.bfloat16, "q", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if out is not None:
        _need(out, torch.bfloat16, "out", q.dim())
    b, nq, hq = check_decode_shapes(pool.head_dim, q.shape, block_tables.shape, context_lens.shape,
                                    None if out is None else out.shape)
    if out is None:
        out = torch.empty_like(q)
    need = decode_workspace_bytes(pool, b, hq, max_context_len, partition_blocks, kernel, nq, window) if b else 0
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(_lib.load().pkv_paged_attention_decode_ex(
        _handle(pool), _ptr(q), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), b, hq,
        int(max_context_len), float(scale), _ptr(out), _ptr(workspace), ws_bytes,
        _options(partition_blocks, kernel, schedule, stages, blocks_per_stage, nq, window), _stream(stream)),
        "paged_attention_decode")
    return out


def get_device_error(pool: PagedKVPool, stream=None) -> int:
    """Read and clear the pool's device error word (DEVERR_* bits)."""
    v = ctypes.c_uint32()
    check(_lib.load().pkv_get_device_error(_handle(pool), ctypes.byref(v), _stream(stream)),
          "get_device_error")
    return v.value


def selftest_bounded_wait(limit_ns: int, stream=None) -> tuple[int, int]:
    """Run the kernels' bounded wait on a barrier nothing completes: (flags, waited_ns).
    The wait is expected to give up with DEVERR_TIMEOUT after about limit_ns."""
    flags, waited = ctypes.c_uint32(), ctypes.c_uint64()
    check(_lib.load().pkv_selftest_bounded_wait(int(limit_ns), ctypes.byref(flags), ctypes.byref(waited),
                                                _stream(stream)), "selftest_bounded_wait")
    return flags.value, waited.value


def paged_attention_decode_static_scratch(pool: PagedKVPool, q: torch.Tensor, block_tables: torch.Tensor,
                                          context_lens: torch.Tensor, scale: float, max_context_len: int,
                                          out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_attention_decode for callers that cannot allocate device memory: the split-K
    scratch lives in a fixed 16 MiB array inside the library instead of a workspace the
    caller allocates.  Calls that overlap on the GPU share that array and must be
    serialised; shapes that need more scratch raise."""
    _need(q, torch.bfloat16, "q", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    if out is not None:
        _need(out, torch.bfloat16, "out", 3)
    b, _, hq = check_decode_shapes(pool.head_dim, q.shape, block_tables.shape, context_lens.shape,
                                   None if out is None else out.shape)
    if out is None:
        out = torch.empty_like(q)
    lib = _lib.load()
    with torch.cuda.device(q.device):  # the library's scratch address is per device
        st = lib.pkv_paged_attention_decode_static_scratch(
            _handle(pool), _ptr(q), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), b, hq,
            int(max_context_len), float(scale), _ptr(out), _stream(stream))
    if st != 0:
        raise _lib.PagedKVError(st, "paged_attention_decode_static_scratch (" +
                                lib.pkv_static_scratch_error().decode() + ")")
    return out


def copy_blocks(pool: PagedKVPool, pairs: torch.Tensor, stream=None) -> None:
    """Copy whole blocks src -> dst for each row (src, dst) of int32 pairs [n, 2] (CUDA)."""
    _need(pairs, torch.int32, "pairs", 2)
    if pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2]")
    check(_lib.load().pkv_copy_blocks(_handle(pool), _ptr(pairs), pairs.shape[0], _stream(stream)),
          "copy_blocks")


class BlockManager:
    """Host-side free list, reference counts and page tables of a block pool (the C
    ``pkv_block_manager``).  Sequences are small integer handles."""

    def __init__(self, num_blocks: int, max_seqs: int, max_blocks_per_seq: int):
        self.lib = _lib.load()
        self.max_blocks_per_seq = max_blocks_per_seq
        self.handle = ctypes.c_void_p()
        check(self.lib.pkv_block_manager_create(num_blocks, max_seqs, max_blocks_per_seq,
                                                ctypes.byref(self.handle)), "block_manager_create")

    def close(self):
        if getattr(self, "handle", None):
            self.lib.pkv_block_manager_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass

    def add_sequence(self) -> int:
        s = ctypes.c_int()
        check(self.lib.pkv_block_manager_add_sequence(self.handle, ctypes.byref(s)), "add_sequence")
        return s.value

    def fork(self, parent: int) -> int:
        c = ctypes.c_int()
        check(self.lib.pkv_block_manager_fork(self.handle, parent, ctypes.byref(c)), "fork")
        return c.value

    def free_sequence(self, seq: int) -> None:
        check(self.lib.pkv_block_manager_free_sequence(self.handle, seq), "free_sequence")

    def append(self, seqs, num_new_tokens):
        """Reserve slots: returns (slot_mapping int32 [sum], copy_pairs int32 [k, 2]) on the host."""
        seqs = (ctypes.c_int * len(seqs))(*seqs)
        counts = (ctypes.c_int * len(num_new_tokens))(*num_new_tokens)
        total = sum(num_new_tokens)
        slots = torch.empty(max(total, 1), dtype=torch.int32)
        pairs = torch.empty(max(len(seqs), 1), 2, dtype=torch.int32)
        k = ctypes.c_int()
        check(self.lib.pkv_block_manager_append(self.handle, seqs, counts, len(seqs), _ptr(slots),
                                                _ptr(pairs), pairs.shape[0], ctypes.byref(k)), "append")
        return slots[:total], pairs[:k.value]

    def truncate(self, seq: int, num_tokens: int) -> None:
        """Keep the first num_tokens tokens of a sequence (drop rejected draft tokens)."""
        check(self.lib.pkv_block_manager_truncate(self.handle, seq, num_tokens), "truncate")

    def release_before(self, seq: int, token: int) -> None:
        """Give back the blocks holding only tokens before position ``token`` (sliding
        window); their table entries become -1."""
        check(self.lib.pkv_block_manager_release_before(self.handle, seq, token), "release_before")

    def tables(self, seqs):
        """(block_tables int32 [n, max_blocks_per_seq] with -1 padding, context_lens int32 [n])."""
        arr = (ctypes.c_int * len(seqs))(*seqs)
        bt = torch.empty(max(len(seqs), 1), self.max_blocks_per_seq, dtype=torch.int32)
        cl = torch.empty(max(len(seqs), 1), dtype=torch.int32)
        check(self.lib.pkv_block_manager_tables(self.handle, arr, len(seqs), _ptr(bt), _ptr(cl)), "tables")
        return bt[:len(seqs)], cl[:len(seqs)]

    def stats(self) -> tuple[int, int]:
        fb, ls = ctypes.c_int64(), ctypes.c_int()
        check(self.lib.pkv_block_manager_stats(self.handle, ctypes.byref(fb), ctypes.byref(ls)), "stats")
        return fb.value, ls.value

    def refcount(self, block: int) -> int:
        return int(self.lib.pkv_block_manager_refcount(self.handle, block))
