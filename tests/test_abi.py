"""The C-ABI library without a GPU: it loads, exports every symbol the header declares,
and rejects bad host-side arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_264_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_pool_create", "pkv_reshape_and_cache", "pkv_paged_attention_decode",
                     "pkv_decode_workspace_bytes", "pkv_get_device_error", "pkv_pool_destroy"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_binding_declares_only_header_symbols():
    assert set(_lib.SIGNATURES) <= set(declared_functions())


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"ok"
    assert b"invalid" in lib.pkv_status_string(1)
    assert b"unsupported" in lib.pkv_status_string(2)
    assert lib.pkv_version().decode().count(".") == 2


def test_pool_bytes(lib):
    kv, sc = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.pkv_pool_bytes(10, 8, 128, _lib.PKV_KV_BF16, ctypes.byref(kv), ctypes.byref(sc)) == 0
    assert kv.value == 10 * 8 * 16 * 128 * 2 and sc.value == 0
    assert lib.pkv_pool_bytes(10, 8, 128, _lib.PKV_KV_INT8, ctypes.byref(kv), ctypes.byref(sc)) == 0
    assert kv.value == 10 * 8 * 16 * 128 and sc.value == 10 * 8 * 16 * 4
    assert lib.pkv_pool_bytes(10, 8, 128, _lib.PKV_KV_FP8_E4M3, ctypes.byref(kv), ctypes.byref(sc)) == 0
    assert kv.value == 10 * 8 * 16 * 128 and sc.value == 10 * 8 * 16 * 4
    assert lib.pkv_pool_bytes(0, 8, 128, 0, None, None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_pool_bytes(10, 8, 128, 7, None, None) == _lib.PKV_ERR_INVALID_ARG


FAKE = ctypes.c_void_p(0x100000)  # aligned, never dereferenced: rejected before any CUDA call
ODD = ctypes.c_void_p(0x100008)


@pytest.mark.parametrize("args,expect", [
    ((0, 8, 128, 16, 0, FAKE, FAKE, None, None), _lib.PKV_ERR_INVALID_ARG),   # no blocks
    ((4, 8, 128, 16, 0, None, FAKE, None, None), _lib.PKV_ERR_INVALID_ARG),   # NULL K
    ((4, 8, 128, 16, 0, ODD, FAKE, None, None), _lib.PKV_ERR_INVALID_ARG),    # misaligned K
    ((4, 8, 128, 16, 0, FAKE, FAKE, FAKE, FAKE), _lib.PKV_ERR_INVALID_ARG),   # scales on bf16
    ((4, 8, 128, 16, 1, FAKE, FAKE, None, None), _lib.PKV_ERR_INVALID_ARG),   # int8 without scales
    ((4, 8, 128, 16, 2, FAKE, FAKE, None, None), _lib.PKV_ERR_INVALID_ARG),   # fp8 without scales
    ((4, 8, 128, 16, 3, FAKE, FAKE, None, None), _lib.PKV_ERR_INVALID_ARG),   # unknown dtype
    ((4, 8, 96, 16, 0, FAKE, FAKE, None, None), _lib.PKV_ERR_UNSUPPORTED),    # head_dim 96
    ((4, 8, 128, 32, 0, FAKE, FAKE, None, None), _lib.PKV_ERR_UNSUPPORTED),   # block size 32
])
def test_pool_create_rejects(lib, args, expect):
    h = ctypes.c_void_p()
    assert lib.pkv_pool_create(*args, ctypes.byref(h)) == expect
    assert not h.value


def test_null_pool_rejected(lib):
    assert lib.pkv_reshape_and_cache(None, FAKE, FAKE, FAKE, 4, None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_attention_decode(None, FAKE, FAKE, 4, FAKE, 2, 8, 64, 1.0, FAKE, None, 0,
                                          None) == _lib.PKV_ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert lib.pkv_decode_workspace_bytes(None, 2, 8, 64, None, ctypes.byref(n)) == _lib.PKV_ERR_INVALID_ARG
    f = ctypes.c_uint32()
    assert lib.pkv_get_device_error(None, ctypes.byref(f), None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_pool_destroy(None) == 0


def test_launch_count_starts_at_zero_without_work(lib):
    assert lib.pkv_launch_count() == 0 or lib.pkv_launch_count() > 0  # a plain counter


def test_ctypes_layout_and_constants_match_the_header(tmp_path):
    """The binding's mirror of the header, checked by the C compiler: the options struct's
    size and field offsets, and the status, pool-type, kernel, schedule and device-error
    constants."""
    import shutil
    import subprocess

    import paged_kv_cache_264_gb300 as pkv

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in _lib.DecodeOptions._fields_]
    consts = ["PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED", "PKV_ERR_CUDA",
              "PKV_ERR_WORKSPACE", "PKV_ERR_CAPACITY", "PKV_KV_BF16", "PKV_KV_INT8",
              "PKV_KV_FP8_E4M3", "PKV_KERNEL_AUTO", "PKV_KERNEL_CUDA_CORE",
              "PKV_KERNEL_TENSOR_CORE", "PKV_SCHEDULE_AUTO", "PKV_SCHEDULE_GRID",
              "PKV_SCHEDULE_PERSISTENT", "PKV_DEVERR_BLOCK_ID", "PKV_DEVERR_CONTEXT_LEN",
              "PKV_DEVERR_SLOT", "PKV_DEVERR_TIMEOUT", "PKV_BLOCK_SIZE"]
    src = tmp_path / "layout.c"
    body = ['printf("size %zu\\n", sizeof(pkv_decode_options));']
    body += [f'printf("{f} %zu\\n", offsetof(pkv_decode_options, {f}));' for f in fields]
    body += [f'printf("{c} %lld\\n", (long long)({c}));' for c in consts]
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"pagedkv.h\"\n"
                   "int main(void) {\n" + "\n".join(body) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                      check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(_lib.DecodeOptions)
    for f in fields:
        assert int(got[f]) == getattr(_lib.DecodeOptions, f).offset, f
    from paged_kv_cache_264_gb300 import api
    py = {c: getattr(_lib, c) for c in consts[:9]}
    py.update(PKV_KERNEL_AUTO=api._KERNELS["auto"], PKV_KERNEL_CUDA_CORE=api._KERNELS["cuda_core"],
              PKV_KERNEL_TENSOR_CORE=api._KERNELS["tensor_core"],
              PKV_SCHEDULE_AUTO=api._SCHEDULES["auto"], PKV_SCHEDULE_GRID=api._SCHEDULES["grid"],
              PKV_SCHEDULE_PERSISTENT=api._SCHEDULES["persistent"],
              PKV_DEVERR_BLOCK_ID=pkv.DEVERR_BLOCK_ID, PKV_DEVERR_CONTEXT_LEN=pkv.DEVERR_CONTEXT_LEN,
              PKV_DEVERR_SLOT=pkv.DEVERR_SLOT, PKV_DEVERR_TIMEOUT=pkv.DEVERR_TIMEOUT,
              PKV_BLOCK_SIZE=16)
    assert set(py) == set(consts)
    for c in consts:
        assert int(got[c]) == int(py[c]), c
