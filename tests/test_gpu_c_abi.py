"""The C ABI without Python in the loop: a C program (tests/c_abi_decode.c) that includes
only pagedkv.h and the CUDA runtime creates a pool, appends a small batch with
pkv_reshape_and_cache, decodes with pkv_paged_attention_decode and prints the bf16 output;
the test builds it with gcc against the in-tree library and compares with the oracle."""

import os
import struct
import subprocess

import numpy as np
import pytest

import oracle
from paged_kv_cache_264_gb300 import build, workloads as W
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_decode(tmp_path):
    lib = build.build()
    oracle.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "c_abi_decode"
    cmd = ["gcc", "-std=c11", "-O2", os.path.join(HERE, "c_abi_decode.c"), "-o", str(exe),
           f"-I{os.path.join(ROOT, 'include')}", f"-I{cuda}/include", f"-L{lib.parent}", "-lpagedkv",
           f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{lib.parent}", f"-Wl,-rpath,{cuda}/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    w = W.build(name="c_abi", context_lens=[5, 17, 40, 129], num_q_heads=8, num_kv_heads=2, head_dim=128,
                seed=81)
    key, value = W.bf16_bits(w.key), W.bf16_bits(w.value)
    q = W.bf16_bits(w.q)
    tables = w.block_tables.numpy().astype(np.int32)
    lens = w.context_lens.numpy().astype(np.int32)
    slots = w.slot_mapping.numpy().astype(np.int32)
    inp = tmp_path / "input.bin"
    with open(inp, "wb") as f:
        f.write(struct.pack("<7i", w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_blocks,
                            tables.shape[1], len(slots)))
        f.write(struct.pack("<f", w.scale))
        for a in (lens, tables, slots, q, key, value):
            f.write(np.ascontiguousarray(a).tobytes())
    r = subprocess.run([str(exe), str(inp)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    bits = np.array([int(x) for x in r.stdout.split()], dtype=np.uint32).astype(np.uint16)
    got = (bits.astype(np.uint32) << 16).view(np.float32).reshape(q.shape)

    o = oracle.load()
    kc = np.zeros((w.num_blocks, w.num_kv_heads, 16, w.head_dim), np.uint16)
    vc = kc.copy()
    o.reshape_and_cache_bf16(key, value, slots, kc, vc)
    ref = o.paged_decode(q, kc, vc, tables, lens, w.scale)

    class _T:  # compare() takes a tensor-like with .float().cpu().numpy()
        def __init__(self, a):
            self.a = a

        def float(self):
            return self

        def cpu(self):
            return self

        def numpy(self):
            return self.a

    compare(_T(got), ref, "C program decode")
