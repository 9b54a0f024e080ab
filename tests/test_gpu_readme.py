"""The README's Python example, run as written.

The code block under "Example (Python)" is extracted from README.md and executed; its
decode output is then checked against attention recomputed in fp32 from what the example
left in the pool (INT8 codes times their scales, gathered through the block tables), so
that the documented calls, argument orders and shapes stay those of the package.
"""

import math
import os
import re

import pytest
import torch

import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example_code() -> str:
    text = open(os.path.join(ROOT, "README.md")).read()
    m = re.search(r"## Example \(Python\)\n\n((?:    .*\n|\n)+)", text)
    assert m, "README.md has no indented code block under 'Example (Python)'"
    lines = [ln[4:] if ln.startswith("    ") else ln for ln in m.group(1).splitlines()]
    return "\n".join(lines).strip() + "\n"


def _reference(pool, q, tables, lens, scale):
    """fp32 attention over the pool's dequantised K/V, walked through the block tables."""
    kc = pool.k_cache.float() * pool.k_scale[..., None]
    vc = pool.v_cache.float() * pool.v_scale[..., None]
    hkv = pool.kv_heads
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    for b in range(q.shape[0]):
        t = int(lens[b])
        blocks = tables[b, : (t + 15) // 16].long()
        k = kc[blocks].permute(1, 0, 2, 3).reshape(hkv, -1, pool.head_dim)[:, :t]  # [Hkv, T, d]
        v = vc[blocks].permute(1, 0, 2, 3).reshape(hkv, -1, pool.head_dim)[:, :t]
        g = q.shape[1] // hkv
        qb = q[b].float().view(hkv, g, -1)
        p = torch.softmax(torch.einsum("hgd,htd->hgt", qb, k) * scale, dim=-1)
        out[b] = torch.einsum("hgt,htd->hgd", p, v).reshape(q.shape[1], -1)
    return out


def test_readme_example_runs_and_matches():
    build.build()
    torch.manual_seed(0)
    env = {}
    exec(compile(_example_code(), "README.md example", "exec"), env)
    pool, q, out, tables, lens, d = (env[k] for k in ("pool", "q", "out", "tables", "lens", "d"))
    torch.cuda.synchronize()
    assert out.shape == q.shape and out.dtype == torch.bfloat16
    assert pool.device_error() == 0
    ref = _reference(pool, q, tables.cuda(), lens, 1.0 / math.sqrt(d))
    err = (out.float() - ref).abs()
    assert err.max().item() < 1e-2 and err.mean().item() < 1e-3, (err.max().item(), err.mean().item())
    pool.close()
