"""Failure detection on the GPU without a fault: every wait in the decode kernels is
bounded.  The library's bounded mbarrier wait, run on a barrier that nothing completes,
must give up after its limit, report PKV_DEVERR_TIMEOUT, and leave the context usable for
the next decode (which must still equal the oracle)."""

import pytest
import torch

import oracle
import paged_kv_cache_264_gb300 as pkv
from paged_kv_cache_264_gb300 import workloads as W
from gpu_helpers import compare, gpu_pool_from, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_264_gb300 import build
    build.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("limit_ms", [1, 20])
def test_bounded_wait_gives_up_and_context_survives(limit_ms):
    limit_ns = limit_ms * 1_000_000
    flags, waited = pkv.selftest_bounded_wait(limit_ns)
    assert flags == pkv.DEVERR_TIMEOUT
    assert limit_ns <= waited < limit_ns + 200_000_000  # gives up soon after the limit
    w = W.build(name="after_timeout", context_lens=[20, 70], num_q_heads=8, num_kv_heads=2, head_dim=128,
                seed=71)
    pool = gpu_pool_from(w, "bf16")
    out = pool.decode(w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda(), w.scale, w.max_context_len)
    torch.cuda.synchronize()
    assert pool.device_error() == 0
    ref, _, _ = oracle_decode(w, "bf16")
    compare(out, ref, "decode after a timed-out wait")
    pool.close()


def test_selftest_rejects_bad_limits():
    for bad in (0, 50_000, 3_000_000_000):
        with pytest.raises(pkv.PagedKVError, match="invalid"):
            pkv.selftest_bounded_wait(bad)
