"""The decode step under CUDA graphs: append + decode (programmatic dependent launches)
captured once into a torch CUDA graph and replayed with new inputs copied into the captured
buffers.  Each replay equals the oracle.  Small batches are launch-bound, which is what
graph replay removes."""

import numpy as np
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


@pytest.mark.parametrize("kv,partition_blocks", [("bf16", 0), ("bf16", 2), ("int8", 0), ("fp8", 3)])
def test_decode_step_in_cuda_graph(kv, partition_blocks):
    w = W.build(name="graph", context_lens=[17, 40, 95, 260], num_q_heads=16, num_kv_heads=4, head_dim=128,
                kv_dtype=kv, seed=61)
    pool = gpu_pool_from(w, kv)
    dev = torch.device("cuda")
    last = w.last_token_rows().to(dev)
    k_new = w.key.to(dev)[last].contiguous()
    v_new = w.value.to(dev)[last].contiguous()
    slots = w.slot_mapping.to(dev)[last].contiguous()
    q = w.q.to(dev).clone()
    tab, lens = w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    nbytes = pkv.decode_workspace_bytes(pool, w.num_seqs, w.num_q_heads, w.max_context_len, partition_blocks)
    ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()

    def step():
        pkv.reshape_and_cache(pool, k_new, v_new, slots, stream)
        pkv.paged_attention_decode(pool, q, tab, lens, w.scale, w.max_context_len, out=out, workspace=ws,
                                   partition_blocks=partition_blocks, stream=stream)

    with torch.cuda.stream(stream):
        step()  # first call outside the capture (kernel attributes, occupancy cache)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    gen = torch.Generator().manual_seed(62)
    for rep in range(3):
        q_host = torch.randn(q.shape, generator=gen).to(torch.bfloat16)
        q.copy_(q_host.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        assert pool.device_error() == 0
        ref, _, _ = oracle_decode(w, kv, q=q_host)
        compare(out, ref, f"graph replay {rep} {kv} P={partition_blocks}")
    pool.close()
