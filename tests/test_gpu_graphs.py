"""A serving step captured once in a CUDA graph and replayed with new inputs.

The library's calls issue only stream work (kernel launches, no host
synchronisation, no allocation inside a call), and every kernel reads the
lengths, block tables and query offsets from device memory when it runs,
so a captured step replays correctly for any batch with the captured
shapes: the same sequence count, query-token count, cache and table
sizes.  Each replay here loads another batch of that shape (other lengths,
tables and values) into the captured tensors and is checked against the
oracle, cache bits and attention alike.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_harness import GpuCase, bits, check_attention, elem_dtype

pytestmark = pytest.mark.gpu

B, HQ, HKV, D, BS, MBS = 16, 32, 8, 128, 16, 64
NUM_BLOCKS = B * MBS + 64


def _case(seed, query_lens):
    rng = np.random.default_rng(seed)
    ctx = np.maximum(rng.integers(1, MBS * BS + 1, size=B), query_lens)
    return W.make_case(f"graph_{seed}", seed=seed, rng=rng, dtype=W.BF16, num_heads=HQ,
                       num_kv_heads=HKV, head_dim=D, block_size=BS, context_lens=ctx,
                       query_lens=query_lens, num_blocks=NUM_BLOCKS, max_blocks_per_seq=MBS)


def _load(g, c):
    """Copy case c into the captured tensors of GpuCase g (same shapes)."""
    et = elem_dtype(c)

    def put(dst, a, dtype=None):
        src = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            src = src.view(torch.int16).view(dtype)
        assert tuple(src.shape) == tuple(dst.shape)
        dst.copy_(src)

    put(g.q, c.q, et)
    put(g.k_cache, c.k_cache, et)
    put(g.v_cache, c.v_cache, et)
    put(g.k_new, c.k_new, et)
    put(g.v_new, c.v_new, et)
    put(g.slot_mapping, c.slot_mapping)
    put(g.block_tables, c.block_tables)
    put(g.context_lens, c.context_lens)
    put(g.cu_query_lens, c.cu_query_lens)


@pytest.mark.parametrize("kind", ["decode", "chunked"])
def test_step_captured_in_a_cuda_graph_replays_with_new_batches(kind):
    import mqa_paged_kv_gb300 as pa
    if kind == "decode":
        ql = np.ones(B, np.int64)
    else:  # query chunks of 1 to 96 tokens beside decode rows
        ql = np.where(np.arange(B) % 3 == 0, 1 + (np.arange(B) * 37) % 96, 1).astype(np.int64)
    cases = [_case(s, ql) for s in (101, 102, 103)]
    c0 = cases[0]
    g = GpuCase(c0)
    tq = c0.total_query_tokens
    out = torch.empty_like(g.q)
    if kind == "decode":
        nb = pa.paged_attn_workspace_bytes(B, HQ, HKV, D, MBS, BS, 0)
    else:
        nb = pa.paged_attn_chunked_prefill_workspace_bytes(B, tq, HQ, HKV, D, MBS, BS, 0)
    ws = pa.alloc_workspace(nb, g.q.device)
    max_ql = int(ql.max())

    def step():
        pa.reshape_and_cache(g.k_new, g.v_new, g.k_cache, g.v_cache, g.slot_mapping)
        if kind == "decode":
            pa.paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                 c0.scale, out=out, workspace=ws)
        else:
            pa.paged_attn_chunked_prefill(g.q, g.k_cache, g.v_cache, g.block_tables,
                                          g.cu_query_lens, g.context_lens, max_ql, c0.scale,
                                          out=out, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # first calls outside the capture (kernel attributes)
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    torch.cuda.synchronize()

    for c in cases[1:] + cases[:1]:
        _load(g, c)
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        o64, ob, kref, vref = oracle.run_case(c)
        assert np.array_equal(bits(g.k_cache), kref), "k_cache differs"
        assert np.array_equal(bits(g.v_cache), vref), "v_cache differs"
        check_attention(bits(out), o64, ob, c.dtype)
        assert pa.pa_read_device_status(ws) == 0
