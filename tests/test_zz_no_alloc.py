"""paged_attn_decode_noalloc: the decode entry point for callers that cannot
allocate device scratch memory (a runtime whose allocator already owns
nearly all of HBM, a plugin host that passes only inputs and outputs).

It keeps its workspace in a device array inside the library, so the test
calls it through the C ABI exactly as such a caller would -- no workspace
argument -- and checks it against paged_attn_decode (which takes a caller
workspace) on two calls in a row with different inputs, so that whatever the
first call leaves in the shared array cannot leak into the second.  This
file is collected last; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_harness import GpuCase, bits, check_attention

pytestmark = pytest.mark.gpu


def _noalloc(g, out, num_splits=0):
    c, pa = g.case, g.pa
    return pa._lib.paged_attn_decode_noalloc(
        ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(g.k_cache.data_ptr()),
        ctypes.c_void_p(g.v_cache.data_ptr()), ctypes.c_void_p(g.block_tables.data_ptr()),
        c.max_blocks_per_seq, ctypes.c_void_p(g.context_lens.data_ptr()), float(c.scale),
        c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks,
        1 if c.dtype == W.BF16 else 0, num_splits, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cases = [W.llama8b_decode(21, batch=48, max_ctx=2048),
             W.tiny_gqa_decode(2)]
    for c in cases:
        g = GpuCase(c)
        g.write_cache()
        ref = bits(g.attention())
        out = torch.full_like(g.q, float("nan"))
        assert _noalloc(g, out) == 0
        torch.cuda.synchronize()
        got = bits(out)
        # same kernels on the same inputs: within the parity tolerance
        # (and in fact bit for bit)
        check_attention(got, oracle.from_bits(ref, c.dtype), ref, c.dtype)
        assert np.array_equal(got, ref)


def test_noalloc_rejects_problems_beyond_its_array():
    c = W.llama8b_decode(22, batch=8, max_ctx=1024)
    g = GpuCase(c)
    big_seqs = 4096  # 4096 x 64 splits x 32 heads x 129 floats >> 32 MiB
    rc = g.pa._lib.paged_attn_decode_noalloc(
        ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(g.k_cache.data_ptr()),
        ctypes.c_void_p(g.v_cache.data_ptr()), ctypes.c_void_p(g.block_tables.data_ptr()),
        4096, ctypes.c_void_p(g.context_lens.data_ptr()), 0.1, big_seqs, 32, 8, 128, 16,
        c.num_blocks, 1, 64, ctypes.c_void_p(g.q.data_ptr()), None)
    assert rc == -6  # PA_ERR_WORKSPACE, nothing launched
