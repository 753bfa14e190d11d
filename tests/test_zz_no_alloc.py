"""paged_attn_decode_noalloc: the decode entry point for callers that cannot
allocate device scratch memory (a runtime whose allocator already owns
nearly all of HBM, a plugin host that passes only inputs and outputs).

It keeps its workspace in a device array inside the library, so the tests
call it through the C ABI exactly as such a caller would -- no workspace
argument.  Each call is checked against the fp64 oracle directly and, bit
for bit, against paged_attn_decode with a caller workspace (the same kernels
on the same inputs).  The calls run back to back with different inputs, in
both orders -- a small problem after one that filled the array nearly to its
end, and the other way round -- so that nothing the previous call left in
the shared array can leak into the next.  This file is collected last; it
also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_harness import GpuCase, bits, check_attention

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20  # the array's size, as the header states


def _noalloc(g, out, num_splits=0):
    c, pa = g.case, g.pa
    return pa._lib.paged_attn_decode_noalloc(
        ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(g.k_cache.data_ptr()),
        ctypes.c_void_p(g.v_cache.data_ptr()), ctypes.c_void_p(g.block_tables.data_ptr()),
        c.max_blocks_per_seq, ctypes.c_void_p(g.context_lens.data_ptr()), float(c.scale),
        c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size, c.num_blocks,
        1 if c.dtype == W.BF16 else 0, num_splits, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _near_limit_case(seed):
    """A decode batch with 16 fixed KV splits per sequence whose workspace is
    the largest that fits the array: every sequence has at least 16 blocks,
    so all of its splits are used and the last partials sit at the array's
    end."""
    import mqa_paged_kv_gb300 as pa
    H, Hkv, D, bs, S, mbs = 32, 8, 128, 16, 16, 40
    B = 1
    while pa.paged_attn_workspace_bytes(B + 1, H, Hkv, D, mbs, bs, S) <= STATIC_SCRATCH_BYTES:
        B += 1
    need = pa.paged_attn_workspace_bytes(B, H, Hkv, D, mbs, bs, S)
    assert STATIC_SCRATCH_BYTES - need < STATIC_SCRATCH_BYTES // 32, need
    rng = np.random.default_rng(seed)
    ctx = rng.integers(16 * bs, mbs * bs + 1, size=B)
    c = W.make_case(f"noalloc_near_limit_b{B}", seed=seed, rng=rng, dtype=W.BF16,
                    num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                    context_lens=ctx, query_lens=np.ones(B, np.int64),
                    max_blocks_per_seq=mbs)
    return c, S


def _cases():
    return [(W.tiny_gqa_decode(2), 0),
            _near_limit_case(23),
            (W.llama8b_decode(21, batch=48, max_ctx=2048), 0),
            (W.head_sweep(24, num_kv_heads=1, batch=40, ctx_len=700), 0)]


def _check_one(c, num_splits):
    g = GpuCase(c)
    g.write_cache()
    ref = bits(g.attention(num_splits=num_splits))
    out = torch.full_like(g.q, float("nan"))
    assert _noalloc(g, out, num_splits) == 0
    torch.cuda.synchronize()
    got = bits(out)
    o64, ob, _, _ = oracle.run_case(c)
    check_attention(got, o64, ob, c.dtype)          # the oracle, directly
    assert np.array_equal(got, ref)                 # same kernels as the workspace path


def test_noalloc_matches_oracle_on_calls_in_a_row_both_orders():
    cases = _cases()
    for c, s in cases + cases[::-1]:
        _check_one(c, s)


def test_noalloc_rejects_problems_beyond_its_array():
    c = W.llama8b_decode(22, batch=8, max_ctx=1024)
    g = GpuCase(c)
    big_seqs = 4096  # 4096 x 64 splits x 32 heads x 129 floats >> 32 MiB
    assert g.pa.paged_attn_workspace_bytes(big_seqs, 32, 8, 128, 4096, 16, 64) > \
        STATIC_SCRATCH_BYTES
    rc = g.pa._lib.paged_attn_decode_noalloc(
        ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(g.k_cache.data_ptr()),
        ctypes.c_void_p(g.v_cache.data_ptr()), ctypes.c_void_p(g.block_tables.data_ptr()),
        4096, ctypes.c_void_p(g.context_lens.data_ptr()), 0.1, big_seqs, 32, 8, 128, 16,
        c.num_blocks, 1, 64, ctypes.c_void_p(g.q.data_ptr()), None)
    assert rc == -6  # PA_ERR_WORKSPACE, nothing launched
