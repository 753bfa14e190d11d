"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every test runs the whole step -- reshape_and_cache of the step's new tokens,
then paged attention -- on seeded synthetic inputs.  reshape_and_cache must
match the oracle bit for bit over the whole cache; attention must stay
within max-abs 1e-2 (vs fp64) and mean-abs 1e-3 (vs the oracle rounded to
the element type).  Small cases compare every output row; the full-size
workloads compare sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_harness import GpuCase, bits, check_attention, run_and_check

pytestmark = pytest.mark.gpu


def _rows_sample(case, n, seed=0):
    rng = np.random.default_rng(seed)
    T = case.total_query_tokens
    return np.sort(rng.choice(T, size=min(n, T), replace=False))


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_gqa_decode(seed):
    run_and_check(W.tiny_gqa_decode(seed))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_llama8b_decode_small(seed):
    run_and_check(W.llama8b_decode(seed, batch=24, max_ctx=1024))


def test_llama8b_decode_full_size_sampled():
    c = W.llama8b_decode(0)
    run_and_check(c, rows=_rows_sample(c, 48))


@pytest.mark.parametrize("hkv", [1, 8, 32])
def test_head_sweep_small(hkv):
    run_and_check(W.head_sweep(0, num_kv_heads=hkv, batch=6))


@pytest.mark.parametrize("hkv", [1, 8, 32])
def test_head_sweep_full_size_sampled(hkv):
    c = W.head_sweep(1, num_kv_heads=hkv)
    run_and_check(c, rows=_rows_sample(c, 12))


@pytest.mark.parametrize("splits", [0, 16, 32, 64])
def test_long_context_split_kv(splits):
    run_and_check(W.long_context_decode(0, batch=2), num_splits=splits)


def test_long_context_full_size():
    run_and_check(W.long_context_decode(1))


# ---------------------------------------------------------------- mixed
def _small_mixed(seed, **kw):
    args = dict(n_prefill=3, n_decode=5, q_range=(2, 150), prior_range=(0, 300),
                dec_range=(1, 700))
    args.update(kw)
    return W.mixed_prefill_decode(seed, **args)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_mixed_small(seed):
    run_and_check(_small_mixed(seed))


def test_mixed_full_size_sampled():
    c = W.mixed_prefill_decode(0)
    ql = c.query_lens
    dec_rows = c.cu_query_lens[:-1][ql == 1]
    last_rows = c.cu_query_lens[1:][ql > 1] - 1   # last token of each chunk
    first_rows = c.cu_query_lens[:-1][ql > 1]
    rows = np.unique(np.concatenate([dec_rows, last_rows, first_rows,
                                     _rows_sample(c, 96, seed=3)]))
    run_and_check(c, rows=rows)


# ---------------------------------------------------------------- shapes
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 12, 16, 24, 32, 48, 64])
def test_group_sizes_decode_and_prefill(G):
    rng = np.random.default_rng(G)
    hkv = 2 if G <= 16 else 1
    B = 5
    ctx = rng.integers(1, 400, size=B)
    ql = np.minimum(ctx, np.array([1, 1, 37, 1, 9]))
    c = W.make_case(f"g{G}", seed=G, dtype=W.BF16, num_heads=G * hkv, num_kv_heads=hkv,
                    head_dim=128, block_size=16, context_lens=ctx, query_lens=ql)
    run_and_check(c)
    d = W.make_case(f"g{G}d", seed=G + 100, dtype=W.BF16, num_heads=G * hkv,
                    num_kv_heads=hkv, head_dim=128, block_size=16, context_lens=ctx,
                    query_lens=np.ones(B, np.int64))
    run_and_check(d)


@pytest.mark.parametrize("dtype,D", [(W.F16, 64), (W.BF16, 64), (W.F16, 128)])
def test_mqa_decode_dtypes(dtype, D):
    """Head-major decode (G > 8) in both element types and head sizes, with
    ragged contexts that end inside a 16-key tile."""
    rng = np.random.default_rng(41 + D)
    ctx = np.concatenate([[1, 15, 17], rng.integers(18, 900, size=5)])
    c = W.make_case(f"mqa_{D}", seed=41 + D, dtype=dtype, num_heads=32, num_kv_heads=1,
                    head_dim=D, block_size=16, context_lens=ctx,
                    query_lens=np.ones(ctx.size, np.int64))
    run_and_check(c)


@pytest.mark.parametrize("bs", [64, 256])
def test_mqa_decode_block_sizes(bs):
    """Head-major decode reads its 16-key tiles through blocks of any size."""
    rng = np.random.default_rng(61 + bs)
    ctx = np.concatenate([[bs - 1, bs, bs + 1], rng.integers(2, 3000, size=5)])
    c = W.make_case(f"mqa_bs{bs}", seed=61 + bs, dtype=W.BF16, num_heads=32, num_kv_heads=1,
                    head_dim=128, block_size=bs, context_lens=ctx,
                    query_lens=np.ones(ctx.size, np.int64))
    run_and_check(c)


@pytest.mark.parametrize("splits", [0, 16, 64])
def test_mqa_long_context_outliers(splits):
    """MQA over 16k-32k keys with 1% of the K rows scaled by 8: the head-major
    path's reference max moves rarely and late; split partials merge."""
    rng = np.random.default_rng(51)
    ctx = rng.integers(16384, 32769, size=2)
    c = W.make_case("mqa_long", seed=51, rng=rng, dtype=W.BF16, num_heads=32, num_kv_heads=1,
                    head_dim=128, block_size=16, context_lens=ctx,
                    query_lens=np.ones(2, np.int64), key_outlier_prob=0.01)
    run_and_check(c, num_splits=splits)


@pytest.mark.parametrize("bs", [32, 48, 64, 96, 128, 256])
def test_block_sizes(bs):
    rng = np.random.default_rng(bs)
    ctx = rng.integers(1, 1200, size=6)
    ql = np.minimum(ctx, np.array([1, 70, 1, 3, 1, 130]))
    c = W.make_case(f"bs{bs}", seed=bs, dtype=W.BF16, num_heads=16, num_kv_heads=4,
                    head_dim=128, block_size=bs, context_lens=ctx, query_lens=ql)
    run_and_check(c)
    d = W.make_case(f"bs{bs}d", seed=bs + 1, dtype=W.BF16, num_heads=16, num_kv_heads=4,
                    head_dim=128, block_size=bs, context_lens=ctx,
                    query_lens=np.ones(6, np.int64))
    run_and_check(d, num_splits=3)


@pytest.mark.parametrize("dtype,D", [(W.F16, 64), (W.F16, 128), (W.BF16, 64)])
def test_dtypes_and_head_dims(dtype, D):
    rng = np.random.default_rng(D + dtype)
    ctx = rng.integers(1, 900, size=7)
    ql = np.minimum(ctx, np.array([1, 1, 64, 1, 17, 1, 2]))
    c = W.make_case("dt", seed=3, dtype=dtype, num_heads=8, num_kv_heads=2, head_dim=D,
                    block_size=16, context_lens=ctx, query_lens=ql)
    run_and_check(c)
    d = W.make_case("dtd", seed=4, dtype=dtype, num_heads=8, num_kv_heads=2, head_dim=D,
                    block_size=16, context_lens=ctx, query_lens=np.ones(7, np.int64))
    run_and_check(d)


# ---------------------------------------------------------------- edges
def test_empty_and_one_token_contexts():
    ctx = np.array([0, 1, 16, 17, 0, 33])
    ql = np.array([0, 1, 1, 1, 0, 1])
    c = W.make_case("edge", seed=5, dtype=W.BF16, num_heads=8, num_kv_heads=2, head_dim=128,
                    block_size=16, context_lens=ctx, query_lens=ql, is_decode=False)
    run_and_check(c)
    # decode entry point: an empty sequence gets a zero row
    d = W.make_case("edged", seed=6, dtype=W.BF16, num_heads=8, num_kv_heads=2,
                    head_dim=128, block_size=16, context_lens=np.array([3, 1, 40]),
                    query_lens=np.ones(3, np.int64))
    d.context_lens[0] = 0
    d.slot_mapping[0] = -1           # nothing to write for it
    g = GpuCase(d)
    g.write_cache()
    out = g.attention()
    torch.cuda.synchronize()
    assert not bits(out)[0].any()
    o64, ob, _, _ = oracle.run_case(d, rows=np.array([1, 2]))
    check_attention(bits(out)[1:], o64, ob, d.dtype)


def test_whole_chunk_in_one_sequence_and_qlen_equal_ctx():
    ctx = np.array([300, 77])
    ql = np.array([300, 77])          # no cached prefix: pure causal prefill
    c = W.make_case("pure", seed=7, dtype=W.BF16, num_heads=32, num_kv_heads=8,
                    head_dim=128, block_size=16, context_lens=ctx, query_lens=ql)
    run_and_check(c)


# ---------------------------------------------------------------- invariants
def test_block_permutation_is_bitwise_invariant():
    c = W.llama8b_decode(4, batch=16, max_ctx=900)
    g1 = GpuCase(c)
    g1.write_cache()
    o1 = bits(g1.attention())
    rng = np.random.default_rng(11)
    perm = rng.permutation(c.num_blocks)
    c2 = W.make_case("p", seed=0, dtype=c.dtype, num_heads=c.num_heads,
                     num_kv_heads=c.num_kv_heads, head_dim=c.head_dim,
                     block_size=c.block_size, context_lens=c.context_lens,
                     query_lens=c.query_lens)
    c2.q = c.q
    c2.k_cache = np.empty_like(c.k_cache)
    c2.v_cache = np.empty_like(c.v_cache)
    c2.k_cache[perm] = c.k_cache
    c2.v_cache[perm] = c.v_cache
    c2.block_tables = np.where(c.block_tables >= 0, perm[np.maximum(c.block_tables, 0)], -1
                               ).astype(np.int32)
    bs = c.block_size
    c2.slot_mapping = perm[c.slot_mapping // bs] * bs + c.slot_mapping % bs
    c2.k_new, c2.v_new = c.k_new, c.v_new
    g2 = GpuCase(c2)
    g2.write_cache()
    o2 = bits(g2.attention())
    assert np.array_equal(o1, o2)


def test_split_count_independence():
    c = W.llama8b_decode(5, batch=12, max_ctx=3000)
    g = GpuCase(c)
    g.write_cache()
    o64, ob, _, _ = oracle.run_case(c)
    outs = {}
    for s in [1, 2, 5, 17, 64, 0]:
        outs[s] = bits(g.attention(num_splits=s))
        check_attention(outs[s], o64, ob, c.dtype)
    assert np.array_equal(outs[1], bits(g.attention(num_splits=1)))   # deterministic


def test_chunked_entry_with_only_decode_rows_equals_decode_bitwise():
    # with a fixed split count both entry points run the same sorted work
    # list; with automatic splits the decode entry point takes equal shares
    # of the key tiles instead, so there both are held to the oracle
    c = W.llama8b_decode(6, batch=20, max_ctx=2000)
    g = GpuCase(c)
    g.write_cache()
    for s in (1, 3):
        a = bits(g.attention(num_splits=s))
        b = bits(g.attention(num_splits=s, force_chunked=True))
        assert np.array_equal(a, b)
    o64, ob, _, _ = oracle.run_case(c)
    check_attention(bits(g.attention()), o64, ob, c.dtype)
    check_attention(bits(g.attention(force_chunked=True)), o64, ob, c.dtype)


def test_gqa_matches_mha_on_duplicated_kv_heads():
    c = W.head_sweep(2, num_kv_heads=8, batch=4, ctx_len=300)
    g = GpuCase(c)
    g.write_cache()
    o_gqa = bits(g.attention())
    G = c.num_heads // c.num_kv_heads
    kc = g.k_cache.repeat_interleave(G, dim=1).contiguous()
    vc = g.v_cache.repeat_interleave(G, dim=1).contiguous()
    ws = g.pa.alloc_workspace(g.pa.paged_attn_workspace_bytes(
        c.num_seqs, c.num_heads, c.num_heads, c.head_dim, c.max_blocks_per_seq,
        c.block_size, 0), g.q.device)
    o_mha = bits(g.pa.paged_attn_decode(g.q, kc, vc, g.block_tables, g.context_lens, c.scale,
                                        workspace=ws))
    a = oracle.from_bits(o_gqa, c.dtype)
    b = oracle.from_bits(o_mha, c.dtype)
    assert np.max(np.abs(a - b)) <= 2 ** -7


def test_repeated_calls_reuse_the_workspace():
    c = _small_mixed(9)
    g = GpuCase(c)
    g.write_cache()
    a = bits(g.attention())
    for _ in range(3):
        assert np.array_equal(a, bits(g.attention()))


# ---------------------------------------------------------------- device checks
def test_bad_block_id_is_flagged_not_read():
    c = W.llama8b_decode(7, batch=4, max_ctx=300)
    c.block_tables = c.block_tables.copy()
    c.block_tables[1, 0] = c.num_blocks + 1000
    g = GpuCase(c)
    g.write_cache()
    out = g.attention()
    torch.cuda.synchronize()
    assert g.status() & g.pa.PA_DEV_BAD_BLOCK_ID
    assert np.all(np.isfinite(oracle.from_bits(bits(out), c.dtype)))


def test_bad_slot_is_flagged_and_skipped():
    c = W.tiny_gqa_decode(1)
    g = GpuCase(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sm = g.slot_mapping.clone()
    sm[0] = c.num_blocks * c.block_size + 3
    before = bits(g.k_cache)
    g.pa.reshape_and_cache(g.k_new, g.v_new, g.k_cache, g.v_cache, sm, status_word=status)
    torch.cuda.synchronize()
    assert int(status.item()) & g.pa.PA_DEV_BAD_SLOT
    after = bits(g.k_cache)
    kref = before.copy()
    vdummy = bits(g.v_cache).copy()
    keep = np.ones(len(c.slot_mapping), bool)
    keep[0] = False
    sm_h = c.slot_mapping.copy()
    sm_h[0] = -1
    oracle.reshape_and_cache(c.k_new, c.v_new, kref, vdummy, sm_h)
    assert np.array_equal(after, kref)


def test_bad_lengths_are_flagged():
    c = _small_mixed(10)
    c.context_lens = c.context_lens.copy()
    i = int(np.argmax(c.query_lens))
    c.context_lens[i] = c.query_lens[i] - 1    # qlen > ctx
    g = GpuCase(c)
    g.write_cache()
    g.attention()
    torch.cuda.synchronize()
    assert g.status() & g.pa.PA_DEV_BAD_LENGTHS


@pytest.mark.parametrize("hkv", [8, 1])
def test_pipeline_wait_timeout_is_flagged_and_the_next_call_recovers(hkv):
    # a wait limit of a nanosecond makes the decode kernel's waits give up
    # before the first copies land (swap-AB path at 4 heads per KV head,
    # head-major at 32): the call returns, its status word says so, and with
    # the default limit back the next call matches the oracle
    c = W.head_sweep(80 + hkv, num_kv_heads=hkv, batch=8, ctx_len=700)
    g = GpuCase(c)
    g.write_cache()
    sweep = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")  # 256 MiB: out of L2
    g.attention()  # the workspace exists before the timed-out call
    float(sweep.sum())
    g.pa.pa_set_pipeline_wait_limit(1)
    try:
        g.attention()
        torch.cuda.synchronize()
        flags = g.status()
    finally:
        g.pa.pa_set_pipeline_wait_limit(0)
    assert flags & g.pa.PA_DEV_WAIT_TIMEOUT
    out = g.attention()
    torch.cuda.synchronize()
    assert g.status() == 0
    o64, ob, _, _ = oracle.run_case(c)
    check_attention(bits(out), o64, ob, c.dtype)


# --------------------------------------------------------------------------
# cross-attention over a static encoder cache (no causal mask)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bs", [16, 64])
def test_cross_attention_mixed_lengths(bs):
    # encoder lengths incl. 0 and shorter than the query chunk; query rows
    # incl. single rows (decode path) and chunks over several tiles
    enc = np.array([700, 0, 37, 1601, 5, 3202, 90])
    ql = np.array([130, 3, 200, 1, 64, 1, 17])
    c = W.make_cross_case(f"cross_bs{bs}", seed=40 + bs, dtype=W.BF16, num_heads=32,
                          num_kv_heads=8, head_dim=128, block_size=bs, encoder_lens=enc,
                          query_lens=ql)
    run_and_check(c)


@pytest.mark.parametrize("hq,hkv,D,dtype", [(8, 8, 64, W.F16), (16, 2, 128, W.F16),
                                            (32, 1, 128, W.BF16)])
def test_cross_attention_head_layouts(hq, hkv, D, dtype):
    enc = np.array([300, 1100, 64])
    ql = np.array([50, 9, 140])
    c = W.make_cross_case("cross_heads", seed=hq + hkv + D, dtype=dtype, num_heads=hq,
                          num_kv_heads=hkv, head_dim=D, block_size=16, encoder_lens=enc,
                          query_lens=ql)
    run_and_check(c)


def test_cross_attention_decode_workload():
    c = W.cross_attention_decode(0)
    stats, g, out = run_and_check(c)
    # one query row per sequence: the plain decode entry point over the same
    # cache is the same computation
    ref = g.pa.paged_attn_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                 c.scale, num_splits=4)
    cross = g.attention(num_splits=4)
    torch.cuda.synchronize()
    assert np.array_equal(bits(ref), bits(cross))


def test_cross_attention_prefill_workload_sampled_rows():
    c = W.cross_attention_prefill(0)
    rows = np.random.default_rng(0).choice(c.total_query_tokens, size=48, replace=False)
    rows.sort()
    run_and_check(c, rows=rows)


# --------------------------------------------------------------------------
# GQA prefill over contiguous varlen K/V (no cache, no expansion)
# --------------------------------------------------------------------------

def _run_varlen(c, rows=None):
    import mqa_paged_kv_gb300 as pa
    from gpu_harness import elem_dtype, to_dev
    et = elem_dtype(c)
    q, k, v = to_dev(c.q, et), to_dev(c.k, et), to_dev(c.v, et)
    cq, ck = to_dev(c.cu_q), to_dev(c.cu_k)
    out = torch.full_like(q, float("nan"))
    ws = pa.alloc_workspace(pa.gqa_varlen_prefill_workspace_bytes(
        c.num_seqs, c.total_query_tokens, c.num_heads, c.num_kv_heads, c.head_dim), q.device)
    pa.gqa_varlen_prefill(q, k, v, cq, ck, c.max_query_len, c.scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == 0
    o64, ob = oracle.varlen_attention(c.q, c.k, c.v, c.cu_q, c.cu_k, c.scale, c.dtype, rows=rows)
    got = bits(out)
    if rows is not None:
        got = got[np.asarray(rows)]
    return check_attention(got, o64, ob, c.dtype)


@pytest.mark.parametrize("hq,hkv,D,dtype", [(32, 8, 128, W.BF16), (16, 16, 64, W.F16),
                                            (32, 4, 128, W.F16), (32, 1, 128, W.BF16)])
def test_varlen_prefill_prompts(hq, hkv, D, dtype):
    # prompt lengths around the 64-key stage and the tile heights, incl. 1
    ql = np.array([1, 63, 64, 65, 200, 513, 7])
    c = W.make_varlen_case("varlen", seed=hq * 3 + hkv + D, dtype=dtype, num_heads=hq,
                           num_kv_heads=hkv, head_dim=D, q_lens=ql)
    _run_varlen(c)


@pytest.mark.parametrize("G", [3, 12, 48])
def test_prefill_long_chunks_odd_group_sizes(G):
    # Long chunks after prefixes: most tiles hold full tokens and leave in
    # one tensor store whose box is G heads by the tile's tokens (rows
    # G * TQ < 128 when G does not divide 128); each chunk's last tile is
    # copied out row by row.  A decode row rides along.
    hkv = 2 if G <= 12 else 1
    ql = np.array([300, 1, 257, 190])
    ctx = ql + np.array([500, 800, 0, 64])
    c = W.make_case(f"long_g{G}", seed=90 + G, dtype=W.BF16, num_heads=G * hkv,
                    num_kv_heads=hkv, head_dim=128, block_size=16, context_lens=ctx,
                    query_lens=ql)
    run_and_check(c)


def test_varlen_prefill_one_token_tiles():
    # 64 query heads over one KV head: a 128-row tile holds two tokens' 64
    # heads, so odd prompt lengths end in a one-token tile (copied out row
    # by row) and every other tile leaves in one tensor store
    c = W.make_varlen_case("varlen_g64", seed=91, dtype=W.BF16, num_heads=64, num_kv_heads=1,
                           head_dim=128, q_lens=[1, 70, 129, 256])
    _run_varlen(c)


def test_varlen_prefill_chunks_after_a_prefix():
    # more keys than query rows: the chunk sits at the end (bottom-right)
    c = W.make_varlen_case("varlen_prefix", seed=77, dtype=W.BF16, num_heads=32, num_kv_heads=8,
                           head_dim=128, q_lens=[40, 1, 130, 64], k_lens=[300, 90, 131, 64])
    _run_varlen(c)


def test_varlen_prefill_workload_sampled_rows():
    c = W.varlen_prefill_llama8b(0)
    rows = np.sort(np.random.default_rng(1).choice(c.total_query_tokens, 48, replace=False))
    _run_varlen(c, rows=rows)


@pytest.mark.parametrize("limit", [1, 7])
def test_cta_limit_gives_the_same_bits(limit):
    # fewer persistent CTAs only change which SM runs which item (one CTA:
    # the mixed call does not split the SMs between its two kernels)
    c = W.mixed_prefill_decode(5, n_prefill=4, n_decode=12, q_range=(40, 200),
                               prior_range=(0, 600), dec_range=(64, 1500))
    g = GpuCase(c)
    g.write_cache()
    ref = bits(g.attention())
    g.pa.pa_limit_next_call_ctas(limit)
    out = g.attention()
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), ref)


# --------------------------------------------------------------------------
# large sizes: batches beyond one work-list pass, long single chunks
# --------------------------------------------------------------------------

@pytest.mark.parametrize("batch,splits", [(1500, 0), (1500, 2), (2100, 0)])
def test_decode_batch_beyond_one_work_list_pass(batch, splits):
    # more sequences than the work-list kernel's 512 threads: the multi-pass
    # path (split offsets read back from the workspace) with fixed splits, and
    # past the equal-share batch limit (2048) with automatic ones; 1500
    # sequences with automatic splits scan the lengths in several passes of
    # the decode kernel's prologue
    c = W.llama8b_decode(31, batch=batch, max_ctx=1024)
    rows = np.sort(np.random.default_rng(3).choice(c.num_seqs, 96, replace=False))
    run_and_check(c, rows=rows, num_splits=splits)


# --------------------------------------------------------------------------
# equal-share decode (automatic splits of the decode entry point)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("limit", [1, 7, 37])
def test_equal_share_under_cta_limits(limit):
    # the groups' tile ranges follow the grid: a smaller grid cuts the units
    # elsewhere (other partials, same result within the tolerance); the same
    # grid twice gives the same bits
    c = W.llama8b_decode(41, batch=40, max_ctx=3000)
    g = GpuCase(c)
    g.write_cache()
    o64, ob, _, _ = oracle.run_case(c)
    g.pa.pa_limit_next_call_ctas(limit)
    a = bits(g.attention())
    g.pa.pa_limit_next_call_ctas(limit)
    b = bits(g.attention())
    torch.cuda.synchronize()
    assert np.array_equal(a, b)
    check_attention(a, o64, ob, c.dtype)
    assert g.status() == 0


@pytest.mark.parametrize("G,splits", [(4, 0), (16, 0), (32, 0), (64, 0), (32, 3)])
def test_repeated_decode_calls_give_the_same_bits(G, splits):
    # the same call on the same grid repeats its arithmetic exactly: a stage
    # read before its copy landed, a query slot reused too early or a
    # partial read before it was written would show up as differing bits
    hkv = 2 if G <= 16 else 1
    c = W.make_case(f"rep_g{G}", seed=70 + G, dtype=W.BF16, num_heads=G * hkv,
                    num_kv_heads=hkv, head_dim=128, block_size=16,
                    context_lens=np.random.default_rng(G).integers(1, 2500, size=24),
                    query_lens=np.ones(24, np.int64))
    g = GpuCase(c)
    g.write_cache()
    first = bits(g.attention(num_splits=splits))
    for _ in range(6):
        assert np.array_equal(bits(g.attention(num_splits=splits)), first)
    o64, ob, _, _ = oracle.run_case(c)
    check_attention(first, o64, ob, c.dtype)


@pytest.mark.parametrize("G", [16, 32, 64])
def test_head_major_bits_repeat_between_other_problems(G):
    # Between calls a GQA decode of 0.7 GB runs, so the next call's keys come
    # from HBM again and its warps are timed differently.  A query slot handed
    # back before the warps' reads of it had finished let the next item's
    # rows into one warp's item in about 7 % of such calls (one sequence,
    # some heads); 300 calls leave no room for that.
    hkv = 2 if G == 16 else 1
    c = W.make_case(f"hm_g{G}", seed=80 + G, dtype=W.BF16, num_heads=G * hkv,
                    num_kv_heads=hkv, head_dim=128, block_size=16,
                    context_lens=np.full(40, 700), query_lens=np.ones(40, np.int64))
    g = GpuCase(c)
    g.write_cache()
    other = GpuCase(W.llama8b_decode(21, batch=48, max_ctx=2048))
    other.write_cache()
    first = g.attention().clone()
    torch.cuda.synchronize()
    o64, ob, _, _ = oracle.run_case(c)
    check_attention(bits(first), o64, ob, c.dtype)
    same = 0
    for _ in range(300):
        other.attention()
        same += int(torch.equal(g.attention().view(torch.int16), first.view(torch.int16)))
    assert same == 300
    assert g.status() == 0


def test_equal_share_one_sequence_over_every_group():
    # one MQA unit of 32k keys cut into a piece per warp group (more pieces
    # than a warp's 32 lanes in the merge), and one GQA sequence beside a run
    # of empty ones
    for hkv, ctx in ((1, [32768]), (8, [0, 0, 0, 20000, 0])):
        ctx = np.array(ctx)
        c = W.make_case("one_long", seed=43 + hkv, dtype=W.BF16, num_heads=32,
                        num_kv_heads=hkv, head_dim=128, block_size=16,
                        context_lens=np.maximum(ctx, 1), query_lens=np.ones(len(ctx), np.int64))
        c.context_lens = c.context_lens.copy()
        c.context_lens[ctx == 0] = 0          # key-less sequences
        c.slot_mapping = np.where(ctx > 0, c.slot_mapping, -1)  # nothing to write for them
        g = GpuCase(c)
        g.write_cache()
        out = g.attention()
        torch.cuda.synchronize()
        got = bits(out)
        live = np.nonzero(c.context_lens > 0)[0]
        o64, ob, _, _ = oracle.run_case(c, rows=live)
        check_attention(got[live], o64, ob, c.dtype)
        assert not got[c.context_lens == 0].any()  # key-less sequences: zero rows


def test_equal_share_bad_length_is_flagged():
    c = W.llama8b_decode(44, batch=6, max_ctx=500)
    g = GpuCase(c)
    g.write_cache()
    ctx = g.context_lens.clone()
    ctx[2] = c.max_blocks_per_seq * c.block_size + 1   # beyond the table
    g.context_lens = ctx
    out = g.attention()
    torch.cuda.synchronize()
    assert g.status() & g.pa.PA_DEV_BAD_LENGTHS
    got = bits(out)
    assert not got[2].any()                            # no keys read: a zero row
    rows = np.array([0, 1, 3, 4, 5])
    o64, ob, _, _ = oracle.run_case(c, rows=rows)
    check_attention(got[rows], o64, ob, c.dtype)


def test_mixed_batch_beyond_one_work_list_pass():
    c = W.mixed_prefill_decode(32, n_prefill=40, n_decode=700, q_range=(2, 96),
                               prior_range=(0, 300), dec_range=(16, 600))
    rows = np.sort(np.random.default_rng(4).choice(c.total_query_tokens, 96, replace=False))
    run_and_check(c, rows=rows)


def test_one_long_chunk():
    # 4096 query tokens of one sequence after a 1000-token prefix: 64 tile pairs
    c = W.make_case("long_chunk", seed=33, dtype=W.BF16, num_heads=32, num_kv_heads=8,
                    head_dim=128, block_size=16, context_lens=[5096, 40],
                    query_lens=[4096, 1])
    rows = np.sort(np.concatenate([np.random.default_rng(5).choice(4096, 40, replace=False),
                                   [0, 4095, 4096]]))
    run_and_check(c, rows=rows)


def test_varlen_one_long_prompt():
    c = W.make_varlen_case("varlen_long", seed=34, dtype=W.BF16, num_heads=32, num_kv_heads=8,
                           head_dim=128, q_lens=[8192, 3])
    rows = np.sort(np.concatenate([np.random.default_rng(6).choice(8192, 40, replace=False),
                                   [8191, 8192, 8194]]))
    _run_varlen(c, rows=rows)
