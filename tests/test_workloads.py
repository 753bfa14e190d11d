"""The seeded input generators keep their stated recipe (CPU only).

Both the oracle and the CUDA path are fed these arrays, so a generator that
silently drifted (a block id handed out twice, a slot past a context that is
not NaN, a new token's slot already holding a value) would make a parity test
pass without exercising what it claims to: the masking of garbage past each
context, the block-table gather, the cache write before attention.  These
checks fix the layout of every named workload and the figures the benchmark's
algorithmic bytes and flops are computed from."""
import math

import numpy as np
import pytest

import workloads as W

EXP_MASK = {W.F16: 0x7C00, W.BF16: 0x7F80}


def _slot_positions(case, b):
    """Cache slot (block id * bs + offset) of every position of sequence b."""
    bs = case.block_size
    pos = np.arange(int(case.context_lens[b]), dtype=np.int64)
    blocks = case.block_tables[b].astype(np.int64)
    return blocks[pos // bs] * bs + pos % bs


def _nonfinite_per_slot(cache, dtype):
    """[NB * bs] -> (all elements non-finite, any element non-finite)."""
    m = EXP_MASK[dtype]
    nf = (cache & np.uint16(m)) == np.uint16(m)                  # [NB, Hkv, bs, D]
    nf = nf.transpose(0, 2, 1, 3).reshape(cache.shape[0] * cache.shape[2], -1)
    return nf.all(axis=1), nf.any(axis=1)


def check_layout(case, new_tokens_written=False):
    B, bs, NB = case.num_seqs, case.block_size, case.num_blocks
    ctx = case.context_lens.astype(np.int64)
    ql = case.query_lens.astype(np.int64)
    bt = case.block_tables
    assert bt.dtype == np.int32 and bt.shape[0] == B
    assert case.cu_query_lens[0] == 0 and np.all(ql >= 0)
    if not case.cross:
        assert np.all(ql <= ctx)
    used = []
    for b in range(B):
        n = -(-int(ctx[b]) // bs)
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, :n] < NB), b
        assert np.all(bt[b, n:] == -1), b           # padding is a -1 suffix
        used.append(bt[b, :n])
    used = np.concatenate(used) if used else np.zeros(0, np.int32)
    assert np.unique(used).size == used.size        # no block shared by two owners

    prior = np.zeros(NB * bs, bool)
    new = np.zeros(NB * bs, bool)
    expect_slots = []
    for b in range(B):
        s = _slot_positions(case, b)
        p = int(ctx[b] - (0 if case.cross else ql[b]))
        prior[s[:p]] = True
        new[s[p:]] = True
        expect_slots.append(s[p:])
    if case.cross:
        assert case.slot_mapping.size == 0 and case.k_new.shape[0] == 0
        assert not new.any()
    else:
        assert np.array_equal(case.slot_mapping, np.concatenate(expect_slots))
        assert case.k_new.shape == (case.total_query_tokens, case.num_kv_heads, case.head_dim)
    for cache in (case.k_cache, case.v_cache):
        all_nf, any_nf = _nonfinite_per_slot(cache, case.dtype)
        assert not any_nf[prior].any()              # every prior token is finite
        assert all_nf[~prior].all()                 # every other slot is NaN, new slots too
        nan_bits = (cache == np.uint16(W.NAN_BITS[case.dtype]))
        assert nan_bits.sum() == (~prior).sum() * case.num_kv_heads * case.head_dim
    for a in (case.q, case.k_new, case.v_new):
        m = EXP_MASK[case.dtype]
        assert not ((a & np.uint16(m)) == np.uint16(m)).any()
    return prior, new


def test_tiny_case_layout():
    c = W.tiny_gqa_decode(0)
    assert (c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim) == (4, 8, 2, 64)
    assert c.dtype == W.F16 and c.block_size == 16 and c.num_blocks == 64
    assert c.scale == 0.125 and c.is_decode
    assert np.all((c.context_lens >= 1) & (c.context_lens <= 256))
    check_layout(c)


@pytest.fixture(scope="module")
def llama():
    return W.llama8b_decode(0)


def test_llama8b_decode_figures(llama):
    # The benchmark's headline bytes: 164,001 context tokens x 8 KV heads x
    # 128 x (K, V) x 2 bytes = 671,748,096 bytes per attention pass.
    assert (llama.num_seqs, llama.num_heads, llama.num_kv_heads, llama.head_dim) == (256, 32, 8, 128)
    assert llama.dtype == W.BF16 and llama.block_size == 16
    assert int(llama.context_lens.sum()) == 164001
    assert llama.kv_bytes() == 671748096
    assert llama.max_blocks_per_seq == 256
    need = int(((llama.context_lens + 15) // 16).sum())
    assert llama.num_blocks == need + math.ceil(0.05 * need)


def test_llama8b_context_lengths_are_clipped_lognormal(llama):
    ctx = llama.context_lens
    assert ctx.min() >= 16 and ctx.max() <= 4096
    # lognormal with median 400 and sigma 1 (256 draws): loose bounds
    assert 300 <= np.median(ctx) <= 520
    assert 0.8 <= np.std(np.log(ctx)) <= 1.2


def test_llama8b_layout_small_batch():
    check_layout(W.llama8b_decode(3, batch=24))


def test_spare_blocks_are_entirely_nan():
    c = W.llama8b_decode(1, batch=16)
    spare = np.setdiff1d(np.arange(c.num_blocks), c.block_tables[c.block_tables >= 0])
    assert spare.size > 0
    assert np.all(c.k_cache[spare] == np.uint16(W.NAN_BITS[c.dtype]))
    assert np.all(c.v_cache[spare] == np.uint16(W.NAN_BITS[c.dtype]))


def test_block_size_changes_paging_not_lengths():
    a, b = W.llama8b_decode(2, batch=12), W.llama8b_decode(2, batch=12, block_size=64)
    assert np.array_equal(a.context_lens, b.context_lens)
    assert b.block_size == 64 and b.max_blocks_per_seq == 64
    check_layout(b)


def test_mixed_batch_recipe():
    c = W.mixed_prefill_decode(0)
    ql, ctx = c.query_lens, c.context_lens
    pre, dec = ql > 1, ql == 1
    assert pre.sum() == 16 and dec.sum() == 48 and not c.is_decode
    assert np.all((ql[pre] >= 32) & (ql[pre] <= 512))
    assert np.all((ctx[pre] - ql[pre] >= 0) & (ctx[pre] - ql[pre] <= 2048))
    assert np.all((ctx[dec] >= 64) & (ctx[dec] <= 4096))
    # the tensor roofline's figures: 4,386 chunk tokens, 95.15 GFLOP over
    # (query row, visible key) pairs under the bottom-right causal mask
    q, k = ql[pre].astype(np.int64), ctx[pre].astype(np.int64)
    assert int(q.sum()) == 4386 and c.total_query_tokens == 4434
    pairs = int((q * (k - q) + q * (q + 1) // 2).sum())
    assert 4 * 32 * 128 * pairs == 95151603712
    # decode rows and chunks are interleaved, not sorted
    assert not np.all(np.diff(pre.astype(int)) <= 0) and not np.all(np.diff(pre.astype(int)) >= 0)


def test_mixed_batch_layout_small():
    c = W.mixed_prefill_decode(5, n_prefill=3, n_decode=5, q_range=(17, 70),
                               prior_range=(0, 90), dec_range=(1, 200))
    prior, new = check_layout(c)
    # a chunk's new tokens sit at its last positions and become finite once
    # written; nothing else changes
    k = c.k_cache.copy()
    Hkv, D, bs = c.num_kv_heads, c.head_dim, c.block_size
    kv = k.transpose(0, 2, 1, 3).reshape(-1, Hkv, D)
    kv[c.slot_mapping] = c.k_new
    all_nf, any_nf = _nonfinite_per_slot(kv.reshape(c.num_blocks, bs, Hkv, D).transpose(0, 2, 1, 3),
                                         c.dtype)
    assert not any_nf[prior | new].any() and all_nf[~(prior | new)].all()


def test_head_sweep_shapes():
    for hkv in (1, 8, 32):
        c = W.head_sweep(0, num_kv_heads=hkv, batch=4, ctx_len=100)
        assert c.num_heads == 32 and c.num_kv_heads == hkv and np.all(c.context_lens == 100)
        check_layout(c)


def test_long_context_outliers_are_one_percent_of_key_rows():
    c = W.long_context_decode(0, lo=1024, hi=2048)
    assert np.all((c.context_lens >= 1024) & (c.context_lens <= 2048))
    prior, _ = check_layout(c)
    k = W.bits_to_f32(c.k_cache, c.dtype)                 # [NB, Hkv, bs, D]
    rms = np.sqrt((k.astype(np.float64) ** 2).mean(axis=3)).transpose(0, 2, 1)
    rows = rms.reshape(-1, c.num_kv_heads)[prior]         # prior (slot, head) rows
    frac = float((rows > 4.0).mean())                     # x8 rows sit near 8, others near 1
    assert 0.007 <= frac <= 0.013, frac
    v = W.bits_to_f32(c.v_cache, c.dtype)
    vrms = np.sqrt((v.astype(np.float64) ** 2).mean(axis=3)).transpose(0, 2, 1)
    assert (vrms.reshape(-1, c.num_kv_heads)[prior] > 4.0).sum() == 0   # V untouched


def test_cross_attention_recipe():
    d = W.cross_attention_decode(0)
    assert d.cross and d.is_decode and d.num_seqs == 16
    assert np.all(d.context_lens % 1601 == 0)
    assert np.all((d.context_lens >= 1601) & (d.context_lens <= 4 * 1601))
    check_layout(d)
    p = W.cross_attention_prefill(0, batch=4)
    assert p.cross and np.all((p.query_lens >= 32) & (p.query_lens <= 512))
    assert np.any(p.query_lens > 1)
    check_layout(p)


def test_varlen_prompts():
    c = W.varlen_prefill_llama8b(0, batch=6, lo=5, hi=40)
    ql = np.diff(c.cu_q)
    assert np.array_equal(c.cu_q, c.cu_k) and np.all((ql >= 5) & (ql <= 40))
    assert c.q.shape == (c.cu_q[-1], 32, 128) and c.k.shape == (c.cu_k[-1], 8, 128)
    assert c.flops() == 4 * 32 * 128 * float((ql * (ql + 1) // 2).sum())


def test_seeded_and_reproducible():
    a, b, c = W.tiny_gqa_decode(7), W.tiny_gqa_decode(7), W.tiny_gqa_decode(8)
    for f in ("q", "k_cache", "v_cache", "k_new", "block_tables", "context_lens", "slot_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert not np.array_equal(a.q, c.q)


def test_values_are_standard_normal_rounded():
    c = W.head_sweep(0, num_kv_heads=8, batch=8, ctx_len=512)
    q = W.bits_to_f32(c.q, c.dtype).astype(np.float64)
    assert abs(q.mean()) < 0.01 and abs(q.std() - 1.0) < 0.01
    # each draw is an exact bf16 value (low 16 bits of the float32 are zero)
    assert np.all(W.bits_to_f32(c.q, c.dtype).view(np.uint32) & 0xFFFF == 0)
