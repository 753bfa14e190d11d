"""Pins for the fp64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: IEEE rounding as
implemented by numpy/torch, a dense brute-force loop written here, PyTorch's
float64 scaled_dot_product_attention, closed forms, hand-derived fixtures and
invariants of paged GQA attention.  A dropped term, a wrong head map, a wrong
causal offset or a transposed operand in the oracle fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# element conversion
# --------------------------------------------------------------------------

def test_from_bits_f16_all_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.from_bits(b, W.F16)
    ref = b.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_from_bits_bf16_all_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.from_bits(b, W.BF16)
    with np.errstate(invalid="ignore"):
        ref = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_to_bits_f16_matches_numpy():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24,
         2.0 ** -25, 3 * 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]])
    got = oracle.to_bits(x, W.F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)  # numpy rounds from double once
    assert np.array_equal(got, ref)


def test_to_bits_bf16_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)
         ).astype(np.float32)
    got = oracle.to_bits(x.astype(np.float64), W.BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_to_bits_bf16_rounds_once_from_double():
    # 1 + 2^-8 + 2^-30 lies above the bf16 midpoint 1 + 2^-8, so it rounds
    # up to 1 + 2^-7; going through float32 first would land on the midpoint
    # and round to even (1.0).
    x = np.array([1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8])
    got = oracle.from_bits(oracle.to_bits(x, W.BF16), W.BF16)
    assert got.tolist() == [1 + 2.0 ** -7, 1.0, 1 + 2.0 ** -6]


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def _small_case(seed=0, B=2, Hq=4, Hkv=2, D=8, bs=4, ctx=None, ql=None,
                dtype=W.BF16, num_blocks=None, **kw):
    rng = np.random.default_rng(seed)
    if ctx is None:
        ctx = rng.integers(1, 41, size=B)
    if ql is None:
        ql = np.ones(B, np.int64)
    return W.make_case("small", seed=seed, rng=rng, dtype=dtype, num_heads=Hq,
                       num_kv_heads=Hkv, head_dim=D, block_size=bs,
                       context_lens=ctx, query_lens=ql, num_blocks=num_blocks, **kw)


def _dense_sequence(case, kc, vc, b):
    """Sequence b's keys/values [ctx, Hkv, D] (fp64), read slot by slot."""
    bs = case.block_size
    ctx = int(case.context_lens[b])
    K = np.empty((ctx, case.num_kv_heads, case.head_dim))
    V = np.empty_like(K)
    for j in range(ctx):
        blk = case.block_tables[b, j // bs]
        K[j] = W.bits_to_f32(kc[blk, :, j % bs, :], case.dtype)
        V[j] = W.bits_to_f32(vc[blk, :, j % bs, :], case.dtype)
    return K, V


def _brute_force(case):
    """Dense loop: for every query row and head, softmax over visible keys,
    grouping heads by reshaping q to [Hkv, G, D] (no paging, no expand)."""
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    bs = case.block_size
    for t, s in enumerate(case.slot_mapping):
        kc[s // bs, :, s % bs] = case.k_new[t]
        vc[s // bs, :, s % bs] = case.v_new[t]
    Hq, Hkv, D = case.num_heads, case.num_kv_heads, case.head_dim
    G = Hq // Hkv
    q = W.bits_to_f32(case.q, case.dtype).astype(np.float64)
    out = np.zeros((case.total_query_tokens, Hq, D))
    for b in range(case.num_seqs):
        K, V = _dense_sequence(case, kc, vc, b)
        ctx = int(case.context_lens[b])
        c0, c1 = int(case.cu_query_lens[b]), int(case.cu_query_lens[b + 1])
        for tok in range(c0, c1):
            pos = ctx - (c1 - c0) + (tok - c0)
            qg = q[tok].reshape(Hkv, G, D)
            for kvh in range(Hkv):
                for g in range(G):
                    s = np.array([case.scale * float(np.dot(qg[kvh, g], K[j, kvh]))
                                  for j in range(pos + 1)])
                    w = np.exp(s - s.max())
                    out[tok, kvh * G + g] = (w[:, None] * V[:pos + 1, kvh]).sum(0) / w.sum()
    return out


# --------------------------------------------------------------------------
# attention pins
# --------------------------------------------------------------------------

def _golden(name, dtype=W.BF16):
    """A hand-derived fixture and its paged cache (one sequence, NaN in every
    slot past the context).  Every key, value and query in the fixtures is
    exact in fp16 and bf16 alike."""
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    Hkv, D, bs = g["num_kv_heads"], g["head_dim"], g["block_size"]
    bt = np.array([g["block_table"]], np.int32)
    kc = np.full((bt.shape[1], Hkv, bs, D), W.NAN_BITS[dtype], np.uint16)
    vc = kc.copy()
    keys = np.array(g["keys"], np.float32)      # [Hkv, ctx, D]
    vals = np.array(g["values"], np.float32)
    for j in range(g["context_len"]):
        blk = bt[0, j // bs]
        kc[blk, :, j % bs] = W.f32_to_bits(keys[:, j], dtype)
        vc[blk, :, j % bs] = W.f32_to_bits(vals[:, j], dtype)
    return g, kc, vc, bt


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
def test_golden_powers_of_two(dtype):
    g, kc, vc, bt = _golden("gqa_powers_of_two.json", dtype)
    q = W.f32_to_bits(np.array(g["queries"], np.float32)[None], dtype)
    o64, ob = oracle.paged_attention(q, kc, vc, bt, np.array([0, 1], np.int32),
                                     np.array([g["context_len"]], np.int32), math.log(2.0),
                                     g["num_kv_heads"], dtype)
    np.testing.assert_allclose(o64[0], np.array(g["expected"]), rtol=0, atol=1e-13)


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
def test_golden_cross_attention_unmasked(dtype):
    # hand-derived: four decoder rows over three encoder keys, no mask
    g, kc, vc, bt = _golden("cross_attention_unmasked.json", dtype)
    q = W.f32_to_bits(np.array(g["queries"], np.float32), dtype)
    assert q.shape == (g["query_len"], g["num_heads"], g["head_dim"])
    o64, ob = oracle.cross_attention(q, kc, vc, bt, np.array([0, g["query_len"]], np.int32),
                                     np.array([g["context_len"]], np.int32), math.log(2.0),
                                     g["num_kv_heads"], dtype)
    exact = np.array(g["expected"])
    np.testing.assert_allclose(o64, exact, rtol=0, atol=1e-13)
    assert np.array_equal(ob, W.f32_to_bits(exact.astype(np.float32), dtype))


@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
def test_golden_causal_chunk_bottom_right(dtype):
    # hand-derived: a two-token chunk after a one-token prefix; the expected
    # rows differ from those of a top-left mask (see the fixture's derivation)
    g, kc, vc, bt = _golden("causal_chunk_bottom_right.json", dtype)
    Hq, Hkv, D = g["num_heads"], g["num_kv_heads"], g["head_dim"]
    ctx, qlen = g["context_len"], g["query_len"]
    q = W.f32_to_bits(np.array(g["queries"], np.float32), dtype)   # [qlen, Hq, D]
    assert q.shape == (qlen, Hq, D)
    o64, ob = oracle.paged_attention(q, kc, vc, bt, np.array([0, qlen], np.int32),
                                     np.array([ctx], np.int32), math.log(2.0), Hkv, dtype)
    np.testing.assert_allclose(o64, np.array(g["expected"]), rtol=0, atol=1e-13)
    # every expected value but 4.2 and 16.8 is exact in the element type:
    # those round to themselves
    exact = np.array(g["expected"])
    ok = W.f32_to_bits(exact.astype(np.float32), dtype)
    same = (exact == W.bits_to_f32(ok, dtype))
    assert same.sum() == exact.size - 2
    assert np.array_equal(ob[same], ok[same])


def test_golden_causal_chunk_varlen_contiguous_kv():
    # the same hand-derived rows through the varlen definition: the three
    # keys as contiguous K/V of one sequence, its two query rows the chunk
    with open(os.path.join(GOLDEN, "causal_chunk_bottom_right.json")) as f:
        g = json.load(f)
    k = W.f32_to_bits(np.array(g["keys"], np.float32).transpose(1, 0, 2), W.BF16)  # [ctx, Hkv, D]
    v = W.f32_to_bits(np.array(g["values"], np.float32).transpose(1, 0, 2), W.BF16)
    q = W.f32_to_bits(np.array(g["queries"], np.float32), W.BF16)
    o64, _ = oracle.varlen_attention(q, k, v, np.array([0, g["query_len"]], np.int32),
                                     np.array([0, g["context_len"]], np.int32),
                                     math.log(2.0), W.BF16)
    np.testing.assert_allclose(o64, np.array(g["expected"]), rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("hq,hkv", [(4, 2), (6, 1), (3, 3), (8, 2)])
def test_brute_force_decode(seed, hq, hkv):
    c = _small_case(seed=seed, B=2, Hq=hq, Hkv=hkv, D=8, bs=4)
    o64, _, _, _ = oracle.run_case(c)
    np.testing.assert_allclose(o64, _brute_force(c), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_brute_force_chunked_prefill(seed):
    rng = np.random.default_rng(100 + seed)
    ctx = np.array([37, 5, 12, 20])
    ql = np.array([9, 5, 1, 0])
    c = _small_case(seed=seed, B=4, Hq=4, Hkv=2, D=8, bs=4, ctx=ctx, ql=ql)
    o64, _, _, _ = oracle.run_case(c)
    np.testing.assert_allclose(o64, _brute_force(c), rtol=0, atol=1e-12)


def test_g1_matches_torch_sdpa():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    c = _small_case(seed=3, B=3, Hq=4, Hkv=4, D=16, bs=8,
                    ctx=np.array([33, 8, 19]), ql=np.array([6, 8, 1]))
    o64, _, kc, vc = oracle.run_case(c)
    q = torch.from_numpy(W.bits_to_f32(c.q, c.dtype).astype(np.float64))
    for b in range(c.num_seqs):
        K, V = _dense_sequence(c, kc, vc, b)
        ctx = int(c.context_lens[b])
        c0, c1 = int(c.cu_query_lens[b]), int(c.cu_query_lens[b + 1])
        qb = q[c0:c1].permute(1, 0, 2)                 # [H, qlen, D]
        Kt = torch.from_numpy(K).permute(1, 0, 2)      # [H, ctx, D]
        Vt = torch.from_numpy(V).permute(1, 0, 2)
        qlen = c1 - c0
        # bottom-right causal mask: row t sees keys 0 .. ctx - qlen + t
        mask = torch.arange(ctx)[None, :] <= (ctx - qlen + torch.arange(qlen))[:, None]
        ref = F.scaled_dot_product_attention(qb, Kt, Vt, attn_mask=mask,
                                             scale=c.scale)
        np.testing.assert_allclose(o64[c0:c1], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def test_block_permutation_invariance_bitwise():
    c = _small_case(seed=5, B=3, Hq=8, Hkv=2, D=16, bs=4,
                    ctx=np.array([30, 17, 1]), ql=np.array([4, 1, 1]),
                    num_blocks=20)
    o1, b1, kc, vc = oracle.run_case(c)
    rng = np.random.default_rng(9)
    perm = rng.permutation(c.num_blocks)          # new id of old block i
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(c.block_tables >= 0, perm[np.maximum(c.block_tables, 0)], -1)
    o2, b2 = oracle.paged_attention(c.q, kc2, vc2, bt2, c.cu_query_lens,
                                    c.context_lens, c.scale, c.num_kv_heads,
                                    c.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(b1, b2)


@pytest.mark.parametrize("bs2", [1, 2, 8, 16])
def test_block_size_invariance_bitwise(bs2):
    """Re-paging the same sequences into blocks of another size, under a
    shuffled table, leaves the result bitwise unchanged: the block size only
    decides where key j of a sequence lives (block j // bs, slot j % bs).
    Unused slots of the new pool hold NaN, so a slot read in error shows."""
    c = _small_case(seed=11, B=3, Hq=8, Hkv=2, D=16, bs=4,
                    ctx=np.array([30, 17, 1]), ql=np.array([4, 1, 1]), num_blocks=20)
    o1, b1, kc, vc = oracle.run_case(c)
    bs = c.block_size
    nb2 = [(int(x) + bs2 - 1) // bs2 for x in c.context_lens]
    total = sum(nb2)
    ids = np.random.default_rng(12).permutation(total)
    nan_bits = np.uint16(0x7FC0)  # a bf16 quiet NaN
    shape = (total, c.num_kv_heads, bs2, c.head_dim)
    kc2 = np.full(shape, nan_bits, np.uint16)
    vc2 = np.full(shape, nan_bits, np.uint16)
    bt2 = np.full((c.num_seqs, max(nb2)), -1, np.int32)
    k = 0
    for b in range(c.num_seqs):
        bt2[b, :nb2[b]] = ids[k:k + nb2[b]]
        k += nb2[b]
        for j in range(int(c.context_lens[b])):
            src = c.block_tables[b, j // bs]
            kc2[bt2[b, j // bs2], :, j % bs2] = kc[src, :, j % bs]
            vc2[bt2[b, j // bs2], :, j % bs2] = vc[src, :, j % bs]
    o2, b2 = oracle.paged_attention(c.q, kc2, vc2, bt2, c.cu_query_lens, c.context_lens,
                                    c.scale, c.num_kv_heads, c.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(b1, b2)


def test_gqa_equals_mha_with_duplicated_kv_heads_bitwise():
    c = _small_case(seed=6, B=2, Hq=8, Hkv=2, D=16, bs=4,
                    ctx=np.array([21, 9]), ql=np.array([3, 1]))
    o_gqa, _, kc, vc = oracle.run_case(c)
    G = c.num_heads // c.num_kv_heads
    kc_m = np.repeat(kc, G, axis=1)   # KV head i -> heads i*G .. i*G+G-1
    vc_m = np.repeat(vc, G, axis=1)
    o_mha, _ = oracle.paged_attention(c.q, kc_m, vc_m, c.block_tables,
                                      c.cu_query_lens, c.context_lens, c.scale,
                                      c.num_heads, c.dtype)
    assert np.array_equal(o_gqa, o_mha)


def test_head_map_is_h_div_g_not_h_mod_hkv():
    # Two KV heads with constant, different V rows: head h must read KV head
    # h // G (heads 0,1 -> 0; heads 2,3 -> 1), which h % Hkv would not.
    c = _small_case(seed=7, B=1, Hq=4, Hkv=2, D=8, bs=4, ctx=np.array([6]))
    kc, vc = c.k_cache.copy(), c.v_cache.copy()
    vc[:, 0] = W.f32_to_bits(np.full(vc[:, 0].shape, 1.0, np.float32), c.dtype)
    vc[:, 1] = W.f32_to_bits(np.full(vc[:, 1].shape, -2.0, np.float32), c.dtype)
    vn = c.v_new.copy()
    vn[:, 0] = W.f32_to_bits(np.full(vn[:, 0].shape, 1.0, np.float32), c.dtype)
    vn[:, 1] = W.f32_to_bits(np.full(vn[:, 1].shape, -2.0, np.float32), c.dtype)
    oracle.reshape_and_cache(c.k_new, vn, kc, vc, c.slot_mapping)
    o, _ = oracle.paged_attention(c.q, kc, vc, c.block_tables, c.cu_query_lens,
                                  c.context_lens, c.scale, 2, c.dtype)
    np.testing.assert_allclose(o[0, :, 0], [1.0, 1.0, -2.0, -2.0], atol=1e-15)


def test_identical_keys_give_mean_of_values():
    c = _small_case(seed=8, B=2, Hq=4, Hkv=1, D=8, bs=4, ctx=np.array([13, 7]))
    kc, vc = c.k_cache.copy(), c.v_cache.copy()
    row = W.f32_to_bits(np.linspace(-1, 1, 8).astype(np.float32), c.dtype)
    kc[...] = row
    kn = np.broadcast_to(row, c.k_new.shape).copy()
    oracle.reshape_and_cache(kn, c.v_new, kc, vc, c.slot_mapping)
    o, _ = oracle.paged_attention(c.q, kc, vc, c.block_tables, c.cu_query_lens,
                                  c.context_lens, c.scale, 1, c.dtype)
    for b in range(2):
        _, V = _dense_sequence(c, kc, vc, b)
        np.testing.assert_allclose(o[b], np.broadcast_to(V[:, 0].mean(0), (4, 8)),
                                   rtol=0, atol=1e-14)


def test_one_token_context_returns_that_value_row():
    c = _small_case(seed=9, B=3, Hq=6, Hkv=3, D=8, bs=4, ctx=np.array([1, 1, 1]))
    o, ob, kc, vc = oracle.run_case(c)
    G = 2
    for b in range(3):
        v = W.bits_to_f32(c.v_new[b], c.dtype)  # [Hkv, D]
        for h in range(6):
            assert np.array_equal(o[b, h], v[h // G].astype(np.float64))
            assert np.array_equal(ob[b, h], c.v_new[b, h // G])


def test_chunk_equals_successive_decode_steps_bitwise():
    c = _small_case(seed=10, B=1, Hq=4, Hkv=2, D=8, bs=4, ctx=np.array([19]),
                    ql=np.array([7]))
    o_chunk, _, kc, vc = oracle.run_case(c)
    for t in range(7):
        ctx_t = np.array([19 - 7 + t + 1], np.int32)
        o_t, _ = oracle.paged_attention(c.q[t:t + 1], kc, vc, c.block_tables,
                                        np.array([0, 1], np.int32), ctx_t,
                                        c.scale, 2, c.dtype)
        assert np.array_equal(o_t[0], o_chunk[t])


@pytest.mark.parametrize("S", [2, 3, 5, 16])
def test_split_combine_identity(S):
    c = _small_case(seed=11, B=3, Hq=4, Hkv=2, D=8, bs=4,
                    ctx=np.array([40, 9, 3]), ql=np.array([1, 3, 1]))
    kc, vc = c.k_cache.copy(), c.v_cache.copy()
    oracle.reshape_and_cache(c.k_new, c.v_new, kc, vc, c.slot_mapping)
    o, _, po, pl = oracle.paged_attention(c.q, kc, vc, c.block_tables,
                                          c.cu_query_lens, c.context_lens,
                                          c.scale, 2, c.dtype, num_splits=S,
                                          want_partials=True)
    np.testing.assert_allclose(oracle.lse_combine(po, pl), o, rtol=0, atol=1e-12)
    # split 0 always holds key 0; splits past the sequence are empty
    assert np.all(np.isfinite(pl[..., 0]))
    if S == 16:
        assert np.any(np.isneginf(pl))


def test_lse_combine_hand_values():
    # Split weights are e^(lse_s - max): lse 0 and ln 3 weigh 1 : 3, so
    # partials (4, 0) and (0, 4) merge to (1, 3); an empty split (lse -inf)
    # weighs nothing, whatever its partial holds; a common shift of every
    # lse changes nothing (here 1000, past exp's range without the max);
    # all splits empty gives zeros.
    inf = float("inf")
    po = np.array([[[4.0, 0.0], [0.0, 4.0], [1e9, -1e9]],
                   [[4.0, 0.0], [0.0, 4.0], [7.0, 7.0]],
                   [[5.0, 5.0], [6.0, 6.0], [7.0, 7.0]]])
    pl = np.array([[0.0, math.log(3.0), -inf],
                   [1000.0, 1000.0 + math.log(3.0), -inf],
                   [-inf, -inf, -inf]])
    out = oracle.lse_combine(po, pl)
    np.testing.assert_allclose(out, [[1.0, 3.0], [1.0, 3.0], [0.0, 0.0]], rtol=0, atol=1e-12)


def test_split_lse_closed_form():
    # one key per split: lse of split s is exactly its scaled logit
    c = _small_case(seed=12, B=1, Hq=2, Hkv=1, D=8, bs=4, ctx=np.array([8]))
    kc, vc = c.k_cache.copy(), c.v_cache.copy()
    oracle.reshape_and_cache(c.k_new, c.v_new, kc, vc, c.slot_mapping)
    _, _, po, pl = oracle.paged_attention(c.q, kc, vc, c.block_tables,
                                          c.cu_query_lens, c.context_lens,
                                          c.scale, 1, c.dtype, num_splits=2,
                                          want_partials=True)
    K, V = _dense_sequence(c, kc, vc, 0)
    q = W.bits_to_f32(c.q[0], c.dtype).astype(np.float64)
    for h in range(2):
        for s in range(2):
            logits = c.scale * K[4 * s:4 * s + 4, 0] @ q[h]
            m = logits.max()
            assert abs(pl[0, h, s] - (m + math.log(np.exp(logits - m).sum()))) < 1e-12


def test_garbage_past_context_is_never_read():
    c = _small_case(seed=13, B=2, Hq=4, Hkv=2, D=8, bs=8, ctx=np.array([5, 11]),
                    num_blocks=6)
    o1, b1, kc, vc = oracle.run_case(c)
    # overwrite every slot that holds no token with other garbage
    valid = np.zeros((c.num_blocks, c.block_size), bool)
    for b in range(2):
        for j in range(int(c.context_lens[b])):
            valid[c.block_tables[b, j // 8], j % 8] = True
    kc2, vc2 = kc.copy(), vc.copy()
    kc2.transpose(0, 2, 1, 3)[~valid] = 0x7F80   # +inf
    vc2.transpose(0, 2, 1, 3)[~valid] = 0x4B00   # large finite
    o2, b2 = oracle.paged_attention(c.q, kc2, vc2, c.block_tables,
                                    c.cu_query_lens, c.context_lens, c.scale,
                                    2, c.dtype)
    assert np.array_equal(o1, o2)


def test_empty_context_and_empty_query():
    c = _small_case(seed=14, B=3, Hq=4, Hkv=2, D=8, bs=4,
                    ctx=np.array([0, 6, 4]), ql=np.array([0, 2, 0]))
    o, ob, _, _ = oracle.run_case(c)
    assert o.shape == (2, 4, 8)  # only the two query tokens of sequence 1
    np.testing.assert_allclose(o, _brute_force(c), atol=1e-12)


def test_decode_row_without_keys_is_zero():
    c = _small_case(seed=17, B=2, Hq=4, Hkv=2, D=8, bs=4, ctx=np.array([5, 3]))
    kc, vc = c.k_cache.copy(), c.v_cache.copy()
    oracle.reshape_and_cache(c.k_new, c.v_new, kc, vc, c.slot_mapping)
    ctx = c.context_lens.copy()
    ctx[0] = 0
    o, ob = oracle.paged_attention(c.q, kc, vc, c.block_tables, c.cu_query_lens, ctx,
                                   c.scale, 2, c.dtype)
    assert not o[0].any() and not ob[0].any()
    o_ref, _ = oracle.paged_attention(c.q, kc, vc, c.block_tables, c.cu_query_lens,
                                      c.context_lens, c.scale, 2, c.dtype)
    assert np.array_equal(o[1], o_ref[1])
    # a query chunk longer than a non-empty context is still an error
    ctx[0] = 1
    cu = np.array([0, 2, 3], np.int32)
    q2 = np.concatenate([c.q[:1], c.q], 0)
    with pytest.raises(ValueError):
        oracle.paged_attention(q2, kc, vc, c.block_tables, cu, ctx, c.scale, 2, c.dtype)


def test_bad_block_id_is_an_error():
    c = _small_case(seed=15, B=1, Hq=2, Hkv=1, D=8, bs=4, ctx=np.array([6]))
    bt = c.block_tables.copy()
    bt[0, 1] = c.num_blocks
    with pytest.raises(ValueError):
        oracle.paged_attention(c.q, c.k_cache, c.v_cache, bt, c.cu_query_lens,
                               c.context_lens, c.scale, 1, c.dtype)


# --------------------------------------------------------------------------
# reshape_and_cache
# --------------------------------------------------------------------------

def test_reshape_and_cache_is_the_slot_copy():
    rng = np.random.default_rng(16)
    NB, Hkv, bs, D, T = 7, 3, 4, 8, 11
    kc = rng.integers(0, 65536, (NB, Hkv, bs, D)).astype(np.uint16)
    vc = rng.integers(0, 65536, (NB, Hkv, bs, D)).astype(np.uint16)
    k = rng.integers(0, 65536, (T, Hkv, D)).astype(np.uint16)
    v = rng.integers(0, 65536, (T, Hkv, D)).astype(np.uint16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[[2, 7]] = -1
    kc2, vc2 = kc.copy(), vc.copy()
    oracle.reshape_and_cache(k, v, kc2, vc2, slots)
    keep = slots >= 0
    # slot-major copies of the caches: [NB * bs, Hkv, D]
    kref = kc.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D).copy()
    vref = vc.transpose(0, 2, 1, 3).reshape(NB * bs, Hkv, D).copy()
    kref[slots[keep]] = k[keep]
    vref[slots[keep]] = v[keep]
    kref = kref.reshape(NB, bs, Hkv, D).transpose(0, 2, 1, 3)
    vref = vref.reshape(NB, bs, Hkv, D).transpose(0, 2, 1, 3)
    assert np.array_equal(kc2, kref) and np.array_equal(vc2, vref)


def test_reshape_and_cache_rejects_out_of_range_slot():
    kc = np.zeros((2, 1, 4, 8), np.uint16)
    vc = kc.copy()
    k = np.ones((1, 1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(k, k, kc, vc, np.array([8], np.int64))
    assert not kc.any()


# --------------------------------------------------------------------------
# workloads: the recipe the inputs follow
# --------------------------------------------------------------------------

def test_workload_tiny_layout():
    c = W.tiny_gqa_decode(0)
    assert c.num_blocks == 64 and c.max_blocks_per_seq == 16
    assert c.q.shape == (4, 8, 64)
    used = c.block_tables[c.block_tables >= 0]
    assert len(np.unique(used)) == len(used)
    assert np.all((c.context_lens >= 1) & (c.context_lens <= 256))


def test_workload_mixed_layout():
    c = W.mixed_prefill_decode(0)
    ql = c.query_lens
    assert (ql == 1).sum() == 48 and ((ql >= 32) & (ql <= 512)).sum() == 16
    assert np.all(c.context_lens >= ql)


# --------------------------------------------------------------------------
# cross-attention (static encoder cache, no causal mask)
# --------------------------------------------------------------------------

def _small_cross(seed=0, B=3, Hq=4, Hkv=2, D=8, bs=4, enc=None, ql=None, dtype=W.BF16):
    rng = np.random.default_rng(seed)
    if enc is None:
        enc = rng.integers(1, 30, size=B)
    if ql is None:
        ql = rng.integers(1, 12, size=B)
    return W.make_cross_case("cross", seed=seed, rng=rng, dtype=dtype, num_heads=Hq,
                             num_kv_heads=Hkv, head_dim=D, block_size=bs,
                             encoder_lens=enc, query_lens=ql)


def test_cross_brute_force_dense_loop():
    # includes a sequence with more query rows than encoder tokens
    c = _small_cross(seed=5, B=3, Hq=6, Hkv=2, enc=np.array([17, 3, 25]),
                     ql=np.array([4, 9, 1]))
    o64, _, kc, vc = oracle.run_case(c)
    Hq, Hkv, D = c.num_heads, c.num_kv_heads, c.head_dim
    G = Hq // Hkv
    q = W.bits_to_f32(c.q, c.dtype).astype(np.float64)
    for b in range(c.num_seqs):
        K, V = _dense_sequence(c, kc, vc, b)
        for tok in range(int(c.cu_query_lens[b]), int(c.cu_query_lens[b + 1])):
            qg = q[tok].reshape(Hkv, G, D)
            for kvh in range(Hkv):
                for g in range(G):
                    s = c.scale * (K[:, kvh] @ qg[kvh, g])       # every key
                    w = np.exp(s - s.max())
                    ref = (w[:, None] * V[:, kvh]).sum(0) / w.sum()
                    np.testing.assert_allclose(o64[tok, kvh * G + g], ref, rtol=0, atol=1e-12)


def test_cross_equals_one_decode_row_per_query_token_bitwise():
    # Without a causal mask, each query row is a decode row (qlen 1, all
    # keys) over its sequence's cache: the decode definition, pinned above.
    c = _small_cross(seed=6, B=3)
    o_cross, _, kc, vc = oracle.run_case(c)
    ql = np.diff(c.cu_query_lens)
    seq = np.repeat(np.arange(c.num_seqs), ql)
    bt = c.block_tables[seq]
    ctx = c.context_lens[seq]
    cu = np.arange(len(seq) + 1, dtype=np.int32)
    o_dec, _ = oracle.paged_attention(c.q, kc, vc, bt, cu, ctx, c.scale,
                                      c.num_kv_heads, c.dtype)
    assert np.array_equal(o_cross, o_dec)


def test_cross_g1_matches_torch_sdpa_without_mask():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    c = _small_cross(seed=7, B=3, Hq=4, Hkv=4, D=16, bs=8,
                     enc=np.array([33, 6, 19]), ql=np.array([5, 11, 1]))
    o64, _, kc, vc = oracle.run_case(c)
    q = torch.from_numpy(W.bits_to_f32(c.q, c.dtype).astype(np.float64))
    for b in range(c.num_seqs):
        K, V = _dense_sequence(c, kc, vc, b)
        c0, c1 = int(c.cu_query_lens[b]), int(c.cu_query_lens[b + 1])
        ref = F.scaled_dot_product_attention(
            q[c0:c1].permute(1, 0, 2), torch.from_numpy(K).permute(1, 0, 2),
            torch.from_numpy(V).permute(1, 0, 2), scale=c.scale)
        np.testing.assert_allclose(o64[c0:c1], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def test_cross_query_order_is_irrelevant_bitwise():
    c = _small_cross(seed=8, B=2, ql=np.array([7, 5]))
    o64, _, kc, vc = oracle.run_case(c)
    perm = np.concatenate([np.random.default_rng(1).permutation(7),
                           7 + np.random.default_rng(2).permutation(5)])
    o_perm, _ = oracle.cross_attention(c.q[perm], kc, vc, c.block_tables,
                                       c.cu_query_lens, c.context_lens, c.scale,
                                       c.num_kv_heads, c.dtype)
    assert np.array_equal(o_perm, o64[perm])


def test_cross_empty_encoder_gives_zero_rows_and_reads_nothing():
    c = _small_cross(seed=9, B=3, enc=np.array([0, 12, 0]), ql=np.array([3, 2, 4]))
    o64, ob, _, _ = oracle.run_case(c)
    for b in (0, 2):
        c0, c1 = int(c.cu_query_lens[b]), int(c.cu_query_lens[b + 1])
        assert np.all(o64[c0:c1] == 0) and np.all(ob[c0:c1] == 0)
    assert np.all(np.isfinite(o64))


def test_cross_workload_layout():
    c = W.cross_attention_decode(0)
    assert c.cross and c.is_decode and c.slot_mapping.size == 0
    assert set(np.unique(c.context_lens)) <= {1601, 3202, 4803, 6404}
    p = W.cross_attention_prefill(0)
    assert p.cross and not p.is_decode
    assert np.all(np.diff(p.cu_query_lens) >= 32) and np.all(np.diff(p.cu_query_lens) <= 512)
    # every slot that holds no encoder token is NaN
    nb = (p.context_lens.astype(np.int64) + p.block_size - 1) // p.block_size
    used = np.zeros(p.num_blocks, bool)
    for b in range(p.num_seqs):
        used[p.block_tables[b, :nb[b]]] = True
    assert np.all(W.bits_to_f32(p.k_cache[~used], p.dtype) != W.bits_to_f32(p.k_cache[~used], p.dtype))


# --------------------------------------------------------------------------
# GQA prefill over contiguous varlen K/V (no cache)
# --------------------------------------------------------------------------

def _varlen(seed=0, Hq=4, Hkv=2, D=8, ql=(5, 1, 9), kl=None, dtype=W.BF16):
    return W.make_varlen_case("varlen", seed=seed, dtype=dtype, num_heads=Hq,
                              num_kv_heads=Hkv, head_dim=D, q_lens=ql, k_lens=kl)


def test_varlen_literal_expand_then_mha():
    # the issue's prefill: k[:, :, None, :].expand(T, Hkv, G, D) flattened to
    # [T, Hq, D], then causal multi-head attention per sequence
    c = _varlen(seed=1, Hq=6, Hkv=2, ql=(7, 3, 1), kl=(7, 8, 4))
    o64, _ = oracle.varlen_attention(c.q, c.k, c.v, c.cu_q, c.cu_k, c.scale, c.dtype)
    G = c.num_heads // c.num_kv_heads
    q = W.bits_to_f32(c.q, c.dtype).astype(np.float64)
    k = W.bits_to_f32(c.k, c.dtype).astype(np.float64)
    v = W.bits_to_f32(c.v, c.dtype).astype(np.float64)
    ke = np.broadcast_to(k[:, :, None, :], (k.shape[0], c.num_kv_heads, G, c.head_dim))
    ve = np.broadcast_to(v[:, :, None, :], ke.shape)
    ke = ke.reshape(k.shape[0], c.num_heads, c.head_dim)
    ve = ve.reshape(k.shape[0], c.num_heads, c.head_dim)
    for b in range(c.num_seqs):
        q0, q1 = int(c.cu_q[b]), int(c.cu_q[b + 1])
        k0, k1 = int(c.cu_k[b]), int(c.cu_k[b + 1])
        for t in range(q1 - q0):
            p = (k1 - k0) - (q1 - q0) + t
            for h in range(c.num_heads):
                s = c.scale * (ke[k0:k0 + p + 1, h] @ q[q0 + t, h])
                w = np.exp(s - s.max())
                ref = (w[:, None] * ve[k0:k0 + p + 1, h]).sum(0) / w.sum()
                np.testing.assert_allclose(o64[q0 + t, h], ref, rtol=0, atol=1e-12)


def test_varlen_equals_paged_oracle_on_the_same_rows_bitwise():
    # K/V laid into a paged cache (block 4, blocks in a shuffled order) give
    # the same numbers through the paged definition
    c = _varlen(seed=2, Hq=4, Hkv=2, ql=(6, 2, 11), kl=(9, 2, 14))
    o_var, _ = oracle.varlen_attention(c.q, c.k, c.v, c.cu_q, c.cu_k, c.scale, c.dtype)
    bs = 4
    kl = np.diff(c.cu_k)
    nb = (kl + bs - 1) // bs
    NB = int(nb.sum())
    perm = np.random.default_rng(3).permutation(NB).astype(np.int32)
    bt = np.full((c.num_seqs, int(nb.max())), -1, np.int32)
    kc = np.full((NB, c.num_kv_heads, bs, c.head_dim), W.NAN_BITS[c.dtype], np.uint16)
    vc = kc.copy()
    off = 0
    for b in range(c.num_seqs):
        bt[b, :nb[b]] = perm[off:off + nb[b]]
        off += nb[b]
        for j in range(kl[b]):
            kc[bt[b, j // bs], :, j % bs] = c.k[c.cu_k[b] + j]
            vc[bt[b, j // bs], :, j % bs] = c.v[c.cu_k[b] + j]
    o_pag, _ = oracle.paged_attention(c.q, kc, vc, bt, c.cu_q, kl.astype(np.int32), c.scale,
                                      c.num_kv_heads, c.dtype)
    assert np.array_equal(o_var, o_pag)


def test_varlen_g1_matches_torch_sdpa_causal():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    c = _varlen(seed=4, Hq=4, Hkv=4, D=16, ql=(12, 5), kl=(12, 9))
    o64, _ = oracle.varlen_attention(c.q, c.k, c.v, c.cu_q, c.cu_k, c.scale, c.dtype)
    q = torch.from_numpy(W.bits_to_f32(c.q, c.dtype).astype(np.float64))
    k = torch.from_numpy(W.bits_to_f32(c.k, c.dtype).astype(np.float64))
    v = torch.from_numpy(W.bits_to_f32(c.v, c.dtype).astype(np.float64))
    for b in range(c.num_seqs):
        q0, q1 = int(c.cu_q[b]), int(c.cu_q[b + 1])
        k0, k1 = int(c.cu_k[b]), int(c.cu_k[b + 1])
        qlen, klen = q1 - q0, k1 - k0
        mask = torch.arange(klen)[None, :] <= (klen - qlen + torch.arange(qlen))[:, None]
        ref = F.scaled_dot_product_attention(q[q0:q1].permute(1, 0, 2),
                                             k[k0:k1].permute(1, 0, 2),
                                             v[k0:k1].permute(1, 0, 2), attn_mask=mask,
                                             scale=c.scale)
        np.testing.assert_allclose(o64[q0:q1], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_varlen_sequences_are_independent_bitwise():
    c = _varlen(seed=5, ql=(4, 7, 2), kl=(6, 7, 5))
    o64, _ = oracle.varlen_attention(c.q, c.k, c.v, c.cu_q, c.cu_k, c.scale, c.dtype)
    order = [2, 0, 1]
    ql, kl = np.diff(c.cu_q), np.diff(c.cu_k)
    qs = np.concatenate([c.q[c.cu_q[b]:c.cu_q[b + 1]] for b in order])
    ks = np.concatenate([c.k[c.cu_k[b]:c.cu_k[b + 1]] for b in order])
    vs = np.concatenate([c.v[c.cu_k[b]:c.cu_k[b + 1]] for b in order])
    cq = np.concatenate([[0], np.cumsum(ql[order])]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kl[order])]).astype(np.int32)
    o2, _ = oracle.varlen_attention(qs, ks, vs, cq, ck, c.scale, c.dtype)
    ref = np.concatenate([o64[c.cu_q[b]:c.cu_q[b + 1]] for b in order])
    assert np.array_equal(o2, ref)


def test_varlen_rejects_fewer_keys_than_queries():
    c = _varlen(seed=6, ql=(3,), kl=(3,))
    with pytest.raises(ValueError):
        oracle.varlen_attention(c.q, c.k[:2], c.v[:2], c.cu_q, np.array([0, 2], np.int32),
                                c.scale, c.dtype)
