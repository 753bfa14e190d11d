"""Seeded synthetic inputs for paged-KV GQA/MQA attention.

This module only draws inputs.  It holds none of the attention arithmetic:
both the CPU oracle and the CUDA path are fed the arrays built here, so that
neither side ever produces the other's inputs.

What is generated, per case (all numpy, host memory):

* ``q``            [Tq, Hq, D]      uint16 bit patterns of fp16 / bf16
* ``k_cache``      [NB, Hkv, bs, D] uint16 bits; every slot that holds no token
                                    of the prior context is NaN (unused blocks,
                                    the tail of each sequence's last block and
                                    the slots this step's new tokens go to)
* ``v_cache``      same as k_cache
* ``k_new, v_new`` [Tq, Hkv, D]     uint16 bits: K/V rows of this step's query
                                    tokens, written into the cache by
                                    reshape_and_cache before attention runs
* ``slot_mapping`` [Tq] int64       cache slot (block_id * bs + offset) of each
                                    new token
* ``block_tables`` [B, MBS] int32   physical block ids, padded with -1
* ``context_lens`` [B] int32        tokens in the cache per sequence, including
                                    this step's query tokens
* ``cu_query_lens``[B+1] int32      prefix sums of the query-token counts

Recipe (seeded with ``numpy.random.default_rng(seed)``):

* values: float32 draws from N(0, 1), rounded to nearest-even into the
  element type;
* physical blocks: a random permutation of all NB block ids, handed out to the
  sequences in order; NB = sum of the blocks the sequences need, plus 5% spare
  (NaN-filled) blocks, except where a case fixes NB;
* optional key outliers: each (token, kv head) K row is multiplied by a power
  of two (exact in bf16/fp16) with a given probability.

The named configurations restate the workloads of the paged GQA/MQA decode and
chunked-prefill benchmarks: a tiny fp16 decode, a Llama-3.1-8B-shaped decode
with lognormal context lengths, a mixed chunked-prefill + decode batch, an
MQA/GQA/MHA sweep at fixed query-head count, and a long-context decode that
needs split-KV.  The pages' own benchmarks ran ShareGPT traffic through trained
Llama models; these synthetic inputs stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

F16 = 0
BF16 = 1
DTYPE_NAMES = {F16: "f16", BF16: "bf16"}
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}


def f32_to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 samples to nearest-even fp16/bf16; returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if not np.all(np.isfinite(x)):
        raise ValueError("only finite samples are rounded here")
    # finite float32 bit patterns are < 0xFF800000, so the sum cannot wrap
    u = x.view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(b: np.ndarray, dtype: int) -> np.ndarray:
    """uint16 bit patterns -> float32 (exact for both element types)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    if dtype == F16:
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bits(rng: np.random.Generator, shape, dtype: int,
                 chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) float32 draws rounded into the element type, drawn in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bits(rng.standard_normal(e - s, dtype=np.float32), dtype)
    return out.reshape(shape)


@dataclasses.dataclass
class Case:
    name: str
    dtype: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    slot_mapping: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    cu_query_lens: np.ndarray
    is_decode: bool
    num_splits: int = 0
    cross: bool = False  # static encoder cache, no causal mask, no new K/V

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.cu_query_lens)

    @property
    def total_query_tokens(self) -> int:
        return int(self.cu_query_lens[-1])

    @property
    def max_query_len(self) -> int:
        ql = self.query_lens
        return int(ql.max()) if ql.size else 0

    @property
    def elem_bytes(self) -> int:
        return 2

    def kv_bytes(self) -> int:
        """Algorithmic KV-cache bytes one attention pass reads: every context
        token's K and V row, once per KV head."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads \
            * self.head_dim * 2 * self.elem_bytes

    def kv_bytes_block_granular(self) -> int:
        nb = (self.context_lens.astype(np.int64) + self.block_size - 1) // self.block_size
        return int(nb.sum()) * self.block_size * self.num_kv_heads * self.head_dim \
            * 2 * self.elem_bytes


def make_case(name: str, *, seed: int, dtype: int, num_heads: int,
              num_kv_heads: int, head_dim: int, block_size: int,
              context_lens, query_lens, scale: Optional[float] = None,
              num_blocks: Optional[int] = None, spare_frac: float = 0.05,
              max_blocks_per_seq: Optional[int] = None,
              key_outlier_prob: float = 0.0, key_outlier_mult: float = 8.0,
              is_decode: Optional[bool] = None, num_splits: int = 0,
              rng: Optional[np.random.Generator] = None) -> Case:
    """Build one case from explicit per-sequence context and query lengths.

    ``context_lens[b]`` counts every token of sequence b in the cache after
    this step, including its ``query_lens[b]`` new tokens (which occupy the
    last positions of the sequence).
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    B = ctx.shape[0]
    assert ql.shape == (B,)
    assert np.all(ql <= ctx) and np.all(ql >= 0)
    bs = block_size
    nb = (ctx + bs - 1) // bs
    need = int(nb.sum())
    if num_blocks is None:
        num_blocks = need + int(math.ceil(spare_frac * need))
    assert num_blocks >= need, (num_blocks, need)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, int(nb.max()) if B else 1)
    assert max_blocks_per_seq >= (int(nb.max()) if B else 0)
    NB = num_blocks
    Hkv, D = num_kv_heads, head_dim
    if scale is None:
        scale = 1.0 / math.sqrt(D)

    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((B, max_blocks_per_seq), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[off:off + nb[b]]
        off += nb[b]

    # Fill the pool with draws, then NaN every slot that holds no prior token.
    k_cache = _normal_bits(rng, (NB, Hkv, bs, D), dtype)
    v_cache = _normal_bits(rng, (NB, Hkv, bs, D), dtype)
    valid = np.zeros((NB, bs), dtype=bool)
    Tq = int(ql.sum())
    slot = np.empty(Tq, dtype=np.int64)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    for b in range(B):
        prior = int(ctx[b] - ql[b])
        blocks = bt[b, :nb[b]].astype(np.int64)
        pos = np.arange(ctx[b], dtype=np.int64)
        slots_b = blocks[pos // bs] * bs + pos % bs
        valid.reshape(-1)[slots_b[:prior]] = True
        slot[cu[b]:cu[b + 1]] = slots_b[prior:]
    nan = np.uint16(NAN_BITS[dtype])
    inv = ~valid
    k_cache.transpose(0, 2, 1, 3)[inv] = nan
    v_cache.transpose(0, 2, 1, 3)[inv] = nan

    q = _normal_bits(rng, (Tq, num_heads, D), dtype)
    k_new = _normal_bits(rng, (Tq, Hkv, D), dtype)
    v_new = _normal_bits(rng, (Tq, Hkv, D), dtype)

    if key_outlier_prob > 0.0:
        mult = np.float32(key_outlier_mult)
        sel = rng.random((NB, Hkv, bs)) < key_outlier_prob
        sel &= valid[:, None, :]
        kc = k_cache[sel]
        k_cache[sel] = f32_to_bits(bits_to_f32(kc, dtype) * mult, dtype)
        seln = rng.random((Tq, Hkv)) < key_outlier_prob
        kn = k_new[seln]
        k_new[seln] = f32_to_bits(bits_to_f32(kn, dtype) * mult, dtype)

    if is_decode is None:
        is_decode = bool(np.all(ql == 1))
    return Case(name=name, dtype=dtype, num_heads=num_heads, num_kv_heads=Hkv,
                head_dim=D, block_size=bs, scale=float(scale), q=q,
                k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
                slot_mapping=slot, block_tables=bt,
                context_lens=ctx.astype(np.int32), cu_query_lens=cu,
                is_decode=is_decode, num_splits=num_splits)


def make_cross_case(name: str, *, seed: int, dtype: int, num_heads: int,
                    num_kv_heads: int, head_dim: int, block_size: int,
                    encoder_lens, query_lens, scale: Optional[float] = None,
                    spare_frac: float = 0.05, max_blocks_per_seq: Optional[int] = None,
                    rng: Optional[np.random.Generator] = None) -> Case:
    """A cross-attention step: every sequence's encoder keys and values
    (``encoder_lens[b]`` tokens) already sit in the paged cache and stay
    there; the step adds ``query_lens[b]`` decoder query rows (any number,
    also more than the encoder tokens) and writes no K/V.  Unused blocks and
    last-block tails are NaN, as in make_case."""
    if rng is None:
        rng = np.random.default_rng(seed)
    ctx = np.asarray(encoder_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    B = ctx.shape[0]
    assert ql.shape == (B,) and np.all(ql >= 0) and np.all(ctx >= 0)
    bs = block_size
    nb = (ctx + bs - 1) // bs
    need = int(nb.sum())
    NB = max(1, need + int(math.ceil(spare_frac * need)))
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, int(nb.max()) if B else 1)
    Hkv, D = num_kv_heads, head_dim
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((B, max_blocks_per_seq), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[off:off + nb[b]]
        off += nb[b]
    k_cache = _normal_bits(rng, (NB, Hkv, bs, D), dtype)
    v_cache = _normal_bits(rng, (NB, Hkv, bs, D), dtype)
    valid = np.zeros((NB, bs), dtype=bool)
    for b in range(B):
        blocks = bt[b, :nb[b]].astype(np.int64)
        pos = np.arange(ctx[b], dtype=np.int64)
        valid.reshape(-1)[blocks[pos // bs] * bs + pos % bs] = True
    nan = np.uint16(NAN_BITS[dtype])
    k_cache.transpose(0, 2, 1, 3)[~valid] = nan
    v_cache.transpose(0, 2, 1, 3)[~valid] = nan
    Tq = int(ql.sum())
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    q = _normal_bits(rng, (Tq, num_heads, D), dtype)
    empty = np.zeros((0, Hkv, D), np.uint16)
    return Case(name=name, dtype=dtype, num_heads=num_heads, num_kv_heads=Hkv,
                head_dim=D, block_size=bs, scale=float(scale), q=q,
                k_cache=k_cache, v_cache=v_cache, k_new=empty, v_new=empty.copy(),
                slot_mapping=np.zeros(0, np.int64), block_tables=bt,
                context_lens=ctx.astype(np.int32), cu_query_lens=cu,
                is_decode=bool(np.all(ql == 1)), cross=True)


# --------------------------------------------------------------------------
# Named workloads
# --------------------------------------------------------------------------

def tiny_gqa_decode(seed: int = 0) -> Case:
    """Batch 4, 8 query / 2 KV heads, head_dim 64, fp16, block 16, context
    lengths uniform in [1, 256], exactly 64 physical blocks."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, 257, size=4)
    return make_case("tiny_gqa_decode", seed=seed, rng=rng, dtype=F16,
                     num_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                     context_lens=ctx, query_lens=np.ones(4, np.int64),
                     scale=1.0 / 8.0, num_blocks=64, max_blocks_per_seq=16)


def _suffix(block_size: int) -> str:
    return "" if block_size == 16 else f"_bs{block_size}"


def llama8b_decode(seed: int = 0, batch: int = 256, max_ctx: int = 4096,
                   sigma: float = 1.0, block_size: int = 16) -> Case:
    """Llama-3.1-8B-shaped decode: 32 query / 8 KV heads, head_dim 128, bf16,
    block 16 (or block_size), context lengths lognormal (median 400,
    sigma 1.0) clipped to [16, 4096].  The lengths depend on the seed only,
    not on the block size."""
    rng = np.random.default_rng(seed)
    ctx = np.exp(rng.normal(math.log(400.0), sigma, size=batch))
    ctx = np.clip(np.rint(ctx), 16, max_ctx).astype(np.int64)
    name = "llama8b_decode" if batch == 256 else f"llama8b_decode_b{batch}"
    return make_case(name + _suffix(block_size),
                     seed=seed, rng=rng, dtype=BF16, num_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=block_size,
                     context_lens=ctx, query_lens=np.ones(batch, np.int64),
                     max_blocks_per_seq=(max_ctx + block_size - 1) // block_size)


def mixed_prefill_decode(seed: int = 0, n_prefill: int = 16, n_decode: int = 48,
                         q_range=(32, 512), prior_range=(0, 2048),
                         dec_range=(64, 4096), block_size: int = 16) -> Case:
    """Chunked prefill mixed with decode on the Llama-3.1-8B shape: 16
    sequences with query chunks of uniform [32, 512] new tokens after a prior
    context uniform in [0, 2048], and 48 decode sequences (one query token,
    context uniform in [64, 4096]); bf16; the sequence order is shuffled."""
    rng = np.random.default_rng(seed)
    qp = rng.integers(q_range[0], q_range[1] + 1, size=n_prefill)
    prior = rng.integers(prior_range[0], prior_range[1] + 1, size=n_prefill)
    dctx = rng.integers(dec_range[0], dec_range[1] + 1, size=n_decode)
    ctx = np.concatenate([prior + qp, dctx])
    ql = np.concatenate([qp, np.ones(n_decode, np.int64)])
    order = rng.permutation(n_prefill + n_decode)
    ctx, ql = ctx[order], ql[order]
    mbs = (max(prior_range[1] + q_range[1], dec_range[1]) + block_size - 1) // block_size
    return make_case("mixed_prefill_decode" + _suffix(block_size), seed=seed, rng=rng,
                     dtype=BF16, num_heads=32, num_kv_heads=8, head_dim=128,
                     block_size=block_size,
                     context_lens=ctx, query_lens=ql, max_blocks_per_seq=mbs,
                     is_decode=False)


def head_sweep(seed: int = 0, num_kv_heads: int = 8, batch: int = 128,
               ctx_len: int = 1024) -> Case:
    """MQA / GQA / MHA at 32 query heads, head_dim 128, bf16, block 16,
    batch 128, context 1024 each; KV heads 1, 8 or 32."""
    rng = np.random.default_rng(seed)
    ctx = np.full(batch, ctx_len, np.int64)
    return make_case(f"head_sweep_kv{num_kv_heads}", seed=seed, rng=rng,
                     dtype=BF16, num_heads=32, num_kv_heads=num_kv_heads,
                     head_dim=128, block_size=16, context_lens=ctx,
                     query_lens=np.ones(batch, np.int64))


def long_context_decode(seed: int = 0, batch: int = 8, lo: int = 16384,
                        hi: int = 32768, num_splits: int = 0) -> Case:
    """Long-context split-KV decode: batch 8, 32 query / 8 KV heads,
    head_dim 128, bf16, block 16, context uniform in [16384, 32768]; 1% of
    the K rows scaled by 8."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi + 1, size=batch)
    return make_case("long_context_decode", seed=seed, rng=rng, dtype=BF16,
                     num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                     context_lens=ctx, query_lens=np.ones(batch, np.int64),
                     max_blocks_per_seq=(hi + 15) // 16, key_outlier_prob=0.01,
                     num_splits=num_splits)


@dataclasses.dataclass
class VarlenCase:
    """A varlen batch with contiguous keys and values (no cache): sequence b
    has query rows q[cu_q[b]:cu_q[b+1]] and key/value rows
    k, v[cu_k[b]:cu_k[b+1]]."""
    name: str
    dtype: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    q: np.ndarray        # [Tq, Hq, D] bits
    k: np.ndarray        # [Tk, Hkv, D] bits
    v: np.ndarray
    cu_q: np.ndarray     # [B+1] int32
    cu_k: np.ndarray

    @property
    def num_seqs(self) -> int:
        return int(self.cu_q.shape[0] - 1)

    @property
    def total_query_tokens(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_query_len(self) -> int:
        d = np.diff(self.cu_q)
        return int(d.max()) if d.size else 0

    def flops(self) -> float:
        """QK^T and PV, 4 * Hq * D per (query row, visible key)."""
        ql, kl = np.diff(self.cu_q).astype(np.int64), np.diff(self.cu_k).astype(np.int64)
        keys = ql * (kl - ql) + ql * (ql + 1) // 2
        return 4.0 * self.num_heads * self.head_dim * float(keys.sum())


def make_varlen_case(name: str, *, seed: int, dtype: int, num_heads: int,
                     num_kv_heads: int, head_dim: int, q_lens, k_lens=None,
                     scale: Optional[float] = None,
                     rng: Optional[np.random.Generator] = None) -> VarlenCase:
    """Seeded N(0,1) q, k, v for a varlen batch; k_lens defaults to q_lens
    (causal self-attention over each prompt); k_lens >= q_lens."""
    if rng is None:
        rng = np.random.default_rng(seed)
    ql = np.asarray(q_lens, dtype=np.int64)
    kl = ql.copy() if k_lens is None else np.asarray(k_lens, dtype=np.int64)
    assert kl.shape == ql.shape and np.all(kl >= ql) and np.all(ql >= 0)
    cu_q = np.zeros(ql.size + 1, np.int32)
    cu_q[1:] = np.cumsum(ql)
    cu_k = np.zeros(kl.size + 1, np.int32)
    cu_k[1:] = np.cumsum(kl)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    q = _normal_bits(rng, (int(cu_q[-1]), num_heads, head_dim), dtype)
    k = _normal_bits(rng, (int(cu_k[-1]), num_kv_heads, head_dim), dtype)
    v = _normal_bits(rng, (int(cu_k[-1]), num_kv_heads, head_dim), dtype)
    return VarlenCase(name=name, dtype=dtype, num_heads=num_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim, scale=float(scale),
                      q=q, k=k, v=v, cu_q=cu_q, cu_k=cu_k)


def varlen_prefill_llama8b(seed: int = 0, batch: int = 16, lo: int = 128,
                           hi: int = 2048) -> VarlenCase:
    """Prompt prefill before any cache write, Llama-3.1-8B shape (32 query /
    8 KV heads, head_dim 128, bf16): 16 prompts of uniform [128, 2048]
    tokens, causal self-attention over each."""
    rng = np.random.default_rng(seed)
    ql = rng.integers(lo, hi + 1, size=batch)
    return make_varlen_case("varlen_prefill_llama8b", seed=seed, rng=rng, dtype=BF16,
                            num_heads=32, num_kv_heads=8, head_dim=128, q_lens=ql)


# Vision tokens per image of a Llama-3.2-Vision-style encoder: 1601 per
# image tile (1600 patches and a class token), 1 to 4 tiles.  The page on
# cross-attention QKV (vLLM PR #7448, discussion) measures that model family
# at batch 16; the token count is the model's, assumed here.
_VISION_TOKENS_PER_TILE = 1601


def cross_attention_decode(seed: int = 0, batch: int = 16, block_size: int = 16) -> Case:
    """Cross-attention decode (one decoder token per sequence) over a static
    encoder cache, Llama-3.2-11B-Vision-shaped cross-attention layer: 32 query
    / 8 KV heads, head_dim 128, bf16; each sequence's encoder output is 1-4
    image tiles of 1601 vision tokens (uniform)."""
    rng = np.random.default_rng(seed)
    enc = rng.integers(1, 5, size=batch) * _VISION_TOKENS_PER_TILE
    return make_cross_case("cross_attention_decode" + _suffix(block_size), seed=seed, rng=rng,
                           dtype=BF16, num_heads=32, num_kv_heads=8, head_dim=128,
                           block_size=block_size, encoder_lens=enc,
                           query_lens=np.ones(batch, np.int64))


def cross_attention_prefill(seed: int = 0, batch: int = 16, q_range=(32, 512),
                            block_size: int = 16) -> Case:
    """The decoder's prompt chunk attending to the same static encoder cache
    (no causal mask): batch 16, decoder chunks uniform [32, 512] tokens."""
    rng = np.random.default_rng(seed)
    enc = rng.integers(1, 5, size=batch) * _VISION_TOKENS_PER_TILE
    ql = rng.integers(q_range[0], q_range[1] + 1, size=batch)
    return make_cross_case("cross_attention_prefill" + _suffix(block_size), seed=seed, rng=rng,
                           dtype=BF16, num_heads=32, num_kv_heads=8, head_dim=128,
                           block_size=block_size, encoder_lens=enc, query_lens=ql)


WORKLOADS = {
    "tiny_gqa_decode": tiny_gqa_decode,
    "llama8b_decode": llama8b_decode,
    "mixed_prefill_decode": mixed_prefill_decode,
    "head_sweep": head_sweep,
    "long_context_decode": long_context_decode,
    "cross_attention_decode": cross_attention_decode,
    "cross_attention_prefill": cross_attention_prefill,
}


def describe(case: Case) -> Dict[str, object]:
    ql = case.query_lens
    return {
        "workload": case.name,
        "dtype": DTYPE_NAMES[case.dtype],
        "num_seqs": case.num_seqs,
        "num_heads": case.num_heads,
        "num_kv_heads": case.num_kv_heads,
        "head_dim": case.head_dim,
        "block_size": case.block_size,
        "num_blocks": case.num_blocks,
        "context_tokens": int(case.context_lens.sum()),
        "query_tokens": int(ql.sum()),
        "max_context": int(case.context_lens.max()),
    }
