// Work-list builder: one small CTA turns context_lens (and cu_query_lens for
// a mixed batch) into the decode (sequence, split) pairs and the prefill
// tiles that the persistent attention kernels hand out, so the host never
// reads device lengths.  Both lists are bucket-sorted longest-first, which
// lets dynamic hand-out finish with the short items (longest-processing-time
// order).
#include "pa_kernels.cuh"

namespace pa {

namespace {
constexpr int kThreads = 1024;
constexpr int kDecBuckets = 128;  // by 16-key stages, clamped
constexpr int kPfBuckets = 256;   // by 64-key stages, clamped

struct SeqPlan {
  int qlen, ctx, tok;
  int nsplit, chunk_keys;  // decode
  int ntile;               // prefill
  bool bad;                // lengths outside the contract: no work, flagged
};

__device__ __forceinline__ SeqPlan plan_seq(const PrepareParams& p, int b) {
  SeqPlan s{0, 0, 0, 0, 0, 0, false};
  if (b >= p.num_seqs) return s;
  s.ctx = p.context_lens[b];
  if (p.cu_query_lens) {
    s.tok = p.cu_query_lens[b];
    s.qlen = p.cu_query_lens[b + 1] - s.tok;
  } else {
    s.tok = b;
    s.qlen = 1;
  }
  const int ctx = s.ctx;
  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  if (ctx < 0 || ctx > max_ctx || s.qlen < 0 || (s.qlen > ctx && ctx > 0) || s.tok < 0 ||
      static_cast<int64_t>(s.tok) + s.qlen > p.total_tokens) {
    s.bad = true;
    s.qlen = 0;
    return s;
  }
  if (ctx == 0) return s;  // no key: the query rows are zero (written in pass 2)
  if (s.qlen == 1) {
    const int nb = (ctx + p.block_size - 1) / p.block_size;
    if (nb > 0) {
      int chunk;
      if (p.num_splits > 0) {
        chunk = (nb + p.num_splits - 1) / p.num_splits;
      } else {
        const int auto_chunk = (kAutoSplitTokens + p.block_size - 1) / p.block_size;
        const int cap_chunk = (nb + kMaxSplits - 1) / kMaxSplits;
        chunk = auto_chunk > cap_chunk ? auto_chunk : cap_chunk;
      }
      s.nsplit = (nb + chunk - 1) / chunk;
      s.chunk_keys = chunk * p.block_size;
    }
  } else if (s.qlen > 1) {
    s.ntile = (s.qlen + p.tokens_per_tile - 1) / p.tokens_per_tile;
  }
  return s;
}

__device__ __forceinline__ int dec_bucket(int nkeys) {
  int st = (nkeys + kKeyTile - 1) / kKeyTile;
  return st >= kDecBuckets ? kDecBuckets - 1 : st;
}

__device__ __forceinline__ int pf_bucket(int kvlen) {
  int st = (kvlen + kPrefillKeys - 1) / kPrefillKeys;
  return st >= kPfBuckets ? kPfBuckets - 1 : st;
}

// Exclusive scan over the block; returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int& excl) {
  const int tid = threadIdx.x;
  scratch[tid] = v;
  __syncthreads();
  for (int off = 1; off < kThreads; off <<= 1) {
    int t = tid >= off ? scratch[tid - off] : 0;
    __syncthreads();
    scratch[tid] += t;
    __syncthreads();
  }
  const int incl = scratch[tid];
  const int total = scratch[kThreads - 1];
  __syncthreads();
  excl = incl - v;
  return total;
}
}  // namespace

__global__ void __launch_bounds__(kThreads) prepare_kernel(PrepareParams p) {
  __shared__ int scan[kThreads];
  __shared__ int dec_cnt[kDecBuckets];
  __shared__ int pf_cnt[kPfBuckets];
  const int tid = threadIdx.x;
  for (int i = tid; i < kDecBuckets; i += kThreads) dec_cnt[i] = 0;
  for (int i = tid; i < kPfBuckets; i += kThreads) pf_cnt[i] = 0;
  if (tid == 0) p.hdr->status = 0;
  __syncthreads();

  // Pass 1: per-sequence plans, split offsets, bucket histograms.
  int carry = 0, tile_total = 0;
  for (int base = 0; base < p.num_seqs; base += kThreads) {
    const int b = base + tid;
    const SeqPlan s = plan_seq(p, b);
    int excl;
    const int tot = block_exclusive_scan(s.nsplit, scan, excl);
    if (s.bad) Status::raise(&p.hdr->status, PA_DEV_BAD_LENGTHS);
    if (b < p.num_seqs) {
      SeqInfo si;
      si.split_offset = carry + excl;
      si.nsplit = s.nsplit;
      si.tok = s.tok;
      si.qlen = s.qlen;
      p.seq_info[b] = si;
      for (int sp = 0; sp < s.nsplit; ++sp) {
        const int k0 = sp * s.chunk_keys;
        int k1 = k0 + s.chunk_keys;
        if (k1 > s.ctx) k1 = s.ctx;
        atomicAdd(&dec_cnt[dec_bucket(k1 - k0)], 1);
      }
      for (int t = 0; t < s.ntile; ++t) {
        int ntok = s.qlen - t * p.tokens_per_tile;
        if (ntok > p.tokens_per_tile) ntok = p.tokens_per_tile;
        const int pos0 = s.ctx - s.qlen + t * p.tokens_per_tile;
        atomicAdd(&pf_cnt[pf_bucket(pos0 + ntok)], 1);
      }
    }
    int tex;
    tile_total += block_exclusive_scan(s.ntile, scan, tex);
    carry += tot;
  }
  __syncthreads();

  // Bucket starts, longest first.
  if (tid == 0) {
    int acc = 0;
    for (int k = kDecBuckets - 1; k >= 0; --k) {
      const int c = dec_cnt[k];
      dec_cnt[k] = acc;
      acc += c;
    }
    acc = 0;
    for (int k = kPfBuckets - 1; k >= 0; --k) {
      const int c = pf_cnt[k];
      pf_cnt[k] = acc;
      acc += c;
    }
  }
  __syncthreads();

  // Pass 2: emit the sorted lists.
  for (int base = 0; base < p.num_seqs; base += kThreads) {
    const int b = base + tid;
    if (b >= p.num_seqs) continue;
    const SeqPlan s = plan_seq(p, b);
    const int split_offset = p.seq_info[b].split_offset;
    for (int sp = 0; sp < s.nsplit; ++sp) {
      DecPair d;
      d.b = b;
      d.tok = s.tok;
      d.key_begin = sp * s.chunk_keys;
      d.key_end = d.key_begin + s.chunk_keys;
      if (d.key_end > s.ctx) d.key_end = s.ctx;
      d.part_idx = s.nsplit > 1 ? split_offset + sp : -1;
      d.pad[0] = d.pad[1] = d.pad[2] = 0;
      const int pos = atomicAdd(&dec_cnt[dec_bucket(d.key_end - d.key_begin)], 1);
      p.pairs[pos] = d;
    }
    for (int t = 0; t < s.ntile; ++t) {
      PfTile tl;
      tl.b = b;
      tl.tok0 = s.tok + t * p.tokens_per_tile;
      tl.ntok = s.qlen - t * p.tokens_per_tile;
      if (tl.ntok > p.tokens_per_tile) tl.ntok = p.tokens_per_tile;
      tl.pos0 = s.ctx - s.qlen + t * p.tokens_per_tile;
      const int pos = atomicAdd(&pf_cnt[pf_bucket(tl.pos0 + tl.ntok)], 1);
      p.tiles[pos] = tl;
    }
    // Query rows of a sequence with no key: zero output rows.
    if (s.ctx == 0 && s.qlen > 0 && p.out) {
      const int64_t n = static_cast<int64_t>(p.num_heads) * p.head_dim * s.qlen;
      uint16_t* o = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(s.tok) * p.num_heads *
                                                        p.head_dim;
      for (int64_t i = 0; i < n; ++i) o[i] = 0;
    }
  }

  if (tid == 0) {
    WsHeader* h = p.hdr;
    h->decode_grab = 0;
    h->decode_pairs = static_cast<uint32_t>(carry);
    h->decode_items = static_cast<uint32_t>(carry) * static_cast<uint32_t>(p.num_kv_heads);
    h->prefill_grab = 0;
    h->prefill_tiles = static_cast<uint32_t>(tile_total);
    h->prefill_items = static_cast<uint32_t>(tile_total) * static_cast<uint32_t>(p.num_kv_heads);
  }
}

int launch_prepare(const PrepareParams& p, bool /*bf16*/, cudaStream_t stream) {
  prepare_kernel<<<1, kThreads, 0, stream>>>(p);
  return 1;
}

}  // namespace pa
