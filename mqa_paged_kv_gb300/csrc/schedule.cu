// Work-list builder: one small CTA turns context_lens (and cu_query_lens for
// a mixed batch) into the decode (sequence, split) pairs and the prefill
// tiles that the persistent attention kernels hand out, so the host never
// reads device lengths.  Both lists are bucket-sorted longest-first, which
// lets dynamic hand-out finish with the short items (longest-processing-time
// order).
//
// Latency matters more than throughput here (it sits on the critical path of
// every call): scans are warp-shuffle scans, and the attention kernel is
// launched as a programmatic dependent of this one, so its prologue overlaps
// this kernel.
#include "pa_kernels.cuh"

namespace pa {

namespace {
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
static_assert(kWarps <= 32, "one warp scans the warp totals");
constexpr int kDecBuckets = 128;  // by 16-key stages, clamped
constexpr int kPfBuckets = 256;   // by 64-key stages, clamped

struct SeqPlan {
  int qlen, ctx, tok, kbase;
  int nsplit, chunk_keys;  // decode
  int ntile;               // prefill
  bool bad;                // lengths outside the contract: no work, flagged
  bool bad_rows;           // query rows outside [0, total) or a negative count
};

__device__ __forceinline__ SeqPlan plan_seq(const PrepareParams& p, int b) {
  SeqPlan s{0, 0, 0, 0, 0, 0, 0, false, false};
  if (b >= p.num_seqs) return s;
  if (p.cu_key_lens) {  // contiguous K/V of a varlen batch
    s.kbase = p.cu_key_lens[b];
    s.ctx = p.cu_key_lens[b + 1] - s.kbase;
  } else {
    s.ctx = p.context_lens[b];
  }
  if (p.cu_query_lens) {
    s.tok = p.cu_query_lens[b];
    s.qlen = p.cu_query_lens[b + 1] - s.tok;
  } else {
    s.tok = b;
    s.qlen = 1;
  }
  const int ctx = s.ctx;
  const int max_ctx = p.cu_key_lens ? ctx : p.max_blocks_per_seq * p.block_size;
  if (ctx < 0 || ctx > max_ctx || s.kbase < 0 || s.qlen < 0 || (p.causal && s.qlen > ctx && ctx > 0) || s.tok < 0 ||
      static_cast<int64_t>(s.tok) + s.qlen > p.total_tokens) {
    s.bad = true;
    s.bad_rows = s.qlen < 0 || s.tok < 0 || static_cast<int64_t>(s.tok) + s.qlen > p.total_tokens;
    s.qlen = 0;
    return s;
  }
  if (ctx == 0) return s;  // no key: the query rows are zero (written below)
  if (s.qlen == 1 && !p.cu_key_lens) {
    const int nb = (ctx + p.block_size - 1) / p.block_size;
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
  } else if (s.qlen >= 1) {  // chunks; with contiguous K/V every row
    s.ntile = (s.qlen + p.tokens_per_tile - 1) / p.tokens_per_tile;
  }
  return s;
}

__device__ __forceinline__ int dec_bucket(int nkeys) {
  const int st = (nkeys + kKeyTile - 1) / kKeyTile;
  return st >= kDecBuckets ? kDecBuckets - 1 : st;
}

__device__ __forceinline__ int pf_bucket(int kvlen) {
  const int st = (kvlen + kPrefillKeys - 1) / kPrefillKeys;
  return st >= kPfBuckets ? kPfBuckets - 1 : st;
}

// Lanes of the warp that hold the same bucket add their counts together: the
// group's first lane reserves the group total with one shared-memory atomic,
// and each lane gets its own start inside that range.  (Hundreds of splits
// land in the same bucket; one atomic each would serialise them.)  Counts are
// below 128, so a lane's offset inside its group is assembled bit by bit from
// ballots over the lower lanes of the group.
__device__ __forceinline__ int warp_aggregated_add(int* counters, int bucket, int count) {
  const int lane = threadIdx.x & 31;
  const unsigned grp = __match_any_sync(0xffffffffu, bucket);
  const unsigned lower = grp & ((1u << lane) - 1u);
  int before = 0, total = 0;
#pragma unroll
  for (int bit = 0; bit < 7; ++bit) {
    const unsigned set = __ballot_sync(0xffffffffu, (count >> bit) & 1);
    before += __popc(set & lower) << bit;
    total += __popc(set & grp) << bit;
  }
  const int leader = __ffs(grp) - 1;
  int base = 0;
  if (lane == leader && total > 0) base = atomicAdd(&counters[bucket], total);
  base = __shfl_sync(0xffffffffu, base, leader);
  return base + before;
}

// Exclusive scan of one int per thread over the CTA; returns the total.
__device__ __forceinline__ int block_scan(int v, int* warp_sums, int& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < kWarps) warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  const int total = warp_sums[kWarps - 1];
  __syncthreads();
  excl = before + x - v;
  return total;
}
}  // namespace

// kSplit: the batch has query chunks and the grid is split between the
// prefill and decode kernels (p.split_ctas > 0); a separate instance, so the
// other calls run the work-list build without the estimate.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads) prepare_kernel(PrepareParams p) {
  griddep_launch_dependents();  // the attention kernel may start its prologue
  if (p.header_only) {
    // Equal-share decode: the decode kernel derives its work from the
    // lengths itself; only the status word of this call starts at zero.
    if (threadIdx.x == 0) p.hdr->status = 0;
    griddep_wait();
    return;
  }
  // The lengths this kernel reads are final before the previous kernel
  // could let it start early: a kernel of the caller triggers this launch
  // only when it completes, and the library's own cache write (the one
  // kernel that triggers early) waits for its predecessors before it does.
  // So the work list is built while a preceding cache write still runs, and
  // the wait at the end only orders this kernel's completion after it: the
  // attention kernels, which wait for this one, then read a complete cache.

  __shared__ int warp_sums[kWarps];
  __shared__ int dec_cnt[kDecBuckets];
  __shared__ int pf_cnt[kPfBuckets];
  // Decode keys (per KV head) and prefill (token, key) pairs (per head).
  __shared__ float work[kSplit ? 2 : 1];
  const int tid = threadIdx.x;
  for (int i = tid; i < kDecBuckets; i += kThreads) dec_cnt[i] = 0;
  for (int i = tid; i < kPfBuckets; i += kThreads) pf_cnt[i] = 0;
  if (tid == 0) {
    p.hdr->status = 0;
    if constexpr (kSplit) work[0] = work[1] = 0.f;
  }
  __syncthreads();

  // Pass 1: per-sequence plans, split offsets, bucket histograms.
  int carry = 0, tile_total = 0;
  int first_split_offset = 0;  // this thread's sequence in the first pass
  SeqPlan first_plan{0, 0, 0, 0, 0, 0, 0, false, false};  // ... and its plan (pass 2 reuses it)
  bool any_bad_rows = false;
  for (int base = 0; base < p.num_seqs; base += kThreads) {
    const int b = base + tid;
    const SeqPlan s = plan_seq(p, b);
    if (base == 0) first_plan = s;
    any_bad_rows |= s.bad_rows;
    if constexpr (kSplit) {  // the two kernels' work, for the SM split of a mixed batch
      float dk = s.nsplit > 0 ? static_cast<float>(s.ctx) : 0.f;
      float pk = 0.f;
      if (s.ntile > 0) {
        const float q = static_cast<float>(s.qlen), c = static_cast<float>(s.ctx);
        pk = p.causal ? q * (c - q) + q * (q + 1.f) * 0.5f : q * c;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        dk += __shfl_xor_sync(0xffffffffu, dk, off);
        pk += __shfl_xor_sync(0xffffffffu, pk, off);
      }
      if ((tid & 31) == 0) {
        atomicAdd(&work[0], dk);
        atomicAdd(&work[1], pk);
      }
    }
    int excl;
    const int tot = block_scan(s.nsplit, warp_sums, excl);
    if (s.bad) Status::raise(&p.hdr->status, PA_DEV_BAD_LENGTHS);
    if (b < p.num_seqs) {
      SeqInfo si;
      si.split_offset = carry + excl;
      if (base == 0) first_split_offset = si.split_offset;
      si.nsplit = s.nsplit;
      si.tok = s.tok;
      si.qlen = s.qlen;
      p.seq_info[b] = si;
      for (int t = 0; t < s.ntile; ++t) {
        const int ntok = min(s.qlen - t * p.tokens_per_tile, p.tokens_per_tile);
        const int pos0 = s.ctx - s.qlen + t * p.tokens_per_tile;
        atomicAdd(&pf_cnt[pf_bucket(p.causal ? pos0 + ntok : s.ctx)], 1);
      }
    }
    // Decode splits: all but the last have the full chunk length.
    {
      const int nfull = s.nsplit > 0 ? s.nsplit - 1 : 0;
      const int tail = s.nsplit > 0 ? s.ctx - nfull * s.chunk_keys : 0;
      warp_aggregated_add(dec_cnt, dec_bucket(s.chunk_keys), nfull);
      warp_aggregated_add(dec_cnt, dec_bucket(tail), s.nsplit > 0 ? 1 : 0);
    }
    int tex;
    tile_total += block_scan(s.ntile, warp_sums, tex);
    carry += tot;
  }
  // Query rows are disjoint and inside [0, total) only if every sequence's
  // range is (cu_query_lens non-decreasing, within the token count).  One
  // range outside that means the offsets themselves are wrong, and the other
  // sequences' ranges may overlap: their tiles and splits could then outgrow
  // the workspace, which is sized for disjoint rows.  Such a call does no
  // work at all (the sequences at fault are flagged).
  const bool bad_rows = __syncthreads_or(any_bad_rows) != 0;

  // Bucket starts, longest first: scan the reversed histograms.
  {
    const int k = kDecBuckets - 1 - tid;
    const int v = (tid < kDecBuckets) ? dec_cnt[k] : 0;
    int excl;
    block_scan(v, warp_sums, excl);
    if (tid < kDecBuckets) dec_cnt[k] = excl;
  }
  {
    const int k = kPfBuckets - 1 - tid;
    const int v = (tid < kPfBuckets) ? pf_cnt[k] : 0;
    int excl;
    block_scan(v, warp_sums, excl);
    if (tid < kPfBuckets) pf_cnt[k] = excl;
  }
  __syncthreads();

  // Pass 2: emit the sorted lists and zero the rows of key-less sequences.
  if (bad_rows) {  // no lists; no sequence left for the split combine
    for (int b = tid; b < p.num_seqs; b += kThreads) {
      SeqInfo si;
      si.split_offset = 0;
      si.nsplit = 0;
      si.tok = 0;
      si.qlen = 0;
      p.seq_info[b] = si;
    }
    carry = 0;
    tile_total = 0;
  }
  for (int base = 0; !bad_rows && base < p.num_seqs; base += kThreads) {
    const int b = base + tid;
    // All lanes take part in the warp aggregation.  When one pass covers the
    // batch the plan of pass 1 is still in registers: no second read of the
    // lengths on the critical path.
    const SeqPlan s = p.num_seqs <= kThreads ? first_plan : plan_seq(p, b);
    const int nfull = s.nsplit > 0 ? s.nsplit - 1 : 0;
    const int tail = s.nsplit > 0 ? s.ctx - nfull * s.chunk_keys : 0;
    const int pos_full = warp_aggregated_add(dec_cnt, dec_bucket(s.chunk_keys), nfull);
    const int pos_tail = warp_aggregated_add(dec_cnt, dec_bucket(tail), s.nsplit > 0 ? 1 : 0);
    if (b >= p.num_seqs) continue;
    const int split_offset = p.num_seqs <= kThreads ? first_split_offset
                                                    : p.seq_info[b].split_offset;
    for (int sp = 0; sp < s.nsplit; ++sp) {
      DecPair d;
      d.b = b;
      d.tok = s.tok;
      d.key_begin = sp * s.chunk_keys;
      d.key_end = min(d.key_begin + s.chunk_keys, s.ctx);
      d.part_idx = s.nsplit > 1 ? split_offset + sp : -1;
      d.pad[0] = d.pad[1] = d.pad[2] = 0;
      p.pairs[sp < nfull ? pos_full + sp : pos_tail] = d;
    }
    for (int t = 0; t < s.ntile; ++t) {
      PfTile tl;
      tl.b = b;
      tl.tok0 = s.tok + t * p.tokens_per_tile;
      tl.ntok = min(s.qlen - t * p.tokens_per_tile, p.tokens_per_tile);
      tl.pos0 = s.ctx - s.qlen + t * p.tokens_per_tile;
      tl.nkv = p.causal ? tl.pos0 + tl.ntok : s.ctx;
      tl.kbase = s.kbase;
      tl.pad[0] = tl.pad[1] = 0;
      const int pos = atomicAdd(&pf_cnt[pf_bucket(tl.nkv)], 1);
      p.tiles[pos] = tl;
    }
    if (s.ctx == 0 && s.qlen > 0 && p.out) {
      const int64_t n = static_cast<int64_t>(p.num_heads) * p.head_dim * s.qlen / 8;
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                          static_cast<int64_t>(s.tok) * p.num_heads * p.head_dim);
      for (int64_t i = 0; i < n; ++i) o[i] = make_uint4(0, 0, 0, 0);
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
    // Batch with query chunks: the prefill kernel leaves k of the grid's SMs
    // to the decode kernel, k / n about the decode kernel's share of the
    // two kernels' estimated times.
    if constexpr (kSplit) {
      uint32_t k = 0;
      const int n = p.split_ctas;
      const float td = work[0] * static_cast<float>(p.num_kv_heads * p.head_dim) *
                       (4.f / static_cast<float>(kDecodeBytesPerSmSec));
      const float tp = work[1] * static_cast<float>(p.num_heads * p.head_dim) *
                       (4.f / static_cast<float>(kPrefillFlopsPerSmSec));
      if (td <= 0.f || n < 2) {  // nothing to split (one CTA: the prefill CTA stays)
        k = 0;
      } else if (tp <= 0.f) {
        k = static_cast<uint32_t>(n);
      } else {
        int kk = static_cast<int>(static_cast<float>(n) * td / (td + tp) *
                                  static_cast<float>(kDecodeShareMargin));
        kk = kk < 1 ? 1 : (kk > n - 1 ? n - 1 : kk);
        k = static_cast<uint32_t>(kk);
      }
      h->decode_ctas = k;
    }
  }
  griddep_wait();
}

int launch_prepare(const PrepareParams& p, bool /*bf16*/, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(p.header_only ? 32 : kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, p.split_ctas > 0 ? prepare_kernel<true> : prepare_kernel<false>,
                            p) == cudaSuccess ? 1 : -1;
}

}  // namespace pa
