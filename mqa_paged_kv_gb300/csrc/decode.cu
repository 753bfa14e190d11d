// Paged GQA/MQA decode attention for sm_103a.
//
// Work unit: one (sequence, KV split, KV head) item.  The G query heads that
// share the KV head are processed together, so each cache block of that KV
// head is read from HBM once for all of them (vLLM issue #1880, "[Performance]
// Use optimized kernels for MQA/GQA": the MQA/GQA saving only appears when
// the kernel exploits the sharing; item 2 names the paged decode kernel).
//
// Structure:
//  * persistent CTAs; warps form groups, and each group pulls items from a
//    device work list with one atomic per item;
//  * per group, a ring of R stages; a stage is a 16-key tile of K and V
//    (one TMA box per 64 columns, 128-byte swizzle); the group's producer
//    issues the copies R stages ahead, so HBM reads of the next tiles (and
//    of the next item) overlap the math on the current one;
//  * the grouped dot products run on tensor cores (mma.sync m16n8k16) in one
//    of two orientations, chosen by G:
//    - G <= 8, "swap AB": the KV tokens sit on the MMA's M side
//      (S^T = K Q^T, O^T += V^T P^T), so a 16-key tile fills the 16 rows and
//      the query heads sit on the 8-wide N side; one warp per group, which
//      also issues its own copies; the G query rows travel with the first
//      stage of an item; P^T becomes the B operand of the second MMA with
//      movmatrix;
//    - G > 8, "head major": each consumer warp owns 16 query heads on the M
//      side (S = Q K^T, O += P V), so P leaves the first MMA already in the
//      A-operand layout of the second; a group is ceil(G / 16) consumer
//      warps plus one warp that only issues copies; the query rows of an
//      item go to one of two slots per group, released by the consumers
//      once they hold them in registers;
//  * online softmax in base 2 with fp32 running max / sum per head; the
//    head-major path moves its reference max only when a row's max grows by
//    more than 2^8 (the exponentials stay below 2^8, which fp32 sums and the
//    16-bit P operand carry at full relative precision), so most tiles skip
//    the rescale of the accumulators;
//  * items that cover a whole sequence write the output row; split items
//    write an fp32 partial and its log-sum-exp, merged by combine_kernel,
//    which is launched as a programmatic dependent of this kernel so that
//    it is resident and waiting when the last item finishes.
#include "pa_kernels.cuh"

namespace pa {

namespace {

struct StageMeta {
  int32_t tok, kvh, key_base, nvalid, part_idx, flags, b, qslot;
};
constexpr int kFirst = 1, kLast = 2, kDone = 4;

// Head-major path: the reference max moves only when a row's max exceeds it
// by more than this many powers of two.
constexpr float kRefSlack = 8.f;

template <int D, int GS, bool kHM>
struct DecodeTile {
  static constexpr int kBoxes = D / 64;        // 64-column TMA boxes per row
  static constexpr int kKV = kBoxes * 2048;    // one 16-key tile of K (or V)
  static constexpr int kRows = kHM ? 16 : 8;   // query heads per consumer warp
  static constexpr int kQ = GS * kRows * D * 2;  // query rows of one group
  // swap AB keeps the query rows in every stage, head major in two slots
  static constexpr int kStage = kHM ? 2 * kKV : 2 * kKV + kQ;
  static_assert(kStage % 1024 == 0 && kQ % 1024 == 0, "1024-byte alignment");
};

template <int D, int GS, int NW, int R, bool kHM>
struct DecodeSmem {
  using T = DecodeTile<D, GS, kHM>;
  static constexpr int kWarpsPerGroup = kHM ? GS + 1 : GS;
  static constexpr int kGroups = NW / kWarpsPerGroup;
  static constexpr int kRing = kGroups * R * T::kStage;
  // Head major: two query slots per group, so that the producer can load
  // the next item's query rows while the consumers still read the slot of
  // the current one (they release it only at the end of the item's first
  // stage, once the MMAs that take its fragments have issued).
  static constexpr int kNQ = kHM ? 2 : 0;
  static constexpr int kQSlots = kGroups * kNQ * T::kQ;
  static constexpr int kBarsPerGroup = 2 * R + kNQ;  // full, empty, query slots
  static constexpr int kBars = kGroups * kBarsPerGroup * 8;
  static constexpr int kMeta = kGroups * R * static_cast<int>(sizeof(StageMeta));
  static constexpr int kUsed = kRing + kQSlots + kBars + kMeta;  // then the equal-share arrays
  static constexpr int kBytes = kUsed + 1024;  // + alignment slack
};

// Producer-side description of the item whose tiles are being issued.
struct Cursor {
  int tok, b, kvh, key, key_end, part;
  int ids, ids_base;  // lane l: physical block of logical block ids_base + l
  bool first;
};

// The next item, fetched a step at a time while the current one is issued.
struct Next {
  int state;  // 0 none, 1 grabbed, 2 record loaded, 3 ready, 4 list exhausted
  uint32_t it;
  int kvh;
  DecPair rec;
  int ids;
};

}  // namespace

template <bool kBF16, int D, int GS, int NW, int R, bool kHM>
__global__ void __launch_bounds__(NW * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
  using T = DecodeTile<D, GS, kHM>;
  using S = DecodeSmem<D, GS, NW, R, kHM>;
  constexpr int kMT = D / 16;  // 16-wide MMA steps along D
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Equal shares: the first lengths are loaded before anything else (the
  // prologue's scan waits on them), and the block table is prefetched into
  // L2, a slice per CTA, for the producers' first block ids after the scan.
  int ctx_first = 0;
  if (p.equal_share) {
    if (static_cast<int>(threadIdx.x) < p.num_seqs) ctx_first = __ldg(p.context_lens + threadIdx.x);
    const int64_t bytes = static_cast<int64_t>(p.num_seqs) * p.mbs * 4;
    const int64_t lines = (bytes + 127) / 128;
    const int64_t per = (lines + gridDim.x - 1) / gridDim.x;
    for (int64_t i = threadIdx.x; i < per; i += blockDim.x) {
      const int64_t line = static_cast<int64_t>(blockIdx.x) * per + i;
      if (line < lines) {
        const int64_t off = line * 128 < bytes - 4 ? line * 128 : bytes - 4;  // inside the table
        prefetch_l2(reinterpret_cast<const char*>(p.block_tables) + off);
      }
    }
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = warp / S::kWarpsPerGroup, wig = warp % S::kWarpsPerGroup;
  uint8_t* ring = smem + group * R * T::kStage;
  uint8_t* qslots = smem + S::kRing + group * S::kNQ * T::kQ;  // head major only
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smem + S::kRing + S::kQSlots) + group * S::kBarsPerGroup;
  uint64_t* empty = full + R;
  uint64_t* qempty = full + 2 * R;  // head major only
  StageMeta* meta =
      reinterpret_cast<StageMeta*>(smem + S::kRing + S::kQSlots + S::kBars) + group * R;

  // Query slots start zeroed: rows past G are never written and feed the
  // padded rows (head major) or N columns (swap AB) of the MMA.
  if constexpr (kHM) {
    for (int i = threadIdx.x; i < S::kQSlots / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(smem + S::kRing)[i] = make_uint4(0, 0, 0, 0);
  } else {
    for (int i = threadIdx.x; i < S::kGroups * R * (T::kQ / 16); i += blockDim.x) {
      const int st = i / (T::kQ / 16), c = i % (T::kQ / 16);
      reinterpret_cast<uint4*>(smem + st * T::kStage + 2 * T::kKV)[c] = make_uint4(0, 0, 0, 0);
    }
  }
  if (threadIdx.x == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRing + S::kQSlots);
    for (int g = 0; g < S::kGroups; ++g) {
      uint64_t* gb = bars + g * S::kBarsPerGroup;
      for (int s = 0; s < R; ++s) {
        mbar_init(gb + s, 1);
        mbar_init(gb + R + s, GS);
      }
      for (int i = 0; i < S::kNQ; ++i) mbar_init(gb + 2 * R + i, GS);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  fence_proxy_async();
  __syncthreads();

  const int G = p.G, Hq = p.num_heads, Hkv = p.num_kv_heads, bs = p.block_size;
  const bool producer = kHM ? (wig == GS) : (wig == 0);
  uint32_t* status = &p.hdr->status;
  const uint16_t* qg = static_cast<const uint16_t*>(p.q);

  // ------------------------------------------------ equal share: prologue
  // Every CTA scans the lengths into a prefix of key tiles per sequence,
  // n_b = ceil(ctx_b / 16) (unit (b, kvh) owns tiles Hkv * P[b] + kvh * n_b
  // onward), and each warp group takes the tile range
  // [g * T / NG, (g + 1) * T / NG) of the T = Hkv * P[B] tiles (integer
  // shares, the first T mod NG groups one tile more).  Lengths and block
  // tables are final before this kernel can start, so all of it runs before
  // the wait for the preceding kernels.
  int32_t* skP = reinterpret_cast<int32_t*>(smem + S::kUsed);  // [B + 1]
  int32_t* skC = skP + p.num_seqs + 1;                         // [B] lengths
  int sk_t = 0, sk_end = 0, sk_gstart = 0, sk_gg = 0;
  bool sk_bad = false;
  if (p.equal_share) {
    int32_t* wsum = skC + p.num_seqs;
    const int nwarps = blockDim.x >> 5;
    const int max_ctx = p.mbs * bs;
    int carry = 0;
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
      const int b = base + threadIdx.x;
      int n = 0;
      if (b < p.num_seqs) {
        int c = base == 0 ? ctx_first : __ldg(p.context_lens + b);
        if (c < 0 || c > max_ctx) {  // outside the contract: no keys, flagged
          sk_bad = true;
          c = 0;
        }
        skC[b] = c;
        n = (c + kKeyTile - 1) / kKeyTile;
      }
      int x = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      if (warp == 0) {
        int w = lane < nwarps ? wsum[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, w, off);
          if (lane >= off) w += y;
        }
        if (lane < nwarps) wsum[lane] = w;
      }
      __syncthreads();
      if (b < p.num_seqs) skP[b] = carry + (warp ? wsum[warp - 1] : 0) + x - n;
      carry += wsum[nwarps - 1];
      __syncthreads();
    }
    if (threadIdx.x == 0) skP[p.num_seqs] = carry;
    sk_bad = __syncthreads_or(sk_bad) != 0;
    const int total = Hkv * carry;
    const int ng = static_cast<int>(gridDim.x) * S::kGroups;
    sk_gg = static_cast<int>(blockIdx.x) * S::kGroups + group;
    const int q = total / ng, r = total - q * ng;
    sk_gstart = sk_gg * q + min(sk_gg, r);
    sk_end = sk_gstart + q + (sk_gg < r ? 1 : 0);
    sk_t = sk_gstart;
  }
  // Sorted list: its length, read once the list is complete (after the wait
  // below; the lambdas that use it only run after that point).
  uint32_t num_items = 0;

  // ---------------------------------------------------------------- producer
  uint32_t p_iter = 0;
  uint32_t q_items = 0;  // items whose query rows were issued (head major)
  bool p_finished = false;
  Cursor cur;
  cur.key = cur.key_end = 0;
  cur.ids = -1;
  cur.ids_base = 0;
  cur.first = false;
  cur.tok = cur.b = cur.kvh = cur.part = 0;
  Next nx;
  nx.state = 0;
  nx.it = 0;
  nx.kvh = 0;
  nx.ids = -1;

  auto load_ids = [&](int b, int lblk0, int key_end) -> int {
    const int lb = lblk0 + lane;
    if (lb * bs < key_end) return __ldg(p.block_tables + static_cast<int64_t>(b) * p.mbs + lb);
    return -1;
  };

  auto advance = [&]() {
    if (nx.state == 0 && p.equal_share) {
      // The next piece of this group's range: the unit holding tile sk_t
      // (the last sequence whose first tile is at or before it; empty
      // sequences share their successor's prefix), cut at the range's end.
      if (sk_t >= sk_end) {
        nx.state = 4;
        return;
      }
      int lo = 0, hi = p.num_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (Hkv * skP[mid] <= sk_t) lo = mid; else hi = mid - 1;
      }
      const int base = Hkv * skP[lo], n = skP[lo + 1] - skP[lo];
      const int kvh = (sk_t - base) / n;
      const int su = base + kvh * n, eu = su + n;
      const int pe = min(sk_end, eu);
      nx.kvh = kvh;
      nx.rec.b = lo;
      nx.rec.tok = lo;
      nx.rec.key_begin = (sk_t - su) * kKeyTile;
      nx.rec.key_end = pe == eu ? skC[lo] : (pe - su) * kKeyTile;
      // a whole unit writes its output row; a cut one its partial, in the
      // group's first slot when it opens the range, else in the second
      nx.rec.part_idx = (sk_t == su && pe == eu) ? -1 : 2 * sk_gg + (sk_t == sk_gstart ? 0 : 1);
      sk_t = pe;
      nx.state = 2;
      return;
    }
    if (nx.state == 0) {
      uint32_t it = 0;
      if (lane == 0) it = atomicAdd(&p.hdr->decode_grab, 1u);
      nx.it = it;
      nx.state = 1;
    } else if (nx.state == 1) {
      const uint32_t it = __shfl_sync(0xffffffffu, nx.it, 0);
      if (it >= num_items) {
        nx.state = 4;
      } else {
        const uint32_t pair = it / static_cast<uint32_t>(Hkv);
        nx.kvh = static_cast<int>(it - pair * static_cast<uint32_t>(Hkv));
        const int4* rp = reinterpret_cast<const int4*>(p.pairs + pair);
        const int4 r0 = p.concurrent ? __ldcg(rp) : __ldg(rp);
        const int4 r1 = p.concurrent ? __ldcg(rp + 1) : __ldg(rp + 1);
        nx.rec.b = r0.x;
        nx.rec.tok = r0.y;
        nx.rec.key_begin = r0.z;
        nx.rec.key_end = r0.w;
        nx.rec.part_idx = r1.x;
        nx.state = 2;
      }
    } else if (nx.state == 2) {
      nx.ids = load_ids(nx.rec.b, nx.rec.key_begin / bs, nx.rec.key_end);
      nx.state = 3;
    }
  };

  auto issue_stage = [&]() {
    if (p_finished) return;
    const int s = static_cast<int>(p_iter % R);
    // A swap-AB group of one warp consumes its own copies in order and never
    // runs more than R stages ahead of itself.
    if ((kHM || GS > 1) && p_iter >= static_cast<uint32_t>(R)) {
      if (!mbar_wait_warp(&empty[s], ((p_iter / R) - 1) & 1, p.wait_ns)) {
        if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
        p_finished = true;
        return;
      }
    }
    if (cur.key >= cur.key_end) {
      while (nx.state < 3) advance();
      if (nx.state == 4) {
        if (lane == 0) {
          meta[s].flags = kDone;
          mbar_arrive(&full[s]);
        }
        p_finished = true;
        ++p_iter;
        return;
      }
      cur.tok = nx.rec.tok;
      cur.b = nx.rec.b;
      cur.kvh = nx.kvh;
      cur.key = nx.rec.key_begin;
      cur.key_end = nx.rec.key_end;
      cur.part = nx.rec.part_idx;
      cur.ids = nx.ids;
      cur.ids_base = nx.rec.key_begin / bs;
      cur.first = true;
      nx.state = 0;
    }
    const int key_base = cur.key;
    int nvalid = cur.key_end - key_base;
    if (nvalid > kKeyTile) nvalid = kKeyTile;
    const int lblk = key_base / bs;
    if (lblk - cur.ids_base >= 32) {
      cur.ids_base = lblk;
      cur.ids = load_ids(cur.b, lblk, cur.key_end);
    }
    int blk = __shfl_sync(0xffffffffu, cur.ids, lblk - cur.ids_base);
    if (blk < 0 || blk >= p.num_blocks) {
      if (lane == 0) Status::raise(status, PA_DEV_BAD_BLOCK_ID);
      blk = 0;
      nvalid = 0;
    }
    const int y = (blk * Hkv + cur.kvh) * bs + (key_base - lblk * bs);
    const bool first = cur.first;
    const bool last = key_base + kKeyTile >= cur.key_end;
    int qslot = 0;
    if (kHM && first) {
      // The slot's previous item must be in the consumers' registers (its
      // first stage is done).
      constexpr uint32_t kNQ = S::kNQ > 0 ? S::kNQ : 1;  // (swap AB has no slots)
      qslot = static_cast<int>(q_items % kNQ);
      if (q_items >= kNQ &&
          !mbar_wait_warp(&qempty[qslot], ((q_items / kNQ) - 1) & 1, p.wait_ns)) {
        if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
        p_finished = true;
        return;
      }
      ++q_items;
    }
    if (lane == 0) {
      StageMeta m;
      m.tok = cur.tok;
      m.kvh = cur.kvh;
      m.key_base = key_base;
      m.nvalid = nvalid;
      m.part_idx = cur.part;
      m.flags = (first ? kFirst : 0) | (last ? kLast : 0);
      m.b = cur.b;
      m.qslot = qslot;
      meta[s] = m;
      const uint32_t qbytes = first ? static_cast<uint32_t>(G * D * 2) : 0u;
      mbar_arrive_expect_tx(&full[s], 2 * T::kKV + qbytes);
      uint8_t* st = ring + s * T::kStage;
#pragma unroll
      for (int bx = 0; bx < T::kBoxes; ++bx) {
        tma_load_2d(st + bx * 2048, &tmk, bx * 64, y, &full[s]);
        tma_load_2d(st + T::kKV + bx * 2048, &tmv, bx * 64, y, &full[s]);
      }
      if (first) {
        const uint16_t* src =
            qg + (static_cast<int64_t>(cur.tok) * Hq + static_cast<int64_t>(cur.kvh) * G) * D;
        bulk_load(kHM ? qslots + qslot * T::kQ : st + 2 * T::kKV, src, qbytes, &full[s]);
      }
    }
    cur.key += kKeyTile;
    cur.first = false;
    ++p_iter;
    if (nx.state < 3) advance();
  };

  // Wait for the preceding kernels (the cache write; the work-list kernel,
  // which writes the sorted list and resets the status word).  With equal
  // shares each producer first prepares its first piece (record and block
  // ids).  Beside a prefill kernel this kernel starts without a wait (the
  // prefill kernel let it start only after its own wait for the list) and
  // reads the list through L2.
  if (p.equal_share) {
    if (producer)
      while (nx.state < 3) advance();
    griddep_wait();
    if (blockIdx.x == 0) {  // the tile prefix, for the combine
      for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) p.sk_prefix[i] = skP[i];
      if (threadIdx.x == 0 && sk_bad) Status::raise(status, PA_DEV_BAD_LENGTHS);
    }
  } else {
    if (!p.concurrent) griddep_wait();
    num_items = p.concurrent ? __ldcg(&p.hdr->decode_items) : p.hdr->decode_items;
  }
  if (p.trigger_dependents) griddep_launch_dependents();  // the split combine may become resident

  const int g = lane >> 2, q4 = lane & 3;   // MMA fragment: row group, column pair
  const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix index, row in it

  if constexpr (kHM) {
    // ------------------------------------------------ head major, G > 8
    if (producer) {
      while (!p_finished) issue_stage();
      // Leave no copy in flight: wait for the latest fill of each slot, so
      // the CTA never exits with TMA writes pending (the fixed 2 s limit,
      // whatever the pipeline limit: copies land within microseconds).
      for (uint32_t i = p_iter > static_cast<uint32_t>(R) ? p_iter - R : 0u; i < p_iter; ++i)
        if (!mbar_wait_warp(&full[i % R], (i / R) & 1)) break;
      if (p.concurrent) griddep_wait();  // complete after the prefill kernel beside this one
      return;
    }
    constexpr int kNT = D / 8;  // 8-column output tiles along D
    float o[kNT][4];
    uint32_t qa[kMT][4];
    float mref[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};  // rows g, g + 8
#pragma unroll
    for (int i = 0; i < kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kMT; ++i) qa[i][0] = qa[i][1] = qa[i][2] = qa[i][3] = 0u;
    const int h0 = 16 * wig + g, h1 = h0 + 8;  // this lane's two heads

    uint32_t c_iter = 0;
    while (true) {
      const int s = static_cast<int>(c_iter % R);
      if (!mbar_wait_warp(&full[s], (c_iter / R) & 1, p.wait_ns)) {
        if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
        break;
      }
      const StageMeta m = meta[s];
      if (m.flags & kDone) break;
      const uint32_t kbase = smem_u32(ring + s * T::kStage);
      const uint32_t vbase = kbase + T::kKV;

      if (m.flags & kFirst) {
#pragma unroll
        for (int i = 0; i < kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        mref[0] = mref[1] = -INFINITY;
        lsum[0] = lsum[1] = 0.f;
        // A operand (Q): this warp's 16 heads, 16-byte chunks along D.
        const uint32_t qbase = smem_u32(qslots + m.qslot * T::kQ) + wig * 16 * (D * 2);
#pragma unroll
        for (int ks = 0; ks < kMT; ++ks)
          ldsm_x4(qbase + (rr + ((mi & 1) << 3)) * (D * 2) + (2 * ks + (mi >> 1)) * 16, qa[ks]);
        // The slot is released with the stage, below: an arrive issued right
        // after these loads, before any instruction takes their registers,
        // let the producer's copy of a later item's rows land while a warp
        // was still reading, and the warp saw a mix of the two items' rows.
      }

      // S[16 heads][16 keys] = Q K^T: keys 0-7 and 8-15 as two 8-wide N
      // tiles, even and odd D steps on separate accumulation chains.
      float sa0[4] = {0.f, 0.f, 0.f, 0.f}, sa1[4] = {0.f, 0.f, 0.f, 0.f};
      float sb0[4] = {0.f, 0.f, 0.f, 0.f}, sb1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < kMT; ++ks) {
        uint32_t b[4];  // keys 0-7 (low, high D half), keys 8-15 (low, high)
        ldsm_x4(kbase + (ks >> 2) * 2048 + swz128(rr + ((mi >> 1) << 3), ((ks & 3) << 1) + (mi & 1)),
                b);
        if (ks & 1) {
          mma_16816<kBF16>(sb0, qa[ks], b[0], b[1]);
          mma_16816<kBF16>(sb1, qa[ks], b[2], b[3]);
        } else {
          mma_16816<kBF16>(sa0, qa[ks], b[0], b[1]);
          mma_16816<kBF16>(sa1, qa[ks], b[2], b[3]);
        }
      }
      // x[nt][0..1]: head g, keys 8nt + 2q4 (+1); x[nt][2..3]: head g + 8.
      float x[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[0][i] = (sa0[i] + sb0[i]) * p.scale_log2;
        x[1][i] = (sa1[i] + sb1[i]) * p.scale_log2;
      }
      const int nv = m.nvalid;
      if (nv < kKeyTile) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int k0 = nt * 8 + 2 * q4;
          if (k0 >= nv) x[nt][0] = x[nt][2] = -INFINITY;
          if (k0 + 1 >= nv) x[nt][1] = x[nt][3] = -INFINITY;
        }
      }

      // Online softmax per head row; the four lanes of a row hold 4 keys each.
      float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const bool up0 = mx0 > mref[0] + kRefSlack, up1 = mx1 > mref[1] + kRefSlack;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        const float al0 = up0 ? ex2(mref[0] - mx0) : 1.f;  // 0 while the row had no key
        const float al1 = up1 ? ex2(mref[1] - mx1) : 1.f;
        if (up0) mref[0] = mx0;
        if (up1) mref[1] = mx1;
        lsum[0] *= al0;
        lsum[1] *= al1;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          o[nt][0] *= al0;
          o[nt][1] *= al0;
          o[nt][2] *= al1;
          o[nt][3] *= al1;
        }
      }
      const float r0 = mref[0] == -INFINITY ? 0.f : mref[0];
      const float r1 = mref[1] == -INFINITY ? 0.f : mref[1];
      // P in the A-operand layout of the PV MMA: a0/a1 keys 0-7, a2/a3 keys 8-15.
      uint32_t pa[4];
      pa[0] = pack2<kBF16>(ex2(x[0][0] - r0), ex2(x[0][1] - r0));
      pa[1] = pack2<kBF16>(ex2(x[0][2] - r1), ex2(x[0][3] - r1));
      pa[2] = pack2<kBF16>(ex2(x[1][0] - r0), ex2(x[1][1] - r0));
      pa[3] = pack2<kBF16>(ex2(x[1][2] - r1), ex2(x[1][3] - r1));
      {
        float e0, e1, e2, e3;
        unpack2<kBF16>(pa[0], e0, e1);
        unpack2<kBF16>(pa[2], e2, e3);
        lsum[0] += (e0 + e1) + (e2 + e3);
        unpack2<kBF16>(pa[1], e0, e1);
        unpack2<kBF16>(pa[3], e2, e3);
        lsum[1] += (e0 + e1) + (e2 + e3);
      }

      // O[16 heads][D] += P V; V rows past the valid keys are zeroed (they
      // may hold any bits, and 0 * NaN would reach the sum).
      const uint32_t vm_lo = keep_mask(2 * q4 < nv, 2 * q4 + 1 < nv);
      const uint32_t vm_hi = keep_mask(8 + 2 * q4 < nv, 9 + 2 * q4 < nv);
#pragma unroll
      for (int j = 0; j < kMT; ++j) {
        uint32_t v[4];  // columns 16j..16j+7 (keys 0-7, 8-15), then 16j+8..16j+15
        ldsm_x4_t(vbase + (j >> 2) * 2048 + swz128(rr + ((mi & 1) << 3), ((j & 3) << 1) + (mi >> 1)),
                  v);
        if (nv < kKeyTile) {
          v[0] &= vm_lo;
          v[1] &= vm_hi;
          v[2] &= vm_lo;
          v[3] &= vm_hi;
        }
        mma_16816<kBF16>(o[2 * j], pa, v[0], v[1]);
        mma_16816<kBF16>(o[2 * j + 1], pa, v[2], v[3]);
      }
      __syncwarp();
      if (lane == 0) {
        // The MMAs above took every K, V and Q fragment of the stage.
        mbar_arrive(&empty[s]);
        if (m.flags & kFirst) mbar_arrive(&qempty[m.qslot]);
      }

      if (m.flags & kLast) {
        float l0 = lsum[0], l1 = lsum[1];
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        const float il0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float il1 = l1 > 0.f ? 1.f / l1 : 0.f;
        if (m.part_idx < 0) {
          uint16_t* out = static_cast<uint16_t*>(p.out) +
                          (static_cast<int64_t>(m.tok) * Hq + static_cast<int64_t>(m.kvh) * G) * D;
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int d = nt * 8 + 2 * q4;
            if (h0 < G)
              *reinterpret_cast<uint32_t*>(out + h0 * D + d) =
                  pack2<kBF16>(o[nt][0] * il0, o[nt][1] * il0);
            if (h1 < G)
              *reinterpret_cast<uint32_t*>(out + h1 * D + d) =
                  pack2<kBF16>(o[nt][2] * il1, o[nt][3] * il1);
          }
        } else {
          const int64_t prow = static_cast<int64_t>(m.part_idx) * p.part_row_stride +
                               static_cast<int64_t>(m.kvh) * p.part_kvh_rows;
          float* po = p.part_o + prow * D;
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int d = nt * 8 + 2 * q4;
            if (h0 < G)
              *reinterpret_cast<float2*>(po + h0 * D + d) =
                  make_float2(o[nt][0] * il0, o[nt][1] * il0);
            if (h1 < G)
              *reinterpret_cast<float2*>(po + h1 * D + d) =
                  make_float2(o[nt][2] * il1, o[nt][3] * il1);
          }
          if (q4 == 0) {
            float* pl = p.part_lse + prow;
            if (h0 < G) pl[h0] = l0 > 0.f ? mref[0] + __log2f(l0) : -INFINITY;
            if (h1 < G) pl[h1] = l1 > 0.f ? mref[1] + __log2f(l1) : -INFINITY;
          }
        }
      }
      ++c_iter;
    }
  } else {
    // ------------------------------------------------ swap AB, G <= 8
    float acc[kMT][4];
    float mrow[2], lrow[2];
    uint32_t qf[kMT][2];
#pragma unroll
    for (int i = 0; i < kMT; ++i) {
      acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      qf[i][0] = qf[i][1] = 0u;
    }
    mrow[0] = mrow[1] = -INFINITY;
    lrow[0] = lrow[1] = 0.f;
    auto finalize = [&](const StageMeta& m) {
      float l0 = lrow[0], l1 = lrow[1];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      const float il0 = l0 > 0.f ? 1.f / l0 : 0.f;
      const float il1 = l1 > 0.f ? 1.f / l1 : 0.f;
      const int hb = 8 * wig;
      if (m.part_idx < 0) {
        uint16_t* out = static_cast<uint16_t*>(p.out) +
                        (static_cast<int64_t>(m.tok) * Hq + static_cast<int64_t>(m.kvh) * G) * D;
        const int h = hb + g;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const uint32_t t0 =
              movmatrix_t(pack2<kBF16>(acc[mt][0] * il0, acc[mt][1] * il1));
          const uint32_t t1 =
              movmatrix_t(pack2<kBF16>(acc[mt][2] * il0, acc[mt][3] * il1));
          if (h < G) {
            uint32_t* o = reinterpret_cast<uint32_t*>(out + h * D + mt * 16 + 2 * q4);
            o[0] = t0;
            o[4] = t1;  // +8 elements
          }
        }
      } else {
        const int64_t prow = static_cast<int64_t>(m.part_idx) * p.part_row_stride +
                             static_cast<int64_t>(m.kvh) * p.part_kvh_rows;
        float* po = p.part_o + prow * D;
        const int h0 = hb + 2 * q4, h1 = h0 + 1;
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int d0 = mt * 16 + g, d1 = d0 + 8;
          if (h0 < G) {
            po[h0 * D + d0] = acc[mt][0] * il0;
            po[h0 * D + d1] = acc[mt][2] * il0;
          }
          if (h1 < G) {
            po[h1 * D + d0] = acc[mt][1] * il1;
            po[h1 * D + d1] = acc[mt][3] * il1;
          }
        }
        if (g == 0) {
          float* pl = p.part_lse + prow;
          if (h0 < G) pl[h0] = l0 > 0.f ? mrow[0] + __log2f(l0) : -INFINITY;
          if (h1 < G) pl[h1] = l1 > 0.f ? mrow[1] + __log2f(l1) : -INFINITY;
        }
      }
    };

    if (producer)
      for (int i = 0; i < R; ++i) issue_stage();

    uint32_t c_iter = 0;
    while (true) {
      const int s = static_cast<int>(c_iter % R);
      if (!mbar_wait_warp(&full[s], (c_iter / R) & 1, p.wait_ns)) {
        if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
        break;
      }
      const StageMeta m = meta[s];
      if (m.flags & kDone) break;
      const uint32_t kbase = smem_u32(ring + s * T::kStage);
      const uint32_t vbase = kbase + T::kKV;
      const uint32_t qbase = kbase + 2 * T::kKV;

      if (m.flags & kFirst) {
#pragma unroll
        for (int i = 0; i < kMT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        mrow[0] = mrow[1] = -INFINITY;
        lrow[0] = lrow[1] = 0.f;
        // B operand (Q^T): rows = this warp's 8 heads, 16-byte chunks along D.
#pragma unroll
        for (int ks = 0; ks < kMT; ks += 2) {
          const int row = 8 * wig + rr;
          const int chunk = 2 * ks + mi;
          uint32_t r[4];
          ldsm_x4(qbase + row * (D * 2) + chunk * 16, r);
          qf[ks][0] = r[0];
          qf[ks][1] = r[1];
          qf[ks + 1][0] = r[2];
          qf[ks + 1][1] = r[3];
        }
      }

      // S^T[16 keys][8 heads] = K Q^T, two accumulation chains.
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < kMT; ++ks) {
        const int key = rr + ((mi & 1) << 3);
        const int chunk = ((ks & 3) << 1) + (mi >> 1);
        uint32_t a[4];
        ldsm_x4(kbase + (ks >> 2) * 2048 + swz128(key, chunk), a);
        if (ks & 1)
          mma_16816<kBF16>(sb, a, qf[ks][0], qf[ks][1]);
        else
          mma_16816<kBF16>(sa, a, qf[ks][0], qf[ks][1]);
      }
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = (sa[i] + sb[i]) * p.scale_log2;
      const int nv = m.nvalid;
      if (nv < kKeyTile) {
        if (g >= nv) x[0] = x[1] = -INFINITY;
        if (g + 8 >= nv) x[2] = x[3] = -INFINITY;
      }

      // Online softmax per head column (this lane: heads 2*q4, 2*q4 + 1).
      float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(mrow[0], mx0), mn1 = fmaxf(mrow[1], mx1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
      const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = ex2(mrow[0] - ref0), al1 = ex2(mrow[1] - ref1);
      mrow[0] = mn0;
      mrow[1] = mn1;
      const uint32_t ptop = pack2<kBF16>(ex2(x[0] - ref0), ex2(x[1] - ref1));
      const uint32_t pbot = pack2<kBF16>(ex2(x[2] - ref0), ex2(x[3] - ref1));
      float p00, p01, p10, p11;
      unpack2<kBF16>(ptop, p00, p01);
      unpack2<kBF16>(pbot, p10, p11);
      lrow[0] = lrow[0] * al0 + (p00 + p10);
      lrow[1] = lrow[1] * al1 + (p01 + p11);
      const uint32_t b0 = movmatrix_t(ptop);  // P^T rows: keys 2*q4.., column: head g
      const uint32_t b1 = movmatrix_t(pbot);  // keys 8 + 2*q4..
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }

      // O^T[D][8 heads] += V^T P^T.
      const uint32_t vm_lo = keep_mask(2 * q4 < nv, 2 * q4 + 1 < nv);
      const uint32_t vm_hi = keep_mask(8 + 2 * q4 < nv, 9 + 2 * q4 < nv);
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int key = rr + ((mi >> 1) << 3);
        const int chunk = ((mt & 3) << 1) + (mi & 1);
        uint32_t a[4];
        ldsm_x4_t(vbase + (mt >> 2) * 2048 + swz128(key, chunk), a);
        if (nv < kKeyTile) {
          a[0] &= vm_lo;
          a[1] &= vm_lo;
          a[2] &= vm_hi;
          a[3] &= vm_hi;
        }
        mma_16816<kBF16>(acc[mt], a, b0, b1);
      }

      __syncwarp();
      if (GS > 1 && lane == 0) mbar_arrive(&empty[s]);
      if (producer) issue_stage();
      if (m.flags & kLast) finalize(m);
      ++c_iter;
    }

    // Leave no copy in flight: wait for stages this group issued but did not
    // consume, so the CTA never exits with TMA writes pending (the fixed 2 s
    // limit, whatever the pipeline limit).
    if (producer) {
      while (c_iter < p_iter) {
        const int s = static_cast<int>(c_iter % R);
        if (!mbar_wait_warp(&full[s], (c_iter / R) & 1)) break;
        ++c_iter;
      }
    }
  }
  if (p.concurrent) griddep_wait();  // complete after the prefill kernel beside this one
}

// Merge the split partials of each decode sequence (one CTA per sequence
// and group of kCombineHeads query heads, one warp per head):
//   M = max_s lse_s, w_s = 2^(lse_s - M), out = sum_s w_s o_s / sum_s w_s,
// with lse in base 2 and splits of lse = -inf weighted 0.  Latency-bound by
// design: all loads of a head are issued before any is used.
// The CTAs are small (4 warps) so that they fit on an SM beside a decode
// CTA and become resident, waiting, while the decode kernel still runs.
constexpr int kCombineHeads = 4;

template <bool kBF16, int D>
__global__ void __launch_bounds__(32 * kCombineHeads) combine_kernel(const CombineParams p) {
  griddep_wait();  // partials are written by the decode kernel
  const int b = blockIdx.x;
  const SeqInfo si = p.seq_info[b];
  if (si.qlen != 1 || si.nsplit <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = blockIdx.y * kCombineHeads;
  const int Hq = p.num_heads, S = si.nsplit;
  constexpr int kV = D / 32;  // floats per lane
  const float* lse = p.part_lse + static_cast<int64_t>(si.split_offset) * Hq;
  const float* po = p.part_o + static_cast<int64_t>(si.split_offset) * Hq * D;
  uint16_t* out = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(si.tok) * Hq * D;
  for (int h = h0 + warp; h < Hq && h < h0 + kCombineHeads; h += kCombineHeads) {
    // Issue the log-sum-exps and the first eight partial rows together.
    auto load_part = [&](int sp, float (&dst)[kV]) {
      const float* src = po + (static_cast<int64_t>(sp) * Hq + h) * D + lane * kV;
      if constexpr (kV == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
        dst[0] = t.x; dst[1] = t.y; dst[2] = t.z; dst[3] = t.w;
      } else {
        const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
        dst[0] = t.x; dst[1] = t.y;
      }
    };
    const float la = lane < S ? __ldcg(lse + static_cast<int64_t>(lane) * Hq + h) : -INFINITY;
    const float lb = lane + 32 < S ? __ldcg(lse + static_cast<int64_t>(lane + 32) * Hq + h)
                                   : -INFINITY;
    float v[8][kV];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < S) {
        load_part(j, v[j]);
      } else {
#pragma unroll
        for (int i = 0; i < kV; ++i) v[j][i] = 0.f;
      }
    }
    float M = fmaxf(la, lb);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float wa = (M == -INFINITY || la == -INFINITY) ? 0.f : ex2(la - M);
    const float wb = (M == -INFINITY || lb == -INFINITY) ? 0.f : ex2(lb - M);
    float W = wa + wb;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    float acc[kV];
#pragma unroll
    for (int i = 0; i < kV; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < S; s0 += 8) {
      if (s0 > 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (s0 + j < S) {
            load_part(s0 + j, v[j]);
          } else {
#pragma unroll
            for (int i = 0; i < kV; ++i) v[j][i] = 0.f;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sp = s0 + j;
        const float w = __shfl_sync(0xffffffffu, sp < 32 ? wa : wb, sp & 31);
        if (sp < S) {
#pragma unroll
          for (int i = 0; i < kV; ++i) acc[i] += w * v[j][i];
        }
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint32_t packed[kV / 2];
#pragma unroll
    for (int i = 0; i < kV / 2; ++i) packed[i] = pack2<kBF16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    uint16_t* dst = out + static_cast<int64_t>(h) * D + lane * kV;
    if constexpr (kV == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    }
  }
}

// Merge of the equal-share partials.  Unit u = (b, kvh) owns tiles
// [S_u, E_u) and group g the range [start(g), start(g + 1)); the unit was
// cut when its first and last tiles lie in different groups, g_f and g_l.
// Each group g in [g_f, g_l] wrote the unit's piece to its first slot (2g)
// when its range opens inside the unit, and to its second (2g + 1) when
// the unit opens inside its range, which only g_f's can.  Per head (one
// warp): M = max_g lse_g, out = sum_g 2^(lse_g - M) o_g / sum_g 2^(lse_g - M),
// lse in base 2.  Units that were not cut were written by the decode
// kernel; sequences without keys get zero rows here.
template <bool kBF16, int D>
__global__ void __launch_bounds__(32 * kCombineHeads) combine_equal_share_kernel(
    const CombineParams p) {
  griddep_wait();  // partials and the tile prefix are written by the decode kernel
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kCombineHeads + warp;
  const int Hq = p.num_heads, Hkv = p.num_kv_heads, G = Hq / Hkv;
  if (h >= Hq) return;
  constexpr int kV = D / 32;  // values per lane
  uint16_t* dst = static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(b) * Hq + h) * D + lane * kV;
  auto store = [&](const float (&v)[kV]) {
    uint32_t packed[kV / 2];
#pragma unroll
    for (int i = 0; i < kV / 2; ++i) packed[i] = pack2<kBF16>(v[2 * i], v[2 * i + 1]);
    if constexpr (kV == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    }
  };
  // The three prefix entries this head needs, loaded together.
  const int pb = __ldcg(p.sk_prefix + b), pe = __ldcg(p.sk_prefix + b + 1);
  const int total = Hkv * __ldcg(p.sk_prefix + p.num_seqs);
  const int n = pe - pb;
  if (n == 0) {  // no keys: a zero row
    float z[kV];
#pragma unroll
    for (int i = 0; i < kV; ++i) z[i] = 0.f;
    store(z);
    return;
  }
  const int ng = p.sk_groups, q = total / ng, r = total - q * ng;
  const int kvh = h / G, hg = h - kvh * G;
  const int su = Hkv * pb + kvh * n, eu = su + n;
  auto group_of = [&](int t) {
    return t < r * (q + 1) ? t / (q + 1) : r + (t - r * (q + 1)) / q;
  };
  const int gf = group_of(su), gl = group_of(eu - 1);
  if (gf == gl) return;  // one piece: written by the decode kernel
  const bool f_second = gf * q + min(gf, r) < su;
  const int np = gl - gf + 1;
  auto slot_row = [&](int i) {  // partial row of piece i (group gf + i)
    const int gg = gf + i;
    return static_cast<int64_t>(2 * gg + (i == 0 && f_second ? 1 : 0)) * G + hg;
  };
  // The pieces' log-sum-exps (lane c: piece c) and the first eight pieces'
  // rows depend only on the prefix: issue them together, one round trip.
  auto load_row = [&](int i, float (&dst)[kV]) {
    const float* src = p.part_o + slot_row(i) * D + lane * kV;
    if constexpr (kV == 4) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
      dst[0] = t.x; dst[1] = t.y; dst[2] = t.z; dst[3] = t.w;
    } else {
      const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
      dst[0] = t.x; dst[1] = t.y;
    }
  };
  const float l0 = lane < np ? __ldcg(p.part_lse + slot_row(lane)) : -INFINITY;
  float v[8][kV];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < np) {
      load_row(j, v[j]);
    } else {
#pragma unroll
      for (int i = 0; i < kV; ++i) v[j][i] = 0.f;
    }
  }
  float M = l0;
  for (int c = 32 + lane; c < np; c += 32) M = fmaxf(M, __ldcg(p.part_lse + slot_row(c)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[kV], W = 0.f;
#pragma unroll
  for (int i = 0; i < kV; ++i) acc[i] = 0.f;
  for (int c0 = 0; c0 < np; c0 += 32) {
    const float l = c0 == 0 ? l0 : (c0 + lane < np ? __ldcg(p.part_lse + slot_row(c0 + lane)) : -INFINITY);
    const float w = (M == -INFINITY || l == -INFINITY) ? 0.f : ex2(l - M);
    W += w;
    const int cnt = min(32, np - c0);
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      if (c0 > 0 || j0 > 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j0 + j < cnt) {
            load_row(c0 + j0 + j, v[j]);
          } else {
#pragma unroll
            for (int i = 0; i < kV; ++i) v[j][i] = 0.f;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
        if (j0 + j < cnt) {
#pragma unroll
          for (int i = 0; i < kV; ++i) acc[i] += wj * v[j][i];
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int i = 0; i < kV; ++i) acc[i] *= inv;
  store(acc);
}

// ---------------------------------------------------------------- launchers
namespace {

template <bool kBF16, int D, int GS, bool kHM>
int launch_decode_t(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                    cudaStream_t stream, int num_sms) {
  using T = DecodeTile<D, GS, kHM>;
  // Swap AB: 8 warps in groups of GS.  Head major: groups of GS consumer
  // warps plus a producer warp, at most 12 warps per CTA.
  constexpr int kGroups = kHM ? (GS == 1 ? 6 : (GS == 2 ? 4 : 8 / GS)) : 8 / GS;
  constexpr int NW = kGroups * (kHM ? GS + 1 : GS);
  // The ring takes the shared memory left beside the query slots, the
  // equal-share arrays, barriers and stage records: the deeper each group's
  // ring, the more bytes in flight per SM (HBM latency under load is a few
  // microseconds, so in-flight bytes set the streaming rate).
  constexpr int kNQ = kHM ? 2 : 0;
  constexpr int kFixed = 1024 + static_cast<int>(sk_smem_bytes(kSkMaxSeqs)) +
                         kGroups * kNQ * T::kQ + 2048;
  constexpr int kR0 = (227 * 1024 - kFixed) / (kGroups * T::kStage);
  constexpr int R = kR0 < 2 ? 2 : (kR0 > 12 ? 12 : kR0);
  using S = DecodeSmem<D, GS, NW, R, kHM>;
  static_assert(S::kGroups == kGroups, "warps split into whole groups");
  static_assert(kGroups == decode_groups_per_cta(kHM ? (GS == 1 ? 16 : 16 * GS) : 8),
                "the host's group count matches the launched configuration");
  constexpr int kMaxBytes = S::kBytes + static_cast<int>(sk_smem_bytes(kSkMaxSeqs));
  static_assert(kMaxBytes <= 227 * 1024, "fits one CTA per SM");
  auto kern = decode_kernel<kBF16, D, GS, NW, R, kHM>;
  static int configured = -1;  // device whose attribute is set
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxBytes) !=
        cudaSuccess)
      return -1;
    configured = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes =
      S::kBytes + (p.equal_share ? static_cast<int>(sk_smem_bytes(p.num_seqs)) : 0);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, p) == cudaSuccess ? 1 : -1;
}

// G <= 8: swap AB, one warp per group.  G > 8: head major, ceil(G / 16)
// consumer warps per group (G <= 64).
template <bool kBF16, int D>
int launch_decode_d(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                    cudaStream_t stream, int num_sms) {
  if (p.G <= 8) return launch_decode_t<kBF16, D, 1, false>(tmk, tmv, p, stream, num_sms);
  if (p.G <= 16) return launch_decode_t<kBF16, D, 1, true>(tmk, tmv, p, stream, num_sms);
  if (p.G <= 32) return launch_decode_t<kBF16, D, 2, true>(tmk, tmv, p, stream, num_sms);
  return launch_decode_t<kBF16, D, 4, true>(tmk, tmv, p, stream, num_sms);
}

}  // namespace

int launch_combine(const CombineParams& p, bool bf16, int head_dim, cudaStream_t stream) {
  if (p.num_seqs <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  const int heads = p.num_heads < kCombineHeads ? p.num_heads : kCombineHeads;
  cfg.gridDim = dim3(p.num_seqs, (p.num_heads + kCombineHeads - 1) / kCombineHeads);
  cfg.blockDim = dim3(32 * heads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (bf16)
    e = head_dim == 64 ? cudaLaunchKernelEx(&cfg, combine_kernel<true, 64>, p)
                       : cudaLaunchKernelEx(&cfg, combine_kernel<true, 128>, p);
  else
    e = head_dim == 64 ? cudaLaunchKernelEx(&cfg, combine_kernel<false, 64>, p)
                       : cudaLaunchKernelEx(&cfg, combine_kernel<false, 128>, p);
  return e == cudaSuccess ? 1 : -1;
}

int launch_combine_equal_share(const CombineParams& p, bool bf16, int head_dim,
                               cudaStream_t stream) {
  if (p.num_seqs <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  const int heads = p.num_heads < kCombineHeads ? p.num_heads : kCombineHeads;
  cfg.gridDim = dim3(p.num_seqs, (p.num_heads + kCombineHeads - 1) / kCombineHeads);
  cfg.blockDim = dim3(32 * heads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (bf16)
    e = head_dim == 64 ? cudaLaunchKernelEx(&cfg, combine_equal_share_kernel<true, 64>, p)
                       : cudaLaunchKernelEx(&cfg, combine_equal_share_kernel<true, 128>, p);
  else
    e = head_dim == 64 ? cudaLaunchKernelEx(&cfg, combine_equal_share_kernel<false, 64>, p)
                       : cudaLaunchKernelEx(&cfg, combine_equal_share_kernel<false, 128>, p);
  return e == cudaSuccess ? 1 : -1;
}

int launch_decode(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                  bool bf16, int head_dim, cudaStream_t stream, int num_sms) {
  if (bf16) {
    return head_dim == 64 ? launch_decode_d<true, 64>(tmk, tmv, p, stream, num_sms)
                          : launch_decode_d<true, 128>(tmk, tmv, p, stream, num_sms);
  }
  return head_dim == 64 ? launch_decode_d<false, 64>(tmk, tmv, p, stream, num_sms)
                        : launch_decode_d<false, 128>(tmk, tmv, p, stream, num_sms);
}

}  // namespace pa
