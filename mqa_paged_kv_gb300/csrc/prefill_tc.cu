// Chunked-prefill attention over the paged KV cache on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), sm_103a.
//
// vLLM PR #14431 ("[Kernel][V1] Further optimizations to ROCm (Triton)
// Backend to better handle GQA") runs query chunks (qlen > 1, causal within
// the chunk after a cached prefix) next to decode rows; vLLM issue #1880
// ("[Performance] Use optimized kernels for MQA/GQA", opening paragraph) asks
// that the G query heads sharing a KV head share its cache reads and do the
// dot products on tensor cores.  A Q tile packs those G heads times 128 / G
// consecutive query tokens as the M = 128 rows of the MMA (row r = token * G
// + head), and each CTA works on two such tiles (A: the first 128 / G
// tokens, B: the next) of one sequence and KV head, so every 64-key K/V
// stage gathered from the cache feeds 256 rows.
//
// Warp roles (one CTA per SM, persistent over a device tile list):
//   warp 0     TMA producer: the two Q tiles (one 3-D box per 64 columns
//              each), then the visible keys in 64-key stages through a
//              5-deep ring; a stage is 16-key boxes gathered through the
//              block table, one box per lane, issued by one instruction;
//   warp 1     MMA issuer (one thread): S_t = Q_t K^T into tensor memory
//              (two S buffers per tile), O_t += P_t V with P_t read from
//              tensor memory (O in tensor memory);
//   warps 2-9  softmax, four warps per tile, one thread per row (= TMEM
//              lane): scale, bottom-right causal mask, running max,
//              P = 2^(x*scale - m) in the element type written back over
//              its own S buffer in tensor memory (so shared memory holds
//              only Q and the K/V ring), fp32 row sum, and the epilogue O / l.
// The running max is a reference that only moves when a row max exceeds it
// by more than 2^8 (then O and l are rescaled in place); between moves P
// stays below 256, well inside the element type.  Row maxima run over raw
// scores in eight independent chains and the scale is folded into the
// exponent's FMA, so the scale must be positive.
#include "pa_kernels.cuh"

namespace pa {

namespace {

constexpr int kTcRows = 128;              // M of one tile
constexpr int kTcKeys = 64;               // keys per stage
constexpr int kTcSub = kTcKeys / 16;      // 16-key boxes per stage
constexpr int kTcStages = 5;              // K/V ring depth
constexpr int kTcSoftmaxWarps = 8;
constexpr int kTcThreads = (2 + kTcSoftmaxWarps) * 32;
constexpr float kRescaleThreshold = 8.f;  // log2 of the largest unnormalised P

struct TcMeta {
  int32_t tok0, ntok, pos0, kvh, nkv, done, b, pad;
};

enum : int {
  kBarQFull = 0,
  kBarQEmpty,
  kBarKvFull,                              // [stages]
  kBarKvEmpty = kBarKvFull + kTcStages,    // [stages]
  kBarSFull = kBarKvEmpty + kTcStages,     // [tile][buffer]
  kBarPFull = kBarSFull + 4,               // [tile][buffer]
  kBarPvDone = kBarPFull + 4,              // [tile][buffer]
  kBarOFull = kBarPvDone + 4,              // [tile]
  kBarOEmpty = kBarOFull + 2,              // [tile]
  kNumBars = kBarOEmpty + 2
};

template <int D>
struct TcSmem {
  static constexpr int kBoxes = D / 64;            // 64-column halves
  static constexpr int kQRegion = 128 * 128;       // 128 rows x 128 B
  static constexpr int kQ = kBoxes * kQRegion;     // one Q tile
  static constexpr int kKVRegion = kTcKeys * 128;  // 64 keys x 128 B
  static constexpr int kKV = kBoxes * kKVRegion;   // 64 keys of K (or V)
  static constexpr int kStage = 2 * kKV;
  static constexpr int kOffKV = 2 * kQ;
  static constexpr int kOffBar = kOffKV + kTcStages * kStage;
  static constexpr int kOffMeta = kOffBar + kNumBars * 8;
  static constexpr int kOffTmem = kOffMeta + static_cast<int>(sizeof(TcMeta));
  static constexpr int kBytes = kOffTmem + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // tile t, buffer b: S (fp32, 64 columns) at t*128 + b*64, later P (16-bit
  // pairs, its first 32 columns); O_t at 256 + t*128
  static constexpr uint32_t col_s(int t, int b) {
    return static_cast<uint32_t>(t * 128 + b * 64);
  }
  static constexpr uint32_t col_o(int t) { return static_cast<uint32_t>(256 + t * 128); }
};

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_wait(bar, parity)) return true;
  Status::raise(status, PA_DEV_WAIT_TIMEOUT);
  return false;
}

// Warp-uniform form: every lane polls and the lanes agree on the outcome,
// so a timeout seen by only some lanes cannot split the warp before the
// warp-wide (elect.sync) MMA issue.
__device__ __forceinline__ bool warp_wait_or_flag(uint64_t* bar, uint32_t parity,
                                                  uint32_t* status) {
  return __all_sync(0xffffffffu, wait_or_flag(bar, parity, status));
}

}  // namespace

template <bool kBF16, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmq, const PrefillParams p) {
  using S = TcSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sq = smem;
  uint8_t* skv = smem + S::kOffKV;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  TcMeta* meta = reinterpret_cast<TcMeta*>(smem + S::kOffMeta);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffTmem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[kBarQFull], 1);
    mbar_init(&bar[kBarQEmpty], 1 + kTcSoftmaxWarps);  // MMA commit + meta reads
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&bar[kBarKvFull + i], 1);
      mbar_init(&bar[kBarKvEmpty + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bar[kBarSFull + i], 1);
      mbar_init(&bar[kBarPFull + i], 4);
      mbar_init(&bar[kBarPvDone + i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar[kBarOFull + t], 1);
      mbar_init(&bar[kBarOEmpty + t], 4);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, S::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the tile list is written by the preceding kernel

  const int G = p.G, Hq = p.num_heads, Hkv = p.num_kv_heads, bs = p.block_size;
  const int TQ = p.tokens_per_tile / 2;  // tokens of one of the two Q tiles
  uint32_t* status = &p.hdr->status;
  const uint32_t num_items = p.hdr->prefill_items;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      tma_prefetch_desc(&tmq);
    }
    const int oob_row = p.num_blocks * Hkv * bs;  // a box here reads zeros
    constexpr int nb = kTcSub * S::kBoxes;        // K boxes per stage (= V boxes)
    static_assert(2 * nb <= 32, "one box per lane");
    const bool is_v = lane >= nb;
    const int box = is_v ? lane - nb : lane;
    const int my_j = box / S::kBoxes, my_bx = box % S::kBoxes;
    uint32_t t_iter = 0, g = 0;
    bool ok = true;
    while (ok) {
      uint32_t it = 0;
      if (lane == 0) it = atomicAdd(&p.hdr->prefill_grab, 1u);
      it = __shfl_sync(0xffffffffu, it, 0);
      if (t_iter > 0 && !warp_wait_or_flag(&bar[kBarQEmpty], (t_iter - 1) & 1, status)) break;
      if (it >= num_items) {
        if (lane == 0) {
          meta->done = 1;
          mbar_arrive(&bar[kBarQFull]);
        }
        break;
      }
      const uint32_t ti = it / static_cast<uint32_t>(Hkv);
      const int kvh = static_cast<int>(it - ti * static_cast<uint32_t>(Hkv));
      const PfTile tile = p.tiles[ti];
      const int nkv = tile.pos0 + tile.ntok;
      if (lane == 0) {
        TcMeta m;
        m.tok0 = tile.tok0;
        m.ntok = tile.ntok;
        m.pos0 = tile.pos0;
        m.kvh = kvh;
        m.nkv = nkv;
        m.done = 0;
        m.b = tile.b;
        m.pad = 0;
        *meta = m;
        mbar_arrive_expect_tx(&bar[kBarQFull],
                              static_cast<uint32_t>(2 * S::kBoxes * 128 * G * TQ));
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int bx = 0; bx < S::kBoxes; ++bx)
            tma_load_3d(sq + t * S::kQ + bx * S::kQRegion, &tmq, bx * 64, kvh * G,
                        tile.tok0 + t * TQ, &bar[kBarQFull]);
      }
      ++t_iter;

      // Physical block ids, 32 per window held one per lane; the next window
      // is loaded while the current one is in use.
      auto load_window = [&](int lblk0) -> int {
        const int lb = lblk0 + lane;
        return (lb * bs < nkv)
                   ? __ldg(p.block_tables + static_cast<int64_t>(tile.b) * p.mbs + lb)
                   : -1;
      };
      int ids_base = 0;
      int ids = load_window(0);
      int ids_next = load_window(32);
      int lblk = 0, off = 0;  // block and slot of the next 16-key box
      for (int kb = 0; kb < nkv; kb += kTcKeys, ++g) {
        const int st = static_cast<int>(g % kTcStages);
        if (g >= kTcStages &&
            !warp_wait_or_flag(&bar[kBarKvEmpty + st], ((g / kTcStages) - 1) & 1, status)) {
          ok = false;
          break;
        }
        int my_row = oob_row;
#pragma unroll
        for (int j = 0; j < kTcSub; ++j) {
          const int key = kb + 16 * j;
          if (key < nkv && lblk - ids_base >= 32) {  // windows advance in order
            ids_base += 32;
            ids = ids_next;
            ids_next = load_window(ids_base + 32);
          }
          int blk = __shfl_sync(0xffffffffu, ids, (lblk - ids_base) & 31);
          if (key < nkv && (blk < 0 || blk >= p.num_blocks)) {
            if (lane == 0) Status::raise(status, PA_DEV_BAD_BLOCK_ID);
            blk = -1;
          }
          const int row = (key < nkv && blk >= 0) ? (blk * Hkv + kvh) * bs + off : oob_row;
          if (j == my_j) my_row = row;
          off += 16;
          if (off == bs) {
            off = 0;
            ++lblk;
          }
        }
        if (lane == 0)
          mbar_arrive_expect_tx(&bar[kBarKvFull + st], static_cast<uint32_t>(S::kStage));
        __syncwarp();
        if (lane < 2 * nb) {
          uint8_t* dst = skv + st * S::kStage + (is_v ? S::kKV : 0) + my_bx * S::kKVRegion +
                         my_j * 2048;
          tma_load_2d(dst, is_v ? &tmv : &tmk, my_bx * 64, my_row, &bar[kBarKvFull + st]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this branch and waits on the barriers together;
    // elect.sync inside each MMA picks the issuing lane.  Each group of MMAs
    // is straight-line code on descriptors prepared up front: the tensor
    // pipe is fed at its full rate only when no branch or runtime trip count
    // sits between two tcgen05.mma (measured on this part: a
    // data-independent branch inside the issue loop halves the rate).
    //
    // Issue order per step j: QK_0(j), PV_0(j-1), QK_1(j), PV_1(j-1).  The
    // tiles alternate, so every barrier a group waits on was armed at least
    // one group earlier: S buffer reuse (QK_t(j) after PV_t(j-2)) has twelve
    // MMAs of slack, and the softmax of tile t on stage j-1 runs while the
    // pipe works on the other tile.
    constexpr uint32_t kIdQK = idesc_f16(kTcRows, kTcKeys, kBF16, false, false);
    constexpr uint32_t kIdPV = idesc_f16(kTcRows, D, kBF16, false, true);
    constexpr int kQkSteps = D / 16;
    // Adding (byte offset >> 4) to a descriptor moves its start address; the
    // 14-bit field cannot carry because shared-memory offsets stay below
    // 256 KB.
    const uint64_t dq = sdesc_sw128(smem_u32(sq), 16, 1024);
    const uint64_t dk = sdesc_sw128(smem_u32(skv), 16, 1024);
    const uint64_t dv = sdesc_sw128(smem_u32(skv) + S::kKV, S::kKVRegion, 1024);
    uint32_t t_iter = 0, g0 = 0;
    bool ok = true;
    while (ok) {
      if (!warp_wait_or_flag(&bar[kBarQFull], t_iter & 1, status)) break;
      const TcMeta m = *meta;
      __syncwarp();
      if (m.done) break;
      const int n = (m.nkv + kTcKeys - 1) / kTcKeys;
      tc_fence_after();

      for (int j = 0; j <= n && ok; ++j) {
        const uint32_t g = g0 + j;  // stage of the QK groups
        const int st = static_cast<int>(g % kTcStages);
        const int b = static_cast<int>(g & 1);
        const uint32_t gp = g - 1;  // stage of the PV groups
        const int stp = static_cast<int>(gp % kTcStages);
        const int pb = static_cast<int>(gp & 1);
        if (j < n && !warp_wait_or_flag(&bar[kBarKvFull + st], (g / kTcStages) & 1, status)) {
          ok = false;
          break;
        }
        const uint64_t dks = dk + static_cast<uint64_t>((st * S::kStage) >> 4);
        const uint64_t dvs = dv + static_cast<uint64_t>((stp * S::kStage) >> 4);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j < n) {
            // S/P buffer b of tile t was last read by PV of stage g - 2.
            if (g >= 2 &&
                !warp_wait_or_flag(&bar[kBarPvDone + 2 * t + b], ((g >> 1) - 1) & 1, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + S::col_s(t, b);
#pragma unroll
            for (int ks = 0; ks < kQkSteps; ++ks)
              umma_f16_warp(d, dq + ((t * S::kQ + (ks >> 2) * S::kQRegion + (ks & 3) * 32) >> 4),
                            dks + (((ks >> 2) * S::kKVRegion + (ks & 3) * 32) >> 4), kIdQK,
                            ks > 0 ? 1u : 0u);
            umma_commit_warp(&bar[kBarSFull + 2 * t + b]);
            if (t == 1 && j == n - 1) umma_commit_warp(&bar[kBarQEmpty]);
          }
          if (j >= 1) {
            // All four 16-key steps run on every stage: past the sequence P
            // is 0 and the V rows are zero (zero-filled boxes, or zeroed by
            // the softmax warps inside the last box).
            if (!warp_wait_or_flag(&bar[kBarPFull + 2 * t + pb], (gp >> 1) & 1, status) ||
                (j == 1 && t_iter > 0 &&
                 !warp_wait_or_flag(&bar[kBarOEmpty + t], (t_iter - 1) & 1, status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + S::col_o(t), a = tmem + S::col_s(t, pb);
            umma_f16_ts_warp(d, a, dvs, kIdPV, j > 1 ? 1u : 0u);
#pragma unroll
            for (int ks = 1; ks < kTcSub; ++ks)
              umma_f16_ts_warp(d, a + ks * 8, dvs + ((ks * 2048) >> 4), kIdPV, 1u);
            umma_commit_warp(&bar[kBarPvDone + 2 * t + pb]);
            if (t == 1) umma_commit_warp(&bar[kBarKvEmpty + stp]);
            if (j == n) umma_commit_warp(&bar[kBarOFull + t]);
          }
        }
      }
      g0 += n;
      ++t_iter;
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) / 4;    // Q tile of this warp
    const int quarter = warp & 3;    // TMEM lanes 32*quarter ..
    const int row = 32 * quarter + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    const int rows_used = G * TQ;
    uint32_t t_iter = 0, g0 = 0;
    while (true) {
      if (!warp_wait_or_flag(&bar[kBarQFull], t_iter & 1, status)) break;
      const TcMeta m = *meta;
      __syncwarp();
      if (m.done) break;
      if (lane == 0) mbar_arrive(&bar[kBarQEmpty]);
      const int tl = t * TQ + row / G;  // token within the pair
      const bool valid = row < rows_used && tl < m.ntok;
      const int pos = m.pos0 + tl;
      const int n = (m.nkv + kTcKeys - 1) / kTcKeys;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t g = g0 + j;
        const int b = static_cast<int>(g & 1);
        if (!warp_wait_or_flag(&bar[kBarSFull + 2 * t + b], (g >> 1) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float x[kTcKeys];
        tmem_ld64f(lane_base + S::col_s(t, b), x);

        const int kb = j * kTcKeys;
        const int lim = min(pos, m.nkv - 1) - kb;  // last visible column of this row
        if (__any_sync(0xffffffffu, lim < kTcKeys - 1)) {
#pragma unroll
          for (int i = 0; i < kTcKeys; ++i)
            if (i > lim) x[i] = -INFINITY;
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = x[e];
#pragma unroll
        for (int i = 8; i < kTcKeys; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], x[i]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                         p.scale_log2;
        const bool need = m_ref != -INFINITY && mx > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O_t must hold PV of stage g - 1 before it is rescaled.
          const uint32_t gp = g - 1;
          if (!warp_wait_or_flag(&bar[kBarPvDone + 2 * t + (gp & 1)], (gp >> 1) & 1, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? ex2(m_ref - mx) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(lane_base + S::col_o(t) + c * 16, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st16(lane_base + S::col_o(t) + c * 16, r);
          }
          tmem_wait_st();
          if (need) {
            l *= alpha;
            m_ref = mx;
          }
        }
        if (m_ref == -INFINITY) m_ref = mx;
        const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;

        // P row into tensor memory over its S: column c holds keys 2c, 2c+1.
        float rs8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rs8[e] = 0.f;
        uint32_t w[kTcKeys / 2];
#pragma unroll
        for (int c = 0; c < kTcKeys / 2; ++c) {
          const float p0 = ex2(fmaf(x[2 * c], p.scale_log2, neg_ref));
          const float p1 = ex2(fmaf(x[2 * c + 1], p.scale_log2, neg_ref));
          rs8[(2 * c) & 7] += p0;
          rs8[(2 * c + 1) & 7] += p1;
          w[c] = pack2<kBF16>(p0, p1);
        }
        tmem_st32(lane_base + S::col_s(t, b), w);
        l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));

        // Keys past the sequence inside the last loaded 16-key box hold
        // whatever the cache slots hold: zero those V rows (P is 0 there,
        // but 0 * NaN is not).  Both tiles' warps write the same zeros.
        if (j == n - 1) {
          const int r0 = m.nkv - kb;
          const int r1 = min(kTcKeys, (r0 + 15) / 16 * 16);
          if (r1 > r0) {
            const int st = static_cast<int>(g % kTcStages);
            if (!warp_wait_or_flag(&bar[kBarKvFull + st], (g / kTcStages) & 1, status)) {
              ok = false;
              break;
            }
            uint8_t* vst = skv + st * S::kStage + S::kKV;
            const int per_row = S::kBoxes * 8;  // 16-byte chunks per key row
            const int total = (r1 - r0) * per_row;
            for (int i = row; i < total; i += 128) {
              const int kr = r0 + i / per_row, c = i % per_row;
              *reinterpret_cast<uint4*>(vst + (c >> 3) * S::kKVRegion + kr * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
        }
        if (j == n - 1) fence_proxy_async();  // the V rows zeroed above
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarPFull + 2 * t + b]);
      }
      if (!ok) break;

      // Epilogue: O_t / l for the valid rows.
      if (!warp_wait_or_flag(&bar[kBarOFull + t], t_iter & 1, status)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = static_cast<uint16_t*>(p.out) +
                       (static_cast<int64_t>(m.tok0 + tl) * Hq + static_cast<int64_t>(m.kvh) * G +
                        row % G) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + S::col_o(t) + c * 32, r);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = pack2<kBF16>(__uint_as_float(r[8 * q + 0]) * inv,
                               __uint_as_float(r[8 * q + 1]) * inv);
            o.y = pack2<kBF16>(__uint_as_float(r[8 * q + 2]) * inv,
                               __uint_as_float(r[8 * q + 3]) * inv);
            o.z = pack2<kBF16>(__uint_as_float(r[8 * q + 4]) * inv,
                               __uint_as_float(r[8 * q + 5]) * inv);
            o.w = pack2<kBF16>(__uint_as_float(r[8 * q + 6]) * inv,
                               __uint_as_float(r[8 * q + 7]) * inv);
            reinterpret_cast<uint4*>(orow + c * 32)[q] = o;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarOEmpty + t]);
      g0 += n;
      ++t_iter;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, S::kTmemCols);
}

namespace {

template <bool kBF16, int D>
int launch_prefill_tc_t(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                        const PrefillParams& p, int64_t max_items, cudaStream_t stream,
                        int num_sms) {
  using S = TcSmem<D>;
  static_assert(S::kBytes <= 227 * 1024, "one CTA per SM");
  auto kern = prefill_tc_kernel<kBF16, D>;
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes) !=
        cudaSuccess)
      return -1;
    configured = dev;
  }
  int64_t grid = num_sms;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = S::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, tmq, p) == cudaSuccess ? 1 : -1;
}

}  // namespace

int launch_prefill_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                      const PrefillParams& p, bool bf16, int head_dim, int64_t max_items,
                      cudaStream_t stream, int num_sms) {
  if (bf16)
    return head_dim == 64
               ? launch_prefill_tc_t<true, 64>(tmk, tmv, tmq, p, max_items, stream, num_sms)
               : launch_prefill_tc_t<true, 128>(tmk, tmv, tmq, p, max_items, stream, num_sms);
  return head_dim == 64
             ? launch_prefill_tc_t<false, 64>(tmk, tmv, tmq, p, max_items, stream, num_sms)
             : launch_prefill_tc_t<false, 128>(tmk, tmv, tmq, p, max_items, stream, num_sms);
}

}  // namespace pa
