// Chunked-prefill attention over the paged KV cache (query chunks with
// qlen > 1, causal within the chunk after a cached prefix), sm_103a.
//
// vLLM PR #14431 ("[Kernel][V1] Further optimizations to ROCm (Triton)
// Backend to better handle GQA") runs such chunks next to decode rows in one
// batch; vLLM issue #1880 asks for GQA kernels that share each KV head's
// blocks across its G query heads.  Here a tile packs the G query heads of
// one KV head times up to 64 / G consecutive query tokens as the 64 M rows
// (row r = token * G + head), so every K/V tile fetched from the cache feeds
// all of them.
//
// Structure: persistent CTAs of 4 MMA warps (16 rows each) + 1 producer
// warp.  The producer grabs tiles from the device work list, loads the Q
// tile with one 3-D TMA box per 64 columns (tokens x heads x dims lands as
// the packed rows, 128-byte swizzle) into one of two Q buffers, then streams
// the visible keys in 64-key stages (four 16-key TMA boxes per 64 columns,
// gathered through the block table) through an R-stage ring.  MMA warps do
// S = Q K^T and O += P V with mma.sync m16n8k16 (fp32 accumulation), the
// online softmax in base 2 with per-row running max/sum, and the
// bottom-right causal mask.
#include "pa_kernels.cuh"

namespace pa {

namespace {

constexpr int kPfConsumers = 4;
constexpr int kPfThreads = (kPfConsumers + 1) * 32;

struct TileMeta {
  int32_t tok0, ntok, pos0, kvh, nkv, done, b, pad;
};

template <int D, int R>
struct PrefillSmem {
  static constexpr int kBoxes = D / 64;
  static constexpr int kQBox = kPrefillRows * 128;         // 64 rows x 128 B
  static constexpr int kQ = kBoxes * kQBox;                // one Q buffer
  static constexpr int kSub = kBoxes * 2048;               // 16 keys of K (or V)
  static constexpr int kSubTiles = kPrefillKeys / 16;
  static constexpr int kStage = 2 * kSubTiles * kSub;      // K then V
  static constexpr int kRing = 2 * kQ + R * kStage;
  static constexpr int kBars = (2 * R + 4) * 8;
  static constexpr int kMeta = 2 * static_cast<int>(sizeof(TileMeta));
  static constexpr int kBytes = kRing + kBars + kMeta + 1024;
};

}  // namespace

template <bool kBF16, int D, int R>
__global__ void __launch_bounds__(kPfThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmq, const PrefillParams p) {
  using S = PrefillSmem<D, R>;
  constexpr int kKS = D / 16;  // k-steps of QK^T
  constexpr int kNT = D / 8;   // n-tiles of PV
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* qbuf = smem;                    // 2 x kQ
  uint8_t* kvbuf = smem + 2 * S::kQ;       // R x kStage
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRing);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + R;
  uint64_t* q_full = bars + 2 * R;
  uint64_t* q_empty = bars + 2 * R + 2;
  TileMeta* tmeta = reinterpret_cast<TileMeta*>(smem + S::kRing + S::kBars);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], kPfConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], kPfConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int G = p.G, Hq = p.num_heads, Hkv = p.num_kv_heads, bs = p.block_size;
  const int TQ = p.tokens_per_tile;
  uint32_t* status = &p.hdr->status;
  const uint32_t num_items = p.hdr->prefill_items;

  if (warp == kPfConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      tma_prefetch_desc(&tmq);
    }
    uint32_t q_iter = 0, kv_iter = 0;
    bool ok = true;
    while (ok) {
      uint32_t it = 0;
      if (lane == 0) it = atomicAdd(&p.hdr->prefill_grab, 1u);
      it = __shfl_sync(0xffffffffu, it, 0);
      const int qs = static_cast<int>(q_iter & 1);
      if (q_iter >= 2 && !mbar_wait(&q_empty[qs], ((q_iter >> 1) - 1) & 1)) {
        if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
        break;
      }
      if (it >= num_items) {
        if (lane == 0) {
          tmeta[qs].done = 1;
          mbar_arrive(&q_full[qs]);
        }
        ++q_iter;
        break;
      }
      const uint32_t ti = it / static_cast<uint32_t>(Hkv);
      const int kvh = static_cast<int>(it - ti * static_cast<uint32_t>(Hkv));
      const PfTile tile = p.tiles[ti];
      const int nkv = tile.pos0 + tile.ntok;  // keys 0 .. nkv - 1 are visible
      if (lane == 0) {
        TileMeta m;
        m.tok0 = tile.tok0;
        m.ntok = tile.ntok;
        m.pos0 = tile.pos0;
        m.kvh = kvh;
        m.nkv = nkv;
        m.done = 0;
        m.b = tile.b;
        m.pad = 0;
        tmeta[qs] = m;
        mbar_arrive_expect_tx(&q_full[qs], static_cast<uint32_t>(S::kBoxes * 128 * G * TQ));
#pragma unroll
        for (int bx = 0; bx < S::kBoxes; ++bx)
          tma_load_3d(qbuf + qs * S::kQ + bx * S::kQBox, &tmq, bx * 64, kvh * G, tile.tok0,
                      &q_full[qs]);
      }
      ++q_iter;

      // Keys in 64-key stages; physical blocks from the table, 32 at a time.
      int ids_base = -1000000, ids = -1;
      for (int kb = 0; kb < nkv; kb += kPrefillKeys) {
        const int s = static_cast<int>(kv_iter % R);
        if (kv_iter >= static_cast<uint32_t>(R) &&
            !mbar_wait(&kv_empty[s], ((kv_iter / R) - 1) & 1)) {
          if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
          ok = false;
          break;
        }
        int nsub = (nkv - kb + 15) / 16;
        if (nsub > S::kSubTiles) nsub = S::kSubTiles;
        int blks[S::kSubTiles];
#pragma unroll
        for (int j = 0; j < S::kSubTiles; ++j) {
          const int key = kb + 16 * j;
          const int lblk = key / bs;
          if (lblk - ids_base >= 32 || lblk < ids_base) {
            ids_base = lblk;
            const int lb = lblk + lane;
            ids = (lb * bs < nkv)
                      ? __ldg(p.block_tables + static_cast<int64_t>(tile.b) * p.mbs + lb)
                      : -1;
          }
          int blk = __shfl_sync(0xffffffffu, ids, lblk - ids_base);
          if (j < nsub && (blk < 0 || blk >= p.num_blocks)) {
            if (lane == 0) Status::raise(status, PA_DEV_BAD_BLOCK_ID);
            blk = 0;  // in-range stand-in; the bad tile's keys still count
          }
          blks[j] = blk;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&kv_full[s], static_cast<uint32_t>(nsub * 2 * S::kSub));
          uint8_t* st = kvbuf + s * S::kStage;
          for (int j = 0; j < nsub; ++j) {
            const int key = kb + 16 * j;
            const int y = (blks[j] * Hkv + kvh) * bs + (key % bs);
#pragma unroll
            for (int bx = 0; bx < S::kBoxes; ++bx) {
              tma_load_2d(st + j * S::kSub + bx * 2048, &tmk, bx * 64, y, &kv_full[s]);
              tma_load_2d(st + (S::kSubTiles + j) * S::kSub + bx * 2048, &tmv, bx * 64, y,
                          &kv_full[s]);
            }
          }
        }
        ++kv_iter;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, q4 = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;
  const int row0 = warp * 16 + g, row1 = row0 + 8;  // rows of this lane
  const int rows_used = G * TQ;
  uint32_t c_q = 0, c_kv = 0;
  while (true) {
    const int qs = static_cast<int>(c_q & 1);
    if (!mbar_wait(&q_full[qs], (c_q >> 1) & 1)) {
      if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
      break;
    }
    const TileMeta tm = tmeta[qs];
    if (tm.done) break;

    // Q A-fragments for this warp's 16 rows, then release the Q buffer.
    uint32_t qa[kKS][4];
    const uint32_t qb = smem_u32(qbuf + qs * S::kQ);
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      const int row = warp * 16 + rr + ((mi & 1) << 3);
      const int chunk = ((ks & 3) << 1) + (mi >> 1);
      ldsm_x4(qb + (ks >> 2) * S::kQBox + swz128(row, chunk), qa[ks]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[qs]);
    ++c_q;

    // Row positions (bottom-right causal); rows past the tile never store.
    const int t0 = row0 / G, t1 = row1 / G;
    const bool v0 = row0 < rows_used && t0 < tm.ntok;
    const bool v1 = row1 < rows_used && t1 < tm.ntok;
    const int pos_r0 = tm.pos0 + t0, pos_r1 = tm.pos0 + t1;

    float o[kNT][4];
#pragma unroll
    for (int i = 0; i < kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    bool ok = true;
    for (int kb = 0; kb < tm.nkv; kb += kPrefillKeys) {
      const int s = static_cast<int>(c_kv % R);
      if (!mbar_wait(&kv_full[s], (c_kv / R) & 1)) {
        if (lane == 0) Status::raise(status, PA_DEV_WAIT_TIMEOUT);
        ok = false;
        break;
      }
      const uint32_t kst = smem_u32(kvbuf + s * S::kStage);
      const uint32_t vst = kst + S::kSubTiles * S::kSub;
      const int nvalid = tm.nkv - kb;  // keys of this stage that exist (may be > 64)

      // S = Q K^T over 64 keys: 8 n-tiles of 8 keys.
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
      for (int j = 0; j < S::kSubTiles; ++j) {
        if (16 * j < nvalid) {
#pragma unroll
          for (int ks = 0; ks < kKS; ++ks) {
            const int key = rr + ((mi >> 1) << 3);
            const int chunk = ((ks & 3) << 1) + (mi & 1);
            uint32_t b[4];
            ldsm_x4(kst + j * S::kSub + (ks >> 2) * 2048 + swz128(key, chunk), b);
            mma_16816<kBF16>(sc[2 * j], qa[ks], b[0], b[1]);
            mma_16816<kBF16>(sc[2 * j + 1], qa[ks], b[2], b[3]);
          }
        }
      }

      // Scale, mask (key > row position, or key past the visible range).
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kb + nt * 8 + 2 * q4 + e;
          float x0 = sc[nt][e] * p.scale_log2;
          float x1 = sc[nt][2 + e] * p.scale_log2;
          if (key > pos_r0 || key >= tm.nkv) x0 = -INFINITY;
          if (key > pos_r1 || key >= tm.nkv) x1 = -INFINITY;
          sc[nt][e] = x0;
          sc[nt][2 + e] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
      const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = ex2(m0 - ref0), al1 = ex2(m1 - ref1);
      m0 = mn0;
      m1 = mn1;

      // P in the element type (A operand of PV); row sums from the rounded P.
      uint32_t pa[4][4];
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int nt = 2 * j + h;
          const uint32_t top = pack2<kBF16>(ex2(sc[nt][0] - ref0), ex2(sc[nt][1] - ref0));
          const uint32_t bot = pack2<kBF16>(ex2(sc[nt][2] - ref1), ex2(sc[nt][3] - ref1));
          float a, b2, c, d;
          unpack2<kBF16>(top, a, b2);
          unpack2<kBF16>(bot, c, d);
          rs0 += a + b2;
          rs1 += c + d;
          pa[j][2 * h] = top;
          pa[j][2 * h + 1] = bot;
        }
      }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        o[nt][0] *= al0;
        o[nt][1] *= al0;
        o[nt][2] *= al1;
        o[nt][3] *= al1;
      }

      // O += P V, 16 keys per k-step.
#pragma unroll
      for (int j = 0; j < S::kSubTiles; ++j) {
        if (16 * j < nvalid) {
          const int kv_lo = nvalid - 16 * j;  // valid keys in this sub-tile
          const uint32_t vm_lo = keep_mask(2 * q4 < kv_lo, 2 * q4 + 1 < kv_lo);
          const uint32_t vm_hi = keep_mask(8 + 2 * q4 < kv_lo, 9 + 2 * q4 < kv_lo);
#pragma unroll
          for (int np = 0; np < kNT / 2; ++np) {
            const int key = rr + ((mi & 1) << 3);
            const int chunk = ((np & 3) << 1) + (mi >> 1);
            uint32_t b[4];
            ldsm_x4_t(vst + j * S::kSub + (np >> 2) * 2048 + swz128(key, chunk), b);
            if (kv_lo < 16) {
              b[0] &= vm_lo;
              b[1] &= vm_hi;
              b[2] &= vm_lo;
              b[3] &= vm_hi;
            }
            mma_16816<kBF16>(o[2 * np], pa[j], b[0], b[1]);
            mma_16816<kBF16>(o[2 * np + 1], pa[j], b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&kv_empty[s]);
      ++c_kv;
    }
    if (!ok) break;

    // Epilogue: normalise and store the valid rows.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float il0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float il1 = l1 > 0.f ? 1.f / l1 : 0.f;
    uint16_t* out = static_cast<uint16_t*>(p.out);
    const int64_t orow0 =
        (static_cast<int64_t>(tm.tok0 + t0) * Hq + static_cast<int64_t>(tm.kvh) * G + row0 % G) * D;
    const int64_t orow1 =
        (static_cast<int64_t>(tm.tok0 + t1) * Hq + static_cast<int64_t>(tm.kvh) * G + row1 % G) * D;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int d = nt * 8 + 2 * q4;
      if (v0)
        *reinterpret_cast<uint32_t*>(out + orow0 + d) =
            pack2<kBF16>(o[nt][0] * il0, o[nt][1] * il0);
      if (v1)
        *reinterpret_cast<uint32_t*>(out + orow1 + d) =
            pack2<kBF16>(o[nt][2] * il1, o[nt][3] * il1);
    }
  }
}

// ---------------------------------------------------------------- launcher
namespace {

template <bool kBF16, int D>
int launch_prefill_t(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                     const PrefillParams& p, int64_t max_items, cudaStream_t stream,
                     int num_sms) {
  constexpr int R = 2;
  using S = PrefillSmem<D, R>;
  static_assert(S::kBytes <= 113 * 1024, "two CTAs per SM");
  auto kern = prefill_kernel<kBF16, D, R>;
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes) !=
        cudaSuccess)
      return -1;
    configured = dev;
  }
  int64_t grid = static_cast<int64_t>(num_sms) * 2;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  kern<<<static_cast<unsigned>(grid), kPfThreads, S::kBytes, stream>>>(tmk, tmv, tmq, p);
  return 1;
}

}  // namespace

int launch_prefill(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                   const PrefillParams& p, bool bf16, int head_dim, int64_t max_items,
                   cudaStream_t stream, int num_sms) {
  if (bf16)
    return head_dim == 64 ? launch_prefill_t<true, 64>(tmk, tmv, tmq, p, max_items, stream, num_sms)
                          : launch_prefill_t<true, 128>(tmk, tmv, tmq, p, max_items, stream, num_sms);
  return head_dim == 64 ? launch_prefill_t<false, 64>(tmk, tmv, tmq, p, max_items, stream, num_sms)
                        : launch_prefill_t<false, 128>(tmk, tmv, tmq, p, max_items, stream, num_sms);
}

}  // namespace pa
