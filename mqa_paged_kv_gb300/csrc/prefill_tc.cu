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
// + head), and each CTA works on two such tiles (0: the first 128 / G
// tokens, 1: the next) of one sequence and KV head, so every 64-key K/V
// stage gathered from the cache feeds 256 rows.
//
// Warp roles (one CTA per SM, persistent over a device tile list):
//   warps 0, 3 TMA producers (0: the item records, the two Q tiles -- one
//              3-D box per 64 columns each -- and K; 3: V): the visible
//              keys in 64-key stages through one ring of slots, in the
//              order the MMAs consume them (K0, K1, V0, K2, V1, ...); a slot
//              is boxes of gcd(block_size, 64) keys gathered through the
//              block table, one box per lane, issued by one instruction;
//   warps 1-2  MMA issuers, one per tile: S_t = Q_t K^T (M 128, N 64)
//              into one of two S buffers in tensor memory, O_t += P_t V
//              with P_t read from tensor memory (O in tensor memory);
//   warps 4-11 softmax, four warps per tile, one thread per row (= TMEM
//              lane): scale, bottom-right causal mask, running max,
//              P = 2^(x*scale - m) in the element type written over the
//              first half of its own S buffer in tensor memory, fp32 row
//              sum, and the epilogue O / l.
// Tensor memory holds two 64-column S buffers per tile and O_0, O_1, so the
// QK of the next stage runs while the softmax works on the current one.
// The running max is a reference that only moves when a row max exceeds it
// by more than 2^8 (then O and l are rescaled in place); between moves P
// stays below 256, well inside the element type.  Row maxima run over raw
// scores in eight independent chains and the scale is folded into the
// exponent's FMA, so the scale must be positive.
#include "pa_kernels.cuh"

namespace pa {

namespace {

constexpr int kTcRows = 128;              // M of one tile
constexpr int kTcKeys = 64;               // keys per stage: N of QK, K of PV
constexpr int kTcSub = kTcKeys / 16;      // 16-key boxes per slot; PV K-steps
constexpr int kTcSoftmaxWarps = 8;
// warp 0 the K producer, warps 1-2 the MMA issuers, warp 3 the V producer;
// with the softmax warps after them every SM sub-partition (warp % 4) holds
// one of these four and one softmax warp of each tile.  Warps 12 and 13
// help the K and V producers: each issues the second half of every slot's
// boxes when a slot takes four or more (keys gathered in boxes of 16 or 32
// rows, where the per-warp issue rate of small boxes limits the stage).
constexpr int kTcVProducerWarp = 3;
constexpr int kTcFirstSoftmaxWarp = 4;
constexpr int kTcKHelperWarp = kTcFirstSoftmaxWarp + kTcSoftmaxWarps;
constexpr int kTcVHelperWarp = kTcKHelperWarp + 1;
constexpr int kTcThreads = (kTcVHelperWarp + 1) * 32;
constexpr float kRescaleThreshold = 8.f;  // log2 of the largest unnormalised P

struct TcMeta {
  int32_t tok0, ntok, pos0, kvh, nkv, done, b, kbase;
};

enum : int {
  kBarQFull = 0,                // [buffer]: the item's record and Q tiles are in place
  kBarBufFree = kBarQFull + 2,  // [buffer]: its record read, its output rows copied out
  kBarMetaFull = kBarBufFree + 2,  // [buffer]: the item's record is written
  kBarSFull = kBarMetaFull + 2,  // [tile][buffer]
  kBarPFull = kBarSFull + 4,  // [tile][buffer]
  kBarPvDone = kBarPFull + 4, // [tile][buffer]
  kBarOFull = kBarPvDone + 4, // [tile]
  kBarOEmpty = kBarOFull + 2, // [tile]
  kBarStaged = kBarOEmpty + 2, // [tile]: the tile's output rows are in shared memory
  kBarSlotFull = kBarStaged + 2  // [slot], then [slot] of empties
};

template <int D>
struct TcCfg {
  static constexpr int kBoxes = D / 64;              // 64-column halves
  static constexpr int kQRegion = 128 * 128;         // 128 rows x 128 B
  static constexpr int kQ = kBoxes * kQRegion;       // one Q tile
  static constexpr int kRegion = kTcKeys * 128;      // 64 keys x 128 B
  static constexpr int kSlot = kBoxes * kRegion;     // 64 keys of K or of V
  static constexpr int kSlots = D == 128 ? 6 : 16;   // ring depth
  static constexpr int kBarSlotEmpty = kBarSlotFull + kSlots;
  static constexpr int kNumBars = kBarSlotEmpty + kSlots;
  static constexpr int kOffRing = 2 * kQ;
  // Output staging of a tile: its 128 rows of D element-type values in the
  // Q tile's layout, so that one tensor store can take a tile out.
  // Two buffers of two Q tiles each take turns: item i loads its Q tiles
  // into buffer i mod 2 and, once its MMAs are done, stages its output
  // rows there over them, so the next item's Q tiles load into the other
  // buffer while item i still runs.
  static constexpr int kStageTile = kTcRows * D * 2;
  static_assert(kStageTile == kQ, "a tile's output rows fit over its Q tile");
  static constexpr int kOffStage = kOffRing + kSlots * kSlot;
  static constexpr int kOffBar = kOffStage + 2 * kStageTile;
  static constexpr int kOffMeta = kOffBar + kNumBars * 8;
  static constexpr int kOffTmem = kOffMeta + 2 * static_cast<int>(sizeof(TcMeta));
  static constexpr int kBytes = kOffTmem + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // S buffer b of tile t (fp32, 64 columns) at t * 128 + b * 64, later P
  // (16-bit pairs) over its first 32 columns; O_t at 256 + t * D.
  static constexpr uint32_t col_s(int t, int b) { return static_cast<uint32_t>(t * 128 + b * 64); }
  static constexpr uint32_t col_o(int t) { return static_cast<uint32_t>(256 + t * D); }
};

// Ring positions, relative to the first load of a work item with n stages:
// K(0), then K(j), V(j - 1) for j = 1 .. n - 1, then V(n - 1).
__device__ __forceinline__ uint32_t kpos(int j) {
  return j == 0 ? 0u : static_cast<uint32_t>(2 * j - 1);
}
__device__ __forceinline__ uint32_t vpos(int j, int n) {
  return static_cast<uint32_t>(j == n - 1 ? 2 * n - 1 : 2 * j + 2);
}

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_wait(bar, parity)) return true;
  Status::raise(status, PA_DEV_WAIT_TIMEOUT);
  return false;
}

// Warp-uniform form: every lane polls and the lanes agree on the outcome,
// so a timeout seen by only some lanes cannot split the warp ahead of
// warp-synchronous instructions (elect.sync issue, tcgen05.ld/st).
__device__ __forceinline__ bool warp_wait_or_flag(uint64_t* bar, uint32_t parity,
                                                  uint32_t* status) {
  return __all_sync(0xffffffffu, wait_or_flag(bar, parity, status));
}

}  // namespace

// Fourteen warps at 120 registers a thread (no spills) hold 53.8 K of the
// SM's 64 K registers, so that a CTA fits beside one CTA of the cache write
// it follows and becomes resident while that kernel still runs.
template <bool kBF16, int D, bool kVarlen>
__global__ void __maxnreg__(120)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmo, const PrefillParams p) {
  using C = TcCfg<D>;
  constexpr int kSlots = C::kSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Q / staging buffer x of the two (each two tiles of kQ bytes).
  auto qbuf = [&](uint32_t x) -> uint8_t* { return smem + (x ? C::kOffStage : 0); };
  uint8_t* ring = smem + C::kOffRing;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  TcMeta* meta = reinterpret_cast<TcMeta*>(smem + C::kOffMeta);  // [buffer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar[kBarQFull + x], 1);
      mbar_init(&bar[kBarMetaFull + x], 1);
      // the V producer and the two helpers once they have read the record,
      // the softmax warps once their output rows are copied out
      mbar_init(&bar[kBarBufFree + x], 3 + kTcSoftmaxWarps);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bar[kBarSFull + i], 1);
      mbar_init(&bar[kBarPFull + i], 4);
      mbar_init(&bar[kBarPvDone + i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar[kBarOFull + t], 1);
      mbar_init(&bar[kBarOEmpty + t], 4);
      mbar_init(&bar[kBarStaged + t], 4);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bar[kBarSlotFull + i], 1);
      mbar_init(&bar[C::kBarSlotEmpty + i], 2);  // one arrival per tile
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the tile list is written by the preceding kernel
  if (p.split_ctas > 0) {
    // The decode kernel of this batch may start now; CTAs past the prefill
    // share leave their SMs to it.
    griddep_launch_dependents();
    if (blockIdx.x + p.hdr->decode_ctas >= static_cast<uint32_t>(p.split_ctas)) {
      tc_fence_before();
      __syncthreads();
      if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
      return;
    }
  }

  const int G = p.G, Hq = p.num_heads, Hkv = p.num_kv_heads, bs = p.block_size;
  const int TQ = p.tokens_per_tile / 2;  // tokens of one of the two Q tiles
  uint32_t* status = &p.hdr->status;
  const uint32_t num_items = p.hdr->prefill_items;

  if (warp == 0 || warp == kTcVProducerWarp || warp >= kTcKHelperWarp) {
    // ------------------------------------------------------------ producers
    // Four warps issue the K/V copies (measured on this part: L2-resident
    // 2 KB boxes arrive about 1.5x faster from two issuing warps than from
    // one): a K pair and a V pair, the second warp of a pair issuing the
    // second half of each slot's boxes onto the same barrier (the first arms
    // its byte count).  The K warp grabs the work items, publishes each
    // item's record and loads its Q tiles; the other three read the record.
    // Each pair fills its own positions of the one ring, whose order
    // K0, K1, V0, K2, V1, ... is the MMAs' consumption order.
    const bool is_v = warp == kTcVProducerWarp || warp == kTcVHelperWarp;
    const bool helper = warp >= kTcKHelperWarp;
    const bool leader = warp == 0;
    if (lane == 0 && leader) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      tma_prefetch_desc(&tmq);
    }
    const CUtensorMap* map = is_v ? &tmv : &tmk;
    const int oob_row = p.num_blocks * Hkv * bs;  // a box here reads zeros
    // A slot is 64 / box_rows boxes of box_rows keys per 64 columns; box j
    // of column half bx belongs to lane j * kBoxes + bx.
    const int box_rows = p.box_rows;               // 16, 32 or 64
    const int kboxes = kTcKeys / box_rows;         // boxes per 64 columns
    const int nb = kboxes * C::kBoxes;             // boxes per slot (<= 8)
    // With four or more boxes a slot the pair splits them; with fewer the
    // first warp issues them all and the helper issues nothing.
    const bool split = nb >= 4;
    const int nb_first = split ? nb / 2 : nb;  // the first warp's share
    const bool boxer = helper ? (split && lane >= nb_first && lane < nb) : lane < nb_first;
    const int my_j = lane / C::kBoxes, my_bx = lane % C::kBoxes;
    uint32_t t_iter = 0, c0 = 0;  // c0: ring position of the item's first load
    int cur_kvh = 0;              // KV head of the current item (contiguous K/V)
    // Lane i < kSlots remembers the position of this warp's i-th newest
    // load (for the final drain); -1 = none.
    int my_pos = -1;
    bool ok = true;

    // Ring position q: K or V of one stage, each lane its own box.
    auto load_slot = [&](uint32_t q, int row) -> bool {
      const int s = static_cast<int>(q % kSlots);
      if (q >= static_cast<uint32_t>(kSlots) &&
          !warp_wait_or_flag(&bar[C::kBarSlotEmpty + s], ((q / kSlots) - 1) & 1, status))
        return false;
      // The pair's boxes may land before the count is armed: the phase
      // cannot complete while its one arrival is pending.
      if (lane == 0 && !helper)
        mbar_arrive_expect_tx(&bar[kBarSlotFull + s], static_cast<uint32_t>(C::kSlot));
      __syncwarp();
      if constexpr (kVarlen) {  // 64 consecutive tokens of one KV head; row = token
        if (boxer)
          tma_load_3d(ring + s * C::kSlot + my_bx * C::kRegion, map, my_bx * 64, cur_kvh, row,
                      &bar[kBarSlotFull + s]);
      } else if (boxer) {
        tma_load_2d(ring + s * C::kSlot + my_bx * C::kRegion + my_j * box_rows * 128, map,
                    my_bx * 64, row, &bar[kBarSlotFull + s]);
      }
      const int prev = __shfl_up_sync(0xffffffffu, my_pos, 1);
      my_pos = lane == 0 ? static_cast<int>(q) : prev;
      return true;
    };

    while (ok) {
      int tb, kvh, nkv, kbase;
      if (leader) {
        uint32_t it = 0;
        if (lane == 0) it = atomicAdd(&p.hdr->prefill_grab, 1u);
        it = __shfl_sync(0xffffffffu, it, 0);
        // Buffer x last served item t_iter - 2: its record read and its
        // output rows copied out.
        const uint32_t x = t_iter & 1;
        if (t_iter > 1 &&
            !warp_wait_or_flag(&bar[kBarBufFree + x], ((t_iter >> 1) - 1) & 1, status))
          break;
        if (it >= num_items) {
          if (lane == 0) {
            meta[x].done = 1;
            mbar_arrive(&bar[kBarMetaFull + x]);
            mbar_arrive(&bar[kBarQFull + x]);
          }
          break;
        }
        const uint32_t ti = it / static_cast<uint32_t>(Hkv);
        kvh = static_cast<int>(it - ti * static_cast<uint32_t>(Hkv));
        const PfTile tile = p.tiles[ti];
        tb = tile.b;
        nkv = tile.nkv;
        kbase = tile.kbase;
        if (lane == 0) {
          TcMeta m;
          m.tok0 = tile.tok0;
          m.ntok = tile.ntok;
          m.pos0 = tile.pos0;
          m.kvh = kvh;
          m.nkv = nkv;
          m.done = 0;
          m.b = tile.b;
          m.kbase = tile.kbase;
          meta[x] = m;
          mbar_arrive(&bar[kBarMetaFull + x]);  // the other producers start on the record
          mbar_arrive_expect_tx(&bar[kBarQFull + x],
                                static_cast<uint32_t>(2 * C::kBoxes * 128 * G * TQ));
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_3d(qbuf(x) + t * C::kQ + bx * C::kQRegion, &tmq, bx * 64, kvh * G,
                          tile.tok0 + t * TQ, &bar[kBarQFull + x]);
        }
      } else {
        const uint32_t x = t_iter & 1;
        if (!warp_wait_or_flag(&bar[kBarMetaFull + x], (t_iter >> 1) & 1, status)) break;
        const TcMeta m = meta[x];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarBufFree + x]);
        if (m.done) break;
        tb = m.b;
        kvh = m.kvh;
        nkv = m.nkv;
        kbase = m.kbase;
      }
      ++t_iter;
      cur_kvh = kvh;

      // Physical block ids, 32 per window held one per lane; the next window
      // is loaded while the current one is in use.
      auto load_window = [&](int lblk0) -> int {
        const int lb = lblk0 + lane;
        return (!kVarlen && lb * bs < nkv)  // contiguous K/V have no block table
                   ? __ldg(p.block_tables + static_cast<int64_t>(tb) * p.mbs + lb)
                   : -1;
      };
      int ids_base = 0;
      int ids = load_window(0);
      int ids_next = load_window(32);
      int lblk = 0, off = 0;  // block and slot of the next box
      // This lane's cache row for the stage of keys kb .. kb + 63.
      auto stage_row = [&](int kb) -> int {
        int my_row = oob_row;
#pragma unroll
        for (int j = 0; j < kTcSub; ++j) {
          if (j >= kboxes) break;
          const int key = kb + box_rows * j;
          if (key < nkv && lblk - ids_base >= 32) {  // windows advance in order
            ids_base += 32;
            ids = ids_next;
            ids_next = load_window(ids_base + 32);
          }
          int blk = __shfl_sync(0xffffffffu, ids, (lblk - ids_base) & 31);
          if (key < nkv && (blk < 0 || blk >= p.num_blocks)) {
            if (lane == 0 && !is_v) Status::raise(status, PA_DEV_BAD_BLOCK_ID);
            blk = -1;
          }
          const int row = (key < nkv && blk >= 0) ? (blk * Hkv + kvh) * bs + off : oob_row;
          if (j == my_j) my_row = row;
          off += box_rows;
          if (off == bs) {
            off = 0;
            ++lblk;
          }
        }
        return my_row;
      };

      // Contiguous K/V: the stage's first token; keys past the sequence
      // read the next sequence's rows (or zeros past the tensor), which the
      // mask and the V-row zeroing cover.
      const int n = (nkv + kTcKeys - 1) / kTcKeys;
      // With fewer than four boxes a slot (64-key boxes) the helpers issue
      // nothing: they only keep pace with the records.
      const bool loads = !helper || split;
      for (int j = 0; j < n && ok && loads; ++j) {
        int row;
        if constexpr (kVarlen)
          row = kbase + j * kTcKeys;
        else
          row = stage_row(j * kTcKeys);
        ok = load_slot(c0 + (is_v ? vpos(j, n) : kpos(j)), row);
      }
      c0 += 2 * n;
    }
    // Leave no copy in flight (the consumers may have stopped early on a
    // timeout): wait, bounded, for this warp's loads among the ring's last
    // kSlots positions, one per lane (an older position's slot has been
    // refilled since, so its load completed and its barrier moved on).
    const bool mine = lane < kSlots && my_pos >= 0 &&
                      static_cast<uint32_t>(my_pos) + kSlots >= c0;
    const uint32_t q = static_cast<uint32_t>(my_pos);
    if (mine && !mbar_wait(&bar[kBarSlotFull + q % kSlots], (q / kSlots) & 1))
      Status::raise(status, PA_DEV_WAIT_TIMEOUT);
    __syncwarp();
  } else if (warp < kTcVProducerWarp) {
    // ------------------------------------------------------------ MMA issuers
    // One warp per Q tile, so each tile's chain advances on its own while
    // the pipe runs the other tile's groups.  Per tile the QK of stage j + 1
    // is issued before the PV of stage j, so it runs while the softmax works
    // on stage j.  The warp waits on the barriers together and elect.sync
    // inside each MMA picks the issuing lane.  Each group of MMAs is
    // straight-line code on descriptors prepared up front: the tensor pipe
    // is fed at its full rate only when no branch or runtime trip count sits
    // between two tcgen05.mma (measured on this part: a data-independent
    // branch inside the issue loop halves the rate).  P lives in the S
    // buffer that the QK two stages later overwrites, and MMAs on different
    // accumulators are not ordered, so that QK waits for the PV to complete.
    const int t = warp - 1;
    constexpr uint32_t kIdQK = idesc_f16(kTcRows, kTcKeys, kBF16, false, false);
    constexpr uint32_t kIdPV = idesc_f16(kTcRows, D, kBF16, false, true);
    constexpr int kQkSteps = D / 16;
    // Adding (byte offset >> 4) to a descriptor moves its start address; the
    // 14-bit field cannot carry because shared-memory offsets stay below
    // 256 KB.
    uint64_t dq = 0;  // this item's Q tile (its buffer's tile t)
    const uint64_t dk = sdesc_sw128(smem_u32(ring), 16, 1024);             // K-major
    const uint64_t dv = sdesc_sw128(smem_u32(ring), C::kRegion, 1024);     // MN-major
    const uint32_t dout = tmem + C::col_o(t);
    uint32_t t_iter = 0, g0 = 0, c0 = 0;
    int vslot[2] = {0, 0};  // V slot read by the last PV on each S buffer
    bool ok = true;

    // S_t(j) = Q_t K(j)^T once K(j) landed and the PV two stages back no
    // longer reads that S buffer -- nor its V slot, which this warp then
    // releases (a plain arrival: a second tcgen05.commit right behind
    // another one costs the issuing warp about 250 cycles on this part).
    auto issue_qk = [&](int j, int n) -> bool {
      const uint32_t g = g0 + j;
      const int b = static_cast<int>(g & 1);
      const uint32_t ck = c0 + kpos(j);
      const int sk = static_cast<int>(ck % kSlots);
      if (!warp_wait_or_flag(&bar[kBarSlotFull + sk], (ck / kSlots) & 1, status)) return false;
      if (g >= 2) {
        if (!warp_wait_or_flag(&bar[kBarPvDone + 2 * t + b], ((g >> 1) - 1) & 1, status))
          return false;
        if (lane == 0) mbar_arrive(&bar[C::kBarSlotEmpty + (b ? vslot[1] : vslot[0])]);
      }
      tc_fence_after();
      const uint64_t dks = dk + static_cast<uint64_t>((sk * C::kSlot) >> 4);
      const uint32_t ds = tmem + C::col_s(t, b);
#pragma unroll
      for (int ks = 0; ks < kQkSteps; ++ks)
        umma_f16_warp(ds, dq + (((ks >> 2) * C::kQRegion + (ks & 3) * 32) >> 4),
                      dks + (((ks >> 2) * C::kRegion + (ks & 3) * 32) >> 4), kIdQK,
                      ks > 0 ? 1u : 0u);
      umma_commit_warp(&bar[kBarSFull + 2 * t + b]);
      return true;
    };
    // O_t += P_t(j) V(j) once V(j) landed, P_t(j) is written and (first
    // stage) the previous item's epilogue has read O_t.  All four 16-key
    // steps run on every stage: past the sequence P is 0 and the V rows are
    // zero (zero-filled boxes, or zeroed by the softmax warps inside the
    // last box).
    auto issue_pv = [&](int j, int n) -> bool {
      const uint32_t g = g0 + j;
      const int b = static_cast<int>(g & 1);
      const uint32_t cv = c0 + vpos(j, n);
      const int sv = static_cast<int>(cv % kSlots);
      if (!warp_wait_or_flag(&bar[kBarSlotFull + sv], (cv / kSlots) & 1, status) ||
          !warp_wait_or_flag(&bar[kBarPFull + 2 * t + b], (g >> 1) & 1, status) ||
          (j == 0 && t_iter > 0 &&
           !warp_wait_or_flag(&bar[kBarOEmpty + t], (t_iter - 1) & 1, status)))
        return false;
      tc_fence_after();
      const uint64_t dvs = dv + static_cast<uint64_t>((sv * C::kSlot) >> 4);
      const uint32_t ap = tmem + C::col_s(t, b);
      umma_f16_ts_warp(dout, ap, dvs, kIdPV, j > 0 ? 1u : 0u);
#pragma unroll
      for (int ks = 1; ks < kTcSub; ++ks)
        umma_f16_ts_warp(dout, ap + ks * 8, dvs + ((ks * 2048) >> 4), kIdPV, 1u);
      umma_commit_warp(&bar[kBarPvDone + 2 * t + b]);
      if (b) vslot[1] = sv; else vslot[0] = sv;
      if (j == n - 1) umma_commit_warp(&bar[kBarOFull + t]);
      return true;
    };

    while (ok) {
      const uint32_t x = t_iter & 1;
      if (!warp_wait_or_flag(&bar[kBarQFull + x], (t_iter >> 1) & 1, status)) break;
      const TcMeta m = meta[x];
      __syncwarp();
      if (m.done) break;
      const int n = (m.nkv + kTcKeys - 1) / kTcKeys;
      dq = sdesc_sw128(smem_u32(qbuf(x) + t * C::kQ), 16, 1024);
      tc_fence_after();
      ok = issue_qk(0, n);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n) ok = issue_qk(j + 1, n);
        if (ok) ok = issue_pv(j, n);
      }
      g0 += n;
      c0 += 2 * n;
      ++t_iter;
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - kTcFirstSoftmaxWarp) / 4;  // Q tile of this warp
    const int quarter = warp & 3;    // TMEM lanes 32*quarter ..
    const int row = 32 * quarter + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    uint32_t t_iter = 0, g0 = 0, c0 = 0;
    // A tensor store of the previous item's rows that this warp has yet to
    // see read out of its buffer (then the warp releases that buffer).
    int pending_buf = -1;
    while (true) {
      const uint32_t qb = t_iter & 1;  // this item's Q / staging buffer
      if (!warp_wait_or_flag(&bar[kBarQFull + qb], (t_iter >> 1) & 1, status)) break;
      const TcMeta m = meta[qb];
      __syncwarp();
      if (m.done) break;
      const int tl = t * TQ + row / G;  // token within the pair
      // causal: the row's absolute position; cross-attention: every key
      const int pos = p.causal ? m.pos0 + tl : m.nkv - 1;
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
        // S_t(j) complete: this tile's QK no longer reads K(j) (one warp per
        // tile releases its slot).
        if (lane == 0 && quarter == 0)
          mbar_arrive(&bar[C::kBarSlotEmpty + (c0 + kpos(j)) % kSlots]);
        tc_fence_after();
        float x[kTcKeys];
        tmem_ld64f(lane_base + C::col_s(t, b), x);

        const int kb = j * kTcKeys;
        const int lim = min(pos, m.nkv - 1) - kb;  // last visible column of this row
        if (__any_sync(0xffffffffu, lim < kTcKeys - 1)) {
#pragma unroll
          for (int i = 0; i < kTcKeys; ++i)
            if (i > lim) x[i] = -INFINITY;
        }
        // Row max: three-input max on eight independent chains.  (The
        // softmax warps' instruction stream, not the tensor pipe, sets the
        // stage time, so the row arithmetic below uses the widest forms:
        // three-input max, and packed two-float FFMA / FADD / FMUL.)
        static_assert(kTcKeys == 64, "the max chains cover 64 columns");
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmax3f(x[e], x[e + 8], x[e + 16]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmax3f(mx8[e], x[e + 24], x[e + 32]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmax3f(mx8[e], x[e + 40], x[e + 48]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], x[e + 56]);
        const float mx = fmax3f(fmax3f(mx8[0], mx8[1], mx8[2]), fmax3f(mx8[3], mx8[4], mx8[5]),
                                fmaxf(mx8[6], mx8[7])) *
                         p.scale_log2;
        const bool need = m_ref != -INFINITY && mx > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O_t must hold PV of stage g - 1 before it is rescaled.
          if (g >= 1 && !warp_wait_or_flag(&bar[kBarPvDone + 2 * t + ((g - 1) & 1)],
                                           ((g - 1) >> 1) & 1, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? ex2(m_ref - mx) : 1.f;
          const float2 alpha2 = make_float2(alpha, alpha);
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(lane_base + C::col_o(t) + c * 16, r);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float2 v = __fmul2_rn(
                  make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), alpha2);
              r[i] = __float_as_uint(v.x);
              r[i + 1] = __float_as_uint(v.y);
            }
            tmem_st16(lane_base + C::col_o(t) + c * 16, r);
          }
          if (need) {
            l *= alpha;
            m_ref = mx;
          }
        }
        if (m_ref == -INFINITY) m_ref = mx;
        const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;

        // P = 2^(x * scale - m_ref), in place, its row sum, and the P row
        // into tensor memory over the first half of its S (column c holds
        // keys 2c, 2c+1; those S values are already in registers) -- half by
        // half, so that the first half's store runs while the second half's
        // exponentials are computed.  The row sum keeps one accumulation
        // order, column groups of eight in ascending order.
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nr2 = make_float2(neg_ref, neg_ref);
        float2 rs[4];
#pragma unroll
        for (int h = 0; h < kTcKeys / 32; ++h) {
#pragma unroll
          for (int i = 32 * h; i < 32 * h + 32; i += 2) {
            const float2 a = __ffma2_rn(make_float2(x[i], x[i + 1]), sc2, nr2);
            x[i] = ex2(a.x);
            x[i + 1] = ex2(a.y);
          }
#pragma unroll
          for (int i = 32 * h; i < 32 * h + 32; i += 8) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 v = make_float2(x[i + 2 * k], x[i + 2 * k + 1]);
              rs[k] = i == 0 ? v : __fadd2_rn(rs[k], v);
            }
          }
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) w[c] = pack2<kBF16>(x[32 * h + 2 * c], x[32 * h + 2 * c + 1]);
          tmem_st16(lane_base + C::col_s(t, b) + 16 * h, w);
        }
        const float2 rsum = __fadd2_rn(__fadd2_rn(rs[0], rs[1]), __fadd2_rn(rs[2], rs[3]));
        l += rsum.x + rsum.y;

        // Keys past the sequence inside the last loaded box hold
        // whatever the cache slots hold: zero those V rows (P is 0 there,
        // but 0 * NaN is not).  Each tile's PV waits only for its own
        // softmax warps, so both tiles' warps write the same zeros.
        if (j == n - 1) {
          const int r0 = m.nkv - kb;
          const int r1 = min(kTcKeys, (r0 + p.box_rows - 1) / p.box_rows * p.box_rows);
          if (r1 > r0) {
            const uint32_t cv = c0 + vpos(j, n);
            const int sv = static_cast<int>(cv % kSlots);
            if (!warp_wait_or_flag(&bar[kBarSlotFull + sv], (cv / kSlots) & 1, status)) {
              ok = false;
              break;
            }
            uint8_t* vst = ring + sv * C::kSlot;
            const int per_row = C::kBoxes * 8;  // 16-byte chunks per key row
            const int total = (r1 - r0) * per_row;
            for (int i = row; i < total; i += 128) {
              const int kr = r0 + i / per_row, cc = i % per_row;
              *reinterpret_cast<uint4*>(vst + (cc >> 3) * C::kRegion + kr * 128 + (cc & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarPFull + 2 * t + b]);
        if (pending_buf >= 0) {
          // A stage later the store has long read its rows: release the
          // previous item's buffer now instead of waiting at its epilogue.
          if (lane == 0) {
            bulk_wait_read();
            mbar_arrive(&bar[kBarBufFree + pending_buf]);
          }
          pending_buf = -1;
        }
      }
      if (!ok) break;

      // Epilogue: O_t / l into shared memory over this item's Q tile t (O_t
      // complete means every MMA of the tile is, so Q_t is no longer read),
      // in the Q tile's own layout: 64-column halves of 128-byte rows, each
      // row's 16-byte chunks XOR-swizzled by the row as a 128-byte-swizzle
      // tensor copy places them (each thread writes its row; the swizzle
      // spreads a warp's stores over all banks).  A tile of full tokens then
      // leaves in one tensor store per half, issued by one thread; a tile with
      // fewer tokens (the last of a chunk) is copied out by its 128 threads,
      // which write only its valid rows.
      if (!warp_wait_or_flag(&bar[kBarOFull + t], t_iter & 1, status)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* stg = qbuf(qb) + t * C::kQ;  // over this item's Q tile t
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + C::col_o(t) + c * 32, r);
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
          const int k = c * 4 + q;  // chunk of the row: half k / 8, chunk k % 8 of it
          *reinterpret_cast<uint4*>(stg + (k >> 3) * C::kQRegion + row * 128 +
                                    (((k & 7) ^ (row & 7)) << 4)) = o;
        }
      }
      // O_t is read: the next item's first PV may overwrite it.  The rows
      // go out through the async proxy (a tensor store).
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar[kBarOEmpty + t]);
        mbar_arrive(&bar[kBarStaged + t]);
      }
      if (!warp_wait_or_flag(&bar[kBarStaged + t], t_iter & 1, status)) break;
      const int ntok_t = min(max(m.ntok - t * TQ, 0), TQ);  // tokens of this tile
      bool defer = false;  // this warp releases the buffer a stage into the next item
      if (ntok_t == TQ) {
        if (quarter == 0 && lane == 0) {
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_store_3d(&tmo, bx * 64, m.kvh * G, m.tok0 + t * TQ, stg + bx * C::kQRegion);
          bulk_commit();
        }
        defer = quarter == 0;
      } else {
        // Thread `row` of the tile copies chunk k = row % kCh of rows
        // row / kCh, + kStep, + 2 kStep, ...; the row's (token, head) steps
        // along with it, so the loop needs no division by G.
        constexpr int kCh = D / 8;  // 16-byte chunks per row
        constexpr int kStep = kTcRows / kCh;
        const int rows_valid = G * ntok_t;
        const int k = row & (kCh - 1);
        int r = row / kCh;
        int tok = r / G, h = r - tok * G;
        const int dtok = kStep / G, dh = kStep - dtok * G;
        uint16_t* obase = static_cast<uint16_t*>(p.out) +
                          (static_cast<int64_t>(m.tok0 + t * TQ) * Hq +
                           static_cast<int64_t>(m.kvh) * G) * D + k * 8;
        const uint8_t* shalf = stg + (k >> 3) * C::kQRegion;
        for (; r < rows_valid; r += kStep) {  // rows in order: the rest are past the tile's tokens
          const uint4 v =
              *reinterpret_cast<const uint4*>(shalf + r * 128 + (((k & 7) ^ (r & 7)) << 4));
          *reinterpret_cast<uint4*>(obase + (static_cast<int64_t>(tok) * Hq + h) * D) = v;
          tok += dtok;
          h += dh;
          if (h >= G) {
            h -= G;
            ++tok;
          }
        }
      }
      // The buffer may take a later item's Q tiles (TMA writes): order this
      // thread's shared-memory accesses before the release.
      fence_proxy_async();
      __syncwarp();
      if (defer)
        pending_buf = static_cast<int>(qb);
      else if (lane == 0)
        mbar_arrive(&bar[kBarBufFree + qb]);
      g0 += n;
      c0 += 2 * n;
      ++t_iter;
    }
    // This thread's tensor stores reach global memory before the CTA ends.
    if (quarter == 0 && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

namespace {

template <bool kBF16, int D, bool kVarlen>
int launch_prefill_tc_t(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                        const CUtensorMap& tmo,
                        const PrefillParams& p, int64_t max_items, cudaStream_t stream,
                        int num_sms) {
  using C = TcCfg<D>;
  static_assert(C::kBytes <= 227 * 1024, "one CTA per SM");
  auto kern = prefill_tc_kernel<kBF16, D, kVarlen>;
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes) !=
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
  cfg.dynamicSmemBytes = C::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmk, tmv, tmq, tmo, p) == cudaSuccess ? 1 : -1;
}

}  // namespace

int launch_prefill_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                      const CUtensorMap& tmo,
                      const PrefillParams& p, bool bf16, int head_dim, int64_t max_items,
                      cudaStream_t stream, int num_sms) {
#define PA_PREFILL_LAUNCH(B, DIM, V) \
  launch_prefill_tc_t<B, DIM, V>(tmk, tmv, tmq, tmo, p, max_items, stream, num_sms)
  const bool v = p.varlen != 0;
  if (bf16) {
    if (head_dim == 64) return v ? PA_PREFILL_LAUNCH(true, 64, true) : PA_PREFILL_LAUNCH(true, 64, false);
    return v ? PA_PREFILL_LAUNCH(true, 128, true) : PA_PREFILL_LAUNCH(true, 128, false);
  }
  if (head_dim == 64) return v ? PA_PREFILL_LAUNCH(false, 64, true) : PA_PREFILL_LAUNCH(false, 64, false);
  return v ? PA_PREFILL_LAUNCH(false, 128, true) : PA_PREFILL_LAUNCH(false, 128, false);
#undef PA_PREFILL_LAUNCH
}

}  // namespace pa
