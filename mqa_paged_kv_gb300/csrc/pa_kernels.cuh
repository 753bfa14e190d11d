// Internal interface between the C-ABI layer (api.cu) and the kernels:
// workspace layout, work-item records and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {

// ------------------------------------------------------------------ sizes
constexpr int kKeyTile = 16;          // keys per decode pipeline stage
constexpr int kAutoSplitTokens = 256; // automatic split length (tokens)
constexpr int kMaxSplits = 64;        // splits per sequence, at most
constexpr int kPrefillTileRows = 128; // (token, head) rows of one MMA tile
constexpr int kPrefillKeys = 64;      // keys per prefill pipeline stage

// Equal-share decode (automatic splits of the decode entry point): every
// warp group of the persistent grid takes an equal contiguous range of the
// batch's key tiles, units (sequence, KV head) being cut where the ranges
// end.  The lengths are scanned in each CTA's shared memory, which bounds
// the batch; the partial slots are sized for a bounded grid.
constexpr int kSkMaxSeqs = 2048;  // larger batches take the sorted work list
constexpr int kSkMaxCtas = 160;   // CTAs of an equal-share grid, at most

// Warp groups per decode CTA for G query heads per KV head (the launcher's
// configurations: swap AB with one warp per group for G <= 8; head major
// with ceil(G / 16) consumer warps and one producer warp per group above).
constexpr int decode_groups_per_cta(int G) {
  return G <= 8 ? 8 : (G <= 16 ? 6 : (G <= 32 ? 4 : 2));
}

// Shared memory of the equal-share prologue: tile prefix [B + 1], lengths
// [B] and the scan's warp sums.
constexpr size_t sk_smem_bytes(int num_seqs) {
  return (static_cast<size_t>(2 * num_seqs + 1) * 4 + 32 * 4 + 15) / 16 * 16;
}

// ------------------------------------------------------------------ records
// Header at the start of every workspace (256 bytes).
struct WsHeader {
  uint32_t decode_grab;      // next decode item to hand out
  uint32_t status;           // PA_DEV_* bits of the most recent call
  uint32_t decode_items;     // decode (split, kv head) items
  uint32_t decode_pairs;     // decode (sequence, split) pairs
  uint32_t prefill_grab;     // next prefill item to hand out
  uint32_t prefill_items;    // prefill (tile, kv head) items
  uint32_t prefill_tiles;
  uint32_t decode_ctas;      // mixed batch: CTAs the decode kernel keeps (the prefill kernel
                             // takes the SMs of the others)
  uint32_t pad[56];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Per sequence: where its split partials live and how its query rows map.
struct SeqInfo {
  int32_t split_offset;  // first partial index of this sequence's splits
  int32_t nsplit;        // decode splits (0: no decode row; 1: no combine)
  int32_t tok;           // query row of a decode sequence
  int32_t qlen;
};

// A decode (sequence, split) pair; item = pair * Hkv + kv head.
struct DecPair {
  int32_t b;
  int32_t tok;         // query / output row
  int32_t key_begin;   // first key (multiple of the block size)
  int32_t key_end;     // one past the last key
  int32_t part_idx;    // partial slot, or -1 when the split is the whole sequence
  int32_t pad[3];
};

// A prefill tile: up to kPrefillRows / G query tokens of one sequence;
// item = tile * Hkv + kv head.
struct PfTile {
  int32_t b;
  int32_t tok0;   // first query row of the tile
  int32_t ntok;   // valid query tokens in the tile
  int32_t pos0;   // absolute position of the first token (ctx - qlen + i)
  int32_t nkv;    // keys the tile reads: pos0 + ntok (causal) or ctx (cross)
  int32_t kbase;  // contiguous (varlen) K/V: row of the sequence's first key
  int32_t pad[2];
};

struct WsLayout {
  size_t seq_info, pairs, part_lse, part_o, tiles, total;
  int64_t max_pairs, max_tiles;
  bool equal_share;  // the decode call runs the equal-share decomposition
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Upper bound of KV splits of one sequence (host side, no device data).
inline int64_t max_splits_per_seq(int max_blocks_per_seq, int block_size, int num_splits) {
  if (num_splits > 0) return num_splits;
  const int64_t chunk = (kAutoSplitTokens + block_size - 1) / block_size;
  int64_t s = (max_blocks_per_seq + chunk - 1) / chunk;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < 1) s = 1;
  return s;
}

// A prefill work item is two MMA tiles of the same sequence and KV head:
// 2 * floor(128 / G) query tokens.
inline int prefill_tokens_per_tile(int G) {
  const int t = kPrefillTileRows / G;
  return 2 * (t < 1 ? 1 : t);
}

inline WsLayout workspace_layout(int num_seqs, int num_heads, int head_dim, int64_t max_pairs,
                                 int64_t max_tiles) {
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.seq_info = off;
  off = align_up(off + sizeof(SeqInfo) * static_cast<size_t>(num_seqs), 256);
  L.pairs = off;
  off = align_up(off + sizeof(DecPair) * static_cast<size_t>(max_pairs), 256);
  L.part_lse = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(max_pairs) * num_heads, 256);
  L.part_o = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(max_pairs) * num_heads * head_dim, 256);
  L.tiles = off;
  off = align_up(off + sizeof(PfTile) * static_cast<size_t>(max_tiles), 256);
  L.total = off;
  L.max_pairs = max_pairs;
  L.max_tiles = max_tiles;
  L.equal_share = false;
  return L;
}

// Whether a decode call with these sizes uses the equal-share decomposition
// (host side, from sizes only): automatic splits, a batch whose lengths fit
// the prologue's shared memory, and tile counts that fit 32-bit indices.
inline bool use_equal_share(int num_seqs, int num_kv_heads, int max_blocks_per_seq,
                            int block_size, int num_splits) {
  if (num_splits != 0 || num_seqs <= 0 || num_seqs > kSkMaxSeqs) return false;
  const int64_t tiles_per_seq =
      (static_cast<int64_t>(max_blocks_per_seq) * block_size + kKeyTile - 1) / kKeyTile;
  return tiles_per_seq * num_seqs * num_kv_heads < (int64_t{1} << 31);
}

// Equal-share workspace: header, the tile prefix over sequences [B + 1]
// (written by the decode kernel for the combine), and two partial slots
// per warp group -- the unit piece at the start of its range and the one
// at its end -- each holding G rows of D fp32 values and G log-sum-exps.
inline WsLayout equal_share_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim) {
  const int G = num_heads / num_kv_heads;
  const int64_t slots = 2 * static_cast<int64_t>(kSkMaxCtas) * decode_groups_per_cta(G);
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.seq_info = off;  // the tile prefix
  off = align_up(off + sizeof(int32_t) * (static_cast<size_t>(num_seqs) + 1), 256);
  L.pairs = off;
  L.part_lse = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(slots) * G, 256);
  L.part_o = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(slots) * G * head_dim, 256);
  L.tiles = off;
  L.total = off;
  L.max_pairs = slots;
  L.max_tiles = 0;
  L.equal_share = true;
  return L;
}

// ------------------------------------------------------------------ params
struct PrepareParams {
  const int32_t* context_lens;
  const int32_t* cu_query_lens;  // nullptr: pure decode (qlen 1, row = b)
  void* out;                     // zero rows of empty decode sequences
  WsHeader* hdr;
  SeqInfo* seq_info;
  DecPair* pairs;
  PfTile* tiles;
  int num_seqs, block_size, num_splits, num_kv_heads, num_heads, head_dim;
  int tokens_per_tile;  // prefill tile height in tokens
  int max_blocks_per_seq;
  int causal;           // 0: cross-attention, every row sees all keys, qlen may exceed ctx
  const int32_t* cu_key_lens;  // varlen K/V (no cache): key rows of sequence b are
                               // [cu_key_lens[b], cu_key_lens[b+1]); all rows take tiles
  int64_t total_tokens;  // rows of q / out
  int split_ctas;        // > 0: a mixed batch's grid, to be split between decode and prefill
  int header_only;       // equal-share decode: only reset the status word (no lists)
};

struct DecodeParams {
  const void* q;
  const int32_t* block_tables;
  void* out;
  float* part_o;
  float* part_lse;
  const DecPair* pairs;
  WsHeader* hdr;
  int mbs, num_heads, num_kv_heads, G, block_size, num_blocks;
  float scale_log2;  // scale * log2(e)
  // 1 when a kernel of this call follows (the split combine, or the prefill
  // kernel of a mixed batch): only then may the next launch start early (a
  // following call's work-list build must not overlap this kernel).
  int trigger_dependents;
  // Partial of item part_idx, KV head kvh, head h of the group at row
  // part_idx * part_row_stride + kvh * part_kvh_rows + h of part_o / part_lse
  // (sorted list: Hq and G; equal share: G and 0).
  int part_row_stride, part_kvh_rows;
  // Equal-share decomposition (1) instead of the sorted work list: the
  // lengths are read and scanned in the prologue, and CTA 0 stores the tile
  // prefix at sk_prefix for the combine.
  int equal_share;
  const int32_t* context_lens;
  int num_seqs;
  int32_t* sk_prefix;
  // Limit of each pipeline wait (a stage's copies, a free stage or query
  // slot).  The bounded drain of copies still in flight before a CTA exits
  // keeps the fixed 2 s limit, so every copy lands first.
  uint64_t wait_ns;
  // 1 in a batch with query chunks: launched after the prefill kernel and
  // beside it, on the SMs its CTAs past the prefill share leave (its other
  // CTAs join as prefill CTAs finish): no wait at the start (the work list
  // is complete -- the prefill kernel lets this one start only after its
  // own wait for it -- and is read through L2), and a wait for the prefill
  // kernel before completing, so what follows sees both kernels' results.
  int concurrent;
};

// The pipeline wait limit the next decode kernels get (pa_set_pipeline_wait_limit).
uint64_t pipeline_wait_ns();

struct CombineParams {
  const SeqInfo* seq_info;
  const float* part_o;
  const float* part_lse;
  void* out;
  int num_seqs, num_heads, head_dim;
  // equal share: the tile prefix over sequences and the decode grid's groups
  const int32_t* sk_prefix;
  int num_kv_heads, sk_groups;
};

// A batch with query chunks runs its prefill and decode kernels side by
// side, the SMs split by the work-list kernel in proportion to the two
// kernels' estimated times at these per-SM rates (measured on this part:
// the decode kernel streams about 6.2 TB/s over 152 SMs, the prefill kernel
// about 940 TFLOP/s), the decode share shaded down: decode CTAs that find
// no SM at first take over the prefill kernel's SMs as its CTAs finish, so
// the decode kernel can grow into a misjudged split and the prefill kernel
// cannot.
constexpr double kDecodeBytesPerSmSec = 41e9;
constexpr double kPrefillFlopsPerSmSec = 6.2e12;
constexpr double kDecodeShareMargin = 0.9;

struct PrefillParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  const PfTile* tiles;
  WsHeader* hdr;
  int mbs, num_heads, num_kv_heads, G, block_size, num_blocks, tokens_per_tile;
  int box_rows;  // keys per K/V box: gcd(block_size, 64), so a box never crosses a block
  int causal;    // 0: cross-attention (every row sees all of the tile's keys)
  int varlen;    // 1: K/V are contiguous [T, Hkv, D] tensors (3-D maps), no block table
  // > 0 in a batch with query chunks: the SMs (n) split between this kernel
  // and the decode kernel that follows and runs beside it.  CTAs with index
  // >= n - decode_ctas leave at once, giving their SMs to it (the grid may
  // be smaller than n when there are few tiles; then none leaves).
  int split_ctas;
  float scale_log2;
};

// ------------------------------------------------------------------ launchers
// Each returns the number of kernels enqueued, or -1 on a launch error.
int launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, uint32_t* status,
                             cudaStream_t stream, int num_sms);

int launch_prepare(const PrepareParams& p, bool bf16, cudaStream_t stream);

int launch_decode(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                  bool bf16, int head_dim, cudaStream_t stream, int num_sms);

int launch_combine(const CombineParams& p, bool bf16, int head_dim, cudaStream_t stream);

// Merge of the equal-share partials (and zero rows of key-less sequences).
int launch_combine_equal_share(const CombineParams& p, bool bf16, int head_dim,
                               cudaStream_t stream);

int launch_prefill_tc(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                      const CUtensorMap& tmo, const PrefillParams& p, bool bf16, int head_dim, int64_t max_items,
                      cudaStream_t stream, int num_sms);

}  // namespace pa
