// C ABI of libpaged_attn.so: argument validation, TMA descriptors, workspace
// layout and the launch sequence of each entry point.  The declarations and
// their contracts are in include/paged_attn.h.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "pa_kernels.cuh"

namespace pa {

// Pipeline wait limit of the decode kernels; 0 = the default 2 s.
std::atomic<uint64_t> g_pipeline_wait_ns{0};

uint64_t pipeline_wait_ns() {
  const uint64_t v = g_pipeline_wait_ns.load(std::memory_order_relaxed);
  return v ? v : kWaitTimeoutNs;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int num_sms = 0;
  int cc_major = 0;
  bool ok = false;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

thread_local int g_last_launches = 0;
thread_local int g_last_cuda_error = 0;

// Takes the CUDA runtime's pending error (the one behind a failed launch,
// attribute or synchronize call) for pa_last_cuda_error and returns
// PA_ERR_CUDA.
int cuda_error() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}
thread_local int g_next_ctas = 0;
thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;

// Records the measurement hook's events around the attention kernels.
struct ProfileScope {
  cudaEvent_t start, stop;
  cudaStream_t st;
  explicit ProfileScope(cudaStream_t s) : start(g_prof_start), stop(g_prof_stop), st(s) {
    g_prof_start = g_prof_stop = nullptr;
  }
  void begin() const {
    if (start) cudaEventRecord(start, st);
  }
  void end() const {
    if (stop) cudaEventRecord(stop, st);
  }
};

// The CTA cap of pa_limit_next_call_ctas, taken by the next attention call:
// its persistent kernels run on at most that many SMs.
int take_cta_limit() {
  const int n = g_next_ctas;
  g_next_ctas = 0;
  return n;
}

int grid_sms(const DeviceInfo& dev, int limit) {
  return (limit > 0 && limit < dev.num_sms) ? limit : dev.num_sms;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Properties of the current device (cached); PA_OK or an error status.
int current_device(DeviceInfo& info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].ok) {
      int sms = 0, major = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return PA_ERR_CUDA;
      g_dev[dev].num_sms = sms;
      g_dev[dev].cc_major = major;
      g_dev[dev].ok = true;
    }
    info = g_dev[dev];
  }
  if (info.cc_major != 10) return PA_ERR_DEVICE;
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D map over a cache [NB * Hkv * bs rows][D]: box_rows-key x 64-column boxes.
int encode_cache_map(CUtensorMap* map, const void* base, int64_t rows, int head_dim,
                     int box_rows = kKeyTile) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 3-D map over contiguous K or V [T][Hkv][D]: boxes of (64 columns, one KV
// head, 64 tokens) -- one 8 KB copy per 64 columns of a 64-key stage.
int encode_varlen_kv_map(CUtensorMap* map, const void* base, int64_t tokens, int num_kv_heads,
                         int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_kv_heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// 3-D map over q [T][Hq][D]: boxes of (64 columns, G heads, TQ tokens).
int encode_query_map(CUtensorMap* map, const void* base, int64_t tokens, int num_heads,
                     int head_dim, int G, int TQ) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(num_heads) * head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(TQ)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Checks shared by both attention entry points.
int check_common(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                 float scale, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                 int block_size, int num_blocks, int dtype, int num_splits, const void* out) {
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEADDIM;
  if (block_size < 16 || block_size > 256 || block_size % 16 != 0) return PA_ERR_BLOCKSIZE;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PA_ERR_SHAPE;
  if (num_heads / num_kv_heads > 64) return PA_ERR_SHAPE;
  if (num_splits < 0 || num_splits > kMaxSplits) return PA_ERR_SHAPE;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;  // softmax scale > 0
  if (num_seqs == 0) return PA_OK;
  if (max_blocks_per_seq <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > (int64_t{1} << 30))
    return PA_ERR_SHAPE;
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size >= (int64_t{1} << 31))
    return PA_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ALIGN;
  return PA_OK;
}

WsLayout decode_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                       int max_blocks_per_seq, int block_size, int num_splits) {
  if (num_heads % num_kv_heads == 0 &&
      use_equal_share(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, num_splits))
    return equal_share_layout(num_seqs, num_heads, num_kv_heads, head_dim);
  const int64_t pairs =
      static_cast<int64_t>(num_seqs) * max_splits_per_seq(max_blocks_per_seq, block_size, num_splits);
  (void)num_kv_heads;
  return workspace_layout(num_seqs, num_heads, head_dim, pairs, 0);
}

WsLayout prefill_layout(int num_seqs, int total_query_tokens, int num_heads, int num_kv_heads,
                        int head_dim, int max_blocks_per_seq, int block_size, int num_splits) {
  const int G = num_heads / num_kv_heads;
  const int TQ = prefill_tokens_per_tile(G);
  const int64_t decode_rows = num_seqs < total_query_tokens ? num_seqs : total_query_tokens;
  const int64_t pairs =
      decode_rows * max_splits_per_seq(max_blocks_per_seq, block_size, num_splits);
  int64_t tiles = (static_cast<int64_t>(total_query_tokens) +
                   static_cast<int64_t>(num_seqs) * (TQ - 1)) / TQ + 1;
  if (tiles > total_query_tokens) tiles = total_query_tokens;
  return workspace_layout(num_seqs, num_heads, head_dim, pairs, tiles);
}

WsLayout varlen_layout(int num_seqs, int total_query_tokens, int num_heads, int num_kv_heads,
                       int head_dim) {
  const int TQ = prefill_tokens_per_tile(num_heads / num_kv_heads);
  int64_t tiles = (static_cast<int64_t>(total_query_tokens) +
                   static_cast<int64_t>(num_seqs) * (TQ - 1)) / TQ + 1;
  if (tiles > total_query_tokens) tiles = total_query_tokens;
  return workspace_layout(num_seqs, num_heads, head_dim, 0, tiles);
}

int check_workspace(const void* ws, size_t bytes, const WsLayout& L) {
  if (!ws) return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return PA_ERR_WORKSPACE;
  if (bytes < L.total) return PA_ERR_WORKSPACE;
  return PA_OK;
}

int finish(int launched) {
  if (launched < 0) return cuda_error();
  g_last_launches = launched;
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return PA_OK;
  g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}

}  // namespace

// The chunked path: causal = 1 is paged_attn_chunked_prefill (bottom-right
// causal chunks), causal = 0 is paged_attn_cross_attention (every query row
// sees all of its sequence's cached keys).
int run_chunked(const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, int max_blocks_per_seq,
                const int32_t* cu_query_lens, const int32_t* context_lens,
                int total_query_tokens, int max_query_len, float scale,
                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                int block_size, int num_blocks, int dtype, int num_splits,
                void* out, void* workspace, size_t workspace_bytes,
                pa_stream_t stream, int causal) {
  g_last_launches = 0;
  const int cta_limit = take_cta_limit();
  int rc = check_common(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        scale, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, dtype, num_splits, out);
  if (rc != PA_OK) return rc;
  if (total_query_tokens < 0 || max_query_len < 0) return PA_ERR_SHAPE;
  if (num_seqs == 0 || total_query_tokens == 0) return PA_OK;
  if (!cu_query_lens) return PA_ERR_NULL;
  const WsLayout L = prefill_layout(num_seqs, total_query_tokens, num_heads, num_kv_heads,
                     head_dim, max_blocks_per_seq, block_size, num_splits);
  if ((rc = check_workspace(workspace, workspace_bytes, L)) != PA_OK) return rc;
  DeviceInfo dev;
  if ((rc = current_device(dev)) != PA_OK) return rc;

  const int G = num_heads / num_kv_heads;
  const int TQ = prefill_tokens_per_tile(G);
  const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
  CUtensorMap tmk, tmv, tmq, tmo;
  if ((rc = encode_cache_map(&tmk, k_cache, rows, head_dim)) != PA_OK) return rc;
  if ((rc = encode_cache_map(&tmv, v_cache, rows, head_dim)) != PA_OK) return rc;
  if ((rc = encode_query_map(&tmq, q, total_query_tokens, num_heads, head_dim, G, TQ / 2)) !=
      PA_OK)
    return rc;
  // The output has q's shape: full tiles leave through the same box.
  if ((rc = encode_query_map(&tmo, out, total_query_tokens, num_heads, head_dim, G, TQ / 2)) !=
      PA_OK)
    return rc;
  // The prefill kernel gathers K/V in boxes of gcd(block_size, 64) keys: a
  // 64-key stage then takes 64 / box_rows boxes per 64 columns, and larger
  // blocks mean fewer, larger TMA copies.
  const int box_rows = (block_size % 64 == 0) ? 64 : (block_size % 32 == 0) ? 32 : 16;
  CUtensorMap tmk_pf = tmk, tmv_pf = tmv;
  if (box_rows != kKeyTile && max_query_len > 1) {
    if ((rc = encode_cache_map(&tmk_pf, k_cache, rows, head_dim, box_rows)) != PA_OK) return rc;
    if ((rc = encode_cache_map(&tmv_pf, v_cache, rows, head_dim, box_rows)) != PA_OK) return rc;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool bf16 = dtype == PA_BF16;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  PrepareParams pp;
  pp.context_lens = context_lens;
  pp.cu_query_lens = cu_query_lens;
  pp.out = out;
  pp.hdr = reinterpret_cast<WsHeader*>(ws);
  pp.seq_info = reinterpret_cast<SeqInfo*>(ws + L.seq_info);
  pp.pairs = reinterpret_cast<DecPair*>(ws + L.pairs);
  pp.tiles = reinterpret_cast<PfTile*>(ws + L.tiles);
  pp.num_seqs = num_seqs;
  pp.block_size = block_size;
  pp.num_splits = num_splits;
  pp.num_kv_heads = num_kv_heads;
  pp.num_heads = num_heads;
  pp.head_dim = head_dim;
  pp.tokens_per_tile = TQ;
  pp.max_blocks_per_seq = max_blocks_per_seq;
  pp.total_tokens = total_query_tokens;
  pp.causal = causal;
  pp.cu_key_lens = nullptr;
  pp.header_only = 0;
  // A batch with query chunks runs its prefill and decode kernels side by
  // side; the work-list kernel splits the grid between them.
  const bool concurrent = max_query_len > 1;
  pp.split_ctas = concurrent ? grid_sms(dev, cta_limit) : 0;

  PrefillParams fp;
  fp.block_tables = block_tables;
  fp.context_lens = context_lens;
  fp.out = out;
  fp.tiles = pp.tiles;
  fp.hdr = pp.hdr;
  fp.mbs = max_blocks_per_seq;
  fp.num_heads = num_heads;
  fp.num_kv_heads = num_kv_heads;
  fp.G = G;
  fp.block_size = block_size;
  fp.num_blocks = num_blocks;
  fp.tokens_per_tile = TQ;
  fp.box_rows = box_rows;
  fp.causal = causal;
  fp.varlen = 0;
  fp.split_ctas = pp.split_ctas;
  fp.scale_log2 = scale * 1.4426950408889634f;

  DecodeParams dp;
  dp.q = q;
  dp.block_tables = block_tables;
  dp.out = out;
  dp.part_o = reinterpret_cast<float*>(ws + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  dp.pairs = pp.pairs;
  dp.hdr = pp.hdr;
  dp.mbs = max_blocks_per_seq;
  dp.num_heads = num_heads;
  dp.num_kv_heads = num_kv_heads;
  dp.G = G;
  dp.block_size = block_size;
  dp.num_blocks = num_blocks;
  dp.scale_log2 = fp.scale_log2;
  dp.trigger_dependents = num_splits != 1;
  dp.concurrent = concurrent ? 1 : 0;
  dp.part_row_stride = num_heads;
  dp.part_kvh_rows = G;
  dp.equal_share = 0;
  dp.context_lens = context_lens;
  dp.num_seqs = num_seqs;
  dp.sk_prefix = nullptr;
  dp.wait_ns = pipeline_wait_ns();

  const ProfileScope prof(st);
  int n = 0, r;
  if ((r = launch_prepare(pp, bf16, st)) < 0) return cuda_error();
  n += r;
  prof.begin();
  // Prefill first: its CTAs past the prefill share leave at once, and the
  // decode kernel, launched as its dependent, takes those SMs (and more as
  // prefill CTAs finish).
  if (concurrent) {
    if ((r = launch_prefill_tc(tmk_pf, tmv_pf, tmq, tmo, fp, bf16, head_dim, L.max_tiles * num_kv_heads, st,
                grid_sms(dev, cta_limit))) < 0)
      return cuda_error();
    n += r;
  }
  if ((r = launch_decode(tmk, tmv, dp, bf16, head_dim, st, grid_sms(dev, cta_limit))) < 0)
    return cuda_error();
  n += r;
  prof.end();
  if (num_splits != 1) {
    CombineParams cp;
    cp.seq_info = pp.seq_info;
    cp.part_o = dp.part_o;
    cp.part_lse = dp.part_lse;
    cp.out = out;
    cp.num_seqs = num_seqs;
    cp.num_heads = num_heads;
    cp.head_dim = head_dim;
    cp.sk_prefix = nullptr;
    cp.num_kv_heads = num_kv_heads;
    cp.sk_groups = 0;
    if ((r = launch_combine(cp, bf16, head_dim, st)) < 0) return cuda_error();
    n += r;
  }
  return finish(n);
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "null pointer argument";
    case PA_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case PA_ERR_DTYPE: return "unsupported element type";
    case PA_ERR_HEADDIM: return "unsupported head_dim (64 or 128)";
    case PA_ERR_BLOCKSIZE: return "unsupported block_size (multiple of 16 in [16, 256])";
    case PA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case PA_ERR_DEVICE: return "current device is not an sm_100-family GPU";
    default: return "unknown status";
  }
}

int pa_version(void) { return 1; }

int pa_last_cuda_error(void) { return g_last_cuda_error; }

const char* pa_last_cuda_error_string(void) {
  return g_last_cuda_error == 0 ? "no error"
                                : cudaGetErrorString(static_cast<cudaError_t>(g_last_cuda_error));
}

int pa_last_launch_count(void) { return g_last_launches; }

void pa_limit_next_call_ctas(int max_ctas) { g_next_ctas = max_ctas > 0 ? max_ctas : 0; }

void pa_set_pipeline_wait_limit(uint64_t limit_ns) {
  g_pipeline_wait_ns.store(limit_ns, std::memory_order_relaxed);
}

void pa_profile_next_call(void* start_event, void* stop_event) {
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
}

int reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, int dtype, uint32_t* status_word,
                      pa_stream_t stream) {
  g_last_launches = 0;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEADDIM;
  if (block_size < 16 || block_size > 256 || block_size % 16 != 0) return PA_ERR_BLOCKSIZE;
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGN;
  DeviceInfo dev;
  const int rc = current_device(dev);
  if (rc != PA_OK) return rc;
  return finish(launch_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                         num_kv_heads, head_dim, block_size, num_blocks,
                                         status_word, stream, dev.num_sms));
}

size_t paged_attn_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int block_size, int num_splits) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
    return 0;
  return decode_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                       block_size, num_splits)
      .total;
}

int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, float scale, int num_seqs, int num_heads,
                      int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                      int num_splits, void* out, void* workspace, size_t workspace_bytes,
                      pa_stream_t stream) {
  g_last_launches = 0;
  const int cta_limit = take_cta_limit();
  int rc = check_common(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        scale, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, dtype, num_splits, out);
  if (rc != PA_OK || num_seqs == 0) return rc;
  const WsLayout L = decode_layout(num_seqs, num_heads, num_kv_heads, head_dim,
                                   max_blocks_per_seq, block_size, num_splits);
  if ((rc = check_workspace(workspace, workspace_bytes, L)) != PA_OK) return rc;
  DeviceInfo dev;
  if ((rc = current_device(dev)) != PA_OK) return rc;

  const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
  CUtensorMap tmk, tmv;
  if ((rc = encode_cache_map(&tmk, k_cache, rows, head_dim)) != PA_OK) return rc;
  if ((rc = encode_cache_map(&tmv, v_cache, rows, head_dim)) != PA_OK) return rc;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool bf16 = dtype == PA_BF16;
  const int G = num_heads / num_kv_heads;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  PrepareParams pp;
  pp.context_lens = context_lens;
  pp.cu_query_lens = nullptr;
  pp.out = out;
  pp.hdr = reinterpret_cast<WsHeader*>(ws);
  pp.seq_info = reinterpret_cast<SeqInfo*>(ws + L.seq_info);
  pp.pairs = reinterpret_cast<DecPair*>(ws + L.pairs);
  pp.tiles = nullptr;
  pp.num_seqs = num_seqs;
  pp.block_size = block_size;
  pp.num_splits = num_splits;
  pp.num_kv_heads = num_kv_heads;
  pp.num_heads = num_heads;
  pp.head_dim = head_dim;
  pp.tokens_per_tile = prefill_tokens_per_tile(G);
  pp.max_blocks_per_seq = max_blocks_per_seq;
  pp.total_tokens = num_seqs;
  pp.causal = 1;
  pp.cu_key_lens = nullptr;
  pp.split_ctas = 0;
  pp.header_only = L.equal_share ? 1 : 0;
  // Equal shares: the grid (one CTA per SM) fixes the groups' tile ranges.
  int grid = grid_sms(dev, cta_limit);
  if (L.equal_share && grid > kSkMaxCtas) grid = kSkMaxCtas;

  DecodeParams dp;
  dp.q = q;
  dp.block_tables = block_tables;
  dp.out = out;
  dp.part_o = reinterpret_cast<float*>(ws + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  dp.pairs = pp.pairs;
  dp.hdr = pp.hdr;
  dp.mbs = max_blocks_per_seq;
  dp.num_heads = num_heads;
  dp.num_kv_heads = num_kv_heads;
  dp.G = G;
  dp.block_size = block_size;
  dp.num_blocks = num_blocks;
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.trigger_dependents = num_splits != 1;
  dp.concurrent = 0;
  dp.equal_share = L.equal_share ? 1 : 0;
  dp.part_row_stride = L.equal_share ? G : num_heads;
  dp.part_kvh_rows = L.equal_share ? 0 : G;
  dp.context_lens = context_lens;
  dp.num_seqs = num_seqs;
  dp.sk_prefix = reinterpret_cast<int32_t*>(ws + L.seq_info);
  dp.wait_ns = pipeline_wait_ns();

  const ProfileScope prof(st);
  int n = 0, r;
  if ((r = launch_prepare(pp, bf16, st)) < 0) return cuda_error();
  n += r;
  prof.begin();
  if ((r = launch_decode(tmk, tmv, dp, bf16, head_dim, st, grid)) < 0) return cuda_error();
  n += r;
  prof.end();
  if (num_splits != 1) {
    CombineParams cp;
    cp.seq_info = pp.seq_info;
    cp.part_o = dp.part_o;
    cp.part_lse = dp.part_lse;
    cp.out = out;
    cp.num_seqs = num_seqs;
    cp.num_heads = num_heads;
    cp.head_dim = head_dim;
    cp.sk_prefix = dp.sk_prefix;
    cp.num_kv_heads = num_kv_heads;
    cp.sk_groups = grid * decode_groups_per_cta(G);
    r = L.equal_share ? launch_combine_equal_share(cp, bf16, head_dim, st)
                      : launch_combine(cp, bf16, head_dim, st);
    if (r < 0) return cuda_error();
    n += r;
  }
  return finish(n);
}

size_t paged_attn_chunked_prefill_workspace_bytes(int num_seqs, int total_query_tokens,
                                                  int num_heads, int num_kv_heads, int head_dim,
                                                  int max_blocks_per_seq, int block_size,
                                                  int num_splits) {
  if (num_seqs < 0 || total_query_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
    return 0;
  return prefill_layout(num_seqs, total_query_tokens, num_heads, num_kv_heads, head_dim,
                        max_blocks_per_seq, block_size, num_splits)
      .total;
}

int paged_attn_chunked_prefill(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* cu_query_lens, const int32_t* context_lens,
                               int total_query_tokens, int max_query_len, float scale,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int dtype, int num_splits,
                               void* out, void* workspace, size_t workspace_bytes,
                               pa_stream_t stream) {
  return pa::run_chunked(q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_query_lens,
                         context_lens, total_query_tokens, max_query_len, scale, num_seqs,
                         num_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype,
                         num_splits, out, workspace, workspace_bytes, stream, 1);
}

int paged_attn_cross_attention(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* cu_query_lens, const int32_t* context_lens,
                               int total_query_tokens, int max_query_len, float scale,
                               int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int dtype, int num_splits,
                               void* out, void* workspace, size_t workspace_bytes,
                               pa_stream_t stream) {
  return pa::run_chunked(q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_query_lens,
                         context_lens, total_query_tokens, max_query_len, scale, num_seqs,
                         num_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype,
                         num_splits, out, workspace, workspace_bytes, stream, 0);
}

size_t gqa_varlen_prefill_workspace_bytes(int num_seqs, int total_query_tokens, int num_heads,
                                          int num_kv_heads, int head_dim) {
  if (num_seqs < 0 || total_query_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || head_dim <= 0)
    return 0;
  return varlen_layout(num_seqs, total_query_tokens, num_heads, num_kv_heads, head_dim).total;
}

int gqa_varlen_prefill(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_k, int total_query_tokens, int total_key_tokens,
                       int max_seqlen_q, float scale, int num_seqs, int num_heads,
                       int num_kv_heads, int head_dim, int dtype, void* out, void* workspace,
                       size_t workspace_bytes, pa_stream_t stream) {
  g_last_launches = 0;
  const int cta_limit = take_cta_limit();
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_HEADDIM;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      num_heads / num_kv_heads > 64)
    return PA_ERR_SHAPE;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;
  if (total_query_tokens < 0 || total_key_tokens < 0 || max_seqlen_q < 0) return PA_ERR_SHAPE;
  if (num_seqs == 0 || total_query_tokens == 0) return PA_OK;
  if (total_key_tokens <= 0) return PA_ERR_SHAPE;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out) return PA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PA_ERR_ALIGN;
  const WsLayout L = varlen_layout(num_seqs, total_query_tokens, num_heads, num_kv_heads, head_dim);
  int rc;
  if ((rc = check_workspace(workspace, workspace_bytes, L)) != PA_OK) return rc;
  DeviceInfo dev;
  if ((rc = current_device(dev)) != PA_OK) return rc;

  const int G = num_heads / num_kv_heads;
  const int TQ = prefill_tokens_per_tile(G);
  CUtensorMap tmk, tmv, tmq, tmo;
  if ((rc = encode_varlen_kv_map(&tmk, k, total_key_tokens, num_kv_heads, head_dim)) != PA_OK)
    return rc;
  if ((rc = encode_varlen_kv_map(&tmv, v, total_key_tokens, num_kv_heads, head_dim)) != PA_OK)
    return rc;
  if ((rc = encode_query_map(&tmq, q, total_query_tokens, num_heads, head_dim, G, TQ / 2)) !=
      PA_OK)
    return rc;
  // The output has q's shape: full tiles leave through the same box.
  if ((rc = encode_query_map(&tmo, out, total_query_tokens, num_heads, head_dim, G, TQ / 2)) !=
      PA_OK)
    return rc;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool bf16 = dtype == PA_BF16;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  PrepareParams pp = {};
  pp.context_lens = nullptr;
  pp.cu_query_lens = cu_seqlens_q;
  pp.cu_key_lens = cu_seqlens_k;
  pp.out = out;
  pp.hdr = reinterpret_cast<WsHeader*>(ws);
  pp.seq_info = reinterpret_cast<SeqInfo*>(ws + L.seq_info);
  pp.pairs = reinterpret_cast<DecPair*>(ws + L.pairs);
  pp.tiles = reinterpret_cast<PfTile*>(ws + L.tiles);
  pp.num_seqs = num_seqs;
  pp.block_size = 16;  // unused with contiguous K/V (no decode list)
  pp.num_splits = 1;
  pp.num_kv_heads = num_kv_heads;
  pp.num_heads = num_heads;
  pp.head_dim = head_dim;
  pp.tokens_per_tile = TQ;
  pp.max_blocks_per_seq = 0;
  pp.total_tokens = total_query_tokens;
  pp.causal = 1;
  PrefillParams fp = {};
  fp.block_tables = nullptr;
  fp.context_lens = nullptr;
  fp.out = out;
  fp.tiles = pp.tiles;
  fp.hdr = pp.hdr;
  fp.mbs = 0;
  fp.num_heads = num_heads;
  fp.num_kv_heads = num_kv_heads;
  fp.G = G;
  fp.block_size = 16;
  fp.num_blocks = 0;
  fp.tokens_per_tile = TQ;
  fp.box_rows = 64;
  fp.causal = 1;
  fp.varlen = 1;
  fp.scale_log2 = scale * 1.4426950408889634f;

  const ProfileScope prof(st);
  int n = 0, r;
  if ((r = launch_prepare(pp, bf16, st)) < 0) return cuda_error();
  n += r;
  prof.begin();
  if ((r = launch_prefill_tc(tmk, tmv, tmq, tmo, fp, bf16, head_dim, L.max_tiles * num_kv_heads, st,
                             grid_sms(dev, cta_limit))) < 0)
    return cuda_error();
  n += r;
  prof.end();
  return finish(n);
}

int pa_read_device_status(const void* workspace, int clear, uint32_t* flags, pa_stream_t stream) {
  if (!workspace || !flags) return PA_ERR_NULL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const WsHeader* hdr = static_cast<const WsHeader*>(workspace);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, &hdr->status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return cuda_error();
  if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_error();
  *flags = v;
  if (clear) {
    if (cudaMemsetAsync(const_cast<uint32_t*>(&hdr->status), 0, sizeof(uint32_t), st) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_error();
  }
  return PA_OK;
}

}  // extern "C"
