// paged_attn_decode_noalloc: the decode entry point for callers that cannot
// hand the library a workspace of their own.
//
// Some callers have no way to obtain device scratch memory: an inference
// runtime whose caching allocator has already reserved nearly all of HBM for
// its KV-cache pool and forbids other allocations, a plugin host that gives
// kernels only their input and output tensors, or a plain C program with no
// device-memory manager.  For them this file keeps the decode workspace in a
// file-scope device array, sized once at load time, and runs the ordinary
// decode path (work-list build, decode kernel, split combine) on it.
//
// Cost of that convenience: every GPU that loads this library holds the
// array (kStaticScratchBytes) until the process exits, and all calls share
// it, so two calls that overlap on the GPU (different streams, or different
// host threads) race on it and must be serialised by the caller.
#include <mutex>

#include "pa_kernels.cuh"

namespace pa {
namespace {

// 32 MiB: enough for 256 sequences x 4 KV splits x 32 heads x 128 dims, or
// for the automatic split policy on batches of up to about 120 sequences of
// 4096 tokens; larger problems are rejected with PA_ERR_WORKSPACE.
constexpr size_t kStaticScratchBytes = size_t{32} << 20;

static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device.  Host code only sees a
// host-side stand-in for `g_decode_scratch`; the real address comes from
// cudaGetSymbolAddress with that device current.  It is looked up again on
// every call made outside a stream capture (a cheap host-side query), since
// a context torn down and created again (cudaDeviceReset) loads the module
// anew and the array may then sit elsewhere.  Inside a capture the address
// of the device's latest uncaptured call is used, so the first call on a
// device must come before any capture.
int scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices)
    return PA_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  } else if (!g_scratch_addr[dev]) {
    return PA_ERR_CUDA;  // first call on this device inside a capture
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" {

PA_API int paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, float scale, int num_seqs,
                                     int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int num_blocks, int dtype, int num_splits,
                                     void* out, pa_stream_t stream) {
  const size_t need = paged_attn_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq, block_size, num_splits);
  if (need > pa::kStaticScratchBytes) return PA_ERR_WORKSPACE;
  if (num_seqs == 0)  // nothing to run; no device set-up needed
    return paged_attn_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                             context_lens, scale, num_seqs, num_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, dtype, num_splits, out, nullptr, 0, stream);
  void* ws = nullptr;
  const int rc = pa::scratch_address(reinterpret_cast<cudaStream_t>(stream), &ws);
  if (rc != PA_OK) return rc;
  // The work-list kernel rewrites every counter and list the decode kernels
  // read, so the contents left by the previous call need no clearing.
  return paged_attn_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           scale, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, dtype, num_splits, out, ws, pa::kStaticScratchBytes,
                           stream);
}

}  // extern "C"
