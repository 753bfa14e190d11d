// reshape_and_cache: scatter this step's K/V rows [T, Hkv, D] into the paged
// cache [NB, Hkv, bs, D] at slot_mapping[t] (-1 = skip).  Pure data movement:
// one thread moves one 16-byte chunk of K and the matching chunk of V, so a
// warp reads 512 contiguous bytes of a token's row and writes them to the
// slot's contiguous D-element rows.  HBM-bound: 2 * T * Hkv * D * e bytes
// read and the same written.
#include "pa_kernels.cuh"

namespace pa {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
    int num_kv_heads, int chunks_per_row /* D * 2 / 16 */, int block_size, int64_t num_slots,
    uint32_t* status) {
  griddep_wait();  // k, v and the slots may come from the previous kernel
  griddep_launch_dependents();
  const int64_t chunks_per_token = static_cast<int64_t>(num_kv_heads) * chunks_per_row;
  const int64_t total = num_tokens * chunks_per_token;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / chunks_per_token;
    const int64_t rem = i - t * chunks_per_token;
    const int h = static_cast<int>(rem / chunks_per_row);
    const int c = static_cast<int>(rem - static_cast<int64_t>(h) * chunks_per_row);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) {
      if (slot < -1 && rem == 0) Status::raise(status, PA_DEV_BAD_SLOT);
      continue;
    }
    if (slot >= num_slots) {
      if (rem == 0) Status::raise(status, PA_DEV_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
    k_cache[dst] = __ldg(k + i);
    v_cache[dst] = __ldg(v + i);
  }
}

int launch_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, uint32_t* status,
                             cudaStream_t stream, int num_sms) {
  const int chunks_per_row = head_dim * 2 / 16;
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * chunks_per_row;
  if (total == 0) return 0;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  // One wave at most (8 CTAs of 256 threads an SM, grid-stride beyond): the
  // attention kernels launched behind this one become resident as its CTAs
  // retire, and a second wave would then find the SMs taken.
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, reshape_and_cache_kernel, static_cast<const uint4*>(k), static_cast<const uint4*>(v),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping,
      static_cast<int64_t>(num_tokens), num_kv_heads, chunks_per_row, block_size,
      static_cast<int64_t>(num_blocks) * block_size, status);
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace pa
