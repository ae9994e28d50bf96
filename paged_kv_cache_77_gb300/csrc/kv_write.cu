// kv_cache_write: scatter new K/V rows into the paged cache through slot_mapping.
//
// The cache viewed as [num_blocks * block_size, row] takes row t at index
// slot_mapping[t] (standalone deployment guide, 模式二 modeling write via
// npu_scatter_nd_update_ on cache.view(-1, H_kv, d)). The copy is bit-exact: 16-byte
// vector loads of the new rows and 16-byte stores into the cache, with 64-bit slot
// offsets (slot * row bytes passes 2^32 at these cache sizes).
//
// Roofline: HBM. Algorithmic bytes per row = 2 * (row_k + row_v) (read the new row,
// write it into the cache) + 4 bytes of slot index.
#include "device_common.cuh"
#include "launch.h"

namespace pkv {

// One thread moves one 16-byte chunk. The flattened index space is
// (token, chunk) with the k chunks of a row first, then its v chunks, so
// consecutive threads touch consecutive bytes of one row.
__global__ void __launch_bounds__(256) kv_write_kernel(uint8_t* __restrict__ k_cache,
                                                       uint8_t* __restrict__ v_cache,
                                                       const uint8_t* __restrict__ k,
                                                       const uint8_t* __restrict__ v,
                                                       const int32_t* __restrict__ slots,
                                                       int64_t num_tokens, int64_t num_slots,
                                                       int ck, int cv, int* dev_status) {
  const int per_row = ck + cv;
  const int64_t total = num_tokens * per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / per_row;
    const int c = (int)(idx - t * per_row);
    const int32_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if ((int64_t)slot >= num_slots) {
      if (c == 0) flag_status(dev_status, PKV_DEV_BAD_SLOT);
      continue;
    }
    if (c < ck) {
      const uint4 w = ld_nc_v4(k + (t * ck + c) * 16);
      *reinterpret_cast<uint4*>(k_cache + ((int64_t)slot * ck + c) * 16) = w;
    } else {
      const int cc = c - ck;
      const uint4 w = ld_nc_v4(v + (t * cv + cc) * 16);
      *reinterpret_cast<uint4*>(v_cache + ((int64_t)slot * cv + cc) * 16) = w;
    }
  }
}

cudaError_t launch_kv_write(void* k_cache, void* v_cache, const void* k, const void* v,
                            const int32_t* slots, int64_t num_tokens, int64_t num_slots,
                            int64_t row_k_bytes, int64_t row_v_bytes, int* dev_status,
                            cudaStream_t stream, int num_sms) {
  const int ck = (int)(row_k_bytes / 16), cv = (int)(row_v_bytes / 16);
  const int64_t total = num_tokens * (ck + cv);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms * 8;  // 8 resident CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  kv_write_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      (uint8_t*)k_cache, (uint8_t*)v_cache, (const uint8_t*)k, (const uint8_t*)v, slots, num_tokens,
      num_slots, ck, cv, dev_status);
  return cudaGetLastError();
}

// copy_blocks: block dst[i] of one cache becomes a bit copy of block src[i] (the
// copied incomplete last block of a forked request, "KV Cache 笔记" fork_blocks).
// One thread moves one 16-byte chunk of the flattened (pair, chunk) space, so a
// few large blocks still spread over the whole GPU. Sources are never destinations
// of the same call, so the non-coherent loads see unchanged data.
// Roofline: HBM; algorithmic bytes per pair = 2 * block_bytes + 8 bytes of ids.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t* __restrict__ cache,
                                                          int64_t num_blocks, int64_t chunks,
                                                          const int32_t* __restrict__ src,
                                                          const int32_t* __restrict__ dst,
                                                          int64_t n, int* dev_status) {
  const int64_t total = n * chunks;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / chunks;
    const int64_t c = idx - i * chunks;
    const int32_t s = __ldg(src + i), d = __ldg(dst + i);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
      if (c == 0) flag_status(dev_status, PKV_DEV_BAD_BLOCK);
      continue;
    }
    const uint4 w = ld_nc_v4(cache + ((int64_t)s * chunks + c) * 16);
    *reinterpret_cast<uint4*>(cache + ((int64_t)d * chunks + c) * 16) = w;
  }
}

cudaError_t launch_copy_blocks(void* cache, int64_t num_blocks, int64_t block_bytes,
                               const int32_t* src, const int32_t* dst, int64_t n, int* dev_status,
                               cudaStream_t stream, int num_sms) {
  const int64_t chunks = block_bytes / 16;
  const int64_t total = n * chunks;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  copy_blocks_kernel<<<(unsigned)blocks, threads, 0, stream>>>((uint8_t*)cache, num_blocks, chunks,
                                                              src, dst, n, dev_status);
  return cudaGetLastError();
}

}  // namespace pkv
