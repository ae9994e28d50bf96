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
#include <cuda_fp8.h>

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
  pdl_launch_dependents();  // the attention kernel after this one may launch now
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

// kv_cache_write_fp8: quantise each new (token, kv head) row of K and V to FP8 E4M3
// with one fp32 scale (scale = amax / 448, codes = e4m3(x / scale), rounded to
// nearest even with saturation; an all-zero row gets scale 0 and zero codes) and
// scatter codes and scales through slot_mapping. Both divisions are IEEE fp32
// (__fdiv_rn), so the codes follow from the inputs exactly. One warp per row of
// 128 values: lane = 4 values (8-byte load, 4-byte store); the row max by shuffles.
// Scales live in [num_blocks, H_kv, block_size] so that one tile's 128 scales are
// contiguous for the decode kernel.
// Roofline: HBM; per row 256 B read + 128 B codes + 4 B scale written (+ 4 B slot
// per token).
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
    float* __restrict__ v_scale, const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
    const int32_t* __restrict__ slots, int64_t num_tokens, int64_t num_slots, int hkv,
    int block_size, int* dev_status) {
  pdl_launch_dependents();  // the attention kernel after this one may launch now
  const int lane = threadIdx.x & 31;
  const int64_t rows = num_tokens * hkv * 2;
  for (int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); w < rows;
       w += (int64_t)gridDim.x * 8) {
    const int is_v = (int)(w & 1);
    const int64_t th = w >> 1;  // token * hkv + head
    const int64_t t = th / hkv;
    const int h = (int)(th - t * hkv);
    const int32_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if ((int64_t)slot >= num_slots) {
      if (lane == 0 && is_v == 0 && h == 0) flag_status(dev_status, PKV_DEV_BAD_SLOT);
      continue;
    }
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>((is_v ? v : k) + th * 256) + lane);
    float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                  __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.f);
    uint32_t packed = 0;
    if (scale > 0.f) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)), __NV_SATFINITE, __NV_E4M3);
      packed = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    const int64_t blk = slot / block_size, off = slot - blk * block_size;
    uint8_t* dst = (is_v ? v_cache : k_cache) + ((int64_t)slot * hkv + h) * 128;
    reinterpret_cast<uint32_t*>(dst)[lane] = packed;
    if (lane == 0) (is_v ? v_scale : k_scale)[(blk * hkv + h) * block_size + off] = scale;
  }
}

cudaError_t launch_kv_write_fp8(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                const void* k, const void* v, const int32_t* slots,
                                int64_t num_tokens, int64_t num_blocks, int block_size, int hkv,
                                int* dev_status, cudaStream_t stream, int num_sms) {
  const int64_t rows = num_tokens * hkv * 2;
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  kv_write_fp8_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      (uint8_t*)k_cache, (uint8_t*)v_cache, k_scale, v_scale, (const uint8_t*)k, (const uint8_t*)v,
      slots, num_tokens, num_blocks * block_size, hkv, block_size, dev_status);
  return cudaGetLastError();
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
