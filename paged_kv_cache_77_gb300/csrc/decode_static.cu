// Decode attention for callers that cannot allocate device memory.
//
// Some callers of this library have no way to hand it a workspace: a plugin
// running inside a host runtime that owns the device allocator and forbids other
// allocations, a serving loop that has already partitioned all of HBM between
// weights and the KV cache, or code that must not call cudaMalloc because it may
// synchronise the device in the middle of a latency-critical step. For them,
// pkv_paged_attention_decode_static runs the same decode as
// pkv_paged_attention_decode but keeps its split-KV partials in a fixed array
// compiled into this library, so the caller passes only inputs and outputs.
//
// The array lives in device global memory of every GPU that loads the library and
// stays allocated until the process exits. Its size is PKV_DECODE_STATIC_SCRATCH_BYTES;
// larger problems are rejected. Host code cannot use the array's name as a device
// address, so its address is looked up once per device with cudaGetSymbolAddress,
// on the first call made while that device is current.
#include <cuda_runtime.h>

#include <mutex>

#include "abi_common.h"
#include "launch.h"

namespace pkv {

static __device__ __align__(256) uint8_t g_decode_static_scratch[PKV_DECODE_STATIC_SCRATCH_BYTES];

// Device address of the scratch array on the current device (looked up once per device).
static int static_scratch_address(void** out) {
  static std::mutex mu;
  static void* cached[64] = {nullptr};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  PKV_REQUIRE(e == cudaSuccess && dev >= 0 && dev < 64, PKV_ERR_LAUNCH,
              "pkv_paged_attention_decode_static: no current CUDA device (%s)", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_static_scratch);
    PKV_REQUIRE(e == cudaSuccess && p != nullptr, PKV_ERR_LAUNCH,
                "pkv_paged_attention_decode_static: cudaGetSymbolAddress failed: %s",
                cudaGetErrorString(e));
    cached[dev] = p;
  }
  *out = cached[dev];
  return PKV_OK;
}

}  // namespace pkv

extern "C" int pkv_paged_attention_decode_static(void* out, int32_t out_dtype, float* lse,
                                                 const void* q, const void* k_cache,
                                                 const void* v_cache, const int32_t* block_table,
                                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                                 int32_t B, int32_t H, int32_t H_kv, int32_t head_dim,
                                                 int32_t block_size, int64_t num_blocks, float scale,
                                                 int32_t window, int* dev_status, void* stream) {
  const size_t need = pkv_decode_workspace_size(B, H, H_kv, head_dim);
  PKV_REQUIRE(need <= PKV_DECODE_STATIC_SCRATCH_BYTES, PKV_ERR_WORKSPACE,
              "pkv_paged_attention_decode_static: this problem needs %zu bytes of scratch, more than "
              "the %d-byte static array; use pkv_paged_attention_decode with a workspace",
              need, (int)PKV_DECODE_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  int rc = pkv::static_scratch_address(&scratch);
  if (rc != PKV_OK) return rc;
  // Every partial the merge reads is written by the same call's attention kernel,
  // so nothing in the array has to start at zero.
  return pkv_paged_attention_decode(out, out_dtype, lse, q, k_cache, v_cache, block_table,
                                    max_blocks_per_seq, seq_lens, B, H, H_kv, head_dim, block_size,
                                    num_blocks, scale, window, scratch, PKV_DECODE_STATIC_SCRATCH_BYTES,
                                    dev_status, stream);
}
