// Host side of the tcgen05 decode kernel (decode_tc.cuh): tensor-map encoding and
// the single-token dispatch over the group size n_rep.
#include "decode_tc.cuh"

namespace pkv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map with a 128-byte swizzle. dims/strides innermost first; strides in
// bytes for dims 1..rank-1.
bool make_tmap_sw128(CUtensorMap* m, CUtensorMapDataType dtype, const void* ptr, int rank,
                     const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                     CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void*>(ptr),
                  (const cuuint64_t*)dims, (const cuuint64_t*)strides, (const cuuint32_t*)box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 maps fetch 256 bytes into L2 per request: a 256-byte K/V row of one kv head
// is read as two 128-byte boxes, and the promotion brings the second in with the first.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box) {
  return make_tmap_sw128(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rank, dims, strides, box,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// bf16 map with a 64-byte swizzle (boxes whose rows are 64 bytes, 32 elements).
bool make_tmap_bf16_sw64(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr),
                  (const cuuint64_t*)dims, (const cuuint64_t*)strides, (const cuuint32_t*)box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.n_rep) {
    case 1: return launch_tc_n<1, 1>(a, stream);
    case 2: return launch_tc_n<2, 1>(a, stream);
    case 4: return launch_tc_n<4, 1>(a, stream);
    case 8: return launch_tc_n<8, 1>(a, stream);
    case 16: return launch_tc_n<16, 1>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
