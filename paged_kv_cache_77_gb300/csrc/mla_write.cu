// Fused MLA cache write: RMSNorm of the latent row, RoPE of the rope row, and the
// write of both through slot_mapping, in one pass over the new rows
// ("昇腾 NPU 独立部署模式 KVCache 自管完整指南", 模式三: the kv_a projection output
// goes through kv_a_layernorm RMSNorm and RoPE and into nope_cache / rope_cache in
// one step, optionally also returning k_nope / k_rope). RoPE takes the rotate_half
// form of the Llama forward ("KV Cache 笔记"): out = x * cos + [-x[32:], x[:32]] * sin.
//
//   y_nope = bf16(x[0:512] / sqrt(mean(x[0:512]^2) + eps) * gamma)
//   y_rope = bf16(x[512:576] * cos + rotate_half(x[512:576]) * sin)
//
// One warp per token. Lane l holds latent elements [8l, 8l+8) and [256+8l, 256+8l+8)
// (two 16-byte loads, coalesced across the warp), reduces the sum of squares with
// xor shuffles, and stores its 16 normalised values as two 16-byte vectors. Every
// lane holds two rope elements (2l, 2l+1) with their cos and sin; element i pairs
// with i+32, which lives in lane l ^ 16. All loads of a token are issued together,
// so each token costs one memory round trip. Arithmetic in fp32, results rounded to
// nearest even.
//
// Roofline: HBM. Algorithmic bytes per token = 1152 (latent read) + 512 (cos, sin
// fp32) + 1152 (cache rows written) + 4 (slot) [+ 1152 with k_nope/k_rope outputs].
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kRank = 512;
constexpr int kRope = 64;
constexpr int kRow = kRank + kRope;  // elements of one latent row

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    u[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(u[0], u[1], u[2], u[3]);
}

}  // namespace

#ifndef PKV_MW_UNROLL
#define PKV_MW_UNROLL 1
#endif
#ifndef PKV_MW_GRID_PER_SM
#define PKV_MW_GRID_PER_SM 8
#endif
// Measured on GB300 (262,144 tokens): 1 token per warp iteration with 8 CTAs per SM
// of grid moves 6.1 TB/s (4 or 32 CTAs per SM: within 2 %); 2 tokens per iteration
// need 106 registers, halve the resident warps and drop to 4.7-4.9 TB/s.
constexpr int kUnroll = PKV_MW_UNROLL;          // tokens in flight per warp iteration
constexpr int kMinBlocks = kUnroll == 1 ? 4 : 2;  // register budget that keeps 0 spills

// Per lane and token: latent elements [8l, 8l+8) and [256+8l, 256+8l+8) (a, b), rope
// elements 2l and 2l+1 (r) with their cos and sin. Element i of the rope row pairs
// with i + 32, two elements per lane, so the partner lives in lane l ^ 16 (lanes
// 0-15 hold i < 32). Every load of a token is issued before any arithmetic on it.
struct TokenIn {
  float a[8], b[8];
  float2 r, c, s;
  int32_t slot;
};

__device__ __forceinline__ void load_token(TokenIn& in, const uint8_t* latent, const float* cosv,
                                           const float* sinv, const int32_t* slots, int64_t t,
                                           int lane) {
  const uint8_t* row = latent + t * (kRow * 2);
  unpack8(ld_nc_v4(row + lane * 16), in.a);
  unpack8(ld_nc_v4(row + 512 + lane * 16), in.b);
  const uint32_t rw = __ldg(reinterpret_cast<const unsigned int*>(row + kRank * 2) + lane);
  in.r = make_float2(__uint_as_float(rw << 16), __uint_as_float(rw & 0xffff0000u));
  in.c = __ldg(reinterpret_cast<const float2*>(cosv + t * kRope) + lane);
  in.s = __ldg(reinterpret_cast<const float2*>(sinv + t * kRope) + lane);
  in.slot = __ldg(slots + t);
}

__global__ void __launch_bounds__(256, kMinBlocks) mla_rmsnorm_rope_write_kernel(
    uint8_t* __restrict__ cache_nope, uint8_t* __restrict__ cache_rope,
    uint8_t* __restrict__ k_nope_out, uint8_t* __restrict__ k_rope_out,
    const uint8_t* __restrict__ latent, const uint8_t* __restrict__ gamma,
    const float* __restrict__ cosv, const float* __restrict__ sinv,
    const int32_t* __restrict__ slots, int64_t num_tokens, int64_t num_slots, float eps,
    int* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  float g0[8], g1[8];
  unpack8(ld_nc_v4(gamma + lane * 16), g0);
  unpack8(ld_nc_v4(gamma + 512 + lane * 16), g1);
  const float sign = lane < 16 ? -1.f : 1.f;
  for (int64_t t0 = warp0; t0 < num_tokens; t0 += kUnroll * wstride) {
    TokenIn in[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (t0 + u * wstride < num_tokens) load_token(in[u], latent, cosv, sinv, slots, t0 + u * wstride, lane);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t t = t0 + u * wstride;
      if (t >= num_tokens) continue;  // warp-uniform
      TokenIn& x = in[u];
      const bool bad = (int64_t)x.slot >= num_slots;
      if (bad && lane == 0) flag_status(dev_status, PKV_DEV_BAD_SLOT);
      const bool store = x.slot >= 0 && !bad;
      // RMSNorm of the latent row.
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(x.a[i], x.a[i], fmaf(x.b[i], x.b[i], ss));
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = rsqrtf(ss * (1.f / kRank) + eps);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x.a[i] = x.a[i] * inv * g0[i];
        x.b[i] = x.b[i] * inv * g1[i];
      }
      const uint4 wa = pack8(x.a), wb = pack8(x.b);
      // RoPE of the rope row: out = r * cos + sign * partner * sin.
      const float p0 = __shfl_xor_sync(0xffffffffu, x.r.x, 16);
      const float p1 = __shfl_xor_sync(0xffffffffu, x.r.y, 16);
      __nv_bfloat162 h = __floats2bfloat162_rn(fmaf(x.r.x, x.c.x, sign * p0 * x.s.x),
                                               fmaf(x.r.y, x.c.y, sign * p1 * x.s.y));
      const uint32_t wr = *reinterpret_cast<uint32_t*>(&h);
      if (k_nope_out) {
        uint8_t* o = k_nope_out + t * (kRank * 2);
        *reinterpret_cast<uint4*>(o + lane * 16) = wa;
        *reinterpret_cast<uint4*>(o + 512 + lane * 16) = wb;
      }
      if (k_rope_out) reinterpret_cast<uint32_t*>(k_rope_out + t * (kRope * 2))[lane] = wr;
      if (store) {
        uint8_t* dn = cache_nope + (int64_t)x.slot * (kRank * 2);
        *reinterpret_cast<uint4*>(dn + lane * 16) = wa;
        *reinterpret_cast<uint4*>(dn + 512 + lane * 16) = wb;
        reinterpret_cast<uint32_t*>(cache_rope + (int64_t)x.slot * (kRope * 2))[lane] = wr;
      }
    }
  }
}

cudaError_t launch_mla_rmsnorm_rope_write(void* cache_nope, void* cache_rope, void* k_nope_out,
                                          void* k_rope_out, const void* latent, const void* gamma,
                                          const float* cosv, const float* sinv,
                                          const int32_t* slots, int64_t num_tokens,
                                          int64_t num_slots, float eps, int* dev_status,
                                          cudaStream_t stream, int num_sms) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256, per_cta = threads / 32;
  int64_t blocks = (num_tokens + kUnroll * per_cta - 1) / (kUnroll * per_cta);
  const int64_t cap = (int64_t)num_sms * PKV_MW_GRID_PER_SM;
  if (blocks > cap) blocks = cap;
  mla_rmsnorm_rope_write_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      (uint8_t*)cache_nope, (uint8_t*)cache_rope, (uint8_t*)k_nope_out, (uint8_t*)k_rope_out,
      (const uint8_t*)latent, (const uint8_t*)gamma, cosv, sinv, slots, num_tokens, num_slots, eps,
      dev_status);
  return cudaGetLastError();
}

}  // namespace pkv
