// Device helpers shared by the kernels: bf16 bit handling, cp.async, streaming loads,
// and the balanced tile partition used by every split-KV decode kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_kv.h"

namespace pkv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Pairs of fp32 values in one 64-bit register, for the paired fp32 instructions
// (one fma.f32x2 / add.f32x2 does the work of two scalar ones).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;\n" : "=f"(lo), "=f"(hi) : "l"(v));
  return make_float2(lo, hi);
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Maximum of v over the 32 lanes of a full warp (one redux instruction; NaN inputs
// are ignored like fmaxf does).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(v));
  return r;
}

// Programmatic dependent launch. An attention kernel lets the merge kernel that
// follows it on the stream be launched at once; the merge runs its prologue (which
// reads only the call's inputs), then waits for the attention kernel to complete and
// its writes to be visible before it reads the workspace or writes any output.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Launch of a kernel that may start while the previous kernel on the stream is still
// running (it must call pdl_wait_primary() before depending on that kernel).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ void flag_status(int* dev_status, int bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

// --------------------------------------------------------------------------
// Balanced split of the decode work.
//
// The work of a decode call is the list of (sequence b, kv head g, live block j)
// tiles, ordered by b, then g, then j. A sequence of length len has live blocks
// [jlo, jhi) with jhi = ceil(len / bs) and, for a window W > 0,
// jlo = floor(max(0, len - W) / bs) (blocks wholly before the window are never
// read). The tiles of one (b, g) form a segment. CTA i of G processes tiles
// [floor(i*T/G), floor((i+1)*T/G)), so every CTA streams the same number of
// blocks (+-1). A maximal run of one CTA's tiles inside one segment is a piece;
// a piece that starts at its segment's first tile stores its partial result in
// slot b*H_kv + g, any other piece in slot B*H_kv + i. A segment whose tiles all
// fall in one CTA is finished by that CTA directly.
// --------------------------------------------------------------------------
struct SeqRange {
  int jlo, n;  // first live block, number of live blocks
};

// Lengths are clamped to [0, max_blocks * bs] so that no table row is indexed past
// its end; the attention kernels flag PKV_DEV_BAD_LENGTH when a clamp happens.
__device__ __forceinline__ int clamp_len(int len, int cap) { return len < 0 ? 0 : (len > cap ? cap : len); }

__device__ __forceinline__ SeqRange live_blocks(int len, int bs, int window) {
  SeqRange r;
  if (len <= 0) {
    r.jlo = 0;
    r.n = 0;
    return r;
  }
  int jhi = (len + bs - 1) / bs;
  int lo = (window > 0 && len > window) ? len - window : 0;
  r.jlo = lo / bs;
  r.n = jhi - r.jlo;
  return r;
}

__device__ __forceinline__ int64_t cta_tile_start(int64_t i, int64_t T, int64_t G) {
  return (i * T) / G;
}

// Cursor over one CTA's tiles. All threads of a CTA walk identical cursors.
struct TileCursor {
  int b, g, j;          // current tile (j relative to jlo)
  int jlo, n;           // live range of sequence b
  int len;              // length of sequence b
  int64_t seg_base;     // global index of tile (b, g, 0)
  int64_t t, t_end;     // current global tile index, end of this CTA's range
};

// Sum of live blocks over all sequences (one warp, result in every lane).
__device__ __forceinline__ int64_t total_live_blocks(const int* seq_lens, int B, int bs, int window,
                                                     int cap, int* dev_status) {
  int64_t s = 0;
  for (int b = threadIdx.x & 31; b < B; b += 32) {
    const int raw = __ldg(seq_lens + b);
    const int len = clamp_len(raw, cap);
    if (len != raw && blockIdx.x == 0) flag_status(dev_status, PKV_DEV_BAD_LENGTH);
    s += live_blocks(len, bs, window).n;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Position the cursor at global tile t (a single thread's scan; B is small).
__device__ inline void cursor_seek(TileCursor& c, const int* seq_lens, int B, int Hkv, int bs,
                                   int window, int cap, int64_t t, int64_t t_end) {
  c.t = t;
  c.t_end = t_end;
  int64_t base = 0;
  c.b = B;
  c.g = 0;
  c.j = 0;
  c.jlo = 0;
  c.n = 0;
  c.len = 0;
  c.seg_base = 0;
  if (t >= t_end) return;
  for (int b = 0; b < B; ++b) {
    int len = clamp_len(__ldg(seq_lens + b), cap);
    SeqRange r = live_blocks(len, bs, window);
    int64_t seg = (int64_t)r.n * Hkv;
    if (t < base + seg) {
      int64_t off = t - base;
      c.b = b;
      c.g = (int)(off / r.n);
      c.j = (int)(off % r.n);
      c.jlo = r.jlo;
      c.n = r.n;
      c.len = len;
      c.seg_base = base + (int64_t)c.g * r.n;
      return;
    }
    base += seg;
  }
}

// Advance to the next tile; returns false when the CTA's range is exhausted.
__device__ inline bool cursor_next(TileCursor& c, const int* seq_lens, int B, int Hkv, int bs,
                                   int window, int cap) {
  ++c.t;
  if (c.t >= c.t_end) return false;
  if (++c.j < c.n) return true;
  c.j = 0;
  c.seg_base += c.n;
  if (++c.g < Hkv) return true;
  c.g = 0;
  for (;;) {
    if (++c.b >= B) return false;
    c.len = clamp_len(__ldg(seq_lens + c.b), cap);
    SeqRange r = live_blocks(c.len, bs, window);
    c.jlo = r.jlo;
    c.n = r.n;
    if (r.n > 0) return true;
  }
}

// First CTA whose range starts at or before tile `t`.
__device__ __forceinline__ int64_t cta_of_tile(int64_t t, int64_t T, int64_t G) {
  return ((t + 1) * G + T - 1) / T - 1;
}

}  // namespace pkv
