// Paged decode attention over an FP8 (E4M3) KV cache, dequantised inside the kernel.
//
// The pages' quantised caches (INT8 / W8A8C8 in the skill note; KIVI-style grouped
// quantisation in "KV Cache 笔记") halve or quarter the bytes decode reads, and the
// latter page warns that dequantising into temporary tensors every step eats that
// saving. Here nothing is materialised: the kernel reads E4M3 codes and per-row
// fp32 scales (one scale per (token, kv head); value = code * scale) and widens
// the codes on chip.
//
// Same contraction as the bf16 tcgen05 kernel (swap AB, N = 16 heads):
//   S^T [128 tok x 16] = K'[128 tok x 128 d] . Q'^T      K' in tensor memory (A operand)
//   O^T [128 d x 16]   = V'^T . P'^T                     V' in shared memory
// with f16 operands (kind::f16, fp32 accumulate):
//   K' = E4M3 codes widened to f16 (exact); the K scale multiplies S^T per token lane.
//   Q' = q * 2^e_h in f16 (exact for bf16 q; e_h puts the head's max near 2^14),
//        undone on S^T.
//   V' = E4M3 codes widened to f16 (exact); rows of invalid positions are zeroed,
//        so unwritten cache bytes (possibly NaN codes) never reach O.
//   P' = p * v_scale[token] / f_j in f16, f_j = the tile's largest V scale; O^T of
//        the tile is multiplied back by f_j when it is folded into the output. The
//        normaliser sums the fp32 weights p.
//
// Work split and merge: the balanced (b, kv head, block) tile list and partial
// pieces of the bf16 kernels (device_common.cuh), one persistent CTA per SM.
// Warp roles (608 threads):
//   warp 0       TMA: Q (bf16) per piece; per tile the K and V code tiles
//                (box {128 bytes, 1 head, 128 tokens}, 128-byte swizzle) and the
//                two 512-byte scale rows (bulk copy), 4-deep ring;
//   warp 1       score-product issuer; warp 18 value-product issuer;
//   warps 2-9    softmax, two groups of four warps: group g owns half of the heads
//                of every token row (thread = token lane of S^T / d lane of O^T);
//                both groups convert Q at each piece start;
//   warps 10-13  K converters: thread = token row; 128 codes -> 64 f16 pairs ->
//                tcgen05.st into the K' ring in tensor memory;
//   warps 14-17  V converters: thread = token row; codes -> f16 rows of V' in the
//                128-byte-swizzled layout the MMA reads, zero for invalid rows.
// All waits are bounded (tc_ptx.cuh); a timeout sets PKV_DEV_TIMEOUT.
//
// Roofline: HBM. Algorithmic bytes per tile = 2 * 128 * 128 (codes) + 2 * 512
// (scales) = 33,792.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "device_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {

bool make_tmap_sw128(CUtensorMap* m, CUtensorMapDataType dtype, const void* ptr, int rank,
                     const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                     CUtensorMapL2promotion promo);

namespace f8d {

constexpr int D = 128;
constexpr int BS = 128;
constexpr int N = 16;                  // MMA N: heads padded to 16
#ifndef PKV_F8_NSTG
#define PKV_F8_NSTG 4
#endif
constexpr int NSTG = PKV_F8_NSTG;      // code / scale staging ring
// K' and V' rings are two deep, like the S^T and O^T buffers: the converters of
// tile j reuse the buffers of tile j-2 once that tile's score (value) product has
// completed, which they learn from the same SFULL (OFULL) barrier the softmax waits
// on, so the MMA thread commits only SFULL and OFULL per tile.
constexpr int NKOP = 2;
constexpr int NVOP = 2;
constexpr int NTHREADS = 608;             // + the value-product issuer (warp 18)
constexpr int NSOFT = 256;             // softmax threads: two warps per TMEM lane quarter
constexpr int CTILE = BS * D;          // 16 KB of codes: [128 tokens x 128 bytes], swizzled
constexpr int HALF = 16384;            // f16 [128 rows x 64], one d half, swizzled
constexpr int VOPB = 2 * HALF;         // one V' tile
constexpr int QBUF = 4096;             // 16 rows x 128 d (16-bit), two 2 KB halves
constexpr int PBUF = 4096;             // 128 tokens x 16 heads (16-bit), MN-major
constexpr int SCB = 1024;              // 128 K scales + 128 V scales

constexpr int OFF_KST = 0;
constexpr int OFF_VST = OFF_KST + NSTG * CTILE;
constexpr int OFF_VOP = OFF_VST + NSTG * CTILE;
constexpr int OFF_QST = OFF_VOP + NVOP * VOPB;   // bf16 Q from TMA
constexpr int OFF_QOP = OFF_QST + 2 * QBUF;      // f16 Q' operand
constexpr int OFF_P = OFF_QOP + 2 * QBUF;
constexpr int OFF_SC = OFF_P + 2 * PBUF;
constexpr int OFF_BAR = OFF_SC + NSTG * SCB;
enum {
  B_KSTF = 0,
  B_KSTE = B_KSTF + NSTG,
  B_VSTF = B_KSTE + NSTG,
  B_VSTE = B_VSTF + NSTG,
  B_SCF = B_VSTE + NSTG,
  B_SCE = B_SCF + NSTG,
  B_KOPF = B_SCE + NSTG,
  B_VOPF = B_KOPF + NKOP,
  B_QSTF = B_VOPF + NVOP,
  B_QSTE = B_QSTF + 2,
  B_QOPF = B_QSTE + 2,
  B_QOPE = B_QOPF + 2,
  B_SFULL = B_QOPE + 2,
  B_PFULL = B_SFULL + 2,
  B_OFULL = B_PFULL + 2,
  B_SEMPTY = B_OFULL + 2,  // the softmax has read S^T (count NSOFT)
  B_COUNT = B_SEMPTY + 2
};
constexpr int OFF_RED = OFF_BAR + B_COUNT * 8;       // float [2][4][16] block max per head
constexpr int OFF_FRED = OFF_RED + 2 * 4 * 16 * 4;   // float [2][4] largest V scale per warp
constexpr int OFF_LRED = OFF_FRED + 2 * 4 * 4;       // float [4][16] normaliser partials
constexpr int OFF_QM = OFF_LRED + 4 * 16 * 4;        // float [16] 2^-e_h of the piece
constexpr int OFF_MISC = OFF_QM + 16 * 4;            // tmem addr, abort, total, snapshots
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// TMEM columns: S^T at 0 and 16, O^T at 32 and 48, K' buffers from 64 on.
constexpr uint32_t TMEM_COLS = 64 + 64 * NKOP <= 256 ? 256 : 512;
__device__ __forceinline__ uint32_t s_col(int b) { return b * 16; }
__device__ __forceinline__ uint32_t o_col(int b) { return 32 + b * 16; }
__device__ __forceinline__ uint32_t k_col(int b) { return 64 + b * 64; }

// Byte offset of 16-byte chunk `c` of row `row` in a 128-byte-swizzled [rows x 128 B] tile.
__device__ __forceinline__ uint32_t sw_chunk(int row, int c) {
  return (uint32_t)(row * 128 + (((c ^ row) & 7) << 4));
}

#ifndef PKV_F8_CVT
#define PKV_F8_CVT 1
#endif
// Widening of E4M3 codes to f16 (kWidenScale = the factor the f16 value carries).
//  1: cvt.rn.f16x2.e4m3x2, the exact value (factor 1).
//  2: bit placement: the code's 7 magnitude bits shifted left by 7 and its sign to
//     bit 15 form the f16 whose value is the code's value times 2^-8. Both formats
//     have 3 mantissa bits under an exponent field; E4M3 has bias 7, f16 bias 15,
//     and E4M3 subnormals (exponent field 0, m * 2^-9) land on f16 subnormals
//     (m * 2^7 * 2^-24) with the same factor. The NaN code 0x7F becomes a finite
//     value, which only matters for positions that are masked or zeroed anyway.
constexpr float kWidenScale = PKV_F8_CVT == 2 ? 256.f : 1.f;

// 16 E4M3 codes -> 8 packed f16 pairs (element 2i in the low half).
__device__ __forceinline__ void widen16(const uint4& w, uint32_t (&h)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#if PKV_F8_CVT == 1
    uint32_t lo, hi;
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
        " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(u[i]));
    h[2 * i] = lo;
    h[2 * i + 1] = hi;
#else
    const uint32_t t0 = __byte_perm(u[i], 0u, 0x4140);  // [0, b1, 0, b0]
    const uint32_t t1 = __byte_perm(u[i], 0u, 0x4342);  // [0, b3, 0, b2]
    h[2 * i] = ((t0 & 0x007F007Fu) << 7) | ((t0 & 0x00800080u) << 8);
    h[2 * i + 1] = ((t1 & 0x007F007Fu) << 7) | ((t1 & 0x00800080u) << 8);
#endif
  }
}

}  // namespace f8d

template <int NREP>
__global__ void __launch_bounds__(f8d::NTHREADS, 1)
    decode_fp8_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q) {
  using namespace f8d;
  using namespace tc;
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();  // the merge may launch now; it waits for this grid
  pdl_wait_primary();      // inputs may come from the kernel before (the cache write)
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  long long* total_s = reinterpret_cast<long long*>(misc + 2);
  volatile uint32_t* abort_snap = misc + 4;  // [2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cap = a.max_blocks * BS;

  if (tid == 0) {
    for (int i = 0; i < NSTG; ++i) {
      mbar_init(bar(B_KSTF + i), 1);
      mbar_init(bar(B_KSTE + i), 128);
      mbar_init(bar(B_VSTF + i), 1);
      mbar_init(bar(B_VSTE + i), 128);
      mbar_init(bar(B_SCF + i), 1);
      mbar_init(bar(B_SCE + i), NSOFT);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_KOPF + i), 128);
      mbar_init(bar(B_VOPF + i), 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_QSTF + i), 1);
      mbar_init(bar(B_QSTE + i), NSOFT);
      mbar_init(bar(B_QOPF + i), NSOFT);
      mbar_init(bar(B_QOPE + i), 1);
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), NSOFT);
      mbar_init(bar(B_OFULL + i), 1);
      mbar_init(bar(B_SEMPTY + i), NSOFT);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    const int64_t tot = total_live_blocks(a.seq_lens, a.B, BS, a.window, cap, a.dev_status);
    if (lane == 0) {
      *total_s = tot * a.Hkv;
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(sbase + OFF_MISC, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int64_t T = *total_s, G = gridDim.x;
  const int64_t t0 = cta_tile_start(blockIdx.x, T, G), t1 = cta_tile_start(blockIdx.x + 1, T, G);
  const int ntiles = (int)(t1 - t0);

  auto fail = [&]() {
    *abort_flag = 1;
    flag_status(a.dev_status, PKV_DEV_TIMEOUT);
  };

  if (ntiles > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap, t0, t1);
    int piece = 0;
    const int rows_oob = (int)(a.num_blocks * BS);  // first row past the cache: zero fill
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      if (j == 0 || c.j == 0) {
        const int qb = piece & 1;
        if (!mbar_wait(bar(B_QSTE + qb), ((piece >> 1) & 1) ^ 1)) { fail(); break; }
        mbar_expect_tx(bar(B_QSTF + qb), QBUF);
        const int qrow = c.b * a.H + c.g * NREP;
        const uint32_t qs = sbase + OFF_QST + qb * QBUF;
        tma_load_2d(qs, &tm_q, bar(B_QSTF + qb), 0, qrow);
        tma_load_2d(qs + QBUF / 2, &tm_q, bar(B_QSTF + qb), 64, qrow);
        ++piece;
      }
      const int st = j % NSTG, ph = ((j / NSTG) & 1) ^ 1;
      if (!mbar_wait(bar(B_KSTE + st), ph) || !mbar_wait(bar(B_VSTE + st), ph) ||
          !mbar_wait(bar(B_SCE + st), ph)) { fail(); break; }
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
      const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      if (!ok) flag_status(a.dev_status, PKV_DEV_BAD_BLOCK);
      const int row = ok ? blk * BS : rows_oob;
      mbar_expect_tx(bar(B_KSTF + st), CTILE);
      tma_load_3d(sbase + OFF_KST + st * CTILE, &tm_k, bar(B_KSTF + st), 0, c.g, row);
      mbar_expect_tx(bar(B_VSTF + st), CTILE);
      tma_load_3d(sbase + OFF_VST + st * CTILE, &tm_v, bar(B_VSTF + st), 0, c.g, row);
      if (ok) {
        const int64_t so = ((int64_t)blk * a.Hkv + c.g) * BS;
        mbar_expect_tx(bar(B_SCF + st), SCB);
        bulk_load(sbase + OFF_SC + st * SCB, a.k_scale + so, SCB / 2, bar(B_SCF + st));
        bulk_load(sbase + OFF_SC + st * SCB + SCB / 2, a.v_scale + so, SCB / 2, bar(B_SCF + st));
      } else {
        mbar_arrive(bar(B_SCF + st));  // no scales: the softmax masks the whole tile
      }
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
    }
  } else if (ntiles > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ score-product issuer
    // Two issuing threads: this one issues S^T(j) once K'(j) is widened and the
    // softmax has read S^T(j-2) (SEMPTY); warp 18 issues the value products. O(j) reuses
    // the O^T buffer and P' buffer of tile j-2, which the softmax has folded (resp.
    // released) before it arrives PFULL(j). Each thread's commits track only its own MMAs.
    constexpr uint32_t ID_S = idesc_f16(128, N, 0, 0);  // K' (TMEM) x Q'^T (K-major smem)
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap, t0, t1);
    int piece = -1;
    bool ok = true;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      const bool last = (j + 1 == ntiles) || (c.j + 1 == c.n);
      if (first) ++piece;
      const int qb = piece & 1, kb = j % NKOP, sb = j & 1;
      if (first && !mbar_wait(bar(B_QOPF + qb), (piece >> 1) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_KOPF + kb), (j / NKOP) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_SEMPTY + sb), ((j >> 1) & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      const uint64_t qd = smem_desc(sbase + OFF_QOP + qb * QBUF, 16, 1024, kSwizzle128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tmem + s_col(sb), tmem + k_col(kb) + kk * 8,
               desc_add(qd, (kk >> 2) * (QBUF / 2) + (kk & 3) * 32), ID_S, kk > 0);
      mma_commit(bar(B_SFULL + sb));
      if (last) mma_commit(bar(B_QOPE + qb));
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
    }
    if (!ok) fail();
  } else if (ntiles > 0 && warp == 18 && lane == 0) {
    // ------------------------------------------------------------ value-product issuer
    constexpr uint32_t ID_O = idesc_f16(128, N, 1, 1);  // V'^T (MN-major) x P'^T (MN-major)
    bool ok = true;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const int vb = j % NVOP, ob = j & 1;
      if (!mbar_wait(bar(B_VOPF + vb), (j / NVOP) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_PFULL + ob), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint64_t vd = smem_desc(sbase + OFF_VOP + vb * VOPB, HALF, 1024, kSwizzle128);
      // P'^T, MN-major without swizzle: 8 heads x 8 tokens per 128-byte core matrix;
      // the stride field (SBO) steps along MN (head groups, 128 bytes apart), the
      // leading field (LBO) along K (8-token groups, 256 bytes apart).
      const uint64_t pd = smem_desc(sbase + OFF_P + ob * PBUF, N * 16, 128, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + o_col(ob), desc_add(vd, kk * 2048),
               desc_add(pd, kk * 2 * N * 16), ID_O, kk > 0);
      mma_commit(bar(B_OFULL + ob));
    }
    if (!ok) fail();
  } else if (ntiles > 0 && warp >= 10 && warp < 14) {
    // ------------------------------------------------------------ K converters
    // Thread = token row r: 128 codes -> 64 f16 pairs in columns k_col(kb)..+63 of
    // TMEM lane r (the A operand of the score product). Warp-uniform decisions only:
    // tcgen05.st is warp-collective.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int st = j % NSTG, kb = j % NKOP;
      bool ok = mbar_wait(bar(B_KSTF + st), (j / NSTG) & 1);
      ok = ok && (j < 2 || mbar_wait(bar(B_SFULL + kb), ((j >> 1) & 1) ^ 1));  // S(j-2) done
      if (!__all_sync(0xffffffffu, ok)) { fail(); break; }
      tc_fence_after();
      const uint8_t* src = base + OFF_KST + st * CTILE;
      uint4 w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const uint4*>(src + sw_chunk(r, c));
      mbar_arrive(bar(B_KSTE + st));
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t h[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t p[8];
          widen16(w[4 * hf + c], p);
#pragma unroll
          for (int i = 0; i < 8; ++i) h[8 * c + i] = p[i];
        }
        tmem_st32(tmem + lane_off + k_col(kb) + 32 * hf, h);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_KOPF + kb));
    }
  } else if (ntiles > 0 && warp >= 14 && warp < 18) {
    // ------------------------------------------------------------ V converters
    // Thread = token row r: codes -> f16 row r of V' (two 64-wide swizzled halves);
    // rows of positions the softmax masks are written as zeros.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap, t0, t1);
    int blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int blk = blk_next;
      const int st = j % NSTG, vb = j % NVOP;
      bool ok = mbar_wait(bar(B_VSTF + st), (j / NSTG) & 1);
      ok = ok && (j < 2 || mbar_wait(bar(B_OFULL + vb), ((j >> 1) & 1) ^ 1));  // O(j-2) done
      tc_fence_after();
      if (!__all_sync(0xffffffffu, ok)) { fail(); break; }
      const int lo = (a.window > 0 && c.len > a.window) ? c.len - a.window : 0;
      const int pos = (c.jlo + c.j) * BS + r;
      const bool valid = blk >= 0 && (int64_t)blk < a.num_blocks && pos < c.len && pos >= lo;
      const uint8_t* src = base + OFF_VST + st * CTILE;
      uint4 w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) w[q] = *reinterpret_cast<const uint4*>(src + sw_chunk(r, q));
      mbar_arrive(bar(B_VSTE + st));
      uint8_t* dst = base + OFF_VOP + vb * VOPB;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t p[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (valid) widen16(w[q], p);
        uint8_t* hb = dst + (q >> 2) * HALF;
        const int kc = 2 * (q & 3);
        *reinterpret_cast<uint4*>(hb + sw_chunk(r, kc)) = make_uint4(p[0], p[1], p[2], p[3]);
        *reinterpret_cast<uint4*>(hb + sw_chunk(r, kc + 1)) = make_uint4(p[4], p[5], p[6], p[7]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_VOPF + vb));
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
      if (j + 1 < ntiles) blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
    }
  } else if (ntiles > 0 && warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ softmax / epilogue
    constexpr int HG = NREP > 1 ? NREP / 2 : 1;   // heads per group
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int grp = (warp - 2) >> 2;              // head group
    const int h0 = grp * HG;                      // first head of the group
    const bool has_heads = h0 < NREP;             // false only for group 1 when NREP == 1
    const int r = quarter * 32 + lane;            // token row of S^T, d row of O^T
    const int ts = grp * 128 + r;                 // thread index among the 256
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float* red = reinterpret_cast<float*>(base + OFF_RED);
    float* fred = reinterpret_cast<float*>(base + OFF_FRED);
    float* lred = reinterpret_cast<float*>(base + OFF_LRED);
    float* qm = reinterpret_cast<float*>(base + OFF_QM);
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap, t0, t1);
    // Online softmax with a lazily moved reference (log2 units): m_run changes only
    // when a block max exceeds it by more than kLazy, so most tiles skip the
    // rescale; it starts at a large finite negative value, so no -inf arithmetic is
    // needed. o_reg is kept in the reference of the newest tile whose scores are
    // done: acc_o(j - 1) runs after tile j's rescale factors are known.
    constexpr float kLazy = 8.f;
    constexpr float kMinit = -1e30f;
    float m_run[HG], l_part[HG], o_reg[HG], alpha[HG], qmul[HG];
    bool resc = false;
    float f_prev = 1.f;
    int pb = 0, pg = 0, piece = -1;
    int64_t p_first = t0, p_segbase = 0;
    bool p_whole = false, aborted = false;

    // Q' of a new piece: thread ts converts 8 values of row h = ts / 16; the row is
    // scaled by 2^e_h with its max near 2^14, widened exactly to f16 and written in the
    // layout the score product reads; 2^-e_h goes to qm[h].
    auto convert_q = [&]() -> bool {
      const int qb = piece & 1;
      bool ok = mbar_wait(bar(B_QSTF + qb), (piece >> 1) & 1);
      ok = mbar_wait(bar(B_QOPE + qb), ((piece >> 1) & 1) ^ 1) && ok;
      const int h = ts >> 4, c16 = ts & 15, kc = c16 & 7;
      const uint8_t* src = base + OFF_QST + qb * QBUF + (c16 >> 3) * (QBUF / 2);
      uint8_t* dst = base + OFF_QOP + qb * QBUF + (c16 >> 3) * (QBUF / 2);
      const uint4 x0 = *reinterpret_cast<const uint4*>(src + sw_chunk(h, kc));
      mbar_arrive(bar(B_QSTE + qb));
      const uint32_t u[4] = {x0.x, x0.y, x0.z, x0.w};
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[i] << 16)),
                                 fabsf(__uint_as_float(u[i] & 0xffff0000u))));
#pragma unroll
      for (int o = 8; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int e = 0;
      if (amax > 0.f) {
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127;  // floor(log2 amax)
        e = min(127, max(-126, 14 - ex));
      }
      const float mul = __uint_as_float((uint32_t)(127 + e) << 23);
      uint32_t y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 hv = __floats2half2_rn(__uint_as_float(u[i] << 16) * mul,
                                             __uint_as_float(u[i] & 0xffff0000u) * mul);
        y[i] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(dst + sw_chunk(h, kc)) = make_uint4(y[0], y[1], y[2], y[3]);
      if (c16 == 0) qm[h] = __uint_as_float((uint32_t)(127 - e) << 23);
      fence_proxy_async_smem();
      named_bar_sync(1, NSOFT);
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) qmul[hh] = has_heads ? qm[h0 + hh] : 0.f;
      mbar_arrive(bar(B_QOPF + qb));
      return ok;
    };
    auto acc_o = [&](int jj, bool rs) {
      const int ob = jj & 1;
      if (!mbar_wait(bar(B_OFULL + ob), (jj >> 1) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(tmem + lane_off + o_col(ob), v);
      tmem_wait_ld();
      tc_fence_before();  // ordered before the next PFULL arrive, which frees O^T(jj)
      if (rs) {
#pragma unroll
        for (int h = 0; h < HG; ++h)
          o_reg[h] = (o_reg[h] + f_prev * __uint_as_float(grp ? v[(HG + h) & 15] : v[h])) * alpha[h];
      } else {
#pragma unroll
        for (int h = 0; h < HG; ++h)
          o_reg[h] += f_prev * __uint_as_float(grp ? v[(HG + h) & 15] : v[h]);
      }
    };
    auto finalize = [&]() {
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float l = l_part[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0 && has_heads) lred[quarter * 16 + h0 + h] = l;
      }
      named_bar_sync(1, NSOFT);
      const int64_t slot = (p_first == p_segbase) ? (int64_t)pb * a.Hkv + pg
                                                  : (int64_t)a.B * a.Hkv + blockIdx.x;
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        const int h = h0 + hh;
        if (!has_heads || h >= NREP) continue;
        const float l = lred[h] + lred[16 + h] + lred[32 + h] + lred[48 + h];
        const float ov = l > 0.f ? o_reg[hh] / l : 0.f;
        const float lse2 = l > 0.f ? m_run[hh] + log2f(l) : -INFINITY;
        if (p_whole) {
          const int64_t row = (int64_t)pb * a.H + (int64_t)pg * NREP + h;
          if (a.out_f32)
            reinterpret_cast<float*>(a.out)[row * D + r] = ov;
          else
            reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + r] = __float2bfloat16_rn(ov);
          if (a.lse && r == 0) a.lse[row] = lse2 * kLn2;
        } else {
          a.ws_o[(slot * NREP + h) * D + r] = ov;
          if (r == 0) a.ws_lse[slot * NREP + h] = lse2;
        }
      }
      named_bar_sync(1, NSOFT);  // lred reused by the next piece
    };

    // The tile's block id is loaded one tile ahead, so that its latency is not on
    // the path from S^T to P'.
    int blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
    for (int j = 0; j < ntiles; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      const int blk = blk_next;
      if (first) {
        ++piece;
        if (!convert_q()) fail();
        if (j > 0) {
          acc_o(j - 1, false);
          finalize();
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          m_run[h] = kMinit;
          l_part[h] = 0.f;
          o_reg[h] = 0.f;
        }
        f_prev = 1.f;
        pb = c.b;
        pg = c.g;
        p_first = c.t;
        p_segbase = c.seg_base;
        p_whole = (c.t == c.seg_base) && (c.t + c.n <= t1);
      }
      // ---- scales and scores of tile j
      const int st = j % NSTG, sb = j & 1;
      if (!mbar_wait(bar(B_SCF + st), (j / NSTG) & 1)) fail();
      const float* scs = reinterpret_cast<const float*>(base + OFF_SC + st * SCB);
      const float sk = scs[r], sv = scs[128 + r];
      mbar_arrive(bar(B_SCE + st));
      if (!mbar_wait(bar(B_SFULL + sb), (j >> 1) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      uint32_t svr[16];
      tmem_ld16(tmem + lane_off + s_col(sb), svr);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SEMPTY + sb));  // S^T(j) is in registers: S^T(j+2) may overwrite it

      const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int lo = (a.window > 0 && c.len > a.window) ? c.len - a.window : 0;
      const int pos = (c.jlo + c.j) * BS + r;
      const bool valid = blk_ok && pos < c.len && pos >= lo;
      const float smul = sk * kWidenScale * a.scale_log2;
      float x[HG];
      bool over = false;  // a score of this thread beats its head's reference by > kLazy
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        // Column h0 + h, chosen between two compile-time indices (no local memory).
        const uint32_t sx = grp ? svr[(HG + h) & 15] : svr[h];
        x[h] = (valid && has_heads) ? __uint_as_float(sx) * (smul * qmul[h]) : -INFINITY;
        over |= x[h] > m_run[h] + kLazy;
      }
      if (grp == 0) {
        const float fv = warp_max(valid ? sv : 0.f);
        if (lane == 0) fred[sb * 4 + quarter] = fv;
      }
      if (ts == 0) abort_snap[sb] = *abort_flag;
      // One barrier publishes the V-scale maxima and tells every thread whether any
      // score of the tile beats its reference: most tiles need no block max at all.
      const bool any_over = named_bar_any(1, NSOFT, over);
      if (abort_snap[sb]) {
        aborted = true;
        break;
      }
      float f = fmaxf(fmaxf(fred[sb * 4], fred[sb * 4 + 1]), fmaxf(fred[sb * 4 + 2], fred[sb * 4 + 3]));
      f = f > 0.f ? f : 1.f;
      const float vmul = valid ? __fdividef(sv, f) : 0.f;
      resc = false;
      if (any_over) {
        // Block max per head and the reference test; both groups read the same
        // maxima for their own heads, so `resc` is uniform within a group.
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float m = warp_max(x[h]);
          if (lane == 0 && has_heads) red[(sb * 4 + quarter) * 16 + h0 + h] = m;
        }
        named_bar_sync(1, NSOFT);
        float mb[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float* rr = red + sb * 64 + h0 + h;
          mb[h] = has_heads ? fmaxf(fmaxf(rr[0], rr[16]), fmaxf(rr[32], rr[48])) : -INFINITY;
          resc |= mb[h] > m_run[h] + kLazy;
        }
        if (resc) {
#pragma unroll
          for (int h = 0; h < HG; ++h) {
            const float mn = fmaxf(m_run[h], mb[h]);
            alpha[h] = exp2f(m_run[h] - mn);
            m_run[h] = mn;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float p = exp2f(x[h] - m_run[h]);  // a masked score is -inf: weight 0
        l_part[h] = resc ? l_part[h] * alpha[h] + p : l_part[h] + p;
        x[h] = p * vmul;  // P' = p * v_scale / f
      }
      // ---- P'^T (f16) of the group's heads into the B operand of the value product
      // (O(j-2), its last reader, is complete: acc_o(j-2) waited for it): heads
      // h0..h0+HG-1 of token r are HG contiguous halves of the 16-byte row r % 8 of
      // core matrix (r / 8, h0 / 8). Columns of heads >= NREP are never written and
      // only feed O^T columns that are never read.
      if (has_heads) {
        uint8_t* ps = base + OFF_P + sb * PBUF + (r >> 3) * (N * 16) + (r & 7) * 16 +
                      (h0 >> 3) * 128 + (h0 & 7) * 2;
        if constexpr (HG == 1) {
          *reinterpret_cast<__half*>(ps) = __float2half_rn(x[0]);
        } else {
          uint32_t pk[HG / 2];
#pragma unroll
          for (int i = 0; i < HG / 2; ++i) {
            const __half2 h2 = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          if constexpr (HG == 2) *reinterpret_cast<uint32_t*>(ps) = pk[0];
          if constexpr (HG == 4) *reinterpret_cast<uint2*>(ps) = make_uint2(pk[0], pk[1]);
          if constexpr (HG == 8) *reinterpret_cast<uint4*>(ps) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_PFULL + sb));
      // Tile j's values are all computed; advance and start the next block-id load.
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
      if (j + 1 < ntiles) blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
      // ---- fold the previous tile's O^T into the registers, with this tile's rescale
      if (!first) acc_o(j - 1, resc);
      f_prev = f * kWidenScale;  // O^T of this tile carries V' = value * code factor / f
    }
    if (!aborted) {
      acc_o(ntiles - 1, false);
      finalize();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
template <int NREP>
static cudaError_t launch_fp8_n(const DecodeArgs& a, cudaStream_t stream) {
  using namespace f8d;
  CUtensorMap tk, tv, tq;
  const uint64_t rows = (uint64_t)a.num_blocks * BS;
  const uint64_t kdims[3] = {D, (uint64_t)a.Hkv, rows};  // bytes: one code per element
  const uint64_t kstr[2] = {D, (uint64_t)a.Hkv * D};
  const uint32_t kbox[3] = {D, 1, BS};
  const uint64_t qdims[2] = {D, (uint64_t)a.B * a.H};
  const uint64_t qstr[1] = {D * 2};
  const uint32_t qbox[2] = {64, 16};
  // A code row of one kv head is 128 bytes and the next head's row follows it: a
  // 256-byte L2 promotion would fetch that neighbour, which this CTA does not read.
  if (!make_tmap_sw128(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_cache, 3, kdims, kstr, kbox,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
      !make_tmap_sw128(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v_cache, 3, kdims, kstr, kbox,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
      !make_tmap_sw128(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, 2, qdims, qstr, qbox,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel<NREP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_fp8_kernel<NREP>, dim3(a.num_ctas), dim3(NTHREADS), SMEM_BYTES, stream,
                          a, tk, tv, tq);
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.n_rep) {
    case 1: return launch_fp8_n<1>(a, stream);
    case 2: return launch_fp8_n<2>(a, stream);
    case 4: return launch_fp8_n<4>(a, stream);
    case 8: return launch_fp8_n<8>(a, stream);
    case 16: return launch_fp8_n<16>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
