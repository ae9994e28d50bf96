// Paged decode attention for GQA head groups on the tcgen05 tensor cores.
//
// Same result as the CUDA-core kernel: for each (b, h), softmax(scale * q . K^T) V
// over the visible positions of sequence b read through block_table ("KV Cache 笔记",
// decode incremental form; GQA mapping h -> h / n_rep). The n_rep query heads of a
// kv head share every K/V tile, so each tile is a small dense contraction:
//
//   S^T [128 tokens x N] = K_tile [128 x 128 d] . Q_g^T        (M = 128)
//   O^T [128 d x N]      = V_tile^T [128 d x 128 tokens] . P^T (M = 128)
//
// ("swap AB": the token / d axis takes the M = 128 side of the MMA). Both products
// run as tcgen05.mma kind::f16 (bf16 in, fp32 accumulate in tensor memory).
//
// The same kernel runs speculative (multi-token) decode: with q_len = QL new rows
// per sequence (standalone guide, appendix C: a multi-token decode step takes the
// bottom-right causal mask of prefill), the QL * n_rep query rows of a kv head are
// the N columns, ordered (token, head). Query token i sits at position
// len - QL + i and sees keys p <= len - QL + i (and, with a window W, p > that
// position - W). The rows are padded to N = 16 or 32; each block of 16 columns has
// its own four softmax warps.
//
// Work split: the balanced (b, kv head, block) tile list of device_common.cuh, one
// persistent CTA per SM. Warp roles:
//   warp 0      TMA producer: Q of each piece (box {64 d, n_rep heads, QL tokens}),
//               K and V halves of each tile (box {64 d, 1 head, 128 tokens}),
//               128-byte swizzle, 3-deep ring;
//   warp 1      score-product issuer (S^T of a tile as soon as its K tile has landed
//               and its S^T buffer is free); warp 6 (N = 16) or 11 (N = 32) issues the
//               value products;
//   warps 2..   softmax, four warps per 16 columns: thread = token lane of S^T.
//               Block max per column by one warp redux plus a shared-memory
//               exchange; exp2 in fp32 with q . k pre-scaled by scale * log2 e;
//               P^T written as bf16 in the MN-major layout of the second
//               product's B operand (a thread's 16 columns are two 16-byte
//               stores); then thread = d lane of O^T, accumulating O in
//               registers with the online-softmax rescale.
// All waits are bounded (tc_ptx.cuh); a timeout sets PKV_DEV_TIMEOUT and every
// role winds down.
//
// Roofline: HBM. Algorithmic bytes per tile = 2 * 128 tokens * 128 d * 2 bytes.
#pragma once

#include <cuda.h>

#include "device_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace tcd {

constexpr int D = 128;
constexpr int BS = 128;
constexpr int NST = 3;
constexpr int HALF = 16384;          // [128 rows x 128 bytes], one 64-wide d half
constexpr int TILE = 2 * HALF;       // one K (or V) tile of one kv head

enum {
  B_KFULL = 0,
  B_VFULL = B_KFULL + NST,
  B_KVEMPTY = B_VFULL + NST,
  B_QFULL = B_KVEMPTY + NST,
  B_QEMPTY = B_QFULL + 2,
  B_SFULL = B_QEMPTY + 2,
  B_SEMPTY = B_SFULL + 2,
  B_PFULL = B_SEMPTY + 2,
  B_PEMPTY = B_PFULL + 2,
  B_OFULL = B_PEMPTY + 2,
  B_OEMPTY = B_OFULL + 2,
  B_COUNT = B_OEMPTY + 2
};

// One kernel instance: NR = QL * n_rep query rows per (b, kv head), padded to the
// MMA N; NCH blocks of 16 columns, each with four softmax warps.
template <int NREP, int QL>
struct Shape {
  static constexpr int NR = NREP * QL;
  static constexpr int N = NR <= 16 ? 16 : 32;
  static constexpr int NCH = N / 16;
  static constexpr int CW = NCH == 1 ? NR : 16;  // columns a softmax thread carries
  // A separate thread issues the value products, on the SM sub-partition with the
  // fewest softmax warps (warp 10 is idle when N = 32).
  static constexpr int OWARP = NCH == 1 ? 6 : 11;
  static constexpr int NTHREADS = 32 * (OWARP + 1);
  static constexpr int QBUF = N * 256;           // N rows x 128 d, two 64-wide halves
  static constexpr int PBUF = N * 256;           // 128 tokens x N columns, MN-major
  // Shared-memory layout (offsets from a 1024-aligned base).
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_Q = OFF_V + NST * TILE;
  static constexpr int OFF_P = OFF_Q + 2 * QBUF;
  static constexpr int OFF_BAR = OFF_P + 2 * PBUF;
  static constexpr int OFF_RED = (OFF_BAR + B_COUNT * 8 + 15) & ~15;  // float [2][4][N]
  static constexpr int OFF_LRED = OFF_RED + 2 * 4 * N * 4;  // float [4][N]
  static constexpr int OFF_MISC = OFF_LRED + 4 * N * 4;     // tmem addr, abort, total, snaps
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;   // + alignment slack
  // TMEM columns: S^T buffers at 0 and N, O^T buffers at 2N and 3N.
  static constexpr uint32_t TMEM_COLS = 4 * N;
  static_assert(NR <= 32, "at most 32 query rows per kv head");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

}  // namespace tcd

// O^T(j) += V^T(j) . P^T(j): waits for V(j), P^T(j) and the O^T buffer, issues the
// value product, and commits O full, P^T free and the K/V stage free (K(j) was read by
// S^T(j), complete before the softmax published P^T(j)). False on a wait timeout.
template <int NREP, int QL>
__device__ __forceinline__ bool issue_value(const DecodeArgs& a, uint32_t sbase, uint32_t tmem, int j) {
  using namespace tcd;
  using namespace tc;
  using L = Shape<NREP, QL>;
  constexpr int N = L::N, PBUF = L::PBUF, OFF_V = L::OFF_V, OFF_P = L::OFF_P, OFF_BAR = L::OFF_BAR;
  constexpr uint32_t ID_O = idesc_bf16(128, N, 1, 1);  // V^T (MN-major) x P^T (MN-major)
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  const int st = j % NST, ob = j & 1;
  if (!mbar_wait(bar(B_VFULL + st), (j / NST) & 1)) return false;
  if (!mbar_wait(bar(B_PFULL + ob), (j >> 1) & 1)) return false;
  if (!mbar_wait(bar(B_OEMPTY + ob), ((j >> 1) & 1) ^ 1)) return false;
  tc_fence_after();
  const uint64_t vd = smem_desc(sbase + OFF_V + st * TILE, HALF, 1024, kSwizzle128);
  // P^T, MN-major without swizzle: 8 columns x 8 tokens per 128-byte core matrix. In
  // this layout the descriptor's stride field (SBO) steps along MN (column groups, 128
  // bytes apart) and the leading field (LBO) along K (8-token groups, N * 16 bytes
  // apart), the reverse of the swizzled MN-major forms.
  const uint64_t pd = smem_desc(sbase + OFF_P + ob * PBUF, N * 16, 128, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ss(tmem + (uint32_t)(2 * N + ob * N), desc_add(vd, kk * 2048), desc_add(pd, kk * 2 * N * 16), ID_O,
           kk > 0);
  mma_commit(bar(B_OFULL + ob));
  mma_commit(bar(B_PEMPTY + ob));
  mma_commit(bar(B_KVEMPTY + st));
  return true;
}

template <int NREP, int QL>
__global__ void __launch_bounds__(tcd::Shape<NREP, QL>::NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q) {
  using namespace tcd;
  using namespace tc;
  using L = Shape<NREP, QL>;
  pdl_launch_dependents();  // the merge may launch now; it waits for this grid
  pdl_wait_primary();      // inputs may come from the kernel before (the cache write)
  constexpr int NR = L::NR, N = L::N, NCH = L::NCH, CW = L::CW;
  constexpr int QBUF = L::QBUF, PBUF = L::PBUF;
  constexpr int OFF_K = L::OFF_K, OFF_V = L::OFF_V, OFF_Q = L::OFF_Q, OFF_P = L::OFF_P;
  constexpr int OFF_BAR = L::OFF_BAR, OFF_MISC = L::OFF_MISC;
  constexpr uint32_t TMEM_COLS = L::TMEM_COLS;
  constexpr int NSOFT = 128 * NCH;  // softmax threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  auto s_col = [](int b) { return (uint32_t)(b * N); };
  auto o_col = [](int b) { return (uint32_t)(2 * N + b * N); };
  float* red = reinterpret_cast<float*>(base + L::OFF_RED);
  float* lred = reinterpret_cast<float*>(base + L::OFF_LRED);
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  long long* total_s = reinterpret_cast<long long*>(misc + 2);
  volatile uint32_t* abort_snap = misc + 4;  // [NCH][2]: flag as seen before each softmax barrier

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cap = a.max_blocks * BS;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_KVEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_QFULL + i), 1);
      mbar_init(bar(B_QEMPTY + i), 1);
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SEMPTY + i), NSOFT);
      mbar_init(bar(B_PFULL + i), NSOFT);
      mbar_init(bar(B_PEMPTY + i), 1);
      mbar_init(bar(B_OFULL + i), 1);
      mbar_init(bar(B_OEMPTY + i), NSOFT);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    const int64_t tot = total_live_blocks(a.seq_lens, a.B, BS, a.window, cap, a.dev_status);
    if (lane == 0) *total_s = tot * a.Hkv;
    if (lane == 0) {
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
  if constexpr (NR < N) {
    // Query rows NR..N-1 of both Q buffers are never loaded: zero them once, so the
    // padding columns of S^T are 0 instead of whatever the memory held.
    constexpr int PAD = (N - NR) * 128;  // bytes per 64-wide half
    for (int o = tid * 16; o < 4 * PAD; o += L::NTHREADS * 16) {
      const int half = o / PAD;  // buffer * 2 + d half
      *reinterpret_cast<uint4*>(base + OFF_Q + half * (QBUF / 2) + NR * 128 + o % PAD) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
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
        if (!mbar_wait(bar(B_QEMPTY + qb), ((piece >> 1) & 1) ^ 1)) { fail(); break; }
        mbar_expect_tx(bar(B_QFULL + qb), NR * 256);
        const uint32_t qs = sbase + OFF_Q + qb * QBUF;
        tma_load_3d(qs, &tm_q, bar(B_QFULL + qb), 0, c.g * NREP, c.b * QL);
        tma_load_3d(qs + QBUF / 2, &tm_q, bar(B_QFULL + qb), 64, c.g * NREP, c.b * QL);
        ++piece;
      }
      const int st = j % NST;
      if (!mbar_wait(bar(B_KVEMPTY + st), ((j / NST) & 1) ^ 1)) { fail(); break; }
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
      const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      if (!ok) flag_status(a.dev_status, PKV_DEV_BAD_BLOCK);
      const int row = ok ? blk * BS : rows_oob;
      const uint32_t ks = sbase + OFF_K + st * TILE, vs = sbase + OFF_V + st * TILE;
      mbar_expect_tx(bar(B_KFULL + st), TILE);
      tma_load_3d(ks, &tm_k, bar(B_KFULL + st), 0, c.g, row);
      tma_load_3d(ks + HALF, &tm_k, bar(B_KFULL + st), 64, c.g, row);
      mbar_expect_tx(bar(B_VFULL + st), TILE);
      tma_load_3d(vs, &tm_v, bar(B_VFULL + st), 0, c.g, row);
      tma_load_3d(vs + HALF, &tm_v, bar(B_VFULL + st), 64, c.g, row);
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
    }
  } else if (ntiles > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ score-product issuer
    // This thread issues the score products: S^T(j) once K(j) has landed and the softmax
    // has read the S^T buffer of tile j-2; warp OWARP issues the value products (one
    // thread issuing both in a fixed order measured 2-4 % slower). Each thread's
    // commits track only its own MMAs.
    constexpr uint32_t ID_S = idesc_bf16(128, N, 0, 0);  // K (K-major) x Q^T (K-major)
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap, t0, t1);
    int piece = -1;
    bool ok = true;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      const bool last = (j + 1 == ntiles) || (c.j + 1 == c.n);
      if (first) ++piece;
      const int qb = piece & 1, st = j % NST, sb = j & 1;
      if (first && !mbar_wait(bar(B_QFULL + qb), (piece >> 1) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_KFULL + st), (j / NST) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_SEMPTY + sb), ((j >> 1) & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      // Base descriptors once per tile; each K step only adds a constant offset.
      const uint64_t kd = smem_desc(sbase + OFF_K + st * TILE, 16, 1024, kSwizzle128);
      const uint64_t qd = smem_desc(sbase + OFF_Q + qb * QBUF, 16, 1024, kSwizzle128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + s_col(sb), desc_add(kd, (kk >> 2) * HALF + (kk & 3) * 32),
               desc_add(qd, (kk >> 2) * (QBUF / 2) + (kk & 3) * 32), ID_S, kk > 0);
      mma_commit(bar(B_SFULL + sb));
      if (last) mma_commit(bar(B_QEMPTY + qb));
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
    }
    if (!ok) fail();
  } else if (ntiles > 0 && warp == L::OWARP && lane == 0) {
    // ------------------------------------------------------------ value-product issuer
    bool ok = true;
    for (int j = 0; j < ntiles && !*abort_flag; ++j)
      if (!issue_value<NREP, QL>(a, sbase, tmem, j)) { ok = false; break; }
    if (!ok) fail();
  } else if (ntiles > 0 && warp >= 2 && warp < 2 + 4 * NCH) {
    // ------------------------------------------------------------ softmax / epilogue
    const int chunk = (warp - 2) >> 2;            // block of 16 columns
    const int qbase = chunk * 16;                 // first column of the block
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;            // token row of S^T, d row of O^T
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int bar_id = 1 + chunk;                 // named barrier of the block's 128 threads
    float* cred = red + qbase;                    // [2][4][N] from this block's first column
    float* clred = lred + qbase;                  // [4][N]
    volatile uint32_t* snap = abort_snap + 2 * chunk;
    // Columns of the block past the last query row (NR not a multiple of 16) see a
    // zero query row: their scores are 0 or masked, and nothing reads them.
    const int nreal = NR - qbase < CW ? NR - qbase : CW;
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap, t0, t1);
    // Online softmax with a lazily moved reference: m_run (log2 units) changes only
    // when a block's max exceeds it by more than kLazy, so most tiles skip the
    // rescale; weights stay below 2^kLazy, well inside bf16 and fp32. The result is
    // the same softmax (o = sum p v / sum p for any reference). m_run starts at a
    // large finite negative value, so no -inf arithmetic is needed anywhere.
    constexpr float kLazy = 8.f;
    constexpr float kMinit = -1e30f;
    // o_reg holds the output of the tiles folded so far. O(j - 1) is folded after
    // P(j) is published, or, when tile j raises the reference, before the rescale
    // of everything accumulated.
    // l_part sums the weights as the value product uses them (rounded to bf16) and
    // divides the output; le_part sums the exact fp32 weights and gives the
    // log-sum-exp (the reported lse and the weight of a split piece in the merge).
    float m_run[CW], l_part[CW], le_part[CW], o_reg[CW];
    // State of the piece being accumulated.
    int pb = 0, pg = 0;
    int64_t p_first = t0, p_segbase = 0;
    bool p_whole = false;
    bool aborted = false;

    auto acc_o = [&](int jj) {
      const int ob = jj & 1;
      if (!mbar_wait(bar(B_OFULL + ob), (jj >> 1) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(tmem + lane_off + o_col(ob) + qbase, v);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_OEMPTY + ob));
#pragma unroll
      for (int i = 0; i < CW; ++i) o_reg[i] += __uint_as_float(v[i]);
    };
    auto finalize = [&]() {
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        float l = l_part[i], le = le_part[i];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          l += __shfl_xor_sync(0xffffffffu, l, o);
          le += __shfl_xor_sync(0xffffffffu, le, o);
        }
        l_part[i] = l;
        le_part[i] = le;
      }
      // The four warps' partial sums of both normalisers, one after the other through
      // the same [4][N] slots (once per piece); the totals replace the partials.
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float* part = k ? le_part : l_part;
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < CW; ++i) clred[quarter * N + i] = part[i];
        }
        named_bar_sync(bar_id, 128);
#pragma unroll
        for (int i = 0; i < CW; ++i) part[i] = clred[i] + clred[N + i] + clred[2 * N + i] + clred[3 * N + i];
        named_bar_sync(bar_id, 128);  // the slots are rewritten next (or by the next piece)
      }
      const int64_t slot = (p_first == p_segbase) ? (int64_t)pb * a.Hkv + pg
                                                  : (int64_t)a.B * a.Hkv + blockIdx.x;
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        const int h = qbase + i;  // column: query token h / NREP, head h % NREP
        if (NCH > 1 && h >= NR) continue;
        const float l = l_part[i], le = le_part[i];
        const float ov = l > 0.f ? o_reg[i] / l : 0.f;
        const float lse2 = le > 0.f ? m_run[i] + log2f(le) : -INFINITY;
        if (p_whole) {
          const int64_t row = ((int64_t)pb * QL + h / NREP) * a.H + (int64_t)pg * NREP + h % NREP;
          if (a.out_f32)
            reinterpret_cast<float*>(a.out)[row * D + r] = ov;
          else
            reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + r] = __float2bfloat16_rn(ov);
          if (a.lse && r == 0) a.lse[row] = lse2 * kLn2;
        } else {
          a.ws_o[(slot * NR + h) * D + r] = ov;
          if (r == 0) a.ws_lse[slot * NR + h] = lse2;
        }
      }
    };

    bool resc = false;
    for (int j = 0; j < ntiles; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      if (first) {
        if (j > 0) {
          acc_o(j - 1);
          finalize();
        }
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          m_run[i] = kMinit;
          l_part[i] = 0.f;
          le_part[i] = 0.f;
          o_reg[i] = 0.f;
        }
        pb = c.b;
        pg = c.g;
        p_first = c.t;
        p_segbase = c.seg_base;
        p_whole = (c.t == c.seg_base) && (c.t + c.n <= t1);
      }
      // ---- scores of tile j (raw q . k; the scale is applied inside exp2)
      const int sb = j & 1;
      if (!mbar_wait(bar(B_SFULL + sb), (j >> 1) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      uint32_t sv[16];
      tmem_ld16(tmem + lane_off + s_col(sb) + qbase, sv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SEMPTY + sb));

      // Visible columns of this token: query tokens [qlo, qhi], i.e. columns
      // [qlo * NREP, (qhi + 1) * NREP) of the piece. dpos = position - (len - QL):
      // token i sees it iff dpos <= i, and with a window iff i <= dpos + W - 1.
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.jlo + c.j);
      const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int dpos = (c.jlo + c.j) * BS + r - (c.len - QL);
      const int qlo = dpos > 0 ? dpos : 0;
      int qhi = QL - 1;
      if (a.row_window > 0 && dpos + a.row_window - 1 < qhi) qhi = dpos + a.row_window - 1;
      const bool any = blk_ok && qlo <= qhi;
      const int ilo = any ? qlo * NREP - qbase : 0;
      const int ihi = any ? (qhi + 1) * NREP - qbase : 0;
      float x[CW];
      if (__all_sync(0xffffffffu, any && ilo <= 0 && ihi >= nreal)) {
        // Every real column of the block sees every token of the warp.
#pragma unroll
        for (int i = 0; i < CW; ++i) x[i] = __uint_as_float(sv[i]);
      } else {
#pragma unroll
        for (int i = 0; i < CW; ++i) x[i] = (i >= ilo && i < ihi) ? __uint_as_float(sv[i]) : -INFINITY;
      }
      const float cs = a.scale_log2;
      // The reference moves only when a column's block max beats it by more than
      // kLazy. One barrier with an OR reduction asks whether any thread of the block
      // sees such a score; the block max per column (warp reductions, an exchange
      // through shared memory and a second barrier) is taken only then.
      bool over = false;
#pragma unroll
      for (int i = 0; i < CW; ++i) over |= x[i] * cs > m_run[i] + kLazy;
      // One thread snapshots the abort flag before the barrier so that every
      // thread of the block takes the same decision after it.
      if (r == 0) snap[sb] = *abort_flag;
      const bool any_over = named_bar_any(bar_id, 128, over);
      if (snap[sb]) {
        aborted = true;
        break;
      }
      resc = false;
      if (any_over) {
        {
          float wm[CW];
#pragma unroll
          for (int i = 0; i < CW; ++i) wm[i] = warp_max(x[i]);
          float* dst = cred + (sb * 4 + quarter) * N;
          if (lane == 0) {
            if constexpr (CW % 4 == 0) {
#pragma unroll
              for (int i = 0; i < CW; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(wm[i], wm[i + 1], wm[i + 2], wm[i + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < CW; ++i) dst[i] = wm[i];
            }
          }
        }
        named_bar_sync(bar_id, 128);
        // Block max per column (raw units; scale > 0), then the reference test. Every
        // thread of the block reads the same maxima, so `resc` is uniform.
        float mb[CW];
        {
          const float* src = cred + sb * 4 * N;
          if constexpr (CW % 4 == 0) {
#pragma unroll
            for (int i = 0; i < CW; i += 4) {
              const float4 q0 = *reinterpret_cast<const float4*>(src + i);
              const float4 q1 = *reinterpret_cast<const float4*>(src + N + i);
              const float4 q2 = *reinterpret_cast<const float4*>(src + 2 * N + i);
              const float4 q3 = *reinterpret_cast<const float4*>(src + 3 * N + i);
              mb[i] = fmaxf(fmaxf(q0.x, q1.x), fmaxf(q2.x, q3.x));
              mb[i + 1] = fmaxf(fmaxf(q0.y, q1.y), fmaxf(q2.y, q3.y));
              mb[i + 2] = fmaxf(fmaxf(q0.z, q1.z), fmaxf(q2.z, q3.z));
              mb[i + 3] = fmaxf(fmaxf(q0.w, q1.w), fmaxf(q2.w, q3.w));
            }
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i)
              mb[i] = fmaxf(fmaxf(src[i], src[N + i]), fmaxf(src[2 * N + i], src[3 * N + i]));
          }
        }
#pragma unroll
        for (int i = 0; i < CW; ++i) resc |= mb[i] * cs > m_run[i] + kLazy;
        if (resc) {
          // Everything accumulated so far moves to the new reference now: O(j - 1),
          // which the value product may still be computing, is folded in first (rare;
          // otherwise it is folded after P(j) is published).
          float alpha[CW];
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            const float mn = fmaxf(m_run[i], mb[i] * cs);
            alpha[i] = exp2f(m_run[i] - mn);
            m_run[i] = mn;
          }
          if (!first) acc_o(j - 1);
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            o_reg[i] *= alpha[i];
            l_part[i] *= alpha[i];
            le_part[i] *= alpha[i];
          }
        }
      }
      // P enters the value product as bf16 (pairs of columns packed with one
      // round-to-nearest-even conversion); the output's normaliser sums the same
      // rounded weights, so the output is an exact convex combination of V rows, and
      // the log-sum-exp's sums the exact fp32 weights. A masked score is -inf and
      // gives weight exp2(-inf) = 0.
#pragma unroll
      for (int i = 0; i < CW; ++i) x[i] = exp2f(fmaf(x[i], cs, -m_run[i]));
      uint32_t pk[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float lo = 2 * jj < CW ? x[2 * jj < CW ? 2 * jj : 0] : 0.f;
        const float hi = 2 * jj + 1 < CW ? x[2 * jj + 1 < CW ? 2 * jj + 1 : 0] : 0.f;
        __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
        pk[jj] = *reinterpret_cast<uint32_t*>(&h2);
      }
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        l_part[i] += (i & 1) ? __uint_as_float(pk[i >> 1] & 0xffff0000u) : __uint_as_float(pk[i >> 1] << 16);
        le_part[i] += x[i];
      }
      // A position no query row sees may hold any bytes (an unwritten tail slot):
      // once the tile has landed, zero its V row so that its weight 0 cannot meet a
      // NaN in the value product (made visible to the MMA by the proxy fence before
      // PFULL). Positions some row sees hold written, finite rows.
      if (!any && chunk == 0) {
        const int st = j % NST;
        if (!mbar_wait(bar(B_VFULL + st), (j / NST) & 1)) fail();
        uint8_t* vrow = base + OFF_V + st * TILE + r * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + HALF + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // ---- P^T (bf16) into the B operand of the value product: token r's columns
      // qbase..qbase+7 and qbase+8..qbase+15 are one 16-byte row each of two core
      // matrices (8-token group r / 8, row r % 8).
      if (!mbar_wait(bar(B_PEMPTY + sb), ((j >> 1) & 1) ^ 1)) fail();
      uint8_t* ps = base + OFF_P + sb * PBUF + (r >> 3) * (N * 16) + (r & 7) * 16 + qbase * 16;
      *reinterpret_cast<uint4*>(ps) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(ps + 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      fence_proxy_async_smem();
      mbar_arrive(bar(B_PFULL + sb));
      // ---- fold the previous tile's O^T into the registers, with this tile's rescale
      if (!first && !resc) acc_o(j - 1);
      cursor_next(c, a.seq_lens, a.B, a.Hkv, BS, a.window, cap);
    }
    if (!aborted) {
      acc_o(ntiles - 1);
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

// bf16 tensor map with a 128-byte swizzle and 256-byte L2 promotion (decode_tc.cu).
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);

template <int NREP, int QL>
static cudaError_t launch_tc_n(const DecodeArgs& a, cudaStream_t stream) {
  using namespace tcd;
  using L = Shape<NREP, QL>;
  CUtensorMap tk, tv, tq;
  const uint64_t rows = (uint64_t)a.num_blocks * BS;
  const uint64_t kdims[3] = {D, (uint64_t)a.Hkv, rows};
  const uint64_t kstr[2] = {D * 2, (uint64_t)a.Hkv * D * 2};
  const uint32_t kbox[3] = {64, 1, BS};
  // q [B * QL, H, D]: one box is the n_rep heads of a kv head for the QL tokens.
  const uint64_t qdims[3] = {D, (uint64_t)a.H, (uint64_t)a.B * QL};
  const uint64_t qstr[2] = {D * 2, (uint64_t)a.H * D * 2};
  const uint32_t qbox[3] = {64, NREP, QL};
  if (!make_tmap_bf16(&tk, a.k_cache, 3, kdims, kstr, kbox) ||
      !make_tmap_bf16(&tv, a.v_cache, 3, kdims, kstr, kbox) ||
      !make_tmap_bf16(&tq, a.q, 3, qdims, qstr, qbox))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<NREP, QL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_tc_kernel<NREP, QL>, dim3(a.num_ctas), dim3(L::NTHREADS), L::SMEM_BYTES, stream,
                          a, tk, tv, tq);
}

}  // namespace pkv
