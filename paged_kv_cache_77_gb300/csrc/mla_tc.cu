// Absorbed MLA paged decode on the tcgen05 tensor cores.
//
// One latent KV head serves all query heads. key = value = cache_nope (kv_lora_rank
// 512) and a separate 64-wide rope key adds to the scores ("KVCache 优化技能" 模式三;
// standalone guide 模式三 "key 和 value 传同一个 cache_nope"; "KV Cache 笔记" MLA):
//
//   s_j = scale * (q_nope . nope_j + q_rope . rope_j),   o = softmax(s) . nope
//
// Tiles are 64 tokens of one sequence, streamed by TMA through a 2-deep ring (72 KB
// a stage). Per tile, with the 128 query heads on the M = 128 side of the MMA:
//
//   S [128 heads x 64] = [Q_nope | Q_rope] [128 x 576] . [nope | rope]_tile^T
//   O_half [128 x 256] += P [128 x 64] . nope_tile[:, half]      (P read from TMEM)
//
// 64-token tiles halve the MMA issues per token of 32-token tiles (an N=64 MMA costs
// about what an N=32 one does) and the handoffs per token; shared memory and tensor
// memory are then full, so S has a single buffer (the next score product waits only
// until the softmax has read S into registers).
//
// O for all 512 latent columns (128 x 512 fp32) would fill the whole 512-column
// tensor memory, so the 512 columns are split across two CTAs ("halves"); each CTA
// computes the full S of its tiles (1.5x the minimum tensor work) and half of O.
// CTA i and CTA i + G/2 walk the same tile range, so the second read of a tile
// usually hits L2. To leave shared memory for the ring, the A operand Q is split:
// columns 0..319 stay in shared memory, columns 320..511 and the rope part are
// written by the softmax warps into tensor memory and read from there by the MMA.
//
// Softmax: thread = head row of S (all 64 scores of a tile in one thread, no
// shuffles); exp2 in fp32 with the scale folded into log2 units; P rounded to bf16
// and stored into TMEM as the A operand of the value product; the normaliser sums
// the rounded weights. The running max is only raised when a tile's max exceeds it
// by more than 8 (log2 units): P stays below 2^8 and O in TMEM is rescaled only then
// (warp-uniform), which is rare after the first tile.
//
// Roofline: HBM and tensor both matter. Algorithmic bytes per token = 1152 (nope +
// rope row); algorithmic flops per token = 128 * (2*576 + 2*512).
#include <cuda.h>

#include "device_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);

namespace mla {

constexpr int DC = 512;          // latent (nope) width
constexpr int DR = 64;           // rope width
constexpr int TT = 64;           // tokens per tile (MMA N of the score product)
constexpr int BS = 128;          // block size
constexpr int M = 128;           // query heads per MMA (rows)
constexpr int DH = 256;          // latent columns per CTA half
constexpr int NCH = 9;           // 64-wide chunks of [nope | rope]
constexpr int QSM = 5;           // Q chunks 0-4 (nope 0..319) live in shared memory,
                                 // chunks 5-8 (nope 320..511 and rope) in tensor memory
constexpr int QCH = M * 128;     // one Q chunk: 128 rows x 128 bytes
constexpr int KCH = TT * 128;    // one K chunk: TT rows x 128 bytes
constexpr int NST = 2;           // K stages (72 KB each)
constexpr int NSB = 1;           // S buffers in tensor memory
constexpr int NTHREADS = 192;

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QSM * QCH;           // 81920
constexpr int OFF_BAR = OFF_K + NST * NCH * KCH;   // 229376
enum {
  B_KFULL = 0,
  B_KEMPTY = B_KFULL + NST,
  B_QFULL = B_KEMPTY + NST,
  B_QEMPTY = B_QFULL + 1,
  B_QTFULL = B_QEMPTY + 1,
  B_SFULL = B_QTFULL + 1,
  B_SEMPTY = B_SFULL + NSB,
  B_PFULL = B_SEMPTY + NSB,
  B_PEMPTY = B_PFULL + 2,
  B_ODONE = B_PEMPTY + 2,
  B_OFREE = B_ODONE + 2,
  B_COUNT = B_OFREE + 1
};
constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// TMEM columns: S 0..63 (one buffer, TT fp32 columns), P 64..127 (two buffers of TT
// bf16 packed in pairs), Q chunks 5-8 128..255 (32 columns each), O half 256..511.
constexpr uint32_t TMEM_COLS = 512;
__device__ __forceinline__ uint32_t s_col(int b) { return b * TT; }
__device__ __forceinline__ uint32_t p_col(int b) { return NSB * TT + b * (TT / 2); }
constexpr uint32_t Q_COL = NSB * TT + TT;
constexpr uint32_t O_COL = 256;
static_assert(Q_COL + (NCH - QSM) * 32 <= O_COL, "tensor memory");

}  // namespace mla

// Arguments of the MLA decode kernel and its merge.
struct MlaArgs {
  const uint16_t* q_nope;     // [B, H, 512] bf16
  const uint16_t* q_rope;     // [B, H, 64] bf16
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;            // [B, H, 512]
  float* lse;           // [B, H] or null
  float* ws_o;          // [(B + Gh) * 2 * 128 * 256]
  float* ws_lse;        // [(B + Gh) * 2 * 128]
  int* dev_status;
  int64_t num_blocks;
  int B, H, max_blocks, out_f32;
  int g_half;           // CTAs per latent half
  float scale_log2;
};

__global__ void __launch_bounds__(mla::NTHREADS, 1)
    mla_tc_kernel(const __grid_constant__ MlaArgs a, const __grid_constant__ CUtensorMap tm_qn,
                  const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_cn,
                  const __grid_constant__ CUtensorMap tm_cr) {
  using namespace mla;
  using namespace tc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  long long* total_s = reinterpret_cast<long long*>(misc + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x / a.g_half;
  const int ci = blockIdx.x % a.g_half;
  const int cap = a.max_blocks * BS;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
    }
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_QTFULL), 128);
    for (int i = 0; i < NSB; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SEMPTY + i), 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_PFULL + i), 128);
      mbar_init(bar(B_PEMPTY + i), 1);
      mbar_init(bar(B_ODONE + i), 1);
    }
    mbar_init(bar(B_OFREE), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // Tiles of TT tokens: the cursor runs with "block size" TT and one kv head.
    const int64_t tot = total_live_blocks(a.seq_lens, a.B, TT, 0, cap, a.dev_status);
    if (lane == 0) {
      *total_s = tot;
      tma_prefetch_desc(&tm_qn);
      tma_prefetch_desc(&tm_qr);
      tma_prefetch_desc(&tm_cn);
      tma_prefetch_desc(&tm_cr);
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
  const int64_t T = *total_s, G = a.g_half;
  const int64_t t0 = cta_tile_start(ci, T, G), t1 = cta_tile_start(ci + 1, T, G);
  const int ntiles = (half < 2) ? (int)(t1 - t0) : 0;
  auto fail = [&]() {
    *abort_flag = 1;
    flag_status(a.dev_status, PKV_DEV_TIMEOUT);
  };

  if (ntiles > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, 1, TT, 0, cap, t0, t1);
    int piece = 0;
    const int rows_oob = (int)(a.num_blocks * BS);
    // L2 prefetch runs kPrefetch tiles ahead of the loads (second cursor `pc`): a
    // stage frees only when O(j-2) completes, and the load then finds its tile in L2.
    constexpr int kPrefetch = 2;
    TileCursor pc = c;
    auto prefetch_next = [&](int jp) {
      if (jp >= ntiles) return;
      const int ptok = pc.j * TT;
      const int pblk = __ldg(a.block_table + (int64_t)pc.b * a.max_blocks + ptok / BS);
      if (pblk >= 0 && (int64_t)pblk < a.num_blocks) {
        const int prow = pblk * BS + (ptok % BS);
        for (int ch = 0; ch < 8; ++ch) tma_prefetch_2d(&tm_cn, ch * 64, prow);
        tma_prefetch_2d(&tm_cr, 0, prow);
      }
      cursor_next(pc, a.seq_lens, a.B, 1, TT, 0, cap);
    };
    for (int jp = 0; jp < kPrefetch; ++jp) prefetch_next(jp);
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      prefetch_next(j + kPrefetch);
      if (j == 0 || c.j == 0) {
        if (!mbar_wait(bar(B_QEMPTY), (piece & 1) ^ 1)) { fail(); break; }
        mbar_expect_tx(bar(B_QFULL), QSM * QCH);
        const int qrow = c.b * a.H;
        for (int ch = 0; ch < QSM; ++ch)
          tma_load_2d(sbase + OFF_Q + ch * QCH, &tm_qn, bar(B_QFULL), ch * 64, qrow);
        ++piece;
      }
      const int st = j % NST;
      const int tok0 = c.j * TT;  // first token of the tile within the sequence
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + tok0 / BS);
      const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int row = ok ? blk * BS + (tok0 % BS) : rows_oob;
      if (!mbar_wait(bar(B_KEMPTY + st), ((j / NST) & 1) ^ 1)) { fail(); break; }
      if (!ok) flag_status(a.dev_status, PKV_DEV_BAD_BLOCK);
      const uint32_t ks = sbase + OFF_K + st * NCH * KCH;
      mbar_expect_tx(bar(B_KFULL + st), NCH * KCH);
      for (int ch = 0; ch < 8; ++ch) tma_load_2d(ks + ch * KCH, &tm_cn, bar(B_KFULL + st), ch * 64, row);
      tma_load_2d(ks + 8 * KCH, &tm_cr, bar(B_KFULL + st), 0, row);
      cursor_next(c, a.seq_lens, a.B, 1, TT, 0, cap);
    }
  } else if (ntiles > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t ID_S = idesc_bf16(M, TT, 0, 0);  // Q (K-major) x K_tile^T (K-major)
    constexpr uint32_t ID_O = idesc_bf16(M, DH, 0, 1);  // P (TMEM) x nope half (MN-major)
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, 1, TT, 0, cap, t0, t1);
    int piece_s = -1;
    // Dynamic issue order: the thread polls (non-blocking) and issues whichever
    // product is ready. With two K stages the load of tile j+2 can only start when
    // O(j) has completed, so O(j) must not wait behind a score product that is itself
    // waiting for its tile; a fixed order exposed the whole TMA latency every tile.
    // Phases cannot alias: S(js) needs the softmax to have read S(js-1), and its K
    // stage is refilled only after O(js-2), so js <= jo + 2 while O(jo) is pending.
    bool first_of[4] = {false, false, false, false};  // by tile index mod 4
    int piece_o = -1;
    auto ready_s = [&](int j) -> bool {
      const bool first = (j == 0) || (c.j == 0);
      const int st = j % NST, sb = j % NSB;
      if (first && (!mbar_try(bar(B_QFULL), (piece_s + 1) & 1) ||
                    !mbar_try(bar(B_QTFULL), (piece_s + 1) & 1)))
        return false;
      return mbar_try(bar(B_KFULL + st), (j / NST) & 1) &&
             mbar_try(bar(B_SEMPTY + sb), ((j / NSB) & 1) ^ 1);
    };
    auto issue_s = [&](int j) {
      const bool first = (j == 0) || (c.j == 0);
      const bool last = (j + 1 == ntiles) || (c.j + 1 == c.n);
      const int st = j % NST, sb = j % NSB;
      first_of[j & 3] = first;
      if (first) ++piece_s;
      tc_fence_after();
      // Base descriptors once per tile; each K step only adds a constant offset.
      const uint64_t kd = smem_desc(sbase + OFF_K + st * NCH * KCH, 16, 1024, kSwizzle128);
      const uint64_t qd = smem_desc(sbase + OFF_Q, 16, 1024, kSwizzle128);
      const uint32_t sd = tmem + s_col(sb), qt = tmem + Q_COL;
#pragma unroll
      for (int ch = 0; ch < QSM; ++ch) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(sd, desc_add(qd, ch * QCH + kk * 32), desc_add(kd, ch * KCH + kk * 32), ID_S,
                 (ch | kk) != 0);
      }
#pragma unroll
      for (int ch = QSM; ch < NCH; ++ch) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(sd, qt + (ch - QSM) * 32 + kk * 8, desc_add(kd, ch * KCH + kk * 32), ID_S, 1);
      }
      mma_commit(bar(B_SFULL + sb));
      if (last) mma_commit(bar(B_QEMPTY));
      cursor_next(c, a.seq_lens, a.B, 1, TT, 0, cap);
    };
    auto ready_o = [&](int j) -> bool {
      const int sb = j & 1;  // P buffer
      if (!mbar_try(bar(B_PFULL + sb), (j >> 1) & 1)) return false;
      return !first_of[j & 3] || mbar_try(bar(B_OFREE), ((piece_o + 1) & 1) ^ 1);
    };
    auto issue_o = [&](int j) {
      const int st = j % NST, sb = j & 1;
      const bool first = first_of[j & 3];
      if (first) ++piece_o;
      tc_fence_after();
      const uint64_t vd = smem_desc(sbase + OFF_K + st * NCH * KCH + (4 * half) * KCH, KCH, 1024,
                                    kSwizzle128);
#pragma unroll
      for (int kk = 0; kk < TT / 16; ++kk)
        mma_ts(tmem + O_COL, tmem + p_col(sb) + kk * 8, desc_add(vd, kk * 2048), ID_O,
               !(first && kk == 0));
      mma_commit(bar(B_ODONE + sb));
      mma_commit(bar(B_PEMPTY + sb));
      mma_commit(bar(B_KEMPTY + st));
    };
    int js = 0, jo = 0;
    long long idle_since = clock64();
    while (jo < ntiles) {
      bool done = false;
      if (jo < js && ready_o(jo)) {
        issue_o(jo++);
        done = true;
      } else if (js < ntiles && ready_s(js)) {
        issue_s(js++);
        done = true;
      }
      if (done) {
        idle_since = clock64();
      } else if (*abort_flag || clock64() - idle_since > kWaitCycles) {
        fail();
        break;
      }
    }
  } else if (ntiles > 0 && warp >= 2) {
    // ------------------------------------------------------------ softmax / epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // head row
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    TileCursor c;
    cursor_seek(c, a.seq_lens, a.B, 1, TT, 0, cap, t0, t1);
    float m_ref = -INFINITY, l = 0.f;
    bool aborted = false;
    int piece_sm = 0;
    // Q columns 256..511 and the rope part of head row r into tensor memory (the A
    // operand of chunks 4-8 of the score product), once the previous piece's score
    // products no longer read them.
    auto load_q_tmem = [&](int b) {
      if (!mbar_wait(bar(B_QEMPTY), (piece_sm & 1) ^ 1)) fail();
      __syncwarp();
      tc_fence_after();
      const bool have = r < a.H;
      const int64_t qrow = (int64_t)b * a.H + r;
      for (int ch = 0; ch < NCH - QSM; ++ch) {
        const int gch = QSM + ch;  // chunk of [nope | rope]: 0-7 nope, 8 rope
        const uint4* src = (gch < 8)
            ? reinterpret_cast<const uint4*>(a.q_nope + qrow * DC + gch * 64)
            : reinterpret_cast<const uint4*>(a.q_rope + qrow * DR);
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = have ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
          w[4 * k] = v.x;
          w[4 * k + 1] = v.y;
          w[4 * k + 2] = v.z;
          w[4 * k + 3] = v.w;
        }
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          lo[k] = w[k];
          hi[k] = w[16 + k];
        }
        tmem_st16(tmem + lane_off + Q_COL + ch * 32, lo);
        tmem_st16(tmem + lane_off + Q_COL + ch * 32 + 16, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_QTFULL));
      ++piece_sm;
    };
    int pb = 0, plast = 0;
    int64_t p_first = t0, p_segbase = 0;
    bool p_whole = false;

    auto finalize = [&](int jl) {
      if (!mbar_wait(bar(B_ODONE + (jl & 1)), (jl >> 1) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_ref + log2f(l) : -INFINITY;
      const bool store = r < a.H;
      const int64_t slot = (p_first == p_segbase) ? (int64_t)pb : (int64_t)a.B + ci;
      for (int c0 = 0; c0 < DH; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + O_COL + c0, v);
        tmem_wait_ld();
        if (!store) continue;
        if (p_whole) {
          const int64_t off = ((int64_t)pb * a.H + r) * DC + half * DH + c0;
          if (a.out_f32) {
            float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                 __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
          } else {
            uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[8 * k + 2 * e]) * inv,
                                                          __uint_as_float(v[8 * k + 2 * e + 1]) * inv);
                w[e] = *reinterpret_cast<uint32_t*>(&h2);
              }
              o[k] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        } else {
          float4* o = reinterpret_cast<float4*>(a.ws_o + ((slot * 2 + half) * M + r) * DH + c0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            o[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                               __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
        }
      }
      if (store) {
        if (p_whole) {
          if (a.lse && half == 0) a.lse[(int64_t)pb * a.H + r] = lse2 * kLn2;
        } else {
          a.ws_lse[(slot * 2 + half) * M + r] = lse2;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE));
      (void)plast;
    };

    for (int j = 0; j < ntiles; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      if (first) {
        if (j > 0) finalize(j - 1);
        load_q_tmem(c.b);
        m_ref = -INFINITY;
        l = 0.f;
        pb = c.b;
        p_first = c.t;
        p_segbase = c.seg_base;
        p_whole = (c.t == c.seg_base) && (c.t + c.n <= t1);
      }
      const int ssb = j % NSB, sb = j & 1;  // S buffer, P buffer
      if (!mbar_wait(bar(B_SFULL + ssb), (j / NSB) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      uint32_t sv[TT];
#pragma unroll
      for (int c0 = 0; c0 < TT; c0 += 32)
        tmem_ld32(tmem + lane_off + s_col(ssb) + c0, *reinterpret_cast<uint32_t(*)[32]>(&sv[c0]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SEMPTY + ssb));

      const int tok0 = c.j * TT;
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + tok0 / BS);
      const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int nvalid = blk_ok ? min(TT, c.len - tok0) : 0;
      float x[TT];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < TT; ++i) {
        x[i] = i < nvalid ? __uint_as_float(sv[i]) * a.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[i]);
      }
      // Raise the reference max only when this tile exceeds it by more than 8.
      const bool need = mt > m_ref + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_ref;
        const float alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
        if (!first) {
          // O must hold the previous tile's product before it is rescaled.
          if (!mbar_wait(bar(B_ODONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) fail();
          __syncwarp();
          tc_fence_after();
          for (int c0 = 0; c0 < DH; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + O_COL + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * (need ? alpha : 1.f));
            // 32 columns as two 16-column stores
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              lo[k] = v[k];
              hi[k] = v[16 + k];
            }
            tmem_st16(tmem + lane_off + O_COL + c0, lo);
            tmem_st16(tmem + lane_off + O_COL + c0 + 16, hi);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m_ref = m_new;
        }
      }
      uint32_t pk[TT / 2];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < TT; i += 2) {
        const float p0 = x[i] == -INFINITY ? 0.f : exp2f(x[i] - m_ref);
        const float p1 = x[i + 1] == -INFINITY ? 0.f : exp2f(x[i + 1] - m_ref);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
        const float2 back = __bfloat1622float2(h2);
        psum += back.x + back.y;
        pk[i / 2] = *reinterpret_cast<uint32_t*>(&h2);
      }
      l += psum;
      // Tokens past the sequence's end (the tile's tail) hold any bytes: the score
      // product is done with this tile (SFULL), so zero those rows of the nope chunks
      // this CTA's value product reads, so that a weight 0 cannot meet a NaN there.
      if (nvalid < TT) {
        uint8_t* kt = base + OFF_K + (j % NST) * NCH * KCH + (4 * half) * KCH;
#pragma unroll
        for (int k = 0; k < TT / 4; ++k) {
          const int pidx = r + 128 * k;           // TT rows x 4 chunks x 8 pieces of 16 B
          const int row = pidx >> 5, ch = (pidx >> 3) & 3, q = pidx & 7;
          if (row >= nvalid)
            *reinterpret_cast<uint4*>(kt + ch * KCH + row * 128 + q * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (!mbar_wait(bar(B_PEMPTY + sb), ((j >> 1) & 1) ^ 1)) fail();
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < TT / 2; c0 += 16)
        tmem_st16(tmem + lane_off + p_col(sb) + c0, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c0]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + sb));
      cursor_next(c, a.seq_lens, a.B, 1, TT, 0, cap);
      // Warp-uniform exit: the tcgen05 loads and stores above are warp-collective.
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        aborted = true;
        break;
      }
    }
    if (!aborted) finalize(ntiles - 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// LSE merge of split MLA pieces: lse = log2 sum_i 2^lse_i, o = sum_i 2^(lse_i - lse) o_i.
// Grid (sequence, latent half, head group of 8); warp = one query head, lane = 8
// consecutive latent columns of the half. Segments finished inside one attention
// CTA are skipped; empty sequences get o = 0, lse = -inf.
__global__ void __launch_bounds__(256) mla_merge_kernel(MlaArgs a) {
  using namespace mla;
  const int b = blockIdx.x, half = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.z * 8 + warp;
  if (h >= a.H) return;
  const int cap = a.max_blocks * BS;
  int64_t tot = 0, before = 0;
  for (int bb = lane; bb < a.B; bb += 32) {
    const int n = live_blocks(clamp_len(__ldg(a.seq_lens + bb), cap), TT, 0).n;
    tot += n;
    if (bb < b) before += n;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
  }
  const int64_t T = tot, G = a.g_half, base = before;
  const int n = live_blocks(clamp_len(__ldg(a.seq_lens + b), cap), TT, 0).n;
  const int64_t out_off = ((int64_t)b * a.H + h) * DC + half * DH + lane * 8;
  auto put = [&](const float (&v)[8]) {
    if (a.out_f32) {
      float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + out_off);
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + out_off) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  };
  if (n == 0) {
    const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    put(z);
    if (a.lse && half == 0 && lane == 0) a.lse[(int64_t)b * a.H + h] = -INFINITY;
    return;
  }
  const int64_t i0 = cta_of_tile(base, T, G), i1 = cta_of_tile(base + n - 1, T, G);
  if (i0 == i1) return;
  auto slot_of = [&](int64_t i) { return (i == i0) ? (int64_t)b : (int64_t)a.B + i; };
  float mx = -INFINITY;
  for (int64_t i = i0; i <= i1; ++i) {
    if (i > i0 && cta_tile_start(i + 1, T, G) == cta_tile_start(i, T, G)) continue;
    mx = fmaxf(mx, a.ws_lse[(slot_of(i) * 2 + half) * M + h]);
  }
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float wsum = 0.f;
  for (int64_t i = i0; i <= i1; ++i) {
    if (i > i0 && cta_tile_start(i + 1, T, G) == cta_tile_start(i, T, G)) continue;
    const int64_t slot = slot_of(i);
    const float l2 = a.ws_lse[(slot * 2 + half) * M + h];
    const float w = (l2 == -INFINITY) ? 0.f : exp2f(l2 - mx);
    const float4* src = reinterpret_cast<const float4*>(a.ws_o + ((slot * 2 + half) * M + h) * DH + lane * 8);
    const float4 x0 = src[0], x1 = src[1];
    acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
    acc[4] += w * x1.x; acc[5] += w * x1.y; acc[6] += w * x1.z; acc[7] += w * x1.w;
    wsum += w;
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] *= inv;
  put(acc);
  if (a.lse && half == 0 && lane == 0)
    a.lse[(int64_t)b * a.H + h] = wsum > 0.f ? (mx + log2f(wsum)) * kLn2 : -INFINITY;
}

size_t mla_workspace_bytes(int B, int g_half) {
  const int64_t slots = (int64_t)B + g_half;
  const size_t o_bytes = (size_t)(slots * 2 * mla::M * mla::DH * 4 + 255) / 256 * 256;
  const size_t l_bytes = (size_t)(slots * 2 * mla::M * 4 + 255) / 256 * 256;
  return o_bytes + l_bytes;
}

cudaError_t launch_mla_decode(const void* q_nope, const void* q_rope, const void* cache_nope,
                              const void* cache_rope, const int32_t* block_table, int max_blocks,
                              const int32_t* seq_lens, void* out, int out_f32, float* lse, int B,
                              int H, int64_t num_blocks, float scale, void* ws, int* dev_status,
                              int num_sms, cudaStream_t stream) {
  using namespace mla;
  MlaArgs a{};
  a.q_nope = (const uint16_t*)q_nope;
  a.q_rope = (const uint16_t*)q_rope;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse = lse;
  a.dev_status = dev_status;
  a.num_blocks = num_blocks;
  a.B = B;
  a.H = H;
  a.max_blocks = max_blocks;
  a.out_f32 = out_f32;
  a.g_half = num_sms / 2;
  a.scale_log2 = scale * 1.4426950408889634f;
  const int64_t slots = (int64_t)B + a.g_half;
  const size_t o_bytes = (size_t)(slots * 2 * M * DH * 4 + 255) / 256 * 256;
  a.ws_o = reinterpret_cast<float*>(ws);
  a.ws_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + o_bytes);

  CUtensorMap tqn, tqr, tcn, tcr;
  const uint64_t rows_q = (uint64_t)B * H, rows_c = (uint64_t)num_blocks * BS;
  const uint64_t dqn[2] = {DC, rows_q}, sqn[1] = {DC * 2};
  const uint64_t dqr[2] = {DR, rows_q}, sqr[1] = {DR * 2};
  const uint64_t dcn[2] = {DC, rows_c}, scn[1] = {DC * 2};
  const uint64_t dcr[2] = {DR, rows_c}, scr[1] = {DR * 2};
  const uint32_t qbox[2] = {64, M}, cbox[2] = {64, TT};
  if (!make_tmap_bf16(&tqn, q_nope, 2, dqn, sqn, qbox) || !make_tmap_bf16(&tqr, q_rope, 2, dqr, sqr, qbox) ||
      !make_tmap_bf16(&tcn, cache_nope, 2, dcn, scn, cbox) ||
      !make_tmap_bf16(&tcr, cache_rope, 2, dcr, scr, cbox))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  mla_tc_kernel<<<2 * a.g_half, NTHREADS, SMEM_BYTES, stream>>>(a, tqn, tqr, tcn, tcr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (B > 0) mla_merge_kernel<<<dim3(B, 2, (H + 7) / 8), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
