// Absorbed MLA paged decode on the tcgen05 tensor cores, one CTA pair per tile range.
//
// One latent KV head serves all query heads. key = value = cache_nope (kv_lora_rank
// 512) and a separate 64-wide rope key adds to the scores ("KVCache 优化技能" 模式三;
// standalone guide 模式三 "key 和 value 传同一个 cache_nope"; "KV Cache 笔记" MLA):
//
//   s_j = scale * (q_nope . nope_j + q_rope . rope_j),   o = softmax(s) . nope
//
// The two CTAs of a cluster walk the same tiles of 64 tokens. CTA `half` owns the
// latent columns [256 half, 256 half + 256) and rope columns [32 half, 32 half + 32):
//
//   S_half [128 heads x 64] = Q[:, own columns] . tile[:, own columns]^T   (K = 288)
//   S = S_0 + S_1          (partial scores swapped through distributed shared memory)
//   O_half [128 x 256]    += P [128 x 64] . nope_tile[:, own latent columns]
//
// The score product is split along its reduction axis, so no product is computed
// twice, and each CTA streams only its 36 KB of a tile (four 64-column latent chunks
// in a 128-byte swizzle, its 32 rope columns in a 64-byte swizzle) through a 4-deep
// TMA ring; the pair reads every byte of the cache once.
//
// The partial score tile crosses to the peer as fp32 st.async stores that count their
// bytes on the peer's mbarrier (the receiver opens each phase with expect_tx, so the
// sender needs no fence). Both CTAs add the same two numbers, hold bit-identical S,
// take identical softmax decisions and write identical P. The exchange is double-
// buffered and software-pipelined: tile j+1's partial is sent while tile j's softmax
// runs.
//
// Warps (the default, SMW = 1): 0 TMA producer, 1 score-product issuer, 3 value-
// product issuer, 4..7 softmax, one per TMEM lane quarter, each thread with a head
// row's 64 score columns and 256 O columns (warp 2 is idle). With SMW = 2 (a build
// option): 2..9 softmax, two per lane quarter with 32 score columns and 128 O columns
// each, agreeing on the row max through shared memory, and 11 the value-product
// issuer. One warp per quarter measured faster (228.6 against 232.5 us on the mla
// workload): it needs no exchange between warps.
//
// Tensor memory (512 columns): S 0..63, P 64..127 (two buffers of 64 bf16 packed in
// pairs, the A operand of the value product), this CTA's 256 Q latent columns
// 128..255 (the A operand of 16 score K-steps), O half 256..511. The rope part of Q
// stays in shared memory (two K-steps from shared memory).
//
// Softmax: thread = head row; exp2 in fp32 with the scale folded into log2 units; P
// rounded to bf16. The output is divided by the sum of the rounded weights, and the
// log-sum-exp is taken from the sum of the exact fp32 weights. The reference max is
// raised only when a tile's max exceeds it by more than 8 (log2 units), so P stays
// below 2^8 and O in TMEM is rescaled only then.
//
// Work: one attention problem per (query row, sequence); q_len rows per sequence
// (1 for plain decode) are walked query-row major, see MlaArgs.
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
bool make_tmap_bf16_sw64(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box);

namespace mla {

constexpr int DC = 512;          // latent (nope) width
constexpr int DR = 64;           // rope width
constexpr int TT = 64;           // tokens per tile (MMA N of the score product)
constexpr int BS = 128;          // block size
constexpr int M = 128;           // query heads per MMA (rows)
constexpr int DH = 256;          // latent columns per CTA
constexpr int NLC = 4;           // 64-wide latent chunks per CTA
constexpr int DRH = DR / 2;      // rope columns per CTA
constexpr int QRB = M * DRH * 2; // this CTA's rope part of Q: 128 rows x 64 bytes
constexpr int KCH = TT * 128;    // one latent chunk of a tile: TT rows x 128 bytes
constexpr int KRB = TT * DRH * 2;  // this CTA's rope part of a tile: TT rows x 64 bytes
constexpr int STAGE = NLC * KCH + KRB;  // 4 latent chunks + 32 rope columns (36 KB)
constexpr int NST = 4;           // K stages
constexpr int XBUF = TT * M * 4; // one partial score tile, fp32 (32 KB)
#ifndef PKV_MLA_SMW
#define PKV_MLA_SMW 1
#endif
// Softmax warps per TMEM lane quarter: each takes TT / SMW score columns of a tile
// and DH / SMW columns of O for its head rows.
constexpr int SMW = PKV_MLA_SMW;
static_assert(SMW == 1 || SMW == 2, "softmax warps per lane quarter");
constexpr int NSMT = 128 * SMW;                 // softmax threads
constexpr int CW = TT / SMW;                   // score columns per softmax thread
constexpr int OW = DH / SMW;                   // O columns per softmax thread
constexpr int SM_W0 = SMW == 2 ? 2 : 4;        // first softmax warp (its warp % 4 is its lane quarter)
constexpr int O_WARP = SMW == 2 ? 11 : 3;      // value-product issuer
// SMW 2: TMA warp, S-issue warp, 8 softmax warps, idle, O-issue warp;
// SMW 1: TMA warp, S-issue warp, idle, O-issue warp, 4 softmax warps.
constexpr int NTHREADS = SMW == 2 ? 384 : 256;

constexpr int OFF_K = 0;
constexpr int OFF_QR = OFF_K + NST * STAGE;        // rope part of Q (64-byte swizzle)
constexpr int OFF_X = OFF_QR + QRB;                // two partial-score buffers
constexpr int OFF_BAR = OFF_X + 2 * XBUF;
enum {
  B_KFULL = 0,
  B_KEMPTY = B_KFULL + NST,
  B_QFULL = B_KEMPTY + NST,
  B_QEMPTY = B_QFULL + 1,
  B_QTFULL = B_QEMPTY + 1,
  B_SFULL = B_QTFULL + 1,
  B_SEMPTY = B_SFULL + 1,
  B_PFULL = B_SEMPTY + 1,
  B_PEMPTY = B_PFULL + 2,
  // One commit after each value product O(j) completes phase j/2 of barrier j%2:
  // "P buffer free" and "O holds block j" are the same event, so one barrier pair
  // serves both.
  B_ODONE = B_PEMPTY,
  B_OFREE = B_PEMPTY + 2,
  B_XFULL = B_OFREE + 1,   // peer's partial scores arrived (transaction bytes)
  B_COUNT = B_XFULL + 2
};
// Exchange between the two softmax warps of a lane quarter: float [2][256] sums, then
// float2 [2][256] (row max, abort flag).
constexpr int OFF_RED = OFF_BAR + B_COUNT * 8;
constexpr int OFF_MISC = OFF_RED + 2 * 256 * 4 + 2 * 256 * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(STAGE % 1024 == 0 && OFF_QR % 1024 == 0 && OFF_X % 1024 == 0, "alignment");
static_assert((NLC * KCH) % 512 == 0, "a 64-byte-swizzled box starts on a 512-byte boundary");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;
__device__ __forceinline__ uint32_t p_col(int b) { return TT + b * (TT / 2); }
constexpr uint32_t Q_COL = 2 * TT;
constexpr uint32_t O_COL = 256;
static_assert(Q_COL + NLC * 32 <= O_COL, "tensor memory");

}  // namespace mla

// Arguments of the MLA decode kernel and its merge.
// With q_len query rows per sequence, query row i of sequence b is its own attention
// problem over the first len_b - q_len + 1 + i positions. The kernels walk those
// problems in "row order" p = i * B + b (query rows major): the q_len rows of a
// sequence then fall G / q_len pair ranges apart (G a multiple of q_len), run at
// the same time, and read each latent tile within a few tiles of one another, so
// that the repeats are served by L2. Row p is stored at index b * q_len + i of the
// [B, q_len, H, ...] query, output and lse arrays.
struct MlaArgs {
  const uint16_t* q_nope;     // [B, q_len, H, 512] bf16
  const uint16_t* q_rope;     // [B, q_len, H, 64] bf16
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;            // [B, q_len, H, 512]
  float* lse;           // [B, q_len, H] or null
  float* ws_o;          // [(Bq + Gh) * 2 * 128 * 256]
  float* ws_lse;        // [(Bq + Gh) * 2 * 128]
  long long* ws_bnd;    // [Gh][4]: first row p of pair i's range (-1: empty range),
                        // that row's first tile, its tile count, total tiles
  int* dev_status;
  int64_t num_blocks;
  int B, H, max_blocks, out_f32;
  int q_len, Bq;        // query rows per sequence, Bq = B * q_len
  int g_half;           // CTA pairs (clusters)
  float scale_log2;
};

namespace mla {
__device__ __forceinline__ int seq_of(const MlaArgs& a, int p) { return a.q_len == 1 ? p : p % a.B; }
// Index of row p in the [B, q_len, ...] arrays.
__device__ __forceinline__ int64_t row_index(const MlaArgs& a, int p) {
  return a.q_len == 1 ? (int64_t)p : (int64_t)(p % a.B) * a.q_len + p / a.B;
}
// Positions row p attends to: len_b - (q_len - 1 - i), at least 0.
__device__ __forceinline__ int row_len(const MlaArgs& a, int p, int cap) {
  const int len = clamp_len(__ldg(a.seq_lens + seq_of(a, p)), cap);
  if (a.q_len == 1) return len;
  const int n = len - (a.q_len - 1 - p / a.B);
  return n > 0 ? n : 0;
}
// Tiles of TT positions over all rows (one warp, result in every lane).
__device__ __forceinline__ int64_t total_tiles(const MlaArgs& a, int cap) {
  int64_t s = 0;
  for (int b = threadIdx.x & 31; b < a.B; b += 32) {
    const int raw = __ldg(a.seq_lens + b);
    const int len = clamp_len(raw, cap);
    if (len != raw && blockIdx.x == 0) flag_status(a.dev_status, PKV_DEV_BAD_LENGTH);
    for (int i = 0; i < a.q_len; ++i) {
      const int n = len - (a.q_len - 1 - i);
      if (n > 0) s += (n + TT - 1) / TT;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}
// Cursor over a pair's tiles in row order (c.b holds the row p; one kv head, no
// window, so c.g and c.jlo stay 0).
__device__ inline void seek(TileCursor& c, const MlaArgs& a, int cap, int64_t t, int64_t t_end) {
  c.t = t;
  c.t_end = t_end;
  c.b = a.Bq;
  c.g = 0;
  c.j = 0;
  c.jlo = 0;
  c.n = 0;
  c.len = 0;
  c.seg_base = 0;
  if (t >= t_end) return;
  int64_t base = 0;
  for (int p = 0; p < a.Bq; ++p) {
    const int len = row_len(a, p, cap);
    const int n = (len + TT - 1) / TT;
    if (t < base + n) {
      c.b = p;
      c.j = (int)(t - base);
      c.n = n;
      c.len = len;
      c.seg_base = base;
      return;
    }
    base += n;
  }
}
__device__ inline bool next(TileCursor& c, const MlaArgs& a, int cap) {
  ++c.t;
  if (c.t >= c.t_end) return false;
  if (++c.j < c.n) return true;
  c.j = 0;
  c.seg_base += c.n;
  for (;;) {
    if (++c.b >= a.Bq) return false;
    c.len = row_len(a, c.b, cap);
    c.n = (c.len + TT - 1) / TT;
    if (c.n > 0) return true;
  }
}
}  // namespace mla

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::NTHREADS, 1)
    mla_tc_kernel(const __grid_constant__ MlaArgs a, const __grid_constant__ CUtensorMap tm_qn,
                  const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_cn,
                  const __grid_constant__ CUtensorMap tm_cr) {
  using namespace mla;
  using namespace tc;
  pdl_launch_dependents();  // the merge may launch now; it waits for this grid
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  long long* total_s = reinterpret_cast<long long*>(misc + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = (int)cluster_ctarank();
  const int ci = blockIdx.x >> 1;  // pair index
  const int cap = a.max_blocks * BS;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
    }
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_QTFULL), NSMT);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SEMPTY), NSMT);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_PFULL + i), NSMT);
      mbar_init(bar(B_PEMPTY + i), 1);
      mbar_init(bar(B_XFULL + i), 1);
    }
    mbar_init(bar(B_OFREE), NSMT);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // Tiles of TT tokens: the cursor runs with "block size" TT and one kv head.
    const int64_t tot = total_tiles(a, cap);
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
  // Both CTAs' barriers are initialised before either arrives on the other's.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int64_t T = *total_s, G = a.g_half;
  const int64_t t0 = cta_tile_start(ci, T, G), t1 = cta_tile_start(ci + 1, T, G);
  const int ntiles = (int)(t1 - t0);
  auto fail = [&]() {
    *abort_flag = 1;
    flag_status(a.dev_status, PKV_DEV_TIMEOUT);
  };
  if (ntiles == 0 && half == 0 && tid == 0) a.ws_bnd[4 * ci] = -1;

  if (ntiles > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    TileCursor c;
    seek(c, a, cap, t0, t1);
    if (half == 0) {
      long long* e = a.ws_bnd + 4 * ci;
      e[0] = c.b;
      e[1] = c.seg_base;
      e[2] = c.n;
      e[3] = T;
    }
    int piece = 0;
    const int rows_oob = (int)(a.num_blocks * BS);
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      if (j == 0 || c.j == 0) {
        if (!mbar_wait_sleepy(bar(B_QEMPTY), (piece & 1) ^ 1)) { fail(); break; }
        mbar_expect_tx(bar(B_QFULL), QRB);
        tma_load_2d(sbase + OFF_QR, &tm_qr, bar(B_QFULL), DRH * half, (int)row_index(a, c.b) * a.H);
        ++piece;
      }
      const int st = j % NST;
      const int tok0 = c.j * TT;  // first token of the tile within the sequence
      const int blk = __ldg(a.block_table + (int64_t)seq_of(a, c.b) * a.max_blocks + tok0 / BS);
      const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int row = ok ? blk * BS + (tok0 % BS) : rows_oob;
      if (!mbar_wait(bar(B_KEMPTY + st), ((j / NST) & 1) ^ 1)) { fail(); break; }
      if (!ok) flag_status(a.dev_status, PKV_DEV_BAD_BLOCK);
      const uint32_t ks = sbase + OFF_K + st * STAGE;
      mbar_expect_tx(bar(B_KFULL + st), STAGE);
      for (int ch = 0; ch < NLC; ++ch)
        tma_load_2d(ks + ch * KCH, &tm_cn, bar(B_KFULL + st), (NLC * half + ch) * 64, row);
      tma_load_2d(ks + NLC * KCH, &tm_cr, bar(B_KFULL + st), DRH * half, row);
      next(c, a, cap);
    }
  } else if (ntiles > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ score-product issuer
    // Two issuing threads: this one issues S(j) once its tile has landed and the
    // softmax has read S(j-1) (and, for a piece's first tile, once its Q is in place);
    // warp 11 issues the value products. Each thread's commits track only its own MMAs.
    constexpr uint32_t ID_S = idesc_bf16(M, TT, 0, 0);  // Q (K-major) x K_tile^T (K-major)
    TileCursor c;
    seek(c, a, cap, t0, t1);
    int piece_s = -1;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      const bool last = (j + 1 == ntiles) || (c.j + 1 == c.n);
      const int st = j % NST;
      if (first) {
        ++piece_s;
        if (!mbar_wait(bar(B_QFULL), piece_s & 1) || !mbar_wait(bar(B_QTFULL), piece_s & 1)) { fail(); break; }
      }
      if (!mbar_wait(bar(B_KFULL + st), (j / NST) & 1) || !mbar_wait(bar(B_SEMPTY), (j & 1) ^ 1)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint64_t kd = smem_desc(sbase + OFF_K + st * STAGE, 16, 1024, kSwizzle128);
      // Rope parts: rows of 64 bytes, 64-byte swizzle, 8-row groups 512 bytes apart.
      const uint64_t qd = smem_desc(sbase + OFF_QR, 16, 512, kSwizzle64);
      const uint64_t krd = smem_desc(sbase + OFF_K + st * STAGE + NLC * KCH, 16, 512, kSwizzle64);
      const uint32_t sd = tmem + S_COL, qt = tmem + Q_COL;
#pragma unroll
      for (int ch = 0; ch < NLC; ++ch) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(sd, qt + ch * 32 + kk * 8, desc_add(kd, ch * KCH + kk * 32), ID_S, (ch | kk) != 0);
      }
      // This CTA's 32 rope columns: two K-steps of 16 (32 bytes) within the 64-byte rows.
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) mma_ss(sd, desc_add(qd, kk * 32), desc_add(krd, kk * 32), ID_S, 1);
      mma_commit(bar(B_SFULL));
      if (last) mma_commit(bar(B_QEMPTY));
      next(c, a, cap);
    }
  } else if (ntiles > 0 && warp == O_WARP && lane == 0) {
    // ------------------------------------------------------------ value-product issuer
    // O(j) reads the latent chunks of stage j % NST; its commit also frees the stage
    // (S(j) completed before the softmax published P(j)).
    constexpr uint32_t ID_O = idesc_bf16(M, DH, 0, 1);  // P (TMEM) x nope half (MN-major)
    TileCursor c;
    seek(c, a, cap, t0, t1);
    int piece_o = -1;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      const int st = j % NST, pb = j & 1;
      if (!mbar_wait(bar(B_PFULL + pb), (j >> 1) & 1)) { fail(); break; }
      if (first) {
        ++piece_o;
        if (!mbar_wait(bar(B_OFREE), (piece_o & 1) ^ 1)) { fail(); break; }
      }
      tc_fence_after();
      const uint64_t vd = smem_desc(sbase + OFF_K + st * STAGE, KCH, 1024, kSwizzle128);
#pragma unroll
      for (int kk = 0; kk < TT / 16; ++kk)
        mma_ts(tmem + O_COL, tmem + p_col(pb) + kk * 8, desc_add(vd, kk * 2048), ID_O,
               !(first && kk == 0));
      mma_commit(bar(B_PEMPTY + pb));
      mma_commit(bar(B_KEMPTY + st));
      next(c, a, cap);
    }
  } else if (ntiles > 0 && warp >= SM_W0 && warp < SM_W0 + 4 * SMW) {
    // ------------------------------------------------------------ softmax / epilogue
    // Eight warps, two per TMEM lane quarter: warp w takes head row r of its quarter
    // and score columns [32 hc, 32 hc + 32) of each tile, O columns [128 hc, +128).
    const int quarter = warp & 3;
    const int hc = (warp - SM_W0) >> 2;  // column part of the row (0 when SMW == 1)
    const int r = quarter * 32 + lane;  // head row
    const int st_id = hc * 128 + r;     // 0 .. NSMT-1
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t peer = (uint32_t)(half ^ 1);
    // Partial-score buffers: [TT/4 token groups][128 heads][4 tokens] fp32, so a warp's
    // 16-byte accesses cover 512 contiguous bytes. This thread's groups are 8 hc + g.
    const uint32_t x_peer = mapa_shared(sbase + OFF_X + (uint32_t)((CW / 4) * hc * M + r) * 16, peer);
    const uint32_t xbar_peer = mapa_shared(bar(B_XFULL), peer);
    float* red = reinterpret_cast<float*>(base + OFF_RED);
    const int qbar = 1 + quarter;                            // named barrier of the two warps
    TileCursor c;
    seek(c, a, cap, t0, t1);
    // Normalisers over this warp's columns: l of the weights as the value product uses
    // them (bf16), which divides the output; le of the exact fp32 weights, which gives
    // the log-sum-exp (the reported lse and the weight of a split piece in the merge).
    float m_ref = -INFINITY, l = 0.f, le = 0.f;
    bool aborted = false;
    int piece_sm = 0;
    // This CTA's 256 latent columns of Q for head row r into tensor memory (the A
    // operand of the score product), once the previous piece's score products no
    // longer read them. Column half hc writes chunks 2 hc and 2 hc + 1.
    auto load_q_tmem = [&](int64_t qi) {
      if (!mbar_wait(bar(B_QEMPTY), (piece_sm & 1) ^ 1)) fail();
      __syncwarp();
      tc_fence_after();
      const bool have = r < a.H;
      const int64_t qrow = qi * a.H + r;
      for (int ch = (NLC / SMW) * hc; ch < (NLC / SMW) * (hc + 1); ++ch) {
        const uint4* src = reinterpret_cast<const uint4*>(a.q_nope + qrow * DC + half * DH + ch * 64);
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = have ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
          const uint4 w = have ? __ldg(src + 4 + k) : make_uint4(0, 0, 0, 0);
          lo[4 * k] = v.x; lo[4 * k + 1] = v.y; lo[4 * k + 2] = v.z; lo[4 * k + 3] = v.w;
          hi[4 * k] = w.x; hi[4 * k + 1] = w.y; hi[4 * k + 2] = w.z; hi[4 * k + 3] = w.w;
        }
        tmem_st16(tmem + lane_off + Q_COL + ch * 32, lo);
        tmem_st16(tmem + lane_off + Q_COL + ch * 32 + 16, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_QTFULL));
      ++piece_sm;
    };
    int pb = 0;
    int64_t p_first = t0, p_segbase = 0;
    bool p_whole = false;
    int red_par = 0;  // alternates per exchange through `red`

    // Sum of a per-row value over the two warps of the quarter.
    auto pair_sum = [&](float v) {
      if (SMW == 1) return v;
      float* slot = red + red_par * 256;
      slot[st_id] = v;
      named_bar_sync(qbar, 64);
      const float o = slot[(hc ^ 1) * 128 + r];
      red_par ^= 1;
      return v + o;
    };
    // Row max over the two warps, together with their views of the abort flag, so
    // that both warps of a quarter leave the loop at the same tile (they meet at a
    // named barrier in every exchange).
    auto pair_max_abort = [&](float v, bool& stop) {
      if (SMW == 1) {
        stop = __any_sync(0xffffffffu, *abort_flag != 0);
        return v;
      }
      float2* slot = reinterpret_cast<float2*>(red + 512) + red_par * 256;
      slot[st_id] = make_float2(v, *abort_flag ? 1.f : 0.f);
      named_bar_sync(qbar, 64);
      const float2 o = slot[(hc ^ 1) * 128 + r];
      red_par ^= 1;
      stop = __any_sync(0xffffffffu, slot[st_id].y != 0.f || o.y != 0.f);
      return fmaxf(v, o.x);
    };

    auto finalize = [&](int jl) {
      const float lt = pair_sum(l), lte = pair_sum(le);
      if (!mbar_wait(bar(B_ODONE + (jl & 1)), (jl >> 1) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float lse2 = lte > 0.f ? m_ref + log2f(lte) : -INFINITY;
      const bool store = r < a.H;
      const int64_t slot = (p_first == p_segbase) ? (int64_t)pb : (int64_t)a.Bq + ci;
      const int64_t orow = row_index(a, pb);
      for (int c0 = OW * hc; c0 < OW * hc + OW; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + O_COL + c0, v);
        tmem_wait_ld();
        if (!store) continue;
        if (p_whole) {
          const int64_t off = (orow * a.H + r) * DC + half * DH + c0;
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
      if (store && hc == 0) {
        if (p_whole) {
          if (a.lse && half == 0) a.lse[orow * a.H + r] = lse2 * kLn2;
        } else {
          a.ws_lse[(slot * 2 + half) * M + r] = lse2;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE));
    };

    // The exchange is software-pipelined: while tile j's softmax runs, this CTA's
    // partial scores of tile j+1 are already on their way to the peer. They travel as
    // st.async stores that count their bytes on the peer's XFULL barrier, whose phase
    // the peer opens (expect_tx) itself, so the sender needs no fence. Two buffers are
    // enough: tile j+1 is sent only after this thread has consumed the peer's tile j
    // (its values feed the max below), and the peer sends tile j+2 into the buffer of
    // tile j only once this CTA's tile j+1 has reached it.
    uint32_t sv[CW];  // this warp's CW partial scores of the tile in flight
    // Read S of tile jn from tensor memory and send it into the peer's buffer.
    auto fetch_send = [&](int jn) {
      if (!mbar_wait(bar(B_SFULL), jn & 1)) fail();
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < CW; c0 += 32)
        tmem_ld32(tmem + lane_off + S_COL + CW * hc + c0, *reinterpret_cast<uint32_t(*)[32]>(&sv[c0]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SEMPTY));
      const uint32_t xo = (uint32_t)(jn & 1) * XBUF, xbar = xbar_peer + 8u * (jn & 1);
#pragma unroll
      for (int g = 0; g < CW / 4; ++g)
        st_async_v4(x_peer + xo + g * (M * 16), sv[4 * g], sv[4 * g + 1], sv[4 * g + 2], sv[4 * g + 3], xbar);
    };
    auto lookup_block = [&](const TileCursor& cc) {
      return __ldg(a.block_table + (int64_t)seq_of(a, cc.b) * a.max_blocks + (cc.j * TT) / BS);
    };
    auto begin_piece = [&]() {
      m_ref = -INFINITY;
      l = 0.f;
      le = 0.f;
      pb = c.b;
      p_first = c.t;
      p_segbase = c.seg_base;
      p_whole = (c.t == c.seg_base) && (c.t + c.n <= t1);
    };
    const bool opener = (hc == 0 && quarter == 2 && lane == 0);  // opens each XFULL phase

    load_q_tmem(row_index(a, c.b));
    begin_piece();
    int blk = lookup_block(c);
    fetch_send(0);
    for (int j = 0; j < ntiles; ++j) {
      const bool first = (j == 0) || (c.j == 0);
      const bool more = j + 1 < ntiles;
      const bool next_first = more && (c.j + 1 == c.n);  // tile j+1 opens a new piece
      const int xb = j & 1;
      // Block id of tile j+1, loaded a whole tile before it is used.
      TileCursor cn = c;
      next(cn, a, cap);
      const int blk_next = more ? lookup_block(cn) : 0;
      // Peer's partial scores of tile j, added to this CTA's.
      if (opener) mbar_expect_tx(bar(B_XFULL + xb), XBUF);
      if (!mbar_wait_cluster(bar(B_XFULL + xb), (j >> 1) & 1)) fail();
      const float4* xin =
          reinterpret_cast<const float4*>(base + OFF_X + xb * XBUF + ((CW / 4) * hc * M + r) * 16);
      const int tok0 = c.j * TT + CW * hc;  // first token of this warp's columns
      const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int nvalid = blk_ok ? min(CW, c.len - tok0) : 0;  // may be <= 0
      const int nvalid_tile = blk_ok ? min(TT, c.len - c.j * TT) : 0;
      // Raw scores of this warp's CW columns (the two partial sums added in pairs);
      // masked columns become -inf. The max is taken on raw scores (scale > 0).
      uint64_t x2[CW / 2];
#pragma unroll
      for (int g = 0; g < CW / 4; ++g) {
        const float4 pv = xin[g * M];
        x2[2 * g] = fadd2(f2pack(__uint_as_float(sv[4 * g]), __uint_as_float(sv[4 * g + 1])), f2pack(pv.x, pv.y));
        x2[2 * g + 1] = fadd2(f2pack(__uint_as_float(sv[4 * g + 2]), __uint_as_float(sv[4 * g + 3])), f2pack(pv.z, pv.w));
      }
      if (!__all_sync(0xffffffffu, nvalid >= CW)) {
#pragma unroll
        for (int q = 0; q < CW / 2; ++q) {
          const float2 t = f2unpack(x2[q]);
          x2[q] = f2pack(2 * q < nvalid ? t.x : -INFINITY, 2 * q + 1 < nvalid ? t.y : -INFINITY);
        }
      }
      float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < CW / 2; ++q) {
        const float2 t = f2unpack(x2[q]);
        m2[q & 1] = max3f(m2[q & 1], t.x, t.y);
      }
      float mt = fmaxf(m2[0], m2[1]) * a.scale_log2;
      if (more && !next_first) fetch_send(j + 1);
      bool stop = false;
      mt = pair_max_abort(mt, stop);
      if (stop) {
        aborted = true;
        break;
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
          // 16 columns at a time: x and the next tile's scores are live here.
#pragma unroll 1
          for (int c0 = OW * hc; c0 < OW * hc + OW; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_off + O_COL + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * (need ? alpha : 1.f));
            tmem_st16(tmem + lane_off + O_COL + c0, v);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          le *= alpha;
          m_ref = m_new;
        }
      }
      // p = exp2(s * scale_log2 - m_ref): one fma.f32x2 per two scores; a masked
      // score (-inf) gives 0, and a row that has seen no visible key (m_ref = -inf)
      // keeps all weights 0. The normaliser sums the weights as the value product
      // sees them, rounded to bf16: with the lazy reference max a dominant key's
      // weight is 2^d (0 < d <= 8) rather than exactly 1, and its rounding error (up to
      // 2^-8) would otherwise scale the whole output row.
      const float mneg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const uint64_t cs2 = f2pack(a.scale_log2, a.scale_log2), mn2 = f2pack(mneg, mneg);
      uint32_t pk[CW / 2];
      uint64_t ps2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)}, pe2[2] = {ps2[0], ps2[1]};
#pragma unroll
      for (int q = 0; q < CW / 2; ++q) {
        const float2 t = f2unpack(ffma2(x2[q], cs2, mn2));
        const float p0 = exp2f(t.x), p1 = exp2f(t.y);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
        pk[q] = *reinterpret_cast<uint32_t*>(&h2);
        ps2[q & 1] = fadd2(ps2[q & 1], f2pack(__uint_as_float(pk[q] << 16), __uint_as_float(pk[q] & 0xffff0000u)));
        pe2[q & 1] = fadd2(pe2[q & 1], f2pack(p0, p1));
      }
      {
        const float2 s0 = f2unpack(ps2[0]), s1 = f2unpack(ps2[1]);
        l += (s0.x + s0.y) + (s1.x + s1.y);
        const float2 e0 = f2unpack(pe2[0]), e1 = f2unpack(pe2[1]);
        le += (e0.x + e0.y) + (e1.x + e1.y);
      }
      // Tokens past the sequence's end (the tile's tail) hold any bytes: the score
      // product is done with this tile (SFULL), so zero those rows of the latent
      // chunks this CTA's value product reads, so that a weight 0 cannot meet a NaN.
      if (nvalid_tile < TT) {
        uint8_t* kt = base + OFF_K + (j % NST) * STAGE;
#pragma unroll
        for (int k = 0; k < TT * 32 / NSMT; ++k) {
          const int pidx = st_id + NSMT * k;      // TT rows x 4 chunks x 8 pieces of 16 B
          const int row = pidx >> 5, ch = (pidx >> 3) & 3, q = pidx & 7;
          if (row >= nvalid_tile)
            *reinterpret_cast<uint4*>(kt + ch * KCH + row * 128 + q * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (!mbar_wait(bar(B_PEMPTY + xb), ((j >> 1) & 1) ^ 1)) fail();
      __syncwarp();
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < CW / 2; c0 += 16)
        tmem_st16(tmem + lane_off + p_col(xb) + (CW / 2) * hc + c0, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c0]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + xb));
      c = cn;
      blk = blk_next;
      if (more) {
        if (next_first) {
          // The score product of a new piece needs that piece's Q in tensor memory
          // (free once this piece's last score product is done): write it first, so
          // that S(j+1) runs while this piece's O is read out and stored.
          load_q_tmem(row_index(a, c.b));
          fetch_send(j + 1);
          finalize(j);
          begin_piece();
        }
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
  // Neither CTA leaves while the other may still write into its shared memory.
  cluster_sync();
}

// LSE merge of split MLA pieces: lse = log2 sum_i 2^lse_i, o = sum_i 2^(lse_i - lse) o_i.
// Only a row (one query row of one sequence) whose tiles straddle a boundary between
// two pairs' tile ranges was split. The attention kernel records, per pair, the row its
// range starts in; block (k, g) takes pair i = k + 1 and merges that row if pair i's
// range starts at the row's first cut. Warp = two (head, latent half) rows of row group g,
// lane = 8 consecutive latent columns; the loads of two pieces are issued before any
// is used. Block (k, g) also writes o = 0, lse = -inf into row group g of the empty
// rows p = k (mod gridDim.x).
__global__ void __launch_bounds__(256) mla_merge_kernel(MlaArgs a) {
  using namespace mla;
  constexpr int kRows = 2, kMaxPieces = 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = a.max_blocks * BS;
  const int64_t G = a.g_half;
  auto put = [&](int64_t orow, int h, int half, const float (&v)[8]) {
    const int64_t off = (orow * a.H + h) * DC + half * DH + lane * 8;
    if (a.out_f32) {
      float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off);
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  };
  const int row0 = (blockIdx.y * 8 + warp) * kRows;  // first (head, half) row of this warp
  pdl_wait_primary();
  for (int p = blockIdx.x; p < a.Bq; p += gridDim.x) {
    if (row_len(a, p, cap) > 0) continue;
    const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int64_t orow = row_index(a, p);
    for (int q = 0; q < kRows; ++q) {
      const int h = (row0 + q) >> 1, half = (row0 + q) & 1;
      if (h >= a.H) continue;
      put(orow, h, half, z);
      if (a.lse && half == 0 && lane == 0) a.lse[orow * a.H + h] = -INFINITY;
    }
  }
  const int64_t i = (int64_t)blockIdx.x + 1;  // pair whose range start may cut a row
  if (i >= G || row0 >= 2 * a.H) return;
  const long long* e = a.ws_bnd + 4 * i;
  const long long b = e[0];
  if (b < 0) return;
  const int64_t base = e[1], n = e[2], T = e[3];
  const int64_t t = cta_tile_start(i, T, G);
  const int64_t i0 = cta_of_tile(base, T, G), i1 = cta_of_tile(base + n - 1, T, G);
  // The row's first cut is at tile start(i0 + 1); pairs with empty ranges share
  // that start with the one non-empty pair that holds it, which merges.
  if (t == base || cta_tile_start(i0 + 1, T, G) != t) return;
  int64_t slots[kMaxPieces];
  float mx[kRows], wsum[kRows], acc[kRows][8];
#pragma unroll
  for (int q = 0; q < kRows; ++q) {
    mx[q] = -INFINITY;
    wsum[q] = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[q][c] = 0.f;
  }
  int64_t k = i0;
  bool first_pass = true;
  while (k <= i1) {
    // Next batch of up to kMaxPieces pieces (pairs with empty ranges hold none).
    int np = 0;
    for (; k <= i1 && np < kMaxPieces; ++k) {
      if (k > i0 && cta_tile_start(k + 1, T, G) == cta_tile_start(k, T, G)) continue;
      slots[np++] = (k == i0) ? (int64_t)b : (int64_t)a.Bq + k;
    }
    float l2[kMaxPieces][kRows];
    float4 x[kMaxPieces][kRows][2];
#pragma unroll
    for (int p = 0; p < kMaxPieces; ++p) {
#pragma unroll
      for (int q = 0; q < kRows; ++q) {
        const int hr = (row0 + q) >> 1, half = (row0 + q) & 1;
        const bool ok = p < np && hr < a.H;
        const int64_t r = ok ? (slots[p] * 2 + half) * M + hr : 0;
        l2[p][q] = ok ? a.ws_lse[r] : -INFINITY;
        const float4* src = reinterpret_cast<const float4*>(a.ws_o + r * DH + lane * 8);
        x[p][q][0] = ok ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        x[p][q][1] = ok ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // Online combination across batches (rescale what was accumulated so far).
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
      float m = mx[q];
#pragma unroll
      for (int p = 0; p < kMaxPieces; ++p) m = fmaxf(m, l2[p][q]);
      const float sc = (first_pass || mx[q] == -INFINITY) ? 0.f : exp2f(mx[q] - m);
      wsum[q] *= sc;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[q][c] *= sc;
      mx[q] = m;
#pragma unroll
      for (int p = 0; p < kMaxPieces; ++p) {
        const float w = (l2[p][q] == -INFINITY) ? 0.f : exp2f(l2[p][q] - m);
        wsum[q] += w;
        acc[q][0] += w * x[p][q][0].x; acc[q][1] += w * x[p][q][0].y;
        acc[q][2] += w * x[p][q][0].z; acc[q][3] += w * x[p][q][0].w;
        acc[q][4] += w * x[p][q][1].x; acc[q][5] += w * x[p][q][1].y;
        acc[q][6] += w * x[p][q][1].z; acc[q][7] += w * x[p][q][1].w;
      }
    }
    first_pass = false;
  }
#pragma unroll
  for (int q = 0; q < kRows; ++q) {
    const int h = (row0 + q) >> 1, half = (row0 + q) & 1;
    if (h >= a.H) continue;
    const float inv = wsum[q] > 0.f ? 1.f / wsum[q] : 0.f;
    float v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = acc[q][c] * inv;
    put(row_index(a, (int)b), h, half, v);
    if (a.lse && half == 0 && lane == 0)
      a.lse[row_index(a, (int)b) * a.H + h] = wsum[q] > 0.f ? (mx[q] + log2f(wsum[q])) * kLn2 : -INFINITY;
  }
}

size_t mla_workspace_bytes(int rows, int g_half) {
  const int64_t slots = (int64_t)rows + g_half;
  const size_t o_bytes = (size_t)(slots * 2 * mla::M * mla::DH * 4 + 255) / 256 * 256;
  const size_t l_bytes = (size_t)(slots * 2 * mla::M * 4 + 255) / 256 * 256;
  const size_t b_bytes = (size_t)(g_half * 4 * 8 + 255) / 256 * 256;
  return o_bytes + l_bytes + b_bytes;
}

// CTA pairs that can be resident at once on the current device (at most num_sms / 2):
// a pair needs two SMs of one GPC, and a pair that had to wait for a second wave
// would double the kernel's time.
static int mla_resident_pairs(int num_sms) {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(mla::NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = mla::SMEM_BYTES;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)mla_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = num_sms / 2;
  }
  n = n < num_sms / 2 ? n : num_sms / 2;
  cached[dev] = n;
  return n;
}

cudaError_t launch_mla_decode(const void* q_nope, const void* q_rope, const void* cache_nope,
                              const void* cache_rope, const int32_t* block_table, int max_blocks,
                              const int32_t* seq_lens, void* out, int out_f32, float* lse, int B,
                              int q_len, int H, int64_t num_blocks, float scale, void* ws,
                              int* dev_status, int num_sms, cudaStream_t stream) {
  using namespace mla;
  cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
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
  a.q_len = q_len;
  a.Bq = B * q_len;
  a.g_half = mla_resident_pairs(num_sms);
  // A multiple of q_len pairs keeps the rows of a sequence in step (see MlaArgs).
  if (a.g_half >= q_len) a.g_half -= a.g_half % q_len;
  a.scale_log2 = scale * 1.4426950408889634f;
  const int64_t slots = (int64_t)a.Bq + a.g_half;
  const size_t o_bytes = (size_t)(slots * 2 * M * DH * 4 + 255) / 256 * 256;
  a.ws_o = reinterpret_cast<float*>(ws);
  const size_t l_bytes = (size_t)(slots * 2 * M * 4 + 255) / 256 * 256;
  a.ws_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + o_bytes);
  a.ws_bnd = reinterpret_cast<long long*>(reinterpret_cast<uint8_t*>(ws) + o_bytes + l_bytes);

  CUtensorMap tqn, tqr, tcn, tcr;
  const uint64_t rows_q = (uint64_t)a.Bq * H, rows_c = (uint64_t)num_blocks * BS;
  const uint64_t dqn[2] = {DC, rows_q}, sqn[1] = {DC * 2};
  const uint64_t dqr[2] = {DR, rows_q}, sqr[1] = {DR * 2};
  const uint64_t dcn[2] = {DC, rows_c}, scn[1] = {DC * 2};
  const uint64_t dcr[2] = {DR, rows_c}, scr[1] = {DR * 2};
  const uint32_t qbox[2] = {64, M}, cbox[2] = {64, TT};
  const uint32_t qrbox[2] = {DRH, M}, crbox[2] = {DRH, TT};
  if (!make_tmap_bf16(&tqn, q_nope, 2, dqn, sqn, qbox) ||
      !make_tmap_bf16_sw64(&tqr, q_rope, 2, dqr, sqr, qrbox) ||
      !make_tmap_bf16(&tcn, cache_nope, 2, dcn, scn, cbox) ||
      !make_tmap_bf16_sw64(&tcr, cache_rope, 2, dcr, scr, crbox))
    return cudaErrorInvalidValue;
  mla_tc_kernel<<<2 * a.g_half, NTHREADS, SMEM_BYTES, stream>>>(a, tqn, tqr, tcn, tcr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.Bq > 0) return launch_dependent(mla_merge_kernel, dim3(a.g_half > 1 ? a.g_half - 1 : 1, 16), dim3(256), 0, stream, a);
  return cudaSuccess;
}

}  // namespace pkv
