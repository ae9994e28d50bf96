// Causal paged prefill (and chunked prefill mixed with decode rows) on tcgen05.
//
// Query row r of sequence b, with q_b new rows after c_b = len_b - q_b cached
// positions, attends to keys j <= c_b + r: bottom-right causal alignment, the
// sparse_mode 3 semantics of the standalone guide ("手写40行" mask of "KV Cache 笔记":
// m = (arange(Skv) > arange(Sq)[:, None] + Skv - Sq) * -inf). GQA: query head h
// reads kv head h / n_rep. Queries are TND-packed; cu_seqlens_q holds cumulative
// ends, seq_lens_kv direct totals (standalone guide, actual_seq_lengths table).
//
// Unit of work: (sequence b, q tile, kv head g). A q tile is 128 / n_rep query
// tokens; its 128 rows are (token, head of the group) in TND memory order, so one
// 3-D TMA box {64 d, n_rep heads, 128/n_rep tokens} loads it and the group's K/V
// tile serves all of them. Per 128-key block of the unit's causal range:
//
//   S [128 x 128] = Q [128 x 128 d] . K_blk^T                  (tcgen05, fp32 in TMEM)
//   O_h [128 x 128] += P_h [128 x 64 keys] . V_blk[64h, 64h + 64)  (P bf16 in TMEM, V MN-major)
//
// S of block j and then its P share one of two tensor-memory buffers (P is written
// over the S columns already read), so the score product runs a block ahead of the
// softmax; two O accumulators hold the unit's output, one per key half.
// Softmax: eight warps, two per TMEM lane quarter. Warp half h owns keys
// [64h, 64h + 64) of every block of its 32 rows, with its own running max, normaliser
// and accumulator O_h, so the two warps of a row never wait for each other inside a
// unit; they combine (m_h, l_h, O_h) by the log-sum-exp rule when the unit ends. Each
// running max is raised only when a block exceeds it by more than 8 (log2 units), and
// O_h in TMEM is rescaled only then (warp-uniform). Each half's normaliser sums the
// weights as the value product uses them (bf16). Built with PKV_PF_SPLIT=0 the two
// warps share one max, normaliser and O (three S/P buffers), exchanging the row max
// through shared memory every block.
// Loads: warp 0 streams Q and K tiles (one Q buffer, K ring 3 deep, a tile freed as
// soon as its score product completes), warp 2 streams V tiles (3 deep). Warp 1
// issues the score products and warp 3 the value products, so neither waits behind
// the other.
// Work split: stream-K over all (unit, key block) tiles in kRounds rounds (see
// pf_vbound), one persistent CTA per SM with an equal share of every round; a unit
// cut by a range boundary leaves partial (o, lse) pieces that prefill_merge_kernel
// combines by LSE. Each range owns at most two such pieces: one that starts inside
// a unit ("head") and one that starts a unit it does not finish ("tail"). The kernel
// records where each range starts, so the merge needs no search.
//
// Roofline: tensor cores (dense contraction). Algorithmic flops per visible
// (query row, key) pair = 4 * 128 (q.k and p.v).
#include <cuda.h>

#include "device_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);

namespace pf {
constexpr int D = 128;
constexpr int BS = 128;
constexpr int M = 128;
#ifndef PKV_PF_NQ
#define PKV_PF_NQ 1
#endif
#ifndef PKV_PF_NK
#define PKV_PF_NK 3
#endif
// Shared memory holds 7 tiles of 32 KB. A unit's Q is needed only at its start, while
// K and V loads take ~3.9k cycles under this traffic (measured), so one Q buffer and
// a deeper K/V ring beat two Q buffers: the next unit's Q load waits for the last
// score product of the previous unit, once per ~40 blocks.
constexpr int NQ = PKV_PF_NQ;    // Q buffers
constexpr int NK = PKV_PF_NK;    // K ring: a K tile is released once its score product is done
constexpr int NV = 7 - NQ - NK;  // V ring: a V tile is released after its value product
#ifndef PKV_PF_SPLIT
#define PKV_PF_SPLIT 1
#endif
#ifndef PKV_PF_NPB
#if PKV_PF_SPLIT
#define PKV_PF_NPB 2
#else
#define PKV_PF_NPB 3
#endif
#endif
#ifndef PKV_PF_NOB
#define PKV_PF_NOB 1
#endif
#ifndef PKV_PF_ALIAS
#define PKV_PF_ALIAS 1
#endif
// PKV_PF_ALIAS 1: NPB buffers of 128 columns each hold S(j) and then, over the
// columns the softmax has read, P(j); S(j) waits only for O(j - NPB) to free its
// buffer, so the score product runs NPB - 1 blocks ahead of the softmax.
// PKV_PF_ALIAS 0: one S buffer (the next score product waits until the softmax has
// read S) and NPB P buffers of 64 columns. Either way NOB O buffers of 128 columns.
// Measured on the mixed prefill workload: unaliased, 3 P buffers and 1 O buffer
// 882.5 us against 904.4 with 2 and 2 and 926.6 with 4 and 1; aliased with 3 buffers
// 877.8 against 890.9 unaliased on one box.
constexpr bool kAlias = PKV_PF_ALIAS != 0;
// PKV_PF_SPLIT 1: the two softmax warps of a row keep separate running maxima,
// normalisers and O accumulators, one for keys [0, 64) and one for keys [64, 128) of
// every block, and combine them once per unit; no per-block exchange couples them.
// Tensor memory then holds two S/P buffers and the two O halves. Measured on the mixed
// prefill workload (per call, two boxes, each A/B on one box): 848 against 877 us and
// 874.7 against 877.4 us for the unsplit kernel with three S/P buffers.
constexpr bool kSplit = PKV_PF_SPLIT != 0;
constexpr int NPB = PKV_PF_NPB;
constexpr int NOB = PKV_PF_NOB;
static_assert(NPB >= 2 && NOB >= 1 &&
                  (kAlias ? NPB * 128 + (kSplit ? 2 : NOB) * 128 : 128 + NPB * 64 + NOB * 128) <= 512,
              "tensor memory");
static_assert(!kSplit || (kAlias && NOB == 1), "split halves need aliased S/P buffers and one O pair");
static_assert(NQ >= 1 && NQ <= 2 && NK >= 2 && NV >= 2,
              "prefill ring");
constexpr int NTHREADS = 384;    // warp 0 Q/K loads, 1 score MMAs, 2 V loads, 3 value MMAs, 4-11 softmax
constexpr int NSM = 256;         // softmax threads: two warps per TMEM lane quarter
constexpr int HALF = 16384;      // [128 rows x 128 bytes]
constexpr int TILE = 2 * HALF;   // K or V tile, or a Q tile
constexpr int OFF_Q = 0;                          // NQ Q buffers
constexpr int OFF_K = OFF_Q + NQ * TILE;          // NK K tiles
constexpr int OFF_V = OFF_K + NK * TILE;          // NV V tiles
constexpr int OFF_BAR = OFF_V + NV * TILE;        // 229376
enum {
  B_KFULL = 0,
  B_KEMPTY = B_KFULL + NK,
  B_VFULL = B_KEMPTY + NK,
  B_VEMPTY = B_VFULL + NV,
  B_QFULL = B_VEMPTY + NV,
  B_QEMPTY = B_QFULL + 2,
  B_SFULL = B_QEMPTY + 2,  // [NPB] aliased, else [0] only
  B_SEMPTY = B_SFULL + NPB,
  B_PFULL = B_SEMPTY + 2,  // [NPB] or, split, [NPB][2 halves]
  B_PEMPTY = B_PFULL + NPB * (kSplit ? 2 : 1),
  // One commit after each value product O(j) completes phase j / NPB of barrier
  // j % NPB: "P buffer free" and "O holds block j" are the same event, so one set of
  // barriers serves both.
  B_ODONE = B_PEMPTY,
  B_OFREE = B_PEMPTY + NPB,  // per O buffer
  B_XCH = B_OFREE + NOB,     // split: per lane quarter, the halves' end-of-unit exchange
  B_COUNT = B_XCH + (kSplit ? 4 : 0)
};
constexpr int OFF_XCH = OFF_BAR + B_COUNT * 8;      // float [2 halves][128 rows], the halves' exchange
constexpr int OFF_AFL = OFF_XCH + 2 * 128 * 4;      // int [2 halves][4 quarters] abort votes (unsplit)
constexpr int OFF_MISC = OFF_AFL + 2 * 4 * 4;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t TMEM_COLS = 512;
// Tensor memory (512 columns): S and P buffers as above (P holds 128 bf16 weights
// packed in pairs in 64 columns), then the O accumulators: with split halves the two
// O_h of 128 columns each, else NOB O buffers. A unit accumulates into the O
// buffer(s) after its predecessor's, which its first value product waits for until
// they are read out.
__device__ __forceinline__ uint32_t s_col(int b) { return kAlias ? b * 128 : 0; }
// P of buffer b; aliased, half h of a row writes its 32 columns at the start of the
// 64 S columns it read (the value product's K-steps 4h..4h+3 read them there).
__device__ __forceinline__ uint32_t p_col(int b, int h) { return kAlias ? b * 128 + h * 64 : 128 + b * 64 + h * 32; }
__device__ __forceinline__ uint32_t o_col(int ob) { return (kAlias ? NPB * 128 : 128 + NPB * 64) + ob * 128; }
// Split: O_h accumulates the value products of keys [64h, 64h + 64) of every block.
__device__ __forceinline__ uint32_t o_half(int h) { return NPB * 128 + h * 128; }
}  // namespace pf

struct PrefillArgs {
  const int32_t* cu_q;        // [B] cumulative query ends
  const int32_t* seq_lens;    // [B] total kv lengths
  const int32_t* block_table;
  void* out;                  // [T, H, D]
  float* lse;                 // [T, H] or null
  float* ws_o;                // [kRounds * G][2][128][128]
  float* ws_lse;              // [kRounds * G][2][128]
  long long* ws_bnd;          // [kRounds * G][8]: per virtual CTA, its range's first tile
                              // (-1: empty range), that tile's unit (first tile, blocks,
                              // b, g, q tile) and the total tile count
  int* dev_status;
  int64_t num_blocks;
  int B, H, Hkv, n_rep, qt_tokens, max_blocks, causal, out_f32, T;
  float scale_log2;
};

// Geometry of sequence b: query start / length, prior length, number of q tiles.
struct PfSeq {
  int q0, qlen, kvlen, c, nqt;
};

__device__ __forceinline__ PfSeq pf_seq(const PrefillArgs& a, int b) {
  PfSeq s;
  s.q0 = b > 0 ? __ldg(a.cu_q + b - 1) : 0;
  const int q1 = __ldg(a.cu_q + b);
  s.qlen = max(q1 - s.q0, 0);
  s.kvlen = clamp_len(__ldg(a.seq_lens + b), a.max_blocks * pf::BS);
  if (s.qlen > s.kvlen) s.qlen = s.kvlen;  // more queries than keys: only the last kvlen rows are meaningful
  s.c = s.kvlen - s.qlen;
  s.nqt = (s.qlen + a.qt_tokens - 1) / a.qt_tokens;
  return s;
}

// Key blocks a q tile needs: its causal range is keys [0, c + last token + 1).
__device__ __forceinline__ int pf_nkv(const PrefillArgs& a, const PfSeq& s, int qt) {
  const int tok_end = min((qt + 1) * a.qt_tokens, s.qlen);
  const int keys = a.causal ? s.c + tok_end : s.kvlen;
  return (keys + pf::BS - 1) / pf::BS;
}

// The (unit, key block) tile list is ordered b -> kv head g -> q tile -> block, so
// the units of one (b, g) are adjacent and stream the same K/V blocks.
//
// Rounds: the list is cut into kRounds equal chunks and chunk c is split across
// the G CTAs as in stream-K (CTA i takes [cb_c + i*W_c/G, cb_c + (i+1)*W_c/G)).
// CTA i walks round 0, then round 1, ...; since every CTA does an equal share of a
// round, all CTAs are inside the same chunk at any time, which keeps that chunk's
// K/V resident in L2. The range of round c on CTA i is "virtual CTA" k = c*G + i;
// pieces and merges work on virtual CTAs. Every range boundary adds a partial piece
// whose O the softmax warps read out. Measured on GB300 (16 sequences, 10.7k query
// rows, 0.33 GB of K/V, 4.7 GB of DRAM reads with one round): with one O buffer the
// next unit's value products waited for that readout and more rounds were slower
// (1 round 742 TFLOP/s, 8: 572); with two O buffers 2 rounds are fastest (1068 us
// for 1 round, 1021 for 2, 1096 for 4, 1234 for 8).
#ifndef PKV_PREFILL_ROUNDS
#define PKV_PREFILL_ROUNDS 2
#endif
constexpr int kRounds = PKV_PREFILL_ROUNDS;

__device__ __forceinline__ int64_t pf_chunk_base(int64_t c, int64_t W) { return (c * W) / kRounds; }

// Start of virtual CTA k's range (k in [0, kRounds*G]).
__device__ __forceinline__ int64_t pf_vbound(int64_t k, int64_t W, int64_t G) {
  const int64_t c = k / G, i = k % G;
  if (c >= kRounds) return W;
  const int64_t cb = pf_chunk_base(c, W), wc = pf_chunk_base(c + 1, W) - cb;
  return cb + (i * wc) / G;
}

// Virtual CTA whose range contains tile t (the last one starting at or before t).
__device__ __forceinline__ int64_t pf_vcta_of_tile(int64_t t, int64_t W, int64_t G) {
  int64_t c = ((t + 1) * kRounds + W - 1) / W - 1;  // chunk containing t
  const int64_t cb = pf_chunk_base(c, W), wc = pf_chunk_base(c + 1, W) - cb;
  return c * G + cta_of_tile(t - cb, wc, G);
}

// Cursor over one CTA's tiles: the concatenation of its kRounds ranges.
struct PfCursor {
  int b, g, qt, j, n;
  PfSeq s;
  int64_t seg_base;      // first tile of the current unit
  int64_t t, t_end;      // current tile, end of the current range
  int64_t W, G;
  int round, cta;
  bool range_start;      // t is the first tile of its range
};

__device__ inline int64_t pf_seq_work(const PrefillArgs& a, const PfSeq& s) {
  int64_t w = 0;
  for (int qt = 0; qt < s.nqt; ++qt) w += pf_nkv(a, s, qt);
  return w * a.Hkv;
}

// Position on tile t of the flat list (b, g, q tile, block).
__device__ inline void pf_locate(PfCursor& c, const PrefillArgs& a, int64_t t) {
  c.t = t;
  c.b = a.B;
  int64_t base = 0;
  for (int b = 0; b < a.B; ++b) {
    const PfSeq s = pf_seq(a, b);
    const int64_t w = pf_seq_work(a, s);
    if (t < base + w) {
      const int64_t wg = w / a.Hkv;  // work of one (b, g)
      const int64_t off = t - base;
      c.b = b;
      c.s = s;
      c.g = (int)(off / wg);
      int64_t o2 = off - (int64_t)c.g * wg;
      int64_t sb = base + (int64_t)c.g * wg;
      for (int qt = 0; qt < s.nqt; ++qt) {
        const int n = pf_nkv(a, s, qt);
        if (o2 < n) {
          c.qt = qt;
          c.n = n;
          c.j = (int)o2;
          c.seg_base = sb;
          return;
        }
        o2 -= n;
        sb += n;
      }
      return;
    }
    base += w;
  }
}

// Move to the first non-empty range at or after `round`; false if none is left.
__device__ inline bool pf_enter_round(PfCursor& c, const PrefillArgs& a, int round) {
  for (; round < kRounds; ++round) {
    const int64_t k = (int64_t)round * c.G + c.cta;
    const int64_t lo = pf_vbound(k, c.W, c.G), hi = pf_vbound(k + 1, c.W, c.G);
    if (lo < hi) {
      c.round = round;
      c.t_end = hi;
      c.range_start = true;
      pf_locate(c, a, lo);
      return true;
    }
  }
  c.round = kRounds;
  return false;
}

__device__ inline bool pf_begin(PfCursor& c, const PrefillArgs& a, int64_t W, int64_t G, int cta) {
  c.W = W;
  c.G = G;
  c.cta = cta;
  return pf_enter_round(c, a, 0);
}

// Total tiles of CTA `cta` over all rounds.
__device__ inline int pf_cta_tiles(int64_t W, int64_t G, int cta) {
  int64_t n = 0;
  for (int r = 0; r < kRounds; ++r) {
    const int64_t k = (int64_t)r * G + cta;
    n += pf_vbound(k + 1, W, G) - pf_vbound(k, W, G);
  }
  return (int)n;
}

__device__ inline bool pf_next(PfCursor& c, const PrefillArgs& a) {
  ++c.t;
  if (c.t >= c.t_end) return pf_enter_round(c, a, c.round + 1);
  c.range_start = false;
  if (++c.j < c.n) return true;
  c.j = 0;
  c.seg_base += c.n;
  for (;;) {
    if (++c.qt < c.s.nqt) {
      c.n = pf_nkv(a, c.s, c.qt);
      if (c.n > 0) return true;
      continue;
    }
    c.qt = -1;
    if (++c.g < a.Hkv) continue;
    c.g = 0;
    if (++c.b >= a.B) return false;
    c.s = pf_seq(a, c.b);
  }
}

__device__ inline int64_t pf_total_work(const PrefillArgs& a) {
  // One warp: lanes take sequences, then reduce.
  int64_t w = 0;
  for (int b = threadIdx.x & 31; b < a.B; b += 32) w += pf_seq_work(a, pf_seq(a, b));
#pragma unroll
  for (int o = 16; o; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
  return w;
}

__global__ void __launch_bounds__(pf::NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using namespace pf;
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

  if (tid == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_QFULL + i), 1);
      mbar_init(bar(B_QEMPTY + i), 1);
      mbar_init(bar(B_SEMPTY + i), NSM);
    }
    for (int i = 0; i < NPB; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PEMPTY + i), 1);
    }
    for (int i = 0; i < NPB * (kSplit ? 2 : 1); ++i) mbar_init(bar(B_PFULL + i), kSplit ? NSM / 2 : NSM);
    for (int i = 0; i < NOB; ++i) mbar_init(bar(B_OFREE + i), NSM);
    if (kSplit)
      for (int i = 0; i < 4; ++i) mbar_init(bar(B_XCH + i), 64);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    const int64_t w = pf_total_work(a);
    if (lane == 0) {
      *total_s = w;
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
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
  const int64_t W = *total_s, G = gridDim.x;
  const int ntiles = pf_cta_tiles(W, G, blockIdx.x);
  auto fail = [&]() {
    *abort_flag = 1;
    flag_status(a.dev_status, PKV_DEV_TIMEOUT);
  };

  if (warp == 2 && lane >= 1 && lane <= kRounds) {
    // Where each of this CTA's ranges starts, for the merge: lane r + 1 takes round r.
    const int64_t k = (int64_t)(lane - 1) * G + blockIdx.x;
    long long* e = a.ws_bnd + 8 * k;
    const int64_t lo = pf_vbound(k, W, G), hi = pf_vbound(k + 1, W, G);
    if (lo < hi) {
      PfCursor c;
      pf_locate(c, a, lo);
      e[1] = c.seg_base;
      e[2] = c.n;
      e[3] = c.b;
      e[4] = c.g;
      e[5] = c.qt;
      e[6] = W;
      e[0] = lo;
    } else {
      e[0] = -1;
    }
  }
  if (ntiles > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    PfCursor c;
    pf_begin(c, a, W, G, blockIdx.x);
    int piece = 0;
    const int rows_oob = (int)(a.num_blocks * BS);
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      if (j == 0 || c.j == 0 || c.range_start) {
        const int qb = piece % NQ;
        if (!mbar_wait(bar(B_QEMPTY + qb), ((piece / NQ) & 1) ^ 1)) { fail(); break; }
        mbar_expect_tx(bar(B_QFULL + qb), TILE);
        const int tok = c.s.q0 + c.qt * a.qt_tokens;
        const uint32_t qs = sbase + OFF_Q + qb * TILE;
        tma_load_3d(qs, &tm_q, bar(B_QFULL + qb), 0, c.g * a.n_rep, tok);
        tma_load_3d(qs + HALF, &tm_q, bar(B_QFULL + qb), 64, c.g * a.n_rep, tok);
        ++piece;
      }
      const int st = j % NK;
      if (!mbar_wait(bar(B_KEMPTY + st), ((j / NK) & 1) ^ 1)) { fail(); break; }
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.j);
      const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      if (!ok) flag_status(a.dev_status, PKV_DEV_BAD_BLOCK);
      const int row = ok ? blk * BS : rows_oob;
      const uint32_t ks = sbase + OFF_K + st * TILE;
      mbar_expect_tx(bar(B_KFULL + st), TILE);
      tma_load_3d(ks, &tm_k, bar(B_KFULL + st), 0, c.g, row);
      tma_load_3d(ks + HALF, &tm_k, bar(B_KFULL + st), 64, c.g, row);
      pf_next(c, a);
    }
  } else if (ntiles > 0 && warp == 2 && lane == 0) {
    // ------------------------------------------------------------ TMA producer (V)
    PfCursor c;
    pf_begin(c, a, W, G, blockIdx.x);
    const int rows_oob = (int)(a.num_blocks * BS);
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const int st = j % NV;
      if (!mbar_wait(bar(B_VEMPTY + st), ((j / NV) & 1) ^ 1)) { fail(); break; }
      const int blk = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.j);
      const bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int row = ok ? blk * BS : rows_oob;
      const uint32_t vs = sbase + OFF_V + st * TILE;
      mbar_expect_tx(bar(B_VFULL + st), TILE);
      tma_load_3d(vs, &tm_v, bar(B_VFULL + st), 0, c.g, row);
      tma_load_3d(vs + HALF, &tm_v, bar(B_VFULL + st), 64, c.g, row);
      pf_next(c, a);
    }
  } else if (ntiles > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ score-product issuer
    // Two issuing threads: this one issues S(j) as soon as K(j) has landed and the
    // softmax has read S(j-1); warp 3 issues the value products. A single thread
    // issuing both in a fixed order made O(j) wait behind S(j+1)'s waits and commits
    // and vice versa. Each thread's commits track only its own MMAs.
    constexpr uint32_t ID_S = idesc_bf16(M, 128, 0, 0);  // Q (K-major) x K^T (K-major)
    PfCursor c;
    pf_begin(c, a, W, G, blockIdx.x);
    int piece_s = -1;
    bool ok = true;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const bool first = (j == 0) || (c.j == 0) || c.range_start;
      const bool last = (j + 1 == ntiles) || (c.j + 1 == c.n) || (c.t + 1 == c.t_end);
      const int st = j % NK;
      if (first) ++piece_s;
      const int qb = piece_s % NQ;
      if (first && !mbar_wait(bar(B_QFULL + qb), (piece_s / NQ) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_KFULL + st), (j / NK) & 1)) { ok = false; break; }
      const int sbuf = kAlias ? j % NPB : 0;
      if (kAlias) {
        // S/P buffer j % NPB is free once O(j - NPB) has read P(j - NPB) from it.
        if (!mbar_wait(bar(B_ODONE + sbuf), ((j / NPB) & 1) ^ 1)) { ok = false; break; }
      } else if (!mbar_wait(bar(B_SEMPTY), (j & 1) ^ 1)) {  // softmax has read S(j-1)
        ok = false;
        break;
      }
      tc_fence_after();
      // Base descriptors once per tile; each K step only adds a constant offset.
      const uint64_t qd = smem_desc(sbase + OFF_Q + qb * TILE, 16, 1024, kSwizzle128);
      const uint64_t kd = smem_desc(sbase + OFF_K + st * TILE, 16, 1024, kSwizzle128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + s_col(sbuf), desc_add(qd, (kk >> 2) * HALF + (kk & 3) * 32),
               desc_add(kd, (kk >> 2) * HALF + (kk & 3) * 32), ID_S, kk > 0);
      mma_commit(bar(B_SFULL + sbuf));
      mma_commit(bar(B_KEMPTY + st));
      if (last) mma_commit(bar(B_QEMPTY + qb));
      pf_next(c, a);
    }
    if (!ok) fail();
  } else if (ntiles > 0 && warp == 3 && lane == 0) {
    // ------------------------------------------------------------ value-product issuer
    constexpr uint32_t ID_O = idesc_bf16(M, 128, 0, 1);  // P (TMEM) x V (MN-major)
    PfCursor c;
    pf_begin(c, a, W, G, blockIdx.x);
    int piece_o = -1;
    bool ok = true;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const bool first = (j == 0) || (c.j == 0) || c.range_start;
      const int st = j % NV, sb = j % NPB;
      if (!mbar_wait(bar(B_VFULL + st), (j / NV) & 1)) { ok = false; break; }
      const uint64_t vd = smem_desc(sbase + OFF_V + st * TILE, HALF, 1024, kSwizzle128);
      if (kSplit) {
        // O_h += P_h . V rows [64h, 64h + 64): each half's product issues as soon as
        // that half's weights are published.
        if (first) {
          ++piece_o;
          if (!mbar_wait(bar(B_OFREE), (piece_o & 1) ^ 1)) { ok = false; break; }
        }
        for (int h = 0; h < 2 && ok; ++h) {
          if (!mbar_wait(bar(B_PFULL + sb * 2 + h), (j / NPB) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + o_half(h), tmem + p_col(sb, h) + kk * 8, desc_add(vd, (4 * h + kk) * 2048), ID_O,
                   !(first && kk == 0));
        }
        if (!ok) break;
      } else {
        if (!mbar_wait(bar(B_PFULL + sb), (j / NPB) & 1)) { ok = false; break; }
        if (first) {
          ++piece_o;
          if (!mbar_wait(bar(B_OFREE + piece_o % NOB), ((piece_o / NOB) & 1) ^ 1)) { ok = false; break; }
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + o_col(piece_o % NOB), tmem + p_col(sb, kk >> 2) + (kk & 3) * 8, desc_add(vd, kk * 2048),
                 ID_O, !(first && kk == 0));
      }
      mma_commit(bar(B_PEMPTY + sb));
      mma_commit(bar(B_VEMPTY + st));
      pf_next(c, a);
    }
    if (!ok) fail();
  } else if (kSplit && ntiles > 0 && warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue (split)
    // Warp w handles rows quarter*32 + lane and keys [half*64, half*64 + 64) of every
    // block, with its own running max m_h, normaliser l_h and accumulator O_h, as if
    // the unit's keys were two sequences merged at the end. The two warps of a row
    // never wait for each other inside a unit, so their exp2 phases need not line up.
    // At the end of a unit they exchange (m_h, l_h) and each writes half of the
    // output columns: o = (2^(m_0 - M) O_0 + 2^(m_1 - M) O_1) / (2^(m_0 - M) l_0 +
    // 2^(m_1 - M) l_1), M = max(m_0, m_1).
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;  // row = token_local * n_rep + head
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float* xch = reinterpret_cast<float*>(base + OFF_XCH);  // [2 halves][128 rows]
    // Keys past the sequence's end: this thread clears key zkey's d-half zdh of the V
    // tile (the half's 128 threads cover its 64 keys).
    const int zkey = half * 64 + (r & 63), zdh = r >> 6;
    int xph = 0;  // phases completed on this quarter's exchange barrier
    // One value to the other half of the row and one back: write, meet, read, meet
    // again so that the next exchange cannot overwrite an unread value. Bounded waits,
    // their outcome made warp-uniform (tensor-memory loads follow).
    auto pair_xch = [&](float v, float& other) -> bool {
      xch[half * 128 + r] = v;
      mbar_arrive(bar(B_XCH + quarter));
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_XCH + quarter), xph & 1))) return false;
      ++xph;
      other = xch[(half ^ 1) * 128 + r];
      mbar_arrive(bar(B_XCH + quarter));
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_XCH + quarter), xph & 1))) return false;
      ++xph;
      return true;
    };
    const int tok_local = r / a.n_rep, hl = r % a.n_rep;
    PfCursor c;
    pf_begin(c, a, W, G, blockIdx.x);
    // l sums the weights as the value product uses them (rounded to bf16, added in
    // fp32), as in the unsplit path.
    float m_ref = -INFINITY, l = 0.f;
    bool aborted = false;
    int pqt = 0, pg = 0;
    int64_t p_vcta = 0;
    PfSeq ps{};
    bool p_start = false, p_whole = false;

    auto finalize = [&](int jl) -> bool {
      float m_o = -INFINITY, l_o = 0.f;
      if (!pair_xch(m_ref, m_o) || !pair_xch(l, l_o)) return false;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ODONE + jl % NPB), (jl / NPB) & 1))) return false;
      __syncwarp();
      tc_fence_after();
      const float mx = fmaxf(m_ref, m_o);
      const float a_own = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - mx);
      const float a_oth = (m_o == -INFINITY) ? 0.f : exp2f(m_o - mx);
      const float lt = l * a_own + l_o * a_oth;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float lse2 = lt > 0.f ? mx + log2f(lt) : -INFINITY;
      const float w0 = (half == 0 ? a_own : a_oth) * inv, w1 = (half == 0 ? a_oth : a_own) * inv;
      const int tok = pqt * a.qt_tokens + tok_local;  // query index inside the sequence
      const bool row_ok = tok < ps.qlen;
      const int64_t grow = (int64_t)(ps.q0 + tok) * a.H + (int64_t)pg * a.n_rep + hl;  // [T, H] row
      const int64_t slot = p_vcta * 2 + (p_start ? 1 : 0);
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 32) {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + o_half(0) + c0, v0);
        tmem_ld32(tmem + lane_off + o_half(1) + c0, v1);
        tmem_wait_ld();
        float f[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) f[k] = fmaf(__uint_as_float(v0[k]), w0, __uint_as_float(v1[k]) * w1);
        if (p_whole) {
          if (!row_ok) continue;
          if (a.out_f32) {
            float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + grow * D + c0);
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
          } else {
            uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + grow * D + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(f[8 * k + 2 * e], f[8 * k + 2 * e + 1]);
                w[e] = *reinterpret_cast<uint32_t*>(&h2);
              }
              o[k] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        } else {
          float4* o = reinterpret_cast<float4*>(a.ws_o + (slot * M + r) * D + c0);
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
        }
      }
      if (half == 0) {
        if (p_whole) {
          if (row_ok && a.lse) a.lse[grow] = lse2 * kLn2;
        } else {
          a.ws_lse[slot * M + r] = lse2;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE));
      return true;
    };

    // The block id of a tile is loaded one tile ahead, off the path from S to P.
    int blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.j);
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        aborted = true;
        break;
      }
      const bool first = (j == 0) || (c.j == 0) || c.range_start;
      const int blk = blk_next;
      if (first) {
        if (j > 0 && !finalize(j - 1)) {
          fail();
          aborted = true;
          break;
        }
        m_ref = -INFINITY;
        l = 0.f;
        pqt = c.qt;
        pg = c.g;
        ps = c.s;
        p_vcta = (int64_t)c.round * G + blockIdx.x;
        p_start = (c.t == c.seg_base);
        p_whole = p_start && (c.seg_base + c.n <= c.t_end);
      }
      const int sb = j % NPB;
      if (!mbar_wait(bar(B_SFULL + sb), (j / NPB) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      // Visible keys of this row in block c.j: key < kvlen and (causal) key <= c + tok.
      const int tok = c.qt * a.qt_tokens + tok_local;
      const int key_end = a.causal ? min(c.s.c + tok + 1, c.s.kvlen) : c.s.kvlen;
      const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      const int nvis = blk_ok ? max(0, min(64, key_end - c.j * BS - half * 64)) : 0;
      uint32_t sv[64];
      tmem_ld32(tmem + lane_off + s_col(sb) + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tmem + lane_off + s_col(sb) + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_wait_ld();
      tc_fence_before();
      if (!__all_sync(0xffffffffu, nvis >= 64)) {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= nvis) sv[k] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < 64; k += 2)
        m4[(k >> 1) & 3] = max3f(m4[(k >> 1) & 3], __uint_as_float(sv[k]), __uint_as_float(sv[k + 1]));
      // This half's max (raw scores; scale_log2 > 0 keeps the order).
      const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
      const bool need = mt > m_ref + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_ref;
        const float alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
        if (!first) {
          if (!mbar_wait(bar(B_ODONE + (j - 1) % NPB), ((j - 1) / NPB) & 1)) fail();
          __syncwarp();
          tc_fence_after();
          // O_h, all 128 columns of this thread's row, 16 at a time.
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_off + o_half(half) + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * (need ? alpha : 1.f));
            tmem_st16(tmem + lane_off + o_half(half) + c0, v);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m_ref = m_new;
        }
      }
      // Keys past the sequence's end in this block hold any bytes (unwritten tail
      // slots): zero this half's V rows once the tile has landed, so that a weight 0
      // cannot meet a NaN in the value product.
      if (c.j * BS + zkey >= c.s.kvlen) {
        const int vst = j % NV;
        if (!mbar_wait(bar(B_VFULL + vst), (j / NV) & 1)) fail();
        uint8_t* vrow = base + OFF_V + vst * TILE + zdh * HALF + zkey * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      tc_fence_after();
      // p = exp2(s * scale_log2 - m_h), pairs of scores per fma.f32x2, as above.
      const float mneg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const uint64_t cs2 = f2pack(a.scale_log2, a.scale_log2), mn2 = f2pack(mneg, mneg);
      float lr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 t = f2unpack(ffma2(f2pack(__uint_as_float(sv[c0 + k]), __uint_as_float(sv[c0 + k + 1])),
                                          cs2, mn2));
          const float p0 = exp2f(t.x), p1 = exp2f(t.y);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pk[k / 2] = *reinterpret_cast<uint32_t*>(&h2);
          add_bf16x2_to_f32(lr4[(k >> 1) & 1], lr4[2 + ((k >> 1) & 1)], pk[k / 2]);
        }
        tmem_st16(tmem + lane_off + p_col(sb, half) + c0 / 2, pk);
      }
      l += (lr4[0] + lr4[1]) + (lr4[2] + lr4[3]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + sb * 2 + half));
      pf_next(c, a);
      if (j + 1 < ntiles) blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.j);
    }
    if (!aborted && !finalize(ntiles - 1)) fail();
  } else if (ntiles > 0 && warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    // Two warps per TMEM lane quarter: warp w handles rows quarter*32 + lane and
    // score columns [half*64, half*64 + 64). The halves of a row exchange their row
    // max every block (and their normaliser at the end) through shared memory, with
    // a 64-thread named barrier per quarter.
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;  // row = token_local * n_rep + head
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int bar_id = 1 + quarter;
    float* xch = reinterpret_cast<float*>(base + OFF_XCH);  // [2 halves][128 rows]
    // Exchange one value with the other half of the row: write, sync the pair, read,
    // sync again so that the next exchange cannot overwrite an unread value.
    volatile int* afl = reinterpret_cast<volatile int*>(base + OFF_AFL);
    bool stop = false;  // set identically in both warps of the pair by exchange()
    auto exchange = [&](float v) -> float {
      // Each warp also votes whether to stop, so that the pair leaves the loop at
      // the same block and never waits alone at the pair barrier.
      const bool ab = __any_sync(0xffffffffu, *abort_flag != 0);
      if (lane == 0) afl[half * 4 + quarter] = ab ? 1 : 0;
      xch[half * 128 + r] = v;
      named_bar_sync(bar_id, 64);
      const float other = xch[(half ^ 1) * 128 + r];
      stop = (afl[quarter] | afl[4 + quarter]) != 0;
      named_bar_sync(bar_id, 64);
      return other;
    };
    const int tok_local = r / a.n_rep, hl = r % a.n_rep;
    PfCursor c;
    pf_begin(c, a, W, G, blockIdx.x);
    // l sums the weights as the value product uses them (rounded to bf16, added in
    // fp32): it divides the output, which is then an exact convex combination of V
    // rows, and gives the log-sum-exp, which then weighs a split piece exactly as its
    // output was normalised. With the lazy reference max a dominant key's weight is
    // 2^d (0 < d <= 8) rather than 1; with the fp32 weights summed instead, that
    // weight's rounding (up to 2^-8) would scale the whole output row. The reported
    // log-sum-exp is within ln(1 + 2^-8) of the exact one.
    float m_ref = -INFINITY, l = 0.f;
    bool aborted = false;
    int pqt = 0, pg = 0;
    int64_t p_vcta = 0;
    PfSeq ps{};
    bool p_start = false, p_whole = false;
    int pob = -1;  // O buffer of the piece being accumulated

    auto finalize = [&](int jl) {
      // Row normaliser: sum of both halves.
      const float lt = l + exchange(l);
      if (!mbar_wait(bar(B_ODONE + jl % NPB), (jl / NPB) & 1)) fail();
      __syncwarp();
      tc_fence_after();
      const int tok = pqt * a.qt_tokens + tok_local;  // query index inside the sequence
      const bool row_ok = tok < ps.qlen;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float lse2 = lt > 0.f ? m_ref + log2f(lt) : -INFINITY;
      const int64_t grow = (int64_t)(ps.q0 + tok) * a.H + (int64_t)pg * a.n_rep + hl;  // [T, H] row
      const int64_t slot = p_vcta * 2 + (p_start ? 1 : 0);
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + o_col(pob) + c0, v);
        tmem_wait_ld();
        if (p_whole) {
          if (!row_ok) continue;
          if (a.out_f32) {
            float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + grow * D + c0);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                 __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
          } else {
            uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + grow * D + c0);
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
          float4* o = reinterpret_cast<float4*>(a.ws_o + (slot * M + r) * D + c0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            o[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                               __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
        }
      }
      if (half == 0) {
        if (p_whole) {
          if (row_ok && a.lse) a.lse[grow] = lse2 * kLn2;
        } else {
          a.ws_lse[slot * M + r] = lse2;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE + pob));
    };

    // The block id of a tile is loaded one tile ahead, off the path from S to P.
    int blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.j);
    for (int j = 0; j < ntiles; ++j) {
      const bool first = (j == 0) || (c.j == 0) || c.range_start;
      const int blk = blk_next;
      if (first) {
        if (j > 0) finalize(j - 1);
        m_ref = -INFINITY;
        l = 0.f;
        pqt = c.qt;
        pg = c.g;
        ps = c.s;
        p_vcta = (int64_t)c.round * G + blockIdx.x;
        p_start = (c.t == c.seg_base);
        p_whole = p_start && (c.seg_base + c.n <= c.t_end);
        pob = (pob < 0) ? 0 : (pob + 1) % NOB;  // O buffer of this piece (in turn)
      }
      const int sb = j % NPB;  // P buffer
      if (kAlias ? !mbar_wait(bar(B_SFULL + sb), (j / NPB) & 1) : !mbar_wait(bar(B_SFULL), j & 1)) fail();
      __syncwarp();
      tc_fence_after();
      // Visible keys of this row in block c.j: key < kvlen and (causal) key <= c + tok.
      const int tok = c.qt * a.qt_tokens + tok_local;
      const int key_end = a.causal ? min(c.s.c + tok + 1, c.s.kvlen) : c.s.kvlen;
      const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      // Visible columns of this half.
      const int nvis = blk_ok ? max(0, min(64, key_end - c.j * BS - half * 64)) : 0;
      uint32_t sv[64];
      tmem_ld32(tmem + lane_off + s_col(sb) + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tmem + lane_off + s_col(sb) + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_wait_ld();
      tc_fence_before();
      if (!kAlias) mbar_arrive(bar(B_SEMPTY));
      if (!__all_sync(0xffffffffu, nvis >= 64)) {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= nvis) sv[k] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int k = 0; k < 64; k += 2)
        m4[(k >> 1) & 3] = max3f(m4[(k >> 1) & 3], __uint_as_float(sv[k]), __uint_as_float(sv[k + 1]));
      // Row max over both halves (raw scores; scale_log2 > 0 keeps the order).
      const float mown = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float mt = fmaxf(mown, exchange(mown)) * a.scale_log2;
      if (stop) {
        aborted = true;
        break;
      }
      const bool need = mt > m_ref + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_ref;
        const float alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
        if (!first) {
          if (!mbar_wait(bar(B_ODONE + (j - 1) % NPB), ((j - 1) / NPB) & 1)) fail();
          __syncwarp();
          tc_fence_after();
          // 16 columns at a time: the 64 scores of this block are live here.
#pragma unroll 1
          for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + lane_off + o_col(pob) + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * (need ? alpha : 1.f));
            tmem_st16(tmem + lane_off + o_col(pob) + c0, v);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m_ref = m_new;
        }
      }
      // Keys past the sequence's end in this block hold any bytes (unwritten tail
      // slots): zero their V rows (this thread: row r, d half `half`) once the tile
      // has landed, so that a weight 0 cannot meet a NaN in the value product.
      if (c.j * BS + r >= c.s.kvlen) {
        const int vst = j % NV;
        if (!mbar_wait(bar(B_VFULL + vst), (j / NV) & 1)) fail();
        uint8_t* vrow = base + OFF_V + vst * TILE + half * HALF + r * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      // Aliased, buffer sb is this tile's until P(j) is published.
      if (!kAlias && !mbar_wait(bar(B_PEMPTY + sb), ((j / NPB) & 1) ^ 1)) fail();
      __syncwarp();
      tc_fence_after();
      // p = exp2(s * scale_log2 - m_ref): one FMA and one exp2 per key. A row with no
      // visible key so far keeps m_ref = -inf; its p are all 0 (exp2(-inf)).
      // Scores are taken in pairs: one fma.f32x2 scales and shifts two of them; the
      // two rounded weights are added to the normaliser by mixed-precision adds.
      const float mneg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const uint64_t cs2 = f2pack(a.scale_log2, a.scale_log2), mn2 = f2pack(mneg, mneg);
      float lr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 t = f2unpack(ffma2(f2pack(__uint_as_float(sv[c0 + k]), __uint_as_float(sv[c0 + k + 1])),
                                          cs2, mn2));
          const float p0 = exp2f(t.x), p1 = exp2f(t.y);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pk[k / 2] = *reinterpret_cast<uint32_t*>(&h2);
          add_bf16x2_to_f32(lr4[(k >> 1) & 1], lr4[2 + ((k >> 1) & 1)], pk[k / 2]);
        }
        tmem_st16(tmem + lane_off + p_col(sb, half) + c0 / 2, pk);
      }
      {
        l += (lr4[0] + lr4[1]) + (lr4[2] + lr4[3]);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + sb));
      pf_next(c, a);
      if (j + 1 < ntiles) blk_next = __ldg(a.block_table + (int64_t)c.b * a.max_blocks + c.j);
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

// LSE merge of units cut by range boundaries. Block (k, y) looks at the boundary
// where virtual CTA k's range starts; if it falls inside a unit and k is the first
// non-empty virtual CTA after the one that started that unit (whose "tail" piece it
// is), it merges rows [32 y, 32 y + 32) of the unit: the tail piece plus the head
// piece of every later virtual CTA the unit reaches. The attention kernel records
// where each range starts, and the other ranges are found in closed form, so the
// merge does no search: one record, then one round of loads per row. Warp = 4 rows,
// lane = 4 output columns; all pieces' loads of a row are issued before any is used.
__global__ void __launch_bounds__(256) prefill_merge_kernel(PrefillArgs a, int G) {
  using namespace pf;
  constexpr int kRowsPerWarp = 4, kMaxPieces = 5;
  const int64_t k = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait_primary();  // the attention kernel wrote the range records and the pieces
  if (k == 0) return;
  const long long* e = a.ws_bnd + 8 * k;
  const int64_t start = e[0], seg_base = e[1];
  if (start < 0 || start == seg_base) return;  // empty range, or it starts a unit: nothing cut here
  const int64_t seg_end = seg_base + e[2], W = e[6];
  const int b = (int)e[3], g = (int)e[4], qt = (int)e[5];
  const PfSeq s = pf_seq(a, b);
  const int64_t i0 = pf_vcta_of_tile(seg_base, W, G);
  // The first non-empty virtual CTA after i0 owns the tile right after i0's range.
  if (pf_vcta_of_tile(pf_vbound(i0 + 1, W, G), W, G) != k) return;
  // Pieces: the tail slot of i0, then the head slot of each non-empty virtual CTA
  // whose range starts inside the unit.
  int64_t slot[kMaxPieces];
  int np = 0;
  slot[np++] = i0 * 2 + 1;
  for (int64_t nxt = pf_vbound(i0 + 1, W, G); nxt < seg_end;) {
    const int64_t v = pf_vcta_of_tile(nxt, W, G);
    if (np < kMaxPieces) slot[np] = v * 2;
    ++np;
    nxt = pf_vbound(v + 1, W, G);
  }
  const int row0 = blockIdx.y * 32 + warp * kRowsPerWarp;
  for (int q = 0; q < kRowsPerWarp; ++q) {
    const int rr = row0 + q;
    const int tok = qt * a.qt_tokens + rr / a.n_rep;
    if (tok >= s.qlen) continue;
    float mx = -INFINITY, wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (np <= kMaxPieces) {
      float l2[kMaxPieces];
      float4 x[kMaxPieces];
#pragma unroll
      for (int p = 0; p < kMaxPieces; ++p) {
        if (p < np) {
          l2[p] = a.ws_lse[slot[p] * M + rr];
          x[p] = reinterpret_cast<const float4*>(a.ws_o + (slot[p] * M + rr) * D)[lane];
        }
      }
#pragma unroll
      for (int p = 0; p < kMaxPieces; ++p)
        if (p < np) mx = fmaxf(mx, l2[p]);
#pragma unroll
      for (int p = 0; p < kMaxPieces; ++p) {
        if (p >= np) continue;
        const float w = (l2[p] == -INFINITY) ? 0.f : exp2f(l2[p] - mx);
        acc.x += w * x[p].x;
        acc.y += w * x[p].y;
        acc.z += w * x[p].z;
        acc.w += w * x[p].w;
        wsum += w;
      }
    } else {
      // More pieces than registers hold (ranges much shorter than a unit): walk them.
      for (int pass = 0; pass < 2; ++pass) {
        for (int64_t v = i0, nxt = pf_vbound(i0 + 1, W, G);;) {
          const int64_t sl = v * 2 + (v == i0 ? 1 : 0);
          const float lv = a.ws_lse[sl * M + rr];
          if (pass == 0) {
            mx = fmaxf(mx, lv);
          } else {
            const float w = (lv == -INFINITY) ? 0.f : exp2f(lv - mx);
            const float4 xv = reinterpret_cast<const float4*>(a.ws_o + (sl * M + rr) * D)[lane];
            acc.x += w * xv.x;
            acc.y += w * xv.y;
            acc.z += w * xv.z;
            acc.w += w * xv.w;
            wsum += w;
          }
          if (nxt >= seg_end) break;
          v = pf_vcta_of_tile(nxt, W, G);
          nxt = pf_vbound(v + 1, W, G);
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int64_t grow = (int64_t)(s.q0 + tok) * a.H + (int64_t)g * a.n_rep + rr % a.n_rep;
    const float4 v = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (a.out_f32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + grow * D)[lane] = v;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + grow * D)[lane] =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
    if (a.lse && lane == 0) a.lse[grow] = wsum > 0.f ? (mx + log2f(wsum)) * kLn2 : -INFINITY;
  }
}

// Rows of queries that see no key at all (q_len > 0 with kv_len = 0 cannot occur
// after the clamp; rows of a zero-length sequence have no queries) need no fill.

size_t prefill_workspace_bytes(int G) {
  const size_t slots = (size_t)kRounds * G * 2;
  const size_t o_bytes = slots * pf::M * pf::D * 4;
  const size_t l_bytes = (slots * pf::M * 4 + 255) / 256 * 256;
  const size_t b_bytes = ((size_t)kRounds * G * 8 * 8 + 255) / 256 * 256;
  return o_bytes + l_bytes + b_bytes;
}

cudaError_t launch_prefill(const void* q, const int32_t* cu_q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table, int max_blocks,
                           const int32_t* seq_lens, void* out, int out_f32, float* lse, int T,
                           int B, int H, int Hkv, int64_t num_blocks, float scale, int causal,
                           void* ws, int* dev_status, int num_sms, cudaStream_t stream) {
  using namespace pf;
  PrefillArgs a{};
  a.cu_q = cu_q;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.out = out;
  a.lse = lse;
  a.dev_status = dev_status;
  a.num_blocks = num_blocks;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.n_rep = H / Hkv;
  a.qt_tokens = M / a.n_rep;
  a.max_blocks = max_blocks;
  a.causal = causal;
  a.out_f32 = out_f32;
  a.T = T;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.ws_o = reinterpret_cast<float*>(ws);
  const size_t slots = (size_t)kRounds * num_sms * 2;
  a.ws_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + slots * M * D * 4);
  a.ws_bnd = reinterpret_cast<long long*>(reinterpret_cast<uint8_t*>(ws) + slots * M * D * 4 +
                                          (slots * M * 4 + 255) / 256 * 256);

  CUtensorMap tq, tk, tv;
  const uint64_t qdims[3] = {D, (uint64_t)H, (uint64_t)T};
  const uint64_t qstr[2] = {D * 2, (uint64_t)H * D * 2};
  const uint32_t qbox[3] = {64, (uint32_t)a.n_rep, (uint32_t)a.qt_tokens};
  const uint64_t rows = (uint64_t)num_blocks * BS;
  const uint64_t kdims[3] = {D, (uint64_t)Hkv, rows};
  const uint64_t kstr[2] = {D * 2, (uint64_t)Hkv * D * 2};
  const uint32_t kbox[3] = {64, 1, BS};
  if (!make_tmap_bf16(&tq, q, 3, qdims, qstr, qbox) || !make_tmap_bf16(&tk, k_cache, 3, kdims, kstr, kbox) ||
      !make_tmap_bf16(&tv, v_cache, 3, kdims, kstr, kbox))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  prefill_tc_kernel<<<num_sms, NTHREADS, SMEM_BYTES, stream>>>(a, tq, tk, tv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_dependent(prefill_merge_kernel, dim3(kRounds * num_sms, M / 32), dim3(256), 0, stream, a,
                          num_sms);
}

}  // namespace pkv
