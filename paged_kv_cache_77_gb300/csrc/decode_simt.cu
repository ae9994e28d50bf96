// Split-KV flash-decoding on CUDA cores, and the LSE merge of split pieces.
//
// Each (b, h) output is softmax(scale * q . K^T) V over the visible positions of
// sequence b ("KV Cache 笔记", decode incremental form; GQA head h reads kv head
// h / n_rep, "MHA -> MQA -> GQA"). The keys are read block by block through
// block_table (skill note §3.1) and never gathered into a contiguous copy.
//
// Kernel shape: one CTA per SM walks its balanced share of (b, kv head, block)
// tiles (device_common.cuh). A tile is 128 tokens of one kv head: 32 KB of K and
// 32 KB of V, staged into shared memory by cp.async in a 3-deep ring with the
// 16-byte chunks XOR-swizzled by row so that both the row-wise (QK) and the
// column-wise (PV) reads are bank-conflict free. Scores are fp32 in log2 units
// (q pre-multiplied by scale * log2 e); the running max and sum follow the online
// softmax with the row max subtracted before exp ("三个工程细节"). The block max
// uses warp-shuffle reductions plus one shared-memory exchange across warps.
//
// Roofline: HBM. Algorithmic bytes per tile = 2 * 128 * 128 * 2 (K and V of one
// kv head); per call add q and out. This kernel is the CUDA-core path (used for
// MHA, and as the comparison point for the tensor-core GQA kernel).
#include "device_common.cuh"
#include "launch.h"

namespace pkv {

namespace simt {
constexpr int D = 128;
constexpr int BS = 128;
constexpr int THREADS = 128;
constexpr int STAGES = 3;
constexpr int ROW_BYTES = D * 2;                 // 256 bytes per token row
constexpr int TILE_BYTES = BS * ROW_BYTES;       // 32 KB for K (or V)
constexpr int STAGE_BYTES = 2 * TILE_BYTES;      // K + V

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * ROW_BYTES + ((chunk ^ (row & 7)) << 4));
}
}  // namespace simt

template <int NREP>
struct SimtSmem {
  alignas(128) uint8_t stage[simt::STAGES][simt::STAGE_BYTES];
  float q[NREP][simt::D];
  float p[simt::BS][NREP];
  float red[4][NREP];
  float lred[4][NREP];
  long long total;
};

template <int NREP>
__global__ void __launch_bounds__(simt::THREADS, 1) decode_simt_kernel(DecodeArgs a) {
  pdl_launch_dependents();  // the merge may launch now; it waits for this grid
  pdl_wait_primary();      // inputs may come from the kernel before (the cache write)
  using namespace simt;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<SimtSmem<NREP>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bs = BS;
  const int cap = a.max_blocks * BS;

  if (warp == 0) {
    int64_t tot = total_live_blocks(a.seq_lens, a.B, bs, a.window, cap, a.dev_status);
    if (lane == 0) S.total = tot * a.Hkv;
  }
  __syncthreads();
  const int64_t T = S.total, G = gridDim.x;
  const int64_t t0 = cta_tile_start(blockIdx.x, T, G), t1 = cta_tile_start(blockIdx.x + 1, T, G);
  if (t0 >= t1) return;

  TileCursor cur, pre;
  cursor_seek(cur, a.seq_lens, a.B, a.Hkv, bs, a.window, cap, t0, t1);
  pre = cur;
  bool pre_valid = true;

  const int64_t kv_row_elems = (int64_t)a.Hkv * D;  // elements between consecutive tokens

  // Issue the cp.async copies of the tile under `pre` into ring slot `slot`.
  auto issue = [&](int slot) {
    if (pre_valid) {
      int blk = __ldg(a.block_table + (int64_t)pre.b * a.max_blocks + pre.jlo + pre.j);
      bool ok = blk >= 0 && (int64_t)blk < a.num_blocks;
      if (!ok && tid == 0) flag_status(a.dev_status, PKV_DEV_BAD_BLOCK);
      const int64_t elem0 = ((int64_t)(ok ? blk : 0) * bs * a.Hkv + pre.g) * D;
      const uint8_t* kb = a.k_cache + elem0 * 2;
      const uint8_t* vb = a.v_cache + elem0 * 2;
      const uint32_t sk = smem_u32(S.stage[slot]);
      const uint32_t sv = sk + TILE_BYTES;
#pragma unroll 4
      for (int k = 0; k < (BS * 16) / THREADS; ++k) {
        const int idx = tid + k * THREADS;
        const int row = idx >> 4, chunk = idx & 15;
        const int64_t goff = (int64_t)row * kv_row_elems * 2 + chunk * 16;
        cp_async_16(sk + swz(row, chunk), kb + goff, ok ? 16u : 0u);
        cp_async_16(sv + swz(row, chunk), vb + goff, ok ? 16u : 0u);
      }
      pre_valid = cursor_next(pre, a.seq_lens, a.B, a.Hkv, bs, a.window, cap);
    }
    cp_async_commit();
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) issue(s);

  float m_run[NREP], l_part[NREP], o_acc[NREP];
  int64_t piece_first = t0;
  int it = 0;
  for (;;) {
    const bool piece_start = (cur.t == t0) || (cur.j == 0);
    if (piece_start) {
      piece_first = cur.t;
      // q of the NREP heads of this group, pre-scaled to log2 units.
      const uint16_t* qg = a.q + ((int64_t)cur.b * a.H + (int64_t)cur.g * NREP) * D;
      for (int e = tid; e < NREP * D; e += THREADS)
        S.q[e / D][e % D] = __uint_as_float((uint32_t)qg[e] << 16) * a.scale_log2;
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
        o_acc[h] = 0.f;
      }
    }
    issue((it + STAGES - 1) % STAGES);
    cp_async_wait<STAGES - 1>();
    __syncthreads();

    const uint8_t* kt = S.stage[it % STAGES];
    const uint8_t* vt = kt + TILE_BYTES;
    const int blk = __ldg(a.block_table + (int64_t)cur.b * a.max_blocks + cur.jlo + cur.j);
    const bool blk_ok = blk >= 0 && (int64_t)blk < a.num_blocks;
    const int lo = (a.window > 0 && cur.len > a.window) ? cur.len - a.window : 0;

    // ---- scores: thread = token ----
    const int pos = (cur.jlo + cur.j) * bs + tid;
    const bool valid = blk_ok && pos < cur.len && pos >= lo;
    float s[NREP];
#pragma unroll
    for (int h = 0; h < NREP; ++h) s[h] = 0.f;
#pragma unroll 2
    for (int c = 0; c < 16; ++c) {
      const uint4 w = *reinterpret_cast<const uint4*>(kt + swz(tid, c));
      const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                           bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        const float4 qa = *reinterpret_cast<const float4*>(&S.q[h][c * 8]);
        const float4 qb = *reinterpret_cast<const float4*>(&S.q[h][c * 8 + 4]);
        s[h] += qa.x * kf[0] + qa.y * kf[1] + qa.z * kf[2] + qa.w * kf[3] + qb.x * kf[4] +
                qb.y * kf[5] + qb.z * kf[6] + qb.w * kf[7];
      }
    }
    // A masked position's V row may hold any bytes (an unwritten tail slot): zero it,
    // so that its weight 0 cannot meet a NaN in the value loop below.
    if (!valid) {
      uint8_t* vrow = const_cast<uint8_t*>(vt);
#pragma unroll
      for (int c = 0; c < 16; ++c) *reinterpret_cast<uint4*>(vrow + swz(tid, c)) = make_uint4(0, 0, 0, 0);
    }
    float mx[NREP];
#pragma unroll
    for (int h = 0; h < NREP; ++h) {
      s[h] = valid ? s[h] : -INFINITY;
      float m = s[h];
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      mx[h] = m;
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < NREP; ++h) S.red[warp][h] = mx[h];
    }
    __syncthreads();
    float alpha[NREP];
#pragma unroll
    for (int h = 0; h < NREP; ++h) {
      const float mb = fmaxf(fmaxf(S.red[0][h], S.red[1][h]), fmaxf(S.red[2][h], S.red[3][h]));
      const float mn = fmaxf(m_run[h], mb);
      alpha[h] = (mn == -INFINITY) ? 1.f : exp2f(m_run[h] - mn);
      const float p = (s[h] == -INFINITY) ? 0.f : exp2f(s[h] - mn);
      S.p[tid][h] = p;
      l_part[h] = l_part[h] * alpha[h] + p;
      m_run[h] = mn;
    }
    __syncthreads();

    // ---- values: thread = output element d ----
    float acc[NREP];
#pragma unroll
    for (int h = 0; h < NREP; ++h) acc[h] = 0.f;
    const int dchunk = tid >> 3, dsub = (tid & 7) * 2;
#pragma unroll 4
    for (int tok = 0; tok < BS; ++tok) {
      const uint16_t vb = *reinterpret_cast<const uint16_t*>(vt + swz(tok, dchunk) + dsub);
      const float vf = __uint_as_float((uint32_t)vb << 16);
#pragma unroll
      for (int h = 0; h < NREP; ++h) acc[h] += S.p[tok][h] * vf;
    }
#pragma unroll
    for (int h = 0; h < NREP; ++h) o_acc[h] = o_acc[h] * alpha[h] + acc[h];

    const bool piece_end = (cur.t + 1 == t1) || (cur.j + 1 == cur.n);
    if (piece_end) {
      // Sum the per-token partial normalisers across the CTA.
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        float l = l_part[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) S.lred[warp][h] = l;
      }
      __syncthreads();
      const bool whole = (piece_first == cur.seg_base) && (cur.j + 1 == cur.n);
      const int64_t slot = (piece_first == cur.seg_base)
                               ? (int64_t)cur.b * a.Hkv + cur.g
                               : (int64_t)a.B * a.Hkv + blockIdx.x;
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        const float l = S.lred[0][h] + S.lred[1][h] + S.lred[2][h] + S.lred[3][h];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float ov = o_acc[h] * inv;
        const float lse2 = l > 0.f ? m_run[h] + log2f(l) : -INFINITY;
        if (whole) {
          const int64_t row = (int64_t)cur.b * a.H + (int64_t)cur.g * NREP + h;
          if (a.out_f32)
            reinterpret_cast<float*>(a.out)[row * D + tid] = ov;
          else
            reinterpret_cast<__nv_bfloat16*>(a.out)[row * D + tid] = __float2bfloat16_rn(ov);
          if (a.lse && tid == 0) a.lse[row] = lse2 * kLn2;
        } else {
          a.ws_o[(slot * NREP + h) * D + tid] = ov;
          if (tid == 0) a.ws_lse[slot * NREP + h] = lse2;
        }
      }
    }
    __syncthreads();  // everyone is done with this ring slot and with S.p / S.q
    ++it;
    if (!cursor_next(cur, a.seq_lens, a.B, a.Hkv, bs, a.window, cap)) break;
  }
  cp_async_wait<0>();
}

// --------------------------------------------------------------------------
// LSE merge of split pieces: lse = log sum_i exp(lse_i), o = sum_i exp(lse_i - lse) o_i.
// Grid (b * Hkv + kv head, block of 16 query rows); one warp per query row of the
// group (q_len * n_rep rows, ordered token then head); lane = 4 consecutive output
// elements. Segments finished inside one attention CTA are skipped; empty
// sequences get o = 0, lse = -inf.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(512) decode_merge_kernel(DecodeArgs a) {
  constexpr int D = 128;
  const int seg = blockIdx.x;  // b * Hkv + g
  const int b = seg / a.Hkv, g = seg % a.Hkv;
  const int h = blockIdx.y * 16 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int n_rep = a.n_rep * a.q_len;  // rows per (b, kv head)
  if (h >= n_rep) return;
  const int bs = 128;
  const int cap = a.max_blocks * bs;
  int64_t tot = 0, before = 0;
  for (int bb = lane; bb < a.B; bb += 32) {
    const int n = live_blocks(clamp_len(__ldg(a.seq_lens + bb), cap), bs, a.window).n;
    tot += n;
    if (bb < b) before += n;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
  }
  const int64_t T = tot * a.Hkv, G = a.num_ctas;
  const int n = live_blocks(clamp_len(__ldg(a.seq_lens + b), cap), bs, a.window).n;
  const int64_t base = before * a.Hkv + (int64_t)g * n;
  const int64_t row =
      ((int64_t)b * a.q_len + h / a.n_rep) * a.H + (int64_t)g * a.n_rep + h % a.n_rep;
  auto put = [&](float4 v) {
    if (a.out_f32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + row * D)[lane] = v;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * D)[lane] =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
  };
  const int64_t i0 = n ? cta_of_tile(base, T, G) : 0, i1 = n ? cta_of_tile(base + n - 1, T, G) : 0;
  if (n > 0 && i0 == i1) return;  // finished by the attention kernel
  // The pieces' workspace slots, found before the wait (they depend on the inputs
  // only), so that after it every piece's loads are issued at once.
  constexpr int kMaxPieces = 8;
  auto slot_of = [&](int64_t i) { return (i == i0) ? (int64_t)seg : (int64_t)a.B * a.Hkv + i; };
  int64_t slots[kMaxPieces];
  int np = 0;
  for (int64_t i = i0; n > 0 && i <= i1; ++i) {
    if (i > i0 && cta_tile_start(i + 1, T, G) == cta_tile_start(i, T, G)) continue;  // empty CTA
    if (np < kMaxPieces) slots[np] = slot_of(i);
    ++np;
  }
  pdl_wait_primary();
  if (n == 0) {
    put(make_float4(0.f, 0.f, 0.f, 0.f));
    if (a.lse && lane == 0) a.lse[row] = -INFINITY;
    return;
  }
  float mx = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (np <= kMaxPieces) {
    float l2[kMaxPieces];
    float4 x[kMaxPieces];
#pragma unroll
    for (int p = 0; p < kMaxPieces; ++p) {
      if (p < np) {
        l2[p] = a.ws_lse[slots[p] * n_rep + h];
        x[p] = reinterpret_cast<const float4*>(a.ws_o + (slots[p] * n_rep + h) * D)[lane];
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
    // More pieces than registers hold (segments far longer than a CTA's share).
    for (int64_t i = i0; i <= i1; ++i) {
      if (i > i0 && cta_tile_start(i + 1, T, G) == cta_tile_start(i, T, G)) continue;
      mx = fmaxf(mx, a.ws_lse[slot_of(i) * n_rep + h]);
    }
    for (int64_t i = i0; i <= i1; ++i) {
      if (i > i0 && cta_tile_start(i + 1, T, G) == cta_tile_start(i, T, G)) continue;
      const int64_t slot = slot_of(i);
      const float l2 = a.ws_lse[slot * n_rep + h];
      const float w = (l2 == -INFINITY) ? 0.f : exp2f(l2 - mx);
      const float4 x = reinterpret_cast<const float4*>(a.ws_o + (slot * n_rep + h) * D)[lane];
      acc.x += w * x.x;
      acc.y += w * x.y;
      acc.z += w * x.z;
      acc.w += w * x.w;
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  put(make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  if (a.lse && lane == 0) a.lse[row] = wsum > 0.f ? (mx + log2f(wsum)) * kLn2 : -INFINITY;
}

// H here counts every query row of a sequence (q_len * heads).
size_t decode_workspace_bytes(int B, int H, int Hkv, int D, int G) {
  const int64_t slots = (int64_t)B * Hkv + G;
  const int64_t n_rep = H / Hkv;
  const size_t o_bytes = (size_t)(slots * n_rep * D * 4 + 255) / 256 * 256;
  const size_t l_bytes = (size_t)(slots * n_rep * 4 + 255) / 256 * 256;
  return o_bytes + l_bytes;
}

void decode_workspace_carve(DecodeArgs& a, void* ws) {
  const int64_t slots = (int64_t)a.B * a.Hkv + a.num_ctas;
  const size_t o_bytes = (size_t)(slots * a.n_rep * a.q_len * 128 * 4 + 255) / 256 * 256;
  a.ws_o = reinterpret_cast<float*>(ws);
  a.ws_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + o_bytes);
}

template <int NREP>
static cudaError_t launch_simt_n(const DecodeArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem<NREP>);
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<NREP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(decode_simt_kernel<NREP>, dim3(a.num_ctas), dim3(simt::THREADS), smem, stream, a);
}

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.n_rep) {
    case 1: return launch_simt_n<1>(a, stream);
    case 2: return launch_simt_n<2>(a, stream);
    case 4: return launch_simt_n<4>(a, stream);
    case 8: return launch_simt_n<8>(a, stream);
    case 16: return launch_simt_n<16>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream) {
  if (a.B * a.Hkv == 0) return cudaSuccess;
  const int rows = a.n_rep * a.q_len;
  const dim3 grid(a.B * a.Hkv, (rows + 15) / 16);
  return launch_dependent(decode_merge_kernel, grid, dim3(32 * (rows < 16 ? rows : 16)), 0, stream, a);
}

}  // namespace pkv
