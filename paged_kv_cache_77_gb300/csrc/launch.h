// Internal launcher interface between the C ABI layer (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

cudaError_t launch_kv_write(void* k_cache, void* v_cache, const void* k, const void* v,
                            const int32_t* slots, int64_t num_tokens, int64_t num_slots,
                            int64_t row_k_bytes, int64_t row_v_bytes, int* dev_status,
                            cudaStream_t stream, int num_sms);
cudaError_t launch_kv_write_fp8(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                const void* k, const void* v, const int32_t* slots,
                                int64_t num_tokens, int64_t num_blocks, int block_size, int hkv,
                                int* dev_status, cudaStream_t stream, int num_sms);
cudaError_t launch_copy_blocks(void* cache, int64_t num_blocks, int64_t block_bytes,
                               const int32_t* src, const int32_t* dst, int64_t n, int* dev_status,
                               cudaStream_t stream, int num_sms);
cudaError_t launch_mla_rmsnorm_rope_write(void* cache_nope, void* cache_rope, void* k_nope_out,
                                          void* k_rope_out, const void* latent, const void* gamma,
                                          const float* cosv, const float* sinv,
                                          const int32_t* slots, int64_t num_tokens,
                                          int64_t num_slots, float eps, int* dev_status,
                                          cudaStream_t stream, int num_sms);

// Arguments of the split-KV decode kernels and their LSE merge.
struct DecodeArgs {
  const uint16_t* q;          // [B, q_len, H, D] bf16
  const uint8_t* k_cache;     // [nb, bs, Hkv, D] bf16
  const uint8_t* v_cache;
  const int32_t* block_table; // [B, max_blocks]
  const int32_t* seq_lens;    // [B]
  void* out;                  // [B, q_len, H, D] bf16 or f32
  float* lse;                 // [B, q_len, H] or null
  float* ws_o;                // [(B*Hkv + G) * q_len * n_rep * D] partial outputs
  float* ws_lse;              // [(B*Hkv + G) * q_len * n_rep] partial log2-sum-exp
  int* dev_status;
  int64_t num_blocks;
  int B, H, Hkv, n_rep, max_blocks, out_f32;
  int q_len;                  // new query rows per sequence (1 = plain decode)
  int row_window;             // window of one query row (0 = full attention)
  int window;                 // live-block span: row_window + q_len - 1 (0 = all)
  int num_ctas;               // G: CTAs of the attention kernel (one per SM)
  float scale_log2;           // scale * log2(e)
  const float* k_scale;       // FP8 cache only: [nb, Hkv, bs] per-row scales
  const float* v_scale;
};

size_t decode_workspace_bytes(int B, int H, int Hkv, int D, int G);
void decode_workspace_carve(DecodeArgs& a, void* ws);

// CUDA-core split-KV decode (any group size 1..16) followed by the LSE merge.
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream);
// tcgen05 split-KV decode for head groups (n_rep 1..16), same partials as above.
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);
// The same kernel for q_len 1..4 query rows per sequence (q_len * n_rep <= 32).
cudaError_t launch_decode_spec(const DecodeArgs& a, cudaStream_t stream);
// tcgen05 split-KV decode over an FP8 (E4M3) cache with per-row scales; same
// partials and merge as above.
cudaError_t launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream);

// Absorbed MLA decode (tcgen05) plus its merge, q_len query rows per sequence
// (1 for plain decode). Workspace: mla_workspace_bytes(B * q_len, num_sms / 2).
size_t mla_workspace_bytes(int rows, int g_half);
cudaError_t launch_mla_decode(const void* q_nope, const void* q_rope, const void* cache_nope,
                              const void* cache_rope, const int32_t* block_table, int max_blocks,
                              const int32_t* seq_lens, void* out, int out_f32, float* lse, int B,
                              int q_len, int H, int64_t num_blocks, float scale, void* ws,
                              int* dev_status, int num_sms, cudaStream_t stream);

// Causal paged prefill (tcgen05, stream-K) plus its merge.
size_t prefill_workspace_bytes(int G);
cudaError_t launch_prefill(const void* q, const int32_t* cu_q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table, int max_blocks,
                           const int32_t* seq_lens, void* out, int out_f32, float* lse, int T,
                           int B, int H, int Hkv, int64_t num_blocks, float scale, int causal,
                           void* ws, int* dev_status, int num_sms, cudaStream_t stream);

// Self-test: a bounded wait that runs out (selftest.cu).
cudaError_t launch_bounded_wait(int* dev_status, cudaStream_t stream);

}  // namespace pkv
