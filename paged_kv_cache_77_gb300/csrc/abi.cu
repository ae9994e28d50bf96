// C ABI entry points for the device calls: argument validation, workspace
// carving and kernel dispatch onto the caller's stream. Nothing here allocates,
// frees or synchronises device memory.
#include <cuda_runtime.h>

#include <cmath>

#include "abi_common.h"
#include "launch.h"

namespace pkv {

// SM count of the current device (queried once per device).
static int current_num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

// Decode kernel choice (process-wide): 0 = automatic, 1 = CUDA cores, 2 = tensor cores.
static int g_decode_kernel = 0;

static int launch_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return PKV_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return PKV_ERR_LAUNCH;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_kv_cache_write(void* k_cache, void* v_cache, const void* k, const void* v,
                       const int32_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim_k,
                       int32_t head_dim_v, int* dev_status, void* stream) {
  PKV_REQUIRE(num_tokens >= 0 && num_blocks > 0 && block_size > 0 && num_kv_heads > 0 &&
                  head_dim_k > 0,
              PKV_ERR_INVALID_ARG, "pkv_kv_cache_write: non-positive size");
  PKV_REQUIRE(k_cache && (num_tokens == 0 || (k && slot_mapping)), PKV_ERR_INVALID_ARG,
              "pkv_kv_cache_write: null pointer");
  // v goes with v_cache; with no rows to write, v may be NULL (an empty tensor's
  // storage) either way.
  PKV_REQUIRE(v_cache ? (num_tokens == 0 || v != nullptr) : (v == nullptr), PKV_ERR_INVALID_ARG,
              "pkv_kv_cache_write: v_cache and v must both be set or both be NULL");
  const int64_t row_k = (int64_t)num_kv_heads * head_dim_k * 2;
  const int64_t row_v = v_cache ? (int64_t)num_kv_heads * head_dim_v * 2 : 0;
  PKV_REQUIRE(row_k % 16 == 0 && row_v % 16 == 0, PKV_ERR_UNSUPPORTED,
              "pkv_kv_cache_write: row sizes must be multiples of 16 bytes");
  PKV_REQUIRE(aligned16(k_cache) && aligned16(k) && aligned16(v_cache) && aligned16(v),
              PKV_ERR_INVALID_ARG, "pkv_kv_cache_write: pointers must be 16-byte aligned");
  const int64_t num_slots = num_blocks * block_size;
  clear_error();
  return launch_status(launch_kv_write(k_cache, v_cache, k, v, slot_mapping, num_tokens, num_slots,
                                       row_k, row_v, dev_status, (cudaStream_t)stream,
                                       current_num_sms()),
                       "pkv_kv_cache_write");
}

int pkv_copy_blocks(void* cache, int64_t num_blocks, int64_t block_bytes, const int32_t* src,
                    const int32_t* dst, int64_t n, int* dev_status, void* stream) {
  PKV_REQUIRE(num_blocks > 0 && n >= 0 && block_bytes > 0 && block_bytes % 16 == 0,
              PKV_ERR_INVALID_ARG, "pkv_copy_blocks: bad sizes");
  PKV_REQUIRE(cache && aligned16(cache) && (n == 0 || (src && dst)), PKV_ERR_INVALID_ARG,
              "pkv_copy_blocks: null or misaligned pointer");
  clear_error();
  return launch_status(launch_copy_blocks(cache, num_blocks, block_bytes, src, dst, n, dev_status,
                                          (cudaStream_t)stream, current_num_sms()),
                       "pkv_copy_blocks");
}

int pkv_mla_rmsnorm_rope_write(void* cache_nope, void* cache_rope, void* k_nope_out,
                               void* k_rope_out, const void* latent, const void* gamma,
                               const float* cos, const float* sin, const int32_t* slot_mapping,
                               int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                               int32_t kv_lora_rank, int32_t rope_dim, float epsilon,
                               int* dev_status, void* stream) {
  PKV_REQUIRE(num_tokens >= 0 && num_blocks > 0 && block_size > 0, PKV_ERR_INVALID_ARG,
              "pkv_mla_rmsnorm_rope_write: bad sizes");
  PKV_REQUIRE(kv_lora_rank == 512 && rope_dim == 64, PKV_ERR_UNSUPPORTED,
              "pkv_mla_rmsnorm_rope_write: only kv_lora_rank 512 and rope_dim 64 are implemented");
  PKV_REQUIRE(std::isfinite(epsilon) && epsilon >= 0.f, PKV_ERR_INVALID_ARG,
              "pkv_mla_rmsnorm_rope_write: epsilon must be finite and >= 0");
  PKV_REQUIRE(cache_nope && cache_rope && gamma &&
                  (num_tokens == 0 || (latent && cos && sin && slot_mapping)),
              PKV_ERR_INVALID_ARG, "pkv_mla_rmsnorm_rope_write: null pointer");
  PKV_REQUIRE(aligned16(cache_nope) && aligned16(cache_rope) && aligned16(k_nope_out) &&
                  aligned16(k_rope_out) && aligned16(latent) && aligned16(gamma) && aligned16(cos) &&
                  aligned16(sin),
              PKV_ERR_INVALID_ARG, "pkv_mla_rmsnorm_rope_write: pointers must be 16-byte aligned");
  clear_error();
  return launch_status(
      launch_mla_rmsnorm_rope_write(cache_nope, cache_rope, k_nope_out, k_rope_out, latent, gamma,
                                    cos, sin, slot_mapping, num_tokens, num_blocks * block_size,
                                    epsilon, dev_status, (cudaStream_t)stream, current_num_sms()),
      "pkv_mla_rmsnorm_rope_write");
}

int pkv_set_decode_kernel(int32_t kernel) {
  PKV_REQUIRE(kernel >= PKV_KERNEL_AUTO && kernel <= PKV_KERNEL_TENSOR_CORE, PKV_ERR_INVALID_ARG,
              "pkv_set_decode_kernel: unknown kernel %d", kernel);
  g_decode_kernel = kernel;
  return PKV_OK;
}

int32_t pkv_get_decode_kernel(void) { return g_decode_kernel; }

size_t pkv_decode_workspace_size(int32_t B, int32_t H, int32_t H_kv, int32_t head_dim) {
  if (B < 0 || H <= 0 || H_kv <= 0 || H % H_kv || head_dim <= 0) return 0;
  return decode_workspace_bytes(B, H, H_kv, head_dim, current_num_sms());
}

}  // extern "C"

namespace {

// Validation and argument set-up shared by the decode entry points. `what` names
// the caller in error messages; *empty is set when B == 0 (nothing to launch).
int decode_setup(pkv::DecodeArgs& a, bool* empty, const char* what, void* out, int32_t out_dtype,
                 float* lse, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                 int32_t B, int32_t H, int32_t H_kv, int32_t head_dim, int32_t block_size,
                 int64_t num_blocks, float scale, int32_t window, void* workspace,
                 size_t workspace_bytes, int* dev_status, int32_t q_len = 1) {
  using namespace pkv;
  *empty = false;
  PKV_REQUIRE(B >= 0 && H > 0 && H_kv > 0 && max_blocks_per_seq > 0 && num_blocks > 0,
              PKV_ERR_INVALID_ARG, "%s: bad sizes", what);
  PKV_REQUIRE(H % H_kv == 0, PKV_ERR_INVALID_ARG, "%s: H (%d) not a multiple of H_kv (%d)", what,
              H, H_kv);
  const int n_rep = H / H_kv;
  PKV_REQUIRE(head_dim == 128 && block_size == 128, PKV_ERR_UNSUPPORTED,
              "%s: only head_dim 128 and block_size 128 are implemented", what);
  PKV_REQUIRE(n_rep == 1 || n_rep == 2 || n_rep == 4 || n_rep == 8 || n_rep == 16,
              PKV_ERR_UNSUPPORTED, "%s: H / H_kv = %d unsupported", what, n_rep);
  PKV_REQUIRE(out_dtype == PKV_BF16 || out_dtype == PKV_F32, PKV_ERR_INVALID_ARG,
              "%s: bad out_dtype", what);
  PKV_REQUIRE(std::isfinite(scale) && scale > 0.f, PKV_ERR_INVALID_ARG,
              "%s: scale must be a positive finite number", what);
  PKV_REQUIRE(window >= 0, PKV_ERR_INVALID_ARG, "%s: negative window", what);
  PKV_REQUIRE(q_len >= 1 && q_len <= 4, PKV_ERR_UNSUPPORTED, "%s: q_len %d outside 1..4", what,
              q_len);
  PKV_REQUIRE(q_len * n_rep <= 32, PKV_ERR_UNSUPPORTED,
              "%s: q_len * H / H_kv = %d exceeds 32 query rows per kv head", what, q_len * n_rep);
  PKV_REQUIRE(window <= INT32_MAX - 4, PKV_ERR_INVALID_ARG, "%s: window too large", what);
  PKV_REQUIRE(num_blocks * block_size <= INT32_MAX, PKV_ERR_UNSUPPORTED,
              "%s: num_blocks * block_size must fit in int32", what);
  if (B == 0) {
    *empty = true;
    return PKV_OK;
  }
  PKV_REQUIRE(out && q && k_cache && v_cache && block_table && seq_lens, PKV_ERR_INVALID_ARG,
              "%s: null pointer", what);
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
              PKV_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", what);
  const int G = current_num_sms();
  PKV_REQUIRE(G > 0, PKV_ERR_LAUNCH, "%s: no CUDA device", what);
  const size_t need = decode_workspace_bytes(B, H * q_len, H_kv, head_dim, G);
  PKV_REQUIRE(workspace && workspace_bytes >= need && (((uintptr_t)workspace) & 255) == 0,
              PKV_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 256-aligned", what, need);
  a = DecodeArgs{};
  a.q = (const uint16_t*)q;
  a.k_cache = (const uint8_t*)k_cache;
  a.v_cache = (const uint8_t*)v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse = lse;
  a.dev_status = dev_status;
  a.num_blocks = num_blocks;
  a.B = B;
  a.H = H;
  a.Hkv = H_kv;
  a.n_rep = n_rep;
  a.max_blocks = max_blocks_per_seq;
  a.q_len = q_len;
  a.row_window = window;
  a.window = window > 0 ? window + q_len - 1 : 0;
  a.out_f32 = out_dtype == PKV_F32;
  a.num_ctas = G;
  a.scale_log2 = scale * 1.4426950408889634f;
  decode_workspace_carve(a, workspace);
  return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_attention_decode(void* out, int32_t out_dtype, float* lse, const void* q,
                               const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* seq_lens, int32_t B, int32_t H, int32_t H_kv,
                               int32_t head_dim, int32_t block_size, int64_t num_blocks,
                               float scale, int32_t window, void* workspace,
                               size_t workspace_bytes, int* dev_status, void* stream) {
  DecodeArgs a;
  bool empty;
  const int rc0 = decode_setup(a, &empty, "pkv_paged_attention_decode", out, out_dtype, lse, q,
                               k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, B, H,
                               H_kv, head_dim, block_size, num_blocks, scale, window, workspace,
                               workspace_bytes, dev_status);
  if (rc0 != PKV_OK || empty) return rc0;
  clear_error();
  cudaStream_t s = (cudaStream_t)stream;
  // Automatic choice: the tcgen05 kernel for every group size (also faster for n_rep 1:
  // 21.7 against 25.1 us on the tiny MHA workload).
  const bool tensor_cores = g_decode_kernel != PKV_KERNEL_CUDA_CORE;
  int rc = launch_status(tensor_cores ? launch_decode_tc(a, s) : launch_decode_simt(a, s),
                         "pkv_paged_attention_decode (attention)");
  if (rc != PKV_OK) return rc;
  return launch_status(launch_decode_merge(a, s), "pkv_paged_attention_decode (merge)");
}

size_t pkv_decode_spec_workspace_size(int32_t B, int32_t q_len, int32_t H, int32_t H_kv,
                                      int32_t head_dim) {
  if (B < 0 || q_len < 1 || H <= 0 || H_kv <= 0 || H % H_kv || head_dim <= 0) return 0;
  return decode_workspace_bytes(B, H * q_len, H_kv, head_dim, current_num_sms());
}

int pkv_paged_attention_decode_spec(void* out, int32_t out_dtype, float* lse, const void* q,
                                    const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                                    int32_t H_kv, int32_t head_dim, int32_t block_size,
                                    int64_t num_blocks, float scale, int32_t window,
                                    void* workspace, size_t workspace_bytes, int* dev_status,
                                    void* stream) {
  DecodeArgs a;
  bool empty;
  const int rc0 = decode_setup(a, &empty, "pkv_paged_attention_decode_spec", out, out_dtype, lse,
                               q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, B,
                               H, H_kv, head_dim, block_size, num_blocks, scale, window, workspace,
                               workspace_bytes, dev_status, q_len);
  if (rc0 != PKV_OK || empty) return rc0;
  clear_error();
  cudaStream_t s = (cudaStream_t)stream;
  int rc = launch_status(launch_decode_spec(a, s), "pkv_paged_attention_decode_spec (attention)");
  if (rc != PKV_OK) return rc;
  return launch_status(launch_decode_merge(a, s), "pkv_paged_attention_decode_spec (merge)");
}

int pkv_kv_cache_write_fp8(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                           const void* k, const void* v, const int32_t* slot_mapping,
                           int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim, int* dev_status, void* stream) {
  PKV_REQUIRE(num_tokens >= 0 && num_blocks > 0 && block_size > 0 && num_kv_heads > 0,
              PKV_ERR_INVALID_ARG, "pkv_kv_cache_write_fp8: bad sizes");
  PKV_REQUIRE(head_dim == 128, PKV_ERR_UNSUPPORTED,
              "pkv_kv_cache_write_fp8: only head_dim 128 is implemented");
  PKV_REQUIRE(k_cache && v_cache && k_scale && v_scale && (num_tokens == 0 || (k && v && slot_mapping)),
              PKV_ERR_INVALID_ARG, "pkv_kv_cache_write_fp8: null pointer");
  PKV_REQUIRE(aligned16(k_cache) && aligned16(v_cache) && aligned16(k) && aligned16(v) &&
                  (((uintptr_t)k_scale) & 3) == 0 && (((uintptr_t)v_scale) & 3) == 0,
              PKV_ERR_INVALID_ARG, "pkv_kv_cache_write_fp8: misaligned pointer");
  clear_error();
  return launch_status(launch_kv_write_fp8(k_cache, v_cache, k_scale, v_scale, k, v, slot_mapping,
                                           num_tokens, num_blocks, block_size, num_kv_heads,
                                           dev_status, (cudaStream_t)stream, current_num_sms()),
                       "pkv_kv_cache_write_fp8");
}

int pkv_paged_attention_decode_fp8(void* out, int32_t out_dtype, float* lse, const void* q,
                                   const void* k_cache, const void* v_cache, const float* k_scale,
                                   const float* v_scale, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t B,
                                   int32_t H, int32_t H_kv, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, float scale, int32_t window,
                                   void* workspace, size_t workspace_bytes, int* dev_status,
                                   void* stream) {
  DecodeArgs a;
  bool empty;
  const int rc0 = decode_setup(a, &empty, "pkv_paged_attention_decode_fp8", out, out_dtype, lse, q,
                               k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, B, H,
                               H_kv, head_dim, block_size, num_blocks, scale, window, workspace,
                               workspace_bytes, dev_status);
  if (rc0 != PKV_OK || empty) return rc0;
  PKV_REQUIRE(k_scale && v_scale && aligned16(k_scale) && aligned16(v_scale), PKV_ERR_INVALID_ARG,
              "pkv_paged_attention_decode_fp8: scale arrays must be set and 16-byte aligned");
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  clear_error();
  cudaStream_t s = (cudaStream_t)stream;
  int rc = launch_status(launch_decode_fp8(a, s), "pkv_paged_attention_decode_fp8 (attention)");
  if (rc != PKV_OK) return rc;
  return launch_status(launch_decode_merge(a, s), "pkv_paged_attention_decode_fp8 (merge)");
}

size_t pkv_prefill_workspace_size(void) { return prefill_workspace_bytes(current_num_sms()); }

int pkv_paged_attention_prefill(void* out, int32_t out_dtype, float* lse, const void* q,
                                const int32_t* cu_seqlens_q, int32_t num_tokens,
                                const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens_kv, int32_t B, int32_t H, int32_t H_kv,
                                int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                float scale, int32_t causal, void* workspace,
                                size_t workspace_bytes, int* dev_status, void* stream) {
  PKV_REQUIRE(B >= 0 && num_tokens >= 0 && H > 0 && H_kv > 0 && max_blocks_per_seq > 0 &&
                  num_blocks > 0,
              PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: bad sizes");
  PKV_REQUIRE(H % H_kv == 0, PKV_ERR_INVALID_ARG,
              "pkv_paged_attention_prefill: H (%d) not a multiple of H_kv (%d)", H, H_kv);
  const int n_rep = H / H_kv;
  PKV_REQUIRE(head_dim == 128 && block_size == 128, PKV_ERR_UNSUPPORTED,
              "pkv_paged_attention_prefill: only head_dim 128 and block_size 128 are implemented");
  PKV_REQUIRE(n_rep == 1 || n_rep == 2 || n_rep == 4 || n_rep == 8 || n_rep == 16,
              PKV_ERR_UNSUPPORTED, "pkv_paged_attention_prefill: H / H_kv = %d unsupported", n_rep);
  PKV_REQUIRE(out_dtype == PKV_BF16 || out_dtype == PKV_F32, PKV_ERR_INVALID_ARG,
              "pkv_paged_attention_prefill: bad out_dtype");
  PKV_REQUIRE(std::isfinite(scale) && scale > 0.f, PKV_ERR_INVALID_ARG,
              "pkv_paged_attention_prefill: scale must be a positive finite number");
  PKV_REQUIRE(causal == 0 || causal == 1, PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: causal");
  PKV_REQUIRE(num_blocks * block_size <= INT32_MAX, PKV_ERR_UNSUPPORTED,
              "pkv_paged_attention_prefill: num_blocks * block_size must fit in int32");
  if (B == 0 || num_tokens == 0) return PKV_OK;
  PKV_REQUIRE(out && q && cu_seqlens_q && k_cache && v_cache && block_table && seq_lens_kv,
              PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: null pointer");
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
              PKV_ERR_INVALID_ARG, "pkv_paged_attention_prefill: pointers must be 16-byte aligned");
  const int G = current_num_sms();
  PKV_REQUIRE(G > 0, PKV_ERR_LAUNCH, "pkv_paged_attention_prefill: no CUDA device");
  const size_t need = prefill_workspace_bytes(G);
  PKV_REQUIRE(workspace && workspace_bytes >= need && (((uintptr_t)workspace) & 255) == 0,
              PKV_ERR_WORKSPACE, "pkv_paged_attention_prefill: workspace needs %zu bytes, 256-aligned",
              need);
  clear_error();
  return launch_status(launch_prefill(q, cu_seqlens_q, k_cache, v_cache, block_table,
                                      max_blocks_per_seq, seq_lens_kv, out, out_dtype == PKV_F32, lse,
                                      num_tokens, B, H, H_kv, num_blocks, scale, causal, workspace,
                                      dev_status, G, (cudaStream_t)stream),
                       "pkv_paged_attention_prefill");
}

// Absorbed MLA decode of q_len query rows per sequence (q_len = 1: plain decode).
static int mla_decode(const char* name, void* out, int32_t out_dtype, float* lse,
                      const void* q_nope, const void* q_rope, const void* cache_nope,
                      const void* cache_rope, const int32_t* block_table, int32_t max_blocks_per_seq,
                      const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                      int32_t kv_lora_rank, int32_t rope_dim, int32_t block_size, int64_t num_blocks,
                      float scale, void* workspace, size_t workspace_bytes, int* dev_status,
                      void* stream) {
  PKV_REQUIRE(B >= 0 && H > 0 && max_blocks_per_seq > 0 && num_blocks > 0, PKV_ERR_INVALID_ARG,
              "%s: bad sizes", name);
  PKV_REQUIRE(q_len >= 1 && q_len <= 4, PKV_ERR_UNSUPPORTED, "%s: q_len must be 1..4", name);
  PKV_REQUIRE(kv_lora_rank == 512 && rope_dim == 64 && block_size == 128 && H <= 128,
              PKV_ERR_UNSUPPORTED,
              "%s: implemented for kv_lora_rank 512, rope 64, block_size 128, H <= 128", name);
  PKV_REQUIRE(out_dtype == PKV_BF16 || out_dtype == PKV_F32, PKV_ERR_INVALID_ARG,
              "%s: bad out_dtype", name);
  PKV_REQUIRE(std::isfinite(scale) && scale > 0.f, PKV_ERR_INVALID_ARG,
              "%s: scale must be a positive finite number", name);
  PKV_REQUIRE(num_blocks * block_size <= INT32_MAX, PKV_ERR_UNSUPPORTED,
              "%s: num_blocks * block_size must fit in int32", name);
  PKV_REQUIRE((int64_t)B * q_len * H <= INT32_MAX, PKV_ERR_UNSUPPORTED,
              "%s: B * q_len * H must fit in int32", name);
  if (B == 0) return PKV_OK;
  PKV_REQUIRE(out && q_nope && q_rope && cache_nope && cache_rope && block_table && seq_lens,
              PKV_ERR_INVALID_ARG, "%s: null pointer", name);
  PKV_REQUIRE(aligned16(out) && aligned16(q_nope) && aligned16(q_rope) && aligned16(cache_nope) &&
                  aligned16(cache_rope),
              PKV_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", name);
  const int G = current_num_sms();
  PKV_REQUIRE(G >= 2, PKV_ERR_LAUNCH, "%s: no CUDA device", name);
  const size_t need = mla_workspace_bytes(B * q_len, G / 2);
  PKV_REQUIRE(workspace && workspace_bytes >= need && (((uintptr_t)workspace) & 255) == 0,
              PKV_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 256-aligned", name, need);
  clear_error();
  return launch_status(launch_mla_decode(q_nope, q_rope, cache_nope, cache_rope, block_table,
                                         max_blocks_per_seq, seq_lens, out, out_dtype == PKV_F32,
                                         lse, B, q_len, H, num_blocks, scale, workspace, dev_status,
                                         G, (cudaStream_t)stream),
                       name);
}

size_t pkv_mla_decode_workspace_size(int32_t B, int32_t H) {
  if (B < 0 || H <= 0) return 0;
  return mla_workspace_bytes(B, current_num_sms() / 2);
}

int pkv_mla_paged_decode(void* out, int32_t out_dtype, float* lse, const void* q_nope,
                         const void* q_rope, const void* cache_nope, const void* cache_rope,
                         const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, int32_t B, int32_t H, int32_t kv_lora_rank,
                         int32_t rope_dim, int32_t block_size, int64_t num_blocks, float scale,
                         void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  return mla_decode("pkv_mla_paged_decode", out, out_dtype, lse, q_nope, q_rope, cache_nope,
                    cache_rope, block_table, max_blocks_per_seq, seq_lens, B, 1, H, kv_lora_rank,
                    rope_dim, block_size, num_blocks, scale, workspace, workspace_bytes, dev_status,
                    stream);
}

size_t pkv_mla_decode_spec_workspace_size(int32_t B, int32_t q_len, int32_t H) {
  if (B < 0 || q_len < 1 || H <= 0) return 0;
  return mla_workspace_bytes(B * q_len, current_num_sms() / 2);
}

int pkv_mla_paged_decode_spec(void* out, int32_t out_dtype, float* lse, const void* q_nope,
                              const void* q_rope, const void* cache_nope, const void* cache_rope,
                              const int32_t* block_table, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                              int32_t kv_lora_rank, int32_t rope_dim, int32_t block_size,
                              int64_t num_blocks, float scale, void* workspace,
                              size_t workspace_bytes, int* dev_status, void* stream) {
  return mla_decode("pkv_mla_paged_decode_spec", out, out_dtype, lse, q_nope, q_rope, cache_nope,
                    cache_rope, block_table, max_blocks_per_seq, seq_lens, B, q_len, H,
                    kv_lora_rank, rope_dim, block_size, num_blocks, scale, workspace,
                    workspace_bytes, dev_status, stream);
}

int pkv_selftest_bounded_wait(int* dev_status, void* stream) {
  PKV_REQUIRE(dev_status != nullptr, PKV_ERR_INVALID_ARG, "pkv_selftest_bounded_wait: null dev_status");
  return launch_status(launch_bounded_wait(dev_status, static_cast<cudaStream_t>(stream)),
                       "pkv_selftest_bounded_wait");
}

}  // extern "C"
