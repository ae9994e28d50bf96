// Speculative (multi-token) decode on the tcgen05 decode kernel (decode_tc.cuh):
// q_len = 2..4 new query rows per sequence, bottom-right causal ("昇腾 NPU 独立部署
// 模式 KVCache 自管完整指南", appendix C: a decode step with q_len > 1 takes the
// prefill mask, sparse_mode 3). Kept apart from decode_tc.cu so that the two
// translation units compile in parallel.
#include "decode_tc.cuh"

namespace pkv {

template <int QL>
static cudaError_t launch_spec_q(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.n_rep) {
    case 1: return launch_tc_n<1, QL>(a, stream);
    case 2: return launch_tc_n<2, QL>(a, stream);
    case 4: return launch_tc_n<4, QL>(a, stream);
    case 8: return launch_tc_n<8, QL>(a, stream);
    case 16:
      if constexpr (QL <= 2) return launch_tc_n<16, QL>(a, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_spec(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.q_len) {
    case 1: return launch_decode_tc(a, stream);
    case 2: return launch_spec_q<2>(a, stream);
    case 3: return launch_spec_q<3>(a, stream);
    case 4: return launch_spec_q<4>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
