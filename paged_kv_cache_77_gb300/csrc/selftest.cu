// Self-test of the kernels' failure path: every wait on an mbarrier inside the
// attention kernels is bounded, and a wait that gives up sets PKV_DEV_TIMEOUT in the
// caller's status word and lets the kernel wind down instead of hanging the GPU. This
// kernel waits, with the same wait routines, on an mbarrier that nothing completes,
// so that a test can watch that path run out and check the status and that the CUDA
// context is still usable afterwards. Nothing here faults or spins without a limit.
#include "device_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {

__global__ void __launch_bounds__(64) bounded_wait_kernel(int* dev_status) {
  using namespace tc;
  __shared__ __align__(8) uint64_t bar;  // initialised with one expected arrival that never comes
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  // Phase 0 never completes: the spinning wait (issuing threads) and the sleeping wait
  // (producer threads) each give up after their cycle limit.
  if (threadIdx.x == 0) ok = mbar_wait(b, 0);
  if (threadIdx.x == 32) ok = mbar_wait_sleepy(b, 0);
  if (!ok) flag_status(dev_status, PKV_DEV_TIMEOUT);
}

cudaError_t launch_bounded_wait(int* dev_status, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 64, 0, stream>>>(dev_status);
  return cudaGetLastError();
}

}  // namespace pkv
