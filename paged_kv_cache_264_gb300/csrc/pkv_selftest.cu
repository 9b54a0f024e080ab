// pkv_selftest.cu -- failure-detection self-test: the decode kernels' bounded mbarrier wait,
// run on a barrier that nothing completes, must give up, report the timeout bit and leave
// the CUDA context usable.  No fault, trap or hang is involved.
#include <cstdio>

#include "../../include/pagedkv.h"
#include "pkv_device.cuh"

namespace {

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, uint32_t* flags,
                                             unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pkv::mbar_init(&bar, 1);  // expects one arrival, which never comes
    pkv::fence_barrier_init();
  }
  __syncwarp();
  const uint64_t t0 = pkv::global_timer_ns();
  const bool done = pkv::mbar_wait_bounded(&bar, 0, limit_ns);
  const uint64_t t1 = pkv::global_timer_ns();
  if (threadIdx.x == 0) {
    if (!done) atomicOr(flags, pkv::kErrTimeout);
    *waited_ns = static_cast<unsigned long long>(t1 - t0);
  }
}

}  // namespace

extern "C" {

PKV_API pkv_status pkv_selftest_bounded_wait(uint64_t limit_ns, uint32_t* flags, uint64_t* waited_ns,
                                             void* stream) {
  if (!flags || !waited_ns || limit_ns < 100000u || limit_ns > pkv::kWaitTimeoutNs)
    return PKV_ERR_INVALID_ARG;
  auto s = static_cast<cudaStream_t>(stream);
  void* d = nullptr;
  if (cudaMalloc(&d, 16) != cudaSuccess) return PKV_ERR_CUDA;
  uint32_t* d_flags = static_cast<uint32_t*>(d);
  auto* d_waited = reinterpret_cast<unsigned long long*>(static_cast<char*>(d) + 8);
  pkv_status st = PKV_OK;
  uint32_t h[4] = {0, 0, 0, 0};
  if (cudaMemsetAsync(d, 0, 16, s) != cudaSuccess) st = PKV_ERR_CUDA;
  if (st == PKV_OK) {
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, d_flags, d_waited);
    if (cudaGetLastError() != cudaSuccess) st = PKV_ERR_CUDA;
  }
  if (st == PKV_OK && (cudaMemcpyAsync(h, d, 16, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                       cudaStreamSynchronize(s) != cudaSuccess))
    st = PKV_ERR_CUDA;
  cudaFree(d);
  if (st != PKV_OK) return st;
  *flags = h[0];
  *waited_ns = uint64_t(h[2]) | (uint64_t(h[3]) << 32);
  return PKV_OK;
}

}  // extern "C"
