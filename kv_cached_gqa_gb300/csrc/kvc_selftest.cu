// Self-test of the kernels' failure path: a bounded wait that runs out.
//
// Every wait in the attention kernels gives up after a time limit, sets the handle's device status
// word and lets the CTA finish, so a stuck pipeline is reported by kvc_status instead of hanging the
// GPU. This kernel exercises exactly that path without any fault: one thread waits on an mbarrier
// phase that nothing will ever complete, gives up after `limit_ns`, and records the timeout.
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace {

__global__ void wait_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = kvc::dev::smem_u32(&bar);
  kvc::dev::mbar_init(b, 1);                  // expects one arrival that never comes
  kvc::dev::fence_mbar_init();
  const unsigned long long t0 = kvc::dev::now_ns();
  bool done = false;
  while (!done) {
    done = kvc::dev::mbar_try(b, 0);
    if (!done && kvc::dev::now_ns() - t0 > limit_ns) break;
  }
  if (!done) atomicExch(status, kvc::kStatusTimeout);
}

}  // namespace

extern "C" int kvc_selftest_wait_timeout(kvc_handle h, int limit_us, void* stream) {
  if (!h || limit_us < 1 || limit_us > 1000000) return KVC_E_INVAL;
  wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      h->d_status, static_cast<unsigned long long>(limit_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return KVC_E_CUDA;
  h->launches += 1;
  return KVC_OK;
}
