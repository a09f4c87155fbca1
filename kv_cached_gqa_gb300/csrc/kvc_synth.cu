// Device side of the seeded input generator (see include/kvc_synth.h). Holds none of the
// attention arithmetic. Philox4x32-10 as defined by Salmon et al. (SC 2011), §3.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kvc_synth.h"

namespace {

struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__global__ void fill_normal_kernel(float* out, size_t n, uint64_t offset, uint64_t seed,
                                   uint32_t stream_id, float std) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint64_t j = offset + i;
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  int64_t total = 0;
#pragma unroll
  for (uint32_t blk = 0; blk < 3; ++blk) {
    const U4 w = philox4x32_10(U4{static_cast<uint32_t>(j), static_cast<uint32_t>(j >> 32), stream_id, blk},
                               k0, k1);
    total += (w.x >> 8) + (w.y >> 8) + (w.z >> 8) + (w.w >> 8);
  }
  // exact in double (|total - 6*2^24| < 2^27), then one rounding to float32
  const float x = __double2float_rn(static_cast<double>(total - 6LL * (1LL << 24)) * 5.9604644775390625e-08);
  out[i] = (std == 1.0f) ? x : __fmul_rn(x, std);
}

}  // namespace

extern "C" int kvc_synth_fill_normal_f32(float* out_dev, size_t n, uint64_t offset, uint64_t seed,
                                         uint32_t stream_id, float std, void* stream) {
  if (n == 0) return 0;
  if (!out_dev) return -1;
  const unsigned threads = 256;
  const size_t blocks = (n + threads - 1) / threads;
  fill_normal_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      out_dev, n, offset, seed, stream_id, std);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
