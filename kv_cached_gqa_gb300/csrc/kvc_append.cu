// Append and length bookkeeping kernels.
//
// Append ("KV cache, incremental decode, ...", §4 update and §2.5 "Storage dtype"; "KV cache
// decoding", step 5): row t of a [B, H, T, D] chunk goes to position lens[b] + delta + t of
// (layer, b, h), rounded to the cache dtype to nearest even. Each thread moves one 16-byte group of
// output elements, so a warp writes 512 contiguous bytes of one row (or of consecutive rows):
// coalesced, vectorised stores with no read-modify-write. The write position comes from the
// device's committed lengths, so the kernel stays correct when replayed from a captured graph.
//
// Rotary positions (fused RoPE): a key row is rotated by its absolute position, the position it is
// written at, in float32 from a float64-built cos/sin table, and then rounded; V rows are stored as
// given. The table is [max_len, D/2] pairs of (cos, sin), built once per handle.
//
// Paged store: the row's physical block comes from the sequence's block table (pool layout
// [L, n_blocks, H, block, D]); the table edits that allocate blocks are one small launch before the
// append, in stream order.
//
// Lengths: commit adds T to every committed length, truncate overwrites them; both are one tiny
// kernel so the device copy changes in stream order with the rest of the forward.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "kvc_append.cuh"
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using app::Pack;

// One thread per 16-byte output group; grid covers 2 (K, V) x B x H x T x D / N groups. Tc is the
// storage type, Tin the input type (float32, the storage type itself, or a 16-bit type for fp8).
template <typename Tc, typename Tin>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  dev::pdl_wait();
  dev::pdl_trigger();
  constexpr int N = Pack<Tc>::N;
  const long long rows = static_cast<long long>(a.B) * a.H * a.T;
  const long long per_k = rows * (a.D / N);             // groups of the first store (K, or the latent)
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= per_k + rows * (a.Dv / N)) return;
  const bool is_v = gid >= per_k;
  const int groups_per_row = (is_v ? a.Dv : a.D) / N;
  const long long g = is_v ? gid - per_k : gid;
  app::append_group<Tc, Tin>(a, g / groups_per_row, static_cast<int>(g % groups_per_row), is_v);
}

__global__ void lens_add_kernel(int32_t* lens, int B, int delta) {
  dev::pdl_wait();
  dev::pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B) lens[i] += delta;
}

__global__ void table_edits_kernel(int32_t* table, const __grid_constant__ TableEdits e) {
  dev::pdl_wait();
  dev::pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < e.n) table[e.slot[i]] = e.value[i];
}

__global__ void rope_table_kernel(float2* table, int max_len, int half, const __grid_constant__ RopeTheta th) {
  dev::pdl_wait();
  dev::pdl_trigger();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(max_len) * half) return;
  const int p = static_cast<int>(i / half), j = static_cast<int>(i % half);
  double sn, c;
  sincos(static_cast<double>(p) * th.theta[j], &sn, &c);     // the angle in float64, then rounded
  table[i] = make_float2(static_cast<float>(c), static_cast<float>(sn));
}

struct LensValues {
  int32_t v[kMaxBatch];
};

__global__ void lens_set_kernel(int32_t* lens, int B, const __grid_constant__ LensValues n) {
  dev::pdl_wait();
  dev::pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B) lens[i] = n.v[i];
}

__global__ void positions_kernel(const int32_t* lens, int B, int T, int32_t* out) {
  dev::pdl_wait();
  dev::pdl_trigger();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < static_cast<long long>(B) * T) out[i] = lens[i / T] + static_cast<int>(i % T);
}

template <typename Tc, typename Tin>
cudaError_t run_append(const AppendArgs& a, cudaStream_t st) {
  constexpr int N = Pack<Tc>::N;
  const long long total = static_cast<long long>(a.B) * a.H * a.T * ((a.D + a.Dv) / N);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  return launch_pdl(append_kernel<Tc, Tin>, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st, a);
}

template <typename Tc>
cudaError_t run_append_in(const AppendArgs& a, cudaStream_t st) {
  switch (a.in_dtype) {
    case KVC_F32: return run_append<Tc, float>(a, st);
    case KVC_F16:
      if constexpr (std::is_same<Tc, __half>::value || std::is_same<Tc, dev::fp8>::value) return run_append<Tc, __half>(a, st);
      break;
    case KVC_BF16:
      if constexpr (std::is_same<Tc, __nv_bfloat16>::value || std::is_same<Tc, dev::fp8>::value)
        return run_append<Tc, __nv_bfloat16>(a, st);
      break;
    default: break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  switch (a.cache_dtype) {
    case KVC_F32: return run_append_in<float>(a, st);
    case KVC_F16: return run_append_in<__half>(a, st);
    case KVC_BF16: return run_append_in<__nv_bfloat16>(a, st);
    case KVC_FP8_E4M3: return run_append_in<dev::fp8>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_rope_table(float2* table, int max_len, int D, const RopeTheta& th, cudaStream_t st) {
  const long long n = static_cast<long long>(max_len) * (D / 2);
  return launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st, table,
                    max_len, D / 2, th);
}

cudaError_t launch_table_edits(int32_t* table, const TableEdits& e, cudaStream_t st) {
  if (e.n <= 0) return cudaSuccess;
  return launch_pdl(table_edits_kernel, dim3((e.n + 255) / 256), dim3(256), 0, st, table, e);
}

cudaError_t launch_lens_add(int32_t* lens, int B, int delta, cudaStream_t st) {
  return launch_pdl(lens_add_kernel, dim3((B + 255) / 256), dim3(256), 0, st, lens, B, delta);
}

cudaError_t launch_lens_set(int32_t* lens, int B, const int32_t* n_host, cudaStream_t st) {
  LensValues v;
  for (int i = 0; i < B; ++i) v.v[i] = n_host[i];
  return launch_pdl(lens_set_kernel, dim3((B + 255) / 256), dim3(256), 0, st, lens, B, v);
}

cudaError_t launch_positions(const int32_t* lens, int B, int T, int32_t* out, cudaStream_t st) {
  const long long n = static_cast<long long>(B) * T;
  return launch_pdl(positions_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st,
                    lens, B, T, out);
}

}  // namespace kvc
