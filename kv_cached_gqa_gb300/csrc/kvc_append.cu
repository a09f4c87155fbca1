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

#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

template <typename Tc>
struct Pack;   // 16 bytes of output elements
template <>
struct Pack<float> {
  static constexpr int N = 4;
  __device__ static uint4 from_f32(const float* x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
};
template <>
struct Pack<__half> {
  static constexpr int N = 8;
  __device__ static uint4 from_f32(const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = __half_as_ushort(__float2half_rn(x[2 * i]));
      const uint16_t hi = __half_as_ushort(__float2half_rn(x[2 * i + 1]));
      w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Pack<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static uint4 from_f32(const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(x[2 * i]));
      const uint16_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(x[2 * i + 1]));
      w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Pack<dev::fp8> {
  static constexpr int N = 16;
  // x already divided by the layer's scale: round to nearest even, saturate to +-448
  __device__ static uint4 from_f32(const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i], x[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i + 2], x[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
      w[i] = (lo & 0xffffu) | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// n consecutive input elements as float32 (float32 input, or a 16-bit input widened exactly).
template <typename Tin, int n>
__device__ __forceinline__ void load_group(const void* src, long long off, float* x) {
  if constexpr (std::is_same<Tin, float>::value) {
    const float* p = static_cast<const float*>(src) + off;
#pragma unroll
    for (int i = 0; i < n; i += 4) {
      const float4 f = *reinterpret_cast<const float4*>(p + i);
      x[i] = f.x; x[i + 1] = f.y; x[i + 2] = f.z; x[i + 3] = f.w;
    }
  } else {
    const Tin* p = static_cast<const Tin*>(src) + off;
#pragma unroll
    for (int i = 0; i < n; ++i) x[i] = dev::to_f32<Tin>(p[i]);
  }
}

// One thread per 16-byte output group; grid covers 2 (K, V) x B x H x T x D / N groups. Tc is the
// storage type, Tin the input type (float32, the storage type itself, or a 16-bit type for fp8).
template <typename Tc, typename Tin>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  dev::pdl_wait();
  dev::pdl_trigger();
  constexpr int N = Pack<Tc>::N;
  constexpr bool kFp8 = std::is_same<Tc, dev::fp8>::value;
  const long long rows = static_cast<long long>(a.B) * a.H * a.T;
  const long long per_k = rows * (a.D / N);             // groups of the first store (K, or the latent)
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= per_k + rows * (a.Dv / N)) return;
  const bool is_v = gid >= per_k;
  const int W = is_v ? a.Dv : a.D;                      // this store's row width
  const int groups_per_row = W / N;
  const long long g = is_v ? gid - per_k : gid;
  const long long row = g / groups_per_row;             // (b, h, t) row of the chunk
  const int grp = static_cast<int>(g % groups_per_row);
  const int t = static_cast<int>(row % a.T);
  const int bh = static_cast<int>(row / a.T);
  const int b = bh / a.H, h = bh % a.H;
  const int pos = a.lens[b] + a.delta + t;
  long long dst_row;
  if (a.pg.table == nullptr) {
    dst_row = ((static_cast<long long>(a.layer) * a.B + b) * a.H + h) * a.max_len + pos;
  } else {
    // paged: the row's block comes from the sequence's table (the host allocated it before this
    // launch); a missing block, which the host never lets happen, drops the write instead of
    // writing outside the pool
    const int blk = a.pg.table[static_cast<long long>(b) * a.pg.max_blocks + (pos >> a.pg.block_shift)];
    if (blk < 0 || blk >= a.pg.n_blocks) return;
    dst_row = (((static_cast<long long>(a.layer) * a.pg.n_blocks + blk) * a.H + h) << a.pg.block_shift) +
              (pos & ((1 << a.pg.block_shift) - 1));
  }
  Tc* dst = static_cast<Tc*>(is_v ? a.v_store : a.k_store) + dst_row * W + grp * N;
  const long long src_off = row * W + grp * N;
  const void* src = is_v ? a.v_new : a.k_new;
  const bool rotate = !is_v && a.rope.table != nullptr;
  uint4 out;
  if (std::is_same<Tc, Tin>::value && !rotate) {
    out = *reinterpret_cast<const uint4*>(static_cast<const Tc*>(src) + src_off);   // same type: a copy
  } else {
    float x[N];
    load_group<Tin, N>(src, src_off, x);
    if (rotate) {
      // RoPE: turn the key row by its absolute position (its write position) in float32. The
      // partners of this group's elements are the group D/2 away (style 0) or its own neighbours.
      float y[N];
      const int e0 = grp * N;
      if (a.rope.style == 0) {
        load_group<Tin, N>(src, src_off + (e0 < a.D / 2 ? a.D / 2 : -(a.D / 2)), y);
      } else {
#pragma unroll
        for (int i = 0; i < N; ++i) y[i] = x[i ^ 1];
      }
      const float2* cs = a.rope.table + static_cast<long long>(pos) * (a.D >> 1);
#pragma unroll
      for (int i = 0; i < N; ++i) {
        int pair;
        bool second;
        dev::rope_partner(e0 + i, a.D, a.rope.style, &pair, &second);
        x[i] = dev::rope_rotate(x[i], y[i], cs[pair], second);
      }
    }
    if constexpr (kFp8) {
      const float sc = is_v ? a.v_scale : a.k_scale;
#pragma unroll
      for (int i = 0; i < N; ++i) x[i] = __fdiv_rn(x[i], sc);
    }
    out = Pack<Tc>::from_f32(x);
  }
  if (dev::in_bounds(dst_row, is_v ? a.v_rows : a.k_rows, a.status)) *reinterpret_cast<uint4*>(dst) = out;
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
