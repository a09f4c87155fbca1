// The append's per-element work, shared by the append kernel and the decode kernel's fused append:
// one 16-byte group of stored elements of one K or V row, rounded (and for keys rotated) exactly as the
// append kernel stores it. See kvc_append.cu for what the append computes and its sources.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace app {

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

// Group `grp` (N = Pack<Tc>::N elements) of chunk row `row` = (b * H + h) * T + t of the first store
// (K, or the latent) or, with is_v, of the second, written at position lens[b] + delta + t of (layer,
// b, h). Tc is the storage type, Tin the input type (float32, the storage type itself, or a 16-bit type
// for fp8).
template <typename Tc, typename Tin>
__device__ __forceinline__ void append_group(const AppendArgs& a, long long row, int grp, bool is_v) {
  constexpr int N = Pack<Tc>::N;
  constexpr bool kFp8 = std::is_same<Tc, dev::fp8>::value;
  const int W = is_v ? a.Dv : a.D;                      // this store's row width
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

// append_group with the input type chosen at run time (a.in_dtype).
template <typename Tc>
__device__ __forceinline__ void append_group_any(const AppendArgs& a, long long row, int grp, bool is_v) {
  if (a.in_dtype == KVC_F32) {
    append_group<Tc, float>(a, row, grp, is_v);
  } else if constexpr (std::is_same<Tc, dev::fp8>::value) {
    if (a.in_dtype == KVC_F16) append_group<Tc, __half>(a, row, grp, is_v);
    else append_group<Tc, __nv_bfloat16>(a, row, grp, is_v);
  } else {
    append_group<Tc, Tc>(a, row, grp, is_v);
  }
}

}  // namespace app
}  // namespace kvc
