// Multi-head latent attention (MLA) over the latent cache, on CUDA cores.
//
// What it computes ("KV cache, incremental decode, ...", §2.6 "The latent cache": per position one latent
// c in R^r and one shared RoPE key k^R in R^{d_R}; the attention that reads it is DeepSeek-V2's MLA in its
// absorbed form): for sequence b and query row (t, h), with q_lat the head's no-RoPE query already taken
// through its key up-projection,
//   score_j = (q_lat . c_j + q_rope . k^R_j) * scale      for keys j <= s_b + t,
//   out     = sum_j softmax_j(score) c_j                  (a latent; the value up-projection follows).
//
// How: one CTA owns (sequence, 16 query rows, key split). All heads share one latent stream, so every
// tile of keys read from memory serves all 16 rows (and, through L2, the sequence's other row tiles).
// Keys stream through two shared-memory tiles (cp.async, 16-byte pieces, zero-filled past the split);
// per tile the 256 threads compute the 16 x 32 scores (thread = key, 2 rows), fold them into running
// row maxima and sums (online softmax in base 2), and add the weighted latent rows into per-thread
// accumulators (thread = latent columns d, d + 256, ...). A unit with several splits writes (m, l, o)
// partials; the CTA that finishes its last split merges them (log-sum-exp) while they are in L2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kThreads = 256;
constexpr int kRows = kMlaRows;               // 16 query rows per CTA
constexpr int kMaxDpt = 4;                    // latent columns per thread: r <= 1024

template <typename Tc>
struct MlaCfg {
  static constexpr int E = sizeof(Tc);
  static constexpr int KT = E == 4 ? 16 : 32;           // keys per tile
  static constexpr int RPT = kRows * KT / kThreads;     // score rows per thread (1 or 2)
  static constexpr int EPC = 16 / E;                    // elements per 16-byte piece
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <typename Tc> __device__ __forceinline__ void unpack(const uint4& r, float* f);
template <> __device__ __forceinline__ void unpack<float>(const uint4& r, float* f) {
  f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y); f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
template <> __device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { f[2 * i] = __uint_as_float(w[i] << 16); f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u); }
}
template <> __device__ __forceinline__ void unpack<__half>(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = x.x; f[2 * i + 1] = x.y;
  }
}

template <typename Tc>
__global__ void __launch_bounds__(kThreads, 2)
mla_kernel(const MlaArgs a, const __grid_constant__ SplitPlan plan) {
  using C = MlaCfg<Tc>;
  constexpr int KT = C::KT, RPT = C::RPT, E = C::E, EPC = C::EPC;
  extern __shared__ __align__(16) unsigned char smem[];
  const int W = a.r + a.dR;                             // score width
  const int RS = W * E + 16;                            // key row stride (bytes): padded, conflict-free
  float* qs = reinterpret_cast<float*>(smem);           // [kRows][W] queries, prescaled
  unsigned char* ktiles = smem + kRows * W * 4;         // [2][KT][RS] keys: latent then RoPE key
  float* ps = reinterpret_cast<float*>(ktiles + 2 * KT * RS);   // [KT][kRows] scores, then weights
  float* st_m = ps + KT * kRows;                        // running row maxima (base 2)
  float* st_l = st_m + kRows;                           // running row sums
  float* st_a = st_l + kRows;                           // this tile's rescale factors
  int* last_flag = reinterpret_cast<int*>(st_a + kRows);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- which (unit = sequence x row tile, split) this CTA owns ------------------------------------
  const int item = blockIdx.x;
  int lo = 0, hi = plan.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (plan.prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int unit = lo;
  const int nsplit = plan.prefix[unit + 1] - plan.prefix[unit];
  const int split = item - plan.prefix[unit];
  const int b = plan.unit_b[unit] / plan.n_rowtiles;
  const int rt = plan.unit_b[unit] % plan.n_rowtiles;
  const int row0 = rt * kRows;
  const int nrows = min(kRows, a.T * a.H - row0);

  if (tid < kRows) { st_m[tid] = -INFINITY; st_l[tid] = 0.f; }
  pdl_wait();
  pdl_trigger();
  const int s_b = a.lens[b];                            // committed length = first query position
  const int n_eff = s_b + (row0 + nrows - 1) / a.H + 1; // keys visible to the tile's last row
  const int chunk = split_chunk(n_eff, nsplit, KT);
  const int k_begin = split * chunk;
  const int k_end = min(k_begin + chunk, n_eff);
  const int ntiles = (k_end - k_begin + KT - 1) / KT;

  // queries: row r = (t, h) with row0 + r = t * H + h, in the query type, prescaled into base-2 units
  const float qscale = a.scale * kLog2e;
  for (int i = tid; i < kRows * W; i += kThreads) {
    const int r = i / W, e = i % W;
    float x = 0.f;
    if (r < nrows) {
      const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
      const long long qrow = (static_cast<long long>(b) * a.H + h) * a.T + t;
      x = e < a.r ? load_query<Tc>(a.q_lat, a.q_dtype, qrow * a.r + e)
                  : load_query<Tc>(a.q_rope, a.q_dtype, qrow * a.dR + (e - a.r));
    }
    qs[i] = x * qscale;
  }

  const long long seq_row0 = (static_cast<long long>(a.layer) * a.B + b) * a.max_len;
  const int cpr = a.r * E / 16, kpr = a.dR * E / 16;     // 16-byte pieces per latent row, per RoPE-key row
  auto load_tile = [&](int i, int buf) {
    const int key0 = k_begin + i * KT;
    for (int j = tid; j < KT * (cpr + kpr); j += kThreads) {
      const int k = j / (cpr + kpr), c = j % (cpr + kpr);
      const int key = key0 + k;
      const bool in = key < k_end;
      const long long row = seq_row0 + (in ? key : 0);
      const unsigned char* src = c < cpr
          ? static_cast<const unsigned char*>(a.c_store) + row * a.r * E + c * 16
          : static_cast<const unsigned char*>(a.kr_store) + row * a.dR * E + (c - cpr) * 16;
      cp_async16(smem_u32(ktiles + (buf * KT + k) * RS + c * 16), src, in ? 16 : 0);   // zeros past the split
    }
    cp_async_commit();
  };

  float o[kRows][kMaxDpt];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int j = 0; j < kMaxDpt; ++j) o[r][j] = 0.f;

  if (ntiles > 0) load_tile(0, 0);
  const int kq = tid % KT, rg = tid / KT;                // score mapping: key kq, rows rg*RPT ..
  for (int i = 0; i < ntiles; ++i) {
    const int buf = i & 1;
    cp_async_wait_all();
    __syncthreads();                                    // tile i visible; every thread past tile i-1
    if (i + 1 < ntiles) load_tile(i + 1, buf ^ 1);

    // ---- scores of this tile ------------------------------------------------------------------
    const unsigned char* krow = ktiles + (buf * KT + kq) * RS;
    float acc[RPT];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) acc[rr] = 0.f;
    for (int e = 0; e < W; e += EPC) {
      float kf[EPC];
      unpack<Tc>(*reinterpret_cast<const uint4*>(krow + e * E), kf);
#pragma unroll
      for (int rr = 0; rr < RPT; ++rr) {
        const float* qr = qs + (rg * RPT + rr) * W + e;
#pragma unroll
        for (int j = 0; j < EPC; ++j) acc[rr] = fmaf(qr[j], kf[j], acc[rr]);
      }
    }
    const int key = k_begin + i * KT + kq;
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
      const int row = rg * RPT + rr;
      const bool vis = row < nrows && key < k_end && key <= s_b + (row0 + row) / a.H;
      ps[kq * kRows + row] = vis ? acc[rr] : -INFINITY;
    }
    __syncthreads();

    // ---- online softmax: warp w owns rows 2w, 2w+1; lanes over the tile's keys ------------------
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = 2 * warp + rr;
      const float x = lane < KT ? ps[lane * kRows + row] : -INFINITY;
      float tmax = x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float m_old = st_m[row];
      const float m_new = fmaxf(m_old, tmax);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
      const float p = (m_new == -INFINITY || x == -INFINITY) ? 0.f : exp2f(x - m_new);
      if (lane < KT) ps[lane * kRows + row] = p;
      float psum = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      __syncwarp();
      if (lane == 0) {
        st_l[row] = st_l[row] * alpha + psum;
        st_m[row] = m_new;
        st_a[row] = alpha;
      }
    }
    __syncthreads();

    // ---- o = o * alpha + P . C_tile: thread owns latent columns tid, tid + 256, ... ----------------
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float al = st_a[r];
#pragma unroll
      for (int j = 0; j < kMaxDpt; ++j) o[r][j] *= al;
    }
    const unsigned char* ctile = ktiles + buf * KT * RS;
#pragma unroll 2
    for (int k = 0; k < KT; ++k) {
      float cv[kMaxDpt];
#pragma unroll
      for (int j = 0; j < kMaxDpt; ++j) {
        const int d = tid + j * kThreads;
        cv[j] = d < a.r ? to_f32<Tc>(*reinterpret_cast<const Tc*>(ctile + k * RS + d * E)) : 0.f;
      }
      const float4* pr = reinterpret_cast<const float4*>(ps + k * kRows);
#pragma unroll
      for (int r4 = 0; r4 < kRows / 4; ++r4) {
        const float4 p = pr[r4];
#pragma unroll
        for (int j = 0; j < kMaxDpt; ++j) {
          o[4 * r4][j] = fmaf(p.x, cv[j], o[4 * r4][j]);
          o[4 * r4 + 1][j] = fmaf(p.y, cv[j], o[4 * r4 + 1][j]);
          o[4 * r4 + 2][j] = fmaf(p.z, cv[j], o[4 * r4 + 2][j]);
          o[4 * r4 + 3][j] = fmaf(p.w, cv[j], o[4 * r4 + 3][j]);
        }
      }
    }
  }
  __syncthreads();

  // ---- write: the output, or this split's partials --------------------------------------------------
  const long long item_row0 = static_cast<long long>(item) * kRows;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (r >= nrows) continue;
    const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
    const long long orow = ((static_cast<long long>(b) * a.H + h) * a.T + t) * a.r;
#pragma unroll
    for (int j = 0; j < kMaxDpt; ++j) {
      const int d = tid + j * kThreads;
      if (d >= a.r) continue;
      if (nsplit == 1) put_out(a, orow + d, o[r][j] / st_l[r]);
      else put_part_o(a, (item_row0 + r) * a.r + d, o[r][j]);
    }
    if (nsplit > 1 && tid == 0) {
      put_part_ml(a, (item_row0 + r) * 2, st_m[r]);
      put_part_ml(a, (item_row0 + r) * 2 + 1, st_l[r]);
    }
  }
  if (nsplit == 1) return;

  // ---- the CTA that finishes a unit's last split merges its partials (log-sum-exp) ----------------
  __threadfence();
  __syncthreads();
  int* counter = a.counters + unit;
  if (tid == 0) *last_flag = (atomicAdd(counter, 1) == nsplit - 1);
  __syncthreads();
  if (!*last_flag) return;
  __threadfence();
  const long long first_row = static_cast<long long>(plan.prefix[unit]) * kRows;
  for (int i = tid; i < nrows * a.r; i += kThreads) {
    const int r = i / a.r, d = i % a.r;
    float m = -INFINITY, l = 0.f, acc = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const long long row = first_row + static_cast<long long>(sp) * kRows + r;
      const float ms = __ldcg(a.part_ml + row * 2), ls = __ldcg(a.part_ml + row * 2 + 1);
      if (!(ls > 0.f)) continue;                         // a split that sees no key of this row
      const float mn = fmaxf(m, ms);
      const float c_old = exp2f(m - mn), c_new = exp2f(ms - mn);
      l = l * c_old + ls * c_new;
      acc = acc * c_old + __ldcg(a.part_o + row * a.r + d) * c_new;
      m = mn;
    }
    const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
    put_out(a, ((static_cast<long long>(b) * a.H + h) * a.T + t) * a.r + d, acc / l);
  }
  if (tid == 0) *counter = 0;
}

template <typename Tc>
cudaError_t run(const MlaArgs& a, const SplitPlan& p, cudaStream_t st) {
  const size_t smem = mla_smem_bytes(a.cache_dtype, a.r, a.dR);
  cudaError_t e = ensure_smem_limit<mla_kernel<Tc>>(227 * 1024);
  if (e != cudaSuccess) return e;
  return launch_pdl(mla_kernel<Tc>, dim3(p.n_items), dim3(kThreads), smem, st, a, p);
}

}  // namespace

int mla_tile_keys(kvc_dtype dt) { return dt == KVC_F32 ? MlaCfg<float>::KT : MlaCfg<__half>::KT; }

size_t mla_smem_bytes(kvc_dtype dt, int r, int dR) {
  const int e = itemsize(dt), kt = mla_tile_keys(dt), W = r + dR;
  return static_cast<size_t>(kRows) * W * 4 + 2ull * kt * (W * e + 16) + static_cast<size_t>(kt) * kRows * 4 +
         3 * kRows * 4 + 16;
}

cudaError_t launch_mla(const MlaArgs& a, const SplitPlan& p, cudaStream_t st) {
  switch (a.cache_dtype) {
    case KVC_F32: return run<float>(a, p, st);
    case KVC_F16: return run<__half>(a, p, st);
    case KVC_BF16: return run<__nv_bfloat16>(a, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvc
