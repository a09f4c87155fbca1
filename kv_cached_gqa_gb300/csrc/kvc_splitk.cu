// Split-K grouped-query attention over the KV cache on CUDA cores (decode T = 1 and short chunks).
//
// What it computes ("KV cache, incremental decode, ...", §2.3; "Generation and the KV Cache",
// fence 3; "Heads, GQA and K/V cache", "Four queries, two sets of K/V"): for sequence b, K/V head
// g and the G query heads h = g*G .. g*G+G-1 that share it, every query row (t, h) of the chunk
// attends over stored keys j <= s_b + t with weights softmax_j(q . k_j / sqrt(d_h)), summing v_j.
//
// How (GB300): the query rows of one K/V head are packed together ("row tile": rows r = t*G + g),
// so each K/V tile read from HBM serves the whole group; K/V are never repeated per query head.
// One CTA handles one (row tile, K/V head, key split). A producer warp streams the split's K tiles
// and then its V tiles, HBM -> shared memory, with TMA (128-byte swizzle, so lane-per-key reads
// are bank-conflict free) through a 4-stage mbarrier ring; four consumer warps compute.
//   QK:  a key's row is split over 1-8 lanes (4 x 16 bytes each), every lane scores 2 keys, so a
//        query chunk broadcast from shared memory serves both; paired fp32 FMAs (fma.rn.f32x2);
//        scores for the whole split are kept in shared memory;
//   softmax: exact within the split (max, exp2, sum), no running rescale; each weight is stored
//        twice so PV reads ready-made pairs;
//   PV:  one lane per d_h slice, paired FMAs over d, warps split the keys and are reduced through
//        shared memory at the end.
// A split writes (m, l, o) partials unless it is its unit's only split, in which case it writes
// the normalised output. The CTA that finishes a unit's last split merges the partials with the
// log-sum-exp rule (a per-unit counter in global memory tells it that it is last), so there is
// no second launch.
//
// Every wait is bounded (about one second); a wait that gives up sets the device status word and
// the CTA skips its remaining work instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kStages = 4;
constexpr int kTileBytes = 16384;
constexpr int kScoreFloats = 8192;             // per-split weights: keys x rows x 2 (duplicated)

template <typename Tc, int D, int RMAX>
struct Cfg {
  static constexpr int E = sizeof(Tc);
  static constexpr int ROWB = D * E;                    // bytes per key row
  static constexpr int SW = ROWB >= 128 ? 128 : 64;     // swizzle span (bytes) = TMA box row
  static constexpr int CPB = SW / 16;                   // 16-byte chunks per box row
  static constexpr int NBOX = ROWB / SW;                // boxes per key row
  static constexpr int BOX_INNER = SW / E;              // elements per box row
  static constexpr int TILE = kTileBytes / ROWB;        // keys per tile
  static constexpr int EPC = 16 / E;                    // elements per 16-byte chunk
  static constexpr int CPR = ROWB / 16;                 // chunks per key row
  // QK: a key's row is split over DSPLIT lanes, 4 chunks each; every lane handles KPT keys, so a
  // query chunk read from shared memory serves KPT keys
  static constexpr int CPL = CPR >= 4 ? 4 : CPR;        // chunks per lane
  static constexpr int DSPLIT = CPR / CPL;              // lanes per key
  static constexpr int KPW = 32 / DSPLIT;               // keys per warp per pass
  static constexpr int KPC = kConsumerWarps * KPW;      // keys per CTA pass
  static constexpr int KPT = TILE / KPC;                // keys per lane per tile
  static constexpr int DPART = D / DSPLIT;              // elements per lane part
  static constexpr int QSTRIDE = D + 4 * DSPLIT;        // padded q row (floats) in shared memory
  static constexpr int EPL = D / 32;                    // V elements per lane in PV
  static_assert(TILE <= 256 && TILE % kConsumerWarps == 0, "tile");
  static_assert(KPT >= 1 && KPT * KPC == TILE, "keys per lane");
  static_assert(RMAX % 4 == 0, "row blocks of 4");
};

struct __align__(8) Smem {
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  int abort;
  int last;
  float m[16];
  float l[16];
};

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" :: "n"(kConsumers) : "memory");
}

// Byte offset, inside one tile, of 16-byte chunk `chunk` of key row `key` (TMA swizzle layout).
template <class C>
__device__ __forceinline__ uint32_t tile_off(int key, int chunk) {
  const int box = chunk / C::CPB, cc = chunk % C::CPB;
  const int sw = (C::SW == 128) ? (key & 7) : ((key >> 1) & 3);
  return box * (C::TILE * C::SW) + key * C::SW + ((cc ^ sw) << 4);
}

// 16 bytes of stored elements -> floats
template <typename Tc> __device__ __forceinline__ void unpack16(const uint4& r, float* f);
template <> __device__ __forceinline__ void unpack16<float>(const uint4& r, float* f) {
  f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
  f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
template <> __device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <> __device__ __forceinline__ void unpack16<fp8>(const uint4& r, float* f) {   // 16 E4M3 codes
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 lo = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xffffu), __NV_E4M3)));
    const float2 hi = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3)));
    f[4 * i] = lo.x; f[4 * i + 1] = lo.y; f[4 * i + 2] = hi.x; f[4 * i + 3] = hi.y;
  }
}
template <> __device__ __forceinline__ void unpack16<__half>(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 x = __half22float2(h);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

// V elements [lane*EPL, lane*EPL + EPL) of key row `key` in a V tile.
template <typename Tc, class C>
__device__ __forceinline__ void load_v(const unsigned char* tile, int key, int lane, float* v) {
  constexpr int BYTES = C::EPL * C::E;                  // bytes per lane: 2, 4, 8 or 16
  const int byte0 = lane * BYTES;
  const unsigned char* p = tile + tile_off<C>(key, byte0 >> 4) + (byte0 & 15);
  if constexpr (sizeof(Tc) == 1) {                     // fp8: 2 or 4 codes
#pragma unroll
    for (int i = 0; i < BYTES; i += 2) {
      const float2 x = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(
          *reinterpret_cast<const __nv_fp8x2_storage_t*>(p + i), __NV_E4M3)));
      v[i] = x.x;
      v[i + 1] = x.y;
    }
  } else if constexpr (BYTES == 16) {
    unpack16<Tc>(*reinterpret_cast<const uint4*>(p), v);
  } else if constexpr (BYTES == 8) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    if constexpr (sizeof(Tc) == 4) {
      v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
    } else {
      uint4 r4 = make_uint4(r.x, r.y, 0, 0);
      float f[8];
      unpack16<Tc>(r4, f);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = f[i];
    }
  } else if constexpr (BYTES == 4) {
    const uint32_t r = *reinterpret_cast<const uint32_t*>(p);
    if constexpr (sizeof(Tc) == 4) {
      v[0] = __uint_as_float(r);
    } else {
      uint4 r4 = make_uint4(r, 0, 0, 0);
      float f[8];
      unpack16<Tc>(r4, f);
      v[0] = f[0]; v[1] = f[1];
    }
  } else {
    v[0] = to_f32<Tc>(*reinterpret_cast<const Tc*>(p));
  }
}

// Two fp32 multiply-adds in one instruction: (c0, c1) += (a0, a1) * (b0, b1).
__device__ __forceinline__ void ffma2(float& c0, float& c1, float a0, float a1, float b0, float b1) {
  const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), make_float2(c0, c1));
  c0 = r.x;
  c1 = r.y;
}

template <typename Tc, int D, int RMAX>
__global__ void __launch_bounds__(kThreads, 2)
splitk_kernel(const AttnArgs a, const __grid_constant__ SplitPlan plan,
              const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using C = Cfg<Tc, D, RMAX>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // layout: [stages x 16 KB tiles][weights: keys x RMAX x 2][q rows][Smem]
  unsigned char* tiles = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* SP = reinterpret_cast<float*>(tiles + kStages * kTileBytes);
  float* qs = SP + kScoreFloats;
  Smem* sm = reinterpret_cast<Smem*>(qs + RMAX * C::QSTRIDE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which (unit, K/V head, split) this CTA owns --------------------------------------------
  const int item = blockIdx.x;
  int lo = 0, hi = plan.n_units - 1;
  while (lo < hi) {                        // last unit u with prefix[u] <= item
    const int mid = (lo + hi + 1) >> 1;
    if (plan.prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int unit = lo;
  const int nsplit = (plan.prefix[unit + 1] - plan.prefix[unit]) / a.H_kv;
  const int rem = item - plan.prefix[unit];
  const int kvh = rem / nsplit, split = rem % nsplit;
  const int b = plan.unit_b[unit] / plan.n_rowtiles;
  const int rt = plan.unit_b[unit] % plan.n_rowtiles;
  const int R = a.T * a.G;                              // query rows of this K/V head
  const int row0 = rt * RMAX;
  const int nrows = min(RMAX, R - row0);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), kConsumerWarps);
    }
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // from here on the lengths and the queries, which earlier kernels write, are read
  pdl_wait();
  pdl_trigger();
  const int s_b = a.lens[b] + a.delta - a.T;            // committed length = first query position
  const int t_max = (row0 + nrows - 1) / a.G;
  const int n_eff = s_b + t_max + 1;                    // keys visible to the tile's last row
  const int chunk = split_chunk(n_eff, nsplit, C::TILE);  // near-equal, whole-tile splits of the unit's keys
  const int k_begin = split * chunk;
  const int k_end = min(k_begin + chunk, n_eff);
  const int n_keys = k_end - k_begin;
  const int nkt = (n_keys + C::TILE - 1) / C::TILE;
  // queries of the tile, prescaled by log2(e) / sqrt(d_h): scores are in base-2 units
  const float qscale = kLog2e * rsqrtf(static_cast<float>(D)) * a.k_scale;   // k_scale: fp8 codes -> keys
  for (int i = tid; i < RMAX * D; i += kThreads) {
    const int r = i / D, e = i % D;
    float x = 0.f;
    if (r < nrows) {
      const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
      const long long qrow = ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * D;
      x = load_query_rot<Tc>(a, qrow, e, s_b + t) * qscale;
    }
    qs[r * C::QSTRIDE + e + (e / C::DPART) * 4] = x;
  }
  __syncthreads();

  volatile int* abort_flag = &sm->abort;

  if (warp == kConsumerWarps) {
    // ---------------------------------- producer ------------------------------------------
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    for (int i = 0; i < 2 * nkt; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      const bool isv = i >= nkt;
      const int y = k_begin + (isv ? i - nkt : i) * C::TILE;
      const TilePiece pc = tile_piece<C::TILE>(a, b, kvh, y, lane);   // a block-table read overlaps the wait
      const uint32_t full = smem_u32(&sm->full[st]);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&sm->empty[st]), ph ^ 1, abort_flag);
        if (ok) mbar_expect_tx(full, kTileBytes);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue_piece<C::TILE, C::NBOX, C::SW, C::BOX_INNER>(pc, isv ? &tv : &tk, smem_u32(tiles + st * kTileBytes), full,
                                                       lane);
    }
    return;
  }

  // ---------------------------------- consumers: QK ------------------------------------------
  // lane = (part, key): `part` owns CPL chunks of the row; each lane scores KPT keys of the tile
  const int part = lane / C::KPW;
  const int key_in_warp = lane % C::KPW;
  for (int i = 0; i < nkt; ++i) {
    const int st = i % kStages;
    const bool ok = mbar_wait(smem_u32(&sm->full[st]), (i / kStages) & 1, abort_flag);
    if (ok) {
      const unsigned char* tile = tiles + st * kTileBytes;
#pragma unroll
      for (int rb = 0; rb < RMAX / 4; ++rb) {
        float acc[C::KPT][4][2];
#pragma unroll
        for (int kp = 0; kp < C::KPT; ++kp)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[kp][j][0] = acc[kp][j][1] = 0.f;
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) {
          float kf[C::KPT][C::EPC];
#pragma unroll
          for (int kp = 0; kp < C::KPT; ++kp) {
            const int key = kp * C::KPC + warp * C::KPW + key_in_warp;
            unpack16<Tc>(*reinterpret_cast<const uint4*>(tile + tile_off<C>(key, part * C::CPL + c)), kf[kp]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float* qr = qs + (rb * 4 + j) * C::QSTRIDE + part * (C::DPART + 4) + c * C::EPC;
#pragma unroll
            for (int e4 = 0; e4 < C::EPC; e4 += 4) {
              const float4 qv = *reinterpret_cast<const float4*>(qr + e4);
#pragma unroll
              for (int kp = 0; kp < C::KPT; ++kp) {
                ffma2(acc[kp][j][0], acc[kp][j][1], qv.x, qv.y, kf[kp][e4], kf[kp][e4 + 1]);
                ffma2(acc[kp][j][0], acc[kp][j][1], qv.z, qv.w, kf[kp][e4 + 2], kf[kp][e4 + 3]);
              }
            }
          }
        }
#pragma unroll
        for (int kp = 0; kp < C::KPT; ++kp) {
          const int key = kp * C::KPC + warp * C::KPW + key_in_warp;
          const int kabs = k_begin + i * C::TILE + key;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float sc = acc[kp][j][0] + acc[kp][j][1];
#pragma unroll
            for (int o = C::KPW; o < 32; o <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
            if (part == 0) {
              const int r = rb * 4 + j;
              const int t = (row0 + r) / a.G;
              const bool vis = kabs < k_end && kabs <= s_b + t;
              SP[((i * C::TILE + key) * RMAX + r) * 2] = vis ? sc : -INFINITY;
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm->empty[st]));
  }
  consumers_sync();

  // ---------------------------------- softmax within the split ---------------------------------
  // exact over the split's keys; each weight is stored twice so PV reads ready-made pairs
  const int n_slots = nkt * C::TILE;
  for (int r = warp; r < RMAX; r += kConsumerWarps) {
    float m = -INFINITY;
    for (int k = lane; k < n_slots; k += 32) m = fmaxf(m, SP[(k * RMAX + r) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int k = lane; k < n_slots; k += 32) {
      float* slot = SP + (k * RMAX + r) * 2;
      const float p = (m == -INFINITY) ? 0.f : exp2f(slot[0] - m);
      slot[0] = p;
      slot[1] = p;
      l += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) { sm->m[r] = m; sm->l[r] = l; }
  }
  consumers_sync();

  // ---------------------------------- consumers: PV ------------------------------------------
  constexpr int EPL = C::EPL;
  constexpr int NP = EPL >= 2 ? EPL / 2 : 1;
  float acc[RMAX][NP][2];
#pragma unroll
  for (int r = 0; r < RMAX; ++r)
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[r][e][0] = acc[r][e][1] = 0.f;
  constexpr int KPWV = C::TILE / kConsumerWarps;       // keys per warp per tile
  for (int i = 0; i < nkt; ++i) {
    const int ti = nkt + i;
    const int st = ti % kStages;
    const bool ok = mbar_wait(smem_u32(&sm->full[st]), (ti / kStages) & 1, abort_flag);
    if (ok) {
      const unsigned char* tile = tiles + st * kTileBytes;
#pragma unroll 4
      for (int kk = 0; kk < KPWV; ++kk) {
        const int key = warp * KPWV + kk;
        float v[EPL];
        load_v<Tc, C>(tile, key, lane, v);
        const float4* pr = reinterpret_cast<const float4*>(SP + (i * C::TILE + key) * RMAX * 2);
#pragma unroll
        for (int r2 = 0; r2 < RMAX / 2; ++r2) {
          const float4 p = pr[r2];                       // (p_r, p_r, p_r+1, p_r+1)
          if constexpr (EPL >= 2) {
#pragma unroll
            for (int e = 0; e < NP; ++e) {
              ffma2(acc[2 * r2][e][0], acc[2 * r2][e][1], p.x, p.y, v[2 * e], v[2 * e + 1]);
              ffma2(acc[2 * r2 + 1][e][0], acc[2 * r2 + 1][e][1], p.z, p.w, v[2 * e], v[2 * e + 1]);
            }
          } else {
            acc[2 * r2][0][0] = fmaf(p.x, v[0], acc[2 * r2][0][0]);
            acc[2 * r2 + 1][0][0] = fmaf(p.z, v[0], acc[2 * r2 + 1][0][0]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm->empty[st]));
  }
  consumers_sync();                                      // every tile consumed: ring is free

  // ---------------------------------- reduce warps, write ------------------------------------
  float* red = reinterpret_cast<float*>(tiles);          // [warps][RMAX][D]
#pragma unroll
  for (int r = 0; r < RMAX; ++r)
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      red[(warp * RMAX + r) * D + lane * EPL + e] = EPL >= 2 ? acc[r][e / 2][e % 2] : acc[r][0][0];
  consumers_sync();
  const bool aborted = *abort_flag != 0;
  if (aborted && tid == 0) atomicExch(a.status, kStatusTimeout);
  const long long item_row0 = static_cast<long long>(item) * RMAX;
  for (int i = tid; i < nrows * D; i += kConsumers) {
    const int r = i / D, d = i % D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) o += red[(w * RMAX + r) * D + d];
    if (aborted) continue;
    if (nsplit == 1) {
      const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
      put_out(a, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * D + d, o / sm->l[r] * a.v_scale);
    } else {
      put_part_o(a, (item_row0 + r) * D + d, o);
      if (d == 0) {
        put_part_ml(a, (item_row0 + r) * 2, sm->m[r]);
        put_part_ml(a, (item_row0 + r) * 2 + 1, sm->l[r]);
      }
    }
  }
  if (nsplit == 1) return;

  // ---------------------------------- the last split merges ----------------------------------
  // o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s over this unit's splits, by the CTA that
  // finishes last; the partials are still in L2. The counter is reset for the next launch.
  __threadfence();
  consumers_sync();
  int* counter = a.counters + unit * a.H_kv + kvh;
  if (tid == 0) sm->last = (atomicAdd(counter, 1) == nsplit - 1);
  consumers_sync();
  if (!sm->last) return;
  __threadfence();
  const long long first_row = static_cast<long long>(plan.prefix[unit] + kvh * nsplit) * RMAX;
  for (int i = tid; i < nrows * D; i += kConsumers) {
    const int r = i / D, d = i % D;
    float m = -INFINITY, l = 0.f, o = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const long long row = first_row + static_cast<long long>(s) * RMAX + r;
      const float ms = __ldcg(a.part_ml + row * 2), ls = __ldcg(a.part_ml + row * 2 + 1);
      if (!(ls > 0.f)) continue;                         // a split that sees no key of this row
      const float mn = fmaxf(m, ms);
      const float c_old = exp2f(m - mn), c_new = exp2f(ms - mn);
      l = l * c_old + ls * c_new;
      o = o * c_old + __ldcg(a.part_o + row * D + d) * c_new;
      m = mn;
    }
    const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
    if (!aborted) put_out(a, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * D + d, o / l * a.v_scale);
  }
  if (tid == 0) *counter = 0;
}

template <typename Tc, int D, int RMAX>
size_t smem_bytes() {
  using C = Cfg<Tc, D, RMAX>;
  return 1024 + kStages * kTileBytes + kScoreFloats * 4 + RMAX * C::QSTRIDE * 4 + sizeof(Smem);
}

template <typename Tc, int D, int RMAX>
cudaError_t run(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk, const CUtensorMap* tv,
                cudaStream_t st) {
  const size_t smem = smem_bytes<Tc, D, RMAX>();
  auto kern = splitk_kernel<Tc, D, RMAX>;
  cudaError_t e = ensure_smem_limit<splitk_kernel<Tc, D, RMAX>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.n_items), dim3(kThreads), smem, st, a, p, *tk, *tv);
}

template <typename Tc, int D>
cudaError_t run_rows(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                     const CUtensorMap* tv, cudaStream_t st) {
  switch (p.rows_per_tile) {
    case 4: return run<Tc, D, 4>(a, p, tk, tv, st);
    case 8: return run<Tc, D, 8>(a, p, tk, tv, st);
    case 16: return run<Tc, D, 16>(a, p, tk, tv, st);
  }
  return cudaErrorInvalidValue;
}

template <typename Tc>
cudaError_t run_d(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk, const CUtensorMap* tv,
                  cudaStream_t st) {
  switch (a.D) {
    case 32:
      if constexpr (sizeof(Tc) > 1) return run_rows<Tc, 32>(a, p, tk, tv, st);   // fp8 rows need >= 64 B
      return cudaErrorInvalidValue;
    case 64: return run_rows<Tc, 64>(a, p, tk, tv, st);
    case 128: return run_rows<Tc, 128>(a, p, tk, tv, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool splitk_shape(kvc_dtype dt, int D, int rows, int* rows_per_tile, int* tile_keys) {
  if (D != 32 && D != 64 && D != 128) return false;
  if (dt == KVC_FP8_E4M3 && D == 32) return false;
  *rows_per_tile = rows <= 4 ? 4 : rows <= 8 ? 8 : 16;
  *tile_keys = kTileBytes / (D * itemsize(dt));
  return true;
}

size_t splitk_workspace_floats(const SplitPlan& p, int D) {
  return static_cast<size_t>(p.n_items) * p.rows_per_tile * (D + 2);
}

cudaError_t launch_splitk(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                          const CUtensorMap* tv, cudaStream_t st) {
  switch (a.cache_dtype) {
    case KVC_F32: return run_d<float>(a, p, tk, tv, st);
    case KVC_F16: return run_d<__half>(a, p, tk, tv, st);
    case KVC_BF16: return run_d<__nv_bfloat16>(a, p, tk, tv, st);
    case KVC_FP8_E4M3: return run_d<fp8>(a, p, tk, tv, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvc
