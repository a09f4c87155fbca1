// Multi-head latent attention over the latent cache on the 5th-generation tensor cores (tcgen05 + TMEM),
// for 16-bit latent caches with r = 256 or 512 and a 64-wide RoPE key.
//
// What it computes ("KV cache, incremental decode, ...", §2.6 "The latent cache"; DeepSeek-V2's MLA in
// absorbed form): for sequence b and query row (t, h), over keys j <= s_b + t,
//   score_j = (q_lat . c_j + q_rope . k^R_j) * scale,   out = sum_j softmax_j(score) c_j.
//
// How: 16 query rows of one sequence are the N dimension; 64-key tiles are M:
//   S^T [64 keys x 16 rows]   = [C | K^R]_tile . Q^T      A = key tile (K-major, 576 wide), B = Q^T
//   O^T [r x 16 rows]        += C_tile^T . P^T            A = latent tile read MN-major (r / 128 blocks
//                                                           of 128 latent columns), B = P^T
// so each tile read from memory serves every query row of the CTA and the latent is both key and value.
// One CTA per (sequence, 16-row tile, key split); one CTA per SM (a 72 KB tile per stage):
//   warp 0     TMA: per tile 8 (or 4) 64 x 64 latent boxes and one RoPE-key box, through a 2-stage ring;
//   warp 1     owns TMEM and issues every MMA from one thread, QK(j + 1) before PV(j);
//   warps 2-5  softmax: lanes 0-15 of warp quadrant q hold keys 16q .. 16q + 15 of a tile (the TMEM
//              layout of an M = 64 result); the tile maximum of each row is reduced across the four
//              warps, and the output in TMEM is rescaled only when a row's maximum passes its
//              reference by more than 8 (online softmax with a lazy reference, as in the chunk kernel);
//              P^T goes to shared memory as a hi + lo pair of 16-bit values; the epilogue (thread =
//              latent column) divides by the row sums.
// A unit with several splits writes (m, l, o) partials; the CTA that finishes its last split merges
// them. Every wait is bounded (~1 s) and reported through the device status word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kKT = 64;                       // keys per tile (MMA M of QK, K of PV)
constexpr int kNR = 16;                       // query rows per CTA (MMA N)
constexpr int kDR = 64;                       // RoPE-key width
constexpr int kBox = kKT * 128;               // one 64-element (128-byte) swizzled box of a tile: 8 KB
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kTmemCols = 128;
constexpr int kStages = 2;
constexpr int kMergeSplits = 31;

template <int R>
struct MLayout {
  static constexpr int kCBoxes = R / 64;                        // latent boxes per tile
  static constexpr int kBoxes = kCBoxes + kDR / 64;             // plus the RoPE-key box
  static constexpr int kStageBytes = kBoxes * kBox;
  static constexpr int kQAtoms = (R + kDR) / 64;
  static constexpr int kQBytes = kQAtoms * kNR * 128;           // Q^T: atoms of 16 rows x 128 B
  static constexpr int kPBytes = kNR * 128;                     // one P^T operand (16 rows x 64 keys)
  static constexpr int kOBlocks = R / 128;                      // O^T blocks of 128 latent columns
  static constexpr int kStageOff = 0;
  static constexpr int kQOff = kStages * kStageBytes;
  static constexpr int kPOff = kQOff + kQBytes;                 // 2 buffers x (hi, lo)
  static constexpr int kCtlOff = kPOff + 4 * kPBytes;
};

struct __align__(8) MCtl {
  unsigned long long full[kStages], empty[kStages];
  unsigned long long s_full[2], s_free[2], p_full[2], p_free[2];
  unsigned long long o_full, done;
  uint32_t tmem;
  int abort, last;
  float red[2][4][kNR];                       // per-warp tile maxima (double-buffered by tile parity)
  float lsum[4][kNR];
  float m[kNR], l[kNR];
};

template <int R>
constexpr size_t mla_tc_smem() { return 1024 + MLayout<R>::kCtlOff + sizeof(MCtl); }
// A CTA holds 128 TMEM columns, so the up to two CTAs that share an SM (r = 256) never wait on
// tcgen05.alloc; r = 512 takes more than half the shared memory, one CTA per SM.
static_assert(mla_tc_smem<512>() <= 227 * 1024 && mla_tc_smem<256>() <= 227 * 1024, "shared memory");
static_assert(4 * kTmemCols <= 512, "TMEM columns for every CTA that fits an SM");
static_assert((2 * kNR * kMergeSplits + kNR) * 4 <= 4 * MLayout<256>::kPBytes, "merge scratch fits the P buffers");

// Byte offset of element (row, col) of a [rows][cols] 16-bit matrix stored as 128-byte-swizzled atoms of
// 64 columns (K-major operand layout).
__device__ __forceinline__ uint32_t sw128(int rows, int row, int col) {
  const int atom = col >> 6, c = col & 63;
  return atom * (rows * 128) + row * 128 + ((((c >> 3) ^ (row & 7))) << 4) + (c & 7) * 2;
}

__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  while (!mbar_try(bar, parity)) {
    if (now_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
         "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
      : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename Tc, int R>
__global__ void __launch_bounds__(kThreads, 1)
mla_tc_kernel(const MlaArgs a, const __grid_constant__ SplitPlan plan,
              const __grid_constant__ CUtensorMap tc, const __grid_constant__ CUtensorMap tr) {
  using Lo = MLayout<R>;
  constexpr uint32_t kFmt = std::is_same<Tc, __nv_bfloat16>::value ? 1u : 0u;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MCtl* ctl = reinterpret_cast<MCtl*>(sm + Lo::kCtlOff);
  const uint32_t s_stage = smem_u32(sm + Lo::kStageOff);
  const uint32_t s_q = smem_u32(sm + Lo::kQOff);
  unsigned char* p_base = sm + Lo::kPOff;
  const uint32_t s_p = smem_u32(p_base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

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
  const int row0 = rt * kNR;
  const int nrows = min(kNR, a.T * a.H - row0);
  const int plane = a.layer * a.B + b;

  // ---- set-up: TMEM, barriers --------------------------------------------------------------------
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&ctl->tmem));
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->s_full[s]), 1);
      mbar_init(smem_u32(&ctl->s_free[s]), kSoftmaxThreads / 32);
      mbar_init(smem_u32(&ctl->p_full[s]), kSoftmaxThreads / 32);
      mbar_init(smem_u32(&ctl->p_free[s]), 1);
    }
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();
  const int s_b = a.lens[b];
  const int n_eff = s_b + (row0 + nrows - 1) / a.H + 1;
  const int chunk = split_chunk(n_eff, nsplit, kKT);
  const int k_begin = split * chunk;
  const int k_end = min(k_begin + chunk, n_eff);
  const int nkt = (k_end - k_begin + kKT - 1) / kKT;
  // Q^T: 16 rows x (r + 64) in the cache dtype, 128-byte swizzled (rows past the chunk are zero). Four
  // elements per load, every load of a thread issued before the first store: the latencies overlap.
  {
    constexpr int kW = R + kDR, kQuads = kNR * kW / 4, kIter = (kQuads + kThreads - 1) / kThreads;
    uint4 x[kIter];
#pragma unroll
    for (int k = 0; k < kIter; ++k) {
      const int i = tid + k * kThreads, r = (4 * i) / kW, d = (4 * i) % kW;
      x[k] = make_uint4(0u, 0u, 0u, 0u);
      if (i < kQuads && r < nrows) {
        const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
        const long long qrow = (static_cast<long long>(b) * a.H + h) * a.T + t;
        x[k] = d < R ? load_query4_raw<Tc>(a.q_lat, a.q_dtype, qrow * R + d)
                     : load_query4_raw<Tc>(a.q_rope, a.q_dtype, qrow * kDR + (d - R));
      }
    }
#pragma unroll
    for (int k = 0; k < kIter; ++k) {
      const int i = tid + k * kThreads, r = (4 * i) / kW, d = (4 * i) % kW;
      if (i < kQuads) *reinterpret_cast<uint2*>(sm + Lo::kQOff + sw128(kNR, r, d)) = query4_to<Tc, Tc>(x[k], a.q_dtype);
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;                    // S^T buffers at columns 0, 16; O^T from column 32
  const uint32_t tmem_o = tmem + 2 * kNR;
  volatile int* abort_flag = &ctl->abort;

  if (warp == 0) {
    // ---------------------------------- TMA producer ----------------------------------------------
    if (lane == 0) {
      prefetch_tmap(&tc);
      prefetch_tmap(&tr);
      int issued = 0;
      for (int j = 0; j < nkt; ++j) {
        const int st = j % kStages;
        if (!mbar_wait(smem_u32(&ctl->empty[st]), ((j / kStages) & 1) ^ 1, abort_flag)) break;
        const uint32_t full = smem_u32(&ctl->full[st]);
        mbar_expect_tx(full, Lo::kStageBytes);
        const uint32_t dst = s_stage + st * Lo::kStageBytes;
        const int y = k_begin + j * kKT;
#pragma unroll
        for (int bx = 0; bx < Lo::kCBoxes; ++bx) tma_load_3d(dst + bx * kBox, &tc, 64 * bx, y, plane, full);
        tma_load_3d(dst + Lo::kCBoxes * kBox, &tr, 0, y, plane, full);
        issued = j + 1;
      }
      for (int j = max(0, issued - kStages); j < issued; ++j)
        mbar_drain(smem_u32(&ctl->full[j % kStages]), (j / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------- MMA issuer -------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc(kKT, kNR, kFmt, 0, 0);
      const uint32_t idesc_o = umma_idesc(128, kNR, kFmt, 1, 0);
      bool ok = true;
      auto issue_qk = [&](int j) -> bool {                 // S^T_j = [C | K^R]_j . Q^T
        const int st = j % kStages, sb = j & 1;
        if (!mbar_wait(smem_u32(&ctl->full[st]), (j / kStages) & 1, abort_flag)) return false;
        if (!mbar_wait(smem_u32(&ctl->s_free[sb]), ((j >> 1) & 1) ^ 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kt = s_stage + st * Lo::kStageBytes;
#pragma unroll
        for (int ks = 0; ks < (R + kDR) / 16; ++ks)
          umma_f16(tmem + sb * kNR,
                   umma_desc(kt + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128),
                   umma_desc(s_q + (ks >> 2) * (kNR * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128),
                   idesc_s, ks > 0);
        umma_commit(smem_u32(&ctl->s_full[sb]));
        return true;
      };
      // QK(j + 1) is issued as soon as its tile has landed, but never ahead of a ready PV(j): with two
      // stages tile j + 1 only starts loading once PV(j - 1) has freed its stage, so blocking on it
      // would serialise every load behind the MMAs
      int qk_next = 0;
      if (nkt > 0) {
        ok = issue_qk(0);
        qk_next = 1;
      }
      for (int j = 0; j < nkt && ok; ++j) {
        const int st = j % kStages, pb = j & 1;
        const unsigned long long t0 = now_ns();
        for (int it = 0;; ++it) {
          if (qk_next == j + 1 && qk_next < nkt &&
              mbar_try(smem_u32(&ctl->full[qk_next % kStages]), (qk_next / kStages) & 1) &&
              mbar_try(smem_u32(&ctl->s_free[qk_next & 1]), ((qk_next >> 1) & 1) ^ 1)) {
            ok = issue_qk(qk_next);                         // both ready: does not block
            ++qk_next;
            if (!ok) break;
          }
          if (mbar_try(smem_u32(&ctl->p_full[pb]), (j >> 1) & 1)) break;
          if ((it & 31) == 31) {
            if (*abort_flag) { ok = false; break; }
            if (now_ns() - t0 > kWaitLimitNs) { *abort_flag = 1; ok = false; break; }
          }
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t ct = s_stage + st * Lo::kStageBytes;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t pt = s_p + (pb * 2 + part) * Lo::kPBytes;
#pragma unroll
          for (int mb = 0; mb < Lo::kOBlocks; ++mb)
#pragma unroll
            for (int ks = 0; ks < kKT / 16; ++ks)
              umma_f16(tmem_o + mb * kNR,
                       umma_desc(ct + 2 * mb * kBox + ks * 2048, kBox, 1024, kSwizzle128),
                       umma_desc(pt + ks * 32, 16, 1024, kSwizzle128),
                       idesc_o, (j | part | ks) != 0);
        }
        umma_commit(smem_u32(&ctl->empty[st]));             // the tile's latent has served as key and value
        umma_commit(smem_u32(&ctl->p_free[pb]));
        if (qk_next == j + 1 && qk_next < nkt) {             // its tile had not landed yet
          ok = issue_qk(qk_next);
          ++qk_next;
        }
      }
      if (ok) umma_commit(smem_u32(&ctl->o_full));
      umma_commit(smem_u32(&ctl->done));
      mbar_drain(smem_u32(&ctl->done), 0);
    }
  } else {
    // ---------------------------------- softmax and epilogue ---------------------------------------
    const int quad = warp & 3;
    const int w4 = warp - 2;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const bool key_lane = lane < 16;                         // M = 64: keys in the lower 16 lanes
    const int kslot = quad * 16 + lane;                      // this lane's key within a tile
    const float scale = a.scale * kLog2e;
    constexpr float kSlack = 8.f;
    int trow[kNR];
#pragma unroll
    for (int r = 0; r < kNR; ++r) trow[r] = (r < nrows) ? s_b + (row0 + r) / a.H : -1;
    float m_ref[kNR], l_part[kNR];
#pragma unroll
    for (int r = 0; r < kNR; ++r) { m_ref[r] = -INFINITY; l_part[r] = 0.f; }
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int sb = j & 1, pb = j & 1;
      ok = mbar_wait(smem_u32(&ctl->s_full[sb]), (j >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      float v[kNR];
      tmem_ld16(tmem + lane_base + sb * kNR, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[sb]));
      const int key = k_begin + j * kKT + kslot;
#pragma unroll
      for (int r = 0; r < kNR; ++r) v[r] = (key_lane && key < k_end && key <= trow[r]) ? v[r] * scale : -INFINITY;
      // tile maximum of each row across the 64 keys (16 lanes x 4 warps)
      float tmax[kNR];
#pragma unroll
      for (int r = 0; r < kNR; ++r) {
        float x = v[r];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        tmax[r] = x;
      }
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kNR; ++r) ctl->red[j & 1][w4][r] = tmax[r];
      }
      named_sync(1, kSoftmaxThreads);
      bool any_bump = false;
      float alpha[kNR];
#pragma unroll
      for (int r = 0; r < kNR; ++r) {
        const float t = fmaxf(fmaxf(ctl->red[j & 1][0][r], ctl->red[j & 1][1][r]),
                              fmaxf(ctl->red[j & 1][2][r], ctl->red[j & 1][3][r]));
        const bool bump = t > m_ref[r] + kSlack;
        const float m_new = bump ? t : m_ref[r];
        alpha[r] = bump ? ((m_ref[r] == -INFINITY) ? 0.f : fast_exp2(m_ref[r] - m_new)) : 1.f;
        any_bump |= bump;
        m_ref[r] = m_new;
      }
      // P buffer pb is free once PV(j - 2) is done; a rescale of O also needs PV(j - 1) done
      ok = mbar_wait(smem_u32(&ctl->p_free[pb]), ((j >> 1) & 1) ^ 1, abort_flag);
      if (ok && any_bump && j > 0) {
        ok = mbar_wait(smem_u32(&ctl->p_free[pb ^ 1]), (((j - 1) >> 1) & 1), abort_flag);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int mb = 0; mb < Lo::kOBlocks; ++mb) {
            float ov[kNR];
            tmem_ld16(tmem_o + lane_base + mb * kNR, ov);
#pragma unroll
            for (int r = 0; r < kNR; ++r) ov[r] *= alpha[r];
            tmem_st16(tmem_o + lane_base + mb * kNR, ov);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
      }
      if (!ok) break;
      unsigned char* ph = p_base + (pb * 2) * Lo::kPBytes;
      unsigned char* pl = ph + Lo::kPBytes;
#pragma unroll
      for (int r = 0; r < kNR; ++r) {
        l_part[r] *= alpha[r];
        const float p = (v[r] == -INFINITY) ? 0.f : fast_exp2(v[r] - m_ref[r]);
        l_part[r] += p;
        if (key_lane) {
          const Tc h16 = from_f32<Tc>(p);
          const Tc l16 = from_f32<Tc>(p - to_f32<Tc>(h16));
          const uint32_t off = sw128(kNR, r, kslot);
          *reinterpret_cast<Tc*>(ph + off) = h16;
          *reinterpret_cast<Tc*>(pl + off) = l16;
        }
      }
      tc_fence_before();
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[pb]));
    }
    // row sums over the 64 key lanes of every tile
#pragma unroll
    for (int r = 0; r < kNR; ++r) {
      float x = key_lane ? l_part[r] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0) ctl->lsum[w4][r] = x;
    }
    named_sync(1, kSoftmaxThreads);
    if (tid == 64) {
#pragma unroll
      for (int r = 0; r < kNR; ++r) {
        ctl->m[r] = m_ref[r];
        ctl->l[r] = ctl->lsum[0][r] + ctl->lsum[1][r] + ctl->lsum[2][r] + ctl->lsum[3][r];
      }
    }
    named_sync(1, kSoftmaxThreads);

    // ---- epilogue: thread = latent column (quad * 32 + lane) of each 128-column block ---------------
    ok = ok && mbar_wait(smem_u32(&ctl->o_full), 0, abort_flag);
    tc_fence_after();
    float o[Lo::kOBlocks][kNR];
#pragma unroll
    for (int mb = 0; mb < Lo::kOBlocks; ++mb) tmem_ld16(tmem_o + lane_base + mb * kNR, o[mb]);
    const bool aborted = *abort_flag != 0;
    const int dcol = quad * 32 + lane;
    const long long item_row0 = static_cast<long long>(item) * kNR;
    if (!aborted) {
#pragma unroll
      for (int r = 0; r < kNR; ++r) {
        if (r >= nrows) continue;
        const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
        const long long orow = ((static_cast<long long>(b) * a.H + h) * a.T + t) * R;
#pragma unroll
        for (int mb = 0; mb < Lo::kOBlocks; ++mb) {
          const int d = mb * 128 + dcol;
          if (nsplit == 1) put_out(a, orow + d, o[mb][r] / ctl->l[r]);
          else put_part_o(a, (item_row0 + r) * R + d, o[mb][r]);
        }
        if (nsplit > 1 && dcol == 0) {
          put_part_ml(a, (item_row0 + r) * 2, ctl->m[r]);
          put_part_ml(a, (item_row0 + r) * 2 + 1, ctl->l[r]);
        }
      }
    } else if (tid == 64) {
      atomicExch(a.status, kStatusTimeout);
    }
    if (nsplit > 1) {
      // ---- the CTA that finishes a unit's last split merges its partials ------------------------
      __threadfence();
      named_sync(1, kSoftmaxThreads);
      int* counter = a.counters + unit;
      if (tid == 64) ctl->last = (atomicAdd(counter, 1) == nsplit - 1);
      named_sync(1, kSoftmaxThreads);
      if (ctl->last) {
        __threadfence();
        const long long first_row = static_cast<long long>(plan.prefix[unit]) * kNR;
        if (nsplit <= kMergeSplits) {
          float* wm = reinterpret_cast<float*>(p_base);             // [kNR][kMergeSplits] m, then weight
          float* wl = wm + kNR * kMergeSplits;
          float* linv = wl + kNR * kMergeSplits;
          for (int i = tid - 64; i < nrows * nsplit; i += kSoftmaxThreads) {
            const int r = i / nsplit, sp = i % nsplit;
            const long long row = first_row + static_cast<long long>(sp) * kNR + r;
            wm[r * kMergeSplits + sp] = __ldcg(a.part_ml + row * 2);
            wl[r * kMergeSplits + sp] = __ldcg(a.part_ml + row * 2 + 1);
          }
          named_sync(1, kSoftmaxThreads);
          if (tid - 64 < nrows) {
            const int r = tid - 64;
            float m = -INFINITY;
            for (int sp = 0; sp < nsplit; ++sp)
              if (wl[r * kMergeSplits + sp] > 0.f) m = fmaxf(m, wm[r * kMergeSplits + sp]);
            float lsum = 0.f;
            for (int sp = 0; sp < nsplit; ++sp) {
              const float ls = wl[r * kMergeSplits + sp];
              const float w = ls > 0.f ? exp2f(wm[r * kMergeSplits + sp] - m) : 0.f;
              wm[r * kMergeSplits + sp] = w;
              lsum += w * ls;
            }
            linv[r] = 1.f / lsum;
          }
          named_sync(1, kSoftmaxThreads);
          for (int r = 0; r < nrows; ++r) {
            const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
            const long long orow = ((static_cast<long long>(b) * a.H + h) * a.T + t) * R;
#pragma unroll
            for (int mb = 0; mb < Lo::kOBlocks; ++mb) {
              const int d = mb * 128 + dcol;
              float acc = 0.f;
              for (int sp = 0; sp < nsplit; ++sp)
                acc = fmaf(wm[r * kMergeSplits + sp],
                           __ldcg(a.part_o + (first_row + static_cast<long long>(sp) * kNR + r) * R + d), acc);
              if (!aborted) put_out(a, orow + d, acc * linv[r]);
            }
          }
        } else {
          for (int r = 0; r < nrows; ++r) {
            const int gr = row0 + r, t = gr / a.H, h = gr % a.H;
            const long long orow = ((static_cast<long long>(b) * a.H + h) * a.T + t) * R;
#pragma unroll
            for (int mb = 0; mb < Lo::kOBlocks; ++mb) {
              const int d = mb * 128 + dcol;
              float m = -INFINITY, l = 0.f, acc = 0.f;
              for (int sp = 0; sp < nsplit; ++sp) {
                const long long row = first_row + static_cast<long long>(sp) * kNR + r;
                const float ms = __ldcg(a.part_ml + row * 2), ls = __ldcg(a.part_ml + row * 2 + 1);
                if (!(ls > 0.f)) continue;
                const float mn = fmaxf(m, ms);
                const float c_old = exp2f(m - mn), c_new = exp2f(ms - mn);
                l = l * c_old + ls * c_new;
                acc = acc * c_old + __ldcg(a.part_o + row * R + d) * c_new;
                m = mn;
              }
              if (!aborted) put_out(a, orow + d, acc / l);
            }
          }
        }
        if (tid == 64) *counter = 0;
      }
    }
  }

  // ---- teardown -----------------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

template <typename Tc, int R>
cudaError_t run(const MlaArgs& a, const SplitPlan& p, const CUtensorMap* tc, const CUtensorMap* tr,
                cudaStream_t st) {
  const size_t smem = mla_tc_smem<R>();
  cudaError_t e = ensure_smem_limit<mla_tc_kernel<Tc, R>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(mla_tc_kernel<Tc, R>, dim3(p.n_items), dim3(kThreads), smem, st, a, p, *tc, *tr);
}

}  // namespace

bool mla_tc_shape(kvc_dtype dt, int r, int dR) {
  return (dt == KVC_F16 || dt == KVC_BF16) && (r == 256 || r == 512) && dR == kDR;
}

cudaError_t launch_mla_tc(const MlaArgs& a, const SplitPlan& p, const CUtensorMap* tc, const CUtensorMap* tr,
                          cudaStream_t st) {
  const bool bf = a.cache_dtype == KVC_BF16;
  if (a.r == 512) return bf ? run<__nv_bfloat16, 512>(a, p, tc, tr, st) : run<__half, 512>(a, p, tc, tr, st);
  if (a.r == 256) return bf ? run<__nv_bfloat16, 256>(a, p, tc, tr, st) : run<__half, 256>(a, p, tc, tr, st);
  return cudaErrorInvalidValue;
}

}  // namespace kvc
