// Chunk (prefill) attention over the KV cache on the 5th-generation tensor cores (tcgen05 + TMEM),
// for 16-bit caches with d_h = 128 and many query rows per K/V head (G * T > 32).
//
// What it computes ("KV cache, incremental decode, ...", §2.3 and §4 test_chunked_prefill_equals_whole;
// "KV cache decoding", "Prefill and decode"; "Heads, GQA and K/V cache"): query row (t, h) of a chunk
// at positions s_b .. s_b + T - 1 attends over stored keys j <= s_b + t.
//
// How: the G query heads of one K/V head and 128 / G consecutive chunk positions form a tile of 128
// query rows (rows r = t * G + g), the M dimension; 128-key tiles are N:
//   S  [128 rows x 128 keys] = Q . K_j^T        A = Q (K-major), B = K tile (K-major)
//   Ot [128 rows x 128 d   ] = P_j . V_j        A = P (K-major, shared memory), B = V tile (MN-major)
// One CTA per (sequence, K/V head, row tile), one CTA per SM (all 512 TMEM columns):
//   warp 0     TMA: K_j and V_j tiles through a ring;
//   warp 1     owns TMEM, issues QK(j + 1) before PV(j) so the tensor cores run ahead of the softmax;
//   warps 2-5  one thread per query row: online softmax in base 2 against a per-row reference
//              maximum m_ref; P = 2^(s - m_ref) goes to shared memory (f16; for bf16 a hi + lo pair,
//              so P keeps ~2^-16 relative accuracy). The output accumulates in TMEM across tiles;
//              it is rescaled (read, multiply, write back) only when a row's maximum passes
//              m_ref + 8, which keeps P <= 2^8 and happens only on the first tiles of a row in
//              practice. The final division by the row sum uses the same reference, so the result
//              is the plain softmax.
// Tiles of keys past a row tile's last visible key are skipped; the diagonal tiles are masked per
// row. Every wait is bounded (~1 s) and reported through the device status word.
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kRows = 128;                   // query rows per CTA (MMA M)
constexpr int kKeys = 128;                   // keys per tile (MMA N of QK, K of PV)
constexpr int kDh = 128;
constexpr int kBox = 128 * 128;              // one 128-byte-swizzled atom column of 128 rows (16 KB)
constexpr int kTile = 2 * kBox;              // 32 KB: 128 rows x 128 16-bit values
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kTmemCols = 512;

template <typename Tc>
struct PLayout {
  static constexpr bool kHiLo = std::is_same<Tc, __nv_bfloat16>::value;
  static constexpr int kParts = kHiLo ? 2 : 1;
  static constexpr int kStages = kHiLo ? 3 : 4;             // K/V ring (each stage one 32 KB tile)
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQOff + kTile;
  static constexpr int kPOff = kRingOff + kStages * kTile;
  static constexpr int kCtlOff = kPOff + kParts * kTile;
};

struct __align__(8) PCtl {
  unsigned long long full[4], empty[4];
  unsigned long long s_full[2], s_free[2];
  unsigned long long p_full, p_free, o_full, done;
  uint32_t tmem;
  int abort;
};

template <typename Tc>
constexpr size_t prefill_smem() { return 1024 + PLayout<Tc>::kCtlOff + sizeof(PCtl); }

// offset of 16-byte chunk `c` (0..15) of row `r` in a [128 rows][128 16-bit] swizzled tile
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
  return (c >> 3) * kBox + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  while (!mbar_try(bar, parity)) {
    if (now_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
         "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]),
         "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]),
         "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

// 2^x with the hardware approximation (relative error ~2^-22), flushing subnormal results to zero
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// two floats -> one 32-bit word of two 16-bit values (round to nearest even), in one conversion
template <typename Tc>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (std::is_same<Tc, __half>::value) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}
// the two floats a packed word stands for
template <typename Tc>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (std::is_same<Tc, __half>::value) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  else return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <typename Tc>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const AttnArgs a, const __grid_constant__ SplitPlan plan,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using Lo = PLayout<Tc>;
  constexpr int kStages = Lo::kStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PCtl* ctl = reinterpret_cast<PCtl*>(sm + Lo::kCtlOff);
  const uint32_t s_q = smem_u32(sm + Lo::kQOff);
  const uint32_t s_ring = smem_u32(sm + Lo::kRingOff);
  unsigned char* p_base = sm + Lo::kPOff;
  const uint32_t s_p = smem_u32(p_base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kFmt = std::is_same<Tc, __nv_bfloat16>::value ? 1u : 0u;

  // ---- work item: (unit = sequence x row tile, K/V head) -----------------------------------------
  const int item = blockIdx.x;
  const int unit = item / a.H_kv, kvh = item % a.H_kv;
  const int b = plan.unit_b[unit] / plan.n_rowtiles;
  const int rt = plan.unit_b[unit] % plan.n_rowtiles;
  const int row0 = rt * kRows;
  const int nrows = min(kRows, a.T * a.G - row0);

  // ---- set-up ------------------------------------------------------------------------------------
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&ctl->tmem));
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->s_full[s]), 1);
      mbar_init(smem_u32(&ctl->s_free[s]), kSoftmaxThreads / 32);
    }
    mbar_init(smem_u32(&ctl->p_full), kSoftmaxThreads / 32);
    mbar_init(smem_u32(&ctl->p_free), 1);
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  // from here on the lengths and the queries, which earlier kernels write, are read
  pdl_wait();
  pdl_trigger();
  const int s_b = a.lens[b] + a.delta - a.T;
  const int first_t = row0 / a.G, last_t = (row0 + nrows - 1) / a.G;
  const int n_keys = s_b + last_t + 1;                       // keys visible to the tile's last row
  const int nkt = (n_keys + kKeys - 1) / kKeys;
  const int unmasked_keys = s_b + first_t + 1;               // keys visible to every row of the tile
  // Q tile: 128 rows x 128 d in the cache dtype, 128-byte swizzled (rows past the chunk are zero)
  for (int i = tid; i < kRows * (kDh / 8); i += kThreads) {
    const int r = i / (kDh / 8), c = i % (kDh / 8);
    uint4 w = make_uint4(0, 0, 0, 0);
    if (r < nrows) {
      const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
      const long long base = ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh + c * 8;
      if (a.rope.table != nullptr) {          // rotated to position s_b + t, element by element
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = load_query_rot<Tc>(a, base - c * 8, c * 8 + j, s_b + t);
        w = make_uint4(pack2<Tc>(x[0], x[1]), pack2<Tc>(x[2], x[3]), pack2<Tc>(x[4], x[5]), pack2<Tc>(x[6], x[7]));
      } else if (a.q_dtype == KVC_F32) {
        const float4 x0 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + base);
        const float4 x1 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + base + 4);
        w = make_uint4(pack2<Tc>(x0.x, x0.y), pack2<Tc>(x0.z, x0.w), pack2<Tc>(x1.x, x1.y), pack2<Tc>(x1.z, x1.w));
      } else {
        w = *reinterpret_cast<const uint4*>(static_cast<const Tc*>(a.q) + base);
      }
    }
    *reinterpret_cast<uint4*>(sm + Lo::kQOff + chunk_off(r, c)) = w;
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  volatile int* abort_flag = &ctl->abort;

  if (warp == 0) {
    // ---------------------------------- TMA producer (whole warp): K0, V0, K1, V1, ... -------------
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    int issued = 0;
    for (int i = 0; i < 2 * nkt; ++i) {
      const int st = i % kStages;
      const TilePiece pc = tile_piece<kKeys>(a, b, kvh, (i >> 1) * kKeys, lane);
      const uint32_t full = smem_u32(&ctl->full[st]);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&ctl->empty[st]), ((i / kStages) & 1) ^ 1, abort_flag);
        if (ok) mbar_expect_tx(full, kTile);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue_piece<kKeys, 2, 128, 64>(pc, (i & 1) ? &tv : &tk, s_ring + st * kTile, full, lane);
      issued = i + 1;
    }
    if (lane == 0)
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_drain(smem_u32(&ctl->full[i % kStages]), (i / kStages) & 1);
  } else if (warp == 1) {
    // ---------------------------------- MMA issuer ------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc(kRows, kKeys, kFmt, 0, 0);
      const uint32_t idesc_o = umma_idesc(kRows, kDh, kFmt, 0, 1);
      bool ok = true;
      auto issue_qk = [&](int j) -> bool {
        const int i = 2 * j, st = i % kStages, sb = j & 1;
        if (!mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag)) return false;
        if (!mbar_wait(smem_u32(&ctl->s_free[sb]), ((j >> 1) & 1) ^ 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kt = s_ring + st * kTile;
#pragma unroll
        for (int ks = 0; ks < kDh / 16; ++ks)
          umma_f16(tmem + sb * kKeys,
                   umma_desc(s_q + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128),
                   umma_desc(kt + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128), idesc_s, ks > 0);
        umma_commit(smem_u32(&ctl->empty[st]));
        umma_commit(smem_u32(&ctl->s_full[sb]));
        return true;
      };
      if (nkt > 0) ok = issue_qk(0);
      for (int j = 0; j < nkt && ok; ++j) {
        if (j + 1 < nkt) ok = issue_qk(j + 1);
        if (!ok) break;
        const int i = 2 * j + 1, st = i % kStages;
        ok = mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag) &&
             mbar_wait(smem_u32(&ctl->p_full), j & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vt = s_ring + st * kTile;
#pragma unroll
        for (int part = 0; part < Lo::kParts; ++part)
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks)
            umma_f16(tmem + 2 * kKeys,
                     umma_desc(s_p + part * kTile + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128),
                     umma_desc(vt + ks * 2048, kBox, 1024, kSwizzle128), idesc_o, (j | part | ks) != 0);
        umma_commit(smem_u32(&ctl->empty[st]));
        umma_commit(smem_u32(&ctl->p_free));
      }
      if (ok) umma_commit(smem_u32(&ctl->o_full));
      umma_commit(smem_u32(&ctl->done));
      mbar_drain(smem_u32(&ctl->done), 0);
    }
  } else {
    // ---------------------------------- softmax and epilogue ---------------------------------------
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                          // this thread's query row (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tmem_o = tmem + lane_base + 2 * kKeys;
    const bool row_ok = r < nrows;
    const int t_row = row_ok ? (row0 + r) / a.G : 0;
    const int last_key = s_b + t_row;                        // this row sees keys <= last_key
    const float scale = kLog2e * rsqrtf(static_cast<float>(kDh));
    constexpr float kSlack = 8.f;                            // P <= 2^kSlack before a rescale is forced
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int sb = j & 1;
      ok = mbar_wait(smem_u32(&ctl->s_full[sb]), (j >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      float v[kKeys];
#pragma unroll
      for (int c = 0; c < kKeys; c += 32) tmem_ld32(tmem + lane_base + sb * kKeys + c, v + c);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[sb]));  // S buffer may be overwritten now
      const int key0 = j * kKeys;
      if ((j + 1) * kKeys > unmasked_keys || !row_ok) {        // diagonal tile (or padding row)
#pragma unroll
        for (int e = 0; e < kKeys; ++e)
          if (!row_ok || key0 + e > last_key) v[e] = -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = v[k];
#pragma unroll
      for (int e = 8; e < kKeys; ++e) mx[e & 7] = fmaxf(mx[e & 7], v[e]);
      const float tmax = scale * fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // a new reference when this row's maximum passes the old one by more than kSlack
      const bool bump = tmax > m_ref + kSlack;
      const float m_new = bump ? tmax : m_ref;
      const float alpha = bump ? ((m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new)) : 1.f;
      // the previous tile's PV must be done before P is overwritten or the output rescaled
      ok = mbar_wait(smem_u32(&ctl->p_free), (j & 1) ^ 1, abort_flag);
      if (!ok) break;
      if (j > 0 && __any_sync(0xffffffffu, bump)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kDh; c += 32) {
          float ov[32];
          tmem_ld32(tmem_o + c, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= alpha;
          tmem_st32(tmem_o + c, ov);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      l *= alpha;
      m_ref = m_new;
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;   // padding rows: every score is -inf
      float ls[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls[k] = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < kKeys / 8; ++c8) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = fast_exp2(fmaf(v[c8 * 8 + e], scale, neg_m));  // 0 for masked keys (-inf)
          ls[e] += p[e];
        }
        const uint4 w = make_uint4(pack2<Tc>(p[0], p[1]), pack2<Tc>(p[2], p[3]), pack2<Tc>(p[4], p[5]),
                                   pack2<Tc>(p[6], p[7]));
        *reinterpret_cast<uint4*>(p_base + chunk_off(r, c8)) = w;
        if constexpr (Lo::kParts == 2) {
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
          uint32_t lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 h = unpack2<Tc>(ww[k]);
            lo[k] = pack2<Tc>(p[2 * k] - h.x, p[2 * k + 1] - h.y);
          }
          *reinterpret_cast<uint4*>(p_base + kTile + chunk_off(r, c8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      tc_fence_before();
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
    }
    // ---- epilogue: O / l ---------------------------------------------------------------------------
    ok = ok && mbar_wait(smem_u32(&ctl->o_full), 0, abort_flag);
    tc_fence_after();
    const bool aborted = *abort_flag != 0;
    if (aborted) {
      if (tid == 64) atomicExch(a.status, kStatusTimeout);
    } else {
      const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
      float* dst = row_ok ? a.out + ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh : nullptr;
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < kDh; c += 32) {
        float ov[32];
        tmem_ld32(tmem_o + c, ov);                             // warp-wide: every lane takes part
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + c + i) =
                make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

template <typename Tc>
cudaError_t run(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk, const CUtensorMap* tv,
                cudaStream_t st) {
  auto kern = prefill_tc_kernel<Tc>;
  const size_t smem = prefill_smem<Tc>();
  cudaError_t e = ensure_smem_limit<prefill_tc_kernel<Tc>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.n_units * a.H_kv), dim3(kThreads), smem, st, a, p, *tk, *tv);
}

static_assert(prefill_smem<__half>() > 114 * 1024 && prefill_smem<__nv_bfloat16>() > 114 * 1024,
              "one CTA per SM: each holds all 512 TMEM columns");
static_assert(prefill_smem<__half>() <= 227 * 1024 && prefill_smem<__nv_bfloat16>() <= 227 * 1024, "smem");

}  // namespace

bool prefill_tc_shape(kvc_dtype dt, int D, int* rows_per_tile) {
  if ((dt != KVC_F16 && dt != KVC_BF16) || D != kDh) return false;
  *rows_per_tile = kRows;
  return true;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                              const CUtensorMap* tv, cudaStream_t st) {
  return a.cache_dtype == KVC_BF16 ? run<__nv_bfloat16>(a, p, tk, tv, st) : run<__half>(a, p, tk, tv, st);
}

}  // namespace kvc
