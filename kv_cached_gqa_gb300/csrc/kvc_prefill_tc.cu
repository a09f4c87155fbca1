// Chunk attention over the KV cache on the 5th-generation tensor cores (tcgen05 + TMEM), for
// 16-bit caches with d_h = 128 and more than 16 query rows per K/V head (verify and prefill chunks).
//
// What it computes ("KV cache, incremental decode, ...", §2.3 and §4 test_chunked_prefill_equals_whole;
// "KV cache decoding", "Prefill and decode"; "Heads, GQA and K/V cache"): query row (t, h) of a chunk
// at positions s_b .. s_b + T - 1 attends over stored keys j <= s_b + t.
//
// How: the G query heads of one K/V head and consecutive chunk positions form query rows
// r = t * G + g; a CTA takes a tile of 128 of them (the M dimension) against 128-key tiles (N):
//   S [128 rows x 128 keys] = Q . K_j^T    A = Q (K-major, shared memory), B = K tile (K-major)
//   O [128 rows x 128 d   ] += P . V_j     A = P (tensor memory), B = V tile (MN-major)
// Each softmax thread writes its row of P to tensor memory in 16-bit form and the PV product takes P
// from there, so P never passes through shared memory. Roles (192 threads):
//   warp 0     TMA: K_j and V_j tiles through a ring;
//   warp 1     owns TMEM and issues every MMA from one thread;
//   warps 2-5  one thread per query row: online softmax in base 2 against a per-row reference
//              maximum m_ref; P = 2^(s - m_ref) in f16 (for bf16 a hi + lo pair, so P keeps ~2^-16
//              relative accuracy). O accumulates in tensor memory across key tiles and is rescaled
//              (read, multiply, write back) only when a row's maximum passes m_ref + 8, which keeps
//              P <= 2^8 and happens only on the first tiles of a row in practice. The final division
//              by the row sum uses the same reference, so the result is the plain softmax.
// Two forms:
//   narrow (more than 128 rows per K/V head: prefill). Two CTAs per SM, 256 TMEM columns: S in 128,
//     P written over it once read, O in the next 128. PV(j) then QK(j+1), which overwrites P(j) and
//     so waits for PV(j). Each CTA's step is a chain (QK, softmax, PV); the SM's other CTA fills the
//     tensor pipe and hides each CTA's query staging and output writes. The planner may split a
//     unit's keys over CTAs; the CTA that finishes a unit's last split merges the partials.
//   wide (at most 128 rows: verify chunks). One CTA per SM, 512 TMEM columns: S alternates between
//     columns 0 and 256, O in 128 .. 255, P in 384 .. 511 of its own, so QK(j+1) goes ahead of PV(j)
//     and the softmax of step j+1 follows that of j without waiting for any product.
// Tiles of keys past a row tile's last visible key are skipped; the diagonal tiles are masked per row.
// Softmax warps whose 32 rows all lie past the chunk sit out (their lanes of S hold the scores of zero
// queries, 0, which read as P = 0, and their rows are not stored). Every wait is bounded (~1 s) and
// reported through the device status word.
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
constexpr int kMaxStages = 5;

template <bool kWide>
struct PConf {
  static constexpr int kTmemCols = kWide ? 512 : 256;
  static constexpr int kStages = kWide ? 5 : 2;                // K/V ring, one 32 KB tile per stage
  static constexpr int kCtasPerSm = kWide ? 1 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQOff + kTile;
  static constexpr int kCtlOff = kRingOff + kStages * kTile;
};

struct __align__(8) PCtl {
  unsigned long long full[kMaxStages], empty[kMaxStages];
  unsigned long long s_full[2], s_free[2], p_full[2], pv_done[2];
  unsigned long long done;
  uint32_t tmem;
  int abort, last;
};

template <bool kWide>
constexpr size_t prefill_smem() { return 1024 + PConf<kWide>::kCtlOff + sizeof(PCtl); }

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

#define KVC_R8(b) "=r"(r[b]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), \
                  "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])

// 128 consecutive 32-bit columns of this thread's TMEM lane in one load (warp w: lanes 32*(w%4)..+31)
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* v) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
      "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127"
      "}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : KVC_R8(0), KVC_R8(8), KVC_R8(16), KVC_R8(24), KVC_R8(32), KVC_R8(40), KVC_R8(48), KVC_R8(56),
        KVC_R8(64), KVC_R8(72), KVC_R8(80), KVC_R8(88), KVC_R8(96), KVC_R8(104), KVC_R8(112), KVC_R8(120)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : KVC_R8(0), KVC_R8(8), KVC_R8(16), KVC_R8(24)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
#undef KVC_R8

// 32 consecutive 32-bit columns of this thread's TMEM lane (completion: tcgen05.wait::st)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
         "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
         "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
         "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
      : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
         "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (tensor memory) [+]= A (tensor memory, K-major) . B (shared memory descriptor)
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      :: "r"(tmem_d), "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// 2^x with the hardware approximation (relative error ~2^-22), flushing subnormal results to zero
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// two floats -> one 32-bit word of two 16-bit values (round to nearest even), in one conversion;
// the first float takes the low half (the lower key index of a K-major operand)
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

template <typename Tc, bool kWide>
__global__ void __launch_bounds__(kThreads, PConf<kWide>::kCtasPerSm)
prefill_tc_kernel(const AttnArgs a, const __grid_constant__ SplitPlan plan,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using C = PConf<kWide>;
  constexpr int kStages = C::kStages, kTmemCols = C::kTmemCols;
  constexpr bool kHiLo = std::is_same<Tc, __nv_bfloat16>::value;
  constexpr uint32_t kFmt = kHiLo ? 1u : 0u;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PCtl* ctl = reinterpret_cast<PCtl*>(sm + C::kCtlOff);
  const uint32_t s_q = smem_u32(sm + C::kQOff);
  const uint32_t s_ring = smem_u32(sm + C::kRingOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work item: (unit = sequence x 128-row tile, K/V head, key split) ----------------------------
  const int item = blockIdx.x;
  int unit, kvh, split = 0, nsplit = 1;
  if constexpr (!kWide) {                      // items of unit u: prefix[u] .. prefix[u + 1]
    int lo = 0, hi = plan.n_units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (plan.prefix[mid] <= item) lo = mid; else hi = mid - 1;
    }
    unit = lo;
    nsplit = (plan.prefix[unit + 1] - plan.prefix[unit]) / a.H_kv;
    const int rem = item - plan.prefix[unit];
    kvh = rem / nsplit;
    split = rem % nsplit;
  } else {
    unit = item / a.H_kv;
    kvh = item % a.H_kv;
  }
  const int b = plan.unit_b[unit] / plan.n_rowtiles;
  const int row0 = (plan.unit_b[unit] % plan.n_rowtiles) * kRows;
  const int n_rows = a.T * a.G;
  const int rows = min(n_rows - row0, kRows);                  // query rows of this tile
  const int warps_live = (rows + 31) / 32;                     // softmax warps that hold any

  // ---- set-up ------------------------------------------------------------------------------------
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&ctl->tmem));
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->s_full[s]), 1);
      mbar_init(smem_u32(&ctl->s_free[s]), warps_live);
      mbar_init(smem_u32(&ctl->p_full[s]), warps_live);
      mbar_init(smem_u32(&ctl->pv_done[s]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  volatile int* abort_flag = &ctl->abort;

  // from here on the lengths and the queries, which earlier kernels write, are read
  pdl_wait();
  pdl_trigger();
  const int s_b = a.lens[b] + a.delta - a.T;
  // key tiles: up to the key the tile's last row sees, or (narrow) this split's whole tiles
  // kt0 .. kt0 + nk - 1, cut by the planner's rule
  const int n_eff = s_b + (row0 + rows - 1) / a.G + 1;
  int kt0 = 0, nk = (n_eff + kKeys - 1) / kKeys;
  if constexpr (!kWide) {
    const int chunk = split_chunk(n_eff, nsplit, kKeys);
    const int k_begin = split * chunk, k_end = min(n_eff, k_begin + chunk);
    kt0 = k_begin / kKeys;
    nk = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;
  }
  // Where step j keeps S and P, and which barriers it uses ({barrier, phase}).
  //   narrow: S and P in columns 0 .. 127 (P over S once the scores are read); every barrier of
  //     slot 0, phase j. QK(j+1) waits for PV(j), which read P(j) from there.
  //   wide: S alternates between columns 0 and 256 (s_full / s_free of slot j & 1, phase j / 2) and P
  //     has its own columns 384 .. 511 (f16: two 64-column buffers, j & 1; bf16: one 128-column hi + lo
  //     buffer), with p_full / pv_done of its buffer. QK(j+1) then waits only until the softmax has
  //     read S(j-1), and the softmax waits for the PV that last read its P buffer.
  struct Slot { int bar, phase; };
  auto s_slot = [](int j) -> Slot { return kWide ? Slot{j & 1, j >> 1} : Slot{0, j}; };
  auto p_slot = [](int j) -> Slot {
    return kWide ? (kHiLo ? Slot{0, j} : Slot{j & 1, j >> 1}) : Slot{0, j};
  };
  auto s_col = [](int j) -> uint32_t { return kWide ? (j & 1) * 256 : 0; };
  auto p_col = [](int j) -> uint32_t { return kWide ? 384 + (kHiLo ? 0 : (j & 1) * 64) : 0; };
  constexpr uint32_t kOCol = 128;                              // O: columns 128 .. 255

  if (warp == 0) {
    // ---------------------------------- TMA producer (whole warp): K0, V0, K1, V1, ... -------------
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    int issued = 0;
    for (int i = 0; i < 2 * nk; ++i) {
      const int st = i % kStages;
      const TilePiece pc = tile_piece<kKeys>(a, b, kvh, (kt0 + (i >> 1)) * kKeys, lane);
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
  } else {
    // ---- Q: 128 rows x 128 d in the cache dtype, 128-byte swizzled (rows past the chunk zero) ------
    constexpr int kChunks = kRows * (kDh / 8);
    constexpr int kStagers = kThreads - 32;
    constexpr int kBatch = (kChunks + kStagers - 1) / kStagers;   // every load in flight at once
    for (int i0 = tid - 32; i0 < kChunks; i0 += kBatch * kStagers) {
      uint4 raw[kBatch][2];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {                     // all of this batch's loads first
        raw[k][0] = raw[k][1] = make_uint4(0, 0, 0, 0);
        const int i = i0 + k * kStagers;
        const int r = i / (kDh / 8), c = i % (kDh / 8);
        if (i < kChunks && r < rows && a.rope.table == nullptr) {
          const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
          const long long base = ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh + c * 8;
          raw[k][0] = load_query4_raw<Tc>(a.q, a.q_dtype, base);
          raw[k][1] = load_query4_raw<Tc>(a.q, a.q_dtype, base + 4);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k * kStagers;
        if (i >= kChunks) break;
        const int r = i / (kDh / 8), c = i % (kDh / 8);
        uint4 w = make_uint4(0, 0, 0, 0);
        if (r < rows) {
          if (a.rope.table != nullptr) {       // rotated to position s_b + t, element by element
            const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
            const long long row = ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = load_query_rot<Tc>(a, row, c * 8 + e, s_b + t);
            w = make_uint4(pack2<Tc>(x[0], x[1]), pack2<Tc>(x[2], x[3]), pack2<Tc>(x[4], x[5]),
                           pack2<Tc>(x[6], x[7]));
          } else {
            const uint2 lo = query4_to<Tc, Tc>(raw[k][0], a.q_dtype);
            const uint2 hi = query4_to<Tc, Tc>(raw[k][1], a.q_dtype);
            w = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
        }
        *reinterpret_cast<uint4*>(sm + C::kQOff + chunk_off(r, c)) = w;
      }
    }
    fence_proxy_async();
    named_sync(1, kStagers);                                   // Q is in place for the MMAs

    if (warp == 1) {
      // ---------------------------------- MMA issuer (one thread) -------------------------------------
      if (lane == 0) {
        const uint32_t idesc_s = umma_idesc(kRows, kKeys, kFmt, 0, 0);
        const uint32_t idesc_o = umma_idesc(kRows, kDh, kFmt, 0, 1);
        // S(j) = Q K_j^T into its slot, once nothing still needs what the slot held
        auto issue_qk = [&](int j) -> bool {
          const int i = 2 * j, st = i % kStages;
          if (!mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag)) return false;
          if (!kWide && j > 0) {                               // P(j-1) over S: PV(j-1) read it
            const Slot q = p_slot(j - 1);
            if (!mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag)) return false;
          }
          if (kWide && j > 1) {                                // the softmax has read S(j-2)
            const Slot q = s_slot(j - 2);
            if (!mbar_wait(smem_u32(&ctl->s_free[q.bar]), q.phase & 1, abort_flag)) return false;
          }
          tc_fence_after();
          const uint32_t kt = s_ring + st * kTile;
#pragma unroll
          for (int ks = 0; ks < kDh / 16; ++ks)
            umma_f16(tmem + s_col(j),
                     umma_desc(s_q + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128),
                     umma_desc(kt + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128), idesc_s, ks > 0);
          umma_commit(smem_u32(&ctl->s_full[s_slot(j).bar]));
          umma_commit(smem_u32(&ctl->empty[st]));              // K_j read
          return true;
        };
        // O += P V_j, P from tensor memory: 16 keys are 8 columns (two 16-bit values each); for bf16
        // the 16 keys of step ks are hi in columns 16 ks .. 16 ks + 7 and lo in the next 8
        auto issue_pv = [&](int j) -> bool {
          const int i = 2 * j + 1, st = i % kStages;
          const Slot sl = p_slot(j);
          if (!mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag) ||
              !mbar_wait(smem_u32(&ctl->p_full[sl.bar]), sl.phase & 1, abort_flag))
            return false;
          tc_fence_after();
          const uint32_t vt = s_ring + st * kTile, p_t = tmem + p_col(j), o_t = tmem + kOCol;
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks) {
            const uint64_t vd = umma_desc(vt + ks * 2048, kBox, 1024, kSwizzle128);
            if constexpr (kHiLo) {
              umma_f16_ts(o_t, p_t + ks * 16, vd, idesc_o, (j | ks) != 0);
              umma_f16_ts(o_t, p_t + ks * 16 + 8, vd, idesc_o, 1);
            } else {
              umma_f16_ts(o_t, p_t + ks * 8, vd, idesc_o, (j | ks) != 0);
            }
          }
          umma_commit(smem_u32(&ctl->pv_done[sl.bar]));
          umma_commit(smem_u32(&ctl->empty[st]));              // V_j read
          return true;
        };
        bool ok = nk > 0 && issue_qk(0);
        for (int j = 0; j < nk && ok; ++j) {
          if constexpr (kWide) {
            // QK(j+1) into the other slot before PV(j): the softmax of j+1 follows j's
            if (j + 1 < nk) ok = issue_qk(j + 1);
            ok = ok && issue_pv(j);
          } else {
            // PV(j), then QK(j+1), which waits for it
            ok = issue_pv(j);
            if (ok && j + 1 < nk) ok = issue_qk(j + 1);
          }
        }
        umma_commit(smem_u32(&ctl->done));
        mbar_drain(smem_u32(&ctl->done), 0);
      }
    } else {
      // ---------------------------------- softmax and epilogue ---------------------------------------
      const int quad = warp & 3;
      const int r = quad * 32 + lane;                        // this thread's query row (TMEM lane)
      const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t tmem_o = tmem + lane_base + kOCol;
      const int gr = row0 + r;
      const bool row_ok = r < rows;
      const int last_key = s_b + (row_ok ? gr / a.G : 0);    // this row sees keys <= last_key
      const int unmasked_keys = s_b + row0 / a.G + 1;        // keys visible to every row of the tile
      const float scale = kLog2e * rsqrtf(static_cast<float>(kDh));
      constexpr float kSlack = 8.f;                          // P <= 2^kSlack before a rescale is forced
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      const bool idle = quad >= warps_live;                  // no row of this warp is in the chunk
      for (int j = 0; j < nk && ok && !idle; ++j) {
        const Slot sl = s_slot(j), pl = p_slot(j);
        const uint32_t tmem_s = tmem + lane_base + s_col(j), tmem_p = tmem + lane_base + p_col(j);
        // warp-uniform waits: the tensor-memory loads and stores below are warp-collective
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full[sl.bar]), sl.phase & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        float v[kKeys];
        tmem_ld128(tmem_s, v);
        if (kWide) {                                           // S(j) is read: QK(j+2) may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[sl.bar]));
        }
        const int key0 = (kt0 + j) * kKeys;
        if ((kt0 + j + 1) * kKeys > unmasked_keys || !row_ok) {   // diagonal tile (or padding row)
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
        l *= alpha;
        m_ref = m_new;
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;   // padding rows: every score is -inf
        if (kWide && j >= (kHiLo ? 1 : 2)) {                   // the PV that last read this P buffer
          const Slot q = p_slot(j - (kHiLo ? 1 : 2));          // is complete
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        float ls[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ls[k] = 0.f;
        // P: f16, keys 2w and 2w+1 in column w; bf16, the 16 keys of MMA step ks as 8 hi columns
        // (16 ks ..) then 8 lo columns (16 ks + 8 ..)
        constexpr int kGroup = kHiLo ? 16 : 32;                  // keys per 16-column store
#pragma unroll
        for (int g0 = 0; g0 < kKeys; g0 += kGroup) {
          uint32_t w[16];
#pragma unroll
          for (int c8 = 0; c8 < kGroup / 8; ++c8) {
            float p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              p[e] = fast_exp2(fmaf(v[g0 + c8 * 8 + e], scale, neg_m));   // 0 for masked keys (-inf)
              ls[e] += p[e];
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t hi = pack2<Tc>(p[2 * k], p[2 * k + 1]);
              w[c8 * 4 + k] = hi;
              if constexpr (kHiLo) {
                const float2 h = unpack2<Tc>(hi);
                w[8 + c8 * 4 + k] = pack2<Tc>(p[2 * k] - h.x, p[2 * k + 1] - h.y);
              }
            }
          }
          tmem_st16(tmem_p + (kHiLo ? g0 : g0 / 2), w);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        // O *= alpha once PV(j-1) is complete (narrow: it is, QK(j) was issued after it); PV(j) waits
        // for p_full, which follows these stores
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          const Slot q = p_slot(j - 1);
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kDh; c += 32) {
            float ov[32];
            tmem_ld32(tmem_o + c, ov);
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(ov[e] * alpha);
            tmem_st32(tmem_o + c, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[pl.bar]));
      }
      // ---- epilogue ---------------------------------------------------------------------------------
      if (!kWide && nsplit > 1) {
        // this split's partial (unnormalised O, m_ref, l) per row; the CTA that finishes the unit's
        // last split merges them (log-sum-exp in base 2), reading the partials from L2
        const int R = plan.rows_per_tile;
        if (!idle) {
          const Slot q = p_slot(nk - 1);
          ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag));
          tc_fence_after();
          const bool aborted = __any_sync(0xffffffffu, !ok || *abort_flag != 0);
          if (!aborted) {
            const long long prow = static_cast<long long>(item) * R + r;
#pragma unroll
            for (int c = 0; c < kDh; c += 32) {
              float ov[32];
              tmem_ld32(tmem_o + c, ov);                         // warp-wide: every lane takes part
              if (row_ok && in_bounds(prow * kDh + c + 31, a.part_o_elems, a.status)) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                  *reinterpret_cast<float4*>(a.part_o + prow * kDh + c + i) =
                      make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
              }
            }
            if (row_ok) {
              put_part_ml(a, prow * 2, m_ref);
              put_part_ml(a, prow * 2 + 1, l);
            }
          } else if (lane == 0) {
            atomicExch(a.status, kStatusTimeout);
          }
        }
        __threadfence();
        named_sync(2, kSoftmaxThreads);                          // every softmax warp, idle or not
        int* counter = a.counters + unit * a.H_kv + kvh;
        if (tid == 64) ctl->last = (atomicAdd(counter, 1) == nsplit - 1);
        named_sync(2, kSoftmaxThreads);
        if (ctl->last) {
          __threadfence();
          if (row_ok && *abort_flag == 0) {
            const long long first = static_cast<long long>(plan.prefix[unit] + kvh * nsplit) * R + r;
            float m_max = -INFINITY, l_sum = 0.f;
            for (int sp = 0; sp < nsplit; ++sp) {
              const long long row = first + static_cast<long long>(sp) * R;
              if (__ldcg(a.part_ml + row * 2 + 1) > 0.f) m_max = fmaxf(m_max, __ldcg(a.part_ml + row * 2));
            }
            for (int sp = 0; sp < nsplit; ++sp) {
              const long long row = first + static_cast<long long>(sp) * R;
              const float ls = __ldcg(a.part_ml + row * 2 + 1);
              if (ls > 0.f) l_sum += exp2f(__ldcg(a.part_ml + row * 2) - m_max) * ls;
            }
            const float inv = 1.f / l_sum;
            const int tq = gr / a.G, g = gr % a.G;
            float* dst = a.out + ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + tq) * kDh;
            for (int c = 0; c < kDh; c += 32) {
              float acc[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.f;
              for (int sp = 0; sp < nsplit; ++sp) {
                const long long row = first + static_cast<long long>(sp) * R;
                const float ls = __ldcg(a.part_ml + row * 2 + 1);
                if (!(ls > 0.f)) continue;
                const float w = exp2f(__ldcg(a.part_ml + row * 2) - m_max);
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                  const float4 o = __ldcg(reinterpret_cast<const float4*>(a.part_o + row * kDh + c + i));
                  acc[i] = fmaf(w, o.x, acc[i]);
                  acc[i + 1] = fmaf(w, o.y, acc[i + 1]);
                  acc[i + 2] = fmaf(w, o.z, acc[i + 2]);
                  acc[i + 3] = fmaf(w, o.w, acc[i + 3]);
                }
              }
              if (in_bounds(dst - a.out + c + 31, a.out_elems, a.status)) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                  *reinterpret_cast<float4*>(dst + c + i) =
                      make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv, acc[i + 3] * inv);
              }
            }
          }
          if (tid == 64) *counter = 0;
        }
      } else if (!idle) {
        // O / l straight to the output
        const Slot q = p_slot(nk - 1);
        ok = __all_sync(0xffffffffu, ok && mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag));
        tc_fence_after();
        const bool aborted = __any_sync(0xffffffffu, !ok || *abort_flag != 0);
        if (aborted) {
          if (lane == 0) atomicExch(a.status, kStatusTimeout);
        } else {
          const int tq = row_ok ? gr / a.G : 0, g = row_ok ? gr % a.G : 0;
          float* dst = a.out + ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + tq) * kDh;
          const float inv = 1.f / l;
#pragma unroll
          for (int c = 0; c < kDh; c += 32) {
            float ov[32];
            tmem_ld32(tmem_o + c, ov);                           // warp-wide: every lane takes part
            if (row_ok && in_bounds(dst - a.out + c + 31, a.out_elems, a.status)) {
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + c + i) =
                    make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
            }
          }
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

template <typename Tc, bool kWide>
cudaError_t run(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk, const CUtensorMap* tv,
                cudaStream_t st) {
  auto kern = prefill_tc_kernel<Tc, kWide>;
  constexpr size_t smem = prefill_smem<kWide>();
  cudaError_t e = ensure_smem_limit<prefill_tc_kernel<Tc, kWide>>(smem);
  if (e != cudaSuccess) return e;
  const int grid = kWide ? p.n_units * a.H_kv : p.n_items;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, a, p, *tk, *tv);
}

static_assert(prefill_smem<true>() > 114 * 1024, "wide: one CTA per SM, each holds all 512 TMEM columns");
static_assert(prefill_smem<true>() <= 227 * 1024, "smem");
static_assert(2 * prefill_smem<false>() + 2048 <= 228 * 1024, "narrow: two CTAs per SM");
static_assert(3 * prefill_smem<false>() > 228 * 1024, "narrow: never three CTAs (768 TMEM columns) on an SM");

}  // namespace

bool prefill_tc_shape(kvc_dtype dt, int D, int* rows_per_tile) {
  if ((dt != KVC_F16 && dt != KVC_BF16) || D != kDh) return false;
  *rows_per_tile = kRows;
  return true;
}

cudaError_t launch_chunk_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                            const CUtensorMap* tv, cudaStream_t st) {
  return a.cache_dtype == KVC_BF16 ? run<__nv_bfloat16, true>(a, p, tk, tv, st) : run<__half, true>(a, p, tk, tv, st);
}

cudaError_t launch_prefill_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                              const CUtensorMap* tv, cudaStream_t st) {
  return a.cache_dtype == KVC_BF16 ? run<__nv_bfloat16, false>(a, p, tk, tv, st) : run<__half, false>(a, p, tk, tv, st);
}

}  // namespace kvc
