// Chunk (prefill) attention over the KV cache on the 5th-generation tensor cores (tcgen05 + TMEM),
// for 16-bit caches with d_h = 128 and many query rows per K/V head (G * T > 16).
//
// What it computes ("KV cache, incremental decode, ...", §2.3 and §4 test_chunked_prefill_equals_whole;
// "KV cache decoding", "Prefill and decode"; "Heads, GQA and K/V cache"): query row (t, h) of a chunk
// at positions s_b .. s_b + T - 1 attends over stored keys j <= s_b + t.
//
// How: the G query heads of one K/V head and consecutive chunk positions form query rows
// r = t * G + g. A CTA takes 256 of them as two MMA tiles of 128 rows (the M dimension), so every
// K/V tile it loads serves both; 128-key tiles are N:
//   S_t [128 rows x 128 keys] = Q_t . K_j^T    A = Q_t (K-major, shared memory), B = K tile (K-major)
//   O_t [128 rows x 128 d   ] += P_t . V_j     A = P_t (tensor memory), B = V tile (MN-major)
// Tensor memory (512 columns) holds, per tile t, S_t in 128 columns and O_t in the next 128. Each
// softmax thread overwrites its row of S_t with P_t in 16-bit form once it has read the scores, and
// the PV product takes P_t straight from there, so P never passes through shared memory. A CTA with
// one tile (short chunks, ragged tails) uses the free half differently: S alternates between two
// slots and P has columns of its own, so QK(j+1) need not wait for PV(j) (see s_slot below).
// Roles (352 threads, one CTA per SM):
//   warp 0      TMA: K_j and V_j tiles through a ring;
//   warps 1, 10 one thread each issues the MMAs of tile 0 and of tile 1: PV_t(j), then QK_t(j+1),
//               so the tensor cores work on one tile while the softmax of the other runs, and the
//               two tiles' products (independent accumulators) overlap in the tensor pipe;
//   warps 2-5   softmax of tile 0, warps 6-9 softmax of tile 1: one thread per query row, online
//               softmax in base 2 against a per-row reference maximum m_ref; P = 2^(s - m_ref) in
//               f16 (for bf16 a hi + lo pair, so P keeps ~2^-16 relative accuracy). O accumulates
//               in tensor memory across key tiles and is rescaled (read, multiply, write back) only
//               when a row's maximum passes m_ref + 8, which keeps P <= 2^8 and happens only on the
//               first tiles of a row in practice. The final division by the row sum uses the same
//               reference, so the result is the plain softmax.
// Tiles of keys past a tile's last visible key are skipped; the diagonal tiles are masked per row.
// Every wait is bounded (~1 s) and reported through the device status word.
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kRows = 128;                   // query rows per MMA tile (MMA M)
constexpr int kTiles = 2;                    // MMA tiles per CTA
constexpr int kUnitRows = kTiles * kRows;    // query rows per CTA
constexpr int kKeys = 128;                   // keys per tile (MMA N of QK, K of PV)
constexpr int kDh = 128;
constexpr int kBox = 128 * 128;              // one 128-byte-swizzled atom column of 128 rows (16 KB)
constexpr int kTile = 2 * kBox;              // 32 KB: 128 rows x 128 16-bit values
constexpr int kSoftmaxThreads = 128;         // per MMA tile
constexpr int kThreads = 32 + kTiles * kSoftmaxThreads + kTiles * 32;   // TMA, softmax, one MMA issuer per tile
constexpr int kTmemCols = 512;               // per tile: S_t / P_t (128 columns), then O_t (128)
constexpr int kStages = 5;                   // K/V ring, one 32 KB tile per stage

constexpr int kQOff = 0;                     // Q_0, Q_1
constexpr int kRingOff = kQOff + kTiles * kTile;
constexpr int kCtlOff = kRingOff + kStages * kTile;

struct __align__(8) PCtl {
  unsigned long long full[kStages], empty[kStages];
  unsigned long long s_full[kTiles], s_free[kTiles], p_full[kTiles], pv_done[kTiles];
  unsigned long long done[kTiles];
  uint32_t tmem;
  int abort;
};

constexpr size_t prefill_smem() { return 1024 + kCtlOff + sizeof(PCtl); }

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

template <typename Tc>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const AttnArgs a, const __grid_constant__ SplitPlan plan,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  constexpr bool kHiLo = std::is_same<Tc, __nv_bfloat16>::value;
  constexpr uint32_t kFmt = kHiLo ? 1u : 0u;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PCtl* ctl = reinterpret_cast<PCtl*>(sm + kCtlOff);
  const uint32_t s_q = smem_u32(sm + kQOff);
  const uint32_t s_ring = smem_u32(sm + kRingOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work item: (unit = sequence x 256-row tile, K/V head) -------------------------------------
  const int item = blockIdx.x;
  const int unit = item / a.H_kv, kvh = item % a.H_kv;
  const int b = plan.unit_b[unit] / plan.n_rowtiles;
  const int row0 = (plan.unit_b[unit] % plan.n_rowtiles) * kUnitRows;
  const int n_rows = a.T * a.G;
  // rows of MMA tile t in this CTA, and its softmax warps that hold any (the others sit out: their
  // lanes of S hold the scores of zero queries, 0, which read as P = 0, and their rows are not stored)
  int rows_t[kTiles], warps_t[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    rows_t[t] = min(max(n_rows - (row0 + t * kRows), 0), kRows);
    warps_t[t] = (rows_t[t] + 31) / 32;
  }
  const bool pair = rows_t[1] > 0;

  // ---- set-up ------------------------------------------------------------------------------------
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&ctl->tmem));
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), kTiles);          // one release per MMA issuer
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(smem_u32(&ctl->s_full[t]), 1);
      // arrivals: the softmax warps that hold rows (with one tile, both slots belong to tile 0)
      const int arrivals = max(1, pair ? warps_t[t] : warps_t[0]);
      mbar_init(smem_u32(&ctl->s_free[t]), arrivals);
      mbar_init(smem_u32(&ctl->p_full[t]), arrivals);
      mbar_init(smem_u32(&ctl->pv_done[t]), 1);
    }
    for (int t = 0; t < kTiles; ++t) mbar_init(smem_u32(&ctl->done[t]), 1);
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
  // key tiles of MMA tile t: up to the key its last row sees; 0 for a tile past the chunk's rows
  int nk[kTiles];
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int first = row0 + t * kRows, last = min(first + kRows, n_rows) - 1;
    nk[t] = last >= first ? (s_b + last / a.G + 1 + kKeys - 1) / kKeys : 0;
  }
  const int nkt = max(nk[0], nk[1]);
  // Where step j of tile t keeps S and P, and which barriers it uses ({barrier, phase}).
  //   Two tiles: S and P share tile t's first 128 columns (P over S once the scores are read); every
  //   barrier of slot t, phase j. QK_t(j+1) waits for PV_t(j), which read P_t(j) from there.
  //   One tile: S alternates between columns 0 and 256 (s_full / s_free of slot j & 1, phase j / 2)
  //   and P has its own columns 384 .. 511 (f16: two 64-column buffers, j & 1; bf16: one 128-column
  //   hi + lo buffer), with p_full / pv_done of its buffer. QK(j+1) then waits only until the softmax
  //   has read S(j-1), and the softmax waits for the PV that last read its P buffer.
  struct Slot { int bar, phase; };
  auto s_slot = [pair](int t, int j) -> Slot { return pair ? Slot{t, j} : Slot{j & 1, j >> 1}; };
  auto p_slot = [pair](int t, int j) -> Slot {
    return pair ? Slot{t, j} : (kHiLo ? Slot{0, j} : Slot{j & 1, j >> 1});
  };
  auto s_col = [pair](int t, int j) -> uint32_t { return pair ? t * 256 : (j & 1) * 256; };
  auto p_col = [pair](int t, int j) -> uint32_t {
    return pair ? t * 256 : 384 + (kHiLo ? 0 : (j & 1) * 64);
  };

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
  } else {
    // ---- Q_0, Q_1: 256 rows x 128 d in the cache dtype, 128-byte swizzled (rows past the chunk zero)
    constexpr int kChunks = kUnitRows * (kDh / 8);
    constexpr int kStagers = kThreads - 32;
    constexpr int kBatch = (kChunks + kStagers - 1) / kStagers;   // every load in flight at once
    for (int i0 = tid - 32; i0 < kChunks; i0 += kBatch * kStagers) {
      uint4 raw[kBatch][2];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {                     // all of this batch's loads first
        raw[k][0] = raw[k][1] = make_uint4(0, 0, 0, 0);
        const int i = i0 + k * kStagers;
        const int r = i / (kDh / 8), c = i % (kDh / 8);
        if (i < kChunks && row0 + r < n_rows && a.rope.table == nullptr) {
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
        if (row0 + r < n_rows) {
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
        *reinterpret_cast<uint4*>(sm + kQOff + (r / kRows) * kTile + chunk_off(r % kRows, c)) = w;
      }
    }
    fence_proxy_async();
    named_sync(1, kStagers);                                   // Q is in place for the MMAs

    if (warp == 1 || warp == kThreads / 32 - 1) {
      // ---------------------------------- MMA issuer of tile t (one thread) --------------------------
      const int t = warp == 1 ? 0 : 1;
      if (lane == 0 && (t == 0 || pair)) {
        const uint32_t idesc_s = umma_idesc(kRows, kKeys, kFmt, 0, 0);
        const uint32_t idesc_o = umma_idesc(kRows, kDh, kFmt, 0, 1);
        // S_t(j) = Q_t K_j^T into its slot. P_t(j') of the slot's previous step lives there until
        // PV_t(j') has read it, so QK_t(j) waits for that product to complete.
        auto issue_qk = [&](int j) -> bool {
          const int i = 2 * j, st = i % kStages;
          if (!mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag)) return false;
          if (pair && j > 0) {                                 // P_t(j-1) over S_t: PV_t(j-1) read it
            const Slot q = p_slot(t, j - 1);
            if (!mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag)) return false;
          }
          if (!pair && j > 1) {                                // the softmax has read S(j-2)
            const Slot q = s_slot(t, j - 2);
            if (!mbar_wait(smem_u32(&ctl->s_free[q.bar]), q.phase & 1, abort_flag)) return false;
          }
          const Slot sl = s_slot(t, j);
          tc_fence_after();
          const uint32_t kt = s_ring + st * kTile, qt = s_q + t * kTile;
#pragma unroll
          for (int ks = 0; ks < kDh / 16; ++ks)
            umma_f16(tmem + s_col(t, j),
                     umma_desc(qt + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128),
                     umma_desc(kt + (ks >> 2) * kBox + (ks & 3) * 32, 16, 1024, kSwizzle128), idesc_s, ks > 0);
          umma_commit(smem_u32(&ctl->s_full[sl.bar]));
          return true;
        };
        // O_t += P_t V_j, P_t from tensor memory: 16 keys are 8 columns (two 16-bit values each); for
        // bf16 the 16 keys of step ks are hi in columns 16 ks .. 16 ks + 7 and lo in the next 8
        auto issue_pv = [&](int j) -> bool {
          const int i = 2 * j + 1, st = i % kStages;
          const Slot sl = p_slot(t, j);
          if (!mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag) ||
              !mbar_wait(smem_u32(&ctl->p_full[sl.bar]), sl.phase & 1, abort_flag))
            return false;
          tc_fence_after();
          const uint32_t vt = s_ring + st * kTile, p_t = tmem + p_col(t, j), o_t = tmem + t * 256 + 128;
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
          return true;
        };
        // a ring stage is refilled after both issuers released it; with one tile, its issuer releases
        // for both
        auto release = [&](int i) {
          umma_commit(smem_u32(&ctl->empty[i % kStages]));
          if (!pair) umma_commit(smem_u32(&ctl->empty[i % kStages]));
        };
        bool ok = issue_qk(0);
        if (ok) release(0);
        for (int j = 0; j < nk[t] && ok; ++j) {
          if (pair) {
            // PV_t(j), then QK_t(j+1) (which waits for it)
            ok = issue_pv(j);
            if (!ok) break;
            release(2 * j + 1);
            if (j + 1 < nk[t]) {
              ok = issue_qk(j + 1);
              if (ok) release(2 * j + 2);
            }
          } else {
            // one tile: QK(j+1) into the other slot before PV(j), so the softmax of j+1 follows j's
            if (j + 1 < nk[t]) {
              ok = issue_qk(j + 1);
              if (!ok) break;
              release(2 * j + 2);
            }
            ok = issue_pv(j);
            if (ok) release(2 * j + 1);
          }
        }
        // loads past this tile's keys (tile 0 may end a key tile before tile 1) still take this
        // issuer's release, in order: wait until each is in place, then arrive
        for (int i = 2 * nk[t]; i < 2 * nkt && ok; ++i) {
          ok = mbar_wait(smem_u32(&ctl->full[i % kStages]), (i / kStages) & 1, abort_flag);
          if (ok) mbar_arrive(smem_u32(&ctl->empty[i % kStages]));
        }
        umma_commit(smem_u32(&ctl->done[t]));
        mbar_drain(smem_u32(&ctl->done[t]), 0);
      }
    } else {
      // ---------------------------------- softmax and epilogue of tile t ---------------------------
      const int t = (warp - 2) / 4;
      const int quad = warp & 3;
      const int r = quad * 32 + lane;                        // this thread's query row (TMEM lane)
      const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t tmem_o = tmem + lane_base + t * 256 + 128;
      const int gr = row0 + t * kRows + r;
      const bool row_ok = gr < n_rows;
      const int t_row = row_ok ? gr / a.G : 0;
      const int last_key = s_b + t_row;                      // this row sees keys <= last_key
      const int first_t = (row0 + t * kRows) / a.G;
      const int unmasked_keys = s_b + first_t + 1;           // keys visible to every row of the tile
      const float scale = kLog2e * rsqrtf(static_cast<float>(kDh));
      constexpr float kSlack = 8.f;                          // P <= 2^kSlack before a rescale is forced
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      const bool idle = quad >= warps_t[t];                  // no row of this warp is in the chunk
      for (int j = 0; j < nk[t] && ok && !idle; ++j) {
        const Slot sl = s_slot(t, j), pl = p_slot(t, j);
        const uint32_t tmem_s = tmem + lane_base + s_col(t, j), tmem_p = tmem + lane_base + p_col(t, j);
        // warp-uniform waits: the tensor-memory loads and stores below are warp-collective
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->s_full[sl.bar]), sl.phase & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        float v[kKeys];
        tmem_ld128(tmem_s, v);
        if (!pair) {                                           // S(j) is read: QK(j+2) may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[sl.bar]));
        }
        const int key0 = j * kKeys;
        if ((j + 1) * kKeys > unmasked_keys || !row_ok) {      // diagonal tile (or padding row)
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
        if (!pair && j >= (kHiLo ? 1 : 2)) {                   // one tile: the PV that last read this
          const Slot q = p_slot(t, j - (kHiLo ? 1 : 2));      // P buffer is complete
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->pv_done[q.bar]), q.phase & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        float ls[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ls[k] = 0.f;
        // P_t over S_t: f16, keys 2w and 2w+1 in column w; bf16, the 16 keys of MMA step ks as 8 hi
        // columns (16 ks ..) then 8 lo columns (16 ks + 8 ..)
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
        // O_t *= alpha once PV_t(j-1) is complete (with two tiles it is: QK_t(j) was issued after
        // it); PV_t(j) waits for p_full, which follows these stores.
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          const Slot q = p_slot(t, j - 1);
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
      // ---- epilogue: O_t / l -------------------------------------------------------------------------
      if (nk[t] > 0 && !idle) {
        const Slot q = p_slot(t, nk[t] - 1);
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
            if (row_ok) {
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

template <typename Tc>
cudaError_t run(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk, const CUtensorMap* tv,
                cudaStream_t st) {
  auto kern = prefill_tc_kernel<Tc>;
  constexpr size_t smem = prefill_smem();
  cudaError_t e = ensure_smem_limit<prefill_tc_kernel<Tc>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.n_units * a.H_kv), dim3(kThreads), smem, st, a, p, *tk, *tv);
}

static_assert(prefill_smem() > 114 * 1024, "one CTA per SM: each holds all 512 TMEM columns");
static_assert(prefill_smem() <= 227 * 1024, "smem");
static_assert(kThreads - 32 == 320, "the named barrier counts warps 1-10");

}  // namespace

bool prefill_tc_shape(kvc_dtype dt, int D, int* rows_per_tile) {
  if ((dt != KVC_F16 && dt != KVC_BF16) || D != kDh) return false;
  *rows_per_tile = kUnitRows;
  return true;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                              const CUtensorMap* tv, cudaStream_t st) {
  return a.cache_dtype == KVC_BF16 ? run<__nv_bfloat16>(a, p, tk, tv, st) : run<__half>(a, p, tk, tv, st);
}

}  // namespace kvc
