// Device-side building blocks shared by the attention kernels: shared-memory addresses, bounded
// mbarrier waits, TMA tile loads, and the tcgen05 (5th-generation tensor core) operations with
// their shared-memory and instruction descriptors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <type_traits>

#include "kvc_internal.h"

namespace kvc {
namespace dev {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // every wait gives up after ~1 s
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase. Returns false when it gave up, or when another thread of the
// CTA already gave up (shared abort flag); the caller then skips its work but keeps its control
// flow, so every barrier of the CTA is still reached and nothing hangs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  unsigned long long t0 = 0;
  for (int it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 31) == 31) {
      if (*abort_flag) return false;
      const unsigned long long t = now_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kWaitLimitNs) { *abort_flag = 1; return false; }
    }
  }
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<unsigned long long>(map)) : "memory");
}
// ---- K/V tile addressing -------------------------------------------------------------------------
// Tensor-map coordinates (row, plane) of key `key` of K/V head kvh of sequence b. A contiguous store
// has one plane per (layer, b, kvh) and row = key. A paged pool has one plane per (layer, physical
// block, kvh) and row = key mod block, the block read from the sequence's table. A logical block with
// no physical block (past the table, or -1) maps to row `block` of a valid plane: past the map's row
// extent, where TMA writes zeros instead of reading memory.
__device__ __forceinline__ void kv_coords(const AttnArgs& a, int b, int kvh, int key, int* row, int* plane) {
  if (a.pg.table == nullptr) {
    *row = key;
    *plane = (a.layer * a.B + b) * a.H_kv + kvh;
    return;
  }
  const int idx = key >> a.pg.block_shift;
  const int phys = idx < a.pg.max_blocks ? a.pg.table[b * a.pg.max_blocks + idx] : -1;
  const bool have = phys >= 0 && phys < a.pg.n_blocks;
  *row = have ? (key & ((1 << a.pg.block_shift) - 1)) : (1 << a.pg.block_shift);
  *plane = (a.layer * a.pg.n_blocks + (have ? phys : 0)) * a.H_kv + kvh;
}

// One lane's share of a K/V tile load. A tile is keys [y, y + kRows) of one K or V head, stored as
// kBoxes boxes of kRows rows x kSpan bytes one after another. A contiguous store loads each box with
// one TMA (lane 0). A paged pool whose blocks are shorter than the tile loads it in pieces of one
// block: lane j issues piece j of every box, at row offset j * rows. The 128- and 64-byte swizzle
// patterns repeat every 8 rows and blocks hold at least 16, so the pieces land exactly where one
// whole-tile box would put them.
struct TilePiece {
  int row, plane, rows;
  bool on;
};
template <int kRows>
__device__ __forceinline__ TilePiece tile_piece(const AttnArgs& a, int b, int kvh, int y, int lane) {
  TilePiece p;
  p.rows = (a.pg.table != nullptr && (1 << a.pg.block_shift) < kRows) ? (1 << a.pg.block_shift) : kRows;
  p.on = lane * p.rows < kRows;
  p.row = 0;
  p.plane = 0;
  if (p.on) kv_coords(a, b, kvh, y + lane * p.rows, &p.row, &p.plane);
  return p;
}
// Issue the piece (after the stage's barrier has been armed for the whole tile's bytes). kInner is
// the element count of one box row, the x step between boxes.
template <int kRows, int kBoxes, int kSpan, int kInner>
__device__ __forceinline__ void issue_piece(const TilePiece& p, const CUtensorMap* map, uint32_t dst,
                                            uint32_t bar, int lane) {
  if (!p.on) return;
#pragma unroll
  for (int bx = 0; bx < kBoxes; ++bx)
    tma_load_3d(dst + static_cast<uint32_t>((bx * kRows + lane * p.rows) * kSpan), map, bx * kInner, p.row,
                p.plane, bar);
}

// generic-proxy shared-memory writes become visible to the async proxy (TMA, tensor cores)
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// ---- debug index checks (KVC_DEBUG_BOUNDS) ------------------------------------------------------
// In a debug build a global store whose index falls outside its buffer is skipped and reported through
// the status word (kvc_status returns KVC_E_DEVICE_BOUNDS); a release build compiles the check away.
__device__ __forceinline__ bool in_bounds(long long i, long long n, int* status) {
#ifdef KVC_DEBUG_BOUNDS
  if (i < 0 || i >= n) {
    atomicExch(status, kStatusBounds);
    return false;
  }
#else
  (void)i; (void)n; (void)status;
#endif
  return true;
}
template <typename A>
__device__ __forceinline__ void put_out(const A& a, long long i, float v) {
  if (in_bounds(i, a.out_elems, a.status)) a.out[i] = v;
}
template <typename A>
__device__ __forceinline__ void put_part_o(const A& a, long long i, float v) {
  if (in_bounds(i, a.part_o_elems, a.status)) a.part_o[i] = v;
}
template <typename A>
__device__ __forceinline__ void put_part_ml(const A& a, long long i, float v) {
  if (in_bounds(i, a.part_ml_elems, a.status)) a.part_ml[i] = v;
}

// ---- programmatic dependent launch ---------------------------------------------------------------
// Every kernel of the library is launched so that it may start while its stream predecessor is
// still finishing. Each kernel first does set-up that touches no global data another kernel writes,
// then `pdl_wait` (the predecessor has completed and its memory is visible), then `pdl_trigger`
// (its own successor may now be scheduled), then its work. Triggering only after waiting keeps the
// usual guarantee: when a kernel starts, every kernel two or more launches back has completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- tcgen05 ------------------------------------------------------------------------------------

// Shared-memory matrix descriptor: start address, leading and stride byte offsets (16-byte units),
// descriptor version 1, swizzle layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout) << 61;
  return d;
}
constexpr uint32_t kSwizzle128 = 2;

// Instruction descriptor of kind::f16: f32 accumulator, A and B both f16 (fmt 0) or both bf16
// (fmt 1), A/B K-major (0) or MN-major (1), M and N.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, uint32_t fmt, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      :: "r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// the mbarrier receives one arrival when every tcgen05 operation issued so far by this thread is done
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

template <int NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "n"(NCOLS) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {     // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "n"(NCOLS) : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (warp w reads lanes 32*(w%4)..+31)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- element types ------------------------------------------------------------------------------

template <typename Tc> __device__ __forceinline__ float to_f32(Tc x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename Tc> __device__ __forceinline__ Tc from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// FP8 E4M3 storage: codes widened exactly to half, then to float (the scale is applied separately).
using fp8 = __nv_fp8_e4m3;
template <> __device__ __forceinline__ float to_f32<fp8>(fp8 x) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(x.__x, __NV_E4M3)));
}

// The type a query is used in: the cache dtype for float32 and 16-bit caches, float16 for fp8 caches
// (which float16 holds exactly).
template <typename Tc> struct QueryOf { using T = Tc; };
template <> struct QueryOf<fp8> { using T = __half; };

// A query element as the attention uses it: an F32 query meets a 16-bit (or fp8) cache rounded to its
// query type; a query given in that type is used as is.
template <typename Tc>
__device__ __forceinline__ float load_query(const void* q, kvc_dtype qt, long long i) {
  using Q = typename QueryOf<Tc>::T;
  if (qt == KVC_F32) {
    const float x = static_cast<const float*>(q)[i];
    if constexpr (sizeof(Q) == 2) return to_f32<Q>(from_f32<Q>(x));
    return x;
  }
  return to_f32<Q>(static_cast<const Q*>(q)[i]);
}

// ---- rotary positions ----------------------------------------------------------------------------
// Element e of a D-wide row turns with one partner: (e, e + D/2) for style 0, (e, e ^ 1) for style 1.
// Returns the partner, the pair index (the column of the cos/sin table) and whether e is the pair's
// second element: the first becomes x cos - y sin, the second x cos + y sin (y = the partner).
__device__ __forceinline__ int rope_partner(int e, int D, int style, int* pair, bool* second) {
  if (style == 0) {
    const int h = D >> 1;
    *second = e >= h;
    *pair = *second ? e - h : e;
    return *second ? e - h : e + h;
  }
  *second = (e & 1) != 0;
  *pair = e >> 1;
  return e ^ 1;
}
__device__ __forceinline__ float rope_rotate(float x, float y, float2 cs, bool second) {
  return second ? fmaf(x, cs.x, y * cs.y) : fmaf(x, cs.x, -(y * cs.y));
}

// A query element as given (float32, or the cache dtype widened), before any rounding.
template <typename Tc>
__device__ __forceinline__ float raw_query(const void* q, kvc_dtype qt, long long i) {
  using Q = typename QueryOf<Tc>::T;
  if (qt == KVC_F32) return static_cast<const float*>(q)[i];
  return to_f32<Q>(static_cast<const Q*>(q)[i]);
}

// Element e of the query row starting at element `row`, as the attention uses it: rotated to
// absolute position `pos` when the call applies RoPE, then (16-bit caches) rounded to the cache dtype.
template <typename Tc>
__device__ __forceinline__ float load_query_rot(const AttnArgs& a, long long row, int e, int pos) {
  if (a.rope.table == nullptr) return load_query<Tc>(a.q, a.q_dtype, row + e);
  int pair;
  bool second;
  const int pe = rope_partner(e, a.D, a.rope.style, &pair, &second);
  float r = rope_rotate(raw_query<Tc>(a.q, a.q_dtype, row + e), raw_query<Tc>(a.q, a.q_dtype, row + pe),
                        a.rope.table[static_cast<long long>(pos) * (a.D >> 1) + pair], second);
  using Q = typename QueryOf<Tc>::T;
  if constexpr (sizeof(Q) == 2) r = to_f32<Q>(from_f32<Q>(r));
  return r;
}

// Four consecutive query elements (element index i, a multiple of 4), as raw bits: a float4 of an F32
// query, or the low 8 bytes of a uint4 holding four elements of the query type. Nothing uses the value
// here, so a thread can issue all of its loads before the first one returns.
template <typename Tc>
__device__ __forceinline__ uint4 load_query4_raw(const void* q, kvc_dtype qt, long long i) {
  using Q = typename QueryOf<Tc>::T;
  if (qt == KVC_F32) return *reinterpret_cast<const uint4*>(static_cast<const float*>(q) + i);
  if constexpr (sizeof(Q) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const Q*>(q) + i);
    return make_uint4(w.x, w.y, 0u, 0u);
  } else {
    return *reinterpret_cast<const uint4*>(static_cast<const float*>(q) + i);
  }
}
// Those four elements in the MMA operand type M (a 16-bit type): an F32 query rounded once to M, which
// is its query-type rounding when M is the query type; a query already in the query type copied.
template <typename Tc, typename M>
__device__ __forceinline__ uint2 query4_to(uint4 raw, kvc_dtype qt) {
  using Q = typename QueryOf<Tc>::T;
  if (qt == KVC_F32 || sizeof(Q) != 2) {
    M v[4] = {from_f32<M>(__uint_as_float(raw.x)), from_f32<M>(__uint_as_float(raw.y)),
              from_f32<M>(__uint_as_float(raw.z)), from_f32<M>(__uint_as_float(raw.w))};
    return *reinterpret_cast<const uint2*>(v);
  }
  return make_uint2(raw.x, raw.y);
}

}  // namespace dev
}  // namespace kvc
