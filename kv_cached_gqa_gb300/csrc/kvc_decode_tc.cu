// Grouped-query attention over the KV cache on the 5th-generation tensor cores (tcgen05 + TMEM),
// for 16-bit caches with d_h = 64 or 128 and up to 16 query rows per K/V head (decode).
//
// What it computes ("KV cache, incremental decode, ...", §2.3; "Generation and the KV Cache",
// fence 3; "Heads, GQA and K/V cache", "Four queries, two sets of K/V"): for sequence b and K/V
// head g, each query row (t, h) of the group h = g*G .. g*G+G-1 attends over stored keys
// j <= s_b + t: softmax_j(q . k_j / sqrt(d_h)) weighted sum of v_j.
//
// How: the group's query rows are the N dimension of the MMAs (N = 16, padded with zero
// rows) and the keys are the M dimension (128 per tile), so one K/V tile read from HBM serves every
// query head of the group and nothing is repeated per head.
//   S^T [128 keys x N] = K_tile . Q^T       A = K tile (K-major, TMA 128-byte swizzle), B = Q^T
//   O^T [d_h x N]     += V_tile^T . P^T     A = V tile read MN-major, B = P^T (K-major)
// One CTA owns one (sequence, row tile, K/V head, key split). Roles:
//   warp 0     TMA producer: the split's K tiles, then its V tiles, through a ring of 2 to 6 stages;
//   warp 1     owns TMEM (256 columns) and issues every MMA from one thread;
//   warps 2-5  one thread per key (= TMEM lane): the scores of every K tile of the split stay in
//              TMEM, so the softmax over the split is exact (max, then exp2 and sum) with no
//              running rescale; the maxima are folded in tile by tile while K still streams; P is written to shared memory as a hi + lo pair of 16-bit values
//              (P ~ hi + lo to ~2^-16 relative), so the PV product keeps fp32-level accuracy;
//              then the epilogue: one thread per d reads O^T from TMEM.
// A unit with several splits writes (m, l, o) partials; the CTA that finishes its last split
// merges them (log-sum-exp) while they are in L2. Every wait is bounded (~1 s): a wait that gives
// up sets the device status word and the CTA skips the rest of its work, frees its TMEM and exits.
#include <type_traits>

#include "kvc_append.cuh"
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kTK = 128;                    // keys per tile = MMA M
constexpr int kBoxBytes = kTK * 128;        // one 64-element (128-byte) swizzled column box of a tile
constexpr int kTmemCols = 256;
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kMergeSplits = 31;            // splits merged through shared memory (else a running merge)

// Shared memory per CTA stays under ~110 KB so that two CTAs share an SM. 16-bit caches, d_h = 128: a
// 2-stage ring of 32 KB tiles and two P^T buffers (hi, lo), so that the softmax warps write P_{i+1}
// while the MMAs run PV_i (measured 2.5% faster than a 3-stage ring with one P^T buffer; a 3-stage ring
// with two no longer fits two CTAs). d_h = 64: 6 stages of 16 KB, one P^T buffer. fp8 caches
// (d_h = 128): a 2-stage ring of 16 KB fp8 tiles, plus two 32 KB float16 tiles the softmax warps widen
// the fp8 tiles into, alternately (the MMAs read those), so that one tile is widened while the MMAs
// work on the other.
template <int NR, int DH, bool F8>
struct Layout {
  static constexpr int kBoxes = DH / 64;                        // 64-element boxes per key row (MMA view)
  static constexpr int kTileBytes = kBoxes * kBoxBytes;         // a tile's K (or V) rows in 16 bits
  static constexpr int kStageBytes = F8 ? kTK * DH : kTileBytes;   // what TMA brings per tile
  static constexpr int kLoadBoxes = F8 ? DH / 128 : kBoxes;     // 128-byte column boxes TMA loads
  static constexpr int kLoadInner = F8 ? 128 : 64;              // elements per loaded box row
  static constexpr int kStages = (F8 || DH == 128) ? 2 : 96 * 1024 / kTileBytes;
  static constexpr int kConvBufs = F8 ? 2 : 0;
  static constexpr int kPBufs = (!F8 && DH == 128) ? 2 : 1;
  static constexpr int kQBytes = NR * DH * 2;                   // Q^T: atoms of NR rows x 128 B
  static constexpr int kPBytes = NR * 256;                      // one P^T operand (hi or lo): 128 keys
  static constexpr int kStageOff = 0;
  static constexpr int kConvOff = kStages * kStageBytes;        // fp8: the widened tile
  static constexpr int kQOff = kConvOff + kConvBufs * kTileBytes;
  static constexpr int kPOff = kQOff + kQBytes;                 // kPBufs buffers x (hi, lo)
  static constexpr int kCtlOff = kPOff + 2 * kPBufs * kPBytes;
  static constexpr int kSTiles = (kTmemCols - NR) / NR;         // S^T tiles that fit beside O^T
};

template <int NR, int DH, bool F8>
struct __align__(8) Ctl {
  using Lo = Layout<NR, DH, F8>;
  unsigned long long full[Lo::kStages], empty[Lo::kStages];
  unsigned long long p_full[Lo::kPBufs], p_empty[Lo::kPBufs];
  unsigned long long s_ready[Lo::kSTiles];                     // one per K tile, used once
  unsigned long long k_conv[2];                                // fp8: a K tile widened into buffer c
  unsigned long long o_full, done;
  unsigned long long cl_ready, cl_done;                        // cluster merge: partials in, reads done
  uint32_t tmem;
  int abort, last;
  float red[4][NR];
  float m[NR], l[NR];
};

// Dynamic shared memory per CTA. At least 80 KB, so that no more than two CTAs are ever resident on
// an SM: each holds 256 of the SM's 512 TMEM columns, and a third could wait forever on tcgen05.alloc.
template <int NR, int DH, bool F8>
constexpr size_t smem_bytes() {
  return (1024 + Layout<NR, DH, F8>::kCtlOff + sizeof(Ctl<NR, DH, F8>)) > 80 * 1024
             ? (1024 + Layout<NR, DH, F8>::kCtlOff + sizeof(Ctl<NR, DH, F8>)) : 80 * 1024;
}
static_assert(3 * 80 * 1024 > 228 * 1024, "three CTAs must not fit on one SM");
static_assert(2 * smem_bytes<16, 128, true>() + 2048 <= 228 * 1024, "two fp8 CTAs fit on one SM");
static_assert(2 * smem_bytes<16, 128, false>() + 2048 <= 228 * 1024, "two 16-bit CTAs fit on one SM");
static_assert(2 * smem_bytes<16, 64, false>() + 2048 <= 228 * 1024, "two 16-bit CTAs fit on one SM");
static_assert((2 * 16 * kMergeSplits + 16) * 4 <= 2 * Layout<16, 64, false>::kPBytes, "merge scratch fits the P buffer");

// Widen this thread's key row of an fp8 tile (128 keys x 128 one-byte codes, 128-byte swizzled as TMA
// wrote it) into the float16 tile the MMAs read (two 64-column 128-byte-swizzled boxes). Codes convert
// exactly; the layer's scale is applied to the scores and outputs instead.
__device__ __forceinline__ void widen_fp8_row(const unsigned char* src, unsigned char* dst, int row) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {                  // 16-byte chunk c = elements 16c .. 16c+15
    const uint4 w = *reinterpret_cast<const uint4*>(src + row * 128 + ((c ^ (row & 7)) << 4));
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i)         // 4 codes -> 2 float16 pairs, in element order
      asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
          " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
          : "=r"(h[2 * i]), "=r"(h[2 * i + 1]) : "r"(in[i]));
#pragma unroll
    for (int k = 0; k < 2; ++k) {                // float16 chunk 2c + k: box (2c + k) / 8, chunk (2c + k) % 8
      const int ch = 2 * c + k, box = ch >> 3, cc = ch & 7;
      *reinterpret_cast<uint4*>(dst + box * kBoxBytes + row * 128 + ((cc ^ (row & 7)) << 4)) =
          make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
    }
  }
}

// Byte offset of element (row, col) in an [rows][128] 16-bit matrix stored as two 128-byte-swizzled
// atoms of 64 columns (the layout TMA writes and the tensor cores read, K-major).
__device__ __forceinline__ uint32_t sw128(int rows, int row, int col) {
  const int atom = col >> 6, c = col & 63;
  return atom * (rows * 128) + row * 128 + ((((c >> 3) ^ (row & 7))) << 4) + (c & 7) * 2;
}

// The fused append's stores: rows [t0, t0 + n) of the chunk for (b, kvh), K and V, one 16-byte group per
// thread t of nt and pass. Kept out of line: it runs once per CTA at most, and inlined into the kernel it
// slowed the main loop of the fp8 instantiation by about 15%.
template <typename Tc, int DH>
__device__ __noinline__ void store_new_rows(const AppendArgs& app, int b, int kvh, int H_kv, int T, int t0, int n,
                                            int t, int nt) {
  constexpr int kGroups = DH * sizeof(Tc) / 16;             // 16-byte groups per stored row
  for (int e = t; e < n * 2 * kGroups; e += nt) {
    const int r = e / (2 * kGroups), c = e % (2 * kGroups);
    const long long row = (static_cast<long long>(b) * H_kv + kvh) * T + (t0 + r);
    app::append_group_any<Tc>(app, row, c % kGroups, c >= kGroups);
  }
}

// ---- thread-block clusters: the splits of one unit merged through distributed shared memory ---------
constexpr int kMaxCluster = 16;             // splits per unit the cluster merge takes (non-portable size)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// one arrival on an mbarrier of another CTA of the cluster, releasing this CTA's earlier writes
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
// bounded wait on a local mbarrier that other CTAs of the cluster arrive on (acquire at cluster scope)
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
    if (now_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Bounded wait that ignores the abort flag (used only to drain in-flight copies and MMAs).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  while (!mbar_try(bar, parity)) {
    if (now_ns() - t0 > kWaitLimitNs) return;
  }
}

// kCl: the plan gives every unit the same number of splits and the launch makes the splits of each
// (unit, K/V head) one thread-block cluster (item order puts them next to each other, so the cluster
// rank is the split); the splits' partials are merged through distributed shared memory by the CTA of
// split 0 instead of through L2 by the CTA that finishes last.
template <typename Tc, int NR, int DH, bool kCl>
__global__ void __launch_bounds__(kThreads, 2)
decode_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ SplitPlan plan,
                 const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  constexpr bool kF8 = std::is_same<Tc, fp8>::value;           // fp8 cache: tiles widened to float16
  using Tm = typename std::conditional<kF8, __half, Tc>::type;  // MMA operand type
  using Lo = Layout<NR, DH, kF8>;
  constexpr int kStages = Lo::kStages, kPBufs = Lo::kPBufs, kDh = DH, kTileBytes = Lo::kTileBytes;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl<NR, DH, kF8>* ctl = reinterpret_cast<Ctl<NR, DH, kF8>*>(sm + Lo::kCtlOff);
  const uint32_t s_stage = smem_u32(sm + Lo::kStageOff);
  const uint32_t s_q = smem_u32(sm + Lo::kQOff);
  unsigned char* p_base = sm + Lo::kPOff;
  const uint32_t s_p = smem_u32(p_base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kFmt = std::is_same<Tm, __nv_bfloat16>::value ? 1u : 0u;
  const uint32_t s_conv = smem_u32(sm + Lo::kConvOff);       // fp8: the widened tile

  // ---- which (unit, K/V head, split) this CTA owns --------------------------------------------
  const int item = blockIdx.x;
  int lo = 0, hi = plan.n_units - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (plan.prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int unit = lo;
  const int nsplit = (plan.prefix[unit + 1] - plan.prefix[unit]) / a.H_kv;
  const int rem = item - plan.prefix[unit];
  const int kvh = rem / nsplit, split = rem % nsplit;
  const int b = plan.unit_b[unit] / plan.n_rowtiles;
  const int rt = plan.unit_b[unit] % plan.n_rowtiles;
  const int row0 = rt * NR;
  const int nrows = min(NR, a.T * a.G - row0);

  // ---- set-up: TMEM, barriers, Q^T, zeroed P^T ------------------------------------------------
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&ctl->tmem));
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      // a stage is free again after the MMAs read it (16-bit) or the four softmax warps widened it (fp8)
      mbar_init(smem_u32(&ctl->empty[s]), kF8 ? kSoftmaxThreads / 32 : 1);
    }
    mbar_init(smem_u32(&ctl->k_conv[0]), kSoftmaxThreads / 32);
    mbar_init(smem_u32(&ctl->k_conv[1]), kSoftmaxThreads / 32);
    for (int s = 0; s < kPBufs; ++s) {
      mbar_init(smem_u32(&ctl->p_full[s]), kSoftmaxThreads / 32);
      mbar_init(smem_u32(&ctl->p_empty[s]), 1);
    }
    for (int s = 0; s < Lo::kSTiles; ++s) mbar_init(smem_u32(&ctl->s_ready[s]), 1);
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->done), 1);
    if (kCl) {
      mbar_init(smem_u32(&ctl->cl_ready), nsplit > 1 ? nsplit - 1 : 1);
      mbar_init(smem_u32(&ctl->cl_done), 1);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  // TMEM address and barriers visible to every warp
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // cluster merge: every CTA of the cluster has its barriers initialised before any arrives remotely
  // (every thread of every CTA of the cluster passes here, once, unconditionally)
  if constexpr (kCl) asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
  // from here on the lengths and the queries, which earlier kernels write, are read
  pdl_wait();
  pdl_trigger();
  const int s_b = a.lens[b] + a.delta - a.T;
  const int n_eff = s_b + (row0 + nrows - 1) / a.G + 1;
  const int chunk = split_chunk(n_eff, nsplit, kTK);    // near-equal, whole-tile splits of the unit's keys
  const int k_begin = split * chunk;
  const int k_end = min(k_begin + chunk, n_eff);
  const int nkt = (k_end - k_begin + kTK - 1) / kTK;
  const uint32_t tmem = ctl->tmem;
  const uint32_t tmem_o = tmem + (kTmemCols - NR);
  volatile int* abort_flag = &ctl->abort;
  // fused append: the new rows [s_b, s_b + T) that fall in this split, and the first K tile holding one
  // (-1: none)
  const int new_lo = max(s_b, k_begin), new_hi = min(s_b + a.T, k_end);
  const int i_new = (a.app.k_new != nullptr && new_lo < new_hi) ? (new_lo - k_begin) / kTK : -1;

  if (warp == 0) {
    // ---------------------------------- TMA producer (whole warp) -------------------------------
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
    }
    // fused append: this warp stores the split's new rows before it loads the first K tile holding one
    // (no other CTA loads those tiles): as soon as the ring is full, where it would otherwise wait for a
    // free stage, or earlier when that tile comes first
    int issued = 0;
    for (int i = 0; i < 2 * nkt; ++i) {
      const int st = i % kStages;
      const bool isv = i >= nkt;
      if (i == min(i_new, kStages)) {
        store_new_rows<Tc, DH>(a.app, b, kvh, a.H_kv, a.T, new_lo - s_b, new_hi - new_lo, lane, 32);
        // the stored rows are visible to this warp's tile loads (async proxy) before they are issued
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      const int y = k_begin + (isv ? i - nkt : i) * kTK;
      const TilePiece pc = tile_piece<kTK>(a, b, kvh, y, lane);   // a block-table read overlaps the wait
      const uint32_t full = smem_u32(&ctl->full[st]);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&ctl->empty[st]), ((i / kStages) & 1) ^ 1, abort_flag);
        if (ok) mbar_expect_tx(full, Lo::kStageBytes);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue_piece<kTK, Lo::kLoadBoxes, 128, Lo::kLoadInner>(pc, isv ? &tv : &tk, s_stage + st * Lo::kStageBytes,
                                                           full, lane);
      issued = i + 1;
    }
    // drain: the last copy issued into each stage has landed before the CTA can exit
    if (lane == 0)
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_drain(smem_u32(&ctl->full[i % kStages]), (i / kStages) & 1);
  } else {
    // ---- warps 1-5, while warp 0 already streams: Q^T and zeroed P^T ----------------------------
    if (a.rope.table != nullptr) {
      // rotated queries, four elements a step: each thread issues every query, partner and cos/sin load
      // of its share before it rotates any (one round of memory latency, not one per element); the
      // arithmetic is load_query_rot's, element for element
      using Q = typename QueryOf<Tc>::T;
      constexpr int kStagers = kThreads - 32, kQuads = NR * kDh / 4, kIter = (kQuads + kStagers - 1) / kStagers;
      constexpr int kHalf = kDh / 2;
      const bool style0 = a.rope.style == 0;                 // pairs (e, e + d_h/2); else (2i, 2i + 1)
      uint4 xr[kIter], yr[kIter];
      float4 c0[kIter], c1[kIter];
  #pragma unroll
      for (int k = 0; k < kIter; ++k) {
        const int i = (tid - 32) + k * kStagers, r = (4 * i) / kDh, d = (4 * i) % kDh;
        xr[k] = yr[k] = make_uint4(0u, 0u, 0u, 0u);
        c0[k] = c1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < kQuads && r < nrows) {
          const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
          const long long row = ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh;
          // (cos, sin) pairs of position s_b + t, two per float4
          const float4* cs = reinterpret_cast<const float4*>(a.rope.table + static_cast<long long>(s_b + t) * kHalf);
          xr[k] = load_query4_raw<Tc>(a.q, a.q_dtype, row + d);
          if (style0) {
            yr[k] = load_query4_raw<Tc>(a.q, a.q_dtype, row + (d < kHalf ? d + kHalf : d - kHalf));
            const int p0 = d < kHalf ? d : d - kHalf;        // pairs p0 .. p0 + 3
            c0[k] = cs[p0 / 2];
            c1[k] = cs[p0 / 2 + 1];
          } else {
            c0[k] = cs[d / 4];                              // pairs d/2 and d/2 + 1
          }
        }
      }
  #pragma unroll
      for (int k = 0; k < kIter; ++k) {
        const int i = (tid - 32) + k * kStagers, r = (4 * i) / kDh, d = (4 * i) % kDh;
        if (i < kQuads) {
          float x[4], y[4];
          if (a.q_dtype == KVC_F32) {
            x[0] = __uint_as_float(xr[k].x); x[1] = __uint_as_float(xr[k].y);
            x[2] = __uint_as_float(xr[k].z); x[3] = __uint_as_float(xr[k].w);
            y[0] = __uint_as_float(yr[k].x); y[1] = __uint_as_float(yr[k].y);
            y[2] = __uint_as_float(yr[k].z); y[3] = __uint_as_float(yr[k].w);
          } else {                                            // four 16-bit elements in the low 8 bytes
            const Q* xq = reinterpret_cast<const Q*>(&xr[k]);
            const Q* yq = reinterpret_cast<const Q*>(&yr[k]);
  #pragma unroll
            for (int c = 0; c < 4; ++c) { x[c] = to_f32<Q>(xq[c]); y[c] = to_f32<Q>(yq[c]); }
          }
          if (!style0) { y[0] = x[1]; y[1] = x[0]; y[2] = x[3]; y[3] = x[2]; }
          const float2 cs[4] = {make_float2(c0[k].x, c0[k].y), make_float2(style0 ? c0[k].z : c0[k].x, style0 ? c0[k].w : c0[k].y),
                                make_float2(style0 ? c1[k].x : c0[k].z, style0 ? c1[k].y : c0[k].w),
                                make_float2(style0 ? c1[k].z : c0[k].z, style0 ? c1[k].w : c0[k].w)};
          Tm out[4];
  #pragma unroll
          for (int c = 0; c < 4; ++c) {
            const bool second = style0 ? d >= kHalf : (c & 1) != 0;
            float v = rope_rotate(x[c], y[c], cs[c], second);
            if constexpr (sizeof(Q) == 2) v = to_f32<Q>(from_f32<Q>(v));
            out[c] = from_f32<Tm>(v);
          }
          *reinterpret_cast<uint2*>(sm + Lo::kQOff + sw128(NR, r, d)) = *reinterpret_cast<const uint2*>(out);
        }
      }
    } else {                                                  // four elements per load, all loads first
      constexpr int kStagers = kThreads - 32, kQuads = NR * kDh / 4, kIter = (kQuads + kStagers - 1) / kStagers;
      uint4 x[kIter];
#pragma unroll
      for (int k = 0; k < kIter; ++k) {
        const int i = (tid - 32) + k * kStagers, r = (4 * i) / kDh, d = (4 * i) % kDh;
        x[k] = make_uint4(0u, 0u, 0u, 0u);
        if (i < kQuads && r < nrows) {
          const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
          x[k] = load_query4_raw<Tc>(a.q, a.q_dtype, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh + d);
        }
      }
#pragma unroll
      for (int k = 0; k < kIter; ++k) {
        const int i = (tid - 32) + k * kStagers, r = (4 * i) / kDh, d = (4 * i) % kDh;
        if (i < kQuads) *reinterpret_cast<uint2*>(sm + Lo::kQOff + sw128(NR, r, d)) = query4_to<Tc, Tm>(x[k], a.q_dtype);
      }
    }
    for (int i = tid - 32; i < 2 * kPBufs * Lo::kPBytes / 16; i += kThreads - 32)
      reinterpret_cast<uint4*>(p_base)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async();
    named_sync(2, kThreads - 32);                             // Q^T and P^T ready for the MMA warp
    if (warp == 1) {
      // ---------------------------------- MMA issuer ----------------------------------------------
      if (lane == 0) {
        const uint32_t idesc_s = umma_idesc(kTK, NR, kFmt, 0, 0);
        const uint32_t idesc_o = umma_idesc(kDh, NR, kFmt, 1, 0);
        bool ok = true;
        for (int i = 0; i < nkt && ok; ++i) {                 // S^T_i = K_i . Q^T
          const int st = i % kStages;
          ok = kF8 ? mbar_wait(smem_u32(&ctl->k_conv[i & 1]), (i >> 1) & 1, abort_flag)
                   : mbar_wait(smem_u32(&ctl->full[st]), (i / kStages) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kt = kF8 ? s_conv + (i & 1) * kTileBytes : s_stage + st * kTileBytes;
  #pragma unroll
          for (int ks = 0; ks < kDh / 16; ++ks)
            umma_f16(tmem + i * NR,
                     umma_desc(kt + (ks >> 2) * kBoxBytes + (ks & 3) * 32, 16, 1024, kSwizzle128),
                     umma_desc(s_q + (ks >> 2) * (NR * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128),
                     idesc_s, ks > 0);
          if (!kF8) umma_commit(smem_u32(&ctl->empty[st]));
          umma_commit(smem_u32(&ctl->s_ready[i]));          // fp8: also "the widened tile is free"
        }
        for (int i = 0; i < nkt && ok; ++i) {                 // O^T += V_i^T . P_i^T (hi, then lo)
          const int ti = nkt + i, st = ti % kStages, pb = i % kPBufs;
          // fp8: p_full also means V_i has been widened
          ok = (kF8 || mbar_wait(smem_u32(&ctl->full[st]), (ti / kStages) & 1, abort_flag)) &&
               mbar_wait(smem_u32(&ctl->p_full[pb]), (i / kPBufs) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vt = kF8 ? s_conv + (ti & 1) * kTileBytes : s_stage + st * kTileBytes;
  #pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t pt = s_p + (pb * 2 + part) * Lo::kPBytes;
  #pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks)
              umma_f16(tmem_o,
                       umma_desc(vt + ks * 2048, kBoxBytes, 1024, kSwizzle128),
                       umma_desc(pt + (ks >> 2) * (NR * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128),
                       idesc_o, (i | part | ks) != 0);
          }
          if (!kF8) umma_commit(smem_u32(&ctl->empty[st]));
          umma_commit(smem_u32(&ctl->p_empty[pb]));          // fp8: also "the widened tile is free"
        }
        if (ok) umma_commit(smem_u32(&ctl->o_full));
        umma_commit(smem_u32(&ctl->done));
        mbar_drain(smem_u32(&ctl->done), 0);                  // every MMA done before TMEM is freed
      }
    } else {
      // ---------------------------------- softmax and epilogue ------------------------------------
      const int quad = warp & 3;                              // this warp's TMEM lane quadrant
      const int kslot = quad * 32 + lane;                     // key within a tile; d in the epilogue
      const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
      const int w4 = warp - 2;
      const float scale = kLog2e * rsqrtf(static_cast<float>(kDh)) * a.k_scale;   // k_scale: fp8 codes -> keys
      int trow[NR];
  #pragma unroll
      for (int r = 0; r < NR; ++r) trow[r] = (r < nrows) ? s_b + (row0 + r) / a.G : -1;   // last visible key

      // pass 1, overlapped with the K stream: fold each score tile into the row maxima as soon as
      // its MMAs complete
      bool ok = true;
      // fp8: widen ring tile `ti` (K tiles 0 .. nkt-1, then V tiles) into float16 buffer ti % 2, release
      // the ring stage and, for a K tile, tell the MMA warp
      auto widen = [&](int ti) -> bool {
        const int st = ti % kStages;
        if (!mbar_wait(smem_u32(&ctl->full[st]), (ti / kStages) & 1, abort_flag)) return false;
        widen_fp8_row(sm + Lo::kStageOff + st * Lo::kStageBytes, sm + Lo::kConvOff + (ti & 1) * kTileBytes, kslot);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&ctl->empty[st]));
          if (ti < nkt) mbar_arrive(smem_u32(&ctl->k_conv[ti & 1]));
        }
        return true;
      };
      if constexpr (kF8) {                                    // two K tiles ahead of the MMAs
        ok = widen(0);
        if (ok && nkt > 1) ok = widen(1);
      }
      float m_run[NR];
  #pragma unroll
      for (int r = 0; r < NR; ++r) m_run[r] = -INFINITY;
      for (int i = 0; i < nkt && ok; ++i) {
        ok = mbar_wait(smem_u32(&ctl->s_ready[i]), 0, abort_flag);
        if (!ok) break;
        // fp8: QK_i has read buffer i % 2, so K_{i+2} takes its place while QK_{i+1} runs
        if constexpr (kF8) {
          if (i + 2 < nkt && !(ok = widen(i + 2))) break;
        }
        tc_fence_after();
        float v[NR];
  #pragma unroll
        for (int c = 0; c < NR; c += 16) tmem_ld16(tmem + lane_base + i * NR + c, v + c);
        const int kabs = k_begin + i * kTK + kslot;
  #pragma unroll
        for (int r = 0; r < NR; ++r)
          if (kabs < k_end && kabs <= trow[r]) m_run[r] = fmaxf(m_run[r], v[r] * scale);
      }
      // row maxima over the split's keys: warp shuffles, then across the four warps
  #pragma unroll
      for (int r = 0; r < NR; ++r) {
  #pragma unroll
        for (int o = 16; o > 0; o >>= 1) m_run[r] = fmaxf(m_run[r], __shfl_xor_sync(0xffffffffu, m_run[r], o));
        if (lane == 0) ctl->red[w4][r] = m_run[r];
      }
      named_sync(1, kSoftmaxThreads);
  #pragma unroll
      for (int r = 0; r < NR; ++r)
        m_run[r] = fmaxf(fmaxf(ctl->red[0][r], ctl->red[1][r]), fmaxf(ctl->red[2][r], ctl->red[3][r]));
      named_sync(1, kSoftmaxThreads);

      float l_run[NR];
  #pragma unroll
      for (int r = 0; r < NR; ++r) l_run[r] = 0.f;
      // fp8: every QK is done (all S tiles were read above), so both buffers are free for V_0 and V_1
      if constexpr (kF8) {
        if (ok) ok = widen(nkt);
        if (ok && nkt > 1) ok = widen(nkt + 1);
      }
      for (int i = 0; i < nkt && ok; ++i) {
        const int pb = i % kPBufs;
        ok = mbar_wait(smem_u32(&ctl->p_empty[pb]), ((i / kPBufs) & 1) ^ 1, abort_flag);
        if (!ok) break;
        float v[NR];
  #pragma unroll
        for (int c = 0; c < NR; c += 16) tmem_ld16(tmem + lane_base + i * NR + c, v + c);
        const int kabs = k_begin + i * kTK + kslot;
        unsigned char* ph = p_base + (pb * 2) * Lo::kPBytes;
        unsigned char* pl = ph + Lo::kPBytes;
  #pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (r < nrows) {
            const float p = (kabs < k_end && kabs <= trow[r]) ? exp2f(v[r] * scale - m_run[r]) : 0.f;
            l_run[r] += p;
            const Tm h16 = from_f32<Tm>(p);
            const Tm l16 = from_f32<Tm>(p - to_f32<Tm>(h16));
            const uint32_t off = sw128(NR, r, kslot);
            *reinterpret_cast<Tm*>(ph + off) = h16;
            *reinterpret_cast<Tm*>(pl + off) = l16;
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[pb]));
        // fp8: PV_{i-1} is done (p_empty above), so V_{i+1} takes V_{i-1}'s buffer while PV_i runs
        if constexpr (kF8) {
          if (i >= 1 && i + 1 < nkt && !(ok = widen(nkt + i + 1))) break;
        }
      }
  #pragma unroll
      for (int r = 0; r < NR; ++r) {
  #pragma unroll
        for (int o = 16; o > 0; o >>= 1) l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], o);
        if (lane == 0) ctl->red[w4][r] = l_run[r];
      }
      named_sync(1, kSoftmaxThreads);
      if (tid == 64) {
  #pragma unroll
        for (int r = 0; r < NR; ++r) {
          ctl->m[r] = m_run[r];
          ctl->l[r] = ctl->red[0][r] + ctl->red[1][r] + ctl->red[2][r] + ctl->red[3][r];
        }
      }
      named_sync(1, kSoftmaxThreads);

      // ---- epilogue: thread = d; O^T row d from TMEM -----------------------------------------------
      ok = ok && mbar_wait(smem_u32(&ctl->o_full), 0, abort_flag);
      tc_fence_after();
      float o[NR];
  #pragma unroll
      for (int c = 0; c < NR; c += 16) tmem_ld16(tmem_o + lane_base + c, o + c);
      const bool aborted = *abort_flag != 0;
      // O^T row d sits in TMEM lane d for M = 128; for M = 64 in lane 32 * (d / 16) + d % 16, i.e. the
      // lower 16 lanes of each warp's quadrant
      const bool d_ok = DH == 128 || lane < 16;
      const int d = DH == 128 ? kslot : quad * 16 + (lane & 15);
      const long long item_row0 = static_cast<long long>(item) * NR;
      if (!aborted && d_ok) {
  #pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (r < nrows) {
            const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
            if (nsplit == 1) {
              put_out(a, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh + d, o[r] / ctl->l[r] * a.v_scale);
            } else if (kCl) {
              // this split's partial output stays in its own shared memory (the P buffers are free)
              reinterpret_cast<float*>(p_base)[r * kDh + d] = o[r];
            } else {
              put_part_o(a, (item_row0 + r) * kDh + d, o[r]);
              if (d == 0) {
                put_part_ml(a, (item_row0 + r) * 2, ctl->m[r]);
                put_part_ml(a, (item_row0 + r) * 2 + 1, ctl->l[r]);
              }
            }
          }
        }
      } else if (tid == 64) {
        atomicExch(a.status, kStatusTimeout);
      }
      if (kCl && nsplit > 1) {
        // ---- cluster merge: split 0 reads every split's (m, l, o) from its CTA's shared memory ----
        named_sync(1, kSoftmaxThreads);                       // this CTA's partial is in place
        const int t = tid - 64;
        if (cluster_rank() != 0) {
          if (t == 0) {
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            arrive_remote(map_rank(smem_u32(&ctl->cl_ready), 0));
            // stay (the teardown waits for this thread) until split 0 has read this CTA's memory
            if (!mbar_wait_cluster(smem_u32(&ctl->cl_done), 0)) atomicExch(a.status, kStatusTimeout);
          }
        } else {
          if (t == 0) ctl->last = mbar_wait_cluster(smem_u32(&ctl->cl_ready), 0) ? 1 : 0;
          named_sync(1, kSoftmaxThreads);
          if (ctl->last && !aborted) {
            const uint32_t m_at = smem_u32(&ctl->m[0]), l_at = smem_u32(&ctl->l[0]), o_at = smem_u32(p_base);
            for (int i = t; i < nrows * kDh; i += kSoftmaxThreads) {
              const int r = i / kDh, dd = i % kDh;
              // every split's (m, l, o) of this output in flight at once
              float ms[kMaxCluster], ls[kMaxCluster], os[kMaxCluster];
  #pragma unroll
              for (int sp = 0; sp < kMaxCluster; ++sp) {
                ms[sp] = -INFINITY;
                ls[sp] = 0.f;
                os[sp] = 0.f;
                if (sp < nsplit) {
                  ms[sp] = ld_cluster(map_rank(m_at + 4 * r, sp));
                  ls[sp] = ld_cluster(map_rank(l_at + 4 * r, sp));
                  os[sp] = ld_cluster(map_rank(o_at + 4 * (r * kDh + dd), sp));
                }
              }
              float mx = -INFINITY;
  #pragma unroll
              for (int sp = 0; sp < kMaxCluster; ++sp)
                if (ls[sp] > 0.f) mx = fmaxf(mx, ms[sp]);
              float lsum = 0.f, acc = 0.f;
  #pragma unroll
              for (int sp = 0; sp < kMaxCluster; ++sp) {
                if (ls[sp] > 0.f) {
                  const float w = exp2f(ms[sp] - mx);
                  lsum = fmaf(w, ls[sp], lsum);
                  acc = fmaf(w, os[sp], acc);
                }
              }
              const int gr = row0 + r, tq = gr / a.G, g = gr % a.G;
              put_out(a, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + tq) * kDh + dd,
                      acc / lsum * a.v_scale);
            }
          } else if (t == 0) {
            atomicExch(a.status, kStatusTimeout);
          }
          named_sync(1, kSoftmaxThreads);                     // every read of the other CTAs is done
          if (t == 0)
            for (int sp = 1; sp < nsplit; ++sp) arrive_remote(map_rank(smem_u32(&ctl->cl_done), sp));
        }
      } else if (nsplit > 1) {
        // ---- the CTA that finishes a unit's last split merges its partials -----------------------
        __threadfence();
        named_sync(1, kSoftmaxThreads);
        int* counter = a.counters + unit * a.H_kv + kvh;
        if (tid == 64) ctl->last = (atomicAdd(counter, 1) == nsplit - 1);
        named_sync(1, kSoftmaxThreads);
        if (ctl->last) {
          __threadfence();
          const long long first_row = static_cast<long long>(plan.prefix[unit] + kvh * nsplit) * NR;
          if (nsplit <= kMergeSplits) {
            // every split's (m, l) at once into the P buffer (free now), then one set of weights per
            // row, then independent loads of the partial outputs
            float* wm = reinterpret_cast<float*>(p_base);            // [NR][kMergeSplits] m, then weight
            float* wl = wm + NR * kMergeSplits;                      // [NR][kMergeSplits] l
            float* linv = wl + NR * kMergeSplits;                    // [NR]
            for (int i = tid - 64; i < nrows * nsplit; i += kSoftmaxThreads) {
              const int r = i / nsplit, sp = i % nsplit;
              const long long row = first_row + static_cast<long long>(sp) * NR + r;
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
            if (d_ok) {
              // every row's partial of a split in one batch of independent loads (no store between
              // them), the output stores after the last split
              float acc[NR];
  #pragma unroll
              for (int r = 0; r < NR; ++r) acc[r] = 0.f;
              for (int sp = 0; sp < nsplit; ++sp) {
                const float* src = a.part_o + (first_row + static_cast<long long>(sp) * NR) * kDh + d;
                float x[NR];
  #pragma unroll
                for (int r = 0; r < NR; ++r) x[r] = r < nrows ? __ldcg(src + r * kDh) : 0.f;
  #pragma unroll
                for (int r = 0; r < NR; ++r) acc[r] = fmaf(wm[r * kMergeSplits + sp], x[r], acc[r]);
              }
              if (!aborted) {
  #pragma unroll
                for (int r = 0; r < NR; ++r) {
                  if (r < nrows) {
                    const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
                    put_out(a, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh + d,
                            acc[r] * linv[r] * a.v_scale);
                  }
                }
              }
            }
          } else {
            for (int r = 0; r < nrows && d_ok; ++r) {
              float m = -INFINITY, l = 0.f, acc = 0.f;
              for (int sp = 0; sp < nsplit; ++sp) {
                const long long row = first_row + static_cast<long long>(sp) * NR + r;
                const float ms = __ldcg(a.part_ml + row * 2), ls = __ldcg(a.part_ml + row * 2 + 1);
                if (!(ls > 0.f)) continue;
                const float mn = fmaxf(m, ms);
                const float c_old = exp2f(m - mn), c_new = exp2f(ms - mn);
                l = l * c_old + ls * c_new;
                acc = acc * c_old + __ldcg(a.part_o + row * kDh + d) * c_new;
                m = mn;
              }
              const int gr = row0 + r, t = gr / a.G, g = gr % a.G;
              if (!aborted) put_out(a, ((static_cast<long long>(b) * a.H_q + kvh * a.G + g) * a.T + t) * kDh + d, acc / l * a.v_scale);
            }
          }
          if (tid == 64) *counter = 0;
        }
      }
    }

  }  // warps 1-5

  // ---- teardown: every TMEM access is complete before the allocating warp frees it -------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

// Cluster sizes past the portable 8 (up to 16) allowed for a kernel, once per device.
template <auto Kernel>
cudaError_t ensure_cluster_size() {
  static unsigned long long done = 0;          // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0;
  if (bit && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && bit) __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
  return e;
}

template <typename Tc, int NR, int DH>
cudaError_t run(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk, const CUtensorMap* tv,
                int cluster, cudaStream_t st) {
  constexpr bool kF8 = std::is_same<Tc, fp8>::value;
  const size_t smem = smem_bytes<NR, DH, kF8>();
  if constexpr (!kF8) {
    if (cluster > 1) {
      auto kern = decode_tc_kernel<Tc, NR, DH, true>;
      cudaError_t e = ensure_smem_limit<decode_tc_kernel<Tc, NR, DH, true>>(smem);
      if (e == cudaSuccess) e = ensure_cluster_size<decode_tc_kernel<Tc, NR, DH, true>>();
      if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.n_items);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, kern, a, p, *tk, *tv);
        if (e == cudaSuccess) return e;
      }
      (void)cudaGetLastError();                // a cluster that cannot be placed: the L2 merge instead
    }
  }
  auto kern = decode_tc_kernel<Tc, NR, DH, false>;
  cudaError_t e = ensure_smem_limit<decode_tc_kernel<Tc, NR, DH, false>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.n_items), dim3(kThreads), smem, st, a, p, *tk, *tv);
}

}  // namespace

// Up to 16 query rows per K/V head (decode, G * T <= 16); longer chunks run on the chunk kernel,
// which measured faster from 32 rows on.
bool decode_tc_shape(kvc_dtype dt, int D, int rows, int* rows_per_tile, int* tile_keys, int* max_tiles) {
  if (rows > 16) return false;
  if (dt == KVC_FP8_E4M3 ? D != 128 : ((dt != KVC_F16 && dt != KVC_BF16) || (D != 64 && D != 128))) return false;
  *rows_per_tile = 16;
  *tile_keys = kTK;
  *max_tiles = Layout<16, 128, false>::kSTiles;
  return true;
}

cudaError_t launch_decode_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                             const CUtensorMap* tv, int cluster, cudaStream_t st) {
  if (p.rows_per_tile != 16) return cudaErrorInvalidValue;
  if (cluster > kMaxCluster) cluster = 0;
  if (a.cache_dtype == KVC_FP8_E4M3)
    return a.D == 128 ? run<fp8, 16, 128>(a, p, tk, tv, 0, st) : cudaErrorInvalidValue;
  if (a.D == 128)
    return a.cache_dtype == KVC_BF16 ? run<__nv_bfloat16, 16, 128>(a, p, tk, tv, cluster, st)
                                     : run<__half, 16, 128>(a, p, tk, tv, cluster, st);
  return a.cache_dtype == KVC_BF16 ? run<__nv_bfloat16, 16, 64>(a, p, tk, tv, cluster, st)
                                   : run<__half, 16, 64>(a, p, tk, tv, cluster, st);
}

}  // namespace kvc
