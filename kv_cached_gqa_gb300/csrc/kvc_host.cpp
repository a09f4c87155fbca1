// Host side of the C ABI (include/kvc.h): argument validation, the host mirrors of the per-layer
// fill counts and committed lengths, device allocation, TMA descriptors and the split-K planner.
//
// Bookkeeping follows "KV cache, incremental decode, ...", §2.3 (each layer keeps its own fill
// count; the committed length moves once per forward, after the last layer) and §2.4 (truncate
// sets every layer's count; nothing is freed or copied). Every call validates against the host
// mirrors first and mutates nothing on error (§4, test_update_copies_and_checks).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "kvc_internal.h"

namespace {
thread_local std::string g_err;
}  // namespace

namespace kvc {

int fail(kvc_handle h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  g_err = buf;
  return code;
}

}  // namespace kvc

namespace {

using kvc::fail;

int cuda_fail(kvc_handle h, cudaError_t e, const char* what) {
  return fail(h, KVC_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_dtype(int t) { return t == KVC_F32 || t == KVC_F16 || t == KVC_BF16 || t == KVC_FP8_E4M3; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(std::string* err) {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return nullptr;
  }
  fn = reinterpret_cast<EncodeTiledFn>(p);
  return fn;
}

// ---- device buffers the handle owns --------------------------------------------------------------
// A debug build (KVC_DEBUG_BOUNDS) allocates kGuard more bytes on each side of every buffer and fills
// them with kGuardByte; kvc_debug_check_guards compares them with that byte, so a kernel that wrote
// past either end of a library buffer (the store, the lengths, the workspace, the counters, the block
// table, the rotary table) is caught after the fact. The guards keep the payload 256-byte aligned.
#ifdef KVC_DEBUG_BOUNDS
constexpr size_t kGuard = 64 * 1024;
#else
constexpr size_t kGuard = 0;
#endif
constexpr unsigned char kGuardByte = 0xA5;

cudaError_t dev_alloc(kvc_handle h, void** p, size_t bytes, const char* what, cudaStream_t st, bool async) {
  void* base = nullptr;
  cudaError_t e = async ? cudaMallocAsync(&base, bytes + 2 * kGuard, st) : cudaMalloc(&base, bytes + 2 * kGuard);
  if (e != cudaSuccess) return e;
  unsigned char* payload = static_cast<unsigned char*>(base) + kGuard;
  if (kGuard) {
    e = cudaMemsetAsync(base, kGuardByte, kGuard, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(payload + bytes, kGuardByte, kGuard, st);
    if (e != cudaSuccess) {
      if (async) cudaFreeAsync(base, st); else cudaFree(base);
      return e;
    }
  }
  h->bufs.push_back({base, payload, bytes, what});
  *p = payload;
  return cudaSuccess;
}

// Free a buffer dev_alloc gave out (stream-ordered when `async`); NULL is a no-op.
void dev_free(kvc_handle h, void* p, cudaStream_t st, bool async) {
  if (!p) return;
  for (size_t i = 0; i < h->bufs.size(); ++i) {
    if (h->bufs[i].payload != p) continue;
    if (async) cudaFreeAsync(h->bufs[i].base, st); else cudaFree(h->bufs[i].base);
    h->bufs.erase(h->bufs.begin() + static_cast<long>(i));
    return;
  }
}

int init_device_state(kvc_handle h, cudaStream_t st) {
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaDeviceGetAttribute");
  e = dev_alloc(h, reinterpret_cast<void**>(&h->d_lens), sizeof(int32_t) * h->B, "lengths", st, false);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMalloc(lengths)");
  e = dev_alloc(h, reinterpret_cast<void**>(&h->d_status), sizeof(int), "status word", st, false);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMalloc(status)");
  e = dev_alloc(h, reinterpret_cast<void**>(&h->d_counters), sizeof(int) * kvc::kMaxUnits * h->H, "merge counters",
                st, false);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMalloc(counters)");
  e = cudaMemsetAsync(h->d_lens, 0, sizeof(int32_t) * h->B, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->d_status, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->d_counters, 0, sizeof(int) * kvc::kMaxUnits * h->H, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemsetAsync");
  if (h->paged) {                                   // every logical block starts unmapped (-1)
    const size_t tb = sizeof(int32_t) * h->table.size();
    e = dev_alloc(h, reinterpret_cast<void**>(&h->d_table), tb, "block table", st, false);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaMalloc(block table)");
    e = cudaMemsetAsync(h->d_table, 0xFF, tb, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemsetAsync(block table)");
  }
  if (h->latent) {                                 // maps for the tensor-core latent attention, 64 x 64 boxes
    if (kvc::mla_tc_shape(h->dtype, h->D, h->Dv)) {
      std::string err;
      const long long planes = static_cast<long long>(h->L) * h->B;
      if (!kvc::encode_store_map(&h->tmap_k_tc, h->k, h->dtype, h->D, h->max_len, planes, kvc::kMlaTcKeys, &err) ||
          !kvc::encode_store_map(&h->tmap_v_tc, h->v, h->dtype, h->Dv, h->max_len, planes, kvc::kMlaTcKeys, &err))
        return fail(h, KVC_E_CUDA, "%s", err.c_str());
      h->has_tc = true;
    }
    return KVC_OK;
  }
  int rows = 0;
  kvc::splitk_shape(h->dtype, h->D, 1, &rows, &h->split_tile_keys);
  std::string err;
  const kvc::Paging pg = kvc_paging(h);
  const long long planes = static_cast<long long>(h->L) * (h->paged ? h->n_blocks : h->B) * h->H;
  const int plane_rows = h->paged ? h->block : h->max_len;
  const int split_box = kvc::paged_box_rows(pg, h->split_tile_keys);
  if (!kvc::encode_store_map(&h->tmap_k_split, h->k, h->dtype, h->D, plane_rows, planes, split_box, &err) ||
      !kvc::encode_store_map(&h->tmap_v_split, h->v, h->dtype, h->D, plane_rows, planes, split_box, &err))
    return fail(h, KVC_E_CUDA, "%s", err.c_str());
  int tc_rows = 0, tc_tile = 0, tc_tiles = 0;
  if (kvc::decode_tc_shape(h->dtype, h->D, 1, &tc_rows, &tc_tile, &tc_tiles)) {
    const int tc_box = kvc::paged_box_rows(pg, tc_tile);
    if (!kvc::encode_store_map(&h->tmap_k_tc, h->k, h->dtype, h->D, plane_rows, planes, tc_box, &err) ||
        !kvc::encode_store_map(&h->tmap_v_tc, h->v, h->dtype, h->D, plane_rows, planes, tc_box, &err))
      return fail(h, KVC_E_CUDA, "%s", err.c_str());
    h->has_tc = true;
  }
  return KVC_OK;
}

void release(kvc_handle h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (const auto& buf : h->bufs) cudaFree(buf.base);     // the store too, when the library owns it
  delete h;
}

int check_sizes(int L, int B, int H_kv, int d_h, int max_len, int dtype) {
  if (L < 1 || B < 1 || H_kv < 1 || max_len < 1)
    return fail(nullptr, KVC_E_INVAL, "sizes must be positive (L=%d B=%d H_kv=%d max_len=%d)", L, B, H_kv, max_len);
  if (!valid_dtype(dtype)) return fail(nullptr, KVC_E_INVAL, "unknown dtype %d", dtype);
  if (B > KVC_MAX_BATCH) return fail(nullptr, KVC_E_INVAL, "B=%d exceeds KVC_MAX_BATCH", B);
  if (d_h != 32 && d_h != 64 && d_h != 128)
    return fail(nullptr, KVC_E_UNSUPPORTED, "d_h=%d: kernels exist for 32, 64 and 128", d_h);
  if (dtype == KVC_FP8_E4M3 && d_h == 32)
    return fail(nullptr, KVC_E_UNSUPPORTED, "fp8 caches need d_h 64 or 128 (rows of at least 64 bytes)");
  if (static_cast<long long>(L) * B * H_kv >= (1LL << 31) || max_len >= (1 << 30))
    return fail(nullptr, KVC_E_INVAL, "cache too large for 32-bit tile coordinates");
  return KVC_OK;
}

kvc_handle new_handle(int L, int B, int H_kv, int d_h, int max_len, kvc_dtype dtype) {
  kvc_handle h = new (std::nothrow) kvc_cache();
  if (!h) return nullptr;
  h->L = L; h->B = B; h->H = H_kv; h->D = d_h; h->Dv = d_h; h->max_len = max_len; h->dtype = dtype;
  h->fill.assign(static_cast<size_t>(L) * B, 0);
  h->lens.assign(B, 0);
  h->k_scale.assign(L, 1.f);
  h->v_scale.assign(L, 1.f);
  return h;
}

// Bytes of one store: [L, B, H, max_len, width], or the pool [L, n_blocks, H, block, width]; the first
// store (K, or the latent) has width D, the second (V, or the RoPE key) width Dv.
size_t store_bytes(kvc_handle h, bool second = false) {
  const size_t per_layer = h->paged ? static_cast<size_t>(h->n_blocks) * h->block : static_cast<size_t>(h->B) * h->max_len;
  return static_cast<size_t>(h->L) * per_layer * h->H * (second ? h->Dv : h->D) * kvc::itemsize(h->dtype);
}

// ---- paged pool bookkeeping ------------------------------------------------------------------------
// Free blocks live in a min-heap, so the lowest-numbered free block is always handed out first; a
// sequence's logical blocks 0 .. held-1 are mapped. Allocation happens at append, for the blocks the
// layer's new fill reaches; truncate returns every block wholly past the new length.
int blocks_for(kvc_handle h, long long rows) { return static_cast<int>((rows + h->block - 1) >> h->block_shift); }

int pop_free(kvc_handle h) {
  std::pop_heap(h->free_heap.begin(), h->free_heap.end(), std::greater<int32_t>());
  const int v = h->free_heap.back();
  h->free_heap.pop_back();
  return v;
}

void push_free(kvc_handle h, int v) {
  h->free_heap.push_back(v);
  std::push_heap(h->free_heap.begin(), h->free_heap.end(), std::greater<int32_t>());
}

// Enqueue table edits (slot, value) in launches of at most kMaxTableEdits.
cudaError_t send_edits(kvc_handle h, const std::vector<std::pair<int32_t, int32_t>>& edits, cudaStream_t st) {
  static thread_local kvc::TableEdits e;    // 8 KB: keep it off the stack
  for (size_t i = 0; i < edits.size(); i += kvc::kMaxTableEdits) {
    e.n = static_cast<int>(std::min<size_t>(kvc::kMaxTableEdits, edits.size() - i));
    for (int j = 0; j < e.n; ++j) {
      e.slot[j] = edits[i + j].first;
      e.value[j] = edits[i + j].second;
    }
    const cudaError_t r = kvc::launch_table_edits(h->d_table, e, st);
    if (r != cudaSuccess) return r;
    h->launches += 1;
  }
  return cudaSuccess;
}

// Map the blocks that `layer`'s fill reaches after T more rows. All or nothing: on error no block is
// taken and the host table is unchanged.
int paged_grow(kvc_handle h, int layer, int T, cudaStream_t st) {
  long long need = 0;
  for (int b = 0; b < h->B; ++b) {
    const int nb = blocks_for(h, static_cast<long long>(h->fill[static_cast<size_t>(layer) * h->B + b]) + T);
    if (nb > h->held[b]) need += nb - h->held[b];
  }
  if (need == 0) return KVC_OK;
  if (need > static_cast<long long>(h->free_heap.size()))
    return fail(h, KVC_E_CAPACITY, "block pool exhausted: the append needs %lld more blocks of %d positions, "
                "%zu of %d are free", need, h->block, h->free_heap.size(), h->n_blocks);
  std::vector<std::pair<int32_t, int32_t>>& edits = h->edit_scratch;
  edits.clear();
  for (int b = 0; b < h->B; ++b) {
    const int nb = blocks_for(h, static_cast<long long>(h->fill[static_cast<size_t>(layer) * h->B + b]) + T);
    for (int i = h->held[b]; i < nb; ++i) edits.push_back({b * h->max_blocks + i, pop_free(h)});
  }
  const cudaError_t e = send_edits(h, edits, st);
  if (e != cudaSuccess) {
    for (const auto& ed : edits) push_free(h, ed.second);
    return cuda_fail(h, e, "block table launch");
  }
  for (const auto& ed : edits) h->table[ed.first] = ed.second;
  for (int b = 0; b < h->B; ++b)
    h->held[b] = std::max(h->held[b], blocks_for(h, static_cast<long long>(h->fill[static_cast<size_t>(layer) * h->B + b]) + T));
  return KVC_OK;
}

// Grow the handle's split workspace (stream-ordered) to at least `need` floats.
int ensure_workspace(kvc_handle h, size_t need, cudaStream_t st) {
  if (need <= h->work_floats) return KVC_OK;
  const size_t grow = need + need / 4;
  float* p = nullptr;
  cudaError_t e = dev_alloc(h, reinterpret_cast<void**>(&p), grow * sizeof(float), "split workspace", st, true);
  if (e != cudaSuccess) return fail(h, KVC_E_NOMEM, "workspace cudaMallocAsync: %s", cudaGetErrorString(e));
  dev_free(h, h->work, st, true);
  h->work = p;
  h->work_floats = grow;
  return KVC_OK;
}

// Uniform difference between one layer's fills and the committed lengths.
int layer_delta(kvc_handle h, int layer, int* delta) {
  const int d0 = h->fill[static_cast<size_t>(layer) * h->B] - h->lens[0];
  for (int b = 1; b < h->B; ++b)
    if (h->fill[static_cast<size_t>(layer) * h->B + b] - h->lens[b] != d0)
      return fail(h, KVC_E_STATE, "layer %d: appended rows differ between sequences", layer);
  *delta = d0;
  return KVC_OK;
}

}  // namespace

namespace kvc {

bool encode_store_map(CUtensorMap* map, void* base, kvc_dtype dt, int D, int max_len,
                      long long planes, int box_rows, std::string* err) {
  EncodeTiledFn fn = encode_fn(err);
  if (!fn) return false;
  const int es = itemsize(dt);
  const int row_bytes = D * es;
  const int span = row_bytes >= 128 ? 128 : 64;
  const CUtensorMapDataType ty = dt == KVC_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dt == KVC_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : dt == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_UINT8;   // fp8 codes
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(max_len),
                              static_cast<cuuint64_t>(planes)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(row_bytes) * max_len};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(span / es), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, ty, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    *err = buf;
    return false;
  }
  return true;
}

// ---- kernel choice and work plan ------------------------------------------------------------------
// Tensor cores serve 16-bit caches with d_h = 128: the split decode kernel for up to 16 query rows
// per K/V head; beyond that the chunk kernels, the one-CTA-per-SM form for up to 128 rows (verify
// chunks, one CTA per (sequence, K/V head)) and the two-CTAs-per-SM form with split keys for longer
// chunks (prefill). Everything else runs on the CUDA-core split-K kernel. For the split kernels, the total key work W = H_kv * sum_u n_u (n_u =
// keys visible to unit u) is cut into about k waves of resident CTAs (two per SM); each unit's keys
// are split into near-equal chunks of about W / (k * slots) keys, at most what one CTA can hold, and
// units are ordered longest chunk first so the hardware scheduler packs the last wave tightly.
int plan_attention(kvc_handle h, int T, int H_q, SplitPlan* plan, AttnPlan* out, std::string* err) {
  const int G = H_q / h->H;
  const int R = T * G;
  int rpt = 0, tile = 0, max_tiles = 0;
  AttnKernel kind;
  if (h->has_tc && decode_tc_shape(h->dtype, h->D, R, &rpt, &tile, &max_tiles)) {
    kind = AttnKernel::DecodeTC;
  } else if (h->has_tc && R > 16 && prefill_tc_shape(h->dtype, h->D, &rpt)) {
    if (R <= rpt) {
      kind = AttnKernel::ChunkTC;
    } else {
      kind = AttnKernel::PrefillTC;                         // 128-row units; its online softmax
      tile = 128;                                           // takes any split length
      max_tiles = 1 << 16;
    }
  } else {
    if (!splitk_shape(h->dtype, h->D, R, &rpt, &tile)) {
      *err = "no attention kernel for this d_h";
      return KVC_E_UNSUPPORTED;
    }
    max_tiles = (8192 / (2 * rpt)) / tile;                  // the kernel's weight buffer
    kind = AttnKernel::SplitK;
  }
  const int n_rt = (R + rpt - 1) / rpt;
  if (static_cast<long long>(h->B) * n_rt > kMaxUnits) {
    *err = "batch x row tiles exceeds the planner's limit of 2048 units";
    return KVC_E_UNSUPPORTED;
  }
  const int n_units = h->B * n_rt;
  plan->n_units = n_units;
  plan->rows_per_tile = rpt;
  plan->n_rowtiles = n_rt;
  std::vector<long long>& n_eff = h->plan_n_eff;
  std::vector<int>& nsplit = h->plan_nsplit;
  std::vector<std::pair<int, int>>& order = h->plan_order;
  n_eff.resize(n_units);
  nsplit.resize(n_units);
  order.resize(n_units);
  long long total_keys = 0;
  for (int b = 0; b < h->B; ++b)
    for (int rt = 0; rt < n_rt; ++rt) {
      const int t_max = std::min(T - 1, ((rt + 1) * rpt - 1) / G);
      n_eff[b * n_rt + rt] = static_cast<long long>(h->lens[b]) + t_max + 1;
      total_keys += n_eff[b * n_rt + rt];
    }
  auto longest_first = [](const std::pair<int, int>& x, const std::pair<int, int>& y) { return x.first > y.first; };
  out->kernel = kind;
  out->rows_per_tile = rpt;
  if (kind == AttnKernel::ChunkTC) {
    // one CTA per (unit, K/V head). Longest sequences first, and a sequence's row tiles together
    // (longest tile first): the CTAs resident at any time then share a few sequences' K/V, which
    // stays in L2 instead of being re-read from HBM by each row tile
    for (int u = 0; u < n_units; ++u) order[u] = {static_cast<int>(std::min<long long>(n_eff[u], 1 << 30)), u};
    std::stable_sort(order.begin(), order.end(), [&](const std::pair<int, int>& x, const std::pair<int, int>& y) {
      const int bx = x.second / n_rt, by = y.second / n_rt;
      if (h->lens[bx] != h->lens[by]) return h->lens[bx] > h->lens[by];
      if (bx != by) return bx < by;
      return x.first > y.first;
    });
    for (int i = 0; i < n_units; ++i) plan->unit_b[i] = order[i].second;
    plan->n_items = n_units * h->H;
    plan->split_keys = n_units ? order[0].first : 0;
    plan->prefix[0] = 0;
    out->workspace_floats = 0;
    out->counters = 0;
    return KVC_OK;
  }
  const int cmax = max_tiles * tile;
  const long long slots = 2LL * h->num_sms;
  const long long work = total_keys * h->H;
  // splits of about w keys: a unit of n keys takes round(n / w) near-equal whole-tile splits, at most
  // cmax keys each; `ns = ceil(n / chunk)` keeps the kernels' recomputed chunk and leaves no split empty
  auto splits_for = [&](long long n, long long w_, int* chunk_out) {
    int ns = static_cast<int>(std::max(1LL, (n + w_ / 2) / w_));
    while (kvc::split_chunk(static_cast<int>(n), ns, tile) > cmax) ++ns;
    const int chunk = kvc::split_chunk(static_cast<int>(n), ns, tile);
    *chunk_out = chunk;
    return static_cast<int>((n + chunk - 1) / chunk);
  };
  long long w = h->split_keys_override;
  if (w <= 0) {
    const long long waves = std::max(1LL, (work + slots * 1536 - 1) / (slots * 1536));
    w = (work + waves * slots - 1) / (waves * slots);
    // at least 4 tiles per split when the work spans several waves (shorter splits cost more in
    // set-up and merging than they return); down to one tile when it fits one wave, where the time is
    // the latency of each CTA's chain of tiles
    w = std::max<long long>(w, (waves > 1 ? 4LL : 1LL) * tile);
    // the per-unit rounding can add CTAs past the whole waves aimed at, leaving a short last wave:
    // take the smallest split size (binary search, the CTA count falls as it grows) whose CTAs fit
    const long long target = waves * slots;
    auto items_at = [&](long long w_) {
      long long n_items = 0;
      int c = 0;
      for (int u = 0; u < n_units; ++u) n_items += static_cast<long long>(h->H) * splits_for(n_eff[u], w_, &c);
      return n_items;
    };
    if (items_at(w) > target) {
      long long lo_w = w, hi_w = std::max<long long>(w, cmax);
      if (items_at(hi_w) <= target) {
        while (hi_w - lo_w > 1) {
          const long long mid = (lo_w + hi_w) / 2;
          if (items_at(mid) <= target) hi_w = mid; else lo_w = mid;
        }
        w = hi_w;
      }
    }
  }
  w = std::max(1LL, w);
  for (int u = 0; u < n_units; ++u) {
    int chunk = 0;
    nsplit[u] = splits_for(n_eff[u], w, &chunk);             // whole tiles, as the kernels recompute it
    order[u] = {chunk, u};
  }
  if (kind == AttnKernel::PrefillTC) {
    // a sequence's row tiles together (longest sequences first, then longest chunk): the CTAs
    // resident at a time then read a few sequences' K/V, which stays in L2 for all their row tiles
    std::stable_sort(order.begin(), order.end(), [&](const std::pair<int, int>& x, const std::pair<int, int>& y) {
      const int bx = x.second / n_rt, by = y.second / n_rt;
      if (h->lens[bx] != h->lens[by]) return h->lens[bx] > h->lens[by];
      if (bx != by) return bx < by;
      return x.first > y.first;
    });
  } else {
    std::stable_sort(order.begin(), order.end(), longest_first);
  }
  long long items = 0;
  int max_chunk = 0;
  plan->prefix[0] = 0;
  for (int i = 0; i < n_units; ++i) {
    const int u = order[i].second;
    items += static_cast<long long>(h->H) * nsplit[u];
    if (items >= (1LL << 31)) {
      *err = "too many work items";
      return KVC_E_UNSUPPORTED;
    }
    plan->prefix[i + 1] = static_cast<int32_t>(items);
    plan->unit_b[i] = u;                                    // = b * n_rowtiles + rt
    max_chunk = std::max(max_chunk, order[i].first);
  }
  plan->n_items = static_cast<int>(items);
  plan->split_keys = max_chunk;
  out->workspace_floats = plan->n_items > n_units * h->H ? splitk_workspace_floats(*plan, h->D) : 0;
  out->counters = static_cast<size_t>(n_units) * h->H;
  // one wave of the decode kernel with the same number of splits for every unit (16-bit caches): the
  // splits of each (unit, K/V head) merge as one thread-block cluster, through distributed shared
  // memory, which takes the merge's L2 round trips off the end of the launch
  out->cluster = 0;
  if (kind == AttnKernel::DecodeTC && h->dtype != KVC_FP8_E4M3 && items <= slots && nsplit[0] > 1 &&
      nsplit[0] <= 16 && std::all_of(nsplit.begin(), nsplit.begin() + n_units, [&](int x) { return x == nsplit[0]; }))
    out->cluster = nsplit[0];
  return KVC_OK;
}

cudaError_t launch_attention(const AttnPlan& ap, const AttnArgs& a, const SplitPlan& p, kvc_handle h,
                             cudaStream_t st) {
  switch (ap.kernel) {
    case AttnKernel::DecodeTC: return launch_decode_tc(a, p, &h->tmap_k_tc, &h->tmap_v_tc, ap.cluster, st);
    case AttnKernel::ChunkTC: return launch_chunk_tc(a, p, &h->tmap_k_tc, &h->tmap_v_tc, st);
    case AttnKernel::PrefillTC: return launch_prefill_tc(a, p, &h->tmap_k_tc, &h->tmap_v_tc, st);
    case AttnKernel::SplitK: return launch_splitk(a, p, &h->tmap_k_split, &h->tmap_v_split, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvc

namespace kvc {

int check_attention_call(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int s, int T, int H_q,
                         const float* out, bool rope) {
  if (h->latent) return fail(h, KVC_E_INVAL, "a latent cache is read by mla_cached_attn");
  if (rope && !h->d_rope) return fail(h, KVC_E_STATE, "no rotary table: call kvc_set_rope first");
  if (layer < 0 || layer >= h->L) return fail(h, KVC_E_INVAL, "layer %d out of range [0, %d)", layer, h->L);
  if (T < 1) return fail(h, KVC_E_INVAL, "T=%d must be >= 1", T);
  if (!q || !out) return fail(h, KVC_E_INVAL, "null q/out");
  if (H_q < 1 || H_q % h->H) return fail(h, KVC_E_INVAL, "H_q=%d must be a positive multiple of H_kv=%d", H_q, h->H);
  if (!query_dtype_ok(h->dtype, q_dtype))
    return fail(h, KVC_E_INVAL, "query dtype %d: F32 or the cache dtype (F16 for an fp8 cache)", q_dtype);
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(h, KVC_E_INVAL, "q/out must be 16-byte aligned");
  if (s < KVC_COMMITTED) return fail(h, KVC_E_INVAL, "s=%d", s);
  for (int b = 0; b < h->B; ++b) {
    if (s >= 0 && h->lens[b] != s)
      return fail(h, KVC_E_STATE, "s=%d but sequence %d has committed length %d", s, b, h->lens[b]);
    if (h->fill[static_cast<size_t>(layer) * h->B + b] != h->lens[b] + T)
      return fail(h, KVC_E_STATE, "layer %d holds %d rows of sequence %d; attention needs s_b + T = %d "
                  "(append the chunk to this layer first)", layer, h->fill[static_cast<size_t>(layer) * h->B + b],
                  b, h->lens[b] + T);
  }
  return KVC_OK;
}

}  // namespace kvc

extern "C" {

int kvc_create(kvc_handle* out, int L, int B, int H_kv, int d_h, int max_len, kvc_dtype dtype,
               void* stream) {
  if (!out) return fail(nullptr, KVC_E_INVAL, "null output handle");
  *out = nullptr;
  int rc = check_sizes(L, B, H_kv, d_h, max_len, dtype);
  if (rc) return rc;
  kvc_handle h = new_handle(L, B, H_kv, d_h, max_len, dtype);
  if (!h) return fail(nullptr, KVC_E_NOMEM, "host allocation failed");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = store_bytes(h), bytes2 = store_bytes(h, true);
  cudaError_t e = dev_alloc(h, &h->k, bytes, "K store", st, false);
  if (e == cudaSuccess) e = dev_alloc(h, &h->v, bytes2, "V store", st, false);
  h->owns_store = true;
  if (e != cudaSuccess) {
    rc = fail(nullptr, KVC_E_NOMEM, "cudaMalloc of %zu + %zu bytes failed: %s", bytes, bytes2, cudaGetErrorString(e));
    cudaGetLastError();
    release(h);
    return rc;
  }
  e = cudaMemsetAsync(h->k, 0, bytes, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->v, 0, bytes2, st);
  if (e != cudaSuccess) {
    rc = cuda_fail(nullptr, e, "cudaMemsetAsync(store)");
    release(h);
    return rc;
  }
  rc = init_device_state(h, st);
  if (rc) {
    g_err = h->err;
    release(h);
    return rc;
  }
  *out = h;
  return KVC_OK;
}

int kvc_create_external(kvc_handle* out, int L, int B, int H_kv, int d_h, int max_len,
                        kvc_dtype dtype, void* k_store, void* v_store, void* stream) {
  if (!out) return fail(nullptr, KVC_E_INVAL, "null output handle");
  *out = nullptr;
  int rc = check_sizes(L, B, H_kv, d_h, max_len, dtype);
  if (rc) return rc;
  if (!k_store || !v_store) return fail(nullptr, KVC_E_INVAL, "null store pointer");
  if (!aligned(k_store, 256) || !aligned(v_store, 256))
    return fail(nullptr, KVC_E_INVAL, "store pointers must be 256-byte aligned");
  kvc_handle h = new_handle(L, B, H_kv, d_h, max_len, dtype);
  if (!h) return fail(nullptr, KVC_E_NOMEM, "host allocation failed");
  h->k = k_store;
  h->v = v_store;
  rc = init_device_state(h, static_cast<cudaStream_t>(stream));
  if (rc) {
    g_err = h->err;
    release(h);
    return rc;
  }
  *out = h;
  return KVC_OK;
}

int kvc_create_paged(kvc_handle* out, int L, int B, int H_kv, int d_h, int max_len, int block_size,
                     int n_blocks, kvc_dtype dtype, void* k_pool, void* v_pool, void* stream) {
  if (!out) return fail(nullptr, KVC_E_INVAL, "null output handle");
  *out = nullptr;
  int rc = check_sizes(L, B, H_kv, d_h, max_len, dtype);
  if (rc) return rc;
  if (block_size < 16 || block_size > (1 << 20) || (block_size & (block_size - 1)))
    return fail(nullptr, KVC_E_INVAL, "block_size=%d must be a power of two in [16, 2^20]", block_size);
  if (n_blocks < 1) return fail(nullptr, KVC_E_INVAL, "n_blocks=%d must be positive", n_blocks);
  const long long max_blocks = (static_cast<long long>(max_len) + block_size - 1) / block_size;
  if (static_cast<long long>(L) * n_blocks * H_kv >= (1LL << 31) || static_cast<long long>(B) * max_blocks >= (1LL << 31))
    return fail(nullptr, KVC_E_INVAL, "pool or block table too large for 32-bit tile coordinates");
  if ((k_pool == nullptr) != (v_pool == nullptr))
    return fail(nullptr, KVC_E_INVAL, "pass both pool pointers or neither");
  if (k_pool && (!aligned(k_pool, 256) || !aligned(v_pool, 256)))
    return fail(nullptr, KVC_E_INVAL, "pool pointers must be 256-byte aligned");
  kvc_handle h = new_handle(L, B, H_kv, d_h, max_len, dtype);
  if (!h) return fail(nullptr, KVC_E_NOMEM, "host allocation failed");
  h->paged = true;
  h->block = block_size;
  h->block_shift = __builtin_ctz(static_cast<unsigned>(block_size));
  h->n_blocks = n_blocks;
  h->max_blocks = static_cast<int>(max_blocks);
  h->table.assign(static_cast<size_t>(B) * h->max_blocks, -1);
  h->held.assign(B, 0);
  h->free_heap.resize(n_blocks);
  for (int i = 0; i < n_blocks; ++i) h->free_heap[i] = i;   // ascending order is already a min-heap
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = store_bytes(h);
  if (k_pool) {
    h->k = k_pool;
    h->v = v_pool;
  } else {
    h->owns_store = true;
    cudaError_t e = dev_alloc(h, &h->k, bytes, "K pool", st, false);
    if (e == cudaSuccess) e = dev_alloc(h, &h->v, bytes, "V pool", st, false);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->k, 0, bytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->v, 0, bytes, st);
    if (e != cudaSuccess) {
      rc = fail(nullptr, KVC_E_NOMEM, "pool allocation of 2 x %zu bytes failed: %s", bytes, cudaGetErrorString(e));
      cudaGetLastError();
      release(h);
      return rc;
    }
  }
  rc = init_device_state(h, st);
  if (rc) {
    g_err = h->err;
    release(h);
    return rc;
  }
  *out = h;
  return KVC_OK;
}

int kvc_block_table(kvc_handle h, int32_t* table_host, int32_t* n_free_host) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (!h->paged) return fail(h, KVC_E_INVAL, "not a paged cache");
  if (table_host) memcpy(table_host, h->table.data(), sizeof(int32_t) * h->table.size());
  if (n_free_host) *n_free_host = static_cast<int32_t>(h->free_heap.size());
  return KVC_OK;
}

int kvc_create_latent(kvc_handle* out, int L, int B, int r, int d_rope, int max_len, kvc_dtype dtype,
                      void* c_store, void* kr_store, void* stream) {
  if (!out) return fail(nullptr, KVC_E_INVAL, "null output handle");
  *out = nullptr;
  if (L < 1 || B < 1 || r < 1 || d_rope < 1 || max_len < 1)
    return fail(nullptr, KVC_E_INVAL, "sizes must be positive (L=%d B=%d r=%d d_R=%d max_len=%d)", L, B, r, d_rope, max_len);
  if (dtype != KVC_F32 && dtype != KVC_F16 && dtype != KVC_BF16)
    return fail(nullptr, KVC_E_INVAL, "latent caches store F32, F16 or BF16 (dtype %d)", dtype);
  if (B > KVC_MAX_BATCH) return fail(nullptr, KVC_E_INVAL, "B=%d exceeds KVC_MAX_BATCH", B);
  if (r % 16 || d_rope % 16 || r > 1024 || d_rope > 256 || r + d_rope > 1152)
    return fail(nullptr, KVC_E_UNSUPPORTED, "r=%d, d_R=%d: multiples of 16 with r <= 1024, d_R <= 256, r + d_R <= 1152",
                r, d_rope);
  if (static_cast<long long>(L) * B * max_len >= (1LL << 31) || max_len >= (1 << 30))
    return fail(nullptr, KVC_E_INVAL, "cache too large");
  if ((c_store == nullptr) != (kr_store == nullptr)) return fail(nullptr, KVC_E_INVAL, "pass both stores or neither");
  if (c_store && (!aligned(c_store, 256) || !aligned(kr_store, 256)))
    return fail(nullptr, KVC_E_INVAL, "store pointers must be 256-byte aligned");
  kvc_handle h = new_handle(L, B, 1, r, max_len, dtype);
  if (!h) return fail(nullptr, KVC_E_NOMEM, "host allocation failed");
  h->Dv = d_rope;
  h->latent = true;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = KVC_OK;
  if (c_store) {
    h->k = c_store;
    h->v = kr_store;
  } else {
    const size_t b1 = store_bytes(h), b2 = store_bytes(h, true);
    h->owns_store = true;
    cudaError_t e = dev_alloc(h, &h->k, b1, "latent store", st, false);
    if (e == cudaSuccess) e = dev_alloc(h, &h->v, b2, "RoPE-key store", st, false);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->k, 0, b1, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->v, 0, b2, st);
    if (e != cudaSuccess) {
      rc = fail(nullptr, KVC_E_NOMEM, "latent store allocation failed: %s", cudaGetErrorString(e));
      cudaGetLastError();
      release(h);
      return rc;
    }
  }
  rc = init_device_state(h, st);
  if (rc) {
    g_err = h->err;
    release(h);
    return rc;
  }
  *out = h;
  return KVC_OK;
}

// Work plan of a latent attention call: units = (sequence, 16-row tile of the T * H query rows), each
// cut into near-equal whole-tile key splits sized so the launch fills whole waves (two CTAs per SM),
// longest first. Returns the workspace floats the partials need (0 when no unit splits).
static int plan_mla(kvc_handle h, int T, int H, int tile, int ctas_per_sm, kvc::SplitPlan* plan,
                    size_t* work_floats, std::string* err) {
  const int R = T * H, rpt = kvc::kMlaRows;
  const int n_rt = (R + rpt - 1) / rpt;
  if (static_cast<long long>(h->B) * n_rt > kvc::kMaxUnits) {
    *err = "batch x row tiles exceeds the planner's limit of 2048 units";
    return KVC_E_UNSUPPORTED;
  }
  const int n_units = h->B * n_rt;
  plan->n_units = n_units;
  plan->rows_per_tile = rpt;
  plan->n_rowtiles = n_rt;
  std::vector<std::pair<int, int>>& order = h->plan_order;
  std::vector<int>& nsplit = h->plan_nsplit;
  order.resize(n_units);
  nsplit.resize(n_units);
  long long total = 0;
  for (int b = 0; b < h->B; ++b)
    for (int rt = 0; rt < n_rt; ++rt) total += h->lens[b] + std::min(T - 1, ((rt + 1) * rpt - 1) / H) + 1;
  const long long slots = static_cast<long long>(ctas_per_sm) * h->num_sms;
  const long long waves = std::max(1LL, (total + slots * 1024 - 1) / (slots * 1024));
  const long long w = std::max<long long>(4LL * tile, (total + waves * slots - 1) / (waves * slots));
  for (int b = 0; b < h->B; ++b)
    for (int rt = 0; rt < n_rt; ++rt) {
      const int u = b * n_rt + rt;
      const int n = h->lens[b] + std::min(T - 1, ((rt + 1) * rpt - 1) / H) + 1;
      int ns = static_cast<int>(std::max(1LL, (n + w / 2) / w));
      const int chunk = kvc::split_chunk(n, ns, tile);
      ns = (n + chunk - 1) / chunk;
      nsplit[u] = ns;
      order[u] = {chunk, u};
    }
  std::stable_sort(order.begin(), order.end(),
                   [](const std::pair<int, int>& x, const std::pair<int, int>& y) { return x.first > y.first; });
  long long items = 0;
  plan->prefix[0] = 0;
  for (int i = 0; i < n_units; ++i) {
    items += nsplit[order[i].second];
    plan->prefix[i + 1] = static_cast<int32_t>(items);
    plan->unit_b[i] = order[i].second;
  }
  plan->n_items = static_cast<int>(items);
  plan->split_keys = n_units ? order[0].first : 0;
  *work_floats = items > n_units ? static_cast<size_t>(items) * rpt * (h->D + 2) : 0;
  return KVC_OK;
}

int mla_cached_attn(kvc_handle h, const void* q_lat, const void* q_rope, kvc_dtype q_dtype, int layer, int s,
                    int T, int H, float scale, float* out, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (!h->latent) return fail(h, KVC_E_INVAL, "mla_cached_attn reads a latent cache (kvc_create_latent)");
  if (layer < 0 || layer >= h->L) return fail(h, KVC_E_INVAL, "layer %d out of range [0, %d)", layer, h->L);
  if (T < 1 || H < 1) return fail(h, KVC_E_INVAL, "T=%d and H=%d must be >= 1", T, H);
  if (!q_lat || !q_rope || !out) return fail(h, KVC_E_INVAL, "null q_lat/q_rope/out");
  if (!kvc::query_dtype_ok(h->dtype, q_dtype)) return fail(h, KVC_E_INVAL, "query dtype %d: F32 or the cache dtype", q_dtype);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(h, KVC_E_INVAL, "scale must be positive and finite");
  if (!aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(out, 16))
    return fail(h, KVC_E_INVAL, "q_lat/q_rope/out must be 16-byte aligned");
  if (s < KVC_COMMITTED) return fail(h, KVC_E_INVAL, "s=%d", s);
  for (int b = 0; b < h->B; ++b) {
    if (s >= 0 && h->lens[b] != s)
      return fail(h, KVC_E_STATE, "s=%d but sequence %d has committed length %d", s, b, h->lens[b]);
    if (h->fill[static_cast<size_t>(layer) * h->B + b] != h->lens[b] + T)
      return fail(h, KVC_E_STATE, "layer %d holds %d rows of sequence %d; attention needs s_b + T = %d",
                  layer, h->fill[static_cast<size_t>(layer) * h->B + b], b, h->lens[b] + T);
  }
  static thread_local kvc::SplitPlan plan;
  size_t work_floats = 0;
  std::string perr;
  const bool tc = h->has_tc && kvc::mla_tc_shape(h->dtype, h->D, h->Dv);
  const int prc = tc ? plan_mla(h, T, H, kvc::kMlaTcKeys, 1, &plan, &work_floats, &perr)
                     : plan_mla(h, T, H, kvc::mla_tile_keys(h->dtype), 2, &plan, &work_floats, &perr);
  if (prc) return fail(h, prc, "%s", perr.c_str());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (work_floats) {
    const int wrc = ensure_workspace(h, work_floats, st);
    if (wrc) return wrc;
  }
  kvc::MlaArgs a{};
  a.q_lat = q_lat; a.q_rope = q_rope; a.q_dtype = q_dtype; a.out = out;
  a.part_o = h->work;
  a.part_ml = h->work ? h->work + static_cast<size_t>(plan.n_items) * kvc::kMlaRows * h->D : nullptr;
  a.counters = h->d_counters;
  a.lens = h->d_lens; a.status = h->d_status;
  a.c_store = h->k; a.kr_store = h->v;
  a.layer = layer; a.B = h->B; a.H = H; a.T = T; a.r = h->D; a.dR = h->Dv; a.max_len = h->max_len;
  a.scale = scale; a.cache_dtype = h->dtype;
  a.out_elems = static_cast<long long>(h->B) * H * T * h->D;
  a.part_o_elems = h->work ? static_cast<long long>(plan.n_items) * kvc::kMlaRows * h->D : 0;
  a.part_ml_elems = h->work ? static_cast<long long>(plan.n_items) * kvc::kMlaRows * 2 : 0;
  cudaError_t e = tc ? kvc::launch_mla_tc(a, plan, &h->tmap_k_tc, &h->tmap_v_tc, st) : kvc::launch_mla(a, plan, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "latent attention launch");
  h->launches += 1;
  return KVC_OK;
}

int kvc_destroy(kvc_handle h) {
  release(h);
  return KVC_OK;
}

// The checks of an append (nothing changes): on success *delta is the layer's fill minus the committed
// lengths (uniform over the batch).
static int check_append(kvc_handle h, int layer, const void* k_new, const void* v_new, kvc_dtype in_dtype,
                        int T, bool rope, int* delta_out) {
  if (rope && h->latent) return fail(h, KVC_E_UNSUPPORTED, "fused RoPE is for K/V caches");
  if (rope && !h->d_rope) return fail(h, KVC_E_STATE, "no rotary table: call kvc_set_rope first");
  if (layer < 0 || layer >= h->L) return fail(h, KVC_E_INVAL, "layer %d out of range [0, %d)", layer, h->L);
  if (T < 1) return fail(h, KVC_E_INVAL, "T=%d must be >= 1", T);
  if (!k_new || !v_new) return fail(h, KVC_E_INVAL, "null k_new/v_new");
  if (!kvc::input_dtype_ok(h->dtype, in_dtype))
    return fail(h, KVC_E_INVAL, "input dtype %d: F32 or the cache dtype (F32, F16 or BF16 for an fp8 cache)", in_dtype);
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(h, KVC_E_INVAL, "k_new/v_new must be 16-byte aligned");
  int delta = 0;
  const int rc = layer_delta(h, layer, &delta);
  if (rc) return rc;
  for (int b = 0; b < h->B; ++b) {
    const long long end = static_cast<long long>(h->fill[static_cast<size_t>(layer) * h->B + b]) + T;
    if (end > h->max_len)
      return fail(h, KVC_E_CAPACITY, "sequence %d: %lld positions exceed max_len=%d", b, end, h->max_len);
  }
  *delta_out = delta;
  return KVC_OK;
}

// What the append kernel (or the decode kernel's fused append) needs to store a [B, H, T, D] chunk at
// the layer's fill.
static kvc::AppendArgs append_args(kvc_handle h, int layer, const void* k_new, const void* v_new,
                                   kvc_dtype in_dtype, int T, int delta, bool rope) {
  kvc::AppendArgs a{};
  a.k_store = h->k; a.v_store = h->v; a.k_new = k_new; a.v_new = v_new; a.lens = h->d_lens;
  a.layer = layer; a.B = h->B; a.H = h->H; a.D = h->D; a.Dv = h->Dv; a.T = T; a.max_len = h->max_len;
  a.delta = delta; a.cache_dtype = h->dtype; a.in_dtype = in_dtype;
  a.pg = kvc_paging(h);
  if (rope) {
    a.rope.table = h->d_rope;
    a.rope.style = h->rope_style;
  }
  a.k_scale = h->k_scale[layer];
  a.v_scale = h->v_scale[layer];
  a.k_rows = static_cast<long long>(store_bytes(h) / (static_cast<size_t>(h->D) * kvc::itemsize(h->dtype)));
  a.v_rows = static_cast<long long>(store_bytes(h, true) / (static_cast<size_t>(h->Dv) * kvc::itemsize(h->dtype)));
  a.status = h->d_status;
  return a;
}

static int append_impl(kvc_handle h, int layer, const void* k_new, const void* v_new, kvc_dtype in_dtype,
                       int T, bool rope, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  int delta = 0;
  int rc = check_append(h, layer, k_new, v_new, in_dtype, T, rope, &delta);
  if (rc) return rc;
  if (h->paged) {
    rc = paged_grow(h, layer, T, static_cast<cudaStream_t>(stream));
    if (rc) return rc;
  }
  const kvc::AppendArgs a = append_args(h, layer, k_new, v_new, in_dtype, T, delta, rope);
  cudaError_t e = kvc::launch_append(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "append launch");
  h->launches += 1;
  for (int b = 0; b < h->B; ++b) h->fill[static_cast<size_t>(layer) * h->B + b] += T;
  return KVC_OK;
}

int kvc_append(kvc_handle h, int layer, const void* k_new, const void* v_new, kvc_dtype in_dtype,
               int T, void* stream) {
  return append_impl(h, layer, k_new, v_new, in_dtype, T, false, stream);
}

int kvc_append_rope(kvc_handle h, int layer, const void* k_new, const void* v_new, kvc_dtype in_dtype,
                    int T, void* stream) {
  return append_impl(h, layer, k_new, v_new, in_dtype, T, true, stream);
}

int kvc_set_rope(kvc_handle h, double base, kvc_rope_style style, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (h->latent) return fail(h, KVC_E_UNSUPPORTED, "fused RoPE is for K/V caches");
  if (!(base > 1.0) || base > 1e12) return fail(h, KVC_E_INVAL, "RoPE base %g must be in (1, 1e12]", base);
  if (style != KVC_ROPE_HALF && style != KVC_ROPE_INTERLEAVED) return fail(h, KVC_E_INVAL, "RoPE style %d", style);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!h->d_rope) {
    const size_t bytes = sizeof(float2) * static_cast<size_t>(h->max_len) * (h->D / 2);
    cudaError_t e = dev_alloc(h, reinterpret_cast<void**>(&h->d_rope), bytes, "rotary table", st, false);
    if (e != cudaSuccess) {
      h->d_rope = nullptr;
      return fail(h, KVC_E_NOMEM, "rotary table (%zu bytes): %s", bytes, cudaGetErrorString(e));
    }
  }
  static thread_local kvc::RopeTheta th;
  for (int i = 0; i < h->D / 2; ++i) th.theta[i] = std::pow(base, -2.0 * i / h->D);
  cudaError_t e = kvc::launch_rope_table(h->d_rope, h->max_len, h->D, th, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "rotary table launch");
  h->launches += 1;
  h->rope_style = style;
  return KVC_OK;
}

int kvc_set_kv_scales(kvc_handle h, const float* k_scale, const float* v_scale) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (h->dtype != KVC_FP8_E4M3) return fail(h, KVC_E_INVAL, "scales belong to fp8 caches");
  if (!k_scale || !v_scale) return fail(h, KVC_E_INVAL, "null scales");
  for (int l = 0; l < h->L; ++l)
    if (!(k_scale[l] > 0.f) || !(v_scale[l] > 0.f) || !std::isfinite(k_scale[l]) || !std::isfinite(v_scale[l]))
      return fail(h, KVC_E_INVAL, "layer %d: scales must be positive and finite", l);
  for (int32_t f : h->fill)
    if (f != 0) return fail(h, KVC_E_STATE, "scales are fixed while the cache holds rows");
  for (int l = 0; l < h->L; ++l) {
    h->k_scale[l] = k_scale[l];
    h->v_scale[l] = v_scale[l];
  }
  return KVC_OK;
}

int kvc_commit(kvc_handle h, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  for (int l = 1; l < h->L; ++l)
    for (int b = 0; b < h->B; ++b)
      if (h->fill[static_cast<size_t>(l) * h->B + b] != h->fill[b])
        return fail(h, KVC_E_STATE, "commit: layer %d holds %d rows of sequence %d, layer 0 holds %d",
                    l, h->fill[static_cast<size_t>(l) * h->B + b], b, h->fill[b]);
  int delta = 0;
  int rc = layer_delta(h, 0, &delta);
  if (rc) return rc;
  if (delta != 0) {
    cudaError_t e = kvc::launch_lens_add(h->d_lens, h->B, delta, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "commit launch");
    h->launches += 1;
  }
  for (int b = 0; b < h->B; ++b) h->lens[b] = h->fill[b];
  return KVC_OK;
}

int kvc_truncate_ragged(kvc_handle h, const int32_t* n, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (!n) return fail(h, KVC_E_INVAL, "null lengths");
  for (int b = 0; b < h->B; ++b) {
    if (n[b] < 0) return fail(h, KVC_E_INVAL, "sequence %d: negative length %d", b, n[b]);
    if (n[b] > h->lens[b])
      return fail(h, KVC_E_STATE, "sequence %d: truncate to %d beyond committed length %d", b, n[b], h->lens[b]);
  }
  std::vector<std::pair<int32_t, int32_t>>& edits = h->edit_scratch;
  edits.clear();
  if (h->paged)                                       // blocks wholly past the new length go back
    for (int b = 0; b < h->B; ++b)
      for (int i = blocks_for(h, n[b]); i < h->held[b]; ++i) edits.push_back({b * h->max_blocks + i, -1});
  cudaError_t e = send_edits(h, edits, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = kvc::launch_lens_set(h->d_lens, h->B, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "truncate launch");
  h->launches += 1;
  for (const auto& ed : edits) {
    push_free(h, h->table[ed.first]);
    h->table[ed.first] = -1;
  }
  if (h->paged)
    for (int b = 0; b < h->B; ++b) h->held[b] = std::min(h->held[b], blocks_for(h, n[b]));
  for (int b = 0; b < h->B; ++b) {
    h->lens[b] = n[b];
    for (int l = 0; l < h->L; ++l) h->fill[static_cast<size_t>(l) * h->B + b] = n[b];
  }
  return KVC_OK;
}

int kvc_truncate(kvc_handle h, int n, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  std::unique_ptr<int32_t[]> v(new (std::nothrow) int32_t[h->B]);
  if (!v) return fail(h, KVC_E_NOMEM, "host allocation failed");
  for (int b = 0; b < h->B; ++b) v[b] = n;
  return kvc_truncate_ragged(h, v.get(), stream);
}

int kvc_set_lengths(kvc_handle h, const int32_t* n, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (!n) return fail(h, KVC_E_INVAL, "null lengths");
  if (h->paged) return fail(h, KVC_E_UNSUPPORTED, "a paged cache takes rows only through kvc_append");
  for (int b = 0; b < h->B; ++b)
    if (n[b] < 0 || n[b] > h->max_len)
      return fail(h, KVC_E_INVAL, "sequence %d: length %d outside [0, max_len=%d]", b, n[b], h->max_len);
  cudaError_t e = kvc::launch_lens_set(h->d_lens, h->B, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "set-lengths launch");
  h->launches += 1;
  for (int b = 0; b < h->B; ++b) {
    h->lens[b] = n[b];
    for (int l = 0; l < h->L; ++l) h->fill[static_cast<size_t>(l) * h->B + b] = n[b];
  }
  return KVC_OK;
}

int kvc_seq_len(kvc_handle h, int layer, int32_t* out) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (!out) return fail(h, KVC_E_INVAL, "null output");
  if (layer < -1 || layer >= h->L) return fail(h, KVC_E_INVAL, "layer %d out of range", layer);
  for (int b = 0; b < h->B; ++b)
    out[b] = layer < 0 ? h->lens[b] : h->fill[static_cast<size_t>(layer) * h->B + b];
  return KVC_OK;
}

int kvc_positions(kvc_handle h, int T, int32_t* out, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (T < 1 || !out) return fail(h, KVC_E_INVAL, "T must be >= 1 and out non-null");
  cudaError_t e = kvc::launch_positions(h->d_lens, h->B, T, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "positions launch");
  h->launches += 1;
  return KVC_OK;
}

size_t kvc_nbytes(kvc_handle h) { return h ? store_bytes(h) + store_bytes(h, true) : 0; }

int kvc_layer_ptrs(kvc_handle h, int layer, void** k, void** v) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (layer < 0 || layer >= h->L || !k || !v) return fail(h, KVC_E_INVAL, "bad layer or null output");
  *k = static_cast<char*>(h->k) + store_bytes(h) / h->L * layer;
  *v = static_cast<char*>(h->v) + store_bytes(h, true) / h->L * layer;
  return KVC_OK;
}

// Plan and launch the attention of a call whose checks passed. With `fused` the chunk has not been
// stored yet: the tensor-core decode kernel stores it itself (one launch); any other kernel gets the
// append kernel launched first (two launches).
static int attn_launch(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int T, int H_q, float* out,
                       bool rope, const kvc::AppendArgs* fused, void* stream) {
  static thread_local kvc::SplitPlan plan;   // large: keep it off the stack
  kvc::AttnPlan ap{};
  std::string perr;
  const int prc = kvc::plan_attention(h, T, H_q, &plan, &ap, &perr);
  if (prc) return fail(h, prc, "%s", perr.c_str());
  const int G = H_q / h->H;
  const int rpt = ap.rows_per_tile;

  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ap.workspace_floats) {
    const int wrc = ensure_workspace(h, ap.workspace_floats, st);
    if (wrc) return wrc;
  }
  kvc::AttnArgs a{};
  a.q = q; a.q_dtype = q_dtype; a.out = out;
  a.part_o = h->work;
  a.part_ml = h->work ? h->work + static_cast<size_t>(plan.n_items) * rpt * h->D : nullptr;
  a.counters = h->d_counters;
  a.lens = h->d_lens; a.status = h->d_status;
  a.layer = layer; a.B = h->B; a.H_kv = h->H; a.H_q = H_q; a.G = G; a.T = T; a.D = h->D;
  a.max_len = h->max_len; a.delta = T; a.cache_dtype = h->dtype;
  a.pg = kvc_paging(h);
  if (rope) {
    a.rope.table = h->d_rope;
    a.rope.style = h->rope_style;
  }
  a.k_scale = h->k_scale[layer];
  a.v_scale = h->v_scale[layer];
  a.out_elems = static_cast<long long>(h->B) * H_q * T * h->D;
  a.part_o_elems = h->work ? static_cast<long long>(plan.n_items) * rpt * h->D : 0;
  a.part_ml_elems = h->work ? static_cast<long long>(plan.n_items) * rpt * 2 : 0;
  cudaError_t e = cudaSuccess;
  if (fused) {
    if (h->paged) {
      const int grc = paged_grow(h, layer, T, st);
      if (grc) return grc;
    }
    if (ap.kernel == kvc::AttnKernel::DecodeTC) {
      a.app = *fused;
    } else {
      e = kvc::launch_append(*fused, st);
      if (e != cudaSuccess) return cuda_fail(h, e, "append launch");
      h->launches += 1;
    }
  }
  e = kvc::launch_attention(ap, a, plan, h, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "attention launch");
  h->launches += 1;
  return KVC_OK;
}

static int attn_impl(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int s, int T, int H_q,
                     float* out, bool rope, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  const int crc = kvc::check_attention_call(h, q, q_dtype, layer, s, T, H_q, out, rope);
  if (crc) return crc;
  return attn_launch(h, q, q_dtype, layer, T, H_q, out, rope, nullptr, stream);
}

// kvc_append followed by gqa_cached_attn over the committed lengths, in one call.
static int attn_append_impl(kvc_handle h, int layer, const void* k_new, const void* v_new, kvc_dtype in_dtype,
                            const void* q, kvc_dtype q_dtype, int T, int H_q, float* out, bool rope, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  int delta = 0;
  int rc = check_append(h, layer, k_new, v_new, in_dtype, T, rope, &delta);
  if (rc) return rc;
  if (delta != 0)
    return fail(h, KVC_E_STATE, "layer %d already holds %d rows appended since the last commit; this call "
                "appends the chunk itself", layer, delta);
  // the attention's checks as they stand once the chunk is in (every fill = committed length + T)
  const size_t f0 = static_cast<size_t>(layer) * h->B;
  for (int b = 0; b < h->B; ++b) h->fill[f0 + b] += T;
  rc = kvc::check_attention_call(h, q, q_dtype, layer, KVC_COMMITTED, T, H_q, out, rope);
  for (int b = 0; b < h->B; ++b) h->fill[f0 + b] -= T;
  if (rc) return rc;
  const kvc::AppendArgs app = append_args(h, layer, k_new, v_new, in_dtype, T, 0, rope);
  rc = attn_launch(h, q, q_dtype, layer, T, H_q, out, rope, &app, stream);
  if (rc) return rc;
  for (int b = 0; b < h->B; ++b) h->fill[f0 + b] += T;
  return KVC_OK;
}

int gqa_cached_attn_append(kvc_handle h, int layer, const void* k_new, const void* v_new, kvc_dtype in_dtype,
                           const void* q, kvc_dtype q_dtype, int T, int H_q, float* out, int rope, void* stream) {
  return attn_append_impl(h, layer, k_new, v_new, in_dtype, q, q_dtype, T, H_q, out, rope != 0, stream);
}

int gqa_cached_attn(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int s, int T, int H_q,
                    float* out, void* stream) {
  return attn_impl(h, q, q_dtype, layer, s, T, H_q, out, false, stream);
}

int gqa_cached_attn_rope(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int s, int T, int H_q,
                         float* out, void* stream) {
  return attn_impl(h, q, q_dtype, layer, s, T, H_q, out, true, stream);
}

int kvc_status(kvc_handle h, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  int flag = 0;
  e = cudaMemcpy(&flag, h->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "status read");
  if (flag) {
    const int zero = 0;
    cudaMemcpy(h->d_status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (flag == kvc::kStatusBounds)
      return fail(h, KVC_E_DEVICE_BOUNDS, "a kernel's bounds check caught an index past its buffer and skipped the store");
    return fail(h, KVC_E_DEVICE_TIMEOUT, "a kernel's bounded wait gave up (status %d)", flag);
  }
  return KVC_OK;
}

int kvc_debug_check_guards(kvc_handle h, void* stream) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
#ifndef KVC_DEBUG_BOUNDS
  (void)stream;
  return fail(h, KVC_E_UNSUPPORTED, "this library was built without KVC_DEBUG_BOUNDS (no guard bands)");
#else
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  std::vector<unsigned char> band(kGuard);
  for (const auto& buf : h->bufs) {
    for (int side = 0; side < 2; ++side) {
      const unsigned char* src = side == 0 ? static_cast<const unsigned char*>(buf.base)
                                           : static_cast<const unsigned char*>(buf.payload) + buf.bytes;
      e = cudaMemcpy(band.data(), src, kGuard, cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) return cuda_fail(h, e, "guard read");
      for (size_t i = 0; i < kGuard; ++i)
        if (band[i] != kGuardByte)
          return fail(h, KVC_E_DEVICE_BOUNDS, "%s: the guard band %s it was overwritten, %zu bytes %s its %s",
                      buf.what, side == 0 ? "before" : "after", side == 0 ? kGuard - i : i + 1,
                      side == 0 ? "before" : "past", side == 0 ? "start" : "end");
    }
  }
  return KVC_OK;
#endif
}

int kvc_last_error(kvc_handle h, char* buf, size_t n) {
  if (!buf || n == 0) return KVC_E_INVAL;
  const std::string& s = h ? h->err : g_err;
  const size_t k = std::min(n - 1, s.size());
  memcpy(buf, s.data(), k);
  buf[k] = '\0';
  return KVC_OK;
}

uint64_t kvc_launch_count(kvc_handle h) { return h ? h->launches : 0; }

size_t kvc_workspace_bytes(kvc_handle h) { return h ? h->work_floats * sizeof(float) : 0; }

int kvc_set_split_keys(kvc_handle h, int keys) {
  if (!h) return fail(nullptr, KVC_E_INVAL, "null handle");
  if (keys < 0) return fail(h, KVC_E_INVAL, "keys=%d", keys);
  h->split_keys_override = keys;
  return KVC_OK;
}

}  // extern "C"
