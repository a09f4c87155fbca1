// Internal declarations shared by the host side (kvc_host.cpp) and the kernels (*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kMaxBatch = KVC_MAX_BATCH;
// Units (sequence, row tile) a split-K launch can plan for; the plan travels in the kernel's
// parameters, so this bounds their size (2 * 4 * kMaxUnits bytes).
constexpr int kMaxUnits = 2048;

inline int itemsize(kvc_dtype t) { return t == KVC_F32 ? 4 : t == KVC_FP8_E4M3 ? 1 : 2; }
// Element types an append may hand to a cache of type `cache`: float32 or the cache dtype; an fp8
// cache takes float32, float16 or bfloat16 rows.
inline bool input_dtype_ok(kvc_dtype cache, int in) {
  if (in == KVC_F32) return true;
  if (cache == KVC_FP8_E4M3) return in == KVC_F16 || in == KVC_BF16;
  return in == cache && in != KVC_FP8_E4M3;
}
// Element types a query may have: float32 or the type the attention uses it in (the cache dtype;
// float16 for an fp8 cache).
inline bool query_dtype_ok(kvc_dtype cache, int q) {
  if (q == KVC_F32) return true;
  return cache == KVC_FP8_E4M3 ? q == KVC_F16 : (q == cache && q != KVC_FP8_E4M3);
}

// Device status word values: a kernel's bounded wait gave up; (debug builds) a store's index failed
// its bound and was skipped.
constexpr int kStatusTimeout = 1;
constexpr int kStatusBounds = 3;

// Where a store keeps its rows. A contiguous store is [L, B, H, max_len, D]. A paged store is a
// pool of fixed-size blocks, [L, n_blocks, H, block, D], and a block table [B, max_blocks] that maps
// each sequence's logical block i (positions [i * block, (i + 1) * block)) to a physical block, the
// same one in every layer; -1 marks a logical block that holds no physical block.
struct Paging {
  const int32_t* table = nullptr;   // device block table; nullptr for a contiguous store
  int max_blocks = 0;               // table row width = ceil(max_len / block)
  int block_shift = 0;              // log2(block)
  int n_blocks = 0;                 // physical blocks in the pool
};

// Rotary positions applied inside the kernels: table[p * (D / 2) + i] = (cos, sin)(p * theta_i), built
// once per handle in float64 and rounded to float32; style 0 rotates pairs (i, i + D/2), style 1 pairs
// (2i, 2i + 1).
struct Rope {
  const float2* table = nullptr;    // nullptr: no rotation
  int style = 0;
};
constexpr int kMaxRopePairs = 64;   // d_h <= 128
struct RopeTheta {
  double theta[kMaxRopePairs];      // base^(-2i/D), computed on the host
};
cudaError_t launch_rope_table(float2* table, int max_len, int D, const RopeTheta& th, cudaStream_t st);

// Tile row split of a paged store: keys per TMA box (a tile of `tile` keys takes tile / box_rows
// boxes per 128-byte column when blocks are shorter than the tile).
inline int paged_box_rows(const Paging& pg, int tile) {
  return pg.table ? (tile < (1 << pg.block_shift) ? tile : (1 << pg.block_shift)) : tile;
}

// ------------------------------------------------------------------------------------------------
// Append: writes a [B, H, T, D] chunk at row lens[b] + delta + t of each (layer, b, h).
// ------------------------------------------------------------------------------------------------
struct AppendArgs {
  void* k_store;            // [L, B, H, max_len, D] cache dtype
  void* v_store;
  const void* k_new;        // [B, H, T, D] in_dtype
  const void* v_new;
  const int32_t* lens;      // device committed lengths [B]
  int layer, B, H, D, T, max_len;
  int Dv;                   // width of the second store's rows (= D, or d_R for a latent cache)
  int delta;                // this layer's fill minus the committed length (uniform over b)
  kvc_dtype cache_dtype, in_dtype;
  Paging pg;                // paged store: rows go through the block table
  Rope rope;                // rotate K rows by their positions before storing them (V untouched)
  float k_scale = 1.f;      // fp8 caches: stored code = e4m3(x / scale)
  float v_scale = 1.f;
  long long k_rows = 0, v_rows = 0;   // rows of each store (debug index checks)
  int* status = nullptr;              // device status word (debug index checks)
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t st);

// Block-table edits: table[slot[i]] = value[i], applied in one launch before the call that needs them.
constexpr int kMaxTableEdits = 1024;
struct TableEdits {
  int n;
  int32_t slot[kMaxTableEdits];
  int32_t value[kMaxTableEdits];
};
cudaError_t launch_table_edits(int32_t* table, const TableEdits& e, cudaStream_t st);

// lens[b] += delta for all b
cudaError_t launch_lens_add(int32_t* lens, int B, int delta, cudaStream_t st);
// lens[b] = n[b]
cudaError_t launch_lens_set(int32_t* lens, int B, const int32_t* n_host, cudaStream_t st);
// out[b * T + t] = lens[b] + t
cudaError_t launch_positions(const int32_t* lens, int B, int T, int32_t* out, cudaStream_t st);

// ------------------------------------------------------------------------------------------------
// Split-K attention on CUDA cores (decode and short chunks): plan built on the host from the
// host mirror of the lengths; the kernel reads the lengths themselves from the device.
// ------------------------------------------------------------------------------------------------
struct SplitPlan {
  int n_units;                       // units = (sequence b, row tile rt)
  int n_items;                       // CTAs: sum over units of H_kv * nsplit
  int split_keys;                    // largest split (keys); a unit's nsplit splits are near-equal
  int rows_per_tile;                 // query rows (t, g) per unit
  int n_rowtiles;                    // row tiles per sequence
  int32_t prefix[kMaxUnits + 1];     // item prefix over units
  int32_t unit_b[kMaxUnits];         // b * n_rowtiles + rt of each unit, in dispatch order
};

struct AttnArgs {
  const void* q;            // [B, H_q, T, D]
  kvc_dtype q_dtype;
  float* out;               // [B, H_q, T, D]
  float* part_o;            // [n_items, rows_per_tile, D] workspace
  float* part_ml;           // [n_items, rows_per_tile, 2] workspace
  int* counters;            // [kMaxUnits, H_kv] finished-split counters, zero between launches
  const int32_t* lens;      // device committed lengths
  int* status;              // device status word
  int layer, B, H_kv, H_q, G, T, D, max_len;
  int delta;                // fill - committed for this layer (== T when the chunk was appended)
  kvc_dtype cache_dtype;
  Paging pg;                // paged store: tiles are gathered through the block table
  Rope rope;                // rotate each query row by its position s_b + t before attending
  float k_scale = 1.f;      // fp8 caches: scores use code * k_scale, outputs code * v_scale
  float v_scale = 1.f;
  long long out_elems = 0, part_o_elems = 0, part_ml_elems = 0;   // buffer sizes (debug index checks)
  // Fused append (tensor-core decode kernel only): when app.k_new is set, the chunk's rows have not
  // been stored yet; the CTA whose split holds a new row stores it, exactly as the append kernel
  // would, before it loads the tile that holds the row.
  AppendArgs app{};
};
// Workspace floats the plan needs (0 when no unit splits).
size_t splitk_workspace_floats(const SplitPlan& p, int D);
// Choose rows per tile and tile keys for (dtype, D, rows); returns false if unsupported.
bool splitk_shape(kvc_dtype dt, int D, int rows, int* rows_per_tile, int* tile_keys);
cudaError_t launch_splitk(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                          const CUtensorMap* tv, cudaStream_t st);

// Tensor-core decode/verify kernel (16-bit caches, d_h = 128, up to 32 query rows per K/V head per
// row tile). Returns false when the shape has no tensor-core kernel.
bool decode_tc_shape(kvc_dtype dt, int D, int rows, int* rows_per_tile, int* tile_keys, int* max_tiles);
// cluster > 1: every unit has `cluster` splits and each (unit, K/V head)'s splits run as one thread-block
// cluster whose partials merge through distributed shared memory (16-bit caches; falls back to the L2
// merge when the cluster cannot be placed).
cudaError_t launch_decode_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                             const CUtensorMap* tv, int cluster, cudaStream_t st);

// Tensor-core chunk kernels: 16-bit caches, d_h = 128, 128 query rows per CTA. launch_chunk_tc:
// at most 128 rows per K/V head (one CTA per (sequence, K/V head), one per SM); launch_prefill_tc:
// units of 128 rows, keys split over CTAs as the split planner cuts them, two CTAs per SM.
bool prefill_tc_shape(kvc_dtype dt, int D, int* rows_per_tile);
cudaError_t launch_chunk_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                            const CUtensorMap* tv, cudaStream_t st);
cudaError_t launch_prefill_tc(const AttnArgs& a, const SplitPlan& p, const CUtensorMap* tk,
                              const CUtensorMap* tv, cudaStream_t st);

// Multi-head latent attention over a latent cache (absorbed form): per query row (t, h), scores
// (q_lat . c_j + q_rope . kR_j) * scale over keys j <= s_b + t, output sum_j softmax_j c_j.
struct MlaArgs {
  const void* q_lat;        // [B, H, T, r]
  const void* q_rope;       // [B, H, T, dR]
  kvc_dtype q_dtype;
  float* out;               // [B, H, T, r]
  float* part_o;            // [n_items, rows_per_tile, r] workspace
  float* part_ml;           // [n_items, rows_per_tile, 2]
  int* counters;            // [units] finished-split counters, zero between launches
  const int32_t* lens;
  int* status;
  const void* c_store;      // [L, B, max_len, r]
  const void* kr_store;     // [L, B, max_len, dR]
  int layer, B, H, T, r, dR, max_len;
  float scale;              // softmax scale (1 / sqrt of the per-head query-key width)
  kvc_dtype cache_dtype;
  long long out_elems = 0, part_o_elems = 0, part_ml_elems = 0;   // buffer sizes (debug index checks)
};
constexpr int kMlaRows = 16;                 // query rows per CTA
int mla_tile_keys(kvc_dtype dt);             // keys per shared-memory tile
size_t mla_smem_bytes(kvc_dtype dt, int r, int dR);
cudaError_t launch_mla(const MlaArgs& a, const SplitPlan& p, cudaStream_t st);
// Tensor-core latent attention: 16-bit caches, r = 256 or 512, d_R = 64 (64-key tiles, one CTA per SM).
constexpr int kMlaTcKeys = 64;
bool mla_tc_shape(kvc_dtype dt, int r, int dR);
cudaError_t launch_mla_tc(const MlaArgs& a, const SplitPlan& p, const CUtensorMap* tc, const CUtensorMap* tr,
                          cudaStream_t st);

// Record an error message for kvc_last_error (on the handle when there is one, and for the calling
// thread) and return `code`.
int fail(kvc_handle h, int code, const char* fmt, ...);
// The argument and state checks every gqa_cached_attn* entry point makes before it plans or enqueues
// anything (h non-null): KVC_OK, or the error code with the message recorded.
int check_attention_call(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int s, int T, int H_q,
                         const float* out, bool rope);

// Which attention kernel serves a call, and its work plan (built from the host mirror of the lengths).
enum class AttnKernel { SplitK, DecodeTC, ChunkTC, PrefillTC };
struct AttnPlan {
  AttnKernel kernel;
  int rows_per_tile;
  int cluster = 0;           // decode kernel: splits per unit when they merge as one cluster (else 0)
  size_t workspace_floats;   // split partials (0 when no unit splits)
  size_t counters;           // merge counters the kernel may use (units x H_kv)
};
// Fills `plan` (a large struct: keep it off the stack); returns KVC_OK or an error code with `err`.
int plan_attention(kvc_handle h, int T, int H_q, SplitPlan* plan, AttnPlan* out, std::string* err);
cudaError_t launch_attention(const AttnPlan& ap, const AttnArgs& a, const SplitPlan& p, kvc_handle h,
                             cudaStream_t st);

// Tensor map over a store viewed as [planes, rows, D] with boxes of (swizzle span, box_rows, 1):
// planes = L*B*H and rows = max_len for a contiguous store, planes = L*n_blocks*H and rows = block
// for a paged pool.
bool encode_store_map(CUtensorMap* map, void* base, kvc_dtype dt, int D, int rows,
                      long long planes, int box_rows, std::string* err);

// Keys per split when a unit's n keys are cut into nsplit splits (split i covers [i * chunk, (i + 1) *
// chunk) clipped to n): the near-equal share rounded up to whole tiles, so every split starts on a
// tile boundary and a paged tile never straddles two blocks at an odd offset. If nsplit = ceil(n /
// chunk) for a chunk computed this way, recomputing the chunk from nsplit gives it back, so the host
// planner and the kernels agree and no split is empty.
__host__ __device__ inline int split_chunk(int n, int nsplit, int tile) {
  const int share = (n + nsplit - 1) / nsplit;
  return (share + tile - 1) / tile * tile;
}

// Launch with programmatic stream serialization: the kernel may be scheduled before its stream
// predecessor finishes and orders itself with griddepcontrol.wait (see kvc_device.cuh).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per device instead of on every launch (the
// attribute persists for the process; the call costs host time that decode launches cannot spare).
// Keyed on the kernel itself: every instantiation keeps its own flags.
template <auto Kernel>
cudaError_t ensure_smem_limit(size_t bytes) {
  static unsigned long long done = 0;          // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0;
  if (bit && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && bit) __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
  return e;
}

}  // namespace kvc

struct kvc_cache {
  int L = 0, B = 0, H = 0, D = 0, max_len = 0;
  // latent (MLA) cache: H = 1, the first store holds the latent c (width D = r), the second the
  // shared RoPE key k^R (width Dv = d_R); for a KV cache Dv = D
  int Dv = 0;
  bool latent = false;
  kvc_dtype dtype = KVC_F32;
  bool owns_store = false;
  // paged store: pool blocks, device table and its host mirror, and the free list
  bool paged = false;
  int block = 0, block_shift = 0, n_blocks = 0, max_blocks = 0;
  int32_t* d_table = nullptr;     // [B * max_blocks]
  std::vector<int32_t> table;     // host mirror
  std::vector<int32_t> held;      // blocks each sequence holds (logical blocks 0 .. held-1)
  std::vector<int32_t> free_heap; // free physical blocks, a min-heap: the lowest is handed out first
  std::vector<std::pair<int32_t, int32_t>> edit_scratch;   // (slot, value) table edits of one call
  // rotary positions (kvc_set_rope): cos/sin table [max_len, D / 2] on the device
  float2* d_rope = nullptr;
  int rope_style = -1;
  // fp8 caches: per-layer scales (stored code = e4m3(x / scale)), 1 until kvc_set_kv_scales
  std::vector<float> k_scale, v_scale;
  void* k = nullptr;
  void* v = nullptr;
  int32_t* d_lens = nullptr;      // committed lengths on the device
  int* d_status = nullptr;        // device status word
  std::vector<int32_t> fill;      // host mirror [L * B]
  std::vector<int32_t> lens;      // host mirror [B]
  CUtensorMap tmap_k_split{}, tmap_v_split{};
  CUtensorMap tmap_k_tc{}, tmap_v_tc{};          // 128-key boxes for the tensor-core kernel
  bool has_tc = false;
  int split_tile_keys = 0;
  float* work = nullptr;          // split-K workspace
  int* d_counters = nullptr;      // split-K merge counters [kMaxUnits * H]
  size_t work_floats = 0;
  int split_keys_override = 0;
  std::vector<long long> plan_n_eff;  // planner scratch
  std::vector<int> plan_nsplit;
  std::vector<std::pair<int, int>> plan_order;
  // every device buffer the library allocated for this handle: (allocation base, payload, bytes,
  // what); a debug build (KVC_DEBUG_BOUNDS) puts guard bands of a known byte on both sides of each
  struct DevBuf {
    void* base;
    void* payload;
    size_t bytes;
    const char* what;
  };
  std::vector<DevBuf> bufs;
  uint64_t launches = 0;          // kernels enqueued by this handle
  int num_sms = 0;
  int device = 0;
  std::string err;
};

// The store addressing the kernels of a handle use.
inline kvc::Paging kvc_paging(const kvc_cache* h) {
  kvc::Paging pg;
  if (h->paged) {
    pg.table = h->d_table;
    pg.max_blocks = h->max_blocks;
    pg.block_shift = h->block_shift;
    pg.n_blocks = h->n_blocks;
  }
  return pg;
}
