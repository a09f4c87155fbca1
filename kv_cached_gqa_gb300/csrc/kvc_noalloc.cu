// gqa_cached_attn_noalloc: the attention call without any device allocation.
//
// gqa_cached_attn keeps a per-handle workspace for the split-K partial results and grows it with
// cudaMallocAsync the first time a larger one is needed. Some callers cannot allow that: a serving
// process that reserves all of its device memory up front (the KV cache takes most of the HBM) and
// forbids allocations once it serves, a caller whose memory belongs to another framework's pool,
// or a latency-critical path that must not stall or fail on an allocation under memory pressure.
// This entry point runs the same kernels, but their scratch (the split partials and the per-unit
// merge counters) lives in one fixed file-scope device array, so the call allocates nothing.
//
// Rules of use:
// * The array holds kNoallocScratchBytes (8 MiB); a call whose plan needs more is rejected with
//   KVC_E_UNSUPPORTED and a message giving both sizes. Every GPU that loads the library holds the
//   array until the process exits.
// * The first call on each device looks up the array's device address (cudaGetSymbolAddress, with
//   that device current) and caches it. Make that first call before any stream capture.
// * All calls share the one array and it keeps the last call's contents. Each call clears the merge
//   counters it uses (cudaMemsetAsync on its stream) before launching. Calls that overlap on the GPU
//   (different streams, no ordering between them) race on the array and give wrong results.
#include <cuda_runtime.h>

#include <algorithm>
#include <string>
#include <mutex>
#include <utility>
#include <vector>

#include "kvc_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

// The scratch itself: split partials (float) preceded by the merge counters (int).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per device.
int scratch_address(void** out, std::string* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = cudaGetErrorString(e); return KVC_E_CUDA; }
  if (dev < 0 || dev >= kMaxDevices) { *err = "device index out of range"; return KVC_E_UNSUPPORTED; }
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      *err = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
      return KVC_E_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" int gqa_cached_attn_noalloc(kvc_handle h, const void* q, kvc_dtype q_dtype, int layer, int s,
                                       int T, int H_q, float* out, void* stream) {
  if (!h) return kvc::fail(nullptr, KVC_E_INVAL, "null handle");
  // ---- the checks of gqa_cached_attn, shared with it (latent handles rejected there too) -------
  const int crc = kvc::check_attention_call(h, q, q_dtype, layer, s, T, H_q, out, false);
  if (crc) return crc;

  // ---- the same kernel choice and split plan ----------------------------------------------------
  static thread_local kvc::SplitPlan plan;
  kvc::AttnPlan ap{};
  std::string perr;
  const int prc = kvc::plan_attention(h, T, H_q, &plan, &ap, &perr);
  if (prc) return kvc::fail(h, prc, "%s", perr.c_str());
  const int G = H_q / h->H;
  const int rpt = ap.rows_per_tile;

  // ---- scratch from the fixed array: [counters | partial o | partial (m, l)] ------------------
  const size_t counter_bytes = (ap.counters * sizeof(int) + 255) / 256 * 256;
  const size_t part_bytes = ap.workspace_floats * sizeof(float);
  if (counter_bytes + part_bytes > kNoallocScratchBytes)
    return kvc::fail(h, KVC_E_UNSUPPORTED, "this call needs %zu bytes of scratch; the fixed array holds %zu",
                   counter_bytes + part_bytes, kNoallocScratchBytes);
  void* base = nullptr;
  std::string err;
  int rc = scratch_address(&base, &err);
  if (rc) return kvc::fail(h, rc, "%s", err.c_str());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (counter_bytes) {
    e = cudaMemsetAsync(base, 0, counter_bytes, st);
    if (e != cudaSuccess) return kvc::fail(h, KVC_E_CUDA, "clearing the merge counters: %s", cudaGetErrorString(e));
  }

  kvc::AttnArgs a{};
  a.q = q; a.q_dtype = q_dtype; a.out = out;
  a.counters = static_cast<int*>(base);
  a.part_o = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + counter_bytes);
  a.part_ml = a.part_o + static_cast<size_t>(plan.n_items) * rpt * h->D;
  a.lens = h->d_lens; a.status = h->d_status;
  a.layer = layer; a.B = h->B; a.H_kv = h->H; a.H_q = H_q; a.G = G; a.T = T; a.D = h->D;
  a.max_len = h->max_len; a.delta = T; a.cache_dtype = h->dtype;
  a.pg = kvc_paging(h);
  a.k_scale = h->k_scale[layer];
  a.v_scale = h->v_scale[layer];
  a.out_elems = static_cast<long long>(h->B) * H_q * T * h->D;
  a.part_o_elems = static_cast<long long>(plan.n_items) * rpt * h->D;
  a.part_ml_elems = static_cast<long long>(plan.n_items) * rpt * 2;
  e = kvc::launch_attention(ap, a, plan, h, st);
  if (e != cudaSuccess) return kvc::fail(h, KVC_E_CUDA, "attention launch: %s", cudaGetErrorString(e));
  h->launches += 1;
  return KVC_OK;
}
