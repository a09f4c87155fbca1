/*
 * kvc.h — C ABI of the KV-cached grouped-query attention library for GB300 (sm_103a).
 *
 * One decode (or prefill, or verify) forward of a decoder with a KV cache, per layer l:
 *   kvc_append(l, k_new, v_new)   write the chunk's post-RoPE keys/values at positions [s_b, s_b + T)
 *   gqa_cached_attn(q, l, ...)    attend the chunk's T queries over all s_b + T stored keys
 * (or both in one call: gqa_cached_attn_append(l, k_new, v_new, q, ...)), and once after the last layer:
 *   kvc_commit()                  s_b += T for every sequence
 * ("KV cache, incremental decode, incremental UTF-8 detokenizer, generate", §2.1-§2.4 and §4
 * "The interface"; "KV cache decoding", steps 1-7).
 *
 * Conventions shared by every call
 * - Shapes are row-major and contiguous. The cache holds K and V, each [L, B, H_kv, max_len, d_h],
 *   in the cache dtype. A chunk's keys/values are [B, H_kv, T, d_h]; its queries and the output
 *   are [B, H_q, T, d_h].
 * - Pointers named *_dev are device pointers on the current CUDA device; *_host are host pointers.
 *   `stream` is a cudaStream_t (NULL = the legacy default stream). Every device-side effect is
 *   enqueued on `stream` in call order; no call synchronises the device except kvc_status and
 *   kvc_destroy.
 * - Every call validates its arguments against host-side mirrors of the lengths before it
 *   enqueues anything. On any error it returns a negative code, changes no state (lengths,
 *   store, handle) and records a message for kvc_last_error ("KV cache, incremental decode, ...",
 *   §4, test_update_copies_and_checks: nothing changed on error).
 * - A handle is not thread-safe; calls on one handle must come from one host thread at a time.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvc_cache* kvc_handle;

/* Storage / input element types. KVC_FP8_E4M3 is a cache (storage) type only: FP8 E4M3 codes (bias 7,
 * no infinities, largest finite 448) of x / scale, with one scale per layer for K and one for V
 * (kvc_set_kv_scales, default 1). Inputs to an fp8 cache may be F32, F16 or BF16; its queries F32 or
 * F16 (the attention uses them in float16, which holds every E4M3 value exactly). */
typedef enum { KVC_F32 = 0, KVC_F16 = 1, KVC_BF16 = 2, KVC_FP8_E4M3 = 3 } kvc_dtype;

/* Return codes. */
enum {
  KVC_OK = 0,
  KVC_E_INVAL = -1,          /* bad argument: null pointer, size, layer, dtype, misalignment */
  KVC_E_CAPACITY = -2,       /* the write would pass max_len ("KV cache decoding", assert t + m <= max_len) */
  KVC_E_STATE = -3,          /* call out of order: commit with unequal fills, truncate beyond s_b,
                                attention on a layer that does not hold exactly s_b + T rows */
  KVC_E_CUDA = -4,           /* a CUDA runtime/driver call failed (message in kvc_last_error) */
  KVC_E_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait gave up; reported by kvc_status */
  KVC_E_UNSUPPORTED = -6,    /* a size this build has no kernel for (d_h not in {32, 64, 128}, ...) */
  KVC_E_NOMEM = -7,          /* device or host allocation failed */
  KVC_E_DEVICE_BOUNDS = -8   /* debug builds: a guard band or a kernel's index check caught a stray store */
};

/* Rotary-position pair layouts (kvc_set_rope). */
typedef enum {
  KVC_ROPE_HALF = 0,        /* element i turns with element i + d_h/2 (the Llama-family layout) */
  KVC_ROPE_INTERLEAVED = 1  /* element 2i turns with element 2i + 1 (the RoFormer paper's layout) */
} kvc_rope_style;

/* Pass as `s` to gqa_cached_attn to use each sequence's own committed length (ragged batches). */
#define KVC_COMMITTED (-1)
/* Largest batch a handle accepts. */
#define KVC_MAX_BATCH 1024

/*
 * kvc_create — allocate and zero a cache of L layers, B sequences, H_kv K/V heads of width d_h and
 * capacity max_len positions, stored as `dtype`.
 * Defined by: "KV cache, incremental decode, ...", §2.5 "Storage dtype" (preallocated
 * 2 L B H_kv N_max d_h elements); "Generation and the KV Cache" ("Module 32 built KVCache(cfg,
 * batch_size, max_len): k, v of shape (L, B, H, max_len, d_head)"); "KV cache decoding",
 * KVCache listing (np.zeros: unfilled slots are zero).
 * The library owns the store (cudaMalloc) and frees it in kvc_destroy. All lengths start at 0.
 * Limits: 1 <= B <= KVC_MAX_BATCH, d_h in {32, 64, 128} ({64, 128} for KVC_FP8_E4M3), L*B*H_kv < 2^31,
 * max_len < 2^30.
 */
int kvc_create(kvc_handle* out, int L, int B, int H_kv, int d_h, int max_len, kvc_dtype dtype,
               void* stream);

/*
 * kvc_create_external — the same cache over caller-owned storage: k_store_dev and v_store_dev each
 * hold L*B*H_kv*max_len*d_h elements of `dtype`, 256-byte aligned and already zeroed by the
 * caller. The caller keeps ownership and must keep them alive until kvc_destroy.
 */
int kvc_create_external(kvc_handle* out, int L, int B, int H_kv, int d_h, int max_len,
                        kvc_dtype dtype, void* k_store_dev, void* v_store_dev, void* stream);

/*
 * kvc_create_paged — a cache whose rows live in a pool of fixed-size blocks mapped by a per-sequence
 * block table, instead of one max_len-long slab per sequence.
 * Defined by: "KV cache decoding", "Batching caches of different lengths" (the cache in fixed-size
 * blocks with a table from each request to its blocks; a sequence takes a new block only when it grows
 * into it and frees its blocks when it ends); "Generation and the KV Cache", "Static versus growing"
 * (the positions a preallocated cache reserves are what a paged cache recovers); "KV cache,
 * incremental decode, ...", Key Takeaways and §2.5 (a float16 paged cache stores what the contiguous
 * one stores and compares with it exactly).
 * Layout: K and V pools, each [L, n_blocks, H_kv, block_size, d_h] in `dtype`; a block table
 * [B, ceil(max_len / block_size)] of int32 (device copy owned by the library, host mirror readable with
 * kvc_block_table). Position p of sequence b is row p % block_size of physical block
 * table[b][p / block_size], the same block in every layer; -1 marks a logical block with none.
 * Allocation: kvc_append maps, lowest-numbered free block first (sequences in order, then logical
 * blocks in order), every block the layer's new fill reaches and the sequence does not hold yet
 * (one small table-edit launch before the append when any is needed). kvc_truncate and
 * kvc_truncate_ragged return every block wholly past the new length to the pool (truncate to 0 frees
 * a sequence's blocks when it ends). A partly filled last block stays with its sequence.
 * Every other call (append, commit, positions, attention, the no-alloc variant, status) works on a
 * paged handle with the same arguments, results and errors, and gqa_cached_attn returns exactly what
 * it returns for a contiguous cache holding the same rows. kvc_nbytes is the pool capacity
 * 2 * L * n_blocks * H_kv * block_size * d_h * itemsize; kvc_layer_ptrs gives a layer's pool
 * [n_blocks, H_kv, block_size, d_h].
 * k_pool_dev, v_pool_dev: both NULL (the library allocates and zeroes the pools) or both caller-owned,
 * 256-byte aligned and zeroed, kept alive until kvc_destroy.
 * Limits: those of kvc_create, block_size a power of two in [16, 2^20], n_blocks >= 1,
 * L * n_blocks * H_kv < 2^31. Errors: KVC_E_INVAL; KVC_E_NOMEM. kvc_append returns KVC_E_CAPACITY,
 * changing nothing, when the pool has too few free blocks for it.
 */
int kvc_create_paged(kvc_handle* out, int L, int B, int H_kv, int d_h, int max_len, int block_size,
                     int n_blocks, kvc_dtype dtype, void* k_pool_dev, void* v_pool_dev, void* stream);

/*
 * kvc_block_table — copy a paged cache's block table (host mirror, the state after every call enqueued
 * so far) into table_host[B * ceil(max_len / block_size)] and the number of free pool blocks into
 * *n_free_host; either pointer may be NULL. KVC_E_INVAL for a contiguous cache.
 */
int kvc_block_table(kvc_handle h, int32_t* table_host, int32_t* n_free_host);

/*
 * kvc_create_latent — a latent cache for multi-head latent attention (MLA): per layer and position one
 * compressed latent c in R^r and one RoPE key k^R in R^{d_rope} shared by all heads, instead of per-head
 * K and V.
 * Defined by: "KV cache, incremental decode, ...", §2.6 "The latent cache" (the same rules as the KV cache
 * — per-layer fill, committed length, rollback — on [B, T, r] and [B, T, d_R] chunks; nbytes is
 * L B N_max (r + d_R) times the item size).
 * Layout: the latent store [L, B, max_len, r] and the RoPE-key store [L, B, max_len, d_rope], in `dtype`
 * (F32, F16 or BF16). c_store_dev and kr_store_dev: both NULL (the library allocates and zeroes them) or
 * both caller-owned, 256-byte aligned and zeroed.
 * The handle works with kvc_append (k_new_dev = the latent chunk [B, T, r], v_new_dev = the RoPE-key
 * chunk [B, T, d_rope]; the RoPE key is stored as given), kvc_commit, kvc_truncate(_ragged),
 * kvc_seq_len, kvc_positions, kvc_nbytes (= L B max_len (r + d_rope) itemsize), kvc_layer_ptrs (the
 * layer's two stores), kvc_status and kvc_destroy, with their usual meaning and errors; it is read by
 * mla_cached_attn. gqa_cached_attn* and kvc_set_rope reject it.
 * Limits: r and d_rope multiples of 16, r <= 1024, d_rope <= 256, r + d_rope <= 1152 (the attention
 * kernel's shared memory), B <= KVC_MAX_BATCH.
 * Errors: KVC_E_INVAL, KVC_E_UNSUPPORTED (r or d_rope out of range), KVC_E_NOMEM.
 */
int kvc_create_latent(kvc_handle* out, int L, int B, int r, int d_rope, int max_len, kvc_dtype dtype,
                      void* c_store_dev, void* kr_store_dev, void* stream);

/*
 * mla_cached_attn — multi-head latent attention of a chunk's T queries per head over every stored row of
 * one layer of a latent cache, in the absorbed form (DeepSeek-V2, §2.1: the key up-projection is folded
 * into the query, the value up-projection is applied to the output by the caller).
 * For sequence b, head h and query t (absolute position s_b + t), over keys j <= s_b + t:
 *   score_j = (q_lat[b,h,t] . c_j + q_rope[b,h,t] . k^R_j) * scale,   out[b,h,t] = sum_j softmax_j c_j.
 * Defined by: "KV cache, incremental decode, ...", §2.6 (the latent cache MLA reads) and §2.3 (query t
 * at absolute position s + t sees keys j <= s + t).
 * q_lat_dev [B, H, T, r], q_rope_dev [B, H, T, d_rope], in `q_dtype` (F32, or the cache dtype; an F32
 * query meets a 16-bit cache rounded to it). out_dev [B, H, T, r] float32, caller-owned. scale > 0 (the
 * model's 1 / sqrt(per-head query-key width)). s as in gqa_cached_attn. Precondition: `layer` holds
 * s_b + T rows (the chunk appended), else KVC_E_STATE. Split partials use the handle's workspace
 * (grown with cudaMallocAsync when needed).
 */
int mla_cached_attn(kvc_handle h, const void* q_lat_dev, const void* q_rope_dev, kvc_dtype q_dtype, int layer,
                    int s, int T, int H, float scale, float* out_dev, void* stream);

/* kvc_destroy — synchronise the device, free everything the library allocated. NULL is a no-op. */
int kvc_destroy(kvc_handle h);

/*
 * kvc_append — write one chunk of T positions for one layer.
 * Defined by: "KV cache, incremental decode, ...", §4 update(layer, k_new, v_new) ([B, Hkv, T, dh]
 * in; written at the layer's fill count, §2.3) and §2.5 (values converted to the storage dtype on
 * the way in); "KV cache decoding", step 5 (write slots t .. t+m-1 of this layer).
 * k_new_dev, v_new_dev: [B, H_kv, T, d_h] in `in_dtype`, which is KVC_F32 or the cache dtype. F32
 * input to a 16-bit cache is rounded to nearest even. The inputs are copied (the caller may reuse
 * its buffers once the stream reaches this call). Each sequence b writes rows
 * [fill_b, fill_b + T) of layer `layer`, fill_b being that layer's fill count, and the layer's
 * fill counts advance by T. The committed length does not move (see kvc_commit).
 * Errors: KVC_E_INVAL (layer, T < 1, null, dtype), KVC_E_CAPACITY (fill_b + T > max_len for any b).
 */
int kvc_append(kvc_handle h, int layer, const void* k_new_dev, const void* v_new_dev,
               kvc_dtype in_dtype, int T, void* stream);

/*
 * kvc_set_rope — give the handle rotary positions: build on the device, once, the table of
 * (cos, sin)(p * theta_i) for every position p < max_len and pair i < d_h/2, theta_i = base^(-2i/d_h),
 * computed in float64 and stored as float32 pairs (max_len * d_h/2 * 8 bytes, owned by the handle).
 * Calling it again rebuilds the table for the new base and style (stream-ordered).
 * Defined by: "KV cache decoding", "Position information with a cache" (query and key rotated by an angle
 * of their absolute position; keys stored already rotated; the new query rotated by its position; the
 * score then depends only on the distance). The pages name RoPE without printing it; the formula is
 * Su et al., "RoFormer", eq. 34.
 * Errors: KVC_E_INVAL (base not in (1, 1e12], unknown style), KVC_E_NOMEM.
 */
int kvc_set_rope(kvc_handle h, double base, kvc_rope_style style, void* stream);

/*
 * kvc_append_rope — kvc_append with the keys rotated inside the append: row t of sequence b is turned
 * by its absolute position (the position it is written at, s_b + t for a forward's chunk) in float32,
 * then rounded to the cache dtype; values are stored as given. k_new_dev holds the keys BEFORE RoPE.
 * Arguments, layout and errors are kvc_append's, plus KVC_E_STATE when kvc_set_rope was not called.
 */
int kvc_append_rope(kvc_handle h, int layer, const void* k_new_dev, const void* v_new_dev,
                    kvc_dtype in_dtype, int T, void* stream);

/*
 * kvc_set_kv_scales — per-layer scales of an fp8 cache: k_scale_host[L] and v_scale_host[L] (host
 * memory, copied), positive and finite. A row x of layer l is stored as E4M3(x / scale_l) (float32
 * division, round to nearest even, saturating at +-448) and read as code * scale_l.
 * Defined by: "KV cache decoding", "What is cached, what is not, and what it costs" (cache quantisation
 * as a lever for decode's memory traffic). The pages give no format; E4M3 with per-layer scales is the
 * reading used here.
 * Errors: KVC_E_INVAL (not an fp8 cache, null, a scale <= 0 or not finite); KVC_E_STATE (any layer
 * already holds rows: scales are fixed while the cache holds data).
 */
int kvc_set_kv_scales(kvc_handle h, const float* k_scale_host, const float* v_scale_host);

/*
 * kvc_commit — advance every committed length s_b to its fill, once per forward after the last
 * layer ("KV cache, incremental decode, ...", §2.3: the length advances only after the last layer;
 * "KV cache decoding", step 7).
 * Error: KVC_E_STATE if the layers' fill counts disagree for any sequence.
 */
int kvc_commit(kvc_handle h, void* stream);

/*
 * kvc_truncate — set every layer's fill count and every committed length to n, for speculative
 * rollback ("KV cache, incremental decode, ...", §2.4 "Rollback": nothing is freed or copied; the
 * next append overwrites from n). Rows at and past n keep their old contents until overwritten.
 * Error: KVC_E_STATE if n exceeds any sequence's committed length; KVC_E_INVAL if n < 0.
 */
int kvc_truncate(kvc_handle h, int n, void* stream);

/* kvc_truncate_ragged — the same with one length per sequence, n_host[B] (host memory, copied). */
int kvc_truncate_ragged(kvc_handle h, const int32_t* n_host, void* stream);

/*
 * kvc_set_lengths — set every layer's fill count and every committed length to n_host[b] (host memory,
 * B values, copied), growing or shrinking. The rows [0, n_b) are then the cache's content for sequence
 * b, whatever the store holds there: zeros in a fresh cache (unfilled slots are zero), rows written
 * earlier after a truncate (truncate frees and clears nothing), or rows the caller wrote into the
 * store directly (kvc_layer_ptrs). It sets up a ragged batch whose context is already in place without
 * re-appending it.
 * Defined by: "KV cache, incremental decode, ...", §2.3 (per-layer fill counts and one committed
 * length per sequence) and §2.4 ("Rollback": a length is moved and nothing is copied); "KV cache
 * decoding", "Batching caches of different lengths" (one length per request).
 * Errors: KVC_E_INVAL (null, any n_b < 0 or n_b > max_len); KVC_E_UNSUPPORTED for a paged cache, whose
 * blocks are mapped only by kvc_append. Nothing changes on error.
 */
int kvc_set_lengths(kvc_handle h, const int32_t* n_host, void* stream);

/*
 * kvc_seq_len — copy lengths into out_host[B]: the committed lengths s_b for layer == -1, or one
 * layer's fill counts ("KV cache, incremental decode, ...", §4 seq_len(layer=None)).
 */
int kvc_seq_len(kvc_handle h, int layer, int32_t* out_host);

/*
 * kvc_positions — write the absolute positions of the next chunk, [s_b, s_b + T), into
 * out_dev[B, T] (int32), from the device's committed lengths ("KV cache, incremental decode, ...",
 * §4 positions(t_new); the positions RoPE rotates by, read once at the start of a forward).
 */
int kvc_positions(kvc_handle h, int T, int32_t* out_dev, void* stream);

/* kvc_nbytes — capacity in bytes, 2 * L * B * H_kv * max_len * d_h * itemsize (§2.5). 0 for NULL. */
size_t kvc_nbytes(kvc_handle h);

/*
 * kvc_layer_ptrs — device addresses of layer `layer`'s K and V blocks, each [B, H_kv, max_len, d_h]
 * in the cache dtype: the stored (rounded) rows that attention reads ("KV cache, incremental
 * decode, ...", §4: update returns all stored rows). Valid until kvc_destroy.
 */
int kvc_layer_ptrs(kvc_handle h, int layer, void** k_dev, void** v_dev);

/*
 * gqa_cached_attn — attend a chunk's T queries over every stored row of one layer.
 * Defined by: "KV cache, incremental decode, ...", §2.3 (query i at absolute position s + i sees
 * keys j <= s + i: causal_mask(T, s + T, q_offset = s)); "Generation and the KV Cache", fence 3
 * (scores q K^T / sqrt(d), offset mask, softmax, times V); "Heads, GQA and K/V cache" ("Four
 * queries, two sets of K/V": query head h uses K/V head h / G, G = H_q / H_kv, without repeating
 * K/V in memory).
 * q_dev: [B, H_q, T, d_h] in `q_dtype` (KVC_F32, or the cache dtype). For a 16-bit cache an F32
 * query is rounded to the cache dtype first. out_dev: [B, H_q, T, d_h] float32, caller-owned.
 * s: KVC_COMMITTED to use each sequence's committed length s_b, or a value every s_b must equal.
 * Precondition: `layer` already holds this chunk, i.e. its fill count is s_b + T for every b
 * (kvc_append(layer, ...) with the same T since the last commit/truncate), else KVC_E_STATE.
 * The library keeps a device workspace for partial results and grows it (stream-ordered
 * cudaMallocAsync) the first time a larger one is needed.
 * Limits: the work plan holds at most 2048 (sequence, row tile) units, where a row tile is at most
 * 16 packed query rows (t, g) on the decode and CUDA-core kernels and 128 on the tensor-core chunk
 * kernel (16-bit caches, d_h = 128, G * T > 16: B * ceil(G * T / 128) <= 2048 there); beyond,
 * KVC_E_UNSUPPORTED.
 */
int gqa_cached_attn(kvc_handle h, const void* q_dev, kvc_dtype q_dtype, int layer, int s, int T,
                    int H_q, float* out_dev, void* stream);

/*
 * gqa_cached_attn_rope — gqa_cached_attn with the queries rotated in the attention kernel's prologue:
 * query row t of sequence b is turned by its absolute position s_b + t in float32 (then, for a 16-bit
 * cache, rounded to the cache dtype) before it attends. q_dev holds the queries BEFORE RoPE; the cache
 * must hold keys stored rotated (kvc_append_rope). Arguments, layout and errors are gqa_cached_attn's,
 * plus KVC_E_STATE when kvc_set_rope was not called.
 */
int gqa_cached_attn_rope(kvc_handle h, const void* q_dev, kvc_dtype q_dtype, int layer, int s, int T,
                         int H_q, float* out_dev, void* stream);

/*
 * gqa_cached_attn_append — one layer's step in one call: store the chunk's K/V rows at positions
 * [s_b, s_b + T) (what kvc_append, or with rope != 0 kvc_append_rope, does), then attend its T queries
 * over all s_b + T stored rows (what gqa_cached_attn / gqa_cached_attn_rope with s = KVC_COMMITTED
 * does). Defined by: "KV cache, incremental decode, ...", §2.3 (write the new keys and values at
 * absolute positions [s, s + T), then attend with causal_mask(T, s + T, q_offset = s)) and §4 (update,
 * then attention over the returned rows).
 * k_new_dev, v_new_dev: [B, H_kv, T, d_h] in `in_dtype` (kvc_append's rule); q_dev, out_dev and
 * q_dtype: gqa_cached_attn's. The caller keeps ownership of every buffer; the chunk is copied into the
 * store before the call's kernels finish, so its buffers may be reused once the stream reaches them.
 * Results are bit-identical to the two separate calls: the stored rows are rounded (and rotated) the
 * same way and the attention reads exactly the stored values. On the tensor-core decode kernel (16-bit
 * caches with d_h 64 or 128, fp8 caches with d_h 128, G * T <= 16) this is ONE launch: the CTA that
 * attends over a new row's tile stores the row first. Other shapes launch the append kernel, then the
 * attention kernel.
 * Precondition: the layer holds no rows appended since the last commit/truncate (its fill equals the
 * committed lengths), else KVC_E_STATE. Every error of kvc_append and gqa_cached_attn applies; on any
 * error nothing changes (a paged cache may keep blocks mapped for the coming positions when a CUDA
 * launch itself fails, as kvc_append does).
 */
int gqa_cached_attn_append(kvc_handle h, int layer, const void* k_new_dev, const void* v_new_dev,
                           kvc_dtype in_dtype, const void* q_dev, kvc_dtype q_dtype, int T, int H_q,
                           float* out_dev, int rope, void* stream);

/*
 * kvc_status — synchronise `stream` and report device-side failures: KVC_E_DEVICE_TIMEOUT if a
 * kernel's bounded wait gave up since the last call (the flag is then cleared), KVC_E_DEVICE_BOUNDS
 * if (debug builds) a kernel's index check skipped a store, KVC_E_CUDA on a sticky CUDA error, else
 * KVC_OK.
 */
int kvc_status(kvc_handle h, void* stream);

/* kvc_last_error — copy the last error message (of h, or of the calling thread when h is NULL). */
int kvc_last_error(kvc_handle h, char* buf, size_t n);

/*
 * kvc_set_split_keys — keys per split of the split-K attention kernel; 0 restores the automatic
 * choice. Rounded up to the kernel's tile. A tuning knob: results do not depend on it beyond
 * floating-point reassociation.
 */
int kvc_set_split_keys(kvc_handle h, int keys);

/*
 * gqa_cached_attn_noalloc — gqa_cached_attn for callers that cannot let the library allocate device
 * memory. The pages have no counterpart: it is an operational variant of the same computation.
 * Who needs it: a serving process that reserves its device memory up front (most of the HBM goes to
 * the KV cache) and forbids allocations while it serves; a caller whose memory is owned by another
 * framework's pool; a latency-critical path that must not stall or fail on an allocation.
 * Arguments, results, errors and kernels are those of gqa_cached_attn. The split-K partial results
 * and merge counters live in one fixed 8 MiB device array inside the library instead of the handle's
 * workspace; nothing is allocated (no cudaMalloc/cudaMallocAsync/cudaFree, no library allocator).
 * - A call whose plan needs more than the 8 MiB returns KVC_E_UNSUPPORTED (the message gives both
 *   sizes); every GPU that loads the library holds the array until the process exits.
 * - The first call on each device looks up the array's address (cudaGetSymbolAddress, with that
 *   device current); make that first call before any stream capture.
 * - All calls share the array and it keeps the last call's contents; each call clears the counters it
 *   needs (cudaMemsetAsync on `stream`) before its kernel. Calls that overlap on the GPU (unordered
 *   streams) race on the array and give wrong results: order them on one stream.
 */
int gqa_cached_attn_noalloc(kvc_handle h, const void* q_dev, kvc_dtype q_dtype, int layer, int s, int T,
                            int H_q, float* out_dev, void* stream);

/*
 * kvc_selftest_wait_timeout — operational self-test (no counterpart on the pages): launch one thread
 * that waits on a barrier phase nothing completes and gives up after `limit_us` microseconds
 * (1 .. 1,000,000), exactly as the attention kernels' bounded waits do. The next kvc_status then
 * returns KVC_E_DEVICE_TIMEOUT and clears the flag; the handle stays usable. No fault is raised.
 */
int kvc_selftest_wait_timeout(kvc_handle h, int limit_us, void* stream);

/*
 * kvc_launch_count — number of kernels this handle has enqueued since kvc_create (host counter,
 * incremented at each successful launch). Instrumentation for benchmarks; 0 for NULL.
 */
uint64_t kvc_launch_count(kvc_handle h);

/*
 * kvc_debug_check_guards — the stand-in for a memory checker (no counterpart on the pages). In a
 * library built with KVC_DEBUG_BOUNDS (libkvc_debug.so), every device buffer the library allocates
 * for the handle (its store when kvc_create* allocated it, the lengths, status word, merge counters,
 * split workspace, block table and rotary table) has a 64 KiB guard band of byte 0xA5 on each side,
 * and every kernel checks the index of each global store against its buffer, skipping and reporting
 * (through kvc_status, KVC_E_DEVICE_BOUNDS) one that fails. This call synchronises `stream` and
 * compares every guard band with its byte: KVC_OK, or KVC_E_DEVICE_BOUNDS naming the buffer, the side
 * and the farthest stray byte. Stores the caller owns (kvc_create_external, caller pools) have no
 * guards. A release build returns KVC_E_UNSUPPORTED.
 */
int kvc_debug_check_guards(kvc_handle h, void* stream);

/*
 * kvc_workspace_bytes — device bytes the handle holds for split-K partial results (grown on demand by
 * gqa_cached_attn, gqa_cached_attn_rope and mla_cached_attn; never by gqa_cached_attn_noalloc).
 * Instrumentation (no counterpart on the pages); 0 for NULL and before the first split call.
 */
size_t kvc_workspace_bytes(kvc_handle h);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
