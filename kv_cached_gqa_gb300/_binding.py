"""ctypes binding to `libkvc.so` — argument marshalling only.

Every function here has the name of the C entry point it calls, converts torch tensors to device
pointers and the current CUDA stream to a `cudaStream_t`, and raises `KvcError` on a negative
return code. No step of the attention path runs in Python: if the library is missing, `load()`
raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os

# KVC_DEBUG_BOUNDS=1 selects the debug build: guard bands around every library buffer and an index
# check on every kernel store (kvc_debug_check_guards); it computes the same results, more slowly.
_LIB_NAME = "libkvc_debug.so" if os.environ.get("KVC_DEBUG_BOUNDS") == "1" else "libkvc.so"
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", _LIB_NAME)
_lib = None

KVC_F32, KVC_F16, KVC_BF16, KVC_FP8_E4M3 = 0, 1, 2, 3
KVC_ROPE_HALF, KVC_ROPE_INTERLEAVED = 0, 1
ROPE_STYLE = {"half": KVC_ROPE_HALF, "interleaved": KVC_ROPE_INTERLEAVED}
KVC_COMMITTED = -1
KVC_MAX_BATCH = 1024
ERRORS = {0: "KVC_OK", -1: "KVC_E_INVAL", -2: "KVC_E_CAPACITY", -3: "KVC_E_STATE", -4: "KVC_E_CUDA",
          -5: "KVC_E_DEVICE_TIMEOUT", -6: "KVC_E_UNSUPPORTED", -7: "KVC_E_NOMEM", -8: "KVC_E_DEVICE_BOUNDS"}

# exported symbols and their C signatures (restype, argtypes)
_c_int, _vp, _sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
_i32p = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = {
    "kvc_create": (_c_int, [ctypes.POINTER(_vp), _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "kvc_create_external": (_c_int, [ctypes.POINTER(_vp), _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     _vp, _vp, _vp]),
    "kvc_create_paged": (_c_int, [ctypes.POINTER(_vp), _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_int, _vp, _vp, _vp]),
    "kvc_block_table": (_c_int, [_vp, _i32p, _i32p]),
    "kvc_create_latent": (_c_int, [ctypes.POINTER(_vp), _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp,
                                   _vp]),
    "mla_cached_attn": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.c_float, _vp, _vp]),
    "kvc_destroy": (_c_int, [_vp]),
    "kvc_append": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _c_int, _vp]),
    "kvc_append_rope": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _c_int, _vp]),
    "kvc_set_rope": (_c_int, [_vp, ctypes.c_double, _c_int, _vp]),
    "kvc_set_kv_scales": (_c_int, [_vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]),
    "kvc_commit": (_c_int, [_vp, _vp]),
    "kvc_truncate": (_c_int, [_vp, _c_int, _vp]),
    "kvc_truncate_ragged": (_c_int, [_vp, _i32p, _vp]),
    "kvc_set_lengths": (_c_int, [_vp, _i32p, _vp]),
    "kvc_seq_len": (_c_int, [_vp, _c_int, _i32p]),
    "kvc_positions": (_c_int, [_vp, _c_int, _vp, _vp]),
    "kvc_nbytes": (_sz, [_vp]),
    "kvc_layer_ptrs": (_c_int, [_vp, _c_int, ctypes.POINTER(_vp), ctypes.POINTER(_vp)]),
    "gqa_cached_attn": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "gqa_cached_attn_rope": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "gqa_cached_attn_noalloc": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "gqa_cached_attn_append": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _vp, _c_int,
                                        _vp]),
    "kvc_status": (_c_int, [_vp, _vp]),
    "kvc_last_error": (_c_int, [_vp, ctypes.c_char_p, _sz]),
    "kvc_set_split_keys": (_c_int, [_vp, _c_int]),
    "kvc_launch_count": (ctypes.c_uint64, [_vp]),
    "kvc_workspace_bytes": (_sz, [_vp]),
    "kvc_debug_check_guards": (_c_int, [_vp, _vp]),
    "kvc_selftest_wait_timeout": (_c_int, [_vp, _c_int, _vp]),
    "kvc_synth_fill_normal_f32": (_c_int, [_vp, _sz, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                           ctypes.c_float, _vp]),
}


class KvcError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load `libkvc.so` (built by `kv_cached_gqa_gb300.build`); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _err(h) -> str:
    buf = ctypes.create_string_buffer(512)
    load().kvc_last_error(h, buf, 512)
    return buf.value.decode(errors="replace")


def _check(rc: int, h=None):
    if rc != 0:
        raise KvcError(rc, _err(h))


def _torch():
    import torch
    return torch


_DTYPE_CODES = None


def dtype_code(t) -> int:
    global _DTYPE_CODES
    if _DTYPE_CODES is None:                  # built once: this runs on every call of the hot path
        torch = _torch()
        _DTYPE_CODES = {torch.float32: KVC_F32, torch.float16: KVC_F16, torch.bfloat16: KVC_BF16,
                        torch.float8_e4m3fn: KVC_FP8_E4M3}
    return _DTYPE_CODES[t]


def torch_dtype(code: int):
    torch = _torch()
    return {KVC_F32: torch.float32, KVC_F16: torch.float16, KVC_BF16: torch.bfloat16,
            KVC_FP8_E4M3: torch.float8_e4m3fn}[code]


def _stream(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


class Cache:
    """A KV cache handle over torch-allocated storage (caller-owned K and V tensors)."""

    def __init__(self, L, B, H_kv, d_h, max_len, dtype, device="cuda", stream=None):
        torch = _torch()
        self.L, self.B, self.H_kv, self.d_h, self.max_len = L, B, H_kv, d_h, max_len
        self.dtype = dtype if isinstance(dtype, int) else dtype_code(dtype)
        shape = (L, B, H_kv, max_len, d_h)
        self.k = torch.zeros(shape, dtype=torch_dtype(self.dtype), device=device)
        self.v = torch.zeros(shape, dtype=torch_dtype(self.dtype), device=device)
        h = ctypes.c_void_p()
        _check(load().kvc_create_external(ctypes.byref(h), L, B, H_kv, d_h, max_len, self.dtype,
                                          self.k.data_ptr(), self.v.data_ptr(), _stream(stream)))
        self.h = h

    def close(self):
        if self.h is not None and self.h.value:
            load().kvc_destroy(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DeviceArray:
    """A device buffer the library owns, described by `__cuda_array_interface__` so torch can view it."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 3, "strides": None}


def device_view(ptr: int, shape, code: int):
    """A torch tensor over `shape` elements of cache dtype `code` at device address `ptr` (no copy)."""
    torch = _torch()
    typestr = {KVC_F32: "<f4", KVC_F16: "<f2", KVC_BF16: "<i2", KVC_FP8_E4M3: "|u1"}[code]
    t = torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")
    return t.view(torch_dtype(code)) if code in (KVC_BF16, KVC_FP8_E4M3) else t


class OwnedCache(Cache):
    """A KV cache whose store the library allocates, zero-fills and frees (kvc_create). `.k` and `.v`
    are views of the library's store (through kvc_layer_ptrs), valid until `close()`."""

    def __init__(self, L, B, H_kv, d_h, max_len, dtype, stream=None):
        self.L, self.B, self.H_kv, self.d_h, self.max_len = L, B, H_kv, d_h, max_len
        self.dtype = dtype if isinstance(dtype, int) else dtype_code(dtype)
        h = ctypes.c_void_p()
        self.h = None
        _check(load().kvc_create(ctypes.byref(h), L, B, H_kv, d_h, max_len, self.dtype, _stream(stream)))
        self.h = h
        k0, v0 = kvc_layer_ptrs(self, 0)
        shape = (L, B, H_kv, max_len, d_h)
        self.k = device_view(k0, shape, self.dtype)
        self.v = device_view(v0, shape, self.dtype)

    def close(self):
        self.k = self.v = None
        super().close()


class PagedCache(Cache):
    """A paged KV cache handle over torch-allocated pools, each [L, n_blocks, H_kv, block_size, d_h]."""

    def __init__(self, L, B, H_kv, d_h, max_len, block_size, n_blocks, dtype, device="cuda", stream=None):
        torch = _torch()
        self.L, self.B, self.H_kv, self.d_h, self.max_len = L, B, H_kv, d_h, max_len
        self.block_size, self.n_blocks = block_size, n_blocks
        self.max_blocks = -(-max_len // block_size)
        self.dtype = dtype if isinstance(dtype, int) else dtype_code(dtype)
        shape = (L, n_blocks, H_kv, block_size, d_h)
        self.k = torch.zeros(shape, dtype=torch_dtype(self.dtype), device=device)
        self.v = torch.zeros(shape, dtype=torch_dtype(self.dtype), device=device)
        h = ctypes.c_void_p()
        self.h = None
        _check(load().kvc_create_paged(ctypes.byref(h), L, B, H_kv, d_h, max_len, block_size, n_blocks,
                                       self.dtype, self.k.data_ptr(), self.v.data_ptr(), _stream(stream)))
        self.h = h


class LatentCache(Cache):
    """A latent (MLA) cache over torch-allocated stores: latent c [L, B, max_len, r] (in .k) and RoPE key
    k^R [L, B, max_len, d_rope] (in .v)."""

    def __init__(self, L, B, r, d_rope, max_len, dtype, device="cuda", stream=None):
        torch = _torch()
        self.L, self.B, self.H_kv, self.max_len = L, B, 1, max_len
        self.r, self.d_rope, self.d_h = r, d_rope, r
        self.dtype = dtype if isinstance(dtype, int) else dtype_code(dtype)
        self.k = torch.zeros((L, B, max_len, r), dtype=torch_dtype(self.dtype), device=device)
        self.v = torch.zeros((L, B, max_len, d_rope), dtype=torch_dtype(self.dtype), device=device)
        h = ctypes.c_void_p()
        self.h = None
        _check(load().kvc_create_latent(ctypes.byref(h), L, B, r, d_rope, max_len, self.dtype,
                                        self.k.data_ptr(), self.v.data_ptr(), _stream(stream)))
        self.h = h


def kvc_create_latent(L, B, r, d_rope, max_len, dtype, stream=None) -> LatentCache:
    return LatentCache(L, B, r, d_rope, max_len, dtype, stream=stream)


def mla_cached_attn(c: LatentCache, q_lat, q_rope, layer: int, scale: float, s: int = KVC_COMMITTED, out=None,
                    stream=None):
    """q_lat [B, H, T, r], q_rope [B, H, T, d_rope] -> out [B, H, T, r] float32 (the attended latent)."""
    torch = _torch()
    if q_lat.dim() != 4 or q_lat.shape[0] != c.B or q_lat.shape[3] != c.r:
        raise ValueError("q_lat must be [B, H, T, r]")
    if tuple(q_rope.shape) != (q_lat.shape[0], q_lat.shape[1], q_lat.shape[2], c.d_rope) or q_rope.dtype != q_lat.dtype:
        raise ValueError("q_rope must be [B, H, T, d_rope] of q_lat's dtype")
    if out is None:
        out = torch.empty(q_lat.shape, dtype=torch.float32, device=q_lat.device)
    _check(load().mla_cached_attn(c.h, _ptr(q_lat), _ptr(q_rope), dtype_code(q_lat.dtype), layer, s,
                                  int(q_lat.shape[2]), int(q_lat.shape[1]), float(scale), _ptr(out),
                                  _stream(stream)), c.h)
    return out


def kvc_create(L, B, H_kv, d_h, max_len, dtype, stream=None) -> OwnedCache:
    """A cache whose store the library allocates and zero-fills (and frees in close())."""
    return OwnedCache(L, B, H_kv, d_h, max_len, dtype, stream=stream)


def kvc_create_external(L, B, H_kv, d_h, max_len, dtype, stream=None) -> Cache:
    """A cache over torch-allocated, zeroed K and V tensors (kept as `.k` and `.v`)."""
    return Cache(L, B, H_kv, d_h, max_len, dtype, stream=stream)


def kvc_append(c: Cache, layer: int, k_new, v_new, stream=None):
    """K/V cache: k_new, v_new [B, H_kv, T, d_h]. Latent cache: k_new = latent [B, T, r], v_new = RoPE key
    [B, T, d_rope]."""
    if isinstance(c, LatentCache):
        if k_new.dim() != 3 or v_new.dim() != 3 or k_new.dtype != v_new.dtype or k_new.shape[:2] != v_new.shape[:2]:
            raise ValueError("latent chunk [B, T, r] and RoPE-key chunk [B, T, d_rope] of one dtype expected")
        if k_new.shape[0] != c.B or k_new.shape[2] != c.r or v_new.shape[2] != c.d_rope:
            raise ValueError("chunk shapes do not match the latent cache")
        T = int(k_new.shape[1])
    else:
        if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype or k_new.dim() != 4:
            raise ValueError("k_new and v_new must both be [B, H_kv, T, d_h] of one dtype")
        if tuple(k_new.shape[:2]) != (c.B, c.H_kv) or k_new.shape[3] != c.d_h:
            raise ValueError("k_new shape does not match the cache")
        T = int(k_new.shape[2])
    _check(load().kvc_append(c.h, layer, _ptr(k_new), _ptr(v_new), dtype_code(k_new.dtype), T, _stream(stream)),
           c.h)


def kvc_create_paged(L, B, H_kv, d_h, max_len, block_size, n_blocks, dtype, stream=None) -> PagedCache:
    return PagedCache(L, B, H_kv, d_h, max_len, block_size, n_blocks, dtype, stream=stream)


def kvc_block_table(c: PagedCache):
    """The block table as B lists of ceil(max_len / block_size) physical blocks (-1 = none), and the
    number of free pool blocks."""
    tab = (ctypes.c_int32 * (c.B * c.max_blocks))()
    n_free = ctypes.c_int32()
    _check(load().kvc_block_table(c.h, tab, ctypes.byref(n_free)), c.h)
    flat = [int(x) for x in tab]
    return [flat[b * c.max_blocks:(b + 1) * c.max_blocks] for b in range(c.B)], int(n_free.value)


def kvc_set_rope(c: Cache, base: float, style="half", stream=None):
    """Build the handle's rotary table (theta_i = base^(-2i/d_h)); style "half" or "interleaved"."""
    code = ROPE_STYLE[style] if isinstance(style, str) else int(style)
    _check(load().kvc_set_rope(c.h, float(base), code, _stream(stream)), c.h)


def kvc_append_rope(c: Cache, layer: int, k_new, v_new, stream=None):
    """kvc_append with the keys (given before RoPE) rotated by their positions inside the append."""
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype or k_new.dim() != 4:
        raise ValueError("k_new and v_new must both be [B, H_kv, T, d_h] of one dtype")
    if tuple(k_new.shape[:2]) != (c.B, c.H_kv) or k_new.shape[3] != c.d_h:
        raise ValueError("k_new shape does not match the cache")
    _check(load().kvc_append_rope(c.h, layer, _ptr(k_new), _ptr(v_new), dtype_code(k_new.dtype),
                                  int(k_new.shape[2]), _stream(stream)), c.h)


def kvc_set_kv_scales(c: Cache, k_scale, v_scale):
    """Per-layer scales of an fp8 cache (sequences of L floats, or one float for every layer)."""
    def arr(x):
        vals = [float(x)] * c.L if isinstance(x, (int, float)) else [float(y) for y in x]
        return (ctypes.c_float * c.L)(*vals)
    _check(load().kvc_set_kv_scales(c.h, arr(k_scale), arr(v_scale)), c.h)


def kvc_commit(c: Cache, stream=None):
    _check(load().kvc_commit(c.h, _stream(stream)), c.h)


def kvc_truncate(c: Cache, n: int, stream=None):
    _check(load().kvc_truncate(c.h, int(n), _stream(stream)), c.h)


def kvc_truncate_ragged(c: Cache, n, stream=None):
    arr = (ctypes.c_int32 * c.B)(*[int(x) for x in n])
    _check(load().kvc_truncate_ragged(c.h, arr, _stream(stream)), c.h)


def kvc_set_lengths(c: Cache, n, stream=None):
    """Set every layer's fill and every committed length to n[b] (the rows [0, n_b) already in the store)."""
    arr = (ctypes.c_int32 * c.B)(*[int(x) for x in n])
    _check(load().kvc_set_lengths(c.h, arr, _stream(stream)), c.h)


def kvc_seq_len(c: Cache, layer: int = -1):
    arr = (ctypes.c_int32 * c.B)()
    _check(load().kvc_seq_len(c.h, layer, arr), c.h)
    return [int(x) for x in arr]


def kvc_positions(c: Cache, T: int, stream=None):
    torch = _torch()
    out = torch.empty((c.B, T), dtype=torch.int32, device=c.k.device)
    _check(load().kvc_positions(c.h, T, out.data_ptr(), _stream(stream)), c.h)
    return out


def kvc_nbytes(c: Cache) -> int:
    return int(load().kvc_nbytes(c.h))


def kvc_layer_ptrs(c: Cache, layer: int):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().kvc_layer_ptrs(c.h, layer, ctypes.byref(k), ctypes.byref(v)), c.h)
    return k.value, v.value


def gqa_cached_attn(c: Cache, q, layer: int, s: int = KVC_COMMITTED, out=None, stream=None):
    """q [B, H_q, T, d_h] (float32 or the cache dtype) -> out [B, H_q, T, d_h] float32."""
    torch = _torch()
    if q.dim() != 4 or q.shape[0] != c.B or q.shape[3] != c.d_h:
        raise ValueError("q must be [B, H_q, T, d_h]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check(load().gqa_cached_attn(c.h, _ptr(q), dtype_code(q.dtype), layer, s, int(q.shape[2]),
                                  int(q.shape[1]), _ptr(out), _stream(stream)), c.h)
    return out


def gqa_cached_attn_rope(c: Cache, q, layer: int, s: int = KVC_COMMITTED, out=None, stream=None):
    """gqa_cached_attn with the queries (given before RoPE) rotated by their positions s_b + t."""
    torch = _torch()
    if q.dim() != 4 or q.shape[0] != c.B or q.shape[3] != c.d_h:
        raise ValueError("q must be [B, H_q, T, d_h]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check(load().gqa_cached_attn_rope(c.h, _ptr(q), dtype_code(q.dtype), layer, s, int(q.shape[2]),
                                       int(q.shape[1]), _ptr(out), _stream(stream)), c.h)
    return out


def gqa_cached_attn_append(c: Cache, layer: int, k_new, v_new, q, out=None, rope: bool = False, stream=None):
    """kvc_append (kvc_append_rope with rope=True) of k_new, v_new [B, H_kv, T, d_h], then
    gqa_cached_attn (gqa_cached_attn_rope) of q [B, H_q, T, d_h] over the committed lengths, in one call
    -> out [B, H_q, T, d_h] float32."""
    torch = _torch()
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype or k_new.dim() != 4:
        raise ValueError("k_new and v_new must both be [B, H_kv, T, d_h] of one dtype")
    if tuple(k_new.shape[:2]) != (c.B, c.H_kv) or k_new.shape[3] != c.d_h:
        raise ValueError("k_new shape does not match the cache")
    if q.dim() != 4 or q.shape[0] != c.B or q.shape[3] != c.d_h or q.shape[2] != k_new.shape[2]:
        raise ValueError("q must be [B, H_q, T, d_h] with the chunk's T")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check(load().gqa_cached_attn_append(c.h, layer, _ptr(k_new), _ptr(v_new), dtype_code(k_new.dtype), _ptr(q),
                                         dtype_code(q.dtype), int(q.shape[2]), int(q.shape[1]), _ptr(out),
                                         1 if rope else 0, _stream(stream)), c.h)
    return out


def gqa_cached_attn_noalloc(c: Cache, q, layer: int, out, s: int = KVC_COMMITTED, stream=None):
    """gqa_cached_attn for callers that cannot let the library allocate: scratch comes from a fixed
    8 MiB device array in the library, so `out` must be supplied by the caller."""
    if q.dim() != 4 or q.shape[0] != c.B or q.shape[3] != c.d_h or out.shape != q.shape:
        raise ValueError("q and out must be [B, H_q, T, d_h]")
    _check(load().gqa_cached_attn_noalloc(c.h, _ptr(q), dtype_code(q.dtype), layer, s, int(q.shape[2]),
                                          int(q.shape[1]), _ptr(out), _stream(stream)), c.h)
    return out


def kvc_status(c: Cache, stream=None):
    _check(load().kvc_status(c.h, _stream(stream)), c.h)


def kvc_set_split_keys(c: Cache, keys: int):
    _check(load().kvc_set_split_keys(c.h, keys), c.h)


def kvc_selftest_wait_timeout(c: Cache, limit_us: int, stream=None):
    _check(load().kvc_selftest_wait_timeout(c.h, int(limit_us), _stream(stream)), c.h)


def kvc_launch_count(c: Cache) -> int:
    return int(load().kvc_launch_count(c.h))


def kvc_workspace_bytes(c: Cache) -> int:
    return int(load().kvc_workspace_bytes(c.h))


def kvc_debug_check_guards(c: Cache, stream=None):
    """Debug builds: raise KvcError (KVC_E_DEVICE_BOUNDS) if a guard band of a library buffer was written."""
    _check(load().kvc_debug_check_guards(c.h, _stream(stream)), c.h)


def synth_fill_normal(out, seed: int, stream_id: int, std: float = 1.0, offset: int = 0, stream=None):
    """Fill a float32 CUDA tensor with the seeded draws of `kvc_synth` (same bits as the host)."""
    torch = _torch()
    if out.dtype != torch.float32:
        raise ValueError("float32 tensor expected")
    rc = load().kvc_synth_fill_normal_f32(_ptr(out), out.numel(), offset, seed, stream_id, std,
                                          _stream(stream))
    if rc != 0:
        raise KvcError(rc, "synthetic fill failed")
    return out
