"""The C-ABI library builds, loads and exports every entry point `include/*.h` declares.

No compute call is made here (no GPU): only the host-side argument checks that return before any
CUDA call.
"""
import ctypes
import glob
import os
import re

import pytest

from tests.conftest import ROOT

DECL = re.compile(r"^\s*(?:int|size_t|uint64_t|const char\s*\*)\s+(\w+)\s*\(", re.M)


def declared_symbols():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(path) as f:
            names.update(DECL.findall(f.read()))
    return names


@pytest.fixture(scope="module")
def lib():
    from kv_cached_gqa_gb300 import build, _binding
    build.build()
    return _binding.load()


def test_headers_declare_the_entry_points():
    names = declared_symbols()
    for n in ("kvc_create", "kvc_append", "kvc_commit", "kvc_truncate", "kvc_nbytes", "gqa_cached_attn",
              "kvc_truncate_ragged", "kvc_seq_len", "kvc_positions", "kvc_layer_ptrs", "kvc_status",
              "kvc_create_paged", "kvc_block_table", "kvc_set_rope", "kvc_append_rope", "gqa_cached_attn_rope", "kvc_set_kv_scales",
              "kvc_create_latent", "mla_cached_attn", "kvc_set_lengths", "gqa_cached_attn_noalloc",
              "kvc_workspace_bytes", "gqa_cached_attn_append"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from kv_cached_gqa_gb300 import _binding
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _binding.SIGNATURES, f"{name} has no binding"


def test_debug_library_exports_the_same_symbols(lib):
    from kv_cached_gqa_gb300 import build
    dbg = ctypes.CDLL(build.LIB_DEBUG)
    for name in declared_symbols():
        assert hasattr(dbg, name), name
    dbg.kvc_debug_check_guards.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert dbg.kvc_debug_check_guards(None, None) == -1
    assert lib.kvc_debug_check_guards(None, None) == -1


def test_library_is_built_for_sm_103a_only():
    from kv_cached_gqa_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _err(lib):
    buf = ctypes.create_string_buffer(256)
    lib.kvc_last_error(None, buf, 256)
    return buf.value.decode()


def test_host_validation_without_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.kvc_create(ctypes.byref(h), 0, 1, 1, 64, 16, 0, None) == -1
    assert "positive" in _err(lib)
    assert lib.kvc_create(ctypes.byref(h), 1, 1, 1, 48, 16, 0, None) == -6     # d_h 48 unsupported
    assert lib.kvc_create(ctypes.byref(h), 1, 1, 1, 64, 16, 7, None) == -1     # unknown dtype
    assert lib.kvc_create(ctypes.byref(h), 1, 2000, 1, 64, 16, 0, None) == -1  # B > KVC_MAX_BATCH
    assert lib.kvc_create(None, 1, 1, 1, 64, 16, 0, None) == -1
    assert lib.kvc_create_external(ctypes.byref(h), 1, 1, 1, 64, 16, 0, None, None, None) == -1
    assert lib.kvc_create_external(ctypes.byref(h), 1, 1, 1, 64, 16, 0, 16, 512, None) == -1  # misaligned
    assert h.value is None
    assert lib.kvc_nbytes(None) == 0
    assert lib.kvc_launch_count(None) == 0
    assert lib.kvc_destroy(None) == 0
    for rc in (lib.kvc_append(None, 0, None, None, 0, 1, None), lib.kvc_commit(None, None),
               lib.kvc_truncate(None, 0, None), lib.kvc_seq_len(None, -1, None),
               lib.gqa_cached_attn(None, None, 0, 0, -1, 1, 1, None, None),
               lib.kvc_status(None, None), lib.kvc_set_split_keys(None, 0)):
        assert rc == -1
    assert "null handle" in _err(lib)
    # paged: rejected before any CUDA call
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 1, 1, 64, 64, 24, 8, 1, None, None, None) == -1   # not 2^k
    assert "power of two" in _err(lib)
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 1, 1, 64, 64, 8, 8, 1, None, None, None) == -1    # < 16
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 1, 1, 64, 64, 16, 0, 1, None, None, None) == -1   # no blocks
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 1, 1, 64, 64, 16, 8, 1, 256, None, None) == -1    # one pool
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 1, 1, 64, 64, 16, 8, 1, 16, 512, None) == -1      # misaligned
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 1, 1, 48, 64, 16, 8, 1, None, None, None) == -6   # d_h 48
    assert lib.kvc_create_paged(None, 1, 1, 1, 64, 64, 16, 8, 1, None, None, None) == -1
    assert h.value is None
    assert lib.kvc_block_table(None, None, None) == -1
    assert lib.kvc_set_rope(None, 10000.0, 0, None) == -1
    assert lib.kvc_set_kv_scales(None, None, None) == -1
    assert lib.kvc_create_latent(ctypes.byref(h), 1, 1, 24, 64, 16, 2, None, None, None) == -6   # r % 16
    assert lib.kvc_create_latent(ctypes.byref(h), 1, 1, 512, 64, 16, 3, None, None, None) == -1  # fp8
    assert lib.kvc_create_latent(ctypes.byref(h), 1, 1, 512, 64, 16, 2, 256, None, None) == -1   # one store
    assert lib.mla_cached_attn(None, None, None, 0, 0, -1, 1, 1, ctypes.c_float(1.0), None, None) == -1
    assert lib.kvc_create(ctypes.byref(h), 1, 1, 1, 32, 16, 3, None) == -6     # fp8 rows of 32 bytes
    assert lib.kvc_create(ctypes.byref(h), 1, 1, 1, 64, 16, 4, None) == -1     # unknown dtype
    assert lib.kvc_append_rope(None, 0, None, None, 0, 1, None) == -1
    assert lib.gqa_cached_attn_rope(None, None, 0, 0, -1, 1, 1, None, None) == -1
    assert lib.kvc_set_lengths(None, None, None) == -1
    assert lib.kvc_workspace_bytes(None) == 0
    lib.kvc_create(None, 1, 1, 1, 64, 16, 0, None)                            # leaves another message
    assert lib.gqa_cached_attn_noalloc(None, None, 0, 0, -1, 1, 1, None, None) == -1
    assert _err(lib) == "null handle"                                        # the call's own message
    lib.kvc_create(None, 1, 1, 1, 64, 16, 0, None)
    assert lib.gqa_cached_attn_append(None, 0, None, None, 0, None, 0, 1, 1, None, 0, None) == -1
    assert _err(lib) == "null handle"


def test_binding_fails_loudly_when_library_missing(monkeypatch, tmp_path):
    from kv_cached_gqa_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load()
