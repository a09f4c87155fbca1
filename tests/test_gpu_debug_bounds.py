"""The debug build as a memory checker: guard bands and store index checks over a small-case sweep.

compute-sanitizer is not used on this pool; in its place the library built with KVC_DEBUG_BOUNDS
surrounds every buffer it allocates with guard bands of a known byte and checks every global store of
every kernel against its buffer. The sweep (tests/debug_bounds_sweep.py) runs in a process of its own,
since the binding loads one library per process.
"""
import ctypes
import json
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT

pytestmark = pytest.mark.gpu


def test_debug_build_sweep_keeps_every_guard_and_bound(gpu_lib):
    env = dict(os.environ, KVC_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, "-m", "tests.debug_bounds_sweep"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["library"] == "libkvc_debug.so" and out["cases"] >= 100


GUARD_PROBE = r"""
import ctypes, json, sys
sys.path.insert(0, %r)
import torch
from kv_cached_gqa_gb300 import _binding as kb
c = kb.OwnedCache(2, 2, 2, 64, 32, kb.KVC_F16)
kb.kvc_debug_check_guards(c)                                 # intact after creation
k_end = kb.kvc_layer_ptrs(c, 1)[0] + kb.kvc_nbytes(c) // 4   # one past the K store's last byte
band = kb.device_view(k_end + 100, (4,), kb.KVC_F16)        # inside the guard band after the store
band.fill_(1.0)
torch.cuda.synchronize()
try:
    kb.kvc_debug_check_guards(c)
    print(json.dumps({"caught": False}))
except kb.KvcError as e:
    print(json.dumps({"caught": True, "code": e.code, "msg": str(e)}))
""" % ROOT


def test_guard_check_reports_a_write_past_the_store(gpu_lib):
    """A write just past the end of the library's K store (into its guard band, memory the library
    allocated) is reported by kvc_debug_check_guards with the buffer's name and side."""
    env = dict(os.environ, KVC_DEBUG_BOUNDS="1")
    r = subprocess.run([sys.executable, "-c", GUARD_PROBE], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["caught"] and out["code"] == -8, out
    assert "K store" in out["msg"] and "after" in out["msg"] and "101 bytes past its end" in out["msg"], out


def test_release_build_has_no_guards(gpu_lib):
    from kv_cached_gqa_gb300 import _binding as kb
    c = kb.OwnedCache(1, 1, 1, 64, 16, kb.KVC_F16)
    with pytest.raises(kb.KvcError) as ei:
        kb.kvc_debug_check_guards(c)
    assert ei.value.code == -6
    c.close()
