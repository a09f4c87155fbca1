"""The library-owned cache through its whole life, and kvc_set_lengths, against the oracle.

kvc_create allocates and zero-fills the store itself ("KV cache decoding", KVCache listing: the
store starts as zeros; "KV cache, incremental decode, ...", §2.5: a preallocated store of
2 L B H_kv N_max d_h elements, §4: nbytes, and update returning every stored row). Here the
library's own store is written by appends, moved by commit, truncate and set_lengths, read back
layer by layer through kvc_layer_ptrs and compared with the oracle bit for bit, never-written zeros
included, and freed by kvc_destroy.
"""
import ctypes

import numpy as np
import pytest

from oracle.kvc_oracle import ITEMSIZE
from tests.gpu_parity import DT, Mirror, check_outputs

pytestmark = pytest.mark.gpu

VIEW = {"f32": np.int32, "f16": np.int16, "bf16": np.int16, "e4m3": np.uint8}


def read_back_every_layer(m):
    """Each layer's K and V through kvc_layer_ptrs, as raw bits, against the oracle's store."""
    kb, torch = m.kb, m.torch
    bits = {np.int32: torch.int32, np.int16: torch.int16, np.uint8: torch.uint8}[VIEW[m.dtype]]
    for layer in range(m.L):
        kp, vp = kb.kvc_layer_ptrs(m.gpu, layer)
        for ptr, want in ((kp, m.ref.k[layer]), (vp, m.ref.v[layer])):
            got = kb.device_view(ptr, (m.B, m.H, m.max_len, m.d), DT[m.dtype]).view(bits)
            np.testing.assert_array_equal(got.cpu().numpy(), want.view(VIEW[m.dtype]))


@pytest.mark.parametrize("dtype,d,H_q", [("bf16", 128, 8), ("f16", 64, 6), ("f32", 32, 4), ("e4m3", 128, 8)])
def test_library_owned_cache_lifecycle(gpu_lib, dtype, d, H_q):
    import torch
    L, B, H_kv, max_len = 3, 3, 2, 300
    m = Mirror(L, B, H_kv, d, max_len, dtype, seed=31, owned=True)
    kb = m.kb
    nbytes = 2 * L * B * H_kv * max_len * d * ITEMSIZE[dtype]
    assert kb.kvc_nbytes(m.gpu) == nbytes == m.ref.nbytes()
    torch.cuda.synchronize()
    read_back_every_layer(m)                                    # the library zero-filled its store
    m.forward(40, H_q, what="prefill")                          # T = 40 on every layer, then commit
    m.truncate([10, 40, 0])
    m.forward(1, H_q, what="decode after a ragged truncate")
    m.set_lengths([40, 25, 7])                                  # over rows a truncate left, and zeros
    m.forward(3, H_q, what="chunk after set_lengths")
    m.check_state()
    read_back_every_layer(m)
    kb.kvc_status(m.gpu)
    lib, h = gpu_lib, m.gpu.h
    m.gpu.k = m.gpu.v = None
    assert lib.kvc_destroy(h) == 0
    m.gpu.h = None


def test_library_owned_store_is_device_memory_of_nbytes(gpu_lib):
    """kvc_create takes its store from the device (free memory drops by at least kvc_nbytes) and
    kvc_destroy gives it back."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    c = kb.kvc_create(4, 8, 4, 128, 4096, kb.KVC_BF16)          # 2 x 64 MiB
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert kb.kvc_nbytes(c) == 2 * 4 * 8 * 4 * 4096 * 128 * 2
    assert free0 - free1 >= kb.kvc_nbytes(c)
    assert not bool(c.k.view(torch.int16).any()) and not bool(c.v.view(torch.int16).any())
    c.close()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    assert torch.cuda.mem_get_info()[0] >= free0 - (16 << 20)


def test_set_lengths_over_rows_left_in_the_store(gpu_lib):
    """A ragged batch set up with set_lengths over rows already in the store (rows a truncate to 0 left
    behind, and zeros) attends as the oracle does, on the tensor-core decode kernel."""
    m = Mirror(2, 4, 2, 128, 600, "bf16", seed=5)
    m.forward(512, 8, check=False)                               # rows for every sequence, then commit
    m.truncate(0)
    m.set_lengths([512, 1, 300, 0])
    errs = m.forward(1, 8, what="decode after set_lengths")
    assert max(errs) <= 2e-3
    m.check_state()
    m.close()


def test_set_lengths_errors_change_nothing(gpu_lib):
    from kv_cached_gqa_gb300 import _binding as kb
    m = Mirror(1, 2, 1, 64, 32, "f16", seed=6)
    m.forward(5, 2, check=False)
    before = (kb.kvc_seq_len(m.gpu), kb.kvc_seq_len(m.gpu, 0))
    for bad in ([33, 0], [-1, 2]):
        with pytest.raises(kb.KvcError) as ei:
            kb.kvc_set_lengths(m.gpu, bad)
        assert ei.value.code == -1
    assert (kb.kvc_seq_len(m.gpu), kb.kvc_seq_len(m.gpu, 0)) == before
    m.check_state()
    m.close()
    p = Mirror(1, 2, 1, 64, 64, "f16", seed=6, block=16)
    with pytest.raises(kb.KvcError) as ei:
        kb.kvc_set_lengths(p.gpu, [16, 16])
    assert ei.value.code == -6
    p.check_state()
    p.close()


def test_library_owned_paged_and_latent_stores(gpu_lib):
    """kvc_create_paged and kvc_create_latent with NULL stores: the library allocates and zero-fills the
    pools, kvc_nbytes is their capacity, kvc_layer_ptrs points into them, kvc_destroy frees them."""
    import torch
    from kv_cached_gqa_gb300 import _binding as kb
    lib = gpu_lib
    stream = torch.cuda.current_stream().cuda_stream
    h = ctypes.c_void_p()
    assert lib.kvc_create_paged(ctypes.byref(h), 2, 3, 2, 128, 100, 16, 20, kb.KVC_F16, None, None, stream) == 0
    assert lib.kvc_nbytes(h) == 2 * 2 * 20 * 2 * 16 * 128 * 2
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    assert lib.kvc_layer_ptrs(h, 1, ctypes.byref(k), ctypes.byref(v)) == 0
    torch.cuda.synchronize()
    pool = kb.device_view(k.value, (20, 2, 16, 128), kb.KVC_F16)
    assert not bool(pool.view(torch.int16).any())
    assert lib.kvc_destroy(h) == 0
    h = ctypes.c_void_p()
    assert lib.kvc_create_latent(ctypes.byref(h), 2, 3, 512, 64, 100, kb.KVC_BF16, None, None, stream) == 0
    assert lib.kvc_nbytes(h) == 2 * 3 * 100 * (512 + 64) * 2
    assert lib.kvc_layer_ptrs(h, 1, ctypes.byref(k), ctypes.byref(v)) == 0
    torch.cuda.synchronize()
    c = kb.device_view(k.value, (3, 100, 512), kb.KVC_BF16)
    kr = kb.device_view(v.value, (3, 100, 64), kb.KVC_BF16)
    assert not bool(c.view(torch.int16).any()) and not bool(kr.view(torch.int16).any())
    assert lib.kvc_destroy(h) == 0
