"""Small-case sweep on the debug build of the library (run in a process of its own with
KVC_DEBUG_BOUNDS=1, by tests/test_gpu_debug_bounds.py).

The debug build puts guard bands around every buffer the library allocates and checks the index of
every global store in every kernel. This sweep drives the library-owned caches (their stores guarded
too) through ragged prefills, truncates and chunks over the sizes where index arithmetic goes wrong
(chunk lengths around tile edges, empty and one-key sequences, the group sizes and head widths the
kernels serve) and checks, after every case: the outputs against the oracle, the stored rows bit for
bit, no index check fired (kvc_status), and every guard band intact (kvc_debug_check_guards). It prints
one JSON line with the case count and exits non-zero on the first failure.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tests.gpu_parity import Mirror, check_outputs  # noqa: E402

LENGTHS = ([0, 1, 63, 64, 65], [129, 0, 7], [255, 256, 1])
CASES = [  # (dtype, d_h, H_kv, G, T values)
    ("f32", 32, 2, 1, (1, 2, 3, 5, 8, 17)),
    ("f16", 64, 2, 3, (1, 2, 3, 5, 8, 17, 64)),
    ("bf16", 128, 2, 4, (1, 2, 3, 5, 8, 17, 64, 128, 129)),
    ("f16", 128, 1, 8, (1, 2, 3, 17, 64)),
    ("e4m3", 128, 2, 4, (1, 8, 17)),
    ("bf16", 64, 3, 1, (1, 4, 16)),
]


def one_case(dtype, d, H_kv, G, T, lengths, block=None):
    m = Mirror(1, len(lengths), H_kv, d, max(lengths) + T + 3, dtype, seed=T * 7 + len(lengths),
               owned=block is None, block=block)
    s0 = max(max(lengths), 1)
    m.append(0, s0)
    m.commit()
    m.truncate(lengths)
    m.append(0, T)
    got, want = m.attend(0, H_kv * G, T)
    check_outputs(got, want, dtype, f"{dtype} d{d} G{G} T{T} s{lengths}")
    m.check_state()
    m.kb.kvc_status(m.gpu)
    m.kb.kvc_debug_check_guards(m.gpu)
    m.close()


def main():
    from kv_cached_gqa_gb300 import _binding as kb
    assert kb.lib_path().endswith("libkvc_debug.so"), kb.lib_path()
    n = 0
    for dtype, d, H_kv, G, Ts in CASES:
        for T in Ts:
            for lengths in LENGTHS:
                one_case(dtype, d, H_kv, G, T, lengths)
                n += 1
    for T in (1, 5, 64):                                     # paged pools (the library's table guarded)
        one_case("bf16", 128, 2, 4, T, [100, 0, 17], block=16)
        n += 1
    print(json.dumps({"cases": n, "library": os.path.basename(kb.lib_path())}))


if __name__ == "__main__":
    main()
