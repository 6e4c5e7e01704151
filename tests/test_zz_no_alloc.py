"""fa_fwd_splitkv_noalloc: split-KV with the library's built-in scratch buffer.

The entry point exists for callers that cannot allocate device memory (a
memory manager that owns the device, a plugin interface that hands over only
input and output tensors, a path where cudaMalloc's synchronisation is not
acceptable).  It must give the same result as fa_fwd_splitkv with a caller
workspace.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

from parity_util import TOL_LSE, TOL_O  # noqa: E402

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    from tiled_exact_attention_gb300 import build

    build.build()
    from tiled_exact_attention_gb300 import _lib

    return _lib.load()


def _problem(b, sq, skv, hq, hkv, d, seed):
    from tiled_exact_attention_gb300.inputs import make_custom

    return [t.to(DEV) for t in make_custom(b, sq, skv, hq, hkv, d, "bf16", seed=seed)]


def _run_noalloc(lib, q, k, v, causal, off):
    from tiled_exact_attention_gb300.api import make_args

    b, sq, hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, hq, sq), dtype=torch.float32, device=DEV)
    a = make_args(q, k, v, o, lse, causal=causal, scale=None, q_pos_offset=off)
    used = ctypes.c_int32(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_fwd_splitkv_noalloc(ctypes.byref(a), 0, ctypes.byref(used), stream)
    return rc, o, lse, used.value


def _run_workspace(q, k, v, causal, off):
    from tiled_exact_attention_gb300 import fa_fwd_splitkv

    return fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, return_splits=True)


def _compare(o1, l1, o2, l2):
    fin = torch.isfinite(l2)
    assert torch.equal(fin, torch.isfinite(l1))
    assert (o1.float() - o2.float()).abs().max().item() <= TOL_O[torch.bfloat16]
    if fin.any():
        assert (l1[fin] - l2[fin]).abs().max().item() <= TOL_LSE


def test_noalloc_matches_workspace_entry_point_twice(lib):
    from tiled_exact_attention_gb300 import fa_sync_status

    # two different problems back to back: the second call reuses the same
    # built-in buffer after the first one filled it
    cases = [
        ((4, 1, 5000, 16, 4, 128, 11), True, 4999),   # decode kernel (GQA fold)
        ((1, 300, 700, 4, 2, 128, 12), True, None),   # tcgen05 kernel in split mode
    ]
    for (shape, causal, off) in cases:
        q, k, v = _problem(*shape)
        rc, o_na, l_na, used_na = _run_noalloc(lib, q, k, v, causal, off)
        assert rc == 0, lib.fa_status_string(rc)
        o_ws, l_ws, used_ws = _run_workspace(q, k, v, causal, off)
        assert fa_sync_status() == 0
        assert used_na == used_ws >= 1
        _compare(o_na, l_na, o_ws, l_ws)


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    from tiled_exact_attention_gb300 import _lib
    from tiled_exact_attention_gb300.api import make_args

    # 2 splits x 8 heads x 4096 rows x (128 + 1) floats > 8 MiB
    q, k, v = _problem(1, 4096, 256, 8, 8, 128, 13)
    o = torch.empty_like(q)
    lse = torch.empty((1, 8, 4096), dtype=torch.float32, device=DEV)
    a = make_args(q, k, v, o, lse, causal=False, scale=None, q_pos_offset=None)
    assert lib.fa_splitkv_workspace_size(ctypes.byref(a), 2) > _lib.NOALLOC_SCRATCH_BYTES
    used = ctypes.c_int32(-1)
    rc = lib.fa_fwd_splitkv_noalloc(ctypes.byref(a), 2, ctypes.byref(used),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.FA_ERR_SCRATCH_LIMIT
    assert used.value == -1  # nothing was launched or written
