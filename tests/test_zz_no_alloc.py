"""fa_fwd_splitkv_noalloc: split-KV with the library's built-in scratch buffer.

The entry point exists for callers that cannot allocate device memory (a
memory manager that owns the device, a plugin interface that hands over only
input and output tensors, a path where cudaMalloc's synchronisation is not
acceptable).  It must give the same result as fa_fwd_splitkv with a caller
workspace, and both must match the fp64 oracle.  Every case asks for several
splits, so the partials really pass through the built-in buffer.  This file is
collected last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect this module
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
from parity_util import TOL_LSE, TOL_O, assert_parity, f64, gather  # noqa: E402

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


def _run_noalloc(lib, q, k, v, causal, off, splits):
    from tiled_exact_attention_gb300.api import make_args

    b, sq, hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, hq, sq), dtype=torch.float32, device=DEV)
    a = make_args(q, k, v, o, lse, causal=causal, scale=None, q_pos_offset=off)
    used = ctypes.c_int32(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_fwd_splitkv_noalloc(ctypes.byref(a), splits, ctypes.byref(used), stream)
    return rc, o, lse, used.value


def _run_workspace(q, k, v, causal, off, splits):
    from tiled_exact_attention_gb300 import fa_fwd_splitkv

    return fa_fwd_splitkv(q, k, v, causal=causal, q_pos_offset=off, num_splits=splits, return_splits=True)


def _compare(o1, l1, o2, l2):
    fin = torch.isfinite(l2)
    assert torch.equal(fin, torch.isfinite(l1))
    assert (o1.float() - o2.float()).abs().max().item() <= TOL_O[torch.bfloat16]
    if fin.any():
        assert (l1[fin] - l2[fin]).abs().max().item() <= TOL_LSE


def _oracle_check(q, k, v, causal, off, o, lse, what):
    b, sq, hq, d = q.shape
    rows = oracle.all_rows(b, hq, sq)
    o_ref, l_ref = oracle.attention(f64(q), f64(k), f64(v), causal=causal, q_pos_offset=off,
                                    scale=1.0 / d ** 0.5, rows=rows)
    og, lg = gather(o, lse, rows)
    assert_parity(og, lg, o_ref, l_ref, q.dtype, what)


CASES = [
    # (b, sq, skv, hq, hkv, d, seed), causal, offset, splits
    ((4, 1, 5000, 16, 4, 128, 11), True, 4999, 5),    # decode kernel (GQA fold of 4 heads), merge fused
    ((1, 300, 700, 4, 2, 128, 12), True, None, 3),    # tcgen05 kernel in split mode, then the combine
    ((2, 1, 3000, 32, 2, 128, 14), True, 2999, 4),    # 16 heads per KV head: heads as tile rows, then the combine
]


def test_noalloc_matches_workspace_entry_point_and_oracle_twice(lib):
    from tiled_exact_attention_gb300 import fa_sync_status

    # several problems back to back, each twice: every call reuses the built-in
    # buffer after the previous one filled it
    for (shape, causal, off, splits) in CASES:
        q, k, v = _problem(*shape)
        for _ in range(2):
            rc, o_na, l_na, used_na = _run_noalloc(lib, q, k, v, causal, off, splits)
            assert rc == 0, lib.fa_status_string(rc)
            o_ws, l_ws, used_ws = _run_workspace(q, k, v, causal, off, splits)
            assert fa_sync_status() == 0
            assert used_na == used_ws == splits  # the partials went through the scratch buffer
            _compare(o_na, l_na, o_ws, l_ws)
            _oracle_check(q, k, v, causal, off, o_na, l_na, f"no-alloc {shape}")


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
