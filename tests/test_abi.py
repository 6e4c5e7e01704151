"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/fa.h declares, validates arguments before touching the
device, and its split heuristic agrees with the oracle's."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    from tiled_exact_attention_gb300 import build as b

    b.build()
    from tiled_exact_attention_gb300 import _lib

    return _lib.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_function(lib):
    from tiled_exact_attention_gb300 import _lib

    declared = _declared_functions()
    assert len(declared) >= 9
    assert sorted(_lib.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.fa_version() == 3
    for code in range(5):
        assert lib.fa_status_string(code)
    assert lib.fa_status_string(99) == b"unknown status"


def test_heuristic_matches_oracle(lib, oracle_mod):
    for units in (1, 3, 8, 48, 64, 100, 152, 300, 1024):
        for slots in (108, 148, 152, 304):
            for nblk in (1, 2, 7, 64, 512):
                assert lib.fa_num_splits_heuristic(units, slots, nblk, 128) == \
                    oracle_mod.num_splits(units, slots, nblk, 128), (units, slots, nblk)
    assert lib.fa_num_splits_heuristic(48, 108, 1000, 128) == 2
    assert lib.fa_num_splits_heuristic(0, 108, 10, 128) == 1


def _args(**kw):
    from tiled_exact_attention_gb300._lib import FwdArgs

    a = FwdArgs()
    a.dtype, a.b, a.sq, a.skv, a.hq, a.hkv, a.d = 0, 1, 128, 128, 2, 2, 128
    for f in ("q_strides", "k_strides", "v_strides", "o_strides"):
        setattr(a, f, (ctypes.c_int64 * 3)(128 * 2 * 128, 2 * 128, 128))
    a.q = a.k = a.v = a.o = 4096
    a.lse = 4096
    a.causal = 0
    a.scale = 0.125
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,expect", [
    ("dtype", 7, 1), ("b", 0, 1), ("hq", 3, 1), ("causal", 2, 1), ("scale", 0.0, 1),
    ("scale", float("nan"), 1), ("d", 96, 2), ("d", 32, 2), ("q", 0, 1), ("lse", 0, 1), ("q", 4100, 1),
    ("local", 2, 1), ("softcap", -1.0, 1), ("softcap", float("nan"), 1), ("softcap", float("inf"), 1),
])
def test_validation_rejects_before_any_launch(lib, field, value, expect):
    a = _args(**{field: value})
    assert lib.fa_fwd(ctypes.byref(a), None) == expect
    assert lib.fa_fwd_splitkv(ctypes.byref(a), 1, None, 0, None, None) == expect


def test_window_widths_below_minus_one_rejected(lib):
    for wl, wr in ((-2, 0), (0, -2), (-5, -5)):
        a = _args(local=1, window_left=wl, window_right=wr)
        assert lib.fa_fwd(ctypes.byref(a), None) == 1
        assert lib.fa_fwd_splitkv(ctypes.byref(a), 1, None, 0, None, None) == 1
    # the widths are not looked at while local == 0
    a = _args(local=0, window_left=-7, window_right=-7, q=4100)
    assert lib.fa_fwd(ctypes.byref(a), None) == 1  # rejected for the misaligned q only
    a = _kv_args(local=1, window_left=-2)
    assert lib.fa_fwd_kvcache(ctypes.byref(a), 0, None, 0, None, None) == 1
    a = _kv_args(local=3)
    assert lib.fa_fwd_kvcache(ctypes.byref(a), 0, None, 0, None, None) == 1


_LAYOUT_PROBE = r'''
#include <stddef.h>
#include <stdio.h>
#include "fa.h"
#define F(T, f) printf(#T " " #f " %zu %zu\n", offsetof(T, f), sizeof(((T*)0)->f));
int main(void) {
  printf("fa_fwd_args size %zu\n", sizeof(fa_fwd_args));
  printf("fa_kvcache_args size %zu\n", sizeof(fa_kvcache_args));
  printf("fa_varlen_args size %zu\n", sizeof(fa_varlen_args));
  printf("fa_bwd_args size %zu\n", sizeof(fa_bwd_args));
  printf("fa_quant_args size %zu\n", sizeof(fa_quant_args));
  printf("fa_fwd_e4m3_args size %zu\n", sizeof(fa_fwd_e4m3_args));
  printf("fa_splitkv_e4m3_args size %zu\n", sizeof(fa_splitkv_e4m3_args));
  FIELDS
  return 0;
}
'''


def test_ctypes_mirrors_match_header_layout(tmp_path):
    """Every field of the ctypes mirrors sits at the offset, with the size, that a C
    compiler gives the structs declared in include/fa.h."""
    from tiled_exact_attention_gb300._lib import (BwdArgs, E4m3Args, FwdArgs, KvcacheArgs, QuantArgs, SplitkvE4m3Args,
                                                  VarlenArgs)

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    fields = []
    mirrors = {"fa_fwd_args": FwdArgs, "fa_kvcache_args": KvcacheArgs, "fa_varlen_args": VarlenArgs,
               "fa_bwd_args": BwdArgs, "fa_quant_args": QuantArgs, "fa_fwd_e4m3_args": E4m3Args,
               "fa_splitkv_e4m3_args": SplitkvE4m3Args}
    for cname, py in mirrors.items():
        for name, _ in py._fields_:
            fields.append(f"F({cname}, {name})")
    src = tmp_path / "layout.c"
    src.write_text(_LAYOUT_PROBE.replace("FIELDS", "\n  ".join(fields)))
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()
    sizes = {ln.split()[0]: int(ln.split()[2]) for ln in out if ln.split()[1] == "size"}
    for cname, py in mirrors.items():
        assert sizes[cname] == ctypes.sizeof(py), cname
    for ln in out:
        parts = ln.split()
        if parts[1] == "size":
            continue
        struct, name, off, size = parts[0], parts[1], int(parts[2]), int(parts[3])
        py = mirrors[struct]
        desc = getattr(py, name)
        assert (desc.offset, desc.size) == (off, size), (struct, name)


def test_validation_strides_and_null(lib):
    a = _args()
    a.q_strides = (ctypes.c_int64 * 3)(100, 20, 4)  # not multiples of 8 elements
    assert lib.fa_fwd(ctypes.byref(a), None) == 1
    assert lib.fa_fwd(None, None) == 1
    a = _args(sq=0)
    assert lib.fa_fwd(ctypes.byref(a), None) == 0  # nothing to do
    assert lib.fa_splitkv_workspace_size(None, 1) == 0
    a = _args(skv=1024)  # 8 key blocks
    ws = lib.fa_splitkv_workspace_size(ctypes.byref(a), 3)
    rows = 3 * 1 * 2 * 128
    assert ws >= rows * 128 * 4 + rows * 4
    # a request above the key blocks there are is sized as the split count the call will
    # use (capped at the blocks): 128 keys are one block, so 3 splits size as 1
    a = _args()
    assert lib.fa_splitkv_workspace_size(ctypes.byref(a), 3) == lib.fa_splitkv_workspace_size(ctypes.byref(a), 1)
    assert lib.fa_fwd_splitkv(ctypes.byref(a), -1, None, 0, None, None) == 1


def test_combine_validation(lib):
    st = (ctypes.c_int64 * 3)(1, 1, 1)
    assert lib.fa_splitkv_combine(None, None, 0, 1, 1, 1, 64, 0, None, st, None, None) == 1
    assert lib.fa_splitkv_combine(None, None, 1, 1, 1, 1, 80, 0, None, st, None, None) == 2
    assert lib.fa_splitkv_combine(None, None, 1, 1, 1, 0, 64, 0, None, st, None, None) == 0


def _kv_args(**kw):
    from tiled_exact_attention_gb300._lib import KvcacheArgs

    a = KvcacheArgs()
    a.dtype, a.b, a.hq, a.hkv, a.d = 0, 2, 8, 2, 128
    a.q = a.k = a.v = a.o = 4096
    a.lse = 4096
    a.q_strides = (ctypes.c_int64 * 2)(8 * 128, 128)
    a.o_strides = (ctypes.c_int64 * 2)(8 * 128, 128)
    a.k_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 128)
    a.v_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 128)
    a.num_pages, a.page_size = 16, 256
    a.block_table = a.seqlens_k = 4096
    a.block_table_stride = 8
    a.max_seqlen_k = 1000
    a.scale = 0.1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,expect", [
    ("page_size", 100, 2), ("page_size", -1, 1), ("block_table", 0, 1), ("seqlens_k", 0, 1), ("d", 80, 2),
    ("hq", 7, 1), ("num_pages", 0, 1), ("max_seqlen_k", -5, 1), ("k", 4100, 1), ("scale", 0.0, 1),
    ("softcap", -2.0, 1), ("softcap", float("nan"), 1),
])
def test_kvcache_validation(lib, field, value, expect):
    a = _kv_args(**{field: value})
    assert lib.fa_fwd_kvcache(ctypes.byref(a), 0, None, 0, None, None) == expect
    assert lib.fa_kvcache_workspace_size(ctypes.byref(a), 2) == 0


def test_kvcache_packed_needs_prefix_sums(lib):
    a = _kv_args(page_size=0, cu_seqlens_k=0)
    assert lib.fa_fwd_kvcache(ctypes.byref(a), 1, None, 0, None, None) == 1
    a = _kv_args(page_size=0, cu_seqlens_k=4096)
    assert lib.fa_kvcache_workspace_size(ctypes.byref(a), 3) >= 3 * 2 * 8 * (128 + 1) * 4


def _varlen_args(**kw):
    from tiled_exact_attention_gb300._lib import VarlenArgs

    a = VarlenArgs()
    a.dtype, a.b, a.hq, a.hkv, a.d = 0, 2, 4, 2, 128
    a.total_q, a.total_k, a.max_seqlen_q = 300, 400, 200
    a.q = a.k = a.v = a.o = 4096
    a.lse = a.cu_seqlens_q = a.cu_seqlens_k = 4096
    a.q_strides = (ctypes.c_int64 * 2)(4 * 128, 128)
    a.o_strides = (ctypes.c_int64 * 2)(4 * 128, 128)
    a.k_strides = (ctypes.c_int64 * 2)(2 * 128, 128)
    a.v_strides = (ctypes.c_int64 * 2)(2 * 128, 128)
    a.scale = 0.1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,expect", [
    ("dtype", 3, 1), ("b", 0, 1), ("hq", 3, 1), ("d", 96, 2), ("total_q", -1, 1), ("max_seqlen_q", -1, 1),
    ("causal", 2, 1), ("local", 2, 1), ("scale", 0.0, 1), ("q", 0, 1), ("cu_seqlens_q", 0, 1),
    ("cu_seqlens_k", 4098, 1), ("k", 4100, 1), ("lse", 0, 1), ("total_k", (1 << 30) + 1, 2),
    ("softcap", -0.5, 1), ("softcap", float("inf"), 1),
])
def test_varlen_validation(lib, field, value, expect):
    a = _varlen_args(**{field: value})
    assert lib.fa_fwd_varlen(ctypes.byref(a), None) == expect


def test_varlen_validation_strides_and_empty(lib):
    a = _varlen_args()
    a.q_strides = (ctypes.c_int64 * 2)(4 * 128, 100)
    assert lib.fa_fwd_varlen(ctypes.byref(a), None) == 1
    a = _varlen_args(local=1, window_left=-3, window_right=0)
    assert lib.fa_fwd_varlen(ctypes.byref(a), None) == 1
    assert lib.fa_fwd_varlen(None, None) == 1
    # nothing to compute: no launch, no device needed
    assert lib.fa_fwd_varlen(ctypes.byref(_varlen_args(total_q=0)), None) == 0
    assert lib.fa_fwd_varlen(ctypes.byref(_varlen_args(max_seqlen_q=0)), None) == 0
    assert lib.fa_status_string(6) == b"an argument read on the device (sequence offsets) failed its check"


def _bwd_args(**kw):
    from tiled_exact_attention_gb300._lib import BwdArgs

    a = BwdArgs()
    a.dtype, a.b, a.sq, a.skv, a.hq, a.hkv, a.d = 0, 1, 128, 128, 2, 2, 128
    for f in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"):
        setattr(a, f, 4096)
    for f in ("q_strides", "k_strides", "v_strides", "o_strides", "do_strides", "dq_strides", "dk_strides",
              "dv_strides"):
        setattr(a, f, (ctypes.c_int64 * 3)(128 * 2 * 128, 2 * 128, 128))
    a.scale = 0.125
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,expect", [
    ("d", 256, 2), ("d", 96, 2), ("dout", 0, 1), ("dq", 4100, 1), ("dk", 0, 1), ("lse", 0, 1), ("hq", 3, 1),
    ("causal", 5, 1), ("scale", -1.0, 1), ("softcap", -3.0, 1), ("softcap", float("nan"), 1),
])
def test_bwd_validation(lib, field, value, expect):
    a = _bwd_args(**{field: value})
    assert lib.fa_bwd(ctypes.byref(a), None, 0, None) == expect
    assert lib.fa_bwd_workspace_size(ctypes.byref(a)) == 0


def test_bwd_workspace_size(lib):
    a = _bwd_args(sq=300)
    rows = 1 * 2 * 384  # padded to 128 rows
    assert lib.fa_bwd_workspace_size(ctypes.byref(a)) == 2 * ((rows * 4 + 255) // 256 * 256)
    bad = _bwd_args(dv_strides=(ctypes.c_int64 * 3)(100, 10, 1))
    assert lib.fa_bwd(ctypes.byref(bad), None, 0, None) == 1


def test_e4m3_validation(lib):
    from tiled_exact_attention_gb300._lib import E4m3Args, QuantArgs

    qa = QuantArgs()
    qa.dtype, qa.b, qa.s, qa.h, qa.d = 0, 1, 256, 2, 128
    qa.x = qa.out = qa.descale = 4096
    qa.x_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 128)
    qa.out_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 128)
    for field, value, expect in (("d", 512, 2), ("d", 96, 2), ("transpose", 2, 1), ("x", 0, 1), ("out", 4104, 1)):
        old = getattr(qa, field)
        setattr(qa, field, value)
        assert lib.fa_quantize_e4m3(ctypes.byref(qa), None) == expect, field
        setattr(qa, field, old)
    qa.out_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 8)  # not a multiple of 16 bytes
    assert lib.fa_quantize_e4m3(ctypes.byref(qa), None) == 1
    a = E4m3Args()
    a.b, a.sq, a.skv, a.hq, a.hkv, a.d = 1, 128, 128, 2, 2, 128
    for f in ("q", "k", "vt", "q_descale", "k_descale", "v_descale", "o", "lse"):
        setattr(a, f, 4096)
    for f in ("q_strides", "k_strides", "vt_strides"):
        setattr(a, f, (ctypes.c_int64 * 3)(128 * 2 * 128, 2 * 128, 128))
    a.o_strides = (ctypes.c_int64 * 3)(128 * 2 * 128, 2 * 128, 128)
    a.scale = 0.1
    for field, value, expect in (("d", 96, 2), ("d", 512, 2), ("vt", 0, 1), ("v_descale", 0, 1), ("causal", 3, 1),
                                 ("scale", 0.0, 1), ("hq", 3, 1)):
        old = getattr(a, field)
        setattr(a, field, value)
        assert lib.fa_fwd_e4m3(ctypes.byref(a), None) == expect, field
        setattr(a, field, old)


def test_splitkv_e4m3_validation(lib):
    from tiled_exact_attention_gb300._lib import SplitkvE4m3Args

    def args(**kw):
        a = SplitkvE4m3Args()
        a.dtype, a.b, a.skv, a.hq, a.hkv, a.d = 0, 2, 256, 8, 2, 128
        for f in ("q", "k", "v", "k_descale", "v_descale", "o", "lse"):
            setattr(a, f, 4096)
        a.q_strides = (ctypes.c_int64 * 2)(8 * 128, 128)
        a.o_strides = (ctypes.c_int64 * 2)(8 * 128, 128)
        a.k_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 128)
        a.v_strides = (ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 128)
        a.scale = 0.1
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    for field, value, expect in (("d", 96, 2), ("d", 256, 2), ("hq", 3, 1), ("q", 0, 1), ("k", 0, 1),
                                 ("k_descale", 0, 1), ("scale", 0.0, 1), ("dtype", 5, 1), ("lse", 4098, 1)):
        a = args(**{field: value})
        assert lib.fa_fwd_splitkv_e4m3(ctypes.byref(a), 0, None, 0, None, None) == expect, field
        assert lib.fa_splitkv_e4m3_workspace_size(ctypes.byref(a), 2) == 0, field
    a = args(k_strides=(ctypes.c_int64 * 3)(256 * 2 * 128, 2 * 128, 8))  # not a multiple of 16 bytes
    assert lib.fa_fwd_splitkv_e4m3(ctypes.byref(a), 0, None, 0, None, None) == 1
    a = args()
    # an explicit split count is sized without a device: two 128-key blocks cap 5 splits at 2
    assert lib.fa_splitkv_e4m3_workspace_size(ctypes.byref(a), 5) == lib.fa_splitkv_e4m3_workspace_size(
        ctypes.byref(a), 2) > 0
    assert lib.fa_fwd_splitkv_e4m3(ctypes.byref(a), 2, None, 0, None, None) in (1, 3)  # no workspace / no device
