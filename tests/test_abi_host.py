"""Host-side checks of the C-ABI library that need no GPU: it builds, loads, exports
every function include/fa.h declares, its parameter structs match the binding's
layout, and it rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    fa_build.build()
    return fa.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function(L):
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_decode_paged" in names
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(L, n)


def test_struct_layouts_match_header(tmp_path):
    src = tmp_path / "layout.c"
    fields = {"fa_fwd_params": [f for f, _ in fa.FwdParams._fields_],
              "fa_decode_params": [f for f, _ in fa.DecodeParams._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "fa.h"', "int main(void){"]
    for st, fs in fields.items():
        lines.append(f'printf("{st} %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines.append("return 0;}")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                 check=True).stdout.splitlines())
    for st, cls in (("fa_fwd_params", fa.FwdParams), ("fa_decode_params", fa.DecodeParams)):
        assert int(got[st]) == ctypes.sizeof(cls)
        for f, _ in cls._fields_:
            assert int(got[f"{st}.{f}"]) == getattr(cls, f).offset, (st, f)


def test_version_and_block_m(L):
    assert L.fa_version() >= 100
    assert L.fa_fwd_block_m() == 128
    assert [L.fa_fwd_default_block_m(m) for m in range(6)] == [256, 256, 256, 128, 256, 128]
    assert L.fa_fwd_default_block_m(6) == 0 and L.fa_fwd_default_block_m(-1) == 0


def test_workspace_size_and_split_rule(L):
    assert L.fa_decode_workspace_size(32, 32, 128, 32, 256) == 32 * 32 * 32 * 130 * 4
    assert L.fa_decode_workspace_size(0, 32, 128, 32, 256) == 0
    for B, H, mp in [(32, 32, 32), (1, 1, 1), (4, 8, 100), (64, 64, 64)]:
        pps = L.fa_decode_default_pages_per_split(B, H, mp)
        assert 1 <= pps <= max(1, mp)


A = 0x10000  # a 16-byte aligned fake device address: validation never dereferences it


def _fwd(L, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=None, B=1, H=1, Sq=4, Sk=4, d=64, scale=0.125,
                mask_mode=0, window=0, n_global=0, dtype=0)
    args.update(kw)
    return L.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                    args["H"], args["Sq"], args["Sk"], args["d"], args["scale"],
                    args["mask_mode"], args["window"], args["n_global"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=A + 8), fa.FA_ERR_INVALID_ARG),
    (dict(lse=A + 2), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sq=-1), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), fa.FA_ERR_INVALID_ARG),  # FP32: fa_fwd_ex with a workspace only
    (dict(dtype=3), fa.FA_ERR_UNSUPPORTED),
    (dict(mask_mode=5), fa.FA_ERR_INVALID_ARG),  # block-sparse without a layout
    (dict(mask_mode=6), fa.FA_ERR_INVALID_ARG),
    (dict(mask_mode=-1), fa.FA_ERR_INVALID_ARG),
    (dict(mask_mode=3, window=-1), fa.FA_ERR_INVALID_ARG),
    (dict(mask_mode=4, n_global=-1), fa.FA_ERR_INVALID_ARG),
    (dict(mask_mode=2, window=0), fa.FA_ERR_INVALID_ARG),
    (dict(mask_mode=2, window=4, n_global=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 20, H=1 << 20), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_rejects_bad_arguments(L, kw, code):
    assert _fwd(L, **kw) == code
    assert fa.fa_last_error_string() != ""


def test_fwd_empty_query_is_a_no_op(L):
    assert _fwd(L, Sq=0) == fa.FA_OK


def test_fwd_ex_rejects_bad_plan(L):
    p = fa.FwdParams(A, A, A, A, None, 1, 1, 4, 4, 64, 0.125, 0, 0, 0, 0, 96, 0, 0, 0, 0, None)
    assert L.fa_fwd_ex(ctypes.byref(p), None) == fa.FA_ERR_UNSUPPORTED
    for bm in (32, 96, 512):  # block_m: 64, 128 or 256
        p = fa.FwdParams(A, A, A, A, None, 1, 1, 4, 4, 64, 0.125, 0, 0, 0, 0, 0, bm, 0, 0, 0,
                         None)
        assert L.fa_fwd_ex(ctypes.byref(p), None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_fwd_ex(None, None) == fa.FA_ERR_INVALID_ARG


def test_fwd_workspace_size(L):
    # FP32: a bf16 high and low plane of every Q, K, V element; nothing for 16-bit inputs
    assert L.fa_fwd_workspace_size(4, 32, 4096, 4096, 128, fa.FA_F32) == 4 * 128 * 4 * 32 * 3 * 4096
    assert L.fa_fwd_workspace_size(1, 2, 100, 7, 64, fa.FA_F32) == 4 * 64 * 2 * (100 + 14)
    assert L.fa_fwd_workspace_size(1, 2, 100, 7, 64, fa.FA_BF16) == 0
    assert L.fa_fwd_workspace_size(0, 2, 100, 7, 64, fa.FA_F32) == 0
    assert fa.fa_fwd_workspace_size(1, 1, 0, 0, 64, fa.FA_F32) == 0


def _fwd32(L, ws=A, wsb=None, block_n=0, block_m=0, Sq=4, Sk=4):
    need = L.fa_fwd_workspace_size(1, 1, Sq, Sk, 64, fa.FA_F32)
    p = fa.FwdParams(A, A, A, A, None, 1, 1, Sq, Sk, 64, 0.125, 0, 0, 0, fa.FA_F32, block_n,
                     block_m, 0, 0, 0, None, None, ws, need if wsb is None else wsb)
    return L.fa_fwd_ex(ctypes.byref(p), None)


def test_fwd_f32_argument_checks(L):
    assert _fwd32(L, ws=None) == fa.FA_ERR_INVALID_ARG
    assert _fwd32(L, ws=A + 8) == fa.FA_ERR_INVALID_ARG
    assert _fwd32(L, wsb=16) == fa.FA_ERR_INVALID_ARG
    assert "needs" in fa.fa_last_error_string()
    assert _fwd32(L, block_n=128) == fa.FA_ERR_UNSUPPORTED
    assert _fwd32(L, block_m=128) == fa.FA_ERR_UNSUPPORTED
    assert _fwd32(L, ws=None, Sq=0) == fa.FA_OK  # nothing to compute, nothing needed
    # the split planes double B * H in the tensor maps: B * H is capped at 2^29
    p = fa.FwdParams(A, A, A, A, None, 1 << 15, 1 << 15, 4, 4, 64, 0.125, 0, 0, 0, fa.FA_F32, 0,
                     0, 0, 0, 0, None, None, A, 1 << 40)
    assert L.fa_fwd_ex(ctypes.byref(p), None) == fa.FA_ERR_INVALID_ARG
    # the paged prefill and the backward take 16-bit inputs only
    assert L.fa_fwd_paged(A, A, A, A, A, A, None, 1, 1, 4, 64, 256, 1, 1, 0.125, 0, 0, 0,
                          fa.FA_F32, None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_bwd(A, A, A, A, A, A, A, A, A, A, 1 << 20, 1, 1, 4, 4, 64, 0.125, 0, 0, 0,
                    fa.FA_F32, None) == fa.FA_ERR_UNSUPPORTED


def _dec(L, **kw):
    args = dict(q=A, kp=A, vp=A, bt=A, cl=A, o=A, lse=None, B=2, H=2, d=128, page=256, mp=4,
                np_=8, scale=0.1, dtype=0, ws=A, wsb=1 << 20)
    args.update(kw)
    return L.fa_decode_paged(args["q"], args["kp"], args["vp"], args["bt"], args["cl"], args["o"],
                             args["lse"], args["B"], args["H"], args["d"], args["page"],
                             args["mp"], args["np_"], args["scale"], args["dtype"], args["ws"],
                             args["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(bt=None), fa.FA_ERR_INVALID_ARG),
    (dict(ws=None), fa.FA_ERR_INVALID_ARG),
    (dict(q=A + 4), fa.FA_ERR_INVALID_ARG),
    (dict(bt=A + 2), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(np_=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=80), fa.FA_ERR_UNSUPPORTED),
    (dict(page=100), fa.FA_ERR_UNSUPPORTED),
    (dict(page=8), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=5), fa.FA_ERR_UNSUPPORTED),
    (dict(wsb=16), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments(L, kw, code):
    assert _dec(L, **kw) == code


def test_decode_ex_rejects_bad_split(L):
    p = fa.DecodeParams(A, A, A, A, A, A, None, 2, 2, 128, 256, 4, 8, 0.1, 0, A, 1 << 20, 5,
                        None, None)
    assert L.fa_decode_paged_ex(ctypes.byref(p), None) == fa.FA_ERR_INVALID_ARG


def test_selftest_rejects_bad_limit(L):
    assert L.fa_selftest_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_selftest_timeout(2_000_000, None) == fa.FA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(fa.FaError):
        fa.lib()


def test_merge_rejects_bad_arguments(L):
    assert L.fa_merge_partials(A, A, A, A, A, None, 10, 96, 0, None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_merge_partials(A, A, A, A, A, None, 10, 64, 7, None) == fa.FA_ERR_UNSUPPORTED
    assert L.fa_merge_partials(None, A, A, A, A, None, 10, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_merge_partials(A + 8, A, A, A, A, None, 10, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_merge_partials(A, A, A, A, A, None, -1, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_merge_partials(None, None, None, None, None, None, 0, 64, 0, None) == fa.FA_OK



def test_bwd_rejects_bad_arguments(L):
    A = 1 << 20  # a 16-byte-aligned fake address; nothing is launched
    base = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, ws=A, wsb=1 << 20, B=1,
                H=2, Sq=64, Sk=64, d=64, scale=0.125, mode=0, w=0, g=0, dtype=0)

    def call(**kw):
        a = dict(base, **kw)
        return L.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"],
                        a["dv"], a["ws"], a["wsb"], a["B"], a["H"], a["Sq"], a["Sk"], a["d"],
                        a["scale"], a["mode"], a["w"], a["g"], a["dtype"], None)
    assert call(mode=5) == fa.FA_ERR_UNSUPPORTED
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(ws=None) == fa.FA_ERR_INVALID_ARG
    assert call(wsb=16) == fa.FA_ERR_INVALID_ARG
    assert call(dout=None) == fa.FA_ERR_INVALID_ARG
    assert call(dk=A + 8) == fa.FA_ERR_INVALID_ARG
    assert call(mode=2, w=0) == fa.FA_ERR_INVALID_ARG
    assert L.fa_bwd_workspace_size(2, 3, 100) == 2 * 3 * (100 * 128 + 100) * 4  # dq accumulator at d = 128, D
    assert L.fa_bwd_workspace_size(1, 1, 5) == (8 * 128 + 5) * 4  # Sq rounded up to 4 for the accumulator


def test_paged_fwd_rejects_bad_arguments(L):
    A = 1 << 20  # a 16-byte-aligned fake address; nothing is launched
    base = dict(q=A, kp=A, vp=A, tab=A, ctx=A, host=A, o=A, lse=A, B=2, H=2, Sq=64, d=64,
                page=256, mp=4, npages=16, scale=0.125, mode=1, w=0, g=0, dtype=0)

    def calls(**kw):
        a = dict(base, **kw)
        r1 = L.fa_fwd_paged(a["q"], a["kp"], a["vp"], a["tab"], a["ctx"], a["o"], a["lse"], a["B"],
                            a["H"], a["Sq"], a["d"], a["page"], a["mp"], a["npages"], a["scale"],
                            a["mode"], a["w"], a["g"], a["dtype"], None)
        r2 = L.fa_fwd_paged_host_lens(a["q"], a["kp"], a["vp"], a["tab"], a["ctx"], a["host"],
                                      a["o"], a["lse"], a["B"], a["H"], a["Sq"], a["d"], a["page"],
                                      a["mp"], a["npages"], a["scale"], a["mode"], a["w"], a["g"],
                                      a["dtype"], None)
        assert r1 == r2, kw
        return r1
    assert calls(kp=None) == fa.FA_ERR_INVALID_ARG
    assert calls(tab=None) == fa.FA_ERR_INVALID_ARG
    assert calls(vp=A + 8) == fa.FA_ERR_INVALID_ARG      # pools 16-byte aligned
    assert calls(ctx=A + 2) == fa.FA_ERR_INVALID_ARG     # lengths 4-byte aligned
    assert calls(mp=0) == fa.FA_ERR_INVALID_ARG
    assert calls(page=96) == fa.FA_ERR_UNSUPPORTED       # pages of a multiple of 64 tokens
    assert calls(page=32) == fa.FA_ERR_UNSUPPORTED
    assert calls(page=4096, mp=1 << 20) == fa.FA_ERR_INVALID_ARG  # capacity past 2^30
    assert calls(d=96) == fa.FA_ERR_UNSUPPORTED
    assert calls(dtype=2) == fa.FA_ERR_UNSUPPORTED       # FP32 inputs are not paged
    assert calls(mode=2, w=0) == fa.FA_ERR_INVALID_ARG   # a window needs window >= 1


def test_bwd_block_sparse_rejects_bad_arguments(L):
    A = 1 << 20
    base = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, ws=A, wsb=1 << 20, B=1,
                H=2, Sq=64, Sk=64, d=64, scale=0.125, lay=A, dtype=0)

    def call(**kw):
        a = dict(base, **kw)
        return L.fa_bwd_block_sparse(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"],
                                     a["dk"], a["dv"], a["ws"], a["wsb"], a["B"], a["H"], a["Sq"],
                                     a["Sk"], a["d"], a["scale"], a["lay"], a["dtype"], None)
    assert call(lay=None) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(ws=None) == fa.FA_ERR_INVALID_ARG
    assert call(wsb=16) == fa.FA_ERR_INVALID_ARG
    assert call(dq=A + 8) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=2) == fa.FA_ERR_UNSUPPORTED


def test_kv_append_rejects_bad_arguments(L):
    A = 1 << 20
    base = dict(kn=A, vn=A, kp=A, vp=A, tab=A, ctx=A, nl=None, B=2, H=2, T=64, d=64, page=256,
                mp=4, npages=16, dtype=0)

    def call(**kw):
        a = dict(base, **kw)
        return L.fa_kv_append(a["kn"], a["vn"], a["kp"], a["vp"], a["tab"], a["ctx"], a["nl"],
                              a["B"], a["H"], a["T"], a["d"], a["page"], a["mp"], a["npages"],
                              a["dtype"], None)
    assert call(T=0) == fa.FA_OK                        # nothing to append: nothing launched
    assert call(B=0) == fa.FA_ERR_INVALID_ARG
    assert call(T=-1) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(dtype=2) == fa.FA_ERR_UNSUPPORTED
    assert call(page=24) == fa.FA_ERR_UNSUPPORTED       # a multiple of 16 tokens
    assert call(kp=None) == fa.FA_ERR_INVALID_ARG
    assert call(vn=A + 8) == fa.FA_ERR_INVALID_ARG
    assert call(nl=A + 2) == fa.FA_ERR_INVALID_ARG      # new_lens 4-byte aligned
    assert call(page=4096, mp=1 << 20) == fa.FA_ERR_INVALID_ARG
