"""Host-side checks of the C-ABI library (no GPU, no compute calls).

* libfa.so builds for sm_103a here (nvcc cross-compiles) and loads;
* it exports every function include/fa.h declares, and nothing in the
  binding refers to a symbol the header does not declare;
* argument validation returns the documented codes before touching CUDA;
* the product package never imports the oracle.
"""
import ctypes
import os
import re
import subprocess

import pytest

import exact_attention_forward_fa_gb300 as fa
from exact_attention_forward_fa_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert _header_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\S+)", out))
    for name in _header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert fa.fa_version() == 100
    names = [fa.status_string(c) for c in range(7)]
    assert names == ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED",
                     "FA_ERR_MISALIGNED", "FA_ERR_TOO_LARGE", "FA_ERR_CUDA",
                     "FA_ERR_TIMEOUT"]
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"
    assert fa.fa_status_detail() == [0, 0, 0, 0]


A = 0x10000          # fake, 16-byte aligned device addresses (never dereferenced)


def _call(lib, q=A, k=A, v=A, o=A, lse=None, B=1, H=1, N=128, d=64, alpha=0.125,
          causal=0, dtype=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, alpha, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=None), fa.FA_ERR_INVALID_ARG),
    (dict(v=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(alpha=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(alpha=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(B=1 << 20, H=1 << 10, N=1 << 20, d=128), fa.FA_ERR_TOO_LARGE),
])
def test_validation_codes(lib, kw, code):
    assert _call(lib, **kw) == code


@pytest.mark.parametrize("H,H_kv,code", [(6, 4, fa.FA_ERR_INVALID_ARG), (4, 0, fa.FA_ERR_INVALID_ARG),
                                         (4, 8, fa.FA_ERR_INVALID_ARG)])
def test_gqa_validation_codes(lib, H, H_kv, code):
    assert lib.fa_fwd_gqa(A, A, A, A, None, 1, H, H_kv, 128, 64, 0.125, 0, 0, None) == code


@pytest.mark.parametrize("H,H_kv,d,code", [(6, 4, 64, fa.FA_ERR_INVALID_ARG),   # H_kv must divide H
                                           (6, 2, 64, fa.FA_ERR_UNSUPPORTED),   # group 3 does not divide 128
                                           (8, 1, 256, fa.FA_ERR_UNSUPPORTED),  # d = 256
                                           (8, 2, 96, fa.FA_ERR_UNSUPPORTED)])
def test_gqa_packed_validation_codes(lib, H, H_kv, d, code):
    assert lib.fa_fwd_gqa_packed(A, A, A, A, None, 1, H, H_kv, 128, d, 0.125, 0, 0, None) == code


def _xcall(lib, q=A, k=A, v=A, o=A, lse=None, B=1, H=2, H_kv=1, N=128, d=128, alpha=0.088,
           wl=-1, wr=0, softcap=0.0, sinks=None, dtype=0):
    return lib.fa_fwd_ext(q, k, v, o, lse, B, H, H_kv, N, d, alpha, wl, wr, softcap, sinks,
                          dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(H=3, H_kv=2), fa.FA_ERR_INVALID_ARG),
    (dict(wl=-2), fa.FA_ERR_INVALID_ARG),
    (dict(wr=-5), fa.FA_ERR_INVALID_ARG),
    (dict(softcap=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(softcap=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(softcap=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(softcap=1e-38, alpha=1e3), fa.FA_ERR_INVALID_ARG),   # alpha / c overflows
    (dict(alpha=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=2), fa.FA_ERR_INVALID_ARG),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(v=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(sinks=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 1), fa.FA_ERR_MISALIGNED),
])
def test_ext_validation_codes(lib, kw, code):
    assert _xcall(lib, **kw) == code


def _scall(lib, q=A, k=A, v=A, o=A, lse=None, B=1, H=1, N=128, d=128, alpha=0.088, causal=0,
           dtype=0, S=2, ws=A):
    return lib.fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, alpha, causal, dtype, S, ws, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ws=None), fa.FA_ERR_INVALID_ARG),
    (dict(S=0), fa.FA_ERR_INVALID_ARG),
    (dict(S=17), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(ws=A + 4), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_splitkv_validation_codes(lib, kw, code):
    assert _scall(lib, **kw) == code


def test_splitkv_workspace_size(lib):
    assert fa.fa_splitkv_workspace_floats(2, 3, 100, 64, 4) == 4 * (2 * 100 * 3 * 64 + 2 * 3 * 100)
    assert fa.fa_splitkv_workspace_floats(1, 1, 1, 64, 0) == -1
    assert 1 <= fa.fa_splitkv_auto(1, 1, 128, 128) <= 16


def _qcall(lib, x=A, x8=A, sc=A, signs=None, B=1, H=1, N=128, d=128):
    return lib.fa_quantize_fp8(x, x8, sc, signs, B, H, N, d, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), fa.FA_ERR_INVALID_ARG),
    (dict(x8=None), fa.FA_ERR_INVALID_ARG),
    (dict(sc=None), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(x=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(sc=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(signs=A + 1), fa.FA_ERR_MISALIGNED),
])
def test_quantize_validation_codes(lib, kw, code):
    assert _qcall(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(sc=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(g=-1), fa.FA_ERR_INVALID_ARG),
    (dict(g=3), fa.FA_ERR_INVALID_ARG),
])
def test_quantize_granular_validation_codes(lib, kw, code):
    g = kw.pop("g", fa.FA_SCALE_TENSOR)
    args = dict(x=A, x8=A, sc=A, signs=None, B=1, H=1, N=128, d=128)
    args.update(kw)
    assert lib.fa_quantize_fp8_granular(args["x"], args["x8"], args["sc"], args["signs"],
                                        args["B"], args["H"], args["N"], args["d"], g,
                                        None) == code


def _f8call(lib, q=A, k=A, v=A, qs=A, ks=A, vs=A, o=A, lse=None, B=1, H=1, N=128, d=128,
            alpha=0.088, causal=0):
    return lib.fa_fwd_fp8(q, k, v, qs, ks, vs, o, lse, B, H, N, d, alpha, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(vs=None), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(alpha=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(d=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(k=A + 4), fa.FA_ERR_MISALIGNED),
    (dict(qs=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_fp8_validation_codes(lib, kw, code):
    assert _f8call(lib, **kw) == code


def _bcall(lib, q=A, k=A, v=A, o=A, do=A, lse=A, ws=A, dq=A, dk=A, dv=A, B=1, H=1,
           N=128, d=128, alpha=0.088, causal=0, dtype=0):
    return lib.fa_bwd(q, k, v, o, do, lse, ws, dq, dk, dv, B, H, N, d, alpha, causal,
                      dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(do=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(ws=None), fa.FA_ERR_INVALID_ARG),
    (dict(dv=None), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(alpha=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=3), fa.FA_ERR_INVALID_ARG),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(o=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(dk=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(ws=A + 4), fa.FA_ERR_MISALIGNED),
    (dict(B=1 << 20, H=1 << 10, N=1 << 20, d=128), fa.FA_ERR_TOO_LARGE),
])
def test_bwd_validation_codes(lib, kw, code):
    assert _bcall(lib, **kw) == code


def _bxcall(lib, q=A, o=A, lse=A, ws=A, dq=A, B=1, H=2, H_kv=1, N=128, d=128, wl=64, wr=0,
            softcap=0.0, alpha=0.088, sinks=None, dsinks=None, dtype=0):
    return lib.fa_bwd_ext(q, A, A, o, A, lse, ws, dq, A, A, B, H, H_kv, N, d, alpha, wl, wr,
                          softcap, sinks, dsinks, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(ws=None), fa.FA_ERR_INVALID_ARG),
    (dict(wl=-2), fa.FA_ERR_INVALID_ARG),
    (dict(wr=-3), fa.FA_ERR_INVALID_ARG),
    (dict(dsinks=A), fa.FA_ERR_INVALID_ARG),            # a sink gradient needs the sinks
    (dict(softcap=-2.0), fa.FA_ERR_INVALID_ARG),
    (dict(H=3, H_kv=2), fa.FA_ERR_INVALID_ARG),
    (dict(H_kv=0), fa.FA_ERR_INVALID_ARG),
    (dict(softcap=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(softcap=1e-38, alpha=1e3), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=5), fa.FA_ERR_INVALID_ARG),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(sinks=A + 2, dsinks=A), fa.FA_ERR_MISALIGNED),
    (dict(sinks=A, dsinks=A + 1), fa.FA_ERR_MISALIGNED),
    (dict(dq=A + 8), fa.FA_ERR_MISALIGNED),
])
def test_bwd_ext_validation_codes(lib, kw, code):
    assert _bxcall(lib, **kw) == code


def test_bwd_noalloc_rejects_problems_beyond_its_workspace(lib):
    # 2 * B * H * ceil(N/128) * 128 floats must fit the 4 Mi-float array;
    # the check comes before any CUDA call, after the arguments fa_bwd
    # itself rejects (which keep fa_bwd's codes).
    args = [A] * 9
    assert lib.fa_bwd_noalloc(*args, 1, 16, 131073, 128, 0.088, 0, 0, None) == fa.FA_ERR_TOO_LARGE
    assert lib.fa_bwd_noalloc(*args, 0, 1, 128, 128, 0.088, 0, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_noalloc(*args, 1, 16, 131073, 256, 0.088, 0, 0, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_noalloc(*args, 1, 16, 131073, 128, 0.088, 2, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_noalloc(*args, 1, 16, 131073, 128, 0.088, 0, 7, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_noalloc(None, *args[1:], 1, 16, 131073, 128, 0.088, 0, 0,
                              None) == fa.FA_ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    assert _call(lib) in (fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "exact_attention_forward_fa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fa_oracle" not in text and "liboracle" not in text, f


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    mod = importlib.import_module("exact_attention_forward_fa_gb300")
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        mod.load()


def test_selftest_validation_codes(lib):
    assert lib.fa_selftest_wait_timeout(None, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(A + 2, None) == fa.FA_ERR_MISALIGNED
