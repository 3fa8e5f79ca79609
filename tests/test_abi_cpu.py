"""C-ABI checks that need no GPU: the library builds and loads, exports every
function the header declares, and rejects bad arguments on the host before
touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import varlen_flashattention_forward_gb300 as fa
from varlen_flashattention_forward_gb300 import build_ext

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(REPO, "include", "fa_gb300.h")


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:fa_status|const char\*)\s+(fa_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build_ext.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for s in range(6):
        assert lib.fa_status_string(s)
    assert lib.fa_status_string(2).decode() == "unsupported configuration"


P = ctypes.c_void_p


def varlen(lib, **kw):
    a = dict(q=P(0x1000), k=P(0x2000), v=P(0x3000), cq=P(0x4000), ck=P(0x5000), batch=2,
             total_q=10, total_k=10, H=4, Hk=4, dqk=64, dv=64, mq=5, mk=5, scale=0.125,
             causal=0, wl=-1, wr=-1, out=P(0x6000), lse=None, stream=None)
    a.update(kw)
    return lib.fa_varlen_fwd(a["q"], a["k"], a["v"], a["cq"], a["ck"], a["batch"], a["total_q"],
                             a["total_k"], a["H"], a["Hk"], a["dqk"], a["dv"], a["mq"], a["mk"],
                             a["scale"], a["causal"], a["wl"], a["wr"], a["out"], a["lse"],
                             a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(out=None), fa.FA_ERR_INVALID_ARG),
    (dict(cq=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=None), fa.FA_ERR_INVALID_ARG),
    (dict(batch=0), fa.FA_ERR_INVALID_ARG),
    (dict(total_q=-1), fa.FA_ERR_INVALID_ARG),
    (dict(H=6, Hk=4), fa.FA_ERR_INVALID_ARG),
    (dict(Hk=0), fa.FA_ERR_INVALID_ARG),
    (dict(wl=-2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(q=P(0x1008)), fa.FA_ERR_INVALID_ARG),
    (dict(lse=P(0x6002)), fa.FA_ERR_INVALID_ARG),
    (dict(dqk=100, dv=100), fa.FA_ERR_UNSUPPORTED),
    (dict(dqk=192, dv=192), fa.FA_ERR_UNSUPPORTED),
])
def test_varlen_host_validation(lib, kw, expect):
    assert varlen(lib, **kw) == expect


def varlen_strided(lib, **kw):
    # V as the upper 64 columns of a combined [tokens, 4 heads, 128] buffer.
    a = dict(q=P(0x1000), qr=4 * 64, qh=64, k=P(0x2000), kr=4 * 64, kh=64, v=P(0x3000),
             vr=4 * 128, vh=128, cq=P(0x4000), ck=P(0x5000), batch=2, total_q=10, total_k=10,
             H=4, Hk=4, dqk=64, dv=64, scale=0.125, causal=0, wl=-1, wr=-1, out=P(0x6000),
             lse=None)
    a.update(kw)
    return lib.fa_varlen_fwd_strided(a["q"], a["qr"], a["qh"], a["k"], a["kr"], a["kh"], a["v"],
                                     a["vr"], a["vh"], a["cq"], a["ck"], a["batch"],
                                     a["total_q"], a["total_k"], a["H"], a["Hk"], a["dqk"],
                                     a["dv"], 0, 0, a["scale"], a["causal"], a["wl"], a["wr"],
                                     a["out"], a["lse"], None)


@pytest.mark.parametrize("kw", [
    dict(vh=60),                # head stride below the head dim
    dict(vh=132),               # not a multiple of 8 elements (16 bytes)
    dict(vr=3 * 128 + 63),      # rows overlap the last head
    dict(kr=0),                 # zero stride
    dict(qh=-64),               # negative stride
    dict(qr=3 * 64 + 56),       # q rows overlap
    dict(v=P(0x3008)),          # base not 16-byte aligned
])
def test_varlen_strided_host_validation(lib, kw):
    assert varlen_strided(lib, **kw) == fa.FA_ERR_INVALID_ARG


def test_varlen_strided_valid_views_pass_validation(lib):
    """Valid strided views get past the host checks (then fail only for want
    of a GPU, or launch when one is present)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert varlen_strided(lib) in (fa.FA_ERR_LAUNCH, fa.FA_ERR_ARCH)
    # The contiguous strides are the plain entry point's.
    assert varlen_strided(lib, vr=4 * 64, vh=64) in (fa.FA_ERR_LAUNCH, fa.FA_ERR_ARCH)


def decode(lib, **kw):
    a = dict(q=P(0x1000), c=P(0x2000), pt=P(0x3000), ti=P(0x4000), T=4, H=64, topk=256,
             pages=100, maxp=16, scale=0.04, out=P(0x5000), lse=None, stream=None)
    a.update(kw)
    return lib.fa_sparse_mla_decode(a["q"], a["c"], a["pt"], a["ti"], a["T"], a["H"], a["topk"],
                                    a["pages"], a["maxp"], a["scale"], a["out"], a["lse"],
                                    a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(ti=None), fa.FA_ERR_INVALID_ARG),
    (dict(T=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(c=P(0x2004)), fa.FA_ERR_INVALID_ARG),
    (dict(H=48), fa.FA_ERR_UNSUPPORTED),
    (dict(topk=200), fa.FA_ERR_UNSUPPORTED),
    (dict(topk=2048, maxp=16), fa.FA_ERR_UNSUPPORTED),   # more slots than the context
    (dict(topk=1100, maxp=64), fa.FA_ERR_UNSUPPORTED),   # not a multiple of 128
])
def test_decode_host_validation(lib, kw, expect):
    assert decode(lib, **kw) == expect


def test_empty_extents_accept_null_buffers(lib):
    """Zero rows may come with null buffers (an empty torch tensor has no
    storage); without a GPU the call then fails only at the device query."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert varlen(lib, q=None, out=None, total_q=0) in (fa.FA_ERR_LAUNCH, fa.FA_ERR_ARCH)
    assert varlen(lib, k=None, v=None, total_k=0) in (fa.FA_ERR_LAUNCH, fa.FA_ERR_ARCH)
    assert decode(lib, q=None, pt=None, ti=None, out=None, T=0) in (fa.FA_ERR_LAUNCH,
                                                                    fa.FA_ERR_ARCH)
    # ... but not with rows.
    assert varlen(lib, q=None, out=None) == fa.FA_ERR_INVALID_ARG
    assert decode(lib, q=None, T=1) == fa.FA_ERR_INVALID_ARG


def test_valid_arguments_without_gpu_fail_cleanly(lib):
    """With no usable device the call returns a status instead of crashing."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert varlen(lib) in (fa.FA_ERR_LAUNCH, fa.FA_ERR_ARCH)


@pytest.mark.parametrize("args,expect", [
    ((4, 64, 256, True, True), None),            # valid: past the checks
    ((4, 64, 256, False, True), fa.FA_ERR_INVALID_ARG),
    ((4, 64, 256, True, False), fa.FA_ERR_INVALID_ARG),
    ((-1, 64, 256, True, True), fa.FA_ERR_INVALID_ARG),
    ((4, 48, 256, True, True), fa.FA_ERR_UNSUPPORTED),
    ((4, 64, 200, True, True), fa.FA_ERR_UNSUPPORTED),
    ((4, 64, 4100, True, True), fa.FA_ERR_UNSUPPORTED),
    ((4, 64, 8192, True, True), None),             # above 2048: always split
])
def test_decode_plan_host_validation(lib, args, expect):
    import torch
    T, H, topk, with_n, with_b = args
    n, b = ctypes.c_int(-5), ctypes.c_size_t(7)
    st = lib.fa_sparse_mla_decode_plan(T, H, topk, ctypes.byref(n) if with_n else None,
                                       ctypes.byref(b) if with_b else None)
    if expect is None:
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
        assert st in (fa.FA_ERR_LAUNCH, fa.FA_ERR_ARCH)
    else:
        assert st == expect
