"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library must build for sm_103a, load, export every function declared in
include/ccc.h, size its workspace by pure host arithmetic, and reject bad
arguments with the documented status codes before touching CUDA.
"""
import ctypes
import os
import re

import pytest

import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ccc.h")

OK, E_NULL, E_SHAPE, E_DTYPE, E_ALIGN, E_WS, E_ALIAS = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ccc_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"ccc_fwd", "ccc_bwd", "ccc_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in ccc.h but not exported"
    assert set(_lib.EXPORTS) <= set(names)


def test_status_strings(lib):
    assert _lib.status_string(0) == "CCC_OK"
    assert _lib.status_string(-6) == "CCC_ERR_ALIAS"
    assert _lib.status_string(5) == "unknown"


def test_workspace_size_rules(lib):
    ws = ccc.ccc_workspace_size
    # forward: never any scratch (the work split is found in-kernel)
    assert ws(16384, 4, 4096, False) == 0
    assert ws(65536, 200, 7168, False) == 0
    assert ws(1 << 24, 100000, 8192, False) == 0
    # backward: the FP32 partial sums, R = min(1216 // ceil(C / 256),
    # ceil(rows / 16)) (at least 1) rows of [5][C] floats, rounded up to 256
    # bytes; a function of rows and C, not of N
    for C in (8, 256, 264, 4096, 7168, 8192, 400000):
        for rows in (1, 15, 16, 17, 1040, 16384, 65536, 1 << 24):
            R = min(max(1, 1216 // ((C + 255) // 256)), (rows + 15) // 16)
            assert ws(rows, 200, C, True) == (R * 5 * C * 4 + 255) // 256 * 256, (C, rows)
            assert ws(rows, 1, C, True) == ws(rows, 9999, C, True)
    # the tiny training batch (1040 rows, C 256): 65 partial rows, not 1216
    assert ws(1040, 4, 256, True) == 65 * 5 * 256 * 4
    # degenerate / invalid
    assert ws(0, 4, 4096, True) == 0
    assert ws(100, 0, 4096, False) == 0
    assert ws(100, 4, 12, False) == 0
    assert ws(-1, 4, 4096, False) == 0


def test_noalloc_scratch_bound(lib):
    """The backward's scratch is R * 5 * C floats with R * ceil(C/256) <= 1216
    and R >= 1: at most max(6,225,920, 20 * C) bytes, so the fixed array
    behind ccc_bwd_noalloc holds every C up to 838,856."""
    for C in list(range(8, 70000, 8)) + [311288, 311296, 311304, 500000, 838856]:
        need = ccc.ccc_workspace_size(1 << 20, 1000, C, True)
        assert need <= max(6225920, (20 * C + 255) // 256 * 256), C
        assert need <= _lib.NOALLOC_SCRATCH_BYTES, C
    assert ccc.ccc_workspace_size(1 << 20, 1000, 838864, True) > _lib.NOALLOC_SCRATCH_BYTES


def test_noalloc_refuses_wider_than_its_array(lib):
    """C = 838,864 needs 16,777,280 bytes of partials, more than the array:
    refused with CCC_ERR_WORKSPACE by the size check, which runs before any
    CUDA call or pointer check (the fake addresses are never used)."""
    C = 838864
    f = lib.ccc_bwd_noalloc
    rc = f(P(A), 64, C, C, P(A * 2), 0, 4, None, -1, 1, None, P(A * 3), 1, None, None,
           P(A * 4), C, None, P(A * 5), C, P(A * 6), None, None, None)
    assert rc == E_WS


P = ctypes.c_void_p
A = 1 << 20  # fake, 16-byte aligned, never dereferenced


def fwd_args(**kw):
    a = dict(x=A, rows=64, C=256, xs=256, w=A * 2, wd=0, W=4, b=None, bd=-1, act=1,
             state=None, slots=0, L=0, s0=0, s1=0, s2=0, cu=A * 3, N=4, ci=None, hi=None,
             out=A * 4, os=256, hist=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return a


def call_fwd(lib, a):
    return lib.ccc_fwd(P(a["x"]), a["rows"], a["C"], a["xs"], P(a["w"]), a["wd"], a["W"], P(a["b"]), a["bd"],
                       a["act"], P(a["state"]), a["slots"], a["L"], a["s0"], a["s1"], a["s2"], P(a["cu"]), a["N"],
                       P(a["ci"]), P(a["hi"]), P(a["out"]), a["os"], P(a["hist"]), P(a["ws"]), a["wsb"],
                       P(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), E_NULL),
    (dict(out=None), E_NULL),
    (dict(cu=None), E_NULL),
    (dict(w=None), E_NULL),
    (dict(C=12, xs=16, os=16), E_SHAPE),
    (dict(C=0), E_SHAPE),
    (dict(xs=128), E_SHAPE),
    (dict(xs=260), E_SHAPE),
    (dict(rows=-1), E_SHAPE),
    (dict(wd=7), E_DTYPE),
    (dict(b=A * 5, bd=-1), E_DTYPE),
    (dict(b=None, bd=0), E_DTYPE),
    (dict(x=A + 8), E_ALIGN),
    (dict(out=A * 4 + 2), E_ALIGN),
    (dict(state=A * 6, slots=8, L=2, s0=1024, s1=4, s2=1, ci=A * 7), E_SHAPE),
    (dict(state=A * 6, slots=8, L=4, s0=1024, s1=2, s2=2, ci=A * 7), E_SHAPE),
    (dict(state=A * 6, slots=8, L=4, s0=100, s1=4, s2=1, ci=A * 7), E_SHAPE),  # slots overlap
    (dict(state=A * 6, slots=8, L=4, s0=1024, s1=4, s2=1, ci=None), E_NULL),
    (dict(out=A + 64 * 2), E_ALIAS),            # out overlaps x
    (dict(hist=A + 256, N=4), E_ALIAS),         # saved_hist inside x
    (dict(N=40, ws=None, rows=0), OK),          # the forward needs no workspace
    (dict(rows=0), OK),                         # nothing to do, nothing launched
    (dict(N=0), OK),
    (dict(W=5), E_SHAPE),                       # widths 2..4
    (dict(W=1), E_SHAPE),
    (dict(act=2), E_SHAPE),
    (dict(W=2, rows=0), OK),
    (dict(W=3, act=0, rows=0), OK),
    (dict(W=3, state=A * 6, slots=8, L=1, s0=1024, s1=1, s2=1, ci=A * 7), E_SHAPE),   # L < W-1
    (dict(W=2, rows=0, state=A * 6, slots=8, L=1, s0=256, s1=1, s2=1, ci=A * 7), OK),
])
def test_fwd_host_checks(lib, kw, code):
    assert call_fwd(lib, fwd_args(**kw)) == code


def test_fwd_state_layouts_accepted_by_checks(lib):
    # history-contiguous [slots, C, L] and channel-contiguous [slots, L, C]
    # views pass the layout check (rows == 0 keeps the call host-only)
    for s in ((1024, 4, 1), (1024, 1, 256), (256, 1, 256 * 8)):
        a = fwd_args(rows=0, state=A * 6, slots=8, L=4, s0=s[0], s1=s[1], s2=s[2], ci=A * 7)
        assert call_fwd(lib, a) == OK, s


def call_bwd(lib, **kw):
    a = dict(x=A, rows=64, C=256, xs=256, w=A * 2, wd=0, W=4, b=None, bd=-1, act=1, hist=None, cu=A * 3,
             N=4, ci=None, hi=None, dy=A * 4, dys=256, df=None, dx=A * 5, dxs=256, dw=A * 6, db=None,
             di=None, ws=A * 9, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.ccc_bwd(P(a["x"]), a["rows"], a["C"], a["xs"], P(a["w"]), a["wd"], a["W"], P(a["b"]), a["bd"],
                       a["act"], P(a["hist"]), P(a["cu"]), a["N"], P(a["ci"]), P(a["hi"]), P(a["dy"]), a["dys"],
                       P(a["df"]), P(a["dx"]), a["dxs"], P(a["dw"]), P(a["db"]), P(a["di"]), P(a["ws"]),
                       a["wsb"], P(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(dy=None), E_NULL),
    (dict(dx=None), E_NULL),
    (dict(dw=None), E_NULL),
    (dict(dx=A + 8), E_ALIGN),
    (dict(df=A * 7 + 4), E_ALIGN),
    (dict(dxs=8), E_SHAPE),
    (dict(ws=None), E_WS),
    (dict(wsb=8), E_WS),
    (dict(dx=A + 128), E_ALIAS),          # dx overlaps x
    (dict(dw=A * 4 + 64), E_ALIAS),       # dweight inside dy
    (dict(di=A * 9 + 256), E_ALIAS),      # d_init inside the workspace
    (dict(W=7), E_SHAPE),
    (dict(act=-1), E_SHAPE),
    (dict(W=4, dw=A * 4 - 256 * 2 * 4), E_ALIAS),   # dweight [C, 4] runs into dy
])
def test_bwd_host_checks(lib, kw, code):
    assert call_bwd(lib, **kw) == code


def call_update(lib, **kw):
    a = dict(x=A, rows=64, C=256, xs=256, w=A * 2, wd=0, W=4, b=None, bd=-1, act=1,
             state=A * 6, slots=8, L=4, s0=1024, s1=4, s2=1, cu=A * 3, N=4, ci=A * 7, na=None,
             out=A * 4, os=256, stream=None)
    a.update(kw)
    return lib.ccc_update(P(a["x"]), a["rows"], a["C"], a["xs"], P(a["w"]), a["wd"], a["W"], P(a["b"]), a["bd"],
                          a["act"], P(a["state"]), a["slots"], a["L"], a["s0"], a["s1"], a["s2"], P(a["cu"]),
                          a["N"], P(a["ci"]), P(a["na"]), P(a["out"]), a["os"], P(a["stream"]))


@pytest.mark.parametrize("kw,code", [
    (dict(state=None), E_NULL),                 # the pool is required
    (dict(ci=None), E_NULL),
    (dict(out=None), E_NULL),
    (dict(L=2), E_SHAPE),                       # L < W-1
    (dict(W=2, L=0), E_SHAPE),
    (dict(s1=2, s2=2), E_SHAPE),                # neither channel nor history axis contiguous
    (dict(W=5), E_SHAPE),
    (dict(act=3), E_SHAPE),
    (dict(na=A * 8 + 2), E_ALIGN),
    (dict(out=A + 64), E_ALIAS),                # out overlaps x
    (dict(na=A * 6 + 64), E_ALIAS),             # accepted counts inside the pool (read-only operand vs written pool)
    (dict(rows=0), OK),                         # nothing to do, nothing launched
    (dict(N=0), OK),
    (dict(W=2, L=1, s0=256, s1=1, s2=1, rows=0), OK),
])
def test_update_host_checks(lib, kw, code):
    assert call_update(lib, **kw) == code


def test_check_status_words(lib):
    w = lib.ccc_check_status_words
    assert [w(0), w(1), w(32), w(33), w(100000)] == [1, 2, 2, 3, 1 + 3125]


def test_check_host_errors(lib):
    """ccc_check's host checks fail before any CUDA call (the fake device
    addresses are never dereferenced)."""
    P = ctypes.c_void_p
    cu, cache, acc, st = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    chk = lib.ccc_check
    assert chk(10, None, 2, None, 0, None, 0, st, 1, None) == E_NULL
    assert chk(10, cu, 2, None, 0, None, 0, None, 1, None) == E_NULL
    assert chk(-1, cu, 2, None, 0, None, 0, st, 1, None) == E_SHAPE
    assert chk(10, cu, -1, None, 0, None, 0, st, 1, None) == E_SHAPE
    assert chk(10, cu, 2, cache, -1, None, 0, st, 9, None) == E_SHAPE
    assert chk(10, cu, 2, None, 0, acc, 0, st, 1, None) == E_SHAPE          # max_accepted < 1
    assert chk(10, P(0x10001), 2, None, 0, None, 0, st, 1, None) == E_ALIGN
    assert chk(10, cu, 2, cache, 0, None, 0, P(0x40002), 1, None) == E_ALIGN
    assert chk(10, cu, 2, cache, 100, None, 0, st, 4, None) == E_WS         # needs 1 + 4 words
    assert chk(10, cu, 2, None, 0, None, 0, st, 0, None) == E_WS
    assert chk(10, cu, 2, None, 0, None, 0, P(0x10008), 1, None) == E_ALIAS  # status inside cu_seqlens
    assert chk(10, cu, 2, cache, 64, None, 0, P(0x1fffc), 3, None) == E_ALIAS  # bitmap runs into cache


def test_binding_rejects_tensors_off_the_current_device(lib):
    """The binding hands raw pointers to kernels launched on the current CUDA
    device, so it refuses CPU tensors (and tensors on another GPU) before
    calling the library."""
    import torch
    x = torch.zeros((16, 8), dtype=torch.bfloat16)
    w = torch.zeros((8, 4))
    cu = torch.tensor([0, 16], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        ccc.ccc_fwd(x, w, None, None, cu, None, None, torch.empty_like(x))
    with pytest.raises(ValueError, match="CUDA tensors"):
        ccc.ccc_bwd_noalloc(x, w, None, None, cu, None, None, x, None, torch.empty_like(x),
                            torch.empty((8, 4)), None, None)


def test_launch_options(lib):
    """ccc_fwd_ex / ccc_bwd_ex / ccc_update_ex take CCC_OPT_OVERLAP_PROLOGUE
    (bit 0) and refuse any other bit before touching CUDA."""
    a = fwd_args()
    args = [P(a["x"]), a["rows"], a["C"], a["xs"], P(a["w"]), a["wd"], a["W"], P(a["b"]), a["bd"], a["act"],
            P(a["state"]), a["slots"], a["L"], a["s0"], a["s1"], a["s2"], P(a["cu"]), a["N"], P(a["ci"]),
            P(a["hi"]), P(a["out"]), a["os"], P(a["hist"]), P(a["ws"]), a["wsb"]]
    for bad in (2, 4, 1 << 31, 3):
        assert lib.ccc_fwd_ex(*args, bad, None) == E_SHAPE
    zero = list(args)
    zero[1] = 0  # rows == 0: checks pass, nothing launched
    assert lib.ccc_fwd_ex(*zero, _lib.OPT_OVERLAP_PROLOGUE, None) == OK
    b = [P(A), 64, 256, 256, P(A * 2), 0, 4, None, -1, 1, None, P(A * 3), 4, None, None, P(A * 4), 256, None,
         P(A * 5), 256, P(A * 6), None, None, P(A * 9), 1 << 30]
    assert lib.ccc_bwd_ex(*b, 2, None) == E_SHAPE
    assert lib.ccc_bwd_ex(*b, 4, None) == E_SHAPE
    u = [P(A), 64, 256, 256, P(A * 2), 0, 4, None, -1, 1, P(A * 6), 8, 4, 1024, 4, 1, P(A * 3), 4, P(A * 7),
         None, P(A * 4), 256]
    for bad in (2, 8, 1 << 31):
        assert lib.ccc_update_ex(*u, bad, None) == E_SHAPE
    u[1] = 0  # rows == 0: checks pass, nothing launched
    assert lib.ccc_update_ex(*u, _lib.OPT_OVERLAP_PROLOGUE, None) == OK


def test_empty_batch_takes_null_row_buffers(lib):
    """rows == 0: the row buffers may be NULL (an empty tensor has no storage);
    the forward and the decode step return CCC_OK without any CUDA call, and
    the pointers that are still required stay required."""
    assert call_fwd(lib, fwd_args(rows=0, x=None, out=None)) == OK
    assert call_fwd(lib, fwd_args(rows=0, x=None, out=None, w=None)) == E_NULL
    assert call_fwd(lib, fwd_args(rows=0, x=None, out=None, cu=None)) == E_NULL
    assert call_fwd(lib, fwd_args(rows=1, x=None)) == E_NULL
    assert call_update(lib, rows=0, x=None, out=None) == OK
    assert call_update(lib, rows=0, x=None, out=None, state=None) == E_NULL
    assert call_update(lib, rows=1, out=None) == E_NULL


@pytest.mark.gpu
def test_stream_handle_is_the_current_stream(cuda_device):
    """The binding's stream argument for stream=None is torch's current stream
    on the current device (also inside a torch.cuda.stream context)."""
    import torch
    import ssm_depthwise_causal_gb300 as ccc
    assert ccc._stream(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert ccc._stream(None) == s.cuda_stream
    assert ccc._stream(s) == s.cuda_stream
