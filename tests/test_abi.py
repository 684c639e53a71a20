"""CPU tests of the C-ABI library: it builds, loads, exports every function
declared in include/etattn.h, and rejects invalid calls with the documented
status codes before touching CUDA (so no GPU is needed)."""

import ctypes
import os
import re

import pytest

from exact_tiled_attention_19_gb300 import binding as B
from exact_tiled_attention_19_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Fake, 16-byte aligned, non-overlapping device addresses: validation never
# dereferences them.
Q, K, V, O, LSE = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def contiguous_strides(B_, H, N, D):
    return [H * N * D, N * D, D, 1]


def good_args(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=LSE, B=2, Hq=4, Hkv=2, N=100, D=64, dtype=1, causal=1, scale=0.125,
             stream=0)
    a.update(kw)
    if "strides" not in a:
        a["strides"] = (contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]) +
                        contiguous_strides(a["B"], a["Hkv"], a["N"], a["D"]) * 2 +
                        contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]))
    return a


def call(**kw):
    a = good_args(**kw)
    return B.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], a["D"],
                      a["dtype"], a["strides"], a["causal"], a["scale"], a["stream"])


def declared_functions():
    with open(os.path.join(ROOT, "include", "etattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text)))


def test_library_builds_and_exports_every_declared_symbol():
    path = build_lib.build()
    lib = ctypes.CDLL(path)
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_varlen", "etattn_status_string", "etattn_version"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/etattn.h but not exported"


def test_status_strings_and_version():
    for code in range(13):
        s = B.etattn_status_string(code)
        assert s and s != "unknown status"
    assert B.etattn_status_string(999) == "unknown status"
    assert B.etattn_version() >= 100


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), 2),
    (dict(D=96), 3), (dict(D=256), 3), (dict(N=-1), 3), (dict(B=-1), 3), (dict(N=2 ** 30 + 1), 3),
    (dict(B=65536), 3), (dict(Hq=65536, Hkv=1), 3),
    (dict(Hkv=0), 4), (dict(Hkv=3), 4), (dict(Hq=4, Hkv=8), 4),
    (dict(scale=0.0), 8), (dict(scale=-1.0), 8), (dict(scale=float("inf")), 8), (dict(scale=float("nan")), 8),
    (dict(q=0), 1), (dict(o=0), 1), (dict(k=0), 1),
    (dict(q=Q + 8), 6), (dict(o=O + 2), 6), (dict(lse=LSE + 2), 6),
    (dict(o=Q + 64), 7), (dict(lse=K), 7), (dict(lse=O + 1024), 7),
])
def test_invalid_arguments_rejected(kw, code):
    assert call(**kw) == code


def test_stride_rules():
    a = good_args()
    s = list(a["strides"])
    s[3] = 2  # q d-stride
    assert call(strides=s) == 5
    s = list(a["strides"])
    s[2] = 60  # q n-stride of 120 bytes: not a multiple of 16
    assert call(strides=s) == 5
    s = list(a["strides"])
    s[14] = -64  # o n-stride negative
    assert call(strides=s) == 5
    s = list(a["strides"])
    s[5] = 0  # k head stride 0 with Hkv = 2 (broadcast) is refused
    assert call(strides=s) == 5


def test_null_strides_rejected():
    lib = B.load_library()
    rc = lib.attn_fwd(Q, K, V, O, LSE, 1, 1, 1, 8, 64, 0, None, 1, ctypes.c_float(0.1), None)
    assert rc == 1


def test_empty_work_is_a_noop_even_with_null_pointers():
    assert call(N=0, q=0, k=0, v=0, o=0, lse=0) == 0
    assert call(B=0) == 0
    assert call(Hq=0, Hkv=1) == 0


def test_valid_call_without_gpu_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() == 12


def varlen_call(cu_host=None, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=LSE, cu=0x60000000, num_seqs=3, max_seqlen=50, T=100, Hq=4, Hkv=4, D=128,
             dtype=1, causal=1, scale=0.1, stream=0)
    a.update(kw)
    st = [a["Hq"] * a["D"], a["D"], 1, a["Hkv"] * a["D"], a["D"], 1, a["Hkv"] * a["D"], a["D"], 1,
          a["Hq"] * a["D"], a["D"], 1]
    host = 0
    if cu_host is not None:
        arr = (ctypes.c_int32 * len(cu_host))(*cu_host)
        host = ctypes.addressof(arr)
        a["_keep"] = arr
    return B.attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], host, a["num_seqs"],
                             a["max_seqlen"], a["T"], a["Hq"], a["Hkv"], a["D"], a["dtype"], st, a["causal"],
                             a["scale"], a["stream"])


@pytest.mark.parametrize("cu,code", [
    ([0, 30, 60, 100], 0), ([1, 30, 60, 100], 9), ([0, 30, 20, 100], 9), ([0, 30, 60, 99], 9),
    ([0, 10, 20, 100], 9),  # last length 80 > max_seqlen 50
])
def test_varlen_host_seqlens_validation(cu, code):
    import torch
    rc = varlen_call(cu_host=cu)
    if code == 0:
        assert rc in (0, 12) if not torch.cuda.is_available() else rc == 0
    else:
        assert rc == code


def test_varlen_argument_errors():
    assert varlen_call(cu=0) == 1
    assert varlen_call(D=48) == 3
    assert varlen_call(Hkv=3) == 4
    assert varlen_call(num_seqs=0) == 0
    assert varlen_call(T=0, max_seqlen=0) == 0
    assert varlen_call(cu=0x60000002) == 6


def test_host_entry_points_validate_before_copying():
    H = 0x70000000  # fake host addresses (never touched: validation fails first or no GPU)
    # lse host/device must be both given or both NULL
    assert B.attn_fwd_host(H, H + 0x100000, H + 0x200000, H + 0x300000, H + 0x400000, Q, K, V, O, 0, 1, 2, 2, 64,
                           64, 1, 1, 0.125, 0) == 1
    assert B.attn_fwd_host(H, H, H, H, 0, Q, K, V, O, 0, 1, 2, 2, 64, 48, 1, 1, 0.125, 0) == 3
    assert B.attn_fwd_host(H, H, H, H, 0, Q, K, V, Q + 64, 0, 1, 2, 2, 64, 64, 1, 1, 0.125, 0) == 7
    assert B.attn_fwd_host(0, 0, 0, 0, 0, Q, K, V, O, 0, 0, 2, 2, 64, 64, 1, 1, 0.125, 0) == 0  # empty
    cu = (ctypes.c_int32 * 3)(0, 10, 30)
    cu_bad = (ctypes.c_int32 * 3)(0, 40, 30)
    args = dict(num_seqs=2, max_seqlen=20, T=30, Hq=2, Hkv=2, D=64, dtype=1, causal=1, scale=0.1)

    def vh(cu_arr, **kw):
        a = dict(args, **kw)
        return B.attn_fwd_varlen_host(H, H, H, H, 0, ctypes.addressof(cu_arr) if cu_arr is not None else 0, Q, K,
                                      V, O, 0, 0x60000000, a["num_seqs"], a["max_seqlen"], a["T"], a["Hq"],
                                      a["Hkv"], a["D"], a["dtype"], a["causal"], a["scale"], 0)
    assert vh(None) == 1
    assert vh(cu_bad) == 9
    assert vh(cu, Hkv=3) == 4
    assert vh(cu, scale=-1.0) == 8


def ex_call(**kw):
    a = good_args(**kw)
    Nk = kw.get("Nk", a["N"])
    st = a["strides"] if "strides" in kw else (contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]) +
                                               contiguous_strides(a["B"], a["Hkv"], Nk, a["D"]) * 2 +
                                               contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]))
    return B.attn_fwd_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], Nk, a["D"],
                         a["dtype"], st, a["causal"], kw.get("wl", -1), kw.get("wr", -1), a["scale"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Nk=-1), 3), (dict(Nk=2 ** 30 + 1), 3), (dict(N=-1), 3),
    (dict(k=0), 1), (dict(v=0), 1), (dict(q=0), 1),
    (dict(k=K + 8), 6), (dict(Hkv=3), 4), (dict(scale=0.0), 8),
])
def test_ex_invalid_arguments_rejected(kw, code):
    assert ex_call(**kw) == code


def test_ex_empty_queries_are_a_noop_and_no_keys_needs_no_key_pointers():
    import torch
    assert ex_call(N=0, q=0, k=0, v=0, o=0, lse=0) == 0
    rc = ex_call(Nk=0, k=0, v=0, wl=5)  # valid: every row is empty; needs a device to run
    assert rc == (12 if not torch.cuda.is_available() else 0)


def varlen_ex_call(cu_q_host=None, cu_k_host=None, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=LSE, cuq=0x60000000, cuk=0x60001000, num_seqs=3, mq=50, mk=80, Tq=100, Tk=150,
             Hq=4, Hkv=2, D=128, dtype=1, causal=1, wl=-1, wr=-1, scale=0.1, stream=0)
    a.update(kw)
    st = [a["Hq"] * a["D"], a["D"], 1, a["Hkv"] * a["D"], a["D"], 1, a["Hkv"] * a["D"], a["D"], 1,
          a["Hq"] * a["D"], a["D"], 1]
    keep = []

    def host(arr):
        if arr is None:
            return 0
        c = (ctypes.c_int32 * len(arr))(*arr)
        keep.append(c)
        return ctypes.addressof(c)
    return B.attn_fwd_varlen_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cuq"], a["cuk"], host(cu_q_host),
                                host(cu_k_host), a["num_seqs"], a["mq"], a["mk"], a["Tq"], a["Tk"], a["Hq"], a["Hkv"],
                                a["D"], a["dtype"], st, a["causal"], a["wl"], a["wr"], a["scale"], a["stream"])


@pytest.mark.parametrize("cq,ck,code", [
    ([0, 30, 60, 100], [0, 80, 80, 150], 0),
    ([0, 30, 60, 100], [0, 80, 70, 150], 9),   # key offsets decrease
    ([0, 30, 60, 100], [0, 10, 20, 149], 9),   # key offsets end short of the key total
    ([0, 30, 60, 100], [0, 90, 100, 150], 9),  # a key length above max_seqlen_k
    ([0, 60, 60, 100], [0, 80, 80, 150], 9),   # a query length above max_seqlen_q
])
def test_varlen_ex_host_offsets_validation(cq, ck, code):
    import torch
    rc = varlen_ex_call(cu_q_host=cq, cu_k_host=ck)
    if code == 0:
        assert rc == (12 if not torch.cuda.is_available() else 0)
    else:
        assert rc == code


def test_varlen_ex_argument_errors():
    assert varlen_ex_call(cuk=0) == 1
    assert varlen_ex_call(cuq=0) == 1
    assert varlen_ex_call(cuk=0x60001002) == 6
    assert varlen_ex_call(mk=-1) == 3
    assert varlen_ex_call(Tk=-1) == 3
    assert varlen_ex_call(Tq=0) == 0
    assert varlen_ex_call(num_seqs=0) == 0


def varlen_split_call(kind="split", num_splits=4, num_global=8, ws=0x70000000, ws_bytes=1 << 30, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=LSE, cuq=0x60000000, cuk=0x60001000, num_seqs=3, mq=50, mk=80, Tq=100, Tk=150,
             Hq=4, Hkv=2, D=128, dtype=1, causal=1, wl=32, wr=-1, scale=0.1, stream=0)
    a.update(kw)
    st = [a["Hq"] * a["D"], a["D"], 1, a["Hkv"] * a["D"], a["D"], 1, a["Hkv"] * a["D"], a["D"], 1,
          a["Hq"] * a["D"], a["D"], 1]
    common = (a["q"], a["k"], a["v"], a["o"], a["lse"], a["cuq"], a["cuk"], 0, 0, a["num_seqs"], a["mq"], a["mk"],
              a["Tq"], a["Tk"], a["Hq"], a["Hkv"], a["D"], a["dtype"], st, a["causal"], a["wl"], a["wr"])
    if kind == "split":
        return B.attn_fwd_varlen_splitkv(*common, a["scale"], num_splits, ws, ws_bytes, a["stream"])
    return B.attn_fwd_varlen_global(*common, num_global, a["scale"], a["stream"])


def test_varlen_splitkv_workspace_formula():
    rows = 100 * 4
    o_bytes = 3 * rows * 128 * 4
    padded = (o_bytes + 255) // 256 * 256
    assert B.attn_fwd_varlen_splitkv_workspace_size(100, 4, 128, 3) == padded + 3 * rows * 4
    assert B.attn_fwd_varlen_splitkv_workspace_size(100, 4, 128, 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), 1), (dict(ws=0x70000010), 6), (dict(ws_bytes=1000), 3), (dict(ws=Q), 7),
])
def test_varlen_splitkv_workspace_errors(kw, code):
    assert varlen_split_call("split", **kw) == code


@pytest.mark.parametrize("kind", ["split", "global"])
@pytest.mark.parametrize("kw,code", [(dict(Hkv=3), 4), (dict(cuk=0), 1), (dict(mk=-1), 3)])
def test_varlen_split_and_global_invalid_arguments_rejected(kind, kw, code):
    assert varlen_split_call(kind, **kw) == code


def test_varlen_split_and_global_special_values():
    import torch
    want = 12 if not torch.cuda.is_available() else 0
    assert varlen_split_call("split", num_splits=0) == 3
    assert varlen_split_call("split", num_splits=1025) == 3
    assert varlen_split_call("global", num_global=-1) == 3
    assert varlen_split_call("split") == want
    assert varlen_split_call("global") == want
    assert varlen_split_call("split", num_splits=1, ws=0, ws_bytes=0) == want   # one slice: no workspace
    assert varlen_split_call("global", num_global=0) == want                    # no global token: plain call
    assert varlen_split_call("split", Tq=0) == 0
    rc, n = B.attn_fwd_varlen_splitkv_plan(8, 32, 8, 1, 32768)
    assert rc == want and (rc != 0 or n >= 1)
    assert B.attn_fwd_varlen_splitkv_plan(8, 32, 3, 1, 32768)[0] == 4    # Hq % Hkv != 0


def test_splitkv_workspace_size_formula():
    rows = 2 * 8 * 3
    o_bytes = 5 * rows * 128 * 4
    padded = (o_bytes + 255) // 256 * 256
    assert B.attn_fwd_splitkv_workspace_size(2, 8, 3, 128, 5) == padded + 5 * rows * 4
    assert B.attn_fwd_splitkv_workspace_size(2, 8, 3, 128, 1) == 0
    assert B.attn_fwd_splitkv_workspace_size(2, 8, 3, 96, 5) == 0      # bad head dim
    assert B.attn_fwd_splitkv_workspace_size(2, 8, 3, 64, 1025) == 0   # too many slices


def splitkv_call(num_splits=4, ws=0x70000000, ws_bytes=1 << 30, **kw):
    a = good_args(**kw)
    Nk = kw.get("Nk", a["N"])
    st = (contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]) + contiguous_strides(a["B"], a["Hkv"], Nk, a["D"]) * 2
          + contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]))
    return B.attn_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], Nk, a["D"],
                              a["dtype"], st, a["causal"], -1, -1, a["scale"], num_splits, ws, ws_bytes, a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(num_splits=0), 3), (dict(num_splits=1025), 3),
    (dict(ws=0), 1), (dict(ws=0x70000010), 6), (dict(ws_bytes=1000), 3),
    (dict(ws=Q), 7), (dict(ws=O - 256), 7),
    (dict(Hkv=3), 4), (dict(N=-1), 3),
])
def test_splitkv_invalid_arguments_rejected(kw, code):
    assert splitkv_call(**kw) == code


def test_splitkv_valid_calls_need_a_device():
    import torch
    want = 12 if not torch.cuda.is_available() else 0
    assert splitkv_call() == want
    assert splitkv_call(num_splits=1, ws=0, ws_bytes=0) == want   # one slice: no workspace needed
    assert splitkv_call(N=0) == 0                                 # no queries: no-op
    rc, n = B.attn_fwd_splitkv_plan(4, 8, 2, 1, 4096)
    assert rc == want and (rc != 0 or n >= 1)


def global_call(num_global=8, wl=32, wr=-1, **kw):
    a = good_args(**kw)
    Nk = kw.get("Nk", a["N"])
    st = (contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]) + contiguous_strides(a["B"], a["Hkv"], Nk, a["D"]) * 2
          + contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]))
    return B.attn_fwd_global(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], Nk, a["D"],
                             a["dtype"], st, a["causal"], wl, wr, num_global, a["scale"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(num_global=-1), 3), (dict(Hkv=3), 4), (dict(N=-1), 3), (dict(q=0), 1),
])
def test_global_invalid_arguments_rejected(kw, code):
    assert global_call(**kw) == code


def test_global_valid_calls_need_a_device():
    import torch
    want = 12 if not torch.cuda.is_available() else 0
    assert global_call() == want
    assert global_call(num_global=0) == want        # plain windowed call
    assert global_call(wl=-1) == want               # causal, no left bound: the window is all
    assert global_call(N=0) == 0                    # no queries: no-op


def noalloc_call(num_splits=4, **kw):
    a = good_args(**kw)
    Nk = kw.get("Nk", a["N"])
    st = (contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]) + contiguous_strides(a["B"], a["Hkv"], Nk, a["D"]) * 2
          + contiguous_strides(a["B"], a["Hq"], a["N"], a["D"]))
    return B.attn_fwd_splitkv_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], Nk,
                                      a["D"], a["dtype"], st, a["causal"], -1, -1, a["scale"], num_splits,
                                      a["stream"])


def test_noalloc_refuses_problems_beyond_its_scratch_before_any_device_work():
    import torch
    # 2 x 4 x 100 rows x 64 slices x (4 * 64 + 4) bytes = 13.3 MB fits in 16 MiB; 128 slices do not.
    want = 12 if not torch.cuda.is_available() else 0
    assert noalloc_call(num_splits=64) == want
    assert noalloc_call(num_splits=128) == 3
    assert noalloc_call(num_splits=0) == 3
    assert noalloc_call(num_splits=4, o=Q + 64) == 7
    assert noalloc_call(num_splits=4, N=0) == 0
    # Without keys nothing is split and no scratch is used: a row count far
    # beyond the scratch passes the size check (and then needs a device).
    assert noalloc_call(num_splits=128, N=20000, Nk=0, k=0, v=0) == want


DQ, DK, DV, DO, OO, WS = 0x80000000, 0x90000000, 0xA0000000, 0xB0000000, 0xC0000000, 0xD0000000


def bwd_call(**kw):
    a = dict(q=Q, k=K, v=V, o=OO, lse=LSE, dout=DO, dq=DQ, dk=DK, dv=DV, B=2, Hq=4, Hkv=2, Nq=100, Nk=120, D=64,
             dtype=1, causal=1, wl=-1, wr=-1, scale=0.125, ws=WS, ws_bytes=1 << 26, stream=0)
    a.update(kw)
    qs = contiguous_strides(a["B"], a["Hq"], a["Nq"], a["D"])
    ks = contiguous_strides(a["B"], a["Hkv"], a["Nk"], a["D"])
    st = qs + ks + ks + qs + qs + qs + ks + ks
    return B.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"], a["dv"], a["B"], a["Hq"],
                      a["Hkv"], a["Nq"], a["Nk"], a["D"], a["dtype"], st, a["causal"], a["wl"], a["wr"], a["scale"],
                      a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), 2), (dict(D=48), 3), (dict(Nk=-1), 3), (dict(Hkv=3), 4), (dict(scale=0.0), 8),
    (dict(lse=0), 1), (dict(dout=0), 1), (dict(dk=0), 1), (dict(ws=0), 1),
    (dict(dq=DQ + 8), 6), (dict(ws=WS + 16), 6), (dict(ws_bytes=1000), 3),
    (dict(dq=Q + 128), 7), (dict(dk=DV), 7), (dict(ws=DQ), 7), (dict(dv=LSE), 7),
])
def test_bwd_invalid_arguments_rejected(kw, code):
    assert bwd_call(**kw) == code


def test_bwd_workspace_and_empty_calls():
    import torch
    rows = 2 * 4 * 100
    n_pad = 2 * 4 * 128
    up = lambda x: (x + 255) // 256 * 256
    assert B.attn_bwd_workspace_size(2, 4, 100, 64) == up(rows * 64 * 4) + 2 * up(n_pad * 4)
    assert B.attn_bwd_workspace_size(2, 4, 0, 64) == 0
    assert bwd_call(B=0) == 0
    assert bwd_call(Nq=0, Nk=0) == 0
    want = 12 if not torch.cuda.is_available() else 0
    assert bwd_call() == want
    assert bwd_call(Nq=0, q=0, o=0, lse=0, dout=0, dq=0, ws=0, ws_bytes=0) == want  # no queries: dk = dv = 0


def test_wait_selftest_checks_its_limit_before_any_device_work():
    import torch
    assert B.etattn_selftest_wait_timeout(0) == 3
    assert B.etattn_selftest_wait_timeout(1000001) == 3
    assert B.etattn_selftest_wait_timeout(1000) == (12 if not torch.cuda.is_available() else 0)
    if torch.cuda.is_available():
        B.etattn_read_device_status(clear=True)


# ---------------------------------------------------------------- host-buffer chunk plan

def _check_plan(lengths, max_chunks):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    k, b = B.attn_fwd_varlen_host_plan(cu, max_chunks)
    n = len(lengths)
    if n == 0:
        assert k == 0 and b == []
        return k, b
    k_max = max(1, min(max_chunks, 8, n))
    assert 1 <= k <= k_max and len(b) == k + 1
    assert b[0] == 0 and b[-1] == n and all(x < y for x, y in zip(b, b[1:]))
    T = cu[-1]
    if T > 0:
        for c in range(k - 1):  # run c (all but the last) ends at its first sequence reaching its share
            share = (c + 1) * T
            assert cu[b[c + 1]] * k_max >= share
            assert b[c + 1] - 1 == b[c] or cu[b[c + 1] - 1] * k_max < share
    return k, b


def test_host_plan_packed_workload_runs():
    # the packed benchmark batch's 16 lengths: runs of about T / 8 tokens, cut by hand
    lengths = [12464, 9413, 538, 10743, 5700, 4308, 920, 13928, 1373, 11450, 7567, 2584, 11849, 4442, 12655, 14891]
    k, b = _check_plan(lengths, 8)
    assert k == 8 and b == [0, 2, 4, 8, 10, 11, 14, 15, 16]


@pytest.mark.parametrize("lengths,max_chunks,want", [
    ([100] * 16, 8, [0, 2, 4, 6, 8, 10, 12, 14, 16]),      # equal lengths: equal runs
    ([100] * 16, 99, [0, 2, 4, 6, 8, 10, 12, 14, 16]),     # at most 8 runs
    ([100] * 3, 8, [0, 1, 2, 3]),                          # at most one run per sequence
    ([100] * 4, 1, [0, 4]),                                # one run: the whole batch
    ([10000, 1, 1, 1], 8, [0, 1, 2, 3, 4]),
    ([1, 1, 1, 10000], 8, [0, 4]),                         # the long last sequence holds every share
    ([0, 0, 0], 8, [0, 3]),                                # no tokens: one run
    ([5, 0, 7, 0, 3], 2, [0, 3, 5]),
])
def test_host_plan_examples(lengths, max_chunks, want):
    k, b = _check_plan(lengths, max_chunks)
    assert b == want


def test_host_plan_random_properties():
    import random
    rng = random.Random(3)
    for _ in range(300):
        n = rng.randint(0, 40)
        lengths = [rng.choice([0, rng.randint(1, 300), rng.randint(1, 20000)]) for _ in range(n)]
        _check_plan(lengths, rng.randint(1, 12))


def test_host_plan_rejects_bad_arguments():
    assert B.attn_fwd_varlen_host_plan([0, 5, 3], 8)[0] == -9     # offsets decrease
    assert B.attn_fwd_varlen_host_plan([0, 5], 0)[0] == -3        # max_chunks < 1
    assert B.attn_fwd_varlen_host_plan([], 8)[0] == -3            # num_seqs = -1
    lib = B.load_library()
    assert lib.attn_fwd_varlen_host_plan(None, 1, 8, (ctypes.c_int32 * 9)()) == -1
