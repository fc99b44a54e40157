"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a,
loads, exports every function include/fa.h declares, and rejects bad arguments with
the documented status codes before touching CUDA."""

import ctypes

import pytest

from tests.helpers import ensure_built


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from flashattention_backward_pass_gb300 import _abi
    return _abi.load()


def test_exports_every_declared_symbol(lib):
    from flashattention_backward_pass_gb300._abi import declared_functions
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_status",
                     "fa_status_string", "fa_abi_version", "fa_fwd_workspace_size"):
        assert required in names
    for n in names:
        assert hasattr(lib, n), f"libfa_gb300.so does not export {n}"


def test_version_and_strings(lib):
    assert lib.fa_abi_version() == 3
    for code in range(0, -12, -1):
        s = lib.fa_status_string(code)
        assert s and s.startswith(b"FA_")
    assert lib.fa_status_string(12345) == b"unknown fa status"


def _view(shape, strides=None, dtype=0, data=4096):
    from flashattention_backward_pass_gb300._abi import FaTensor
    t = FaTensor()
    t.data = data
    nd = len(shape)
    if strides is None:
        strides = [0] * nd
        acc = 1
        for i in reversed(range(nd)):
            strides[i] = acc
            acc *= shape[i]
    for i in range(4):
        t.shape[i] = shape[i] if i < nd else 0
        t.stride[i] = strides[i] if i < nd else 0
    t.ndim = nd
    t.dtype = dtype
    return t


def _bwd_args(B=1, Sq=128, Sk=128, H=2, Hk=2, D=64, **over):
    a = dict(dout=_view((B, Sq, H, D)), q=_view((B, Sq, H, D)), k=_view((B, Sk, Hk, D)),
             v=_view((B, Sk, Hk, D)), out=_view((B, Sq, H, D)), lse=_view((B, H, Sq), dtype=1),
             dq=_view((B, Sq, H, D)), dk=_view((B, Sk, Hk, D)), dv=_view((B, Sk, Hk, D)))
    a.update(over)
    return a


def _call_bwd(lib, a, scale=0.125, causal=0, wl=-1, wr=-1, softcap=0.0, det=0, ws=4096, ws_bytes=1 << 30):
    order = ("dout", "q", "k", "v", "out", "lse", "dq", "dk", "dv")
    ptrs = [ctypes.byref(a[n]) if a[n] is not None else None for n in order]
    return lib.fa_bwd(*ptrs, scale, causal, wl, wr, softcap, det, ctypes.c_void_p(ws), ws_bytes, None)


def test_bwd_validation_codes(lib):
    assert _call_bwd(lib, _bwd_args(q=None)) == -1                       # FA_ERR_NULL
    a = _bwd_args(); a["k"] = _view((1, 128, 2, 32))
    assert _call_bwd(lib, a) == -2                                       # K head dim mismatch
    a = _bwd_args(); a["v"] = _view((1, 64, 2, 64))
    assert _call_bwd(lib, a) == -2                                       # K/V mismatch
    assert _call_bwd(lib, _bwd_args(H=3, Hk=2)) == -2                    # H % Hk
    a = _bwd_args(); a["q"] = _view((1, 128, 2, 64), dtype=1)
    assert _call_bwd(lib, a) == -3                                       # dtype
    a = _bwd_args(); a["lse"] = _view((1, 2, 128), dtype=0)
    assert _call_bwd(lib, a) == -3                                       # LSE must be fp32
    assert _call_bwd(lib, _bwd_args(D=60)) == -4                         # D % 8
    assert _call_bwd(lib, _bwd_args(D=264)) == -4                        # D > 256
    assert _call_bwd(lib, _bwd_args(B=65536)) == -8                      # B above the grid limit
    a = _bwd_args(); a["q"] = _view((1, 128, 2, 64), strides=(128 * 2 * 64, 2 * 64, 64, 2))
    assert _call_bwd(lib, a) == -5                                       # last dim not contiguous
    a = _bwd_args(); a["q"] = _view((1, 128, 2, 64), data=4096 + 8)
    assert _call_bwd(lib, a) == -6                                       # base misaligned
    a = _bwd_args(); a["q"] = _view((1, 128, 2, 64), strides=(128 * 2 * 68, 2 * 68, 68, 1))
    assert _call_bwd(lib, a) == -6                                       # stride not 16 B
    assert _call_bwd(lib, _bwd_args(), ws_bytes=16) == -7                # workspace too small
    assert _call_bwd(lib, _bwd_args(), ws=0) == -7                       # no workspace
    assert _call_bwd(lib, _bwd_args(), scale=0.0) == -9                  # scale <= 0
    assert _call_bwd(lib, _bwd_args(), scale=float("nan")) == -9
    assert _call_bwd(lib, _bwd_args(), softcap=-1.0) == -9
    a = _bwd_args(); a["dq"] = _view((1, 128, 2, 64), data=0)
    assert _call_bwd(lib, a) == -1                                       # null output


def _f16_args(**kw):
    a = _bwd_args(**kw)
    for n in ("dout", "q", "k", "v", "out", "dq", "dk", "dv"):
        a[n].dtype = 2                                                   # FA_DTYPE_F16
    return a


def test_f16_validation(lib):
    # every 16-bit tensor f16 passes validation (an empty problem then launches nothing)
    assert _call_bwd(lib, _f16_args(Sq=0)) == 0
    for n in ("dout", "k", "v", "out", "dq", "dk", "dv"):
        a = _f16_args()
        a[n].dtype = 0                                                   # one bf16 among f16
        assert _call_bwd(lib, a) == -3, n
    a = _bwd_args(); a["dq"].dtype = 2                                   # one f16 among bf16
    assert _call_bwd(lib, a) == -3
    # the split algorithm is bf16 only: refused before any launch
    assert lib.fa_bwd_set_algorithm(0) == 0
    try:
        assert _call_bwd(lib, _f16_args()) == -8                         # FA_ERR_UNSUPPORTED
    finally:
        assert lib.fa_bwd_set_algorithm(2) == 0


def test_empty_problems_launch_nothing(lib):
    # Sq == 0 and B == 0 return FA_OK without any CUDA call (this machine has no GPU,
    # so reaching a launch would fail with FA_ERR_CUDA).
    assert _call_bwd(lib, _bwd_args(Sq=0)) == 0
    assert _call_bwd(lib, _bwd_args(B=0)) == 0


def test_workspace_size(lib):
    f = lib.fa_bwd_workspace_size
    f.restype = ctypes.c_size_t
    # header 256 + LSE2 + D (B*H*Sq_r fp32 each) + accumulator (B*H*Mb*128*Dp fp32) + counters
    B, H, Sq, D = 4, 32, 2048, 128
    rows = B * H * Sq
    want = 256 + rows * 4 + rows * 4 + B * H * 16 * 128 * 128 * 4 + B * H * 16 * 4
    assert f(B, H, 8, Sq, Sq, D, 0) == want
    assert f(1, 1, 1, 77, 99, 72, 1) >= 256 + 2 * 128 * 4 + 128 * 80 * 4


def test_fwd_validation_codes(lib):
    q = _view((1, 64, 2, 64)); k = _view((1, 64, 2, 64)); v = _view((1, 64, 2, 64))
    o = _view((1, 64, 2, 64)); l = _view((1, 2, 64), dtype=1)
    args = lambda **kw: [ctypes.byref(x) for x in (kw.get("q", q), kw.get("k", k), v, kw.get("o", o), l)]
    assert lib.fa_fwd(*args(o=_view((1, 64, 2, 32))), ctypes.c_float(0.1), 0, -1, -1, ctypes.c_float(0), None, 0, None) == -2
    assert lib.fa_fwd(*args(), ctypes.c_float(-1.0), 0, -1, -1, ctypes.c_float(0), None, 0, None) == -9
    q0 = _view((1, 0, 2, 64))
    o0 = _view((1, 0, 2, 64))
    l0 = _view((1, 2, 0), dtype=1)
    assert lib.fa_fwd(ctypes.byref(q0), ctypes.byref(k), ctypes.byref(v), ctypes.byref(o0), ctypes.byref(l0),
                      ctypes.c_float(0.1), 0, -1, -1, ctypes.c_float(0), None, 0, None) == 0


def _varlen_fwd(lib, q=None, lse=None, cu=4096, batch=2, mq=100, mk=100, **kw):
    tq, H, D = 300, 2, 64
    qv = q or _view((tq, H, D))
    kv = _view((250, H, D))
    out = _view((tq, H, D))
    lv = lse or _view((H, tq), dtype=1)
    return lib.fa_fwd_varlen(ctypes.byref(qv), ctypes.byref(kv), ctypes.byref(kv), ctypes.byref(out),
                             ctypes.byref(lv), cu, cu, None, None, batch, mq, mk, 0.125, 0, -1, -1, 0.0,
                             None, 0, None)


def test_varlen_validation(lib):
    assert _varlen_fwd(lib, q=_view((1, 300, 2, 64))) == -2            # q must be (total, H, D)
    assert _varlen_fwd(lib, lse=_view((1, 2, 300), dtype=1)) == -2     # lse must be (H, total)
    assert _varlen_fwd(lib, lse=_view((2, 299), dtype=1)) == -2        # lse rows != total_q
    assert _varlen_fwd(lib, batch=-1) == -9                            # negative batch
    assert _varlen_fwd(lib, mq=301) == -9                              # max_seqlen_q > total_q
    assert _varlen_fwd(lib, mk=-1) == -9
    assert _varlen_fwd(lib, batch=70000) == -8                         # above the grid limit
    assert _varlen_fwd(lib, cu=None) == -1                             # offsets missing
    assert _varlen_fwd(lib, batch=0) == 0                              # nothing to do, no launch
    assert _varlen_fwd(lib, mq=0) == 0
    # the backward: split algorithm refused for packed sequences, before any launch
    tq, tk, H, D = 300, 250, 2, 64
    a = [_view((tq, H, D)), _view((tq, H, D)), _view((tk, H, D)), _view((tk, H, D)),
         _view((tq, H, D)), _view((H, tq), dtype=1), _view((tq, H, D)), _view((tk, H, D)),
         _view((tk, H, D))]
    args = [ctypes.byref(x) for x in a]
    assert lib.fa_bwd_set_algorithm(0) == 0
    try:
        assert lib.fa_bwd_varlen(*args, 4096, 4096, None, None, 2, 100, 100, 0.125, 0, -1, -1, 0.0, 0,
                                 ctypes.c_void_p(4096), 1 << 30, None) == -8
    finally:
        assert lib.fa_bwd_set_algorithm(2) == 0
    assert lib.fa_bwd_varlen(*args, 4096, 4096, None, None, 0, 100, 100, 0.125, 0, -1, -1, 0.0, 0,
                             ctypes.c_void_p(4096), 1 << 30, None) == 0           # batch 0
    assert lib.fa_bwd_varlen(*args, 4096, 4096, None, None, 2, 100, 100, 0.125, 0, -1, -1, 0.0, 0,
                             ctypes.c_void_p(4096), 16, None) == -7               # workspace
    # workspace: per head total_q // 128 + batch slots of 128 rows
    f = lib.fa_bwd_varlen_workspace_size
    f.restype = ctypes.c_size_t
    T = 300 // 128 + 2
    rows = H * T * 128
    want = 256 + rows * 4 + rows * 4 + rows * 64 * 4 + ((H * T * 4 + 15) // 16) * 16
    want = (want + 255) // 256 * 256
    assert f(2, H, 300, 64, 0) == want


def test_blocksparse_validation(lib):
    a = _bwd_args()
    order = ("dout", "q", "k", "v", "out", "lse", "dq", "dk", "dv")
    ptrs = [ctypes.byref(a[n]) for n in order]
    # the block mask is required
    assert lib.fa_bwd_blocksparse(*ptrs, None, 0.125, 0, -1, -1, 0.0, 0, ctypes.c_void_p(4096),
                                  1 << 30, None) == -1
    fwd = [ctypes.byref(a[n]) for n in ("q", "k", "v", "out", "lse")]
    assert lib.fa_fwd_blocksparse(*fwd, None, 0.125, 0, -1, -1, 0.0, None, 0, None) == -1
    # split algorithm: refused before any launch
    assert lib.fa_bwd_set_algorithm(0) == 0
    try:
        assert lib.fa_bwd_blocksparse(*ptrs, 4096, 0.125, 0, -1, -1, 0.0, 0, ctypes.c_void_p(4096),
                                      1 << 30, None) == -8
    finally:
        assert lib.fa_bwd_set_algorithm(2) == 0
    # workspace: fa_bwd's plus per key tile a count and G * Mb list entries
    f = lib.fa_bwd_blocksparse_workspace_size
    f.restype = ctypes.c_size_t
    g = lib.fa_bwd_workspace_size
    g.restype = ctypes.c_size_t
    base = g(1, 2, 2, 128, 128, 64, 0)
    assert f(1, 2, 2, 128, 128, 64) == (((base + 2 * 4 + 255) // 256 * 256 + 2 * 1 * 1 * 4 + 255) // 256) * 256
    assert lib.fa_bwd_blocksparse(*ptrs, 4096, 0.125, 0, -1, -1, 0.0, 0, ctypes.c_void_p(4096),
                                  base, None) == -7        # fa_bwd's size is not enough


def test_binding_checks_used_lengths():
    """The binding accepts no used lengths, or a 1-D int32 device tensor of one entry per
    sequence, and refuses anything else before calling the library."""
    import torch
    from flashattention_backward_pass_gb300 import _abi
    assert _abi._used(None, 3) is None
    with pytest.raises(ValueError):
        _abi._used(torch.zeros(3, dtype=torch.int32), 3)       # host tensor
    with pytest.raises(ValueError):
        _abi._used(torch.zeros(3, dtype=torch.int64), 3)       # wrong type
    with pytest.raises(ValueError):
        _abi._used(torch.zeros((3, 1), dtype=torch.int32), 3)  # not 1-D


def _prototype(name):
    """The parameter list of `name` in include/fa.h, whitespace-normalised."""
    import re
    from flashattention_backward_pass_gb300._abi import HEADER_PATH
    text = re.sub(r"/\*.*?\*/", "", open(HEADER_PATH).read(), flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, name
    return " ".join(m.group(1).split())


def test_boundary_signatures_match_the_scope_table():
    """The calls the hot path's boundary lists, with their argument lists as given there:
    fa_fwd / fa_bwd take (tensors..., scalars..., workspace, workspace_bytes, stream),
    fa_bwd_workspace_size the problem sizes, fa_bwd_status (workspace, stream, status)."""
    assert _prototype("fa_bwd_status") == "void* workspace, void* stream, int* device_status"
    assert _prototype("fa_bwd_workspace_size") == (
        "int B, int H, int Hk, int Sq, int Sk, int D, int deterministic")
    assert _prototype("fa_fwd") == (
        "const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, fa_tensor* out, "
        "fa_tensor* lse, float softmax_scale, int causal, int window_left, int window_right, "
        "float softcap, void* workspace, size_t workspace_bytes, void* stream")
    assert _prototype("fa_bwd") == (
        "const fa_tensor* dout, const fa_tensor* q, const fa_tensor* k, const fa_tensor* v, "
        "const fa_tensor* out, const fa_tensor* lse, fa_tensor* dq, fa_tensor* dk, fa_tensor* dv, "
        "float softmax_scale, int causal, int window_left, int window_right, float softcap, "
        "int deterministic, void* workspace, size_t workspace_bytes, void* stream")
    assert _prototype("fa_status_string") == "int status"


def test_status_readers_reject_null_pointers(lib):
    # argument checks come before any CUDA call (there is no GPU here)
    out = ctypes.c_int(7)
    assert lib.fa_bwd_status(None, None, ctypes.byref(out)) == -1
    assert lib.fa_bwd_status(ctypes.c_void_p(4096), None, None) == -1
    assert lib.fa_bwd_noalloc_status(None, None) == -1
    assert out.value == 7



def _dv_args(D=192, Dv=128, B=1, Sq=128, Sk=128, H=2, Hk=2):
    """fa_bwd arguments with v, O, dO and dV of head dim Dv and q, k, dQ, dK of D."""
    return _bwd_args(B=B, Sq=Sq, Sk=Sk, H=H, Hk=Hk, D=D,
                     dout=_view((B, Sq, H, Dv)), v=_view((B, Sk, Hk, Dv)), out=_view((B, Sq, H, Dv)),
                     dv=_view((B, Sk, Hk, Dv)))


def test_own_v_head_dim_validation(lib):
    """A V head dim of its own (the sm90 page's head_dim_v): O, dO and dV follow v; every
    dim a multiple of 8 and at most 256; the wide kernels take no packed sequences and no
    block mask (refused before any launch)."""
    assert _call_bwd(lib, _dv_args(Sq=0)) == 0                           # valid, empty
    assert _call_bwd(lib, _dv_args(D=256, Dv=256, Sq=0)) == 0
    assert _call_bwd(lib, _dv_args(Dv=60)) == -4                         # Dv % 8
    assert _call_bwd(lib, _dv_args(Dv=264)) == -4                        # Dv > 256
    a = _dv_args(); a["dv"] = _view((1, 128, 2, 192))
    assert _call_bwd(lib, a) == -2                                       # dV must have Dv
    a = _dv_args(); a["out"] = _view((1, 128, 2, 192))
    assert _call_bwd(lib, a) == -2                                       # O must have Dv
    a = _dv_args(); a["dq"] = _view((1, 128, 2, 128))
    assert _call_bwd(lib, a) == -2                                       # dQ must have D
    order = ("dout", "q", "k", "v", "out", "lse", "dq", "dk", "dv")
    a = _dv_args()
    ptrs = [ctypes.byref(a[n]) for n in order]
    assert lib.fa_bwd_blocksparse(*ptrs, 4096, 0.125, 0, -1, -1, 0.0, 0, ctypes.c_void_p(4096),
                                  1 << 30, None) == -8
    fwd = [ctypes.byref(a[n]) for n in ("q", "k", "v", "out", "lse")]
    assert lib.fa_fwd_blocksparse(*fwd, 4096, 0.125, 0, -1, -1, 0.0, None, 0, None) == -8
    tq, tk, H = 300, 250, 2
    v3 = [_view((tq, H, 192)), _view((tk, H, 192)), _view((tk, H, 128)), _view((tq, H, 128)),
          _view((H, tq), dtype=1)]
    assert lib.fa_fwd_varlen(*[ctypes.byref(x) for x in v3], 4096, 4096, None, None, 2, 100, 100,
                             0.125, 0, -1, -1, 0.0, None, 0, None) == -8


def test_wide_workspace_size(lib):
    """Wide head dims: LSE2 and D as before, a dQ accumulator of (B, H, ceil(Sq/64),
    ceil(pad64(D)/128)) blocks of 128 x 64 fp32 and one ordering counter per block; v's
    head dim does not change it."""
    f = lib.fa_bwd_workspace_size_dv
    f.restype = ctypes.c_size_t
    B, H, Sq = 2, 3, 200
    Sq_r = 256
    rows = B * H * Sq_r
    lse2_end = (256 + rows * 4 + 255) // 256 * 256
    dsum_end = (lse2_end + rows * 4 + 255) // 256 * 256
    for D, nks in ((192, 2), (256, 2), (128, 1), (72, 1)):
        blocks = B * H * 4 * nks
        want = dsum_end + blocks * 32768 + (blocks * 4 + 15) // 16 * 16   # + ordering counters
        want = (want + 255) // 256 * 256
        assert f(B, H, 1, Sq, 77, D, 64 if D != 64 else 128, 0) == want, D
    g = lib.fa_bwd_workspace_size
    g.restype = ctypes.c_size_t
    assert g(B, H, 1, Sq, 77, 256, 0) == f(B, H, 1, Sq, 77, 256, 256, 0)
    assert g(B, H, 1, Sq, 77, 128, 0) == f(B, H, 1, Sq, 77, 128, 128, 0)


def test_algorithm_selection(lib):
    """AUTO (2) is the default; 0, 1 and 2 are accepted, anything else is FA_ERR_ARG."""
    assert lib.fa_bwd_get_algorithm() == 2
    try:
        for a in (0, 1, 2):
            assert lib.fa_bwd_set_algorithm(a) == 0
            assert lib.fa_bwd_get_algorithm() == a
        assert lib.fa_bwd_set_algorithm(3) == -9
        assert lib.fa_bwd_set_algorithm(-1) == -9
    finally:
        lib.fa_bwd_set_algorithm(2)
