"""Host-side checks of the C-ABI (no GPU needed): libittt.so builds and loads,
exports every entry point include/ittt.h declares, and rejects bad
arguments with the documented status before touching any memory."""
import ctypes
import math

import pytest

from chunk_wise_weight_gb300 import build, ittt


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ittt.load()


def test_exports_every_declared_entry_point(lib):
    names = ittt.header_functions()
    assert set(names) >= {"ittt_forward", "ittt_forward_ex", "ittt_workspace_bytes",
                          "ittt_stream_status", "ittt_last_error", "ittt_version",
                          "ittt_launch_count"}
    for name in names:
        assert hasattr(lib, name), f"{name} is declared in ittt.h but not exported"


def test_only_c_abi_symbols_are_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(ittt.header_functions())


def test_version(lib):
    assert ittt.version() == 100


# A fake, never-dereferenced device address: validation fails before any use.
FAKE = 1 << 20


def _desc(shape, dtype=ittt.BF16, data=FAKE, strides=None):
    d = ittt.Tensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    st = strides
    if st is None:
        st, acc = [], 1
        for s in reversed(shape):
            st.insert(0, acc)
            acc *= s
    for k, s in enumerate(shape):
        d.shape[k] = s
        d.stride[k] = st[k]
    return d


def _args(B=1, T=256, d=64, f=256, out_dtype=ittt.BF16):
    base = [FAKE * (k + 1) * 1024 for k in range(8)]  # disjoint, aligned
    return dict(
        H=_desc([B, T, d], data=base[0]), X0=_desc([B, T, d], data=base[1]),
        Wg=_desc([f, d], data=base[2]), Wu=_desc([f, d], data=base[3]),
        W0=_desc([d, f], data=base[4]), Wt=_desc([d, d], data=base[5]),
        cw=_desc([d, 3], ittt.FP32, data=base[6]),
        out=_desc([B, T, d], out_dtype, data=base[7]))


def _call(lib, a, eta=0.1, chunk=64, opts=None):
    r = lambda x: None if x is None else ctypes.byref(x)  # noqa: E731
    return lib.ittt_forward_ex(r(a["H"]), r(a["X0"]), r(a["Wg"]), r(a["Wu"]), r(a["W0"]),
                               r(a["Wt"]), r(a["cw"]), ctypes.c_float(eta), ctypes.c_int64(chunk),
                               r(a["out"]), None, None if opts is None else ctypes.byref(opts))


@pytest.mark.parametrize("mutate,status,msg", [
    (lambda a: a.update(H=None), ittt.ERR_INVALID_ARG, "H"),
    (lambda a: a.update(X0=_desc([1, 255, 64])), ittt.ERR_INVALID_ARG, "X0"),
    (lambda a: a.update(Wg=_desc([256, 64], ittt.FP32)), ittt.ERR_INVALID_ARG, "W_gate"),
    (lambda a: a.update(Wt=_desc([64, 64], data=FAKE + 8)), ittt.ERR_INVALID_ARG, "aligned"),
    (lambda a: a.update(Wu=_desc([256, 64], strides=[1, 256])), ittt.ERR_INVALID_ARG, "dense"),
    (lambda a: a.update(cw=_desc([64, 3], ittt.BF16)), ittt.ERR_INVALID_ARG, "conv_w"),
    (lambda a: a.update(W0=None), ittt.ERR_INVALID_ARG, "W_down0"),
    (lambda a: a.update(out=_desc([1, 256, 64], data=a["H"].data)), ittt.ERR_INVALID_ARG,
     "overlaps"),
])
def test_rejects_bad_descriptors(lib, mutate, status, msg):
    a = _args()
    mutate(a)
    assert _call(lib, a) == status
    assert msg in ittt.last_error()


def test_rejects_bad_sizes(lib):
    assert _call(lib, _args(), chunk=0) == ittt.ERR_INVALID_ARG
    assert "positive" in ittt.last_error()
    assert _call(lib, _args(), chunk=100) == ittt.ERR_UNSUPPORTED   # not a multiple of 64
    assert "multiples of 64" in ittt.last_error()
    assert _call(lib, _args(T=96), chunk=32) == ittt.ERR_UNSUPPORTED
    assert _call(lib, _args(T=200), chunk=64) == ittt.ERR_UNSUPPORTED  # T not a multiple of 64
    assert _call(lib, _args(d=60), chunk=64) == ittt.ERR_UNSUPPORTED
    assert _call(lib, _args(f=100), chunk=64) == ittt.ERR_UNSUPPORTED
    assert _call(lib, _args(), eta=math.nan) == ittt.ERR_INVALID_ARG
    assert _call(lib, _args(), eta=math.inf) == ittt.ERR_INVALID_ARG


def test_rejects_bad_options(lib):
    a = _args()
    o = ittt.Opts()
    o.pad_mode = 7
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    o = ittt.Opts()
    o.flags = 4
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "flags" in ittt.last_error()
    o = ittt.Opts()
    o.flags = ittt.FLAG_DUAL
    st = _desc([1, 64, 256], ittt.FP32, data=FAKE * 9 * 1024)
    o.state_out = ctypes.pointer(st)
    assert _call(lib, a, opts=o) == ittt.ERR_UNSUPPORTED
    assert "dual" in ittt.last_error()
    o = ittt.Opts()
    bad = _desc([1, 64, 256], ittt.BF16, data=FAKE * 9 * 1024)   # state_out wrong dtype/shape
    o.state_out = ctypes.pointer(bad)
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "state_out" in ittt.last_error()
    o = ittt.Opts()
    o.flags = ittt.FLAG_DUAL
    assert _call(lib, _args(T=320), chunk=128, opts=o) == ittt.ERR_UNSUPPORTED  # partial chunk
    o = ittt.Opts()
    et = _desc([1, 256], ittt.BF16, data=FAKE * 9 * 1024)           # eta_tok must be fp32
    o.eta_tok = ctypes.pointer(et)
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "eta_tok" in ittt.last_error()
    o = ittt.Opts()
    zb = _desc([1, 256, 256], ittt.BF16, data=a["X0"].data)      # z_buf aliases X0
    o.z_buf = ctypes.pointer(zb)
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG


def test_workspace_bytes_and_launch_count(lib):
    def r(x):
        return (x + 255) // 256 * 256
    B, T, d, f, C = 2, 1024, 320, 1000, 256
    n = T // C
    want = r(B * T * f * 2) + 2 * r(B * T * d * 2) + r(B * n * d * f * 2)
    assert ittt.workspace_bytes(B, T, d, f, C) == want
    want3 = r(B * T * f * 2) + 2 * r(B * T * d * 2) + r(B * 3 * d * f * 2)   # 1024 = 2*384+256
    assert ittt.workspace_bytes(B, T, d, f, 384) == want3
    assert ittt.workspace_bytes(B, T, d, f, 100) == 0
    assert ittt.launch_count(B, T, d, f, C) == 6
    assert ittt.launch_count(B, T, d, f, T) == 5
    assert ittt.launch_count(B, T, d, f, 100) == 0


def test_python_binding_has_no_compute_fallback():
    """The binding only marshals arguments: it never imports the oracle and
    has no torch math on the layer's tensors."""
    import inspect
    src = inspect.getsource(ittt)
    assert "oracle" not in src.replace("no fallback", "")
    for op in ("torch.matmul", "F.linear", "silu", "conv1d", "einsum", "@"):
        assert op not in src
