"""Host-side checks of the C-ABI (no GPU needed): libittt.so builds and loads,
exports every entry point include/ittt.h declares, and rejects bad
arguments with the documented status before touching any memory."""
import ctypes
import math
import os

import pytest
import torch

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
    # The descriptors hold fake device addresses: a call that passed
    # validation on a machine with a GPU would launch kernels on them.
    if torch.cuda.is_available():
        pytest.skip("argument checks with fake device pointers run on hosts without a GPU")
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


def _fp32_args(**kw):
    a = _args(**kw)
    for k in ("H", "X0", "Wg", "Wu", "Wt"):
        a[k].dtype = ittt.FP32
    # fp32 tensors are twice as large: spread the fake addresses apart again
    for j, k in enumerate(("H", "X0", "Wg", "Wu", "W0", "Wt", "cw", "out")):
        a[k].data = FAKE * (j + 1) * 4096
    return a


def test_fp32_inputs_validation(lib):
    """fp32 inputs: H's dtype selects the mode, and then all five of H, X0,
    W_gate, W_up and W_target must be fp32; the flag with a bf16 H and the
    fused convolution are refused before any work."""
    for k, name in (("X0", "X0"), ("Wg", "W_gate"), ("Wu", "W_up"), ("Wt", "W_target")):
        a = _fp32_args()
        a[k].dtype = ittt.BF16
        assert _call(lib, a) == ittt.ERR_INVALID_ARG, k
        assert name in ittt.last_error()
    a = _args()
    a["H"].dtype = ittt.FP32                  # H alone fp32: X0 is the first mismatch
    assert _call(lib, a) == ittt.ERR_INVALID_ARG and "X0" in ittt.last_error()
    o = ittt.Opts()
    o.flags = ittt.FLAG_FP32_INPUTS            # flag set, H bf16
    assert _call(lib, _args(), opts=o) == ittt.ERR_INVALID_ARG
    assert "FP32_INPUTS" in ittt.last_error()
    o = ittt.Opts()
    o.flags = ittt.FLAG_FUSED_CONV
    assert _call(lib, _fp32_args(), opts=o) == ittt.ERR_UNSUPPORTED
    assert "split convolution" in ittt.last_error()
    assert ittt.workspace_bytes_ex(1, 256, 64, 256, 64, fused_conv=True, fp32_inputs=True) == 0


def test_rejects_bad_sizes(lib):
    assert _call(lib, _args(), chunk=0) == ittt.ERR_INVALID_ARG
    assert "positive" in ittt.last_error()
    # empty inputs (no sequence, no token) are argument errors, before any work
    for B, T in ((0, 256), (1, 0), (0, 0)):
        assert _call(lib, _args(B=B, T=T)) == ittt.ERR_INVALID_ARG, (B, T)
        assert "positive" in ittt.last_error()
        assert ittt.workspace_bytes(B, T, 64, 256, 64) == 0
    assert _call(lib, _args(), chunk=-64) == ittt.ERR_INVALID_ARG
    assert _call(lib, _args(d=60), chunk=64) == ittt.ERR_UNSUPPORTED
    assert _call(lib, _args(f=100), chunk=64) == ittt.ERR_UNSUPPORTED
    assert _call(lib, _args(), eta=math.nan) == ittt.ERR_INVALID_ARG
    assert _call(lib, _args(), eta=math.inf) == ittt.ERR_INVALID_ARG


def test_any_chunk_and_length_plan():
    """Chunks and lengths that are not multiples of 64 are planned (no call
    with fake pointers gets past validation here: only the planner runs)."""
    for T, C in ((256, 100), (96, 32), (200, 64), (257, 1), (5, 7)):
        assert ittt.workspace_bytes(1, T, 64, 256, C) > 0, (T, C)
    # narrower limits of the two options
    assert ittt.workspace_bytes_ex(1, 256, 64, 256, 100, fused_conv=True) == 0
    assert ittt.workspace_bytes_ex(1, 200, 64, 256, 64, fused_conv=True) == 0
    assert ittt.workspace_bytes_ex(1, 320, 64, 256, 128, dual=True) == 0
    assert ittt.workspace_bytes_ex(1, 256, 64, 256, 128, dual=True) > 0


def test_rejects_bad_options(lib):
    a = _args()
    o = ittt.Opts()
    o.pad_mode = 7
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    o = ittt.Opts()
    o.flags = 256
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
    o.flags = ittt.FLAG_FUSED_CONV
    assert _call(lib, _args(), chunk=100, opts=o) == ittt.ERR_UNSUPPORTED
    o = ittt.Opts()
    o.flags = ittt.FLAG_L2_NORM | ittt.FLAG_DUAL
    assert _call(lib, a, opts=o) == ittt.ERR_UNSUPPORTED
    assert "dual" in ittt.last_error()
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
    tk = 768   # the apply's counters: its unit counter (4 slots) and 152 tail counters
    want = tk + r(B * T * f * 2) + 2 * r(B * T * d * 2) + r(B * n * d * f * 2)
    assert ittt.workspace_bytes(B, T, d, f, C) == want
    assert ittt.workspace_bytes_ex(B, T, d, f, C) == want
    want3 = tk + r(B * T * f * 2) + 2 * r(B * T * d * 2) + r(B * 3 * d * f * 2)  # 1024 = 2*384+256
    assert ittt.workspace_bytes(B, T, d, f, 384) == want3
    assert ittt.workspace_bytes(B, T, d, f, 0) == 0
    assert ittt.workspace_bytes(B, T, 60, f, C) == 0
    # caller buffers and the fused convolution take parts out of the scratch
    assert ittt.workspace_bytes_ex(B, T, d, f, C, fused_conv=True) == want - r(B * T * d * 2)
    fake_z = torch.empty(0)
    assert (ittt.workspace_bytes_ex(B, T, d, f, C, z_buf=fake_z) == want - r(B * T * f * 2))
    # the dual form: scores [B,T,T] bf16, no snapshots (W_0 dtype unknown:
    # a bf16 copy of it is planned)
    want_dual = r(B * T * f * 2) + 2 * r(B * T * d * 2) + r(B * T * T * 2) + r(d * f * 2)
    assert ittt.workspace_bytes_ex(B, T, d, f, C, dual=True) == want_dual
    # packed documents 300 + 724 tokens: ceil(300/256) + ceil(724/256) = 2 + 3
    # slots, and a table of starts and slot bases 2*(2+1), the slot-to-
    # document map 5, the 128- and 256-row tile bases 2*(5+1) and the
    # updating documents 2 ints
    cu = [0, 300, 1024]
    want_packed = (tk + r(T * f * 2) + 2 * r(T * d * 2) + r(5 * d * f * 2)
                   + r((6 + 5 + 12 + 2) * 4))
    assert ittt.workspace_bytes_ex(1, T, d, f, C, cu_seqlens=cu) == want_packed
    # the normalised walk keeps an fp32 state and row partial sums per
    # 256-column block (for the walk with the state in HBM), and, for a
    # regular batch, the row sums and arrival counters of the walk with the
    # state in TMEM (groups of ceil(f/256) CTA pairs, up to 128 pairs)
    nblk = -(-f // 256)
    tiles = -(-d // 128) * -(-f // 32)      # the fp32 state in 128 x 32 tiles
    groups = max(1, 128 // nblk)
    walk = r(2 * groups * 2 * nblk * 256 * 4) + r(2 * 128 * 4)
    assert (ittt.workspace_bytes_ex(B, T, d, f, C, l2norm=True)
            == want + r(B * tiles * 128 * 32 * 4) + r(2 * B * 2 * nblk * d * 4) + walk)
    assert ittt.workspace_bytes_ex(B, T, d, f, C, l2norm=True, dual=True) == 0
    # fp32 inputs: the split copies [A_hi | A_hi | A_lo] of Xc and H
    # (M x 3d each, Xc's in place of the bf16 Xc), [W_hi | W_lo | W_hi] of
    # W_gate and W_up (f x 3d each) and of W_target (d x 3d)
    M = B * T
    want_fp32 = (want - r(M * d * 2) + 2 * r(M * 3 * d * 2)
                 + 2 * r(f * 3 * d * 2) + r(d * 3 * d * 2))
    assert ittt.workspace_bytes_ex(B, T, d, f, C, fp32_inputs=True, primal=True) == want_fp32
    assert (ittt.workspace_bytes_ex(B, T, d, f, C, fp32_inputs=True, reuse_zv=True,
                                    z_buf=fake_z, vhat_buf=fake_z)
            == ittt.workspace_bytes_ex(B, T, d, f, C, reuse_zv=True, z_buf=fake_z,
                                       vhat_buf=fake_z))
    # the apply's split last round: fp32 partials for up to 76 pieces of
    # 256 x 256 tiles, planned when the apply has at least two rounds of
    # units on 76 CTA pairs: 8 sequences x 4 chunks of 256 rows x 5 column
    # tiles (d 1280) = 160 units; half the sequences, 80 units: none
    def plain(Bq, Tq, dq, fq, Cq):
        return (tk + r(Bq * Tq * fq * 2) + 2 * r(Bq * Tq * dq * 2)
                + r(Bq * (Tq // Cq) * dq * fq * 2))
    assert (ittt.workspace_bytes(8, 1024, 1280, 512, 256)
            == plain(8, 1024, 1280, 512, 256) + r(76 * 2 * 128 * 256 * 4))
    assert ittt.workspace_bytes(4, 1024, 1280, 512, 256) == plain(4, 1024, 1280, 512, 256)
    assert ittt.launch_count(B, T, d, f, C) == 5
    assert ittt.launch_count(B, T, d, f, T) == 4
    assert ittt.launch_count(B, 1000, d, f, 512) == 5   # two chunks, the last partial
    assert ittt.launch_count(B, T, d, f, 0) == 0


def _packed_opts(cu, **kw):
    o = ittt.Opts()
    arr = (ctypes.c_int64 * len(cu))(*cu)
    o.cu_seqlens = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64))
    o.num_docs = len(cu) - 1
    for k, v in kw.items():
        setattr(o, k, v)
    return o, arr


@pytest.mark.parametrize("cu,msg", [
    ([1, 100, 256], "cu_seqlens[0]"),
    ([0, 100, 250], "cu_seqlens[num_docs]"),
    ([0, 100, 100, 256], "strictly"),
    ([0, 150, 100, 256], "strictly"),
    ([0], "num_docs"),
])
def test_rejects_bad_document_offsets(lib, cu, msg):
    o, _arr = _packed_opts(cu)
    assert _call(lib, _args(), opts=o) == ittt.ERR_INVALID_ARG
    assert msg in ittt.last_error()


def test_rejects_bad_packed_options(lib):
    o, _arr = _packed_opts([0, 100, 256])
    assert _call(lib, _args(B=2), opts=o) == ittt.ERR_INVALID_ARG      # packed needs B = 1
    assert "B = 1" in ittt.last_error()
    for flag in (ittt.FLAG_FUSED_CONV, ittt.FLAG_DUAL):
        o, _arr = _packed_opts([0, 128, 256], flags=flag)
        assert _call(lib, _args(), opts=o) == ittt.ERR_UNSUPPORTED
    o = ittt.Opts()
    o.num_docs = 2                                                     # count without offsets
    assert _call(lib, _args(), opts=o) == ittt.ERR_INVALID_ARG
    # per-document states are [num_docs, d, f]; snapshots [1, slots, d, f]
    st = _desc([1, 64, 256], ittt.FP32, data=FAKE * 9 * 1024)
    o, _arr = _packed_opts([0, 100, 256], state_out=ctypes.pointer(st))
    assert _call(lib, _args(), opts=o) == ittt.ERR_INVALID_ARG
    assert "state_out" in ittt.last_error()
    sb = _desc([1, 4, 64, 256], ittt.BF16, data=FAKE * 9 * 1024)       # 2 + 3 slots at C=64
    o, _arr = _packed_opts([0, 100, 256], snap_buf=ctypes.pointer(sb))
    assert _call(lib, _args(), opts=o) == ittt.ERR_INVALID_ARG
    assert "snap_buf" in ittt.last_error()


def test_python_binding_has_no_compute_fallback():
    """The binding only marshals arguments: it never imports the oracle and
    has no torch math on the layer's tensors."""
    import inspect
    src = inspect.getsource(ittt)
    assert "oracle" not in src.replace("no fallback", "")
    for op in ("torch.matmul", "F.linear", "silu", "conv1d", "einsum", "@"):
        assert op not in src


def test_update_only_and_reuse_options(lib):
    a = _args()
    st = _desc([1, 64, 256], ittt.FP32, data=FAKE * 9 * 1024)
    sb = _desc([1, 4, 64, 256], ittt.BF16, data=FAKE * 10 * 1024)
    o = ittt.Opts()
    o.flags = ittt.FLAG_UPDATE_ONLY                                     # nowhere to put the state
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "state_out" in ittt.last_error()
    o.state_out = ctypes.pointer(st)
    o.snap_buf = ctypes.pointer(sb)                                     # no snapshots are formed
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "snap_buf" in ittt.last_error()
    for extra in (ittt.FLAG_DUAL, ittt.FLAG_L2_NORM):
        o = ittt.Opts()
        o.flags = ittt.FLAG_UPDATE_ONLY | extra
        o.state_out = ctypes.pointer(st)
        assert _call(lib, a, opts=o) == ittt.ERR_UNSUPPORTED
    o = ittt.Opts()
    o.flags = ittt.FLAG_REUSE_ZV                                        # nothing to reuse
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "z_buf" in ittt.last_error()


def test_update_only_and_reuse_scratch():
    def r(x):
        return (x + 255) // 256 * 256
    B, T, d, f, C = 2, 1024, 320, 1000, 256
    n = T // C
    z, vh, xc, snap = r(B * T * f * 2), r(B * T * d * 2), r(B * T * d * 2), r(B * n * d * f * 2)
    tk = 768   # the apply's counters (none when the call applies nothing)
    fake = torch.empty(0)
    # folding chunks only forms no snapshots
    assert (ittt.workspace_bytes_ex(B, T, d, f, C, update_only=True, state_out=fake)
            == z + vh + xc)
    assert ittt.workspace_bytes_ex(B, T, d, f, C, update_only=True) == 0   # needs state_out
    # reusing Z and eta*Vhat needs neither the producers' scratch nor Xc
    assert (ittt.workspace_bytes_ex(B, T, d, f, C, reuse_zv=True, z_buf=fake, vhat_buf=fake)
            == tk + snap)
    assert ittt.workspace_bytes_ex(B, T, d, f, C, reuse_zv=True, z_buf=fake) == 0
    assert ittt.workspace_bytes_ex(B, T, d, f, C, update_only=True, reuse_zv=True,
                                   state_out=fake, z_buf=fake, vhat_buf=fake) == 0


def _prefix_call(lib, W_start, deltas, count, state):
    if torch.cuda.is_available():
        pytest.skip("argument checks with fake device pointers run on hosts without a GPU")
    r = lambda x: None if x is None else ctypes.byref(x)  # noqa: E731
    return lib.ittt_state_prefix(r(W_start), r(deltas), ctypes.c_int32(count), r(state), None)


def test_state_prefix_rejects_bad_arguments(lib):
    R, S, d, f = 3, 2, 64, 256
    dl = _desc([R, S, d, f], ittt.FP32, data=FAKE)
    st = _desc([S, d, f], ittt.FP32, data=FAKE * 1024)
    w0 = _desc([d, f], ittt.BF16, data=FAKE * 2048)
    assert _prefix_call(lib, w0, _desc([S, d, f], ittt.FP32), 1, st) == ittt.ERR_INVALID_ARG
    assert _prefix_call(lib, w0, dl, R + 1, st) == ittt.ERR_INVALID_ARG
    assert "count" in ittt.last_error()
    assert _prefix_call(lib, w0, dl, -1, st) == ittt.ERR_INVALID_ARG
    assert _prefix_call(lib, w0, dl, 1, _desc([S, d, f], ittt.BF16, data=FAKE * 1024)) \
        == ittt.ERR_INVALID_ARG
    assert _prefix_call(lib, _desc([d, f + 8], ittt.BF16, data=FAKE * 2048), dl, 1, st) \
        == ittt.ERR_INVALID_ARG
    assert _prefix_call(lib, _desc([S, d, f], ittt.BF16, data=FAKE * 2048), dl, 1, st) \
        == ittt.ERR_INVALID_ARG                                         # per-state starts are fp32
    assert _prefix_call(lib, w0, dl, 1, _desc([S, d, f], ittt.FP32, data=FAKE + 4096)) \
        == ittt.ERR_INVALID_ARG                                         # state inside the deltas
    assert "overlaps" in ittt.last_error()
    odd = _desc([R, S, 60, f], ittt.FP32, data=FAKE)
    assert _prefix_call(lib, None, odd, 1, _desc([S, 60, f], ittt.FP32, data=FAKE * 1024)) \
        == ittt.ERR_UNSUPPORTED


def test_scratch_limit_fails_before_any_work(lib):
    """Over the scratch cap a call returns ITTT_ERR_OOM before it touches the
    device (fake pointers: nothing may run); a caller workspace is exempt."""
    a = _args()
    need = ittt.workspace_bytes(1, 256, 64, 256, 64)
    try:
        ittt.set_scratch_limit(need - 1)
        assert _call(lib, a) == ittt.ERR_OOM
        assert "limit" in ittt.last_error()
        o = ittt.Opts()
        o.workspace = FAKE * 64
        o.workspace_bytes = need
        assert _call(lib, a, opts=o) != ittt.ERR_OOM      # no allocation: past the cap check
    finally:
        ittt.set_scratch_limit(0)


def test_wait_check_rejects_limits_out_of_range(lib):
    """ittt_check_wait_timeout validates its limit before it enqueues anything
    (no device needed for these)."""
    for bad in (0, 999, 10**9 + 1):
        assert lib.ittt_check_wait_timeout(ctypes.c_uint64(bad), None) == ittt.ERR_INVALID_ARG
        assert "limit_ns" in ittt.last_error()


C_PROGRAM = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_abi", "forward_from_c.c")


def build_c_program(out_path):
    """gcc, C99, against include/ittt.h, libittt.so and the CUDA runtime."""
    import subprocess
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(build.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-o", out_path, C_PROGRAM,
           "-I", build.INCLUDE, "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-Wl,-rpath," + libdir, "-l:" + os.path.basename(build.LIB_PATH),
           "-L", os.path.join(cuda, "lib64"), "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-lcudart"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out_path


def test_header_and_a_c_caller_build_as_c99(lib, tmp_path):
    """The boundary is plain C: a C99 program using only ittt.h and the CUDA
    runtime compiles (-Wall -Werror) and links against libittt.so."""
    exe = build_c_program(str(tmp_path / "forward_from_c"))
    assert os.path.exists(exe)


def test_state_in_place_only_as_exact_alias(lib):
    a = _args()
    st = _desc([1, 64, 256], ittt.FP32, data=FAKE * 9 * 1024)
    part = _desc([1, 64, 256], ittt.FP32, data=FAKE * 9 * 1024 + 4096)   # overlaps, not equal
    o = ittt.Opts()
    o.state_in = ctypes.pointer(st)
    o.state_out = ctypes.pointer(part)
    assert _call(lib, a, opts=o) == ittt.ERR_INVALID_ARG
    assert "overlaps" in ittt.last_error()
    o.state_out = ctypes.pointer(st)                                   # the same buffer
    assert _call(lib, a, opts=o) != ittt.ERR_INVALID_ARG               # past validation


def test_form_choice_by_sequence_length():
    """The dual form for short sequences (T < 2.5 d f / (d + f)) where it is
    allowed, the primal walk otherwise; DUAL / PRIMAL force one."""
    P, D = ittt.FORM_PRIMAL, ittt.FORM_DUAL
    cases = [
        ((8, 2048, 2560, 9728, 512), D),      # 2048 < 5068
        ((64, 256, 2560, 9728, 64), D),
        ((4, 4096, 2560, 9728, 1024), D),     # 4096 < 5068
        ((2, 8192, 2560, 9728, 2048), P),     # 8192 > 5068
        ((2, 32768, 2560, 9728, 2048), P),    # the bench workload
        ((4, 4096, 4096, 14336, 1024), D),    # 4096 < 7964
        ((2, 8192, 4096, 14336, 1024), P),    # 8192 > 7964
        ((8, 1024, 1024, 3072, 256), D),      # 1024 < 1920
        ((4, 2048, 1024, 3072, 512), P),      # 2048 > 1920
        ((1, 256, 64, 256, 64), P),           # 256 > 128
        ((8, 2048, 2560, 9728, 2048), P),     # one chunk: nothing to update
        ((8, 2000, 2560, 9728, 500), P),      # chunk not a multiple of 64
        ((8, 2048, 2560, 9728, 768), P),      # chunk does not divide T
    ]
    for args, want in cases:
        assert ittt.plan_form(*args) == want, args
        assert ittt.plan_form(*args, primal=True) == P
        assert ittt.plan_form(*args, dual=True, primal=True) == -1
    short = (8, 2048, 2560, 9728, 512)
    fake = torch.empty(0)
    for kw in ({"state_out": fake}, {"snap_buf": fake}, {"l2norm": True}, {"fused_conv": True},
               {"cu_seqlens": [0, 8192, 16384]}):
        if "cu_seqlens" in kw:
            assert ittt.plan_form(1, 16384, 2560, 9728, 512, **kw) == P
        else:
            assert ittt.plan_form(*short, **kw) == P, kw
    # the plan's scratch is the dual form's: no snapshots, the scores instead
    assert ittt.workspace_bytes(*short) == ittt.workspace_bytes_ex(*short, dual=True)
    assert ittt.workspace_bytes(*short) != ittt.workspace_bytes_ex(*short, primal=True)
