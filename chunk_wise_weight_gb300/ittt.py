"""ctypes binding of libittt.so -- argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module turns
torch tensors into ``ittt_tensor`` descriptors (device pointer, dtype, shape,
strides), passes the current CUDA stream, and raises :class:`IttError` when
the library returns a non-OK status.  torch only provides device memory and
streams.  There is no fallback: if libittt.so is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "ITTT_OK", 1: "ITTT_ERR_INVALID_ARG", 2: "ITTT_ERR_UNSUPPORTED",
                3: "ITTT_ERR_CUDA", 4: "ITTT_ERR_OOM", 5: "ITTT_ERR_TIMEOUT"}
BF16, FP32 = 0, 1
PAD_CHUNK, PAD_SEQUENCE = 0, 1
PHASES = ("conv", "target", "gateup", "snapshot0", "update", "apply")
FLAG_FUSED_CONV = 1
FLAG_DUAL = 2
FLAG_L2_NORM = 4
FLAG_SINGLE_CTA = 8
FLAG_UPDATE_ONLY = 16
FLAG_REUSE_ZV = 32
FLAG_PRIMAL = 64
FLAG_FP32_INPUTS = 128
FORM_PRIMAL, FORM_DUAL = 0, 1

_DTYPES = {torch.bfloat16: BF16, torch.float32: FP32}


class IttError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class Opts(ctypes.Structure):
    _fields_ = [("pad_mode", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("state_in", ctypes.POINTER(Tensor)), ("state_out", ctypes.POINTER(Tensor)),
                ("z_buf", ctypes.POINTER(Tensor)), ("vhat_buf", ctypes.POINTER(Tensor)),
                ("snap_buf", ctypes.POINTER(Tensor)), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("events", ctypes.POINTER(ctypes.c_void_p)),
                ("eta_tok", ctypes.POINTER(Tensor)), ("cu_seqlens", ctypes.POINTER(ctypes.c_int64)),
                ("num_docs", ctypes.c_int64)]


_TP = ctypes.POINTER(Tensor)
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libittt.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "or `python -m chunk_wise_weight_gb300.build`")
    lib = ctypes.CDLL(path)
    fwd_args = [_TP, _TP, _TP, _TP, _TP, _TP, _TP, ctypes.c_float, ctypes.c_int64, _TP,
                ctypes.c_void_p]
    lib.ittt_forward.argtypes = fwd_args
    lib.ittt_forward.restype = ctypes.c_int
    lib.ittt_forward_ex.argtypes = fwd_args + [ctypes.POINTER(Opts)]
    lib.ittt_forward_ex.restype = ctypes.c_int
    lib.ittt_workspace_bytes.argtypes = [ctypes.c_int64] * 5
    lib.ittt_workspace_bytes.restype = ctypes.c_size_t
    lib.ittt_workspace_bytes_ex.argtypes = [ctypes.c_int64] * 5 + [ctypes.POINTER(Opts)]
    lib.ittt_workspace_bytes_ex.restype = ctypes.c_size_t
    lib.ittt_stream_status.argtypes = [ctypes.c_void_p]
    lib.ittt_stream_status.restype = ctypes.c_int
    lib.ittt_last_error.argtypes = []
    lib.ittt_last_error.restype = ctypes.c_char_p
    lib.ittt_version.argtypes = []
    lib.ittt_version.restype = ctypes.c_int32
    lib.ittt_launch_count.argtypes = [ctypes.c_int64] * 5
    lib.ittt_launch_count.restype = ctypes.c_int32
    lib.ittt_state_prefix.argtypes = [_TP, _TP, ctypes.c_int32, _TP, ctypes.c_void_p]
    lib.ittt_state_prefix.restype = ctypes.c_int
    lib.ittt_set_scratch_limit.argtypes = [ctypes.c_size_t]
    lib.ittt_set_scratch_limit.restype = None
    lib.ittt_plan_form.argtypes = [ctypes.c_int64] * 5 + [ctypes.POINTER(Opts)]
    lib.ittt_plan_form.restype = ctypes.c_int32
    lib.ittt_check_wait_timeout.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    lib.ittt_check_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the entry points include/ittt.h declares."""
    with open(os.path.join(_build.INCLUDE, "ittt.h")) as fh:
        text = fh.read()
    return re.findall(r"ITTT_API\s+[\w\s\*]+?\b(ittt_\w+)\s*\(", text)


def describe(t: torch.Tensor | None) -> Tensor | None:
    """ittt_tensor descriptor of a torch tensor (no copy, no check)."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("at most 4 dimensions")
    d = Tensor()
    d.data = t.data_ptr()
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for k in range(t.dim()):
        d.shape[k] = t.shape[k]
        d.stride[k] = t.stride(k)
    return d


def _ref(desc):
    return None if desc is None else ctypes.byref(desc)


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def last_error() -> str:
    return load().ittt_last_error().decode()


def _check(status: int):
    if status != OK:
        raise IttError(status, last_error())


def _seqlens(cu_seqlens):
    """int64 ctypes array of host token offsets (list, tuple or CPU tensor)."""
    if cu_seqlens is None:
        return None
    vals = [int(v) for v in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                             else cu_seqlens)]
    return (ctypes.c_int64 * len(vals))(*vals)


def _opts(pad_mode, fused_conv, dual, cu_seqlens, keep: dict, l2norm=False,
          single_cta=False, update_only=False, reuse_zv=False, primal=False,
          fp32_inputs=False, **tensors) -> Opts:
    opts = Opts()
    opts.pad_mode = int(pad_mode)
    opts.flags = ((FLAG_FUSED_CONV if fused_conv else 0) | (FLAG_DUAL if dual else 0)
                  | (FLAG_L2_NORM if l2norm else 0) | (FLAG_SINGLE_CTA if single_cta else 0)
                  | (FLAG_UPDATE_ONLY if update_only else 0)
                  | (FLAG_REUSE_ZV if reuse_zv else 0) | (FLAG_PRIMAL if primal else 0)
                  | (FLAG_FP32_INPUTS if fp32_inputs else 0))
    for name, t in tensors.items():
        if t is not None:
            keep[name] = describe(t)
            setattr(opts, name, ctypes.pointer(keep[name]))
    arr = _seqlens(cu_seqlens)
    if arr is not None:
        keep["cu_seqlens"] = arr
        opts.cu_seqlens = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64))
        opts.num_docs = len(arr) - 1
    return opts


def forward(H, X0, W_gate, W_up, W_down0, W_target, conv_w, eta: float, chunk: int,
            out: torch.Tensor | None = None, *, out_dtype=torch.bfloat16, stream=None,
            pad_mode: int = PAD_CHUNK, state_in=None, state_out=None, z_buf=None,
            vhat_buf=None, snap_buf=None, workspace=None, events=None,
            fused_conv: bool = False, dual: bool = False, eta_tok=None,
            cu_seqlens=None, l2norm: bool = False, single_cta: bool = False,
            update_only: bool = False, reuse_zv: bool = False, primal: bool = False):
    """Enqueue one layer forward on `stream` (default: current stream) and
    return `out` [B,T,d].  Extra keyword buffers map to ittt_opts; `events`
    is a list of 2 * len(PHASES) torch.cuda.Event(enable_timing=True) or
    None entries: a (start, end) pair per phase, None where not wanted.  `cu_seqlens` (host ints, num_docs + 1
    offsets) packs documents into the one row of H [1,T,d].
    `update_only` folds every chunk into `state_out` and applies nothing
    (returns None; W_down0 None starts from zero); `reuse_zv` takes Z and
    eta * Vhat from `z_buf` / `vhat_buf` instead of computing them.  The
    library picks the primal or dual form by measured cost (plan_form);
    `dual` / `primal` force one.  fp32 H, X0, W_gate, W_up and W_target
    (all five) select the fp32-input mode: the library splits each into
    bf16 hi/lo parts instead of rounding it."""
    lib = load()
    if update_only:
        out = None
    elif out is None:
        out = torch.empty(H.shape, dtype=out_dtype, device=H.device)
    keep = [describe(x) for x in (H, X0, W_gate, W_up, W_down0, W_target, conv_w, out)]
    extra = {}
    opts = _opts(pad_mode, fused_conv, dual, cu_seqlens, extra, l2norm=l2norm,
                 single_cta=single_cta, update_only=update_only, reuse_zv=reuse_zv,
                 primal=primal, state_in=state_in,
                 state_out=state_out, z_buf=z_buf, vhat_buf=vhat_buf, snap_buf=snap_buf,
                 eta_tok=eta_tok)
    if workspace is not None:
        opts.workspace = workspace.data_ptr()
        opts.workspace_bytes = workspace.numel() * workspace.element_size()
    ev_arr = None
    if events is not None:
        if len(events) != 2 * len(PHASES):
            raise ValueError(f"events needs {2 * len(PHASES)} entries")
        for e in events:  # torch creates the CUDA event on its first record
            if e is not None and not e.cuda_event:
                e.record(torch.cuda.current_stream(H.device) if stream is None else stream)
        ev_arr = (ctypes.c_void_p * len(events))(
            *[0 if e is None else int(e.cuda_event) for e in events])
        opts.events = ctypes.cast(ev_arr, ctypes.POINTER(ctypes.c_void_p))
    s = _stream_handle(stream, H.device)
    status = lib.ittt_forward_ex(*[_ref(k) for k in keep[:7]], ctypes.c_float(eta),
                                 ctypes.c_int64(chunk), _ref(keep[7]), ctypes.c_void_p(s),
                                 ctypes.byref(opts))
    _check(status)
    return out


def forward_plain(H, X0, W_gate, W_up, W_down0, W_target, conv_w, eta: float, chunk: int,
                  out: torch.Tensor, stream=None) -> torch.Tensor:
    """The plain ittt_forward entry point (no options)."""
    lib = load()
    keep = [describe(x) for x in (H, X0, W_gate, W_up, W_down0, W_target, conv_w, out)]
    s = _stream_handle(stream, H.device)
    _check(lib.ittt_forward(*[_ref(k) for k in keep[:7]], ctypes.c_float(eta),
                            ctypes.c_int64(chunk), _ref(keep[7]), ctypes.c_void_p(s)))
    return out


def state_prefix(W_start, deltas: torch.Tensor, count: int, state: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """ittt_state_prefix: state = W_start + deltas[0] + ... + deltas[count-1]
    (fp32, in that order).  W_start: [d,f] bf16/fp32 shared by every state,
    [S,d,f] fp32, or None (zero); deltas: fp32 [R,S,d,f]; returns `state`
    [S,d,f] fp32."""
    lib = load()
    if state is None:
        state = torch.empty(deltas.shape[1:], dtype=torch.float32, device=deltas.device)
    keep = [describe(W_start), describe(deltas), describe(state)]
    s = _stream_handle(stream, deltas.device)
    _check(lib.ittt_state_prefix(_ref(keep[0]), _ref(keep[1]), ctypes.c_int32(count),
                                 _ref(keep[2]), ctypes.c_void_p(s)))
    return state


def set_scratch_limit(nbytes: int) -> None:
    """ittt_set_scratch_limit: cap on the scratch one call may allocate (0:
    none); a call over it raises IttError(ERR_OOM) before anything runs."""
    load().ittt_set_scratch_limit(ctypes.c_size_t(int(nbytes)))


def check_wait_timeout(limit_ns: int, stream=None, device=None) -> None:
    """ittt_check_wait_timeout: enqueue a kernel whose bounded wait runs out
    after `limit_ns`; the next stream_status() then raises
    IttError(ERR_TIMEOUT)."""
    _check(load().ittt_check_wait_timeout(ctypes.c_uint64(int(limit_ns)),
                                          ctypes.c_void_p(_stream_handle(stream, device))))


def stream_status(stream=None, device=None) -> None:
    """Synchronise and raise IttError if a kernel recorded a failure."""
    _check(load().ittt_stream_status(ctypes.c_void_p(_stream_handle(stream, device))))


def workspace_bytes(B: int, T: int, d: int, f: int, chunk: int) -> int:
    return int(load().ittt_workspace_bytes(B, T, d, f, chunk))


def workspace_bytes_ex(B: int, T: int, d: int, f: int, chunk: int, *, pad_mode: int = PAD_CHUNK,
                       fused_conv: bool = False, dual: bool = False, cu_seqlens=None,
                       l2norm: bool = False, update_only: bool = False, reuse_zv: bool = False,
                       primal: bool = False, fp32_inputs: bool = False, **buffers) -> int:
    """ittt_workspace_bytes_ex: scratch for a forward call with these
    options; `buffers` name the ittt_opts tensors the call passes (state_in,
    state_out, z_buf, vhat_buf, snap_buf, eta_tok) -- only whether each is
    given matters; `fp32_inputs` sizes the hi/lo split copies."""
    keep = {}
    opts = _opts(pad_mode, fused_conv, dual, cu_seqlens, keep, l2norm=l2norm,
                 update_only=update_only, reuse_zv=reuse_zv, primal=primal,
                 fp32_inputs=fp32_inputs, **buffers)
    return int(load().ittt_workspace_bytes_ex(B, T, d, f, chunk, ctypes.byref(opts)))


def plan_form(B: int, T: int, d: int, f: int, chunk: int, *, pad_mode: int = PAD_CHUNK,
              fused_conv: bool = False, dual: bool = False, cu_seqlens=None,
              l2norm: bool = False, update_only: bool = False, reuse_zv: bool = False,
              primal: bool = False, fp32_inputs: bool = False, **buffers) -> int:
    """ittt_plan_form: FORM_PRIMAL or FORM_DUAL for a call with these sizes
    and options (-1 if it would be rejected)."""
    keep = {}
    opts = _opts(pad_mode, fused_conv, dual, cu_seqlens, keep, l2norm=l2norm,
                 update_only=update_only, reuse_zv=reuse_zv, primal=primal,
                 fp32_inputs=fp32_inputs, **buffers)
    return int(load().ittt_plan_form(B, T, d, f, chunk, ctypes.byref(opts)))


def launch_count(B: int, T: int, d: int, f: int, chunk: int) -> int:
    return int(load().ittt_launch_count(B, T, d, f, chunk))


def version() -> int:
    return int(load().ittt_version())
