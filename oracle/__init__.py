"""fp64 CPU oracle for the In-Place TTT fast-weight layer (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product library never
does.  The arithmetic lives in ``ittt_oracle.c`` (plain C, double precision,
OpenMP over output rows); this module only compiles it with gcc, loads it with
ctypes and converts numpy arrays.

Every function here evaluates the layer as the In-Place TTT pages define it
("[논문리뷰] In-Place Test-Time Training", Method §1 eq. (2)-(4), §2 eq. (5)-(6),
§3 "Implementation Details"); see the C file's header for the readings taken
where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ittt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libittt_oracle.so")

PAD_CHUNK = 0
PAD_SEQUENCE = 1

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_int = ctypes.c_int
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ittt_oracle.c into a shared library (gcc -O2 -fopenmp)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # ITTT_ORACLE_LIB lets the oracle's own mutation test load a copy of
        # this library built from a deliberately broken source.
        lib = ctypes.CDLL(os.environ.get("ITTT_ORACLE_LIB") or build())
        lib.oracle_gated_activation.argtypes = [_i64, _i64, _i64, _fp, _fp, _fp, _dp]
        lib.oracle_conv1d.argtypes = [_i64, _i64, _i64, _int, _fp, _fp, _dp]
        lib.oracle_value_target.argtypes = [_i64, _i64, _i64, _int, _fp, _fp, _fp, _dp]
        lib.oracle_forward_sequential.argtypes = [
            _i64, _i64, _i64, _i64, _i64, _dbl, _int, _fp, _fp, _fp, _fp, _fp,
            _i64, _fp, _fp, _fp, _dp, _dp, _dp, _dp]
        lib.oracle_forward_prefix.argtypes = [
            _i64, _i64, _i64, _i64, _i64, _dbl, _int, _fp, _fp, _fp, _fp, _fp,
            _i64, _fp, _fp, _fp, _dp, _dp]
        lib.oracle_forward_l2norm.argtypes = [
            _i64, _i64, _i64, _i64, _i64, _dbl, _int, _fp, _fp, _fp, _fp, _fp,
            _i64, _fp, _fp, _fp, _dp, _dp]
        lib.oracle_forward_dual.argtypes = [
            _i64, _i64, _i64, _i64, _i64, _dbl, _int, _fp, _fp, _fp, _fp, _fp,
            _i64, _fp, _fp, _fp, _dp]
        lib.oracle_z_entries.argtypes = [_i64, _fp, _fp, _fp, _i64, _ip, _ip, _dp]
        lib.oracle_vhat_entries.argtypes = [_i64, _i64, _i64, _int, _fp, _fp, _fp,
                                            _i64, _ip, _ip, _dp]
        lib.oracle_state_entries.argtypes = [
            _i64, _i64, _i64, _i64, _dbl, _int, _fp, _fp, _fp, _fp, _fp, _fp,
            _fp, _fp, _i64, _ip, _ip, _dp]
        lib.oracle_first_chunk_rows.argtypes = [_i64, _i64, _fp, _fp, _fp, _fp,
                                                _i64, _ip, _dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _f32(a) -> np.ndarray:
    """C-contiguous float32 view/copy of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _fptr(a):
    return None if a is None else a.ctypes.data_as(_fp)


def _dptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(_ip)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's OpenMP loops use from now on (results do not
    depend on it)."""
    _load().oracle_set_num_threads(int(n))


def _unpack(inp):
    H, X0 = _f32(inp["H"]), _f32(inp["X0"])
    Wg, Wu = _f32(inp["W_gate"]), _f32(inp["W_up"])
    W0, Wt, cw = _f32(inp["W_down0"]), _f32(inp["W_target"]), _f32(inp["conv_w"])
    if H.ndim == 2:
        H, X0 = H[None], X0[None]
    B, T, d = H.shape
    f = Wg.shape[0]
    assert X0.shape == (B, T, d) and Wg.shape == (f, d) and Wu.shape == (f, d)
    assert Wt.shape == (d, d) and cw.shape == (d, 3)
    if W0.ndim == 3:  # per-sequence initial state
        assert W0.shape == (B, d, f)
        w0_stride = d * f
    else:
        assert W0.shape == (d, f)
        w0_stride = 0
    return H, X0, Wg, Wu, W0, Wt, cw, B, T, d, f, w0_stride


def _eta_tok(eta_tok, B, T):
    if eta_tok is None:
        return None
    e = _f32(eta_tok).reshape(B, T)
    return np.ascontiguousarray(e)


def _chunks(T: int, chunk: int) -> int:
    """Chunk count; the last chunk is the remainder when chunk does not divide T."""
    if chunk <= 0:
        raise ValueError("chunk must be positive")
    return -(-T // chunk)


def forward(inp, eta: float, chunk: int, pad_mode: int = PAD_CHUNK,
            want_z: bool = False, want_vhat: bool = False,
            want_states: bool = False, eta_tok=None, l2norm: bool = False) -> dict:
    """Sequential apply-then-update loop over chunks (the defining form).

    Returns {"O": [B,T,d]} plus optional "Z" [B,T,f], "Vhat" [B,T,d] and
    "states" [B,n+1,d,f] (W^(0)..W^(n)), all float64.  eta_tok: optional
    per-token learning-rate weights [B,T].  l2norm: normalise every updated
    state row by row (the normalised update rule; Z and Vhat are then not
    returned).
    """
    H, X0, Wg, Wu, W0, Wt, cw, B, T, d, f, w0s = _unpack(inp)
    n = _chunks(T, chunk)
    et = _eta_tok(eta_tok, B, T)
    if l2norm:
        if want_z or want_vhat:
            raise ValueError("the normalised form returns O and the states only")
        O = np.zeros((B, T, d), np.float64)
        S = np.zeros((B, n + 1, d, f), np.float64) if want_states else None
        _load().oracle_forward_l2norm(
            B, T, d, f, chunk, float(eta), pad_mode, _fptr(H), _fptr(X0), _fptr(Wg),
            _fptr(Wu), _fptr(W0), w0s, _fptr(Wt), _fptr(cw), _fptr(et), _dptr(O), _dptr(S))
        out = {"O": O}
        if want_states:
            out["states"] = S
        return out
    O = np.zeros((B, T, d), np.float64)
    Z = np.zeros((B, T, f), np.float64) if want_z else None
    V = np.zeros((B, T, d), np.float64) if want_vhat else None
    S = np.zeros((B, n + 1, d, f), np.float64) if want_states else None
    _load().oracle_forward_sequential(
        B, T, d, f, chunk, float(eta), pad_mode, _fptr(H), _fptr(X0), _fptr(Wg),
        _fptr(Wu), _fptr(W0), w0s, _fptr(Wt), _fptr(cw), _fptr(et), _dptr(O), _dptr(Z),
        _dptr(V), _dptr(S))
    out = {"O": O}
    if want_z:
        out["Z"] = Z
    if want_vhat:
        out["Vhat"] = V
    if want_states:
        out["states"] = S
    return out


def forward_prefix(inp, eta: float, chunk: int, pad_mode: int = PAD_CHUNK,
                   want_states: bool = False, eta_tok=None) -> dict:
    """Three-stage form: per-chunk deltas, exclusive prefix sum, apply."""
    H, X0, Wg, Wu, W0, Wt, cw, B, T, d, f, w0s = _unpack(inp)
    n = _chunks(T, chunk)
    et = _eta_tok(eta_tok, B, T)
    O = np.zeros((B, T, d), np.float64)
    S = np.zeros((B, n + 1, d, f), np.float64) if want_states else None
    _load().oracle_forward_prefix(
        B, T, d, f, chunk, float(eta), pad_mode, _fptr(H), _fptr(X0), _fptr(Wg),
        _fptr(Wu), _fptr(W0), w0s, _fptr(Wt), _fptr(cw), _fptr(et), _dptr(O), _dptr(S))
    out = {"O": O}
    if want_states:
        out["states"] = S
    return out


def forward_dual(inp, eta: float, chunk: int, pad_mode: int = PAD_CHUNK,
                 eta_tok=None) -> dict:
    """Dual form O_[i] = Z_[i] W0^T + eta * sum_{j<i} (Z_[i] Z_[j]^T) Vhat_[j]."""
    H, X0, Wg, Wu, W0, Wt, cw, B, T, d, f, w0s = _unpack(inp)
    _chunks(T, chunk)
    et = _eta_tok(eta_tok, B, T)
    O = np.zeros((B, T, d), np.float64)
    _load().oracle_forward_dual(
        B, T, d, f, chunk, float(eta), pad_mode, _fptr(H), _fptr(X0), _fptr(Wg),
        _fptr(Wu), _fptr(W0), w0s, _fptr(Wt), _fptr(cw), _fptr(et), _dptr(O))
    return {"O": O}


def gated_activation(H, W_gate, W_up) -> np.ndarray:
    """Z = SiLU(H W_gate^T) * (H W_up^T) for one sequence H [T, d]."""
    H, Wg, Wu = _f32(H), _f32(W_gate), _f32(W_up)
    T, d = H.shape
    f = Wg.shape[0]
    Z = np.zeros((T, f), np.float64)
    _load().oracle_gated_activation(T, d, f, _fptr(H), _fptr(Wg), _fptr(Wu), _dptr(Z))
    return Z


def conv1d(X0, conv_w, chunk: int, pad_mode: int = PAD_CHUNK) -> np.ndarray:
    """Depthwise three-tap convolution of one sequence X0 [T, d]."""
    X0, cw = _f32(X0), _f32(conv_w)
    T, d = X0.shape
    Xc = np.zeros((T, d), np.float64)
    _load().oracle_conv1d(T, d, chunk, pad_mode, _fptr(X0), _fptr(cw), _dptr(Xc))
    return Xc


def value_target(X0, conv_w, W_target, chunk: int,
                 pad_mode: int = PAD_CHUNK) -> np.ndarray:
    """Vhat = Conv1D(X0) W_target^T for one sequence X0 [T, d]."""
    X0, cw, Wt = _f32(X0), _f32(conv_w), _f32(W_target)
    T, d = X0.shape
    V = np.zeros((T, d), np.float64)
    _load().oracle_value_target(T, d, chunk, pad_mode, _fptr(X0), _fptr(cw),
                                _fptr(Wt), _dptr(V))
    return V


# --------------------------------------------------------------------------
# Entry-wise evaluators (full-size workloads).  `H`, `X0` are ONE sequence.
# --------------------------------------------------------------------------

def z_entries(H, W_gate, W_up, t_idx, j_idx) -> np.ndarray:
    H, Wg, Wu = _f32(H), _f32(W_gate), _f32(W_up)
    t = np.ascontiguousarray(t_idx, np.int64)
    j = np.ascontiguousarray(j_idx, np.int64)
    out = np.zeros(len(t), np.float64)
    _load().oracle_z_entries(H.shape[1], _fptr(H), _fptr(Wg), _fptr(Wu), len(t),
                             _iptr(t), _iptr(j), _dptr(out))
    return out


def vhat_entries(X0, conv_w, W_target, chunk: int, t_idx, m_idx,
                 pad_mode: int = PAD_CHUNK) -> np.ndarray:
    X0, cw, Wt = _f32(X0), _f32(conv_w), _f32(W_target)
    T, d = X0.shape
    t = np.ascontiguousarray(t_idx, np.int64)
    m = np.ascontiguousarray(m_idx, np.int64)
    out = np.zeros(len(t), np.float64)
    _load().oracle_vhat_entries(T, d, chunk, pad_mode, _fptr(X0), _fptr(cw),
                                _fptr(Wt), len(t), _iptr(t), _iptr(m), _dptr(out))
    return out


def state_entries(H, X0, W_gate, W_up, w0, W_target, conv_w, eta: float,
                  chunk: int, m_idx, j_idx, pad_mode: int = PAD_CHUNK,
                  eta_tok=None) -> np.ndarray:
    """W^(i)[m, j] for i = 0..n at each (m, j) pair: returns [count, n+1]."""
    H, X0 = _f32(H), _f32(X0)
    Wg, Wu, w0 = _f32(W_gate), _f32(W_up), _f32(w0)
    Wt, cw = _f32(W_target), _f32(conv_w)
    T, d = H.shape
    f = Wg.shape[0]
    n = _chunks(T, chunk)
    et = None if eta_tok is None else np.ascontiguousarray(_f32(eta_tok).reshape(T))
    m = np.ascontiguousarray(m_idx, np.int64)
    j = np.ascontiguousarray(j_idx, np.int64)
    out = np.zeros((len(m), n + 1), np.float64)
    _load().oracle_state_entries(T, d, f, chunk, float(eta), pad_mode, _fptr(H),
                                 _fptr(X0), _fptr(Wg), _fptr(Wu), _fptr(w0),
                                 _fptr(Wt), _fptr(cw), _fptr(et), len(m), _iptr(m),
                                 _iptr(j), _dptr(out))
    return out


def first_chunk_rows(H, W_gate, W_up, w0, rows) -> np.ndarray:
    """O[t, :] = Z[t, :] W_down0^T for tokens t of the first chunk: [count, d]."""
    H, Wg, Wu, w0 = _f32(H), _f32(W_gate), _f32(W_up), _f32(w0)
    d = H.shape[1]
    f = Wg.shape[0]
    r = np.ascontiguousarray(rows, np.int64)
    out = np.zeros((len(r), d), np.float64)
    _load().oracle_first_chunk_rows(d, f, _fptr(H), _fptr(Wg), _fptr(Wu),
                                    _fptr(w0), len(r), _iptr(r), _dptr(out))
    return out


# --------------------------------------------------------------------------
# Packed documents
# --------------------------------------------------------------------------

def forward_packed(inp, cu_seqlens, eta: float, chunk: int, pad_mode: int = PAD_CHUNK,
                   want_z: bool = False, want_vhat: bool = False, want_states: bool = False,
                   eta_tok=None, l2norm: bool = False) -> dict:
    """Documents packed along one token axis, the fast weight reset to W_0 at
    every document boundary ("[논문리뷰] In-Place Test-Time Training",
    Method §3, causality and boundary handling): document k, the tokens
    [cu_seqlens[k], cu_seqlens[k+1]), is run as a sequence of its own -- its
    chunks start at its first token and no convolution tap crosses into a
    neighbour.

    inp["H"], inp["X0"]: [T, d] or [1, T, d]; inp["W_down0"]: [d, f] shared
    or [num_docs, d, f] per document; eta_tok: [T] or [1, T].  Returns "O"
    [T, d] (and "Z" [T, f], "Vhat" [T, d] when asked), plus "states": a list
    with document k's W^(0)..W^(n_k) as [n_k + 1, d, f].
    """
    cu = [int(v) for v in cu_seqlens]
    H = _f32(inp["H"]).reshape(-1, _f32(inp["H"]).shape[-1])
    X0 = _f32(inp["X0"]).reshape(H.shape)
    W0 = _f32(inp["W_down0"])
    T, d = H.shape
    if cu[0] != 0 or cu[-1] != T or any(b <= a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must rise strictly from 0 to T")
    et = None if eta_tok is None else _f32(eta_tok).reshape(T)
    f = _f32(inp["W_gate"]).shape[0]
    O = np.zeros((T, d), np.float64)
    Z = np.zeros((T, f), np.float64) if want_z else None
    V = np.zeros((T, d), np.float64) if want_vhat else None
    states = []
    for k in range(len(cu) - 1):
        a, b = cu[k], cu[k + 1]
        doc = dict(inp)
        doc["H"], doc["X0"] = H[a:b][None], X0[a:b][None]
        doc["W_down0"] = W0[k] if W0.ndim == 3 else W0
        r = forward(doc, eta, chunk, pad_mode, want_z=want_z, want_vhat=want_vhat,
                    want_states=want_states, eta_tok=None if et is None else et[a:b][None],
                    l2norm=l2norm)
        O[a:b] = r["O"][0]
        if want_z:
            Z[a:b] = r["Z"][0]
        if want_vhat:
            V[a:b] = r["Vhat"][0]
        if want_states:
            states.append(r["states"][0])
    out = {"O": O}
    if want_z:
        out["Z"] = Z
    if want_vhat:
        out["Vhat"] = V
    if want_states:
        out["states"] = states
    return out
