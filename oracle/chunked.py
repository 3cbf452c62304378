"""fp64 chunk-by-chunk oracle for full-size workloads (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module; the product library never
does.  It shares no code with the CUDA path.

This is the same sequential layer as ``oracle_forward_sequential`` in
``ittt_oracle.c``, written with numpy float64 matrix products as its steps so
that workloads with 10^4-10^5 tokens at d_model 2560 finish in seconds on a
many-core host (the plain C loops take hours there).  Per sequence, chunk by
chunk, in the pages' order ("[논문리뷰] In-Place Test-Time Training",
Method §1 eq. (2)-(4), §2 eq. (5)-(6); reading notes 整体框架):

    Z_[i]    = SiLU(H_[i] W_gate^T) * (H_[i] W_up^T)          eq. (2)
    Vhat_[i] = Conv1D(X0)_[i] W_target^T                       eq. (5)
    O_[i]    = Z_[i] (W^(i))^T                                 eq. (3), apply
    W^(i+1)  = W^(i) + eta * (r_[i] * Vhat_[i])^T Z_[i]        eq. (6), update

with W^(0) = W_down0 at every sequence (or document) start (Method §3, reset
at document boundaries) and r the optional per-token rates ("[논문리뷰]
Test-Time Training Done Right", Large-Chunk TTT Layer, per-token eta_i; 1 when
absent).  With ``l2norm`` every updated state is divided row by row by its
norm over the f inputs (same page, Non-Linear Update of Fast-Weight,
L2-Normalize(W - g); floor 1e-12); W_down0 is used as given.

The readings are those of the C oracle: SiLU(x) = x / (1 + exp(-x)); the
convolution is depthwise, taps (t-1, t, t+1) in cross-correlation order, no
bias; a tap outside the current chunk reads 0 under chunk-edge padding, one
outside the sequence under sequence padding; chunks are 0-based and the last
may be the shorter remainder.

Nothing is blocked, fused or reordered beyond the per-chunk loop the
definition states; every matrix product is one numpy ``@`` in float64.
"""
from __future__ import annotations

import numpy as np

PAD_CHUNK = 0
PAD_SEQUENCE = 1


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) = x / (1 + exp(-x)); exp overflow gives -0 (the limit)."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def conv_rows(X0: np.ndarray, conv_w: np.ndarray, lo: int, hi: int,
              seg_lo: int, seg_hi: int) -> np.ndarray:
    """Depthwise three-tap Conv1D of rows [lo, hi) of one sequence X0 [T, d]
    (Method §2 eq. (5)); taps may read only rows in [seg_lo, seg_hi), every
    other tap reads 0."""
    d = X0.shape[1]
    pad = np.zeros((hi - lo + 2, d), np.float64)   # rows lo-1 .. hi
    a, b = max(lo - 1, seg_lo), min(hi + 1, seg_hi)
    pad[a - (lo - 1):b - (lo - 1)] = _f64(X0[a:b])
    w = _f64(conv_w)
    return pad[:-2] * w[:, 0] + pad[1:-1] * w[:, 1] + pad[2:] * w[:, 2]


def _normalise_rows(W: np.ndarray) -> np.ndarray:
    norm = np.sqrt((W * W).sum(axis=1))
    return W / np.maximum(norm, 1e-12)[:, None]


def walk_sequence(H, X0, W_gate, W_up, W0, W_target, conv_w, eta: float,
                  chunk: int, pad_mode: int = PAD_CHUNK, eta_tok=None,
                  l2norm: bool = False, want_final: bool = False,
                  weights64: dict | None = None):
    """The layer over ONE sequence H, X0 [T, d], chunk by chunk.

    Yields, for chunk i = 0..n-1, a dict with "i", "lo", "hi" (its token
    range), "Z" [len, f], "Vhat" [len, d] (not scaled by eta), "W" (the state
    W^(i) [d, f] applied to it) and "O" [len, d]; the last chunk's dict also
    holds "W_next" = W^(n) when ``want_final``.  All float64.  ``weights64``
    may hold the float64 weights already converted (keys W_gate, W_up,
    W_target), to share them across sequences.
    """
    if chunk <= 0:
        raise ValueError("chunk must be positive")
    T = H.shape[0]
    w = weights64 if weights64 is not None else {}
    Wg = w["W_gate"] if "W_gate" in w else _f64(W_gate)
    Wu = w["W_up"] if "W_up" in w else _f64(W_up)
    Wt = w["W_target"] if "W_target" in w else _f64(W_target)
    W = _f64(W0).copy()
    rates = None if eta_tok is None else _f64(eta_tok).reshape(T)
    n = -(-T // chunk)
    for i in range(n):
        lo, hi = i * chunk, min((i + 1) * chunk, T)
        Hi = _f64(H[lo:hi])
        Z = silu(Hi @ Wg.T) * (Hi @ Wu.T)
        seg = (lo, hi) if pad_mode == PAD_CHUNK else (0, T)
        V = conv_rows(X0, conv_w, lo, hi, *seg) @ Wt.T
        O = Z @ W.T
        out = {"i": i, "lo": lo, "hi": hi, "Z": Z, "Vhat": V, "W": W, "O": O}
        if i < n - 1 or want_final:
            Vr = V if rates is None else V * rates[lo:hi, None]
            W_next = W + eta * (Vr.T @ Z)
            if l2norm:
                W_next = _normalise_rows(W_next)
            if i == n - 1:
                out["W_next"] = W_next
            W = W_next
        yield out


def weights64(inp: dict) -> dict:
    """float64 copies of the shared weights of an input set."""
    return {k: _f64(inp[k]) for k in ("W_gate", "W_up", "W_target")}


def forward(inp, eta: float, chunk: int, pad_mode: int = PAD_CHUNK,
            eta_tok=None, l2norm: bool = False) -> dict:
    """Whole-batch form of ``walk_sequence`` for small problems: returns "O"
    [B,T,d], "Z" [B,T,f], "Vhat" [B,T,d] and "states" [B,n+1,d,f]
    (W^(0)..W^(n)).  inp holds H, X0 [B,T,d] and W_down0 [d,f] or [B,d,f]."""
    H, X0 = _f64(inp["H"]), _f64(inp["X0"])
    if H.ndim == 2:
        H, X0 = H[None], X0[None]
    W0 = _f64(inp["W_down0"])
    B, T, d = H.shape
    f = inp["W_gate"].shape[0]
    n = -(-T // chunk)
    rates = None if eta_tok is None else _f64(eta_tok).reshape(B, T)
    w64 = weights64(inp)
    O = np.zeros((B, T, d)); Z = np.zeros((B, T, f)); V = np.zeros((B, T, d))
    S = np.zeros((B, n + 1, d, f))
    for b in range(B):
        for c in walk_sequence(H[b], X0[b], None, None, W0[b] if W0.ndim == 3 else W0,
                               None, inp["conv_w"], eta, chunk, pad_mode,
                               None if rates is None else rates[b], l2norm,
                               want_final=True, weights64=w64):
            lo, hi = c["lo"], c["hi"]
            O[b, lo:hi], Z[b, lo:hi], V[b, lo:hi] = c["O"], c["Z"], c["Vhat"]
            S[b, c["i"]] = c["W"]
            if "W_next" in c:
                S[b, n] = c["W_next"]
    return {"O": O, "Z": Z, "Vhat": V, "states": S}


def state_grid(H, X0, W_gate, W_up, W0, W_target, conv_w, eta: float, chunk: int,
               m_idx, j_idx, pad_mode: int = PAD_CHUNK, eta_tok=None) -> np.ndarray:
    """Entries W^(i)[m, j] of the additive walk over ONE sequence for every m
    in m_idx and j in j_idx, at every chunk boundary i = 0..n:

        W^(i)[m, j] = W_down0[m, j] + eta * sum_{s < start of chunk i} r_s Vhat[s, m] Z[s, j]

    (Method §1 eq. (6) summed over chunks; reading notes 实现细节, prefix sum).
    Only the needed columns of Z and Vhat are formed: Z[:, j] from the rows
    j of W_gate and W_up, Vhat[:, m] from the rows m of W_target.  Returns
    [n+1, len(m_idx), len(j_idx)] float64.
    """
    m_idx = np.asarray(m_idx, np.int64)
    j_idx = np.asarray(j_idx, np.int64)
    T = H.shape[0]
    Wg, Wu = _f64(W_gate)[j_idx], _f64(W_up)[j_idx]
    Wt = _f64(W_target)[m_idx]
    rates = None if eta_tok is None else _f64(eta_tok).reshape(T)
    n = -(-T // chunk)
    out = np.zeros((n + 1, len(m_idx), len(j_idx)))
    out[0] = _f64(W0)[np.ix_(m_idx, j_idx)]
    acc = np.zeros((len(m_idx), len(j_idx)))
    for i in range(n):
        lo, hi = i * chunk, min((i + 1) * chunk, T)
        Hi = _f64(H[lo:hi])
        Z = silu(Hi @ Wg.T) * (Hi @ Wu.T)
        seg = (lo, hi) if pad_mode == PAD_CHUNK else (0, T)
        V = conv_rows(X0, conv_w, lo, hi, *seg) @ Wt.T
        if rates is not None:
            V = V * rates[lo:hi, None]
        acc = acc + V.T @ Z
        out[i + 1] = out[0] + eta * acc
    return out
