"""Pins for the fp64 oracle: every check compares it with something other than
itself -- a library routine, a closed form, an invariant of the method, brute
force finite differences or a hand-derived worked example.

Citations are to the In-Place TTT pages:
  "[논문리뷰] In-Place Test-Time Training" (kimjy99 review), Method §1 eq.
  (1)-(4), §2 eq. (5)-(6), §3 "Implementation Details";
  "In-Place Test-Time Training" reading notes (gitcode), 实现细节.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from chunk_wise_weight_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _t64(x):
    return torch.as_tensor(np.asarray(x), dtype=torch.float64)


def _inputs(B=2, T=12, d=6, f=10, seed=7, round_bf16=False):
    return make_inputs(B, T, d, f, seed, round_bf16=round_bf16)


def _lib_gated_mlp_z(H, Wg, Wu):
    """torch fp64 library evaluation of SiLU(H Wg^T) * (H Wu^T)."""
    H, Wg, Wu = _t64(H), _t64(Wg), _t64(Wu)
    return F.silu(F.linear(H, Wg)) * F.linear(H, Wu)


def _lib_conv_target(X0, conv_w, Wt, chunk, pad_mode):
    """torch fp64 library evaluation of Conv1D(X0) W_target^T for one
    sequence: depthwise conv1d (cross-correlation, padding 1) run per chunk
    (chunk-edge zero padding) or on the whole sequence."""
    X0, cw, Wt = _t64(X0), _t64(conv_w), _t64(Wt)
    T, d = X0.shape
    seg = chunk if pad_mode == oracle.PAD_CHUNK else T
    parts = []
    for s in range(0, T, seg):
        x = X0[s:s + seg].T.unsqueeze(0)                      # [1, d, seg]
        y = F.conv1d(x, cw.unsqueeze(1), padding=1, groups=d)  # [1, d, seg]
        parts.append(y[0].T)
    Xc = torch.cat(parts, 0)
    return F.linear(Xc, Wt)


# --------------------------------------------------------------------------
# Special cases that reduce to library routines
# --------------------------------------------------------------------------

@pytest.mark.parametrize("B,T,d,f,C", [(1, 8, 4, 6, 2), (2, 12, 6, 10, 4), (1, 9, 5, 3, 3)])
def test_eta_zero_is_plain_gated_mlp(B, T, d, f, C):
    """eta = 0 leaves W_down fixed: the layer is exactly the gated MLP of
    Method §1 eq. (1), O = (SiLU(H Wg^T) * (H Wu^T)) W_down^T."""
    inp = _inputs(B, T, d, f, seed=11)
    got = oracle.forward(inp, eta=0.0, chunk=C)["O"]
    ref = F.linear(_lib_gated_mlp_z(inp["H"], inp["W_gate"], inp["W_up"]), _t64(inp["W_down0"]))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("eta", [0.3, -1.7])
def test_single_chunk_applies_initial_weight(eta):
    """C = T: the only chunk is applied before any update (Method §1 eq. (3)
    with W^(0) = W_down), so O = Z W_down0^T whatever eta is."""
    inp = _inputs(2, 10, 4, 7, seed=3)
    got = oracle.forward(inp, eta=eta, chunk=10)["O"]
    ref = F.linear(_lib_gated_mlp_z(inp["H"], inp["W_gate"], inp["W_up"]), _t64(inp["W_down0"]))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_z_matches_library():
    """Method §1 eq. (2): Z = SiLU(H Wg^T) * (H Wu^T)."""
    inp = _inputs(2, 9, 5, 11, seed=5)
    out = oracle.forward(inp, eta=0.1, chunk=3, want_z=True)
    ref = _lib_gated_mlp_z(inp["H"], inp["W_gate"], inp["W_up"])
    np.testing.assert_allclose(out["Z"], ref.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.gated_activation(inp["H"][1], inp["W_gate"], inp["W_up"]),
                               ref[1].numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("pad_mode", [oracle.PAD_CHUNK, oracle.PAD_SEQUENCE])
@pytest.mark.parametrize("T,C", [(12, 4), (12, 12), (10, 1), (9, 3), (10, 4), (7, 3), (5, 8)])
def test_value_target_matches_library(pad_mode, T, C):
    """Method §2 eq. (5): Vhat = Conv1D(X0) W_target^T, depthwise 3-tap conv,
    zero padded at chunk edges (chunk mode) or at sequence ends."""
    inp = _inputs(2, T, 6, 4, seed=9)
    out = oracle.forward(inp, eta=0.2, chunk=C, pad_mode=pad_mode, want_vhat=True)
    for b in range(2):
        ref = _lib_conv_target(inp["X0"][b], inp["conv_w"], inp["W_target"], C, pad_mode)
        np.testing.assert_allclose(out["Vhat"][b], ref.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(
            oracle.value_target(inp["X0"][b], inp["conv_w"], inp["W_target"], C, pad_mode),
            ref.numpy(), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# The update is the gradient step of the stated loss (brute force)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,C,per_token", [(6, 3, False), (7, 3, False), (7, 3, True)])
def test_update_is_gradient_of_inner_product_loss(T, C, per_token):
    """Method §2: with L(W) = -<Z_[i] W^T, Vhat_[i]>_F the step
    W <- W - eta grad L is W + eta Vhat_[i]^T Z_[i] (eq. (6)).  Central finite
    differences of L over every entry of W (L is linear in W, so they are
    exact up to rounding) must equal -(W^(i+1) - W^(i)) / eta for each chunk,
    the partial last chunk included.  With per-token rates the loss is
    sum_t eta_t L_t (the large-chunk update of "Test-Time Training Done
    Right", per-token eta_i)."""
    d, f, eta = 4, 8, 0.37
    inp = _inputs(1, T, d, f, seed=21)
    rates = (torch.rand(1, T, generator=torch.Generator().manual_seed(5)) + 0.25
             if per_token else None)
    out = oracle.forward(inp, eta=eta, chunk=C, want_z=True, want_vhat=True, want_states=True,
                         eta_tok=rates)
    Z, V, S = out["Z"][0], out["Vhat"][0], out["states"][0]
    wt = np.ones(T) if rates is None else rates[0].double().numpy()
    h = 1e-3
    for i in range(-(-T // C)):
        Zi, Vi = Z[i * C:(i + 1) * C], V[i * C:(i + 1) * C]
        wi = wt[i * C:(i + 1) * C, None]

        def loss(W):
            return -np.sum(wi * (Zi @ W.T) * Vi)

        W = S[i].copy()
        grad = np.zeros_like(W)
        for m in range(d):
            for j in range(f):
                Wp, Wm = W.copy(), W.copy()
                Wp[m, j] += h
                Wm[m, j] -= h
                grad[m, j] = (loss(Wp) - loss(Wm)) / (2 * h)
        step = (S[i + 1] - S[i]) / eta
        np.testing.assert_allclose(step, -grad, rtol=1e-9, atol=1e-10)


# --------------------------------------------------------------------------
# The three forms agree (Method §3, reading notes 实现细节, dual expansion)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("B,T,d,f,C,pad", [(2, 16, 5, 7, 4, 0), (1, 15, 3, 9, 5, 1), (3, 8, 4, 4, 1, 0)])
def test_prefix_form_equals_sequential(B, T, d, f, C, pad):
    inp = _inputs(B, T, d, f, seed=13)
    eta = 0.23
    seq = oracle.forward(inp, eta, C, pad, want_states=True)
    pre = oracle.forward_prefix(inp, eta, C, pad, want_states=True)
    np.testing.assert_allclose(pre["O"], seq["O"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(pre["states"], seq["states"], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("B,T,d,f,C,pad", [(2, 16, 5, 7, 4, 0), (1, 15, 3, 9, 5, 1), (1, 8, 4, 4, 8, 0)])
def test_dual_form_equals_sequential(B, T, d, f, C, pad):
    inp = _inputs(B, T, d, f, seed=17)
    eta = -0.4
    seq = oracle.forward(inp, eta, C, pad)
    dual = oracle.forward_dual(inp, eta, C, pad)
    np.testing.assert_allclose(dual["O"], seq["O"], rtol=1e-11, atol=1e-11)


def test_states_start_at_initial_weight_and_accumulate():
    """W^(0) = W_down0 (Method §1) and consecutive states differ by eta times
    a rank-<=C matrix built from that chunk only."""
    inp = _inputs(1, 12, 5, 6, seed=2)
    out = oracle.forward(inp, 0.5, 4, want_states=True, want_z=True, want_vhat=True)
    S = out["states"][0]
    np.testing.assert_array_equal(S[0], inp["W_down0"].double().numpy())
    for i in range(3):
        r = np.linalg.matrix_rank(S[i + 1] - S[i], tol=1e-9)
        assert r <= 4


# --------------------------------------------------------------------------
# Causality and boundary handling (Method §3)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pad_mode", [oracle.PAD_CHUNK, oracle.PAD_SEQUENCE])
@pytest.mark.parametrize("p", [0, 3, 4, 5, 11])
@pytest.mark.parametrize("which", ["H", "X0"])
def test_causality(pad_mode, p, which):
    """Perturbing H or X0 at position p leaves every output at t < p exactly
    unchanged (apply-then-update order plus causal padding)."""
    T, C = 12, 4
    inp = _inputs(1, T, 4, 6, seed=31)
    base = oracle.forward(inp, 0.7, C, pad_mode, want_states=True)
    pert = {k: v.clone() for k, v in inp.items()}
    pert[which][0, p] += 3.0
    new = oracle.forward(pert, 0.7, C, pad_mode, want_states=True)
    np.testing.assert_array_equal(new["O"][0, :p], base["O"][0, :p])
    assert not np.array_equal(new["O"][0, p:], base["O"][0, p:]) or p == T - 1
    if which == "X0" and pad_mode == oracle.PAD_CHUNK:
        # chunk-edge padding isolates the delta: W^(j) for j <= chunk(p)
        # does not see X0[p]
        cp = p // C
        np.testing.assert_array_equal(new["states"][0, :cp + 1], base["states"][0, :cp + 1])


def test_output_within_chunk_uses_only_earlier_chunks():
    """The state used for chunk i excludes chunk i itself: changing a late
    token of chunk i leaves every earlier token of chunk i unchanged, and
    changing the first chunk changes later chunks."""
    T, C = 12, 6
    inp = _inputs(1, T, 3, 5, seed=41)
    base = oracle.forward(inp, 1.0, C)["O"]
    pert = {k: v.clone() for k, v in inp.items()}
    pert["H"][0, 5] *= -2.0
    new = oracle.forward(pert, 1.0, C)["O"]
    np.testing.assert_array_equal(new[0, :5], base[0, :5])
    assert np.abs(new[0, 6:] - base[0, 6:]).max() > 1e-6


# --------------------------------------------------------------------------
# Linearity in eta, batch independence
# --------------------------------------------------------------------------

def test_output_is_affine_in_eta():
    """Deltas do not depend on eta or W, so O(eta) is affine in eta:
    O(2e) - O(e) = O(e) - O(0)."""
    inp = _inputs(2, 12, 4, 6, seed=43)
    e = 0.37
    o0, o1, o2 = (oracle.forward(inp, k * e, 4)["O"] for k in (0, 1, 2))
    np.testing.assert_allclose(o2 - o1, o1 - o0, rtol=1e-10, atol=1e-12)
    assert np.abs(o1 - o0).max() > 1e-3


def test_batch_rows_are_independent():
    """Every sequence starts from W_down0 (reset at document boundaries):
    permuting the batch permutes the output, and each row equals the B = 1
    result."""
    inp = _inputs(3, 8, 4, 5, seed=47)
    out = oracle.forward(inp, 0.5, 4)["O"]
    perm = [2, 0, 1]
    pinp = dict(inp)
    pinp["H"], pinp["X0"] = inp["H"][perm], inp["X0"][perm]
    np.testing.assert_array_equal(oracle.forward(pinp, 0.5, 4)["O"], out[perm])
    for b in range(3):
        one = dict(inp)
        one["H"], one["X0"] = inp["H"][b:b + 1], inp["X0"][b:b + 1]
        np.testing.assert_array_equal(oracle.forward(one, 0.5, 4)["O"][0], out[b])


def test_per_sequence_initial_state():
    """A [B, d, f] initial state gives each sequence its own W^(0)."""
    inp = _inputs(2, 8, 3, 4, seed=53)
    w0b = torch.stack([inp["W_down0"], -2.0 * inp["W_down0"]])
    binp = dict(inp)
    binp["W_down0"] = w0b
    out = oracle.forward(binp, 0.3, 4, want_states=True)
    for b in range(2):
        one = dict(inp)
        one["H"], one["X0"], one["W_down0"] = inp["H"][b:b + 1], inp["X0"][b:b + 1], w0b[b]
        ref = oracle.forward(one, 0.3, 4, want_states=True)
        np.testing.assert_array_equal(out["O"][b], ref["O"][0])
        np.testing.assert_array_equal(out["states"][b], ref["states"][0])


# --------------------------------------------------------------------------
# Closed form: the next-token target (Method §2)
# --------------------------------------------------------------------------

def test_next_token_target_closed_form():
    """W_target = I and a conv kernel that is 1 on the next token and 0
    elsewhere give the plain next-token target: Vhat_t = X0_{t+1} inside a
    chunk and 0 on a chunk's last row (chunk-edge padding), so
    dW_i = sum_{t, t+1 in chunk i} X0_{t+1}^T Z_t."""
    T, C, d, f = 12, 4, 5, 6
    inp = _inputs(1, T, d, f, seed=59)
    inp["W_target"] = torch.eye(d)
    inp["conv_w"] = torch.tensor([[0.0, 0.0, 1.0]] * d)
    out = oracle.forward(inp, 0.5, C, want_vhat=True, want_z=True, want_states=True)
    X0 = inp["X0"][0].double().numpy()
    V = out["Vhat"][0]
    for t in range(T):
        if (t + 1) % C == 0:
            np.testing.assert_array_equal(V[t], np.zeros(d))
        else:
            np.testing.assert_array_equal(V[t], X0[t + 1])
    Z = out["Z"][0]
    S = out["states"][0]
    for i in range(T // C):
        dW = sum(np.outer(X0[t + 1], Z[t]) for t in range(i * C, (i + 1) * C - 1))
        np.testing.assert_allclose(S[i + 1] - S[i], 0.5 * dW, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["scalar_two_chunks.json", "next_token_d2_f1.json",
                                  "l2norm_d1_f2.json", "packed_two_documents.json"])
def test_golden_worked_example(name):
    """Worked examples derived by hand from Method §1 eq. (2)-(3), §2 eq.
    (5)-(6) (and, where the fixture says so, the normalised update and
    packed documents with the reset at document boundaries); each fixture
    carries its derivation and citation."""
    with open(os.path.join(GOLDEN, name)) as fh:
        g = json.load(fh)
    inp = {k: torch.tensor(v, dtype=torch.float32) for k, v in g["inputs"].items()}
    l2 = g.get("l2norm", False)
    if "cu_seqlens" in g:
        out = oracle.forward_packed(inp, g["cu_seqlens"], g["eta"], g["chunk"],
                                    g.get("pad_mode", 0), want_states=True, want_vhat=not l2,
                                    l2norm=l2)
        O, V = out["O"], out.get("Vhat")
        states = out["states"]          # per document: [n_k + 1, d, f]
    else:
        out = oracle.forward(inp, g["eta"], g["chunk"], g.get("pad_mode", 0),
                             want_states=True, want_vhat=not l2, l2norm=l2)
        O, V = out["O"][0], out.get("Vhat")
        V = None if V is None else V[0]
        states = [out["states"][0]]
    env = {"math": math}
    for name_, expr in g.get("let", {}).items():
        env[name_] = _ev(expr, env)

    def mat(rows):
        return np.array([[_ev(e, env) for e in row] for row in rows], dtype=np.float64)

    if "Vhat" in g["expected"]:
        np.testing.assert_allclose(V, mat(g["expected"]["Vhat"]), rtol=1e-14, atol=0)
    np.testing.assert_allclose(O, mat(g["expected"]["O"]), rtol=1e-13, atol=1e-15)
    exp_states = g["expected"]["states"]
    if "cu_seqlens" not in g:
        exp_states = [exp_states]
    for k, doc in enumerate(exp_states):
        for i, st in enumerate(doc):
            np.testing.assert_allclose(states[k][i], mat(st), rtol=1e-13, atol=1e-15)


def _ev(e, env):
    """Fixture entries are numbers or closed-form expressions over `math` and
    the fixture's named sub-expressions."""
    if isinstance(e, (int, float)):
        return float(e)
    return float(eval(e, {"__builtins__": {}}, env))


# --------------------------------------------------------------------------
# The entry-wise evaluators used at full size agree with the full layer
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pad_mode", [oracle.PAD_CHUNK, oracle.PAD_SEQUENCE])
def test_entrywise_evaluators_agree_with_forward(pad_mode):
    B, T, d, f, C, eta = 2, 12, 5, 7, 4, 0.3
    inp = _inputs(B, T, d, f, seed=61)
    full = oracle.forward(inp, eta, C, pad_mode, want_z=True, want_vhat=True, want_states=True)
    rng = np.random.default_rng(0)
    b = 1
    t = rng.integers(0, T, 20)
    j = rng.integers(0, f, 20)
    m = rng.integers(0, d, 20)
    np.testing.assert_allclose(oracle.z_entries(inp["H"][b], inp["W_gate"], inp["W_up"], t, j),
                               full["Z"][b][t, j], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(
        oracle.vhat_entries(inp["X0"][b], inp["conv_w"], inp["W_target"], C, t, m, pad_mode),
        full["Vhat"][b][t, m], rtol=1e-13, atol=1e-14)
    st = oracle.state_entries(inp["H"][b], inp["X0"][b], inp["W_gate"], inp["W_up"],
                              inp["W_down0"], inp["W_target"], inp["conv_w"], eta, C, m, j,
                              pad_mode)
    np.testing.assert_allclose(st, full["states"][b][:, m, j].T, rtol=1e-12, atol=1e-13)
    rows = np.array([0, 1, 3])
    np.testing.assert_allclose(
        oracle.first_chunk_rows(inp["H"][b], inp["W_gate"], inp["W_up"], inp["W_down0"], rows),
        full["O"][b][rows], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# Partial last chunk (streams whose length is not a multiple of C)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,C", [(10, 4), (7, 3), (13, 5)])
def test_partial_last_chunk_extends_the_full_chunks(T, C):
    """The chunks before the partial one are exactly the run on the first
    floor(T/C) chunks (causality of the chunk order), and the partial chunk
    is applied with the state that run ends with."""
    inp = _inputs(2, T, 4, 6, seed=71)
    full = oracle.forward(inp, 0.4, C, want_states=True, want_z=True)
    Tk = (T // C) * C
    head = dict(inp)
    head["H"], head["X0"] = inp["H"][:, :Tk], inp["X0"][:, :Tk]
    part = oracle.forward(head, 0.4, C, want_states=True)
    np.testing.assert_array_equal(full["O"][:, :Tk], part["O"])
    np.testing.assert_array_equal(full["states"][:, :T // C + 1], part["states"])
    Wl = full["states"][:, T // C]
    for b in range(2):
        np.testing.assert_allclose(full["O"][b, Tk:], full["Z"][b, Tk:] @ Wl[b].T,
                                   rtol=1e-12, atol=1e-13)


def test_chunk_longer_than_sequence_is_one_partial_chunk():
    inp = _inputs(1, 5, 3, 4, seed=73)
    got = oracle.forward(inp, 0.9, 8)["O"]
    ref = F.linear(_lib_gated_mlp_z(inp["H"], inp["W_gate"], inp["W_up"]), _t64(inp["W_down0"]))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("T,C", [(10, 4), (13, 5)])
def test_forms_agree_with_partial_last_chunk(T, C):
    inp = _inputs(2, T, 4, 5, seed=75)
    seq = oracle.forward(inp, 0.3, C, want_states=True)
    pre = oracle.forward_prefix(inp, 0.3, C, want_states=True)
    dual = oracle.forward_dual(inp, 0.3, C)
    np.testing.assert_allclose(pre["O"], seq["O"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(pre["states"], seq["states"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dual["O"], seq["O"], rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------
# Per-token learning rates ("Test-Time Training Done Right", per-token eta_i)
# --------------------------------------------------------------------------

def test_unit_token_rates_are_the_plain_update():
    inp = _inputs(2, 12, 4, 6, seed=81)
    plain = oracle.forward(inp, 0.3, 4, want_states=True)
    ones = oracle.forward(inp, 0.3, 4, want_states=True, eta_tok=torch.ones(2, 12))
    np.testing.assert_array_equal(ones["O"], plain["O"])
    np.testing.assert_array_equal(ones["states"], plain["states"])


def test_constant_token_rate_scales_eta():
    inp = _inputs(2, 12, 4, 6, seed=83)
    a = oracle.forward(inp, 0.3 * 0.25, 4, want_states=True)
    b = oracle.forward(inp, 0.3, 4, want_states=True, eta_tok=torch.full((2, 12), 0.25))
    np.testing.assert_allclose(b["O"], a["O"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["states"], a["states"], rtol=1e-12, atol=1e-13)


def test_zero_token_rates_freeze_the_state():
    """Rate 0 on every token of chunk 1 leaves the state unchanged by it."""
    inp = _inputs(1, 12, 4, 6, seed=85)
    rates = torch.ones(1, 12)
    rates[0, 4:8] = 0.0
    out = oracle.forward(inp, 0.3, 4, want_states=True, eta_tok=rates)
    np.testing.assert_array_equal(out["states"][0, 2], out["states"][0, 1])
    assert np.abs(out["states"][0, 3] - out["states"][0, 2]).max() > 1e-6


def test_forms_agree_with_token_rates():
    inp = _inputs(2, 13, 4, 5, seed=87)
    rates = torch.rand(2, 13, generator=torch.Generator().manual_seed(9))
    seq = oracle.forward(inp, 0.3, 4, want_states=True, eta_tok=rates)
    pre = oracle.forward_prefix(inp, 0.3, 4, want_states=True, eta_tok=rates)
    dual = oracle.forward_dual(inp, 0.3, 4, eta_tok=rates)
    np.testing.assert_allclose(pre["O"], seq["O"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(pre["states"], seq["states"], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dual["O"], seq["O"], rtol=1e-11, atol=1e-11)
    m, j = np.array([0, 3, 1]), np.array([4, 0, 2])
    st = oracle.state_entries(inp["H"][1], inp["X0"][1], inp["W_gate"], inp["W_up"],
                              inp["W_down0"], inp["W_target"], inp["conv_w"], 0.3, 4, m, j,
                              eta_tok=rates[1])
    np.testing.assert_allclose(st, seq["states"][1][:, m, j].T, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Packed documents: the fast weight is reset at every document boundary
# (Method §3, causality and boundary handling)
# --------------------------------------------------------------------------

def test_packed_equal_documents_are_the_batch():
    """Documents of equal length packed in one row give the same outputs and
    states as the same documents run as a batch."""
    B, L, d, f, C = 3, 10, 4, 6, 4
    inp = _inputs(B, L, d, f, seed=91)
    batch = oracle.forward(inp, 0.4, C, want_z=True, want_vhat=True, want_states=True)
    packed = dict(inp)
    packed["H"], packed["X0"] = inp["H"].reshape(1, B * L, d), inp["X0"].reshape(1, B * L, d)
    cu = [0, L, 2 * L, 3 * L]
    got = oracle.forward_packed(packed, cu, 0.4, C, want_z=True, want_vhat=True,
                                want_states=True)
    np.testing.assert_array_equal(got["O"], batch["O"].reshape(B * L, d))
    np.testing.assert_array_equal(got["Z"], batch["Z"].reshape(B * L, f))
    np.testing.assert_array_equal(got["Vhat"], batch["Vhat"].reshape(B * L, d))
    for k in range(B):
        np.testing.assert_array_equal(got["states"][k], batch["states"][k])


@pytest.mark.parametrize("cu", [[0, 3, 7, 11, 12], [0, 4, 8, 12], [0, 12]])
def test_packed_short_documents_are_the_plain_mlp(cu):
    """Documents no longer than a chunk are one chunk each, applied with the
    reset weight before any update: O = Z W0_k^T per document (torch fp64),
    whatever eta is.  Without the reset, documents after the first chunk
    boundary of the packed row would see updates."""
    T, d, f, C = 12, 5, 7, 4 if len(cu) > 2 else 12
    inp = _inputs(1, T, d, f, seed=93)
    nd = len(cu) - 1
    w0 = torch.stack([inp["W_down0"] * (1.0 + 0.5 * k) for k in range(nd)])
    pk = dict(inp)
    pk["W_down0"] = w0
    got = oracle.forward_packed(pk, cu, 0.8, C)["O"]
    Z = _lib_gated_mlp_z(inp["H"][0], inp["W_gate"], inp["W_up"])
    for k in range(nd):
        ref = F.linear(Z[cu[k]:cu[k + 1]], _t64(w0[k]))
        np.testing.assert_allclose(got[cu[k]:cu[k + 1]], ref.numpy(), rtol=1e-12, atol=1e-13)
    if nd > 1:
        # the same row with no reset (one long sequence) differs
        whole = dict(inp)
        noreset = oracle.forward(whole, 0.8, C)["O"][0]
        assert np.abs(noreset - got).max() > 1e-3


@pytest.mark.parametrize("pad_mode", [oracle.PAD_CHUNK, oracle.PAD_SEQUENCE])
@pytest.mark.parametrize("which", ["H", "X0"])
def test_packed_documents_do_not_leak(pad_mode, which):
    """Perturbing one document's tokens leaves every other document's
    output exactly unchanged (no state and no convolution tap crosses a
    boundary), in both padding modes."""
    cu = [0, 5, 13, 20]
    inp = _inputs(1, 20, 4, 6, seed=95)
    base = oracle.forward_packed(inp, cu, 0.5, 3, pad_mode=pad_mode)["O"]
    for k in range(3):
        pert = dict(inp)
        x = inp[which].clone()
        x[0, cu[k]:cu[k + 1]] += 1.0
        pert[which] = x
        got = oracle.forward_packed(pert, cu, 0.5, 3, pad_mode=pad_mode)["O"]
        for j in range(3):
            seg = slice(cu[j], cu[j + 1])
            if j == k:
                assert np.abs(got[seg] - base[seg]).max() > 1e-6
            else:
                np.testing.assert_array_equal(got[seg], base[seg])


def test_packed_chunks_restart_at_each_document():
    """Next-token target (W_target = I, taps (0, 0, 1)): inside document k
    the chunks start at its first token, so Vhat_t = X0_{t+1} unless t is
    the last token of its chunk or of its document, and each chunk's update
    is the closed-form sum over its own tokens."""
    cu, C, d, f = [0, 7, 17], 4, 3, 5
    T = cu[-1]
    inp = _inputs(1, T, d, f, seed=97)
    inp["W_target"] = torch.eye(d)
    inp["conv_w"] = torch.tensor([[0.0, 0.0, 1.0]] * d)
    out = oracle.forward_packed(inp, cu, 0.5, C, want_z=True, want_vhat=True, want_states=True)
    X0 = inp["X0"][0].double().numpy()
    Z = out["Z"]
    for k in range(2):
        a, b = cu[k], cu[k + 1]
        for t in range(a, b):
            last = (t - a + 1) % C == 0 or t + 1 == b
            np.testing.assert_array_equal(out["Vhat"][t], np.zeros(d) if last else X0[t + 1])
        S = out["states"][k]
        n = -(-(b - a) // C)
        assert S.shape[0] == n + 1
        for i in range(n):
            lo, hi = a + i * C, min(a + (i + 1) * C, b)
            dW = sum((np.outer(X0[t + 1], Z[t]) for t in range(lo, hi - 1)), np.zeros((d, f)))
            np.testing.assert_allclose(S[i + 1] - S[i], 0.5 * dW, rtol=1e-12, atol=1e-12)


def test_packed_token_rates_follow_their_document():
    """Zero per-token rates over one document freeze its state; the other
    documents are as with unit rates."""
    cu = [0, 9, 16]
    inp = _inputs(1, 16, 4, 5, seed=99)
    ones = torch.ones(1, 16)
    rates = ones.clone()
    rates[0, 9:] = 0.0
    ref = oracle.forward_packed(inp, cu, 0.3, 4, want_states=True, eta_tok=ones)
    got = oracle.forward_packed(inp, cu, 0.3, 4, want_states=True, eta_tok=rates)
    np.testing.assert_array_equal(got["O"][:9], ref["O"][:9])
    np.testing.assert_array_equal(got["states"][0], ref["states"][0])
    for s in got["states"][1]:
        np.testing.assert_array_equal(s, got["states"][1][0])


# --------------------------------------------------------------------------
# Fast-weight L2 normalisation ("[논문리뷰] Test-Time Training Done Right",
# Non-Linear Update of Fast-Weight): W <- L2-Normalize(W + eta dW), rows of
# W_down normalised over their f inputs
# --------------------------------------------------------------------------

def test_l2norm_first_update_matches_library():
    """The first update, from library pieces: torch F.normalize (dim=1, the
    input dimension of W_down [d, f]) of W_0 + eta Vhat_[0]^T Z_[0], with
    Z and Vhat from torch's silu/linear/conv1d."""
    T, C, d, f, eta = 12, 4, 5, 7, 0.6
    inp = _inputs(1, T, d, f, seed=101)
    out = oracle.forward(inp, eta, C, want_states=True, l2norm=True)
    Z = _lib_gated_mlp_z(inp["H"][0], inp["W_gate"], inp["W_up"])
    V = _lib_conv_target(inp["X0"][0], inp["conv_w"], inp["W_target"], C, oracle.PAD_CHUNK)
    W1 = F.normalize(_t64(inp["W_down0"]) + eta * V[:C].T @ Z[:C], dim=1)
    np.testing.assert_allclose(out["states"][0, 1], W1.numpy(), rtol=1e-12, atol=1e-13)
    # the first chunk is applied with W_0 as given
    np.testing.assert_allclose(out["O"][0, :C], (Z[:C] @ _t64(inp["W_down0"]).T).numpy(),
                               rtol=1e-12, atol=1e-13)


def test_l2norm_rows_of_every_updated_state_are_unit():
    inp = _inputs(2, 13, 4, 9, seed=103)
    S = oracle.forward(inp, 0.2, 4, want_states=True, l2norm=True)["states"]
    norms = np.linalg.norm(S[:, 1:], axis=3)
    np.testing.assert_allclose(norms, np.ones_like(norms), rtol=1e-13)
    assert abs(np.linalg.norm(S[0, 0], axis=1) - 1.0).max() > 1e-3   # W_0 is not normalised


def test_l2norm_eta_zero_applies_the_normalised_initial_weight():
    """eta = 0: every update just normalises, and normalising twice changes
    nothing, so chunks after the first see F.normalize(W_0, dim=1)."""
    T, C, d, f = 12, 4, 5, 6
    inp = _inputs(1, T, d, f, seed=105)
    got = oracle.forward(inp, 0.0, C, l2norm=True)["O"][0]
    Z = _lib_gated_mlp_z(inp["H"][0], inp["W_gate"], inp["W_up"])
    W0 = _t64(inp["W_down0"])
    ref = torch.cat([Z[:C] @ W0.T, Z[C:] @ F.normalize(W0, dim=1).T])
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_l2norm_first_update_is_scale_invariant():
    """Scaling W_0 and eta by the same a > 0 scales the first update's
    argument by a, which the row normalisation removes: W^(1) and the
    output of chunk 1 are unchanged, chunk 0's output scales by a, and the
    later states (whose steps start from a unit-row W^(1) with a step a
    times larger) change."""
    T, C, a = 12, 4, 4.0   # a power of two: a * W_0 is exact in float32
    inp = _inputs(1, T, 4, 6, seed=107)
    ref = oracle.forward(inp, 0.3, C, want_states=True, l2norm=True)
    sc = dict(inp)
    sc["W_down0"] = inp["W_down0"] * a
    got = oracle.forward(sc, 0.3 * a, C, want_states=True, l2norm=True)
    np.testing.assert_allclose(got["states"][:, 1], ref["states"][:, 1], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(got["O"][:, C:2 * C], ref["O"][:, C:2 * C], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(got["O"][:, :C], a * ref["O"][:, :C], rtol=1e-12, atol=1e-12)
    assert np.abs(got["states"][:, 2] - ref["states"][:, 2]).max() > 1e-3


def test_l2norm_differs_from_the_plain_update_and_keeps_causality():
    inp = _inputs(1, 16, 4, 6, seed=109)
    plain = oracle.forward(inp, 0.5, 4)["O"]
    norm = oracle.forward(inp, 0.5, 4, l2norm=True)["O"]
    np.testing.assert_array_equal(norm[:, :4], plain[:, :4])
    assert np.abs(norm[:, 4:] - plain[:, 4:]).max() > 1e-3
    for which in ("H", "X0"):
        pert = dict(inp)
        x = inp[which].clone()
        x[0, 9] += 1.0
        pert[which] = x
        got = oracle.forward(pert, 0.5, 4, l2norm=True)["O"]
        np.testing.assert_array_equal(got[:, :9], norm[:, :9])


def test_l2norm_packed_equal_documents_are_the_batch():
    B, L, d, f, C = 2, 10, 4, 6, 4
    inp = _inputs(B, L, d, f, seed=111)
    batch = oracle.forward(inp, 0.4, C, want_states=True, l2norm=True)
    packed = dict(inp)
    packed["H"], packed["X0"] = inp["H"].reshape(1, B * L, d), inp["X0"].reshape(1, B * L, d)
    got = oracle.forward_packed(packed, [0, L, 2 * L], 0.4, C, want_states=True, l2norm=True)
    np.testing.assert_array_equal(got["O"], batch["O"].reshape(B * L, d))
    for k in range(B):
        np.testing.assert_array_equal(got["states"][k], batch["states"][k])
