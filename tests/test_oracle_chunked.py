"""Pins for the chunk-by-chunk fp64 oracle (oracle/chunked.py), the one the
GPU tests use at full size.

It is checked against the pinned C oracle (the plain sequential loop of
"[논문리뷰] In-Place Test-Time Training", Method §1 eq. (2)-(4), §2 eq.
(5)-(6)) on small problems that cover every option it takes, against the
hand-derived worked examples in tests/golden, and against library routines
on the special cases that reduce to them.
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
from oracle import chunked

# The mutation test (tests/test_oracle_mutants.py) points this at a copy of
# oracle/chunked.py with one planted mistake; the pins below must then fail.
if os.environ.get("ITTT_CHUNKED_ORACLE"):
    import importlib.util
    _spec = importlib.util.spec_from_file_location("chunked_mutant",
                                                   os.environ["ITTT_CHUNKED_ORACLE"])
    chunked = importlib.util.module_from_spec(_spec)
    _spec.loader.exec_module(chunked)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def close(got, ref, rel=1e-11):
    got, ref = np.asarray(got), np.asarray(ref)
    scale = max(float(np.abs(ref).max()), 1e-300)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = float(np.abs(got - ref).max()) / scale
    assert err <= rel, f"max |diff| / max |ref| = {err:.3e}"


CASES = [
    # B, T, d, f, C, pad mode, per-token rates, per-sequence W0, l2norm
    (1, 16, 4, 6, 4, 0, False, False, False),
    (2, 23, 5, 7, 6, 0, True, False, False),      # partial last chunk, rates
    (2, 20, 6, 9, 5, 1, False, True, False),      # sequence padding, per-sequence W0
    (3, 17, 4, 10, 17, 0, False, False, False),   # one chunk
    (1, 9, 3, 5, 20, 1, True, False, False),      # chunk longer than the sequence
    (2, 21, 5, 8, 4, 0, True, True, True),        # normalised update, everything on
    (1, 30, 6, 6, 7, 1, False, False, True),
]


@pytest.mark.parametrize("B,T,d,f,C,pad,rates,w0_seq,l2", CASES)
def test_chunked_equals_sequential_c_oracle(B, T, d, f, C, pad, rates, w0_seq, l2):
    inp = make_inputs(B, T, d, f, seed=500 + T + d, round_bf16=False)
    if w0_seq:
        inp["W_down0"] = torch.randn(B, d, f, generator=torch.Generator().manual_seed(3)) * 0.3
    et = (torch.rand(B, T, generator=torch.Generator().manual_seed(4)) + 0.5) if rates else None
    eta = 0.37
    ref = oracle.forward(inp, eta, C, pad, want_z=not l2, want_vhat=not l2, want_states=True,
                         eta_tok=et, l2norm=l2)
    got = chunked.forward(inp, eta, C, pad, eta_tok=et, l2norm=l2)
    close(got["O"], ref["O"])
    close(got["states"], ref["states"])
    if not l2:
        close(got["Z"], ref["Z"])
        close(got["Vhat"], ref["Vhat"])


def test_chunked_walk_per_document_equals_packed_c_oracle():
    """Packed documents: each document walked on its own from W_down0 (the
    reset at document boundaries, Method §3) equals the C oracle's packed
    form."""
    cu = [0, 5, 6, 19, 30]
    d, f, C, eta = 5, 8, 4, 0.4
    inp = make_inputs(1, 30, d, f, seed=41, round_bf16=False)
    ref = oracle.forward_packed(inp, cu, eta, C, oracle.PAD_SEQUENCE, want_states=True)
    w64 = chunked.weights64(inp)
    for k, (a, b) in enumerate(zip(cu, cu[1:])):
        H, X0 = inp["H"][0, a:b], inp["X0"][0, a:b]
        for c in chunked.walk_sequence(H, X0, None, None, inp["W_down0"], None, inp["conv_w"],
                                       eta, C, chunked.PAD_SEQUENCE, want_final=True,
                                       weights64=w64):
            close(c["O"], ref["O"][a + c["lo"]:a + c["hi"]])
            close(c["W"], ref["states"][k][c["i"]])
            if "W_next" in c:
                close(c["W_next"], ref["states"][k][-1])


@pytest.mark.parametrize("name", ["scalar_two_chunks.json", "next_token_d2_f1.json",
                                  "l2norm_d1_f2.json", "packed_two_documents.json"])
def test_chunked_worked_examples(name):
    """The hand-derived worked examples of tests/golden (derivations and
    citations inside each fixture)."""
    with open(os.path.join(GOLDEN, name)) as fh:
        g = json.load(fh)
    inp = {k: torch.tensor(v, dtype=torch.float32) for k, v in g["inputs"].items()}
    env = {"math": math}
    for k, expr in g.get("let", {}).items():
        env[k] = float(eval(expr, {"__builtins__": {}}, env))

    def mat(rows):
        return np.array([[float(e) if isinstance(e, (int, float))
                          else float(eval(e, {"__builtins__": {}}, env)) for e in row]
                         for row in rows])

    l2 = g.get("l2norm", False)
    pad = g.get("pad_mode", 0)
    cu = g.get("cu_seqlens", [0, inp["H"].shape[-2]])
    H = inp["H"].reshape(-1, inp["H"].shape[-1])
    X0 = inp["X0"].reshape(H.shape)
    W0 = inp["W_down0"]
    O = np.zeros((H.shape[0], inp["W_target"].shape[0]))
    V = np.zeros_like(O)
    states = []
    w64 = chunked.weights64(inp)
    for k, (a, b) in enumerate(zip(cu, cu[1:])):
        doc = []
        for c in chunked.walk_sequence(H[a:b], X0[a:b], None, None,
                                       W0[k] if W0.ndim == 3 else W0, None, inp["conv_w"],
                                       g["eta"], g["chunk"], pad, l2norm=l2, want_final=True,
                                       weights64=w64):
            O[a + c["lo"]:a + c["hi"]] = c["O"]
            V[a + c["lo"]:a + c["hi"]] = c["Vhat"]
            doc.append(c["W"])
            if "W_next" in c:
                doc.append(c["W_next"])
        states.append(doc)
    np.testing.assert_allclose(O, mat(g["expected"]["O"]), rtol=1e-13, atol=1e-15)
    if "Vhat" in g["expected"]:
        np.testing.assert_allclose(V, mat(g["expected"]["Vhat"]), rtol=1e-14, atol=0)
    exp_states = g["expected"]["states"]
    if "cu_seqlens" not in g:
        exp_states = [exp_states]
    for k, doc in enumerate(exp_states):
        for i, st in enumerate(doc):
            np.testing.assert_allclose(states[k][i], mat(st), rtol=1e-13, atol=1e-15)


def test_chunked_eta_zero_is_plain_gated_mlp():
    """eta = 0: O = (SiLU(H Wg^T) * (H Wu^T)) W_down0^T (Method §1 eq. (1)),
    evaluated with torch fp64 library routines."""
    inp = make_inputs(2, 13, 5, 9, seed=8, round_bf16=False)
    got = chunked.forward(inp, 0.0, 4)["O"]
    t = {k: v.double() for k, v in inp.items()}
    ref = F.linear(F.silu(F.linear(t["H"], t["W_gate"])) * F.linear(t["H"], t["W_up"]),
                   t["W_down0"])
    close(got, ref.numpy(), rel=1e-13)


def test_chunked_conv_matches_library():
    """Conv1D(X0) W_target^T of Method §2 eq. (5) against torch conv1d
    (groups = d, padding 1) run per chunk, and on the whole sequence for
    sequence padding."""
    T, d, C = 19, 6, 5
    inp = make_inputs(1, T, d, 4, seed=9, round_bf16=False)
    X0, cw, Wt = inp["X0"][0].double(), inp["conv_w"].double(), inp["W_target"].double()
    for pad in (chunked.PAD_CHUNK, chunked.PAD_SEQUENCE):
        seg = C if pad == chunked.PAD_CHUNK else T
        parts = [F.conv1d(X0[s:s + seg].T[None], cw[:, None], padding=1, groups=d)[0].T
                 for s in range(0, T, seg)]
        ref = F.linear(torch.cat(parts), Wt).numpy()
        got = np.concatenate([c["Vhat"] for c in chunked.walk_sequence(
            inp["H"][0], inp["X0"][0], inp["W_gate"], inp["W_up"], inp["W_down0"],
            inp["W_target"], inp["conv_w"], 0.1, C, pad)])
        close(got, ref, rel=1e-13)


@pytest.mark.parametrize("pad", [0, 1])
def test_state_grid_equals_c_state_entries(pad):
    """The column-restricted prefix sum equals the C oracle's entry-wise
    state evaluator and the full walk's states."""
    T, d, f, C = 29, 7, 11, 6
    inp = make_inputs(1, T, d, f, seed=12, round_bf16=False)
    et = torch.rand(T, generator=torch.Generator().manual_seed(2)) + 0.5
    m, j = np.array([0, 3, 6]), np.array([1, 4, 10, 7])
    eta = 0.21
    grid = chunked.state_grid(inp["H"][0], inp["X0"][0], inp["W_gate"], inp["W_up"],
                              inp["W_down0"], inp["W_target"], inp["conv_w"], eta, C, m, j,
                              pad, eta_tok=et)
    mm, jj = np.meshgrid(m, j, indexing="ij")
    ref = oracle.state_entries(inp["H"][0], inp["X0"][0], inp["W_gate"], inp["W_up"],
                               inp["W_down0"], inp["W_target"], inp["conv_w"], eta, C,
                               mm.ravel(), jj.ravel(), pad, eta_tok=et)
    close(grid, ref.T.reshape(-1, len(m), len(j)))
    full = chunked.forward(inp, eta, C, pad, eta_tok=et[None])["states"][0]
    close(grid, full[:, m][:, :, j])
