"""Randomised property tests (hypothesis): the oracle's invariants over random
small shapes, chunk lengths that need not divide T, both padding modes and
random rates, and the host-side partition and planning rules over random
sizes.  Each property is something the In-Place TTT pages or the
mathematics fix, checked against the oracle's own sequential walk or
against a plain restatement:

  "[논문리뷰] In-Place Test-Time Training" Method §1 eq. (3)-(4) (apply then
  update), §2 eq. (6) (the update), §3 "Implementation Details" (the prefix
  form, causal padding, the reset per document).
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from chunk_wise_weight_gb300 import ittt  # noqa: E402
from chunk_wise_weight_gb300.inputs import make_inputs  # noqa: E402
from chunk_wise_weight_gb300.shard import sequence_span, shard_range  # noqa: E402

SETTINGS = settings(max_examples=30, deadline=None, derandomize=True)


@st.composite
def small_problem(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 14))
    d = draw(st.integers(1, 5))
    f = draw(st.integers(1, 6))
    C = draw(st.integers(1, 16))
    pad = draw(st.sampled_from([oracle.PAD_CHUNK, oracle.PAD_SEQUENCE]))
    eta = draw(st.floats(-1.0, 1.0, allow_nan=False, allow_subnormal=False))
    seed = draw(st.integers(0, 10_000))
    return B, T, d, f, C, pad, eta, seed


# --------------------------------------------------------------------------
# Oracle invariants
# --------------------------------------------------------------------------

@SETTINGS
@given(small_problem())
def test_prefix_and_dual_forms_equal_the_walk(prob):
    """The exclusive-prefix form (Method §3) and the dual expansion give the
    walk's outputs for any chunking, partial last chunk included."""
    B, T, d, f, C, pad, eta, seed = prob
    inp = make_inputs(B, T, d, f, seed)
    seq = oracle.forward(inp, eta, C, pad, want_states=True)
    pre = oracle.forward_prefix(inp, eta, C, pad, want_states=True)
    dual = oracle.forward_dual(inp, eta, C, pad)
    scale = max(1.0, float(np.abs(seq["O"]).max()))
    np.testing.assert_allclose(pre["O"], seq["O"], rtol=1e-10, atol=1e-11 * scale)
    np.testing.assert_allclose(pre["states"], seq["states"], rtol=1e-10, atol=1e-11 * scale)
    np.testing.assert_allclose(dual["O"], seq["O"], rtol=1e-10, atol=1e-11 * scale)


@SETTINGS
@given(small_problem(), st.data())
def test_perturbing_a_token_leaves_earlier_outputs_unchanged(prob, data):
    """Apply before update (eq. (3)-(4)) and causal padding: a change at
    token p changes no output before p, bit for bit."""
    B, T, d, f, C, pad, eta, seed = prob
    inp = make_inputs(B, T, d, f, seed)
    p = data.draw(st.integers(0, T - 1))
    which = data.draw(st.sampled_from(["H", "X0"]))
    base = oracle.forward(inp, eta, C, pad)["O"]
    pert = {k: v.clone() for k, v in inp.items()}
    pert[which][:, p] += 2.5
    new = oracle.forward(pert, eta, C, pad)["O"]
    np.testing.assert_array_equal(new[:, :p], base[:, :p])


@SETTINGS
@given(small_problem())
def test_outputs_are_affine_in_eta(prob):
    """The deltas depend on neither eta nor W (eq. (6)), so
    O(2e) - O(e) = O(e) - O(0)."""
    B, T, d, f, C, pad, eta, seed = prob
    inp = make_inputs(B, T, d, f, seed)
    o0, o1, o2 = (oracle.forward(inp, k * eta, C, pad)["O"] for k in (0, 1, 2))
    scale = max(1.0, float(np.abs(o2).max()))
    np.testing.assert_allclose(o2 - o1, o1 - o0, rtol=1e-9, atol=1e-11 * scale)


@SETTINGS
@given(small_problem(), st.data())
def test_packed_documents_equal_separate_runs(prob, data):
    """The state resets at every document boundary (Method §3): a packed row
    of documents gives each document's own single-sequence result."""
    _, T, d, f, C, pad, eta, seed = prob
    cuts = sorted(set(data.draw(st.lists(st.integers(1, T - 1), max_size=3)) if T > 1 else []))
    cu = [0] + cuts + [T]
    inp = make_inputs(1, T, d, f, seed)
    packed = np.asarray(oracle.forward_packed(inp, cu, eta, C, pad)["O"]).reshape(T, d)
    for a, b in zip(cu[:-1], cu[1:]):
        doc = dict(inp)
        doc["H"] = inp["H"][:, a:b]
        doc["X0"] = inp["X0"][:, a:b]
        alone = oracle.forward(doc, eta, C, pad)["O"][0]
        np.testing.assert_allclose(packed[a:b], alone, rtol=1e-12, atol=1e-13)


@SETTINGS
@given(small_problem(), st.data())
def test_constant_token_rates_scale_eta(prob, data):
    """A per-token rate weight that is the same c for every token is the
    scalar rate c * eta."""
    B, T, d, f, C, pad, eta, seed = prob
    c = data.draw(st.floats(0.0, 2.0, allow_nan=False, allow_subnormal=False))
    inp = make_inputs(B, T, d, f, seed)
    rated = oracle.forward(inp, eta, C, pad, eta_tok=np.full((B, T), c, np.float32))["O"]
    plain = oracle.forward(inp, float(np.float32(c)) * eta, C, pad)["O"]
    scale = max(1.0, float(np.abs(plain).max()))
    np.testing.assert_allclose(rated, plain, rtol=1e-9, atol=1e-11 * scale)


# --------------------------------------------------------------------------
# Host-side partition and planning rules
# --------------------------------------------------------------------------

@settings(max_examples=200, deadline=None, derandomize=True)
@given(st.integers(0, 10_000), st.integers(1, 64))
def test_shard_range_partitions_the_units(total, world):
    spans = [shard_range(total, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == total
    for (a, b), (c, _) in zip(spans, spans[1:]):
        assert b == c
    sizes = [b - a for a, b in spans]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1


@settings(max_examples=200, deadline=None, derandomize=True)
@given(st.integers(0, 5_000), st.integers(1, 700), st.integers(1, 16))
def test_sequence_spans_are_whole_chunks_in_order(T, chunk, world):
    spans = [sequence_span(T, chunk, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == T
    for (a, b), (c, _) in zip(spans, spans[1:]):
        assert b == c
    nonempty = [(a, b) for a, b in spans if b > a]
    for a, b in nonempty:
        assert a % chunk == 0
    for a, b in nonempty[:-1]:
        assert (b - a) % chunk == 0
    # no non-empty span after an empty one
    seen_empty = False
    for a, b in spans:
        if b == a:
            seen_empty = True
        else:
            assert not seen_empty


@settings(max_examples=300, deadline=None, derandomize=True)
@given(st.integers(1, 64), st.sampled_from([64, 128, 192, 256, 512, 1024, 2048]),
       st.integers(1, 64), st.sampled_from([64, 256, 1024, 2048, 2560, 4096]),
       st.sampled_from([256, 1024, 3072, 6144, 9728, 14336]))
def test_form_choice_follows_the_measured_rule(B, chunk, nchunks, d, f):
    """Unforced, the dual form exactly when it is allowed (two chunks or more
    of a multiple of 64 tokens) and T (d + f) < 2.5 d f; forcing flags win."""
    T = chunk * nchunks
    form = ittt.plan_form(B, T, d, f, chunk)
    want = ittt.FORM_DUAL if (nchunks >= 2 and 2 * T * (d + f) < 5 * d * f) \
        else ittt.FORM_PRIMAL
    assert form == want
    assert ittt.plan_form(B, T, d, f, chunk, primal=True) == ittt.FORM_PRIMAL
    # forced, the dual form takes any whole number of 64-multiple chunks
    assert ittt.plan_form(B, T, d, f, chunk, dual=True) == ittt.FORM_DUAL
