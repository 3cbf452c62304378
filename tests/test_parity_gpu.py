"""GPU path vs the fp64 oracle, through the C-ABI (libittt.so).

Tolerance (the layer's stated bar): relative Frobenius error <= 5e-3 and
max elementwise error <= 2e-2 * max|reference|, on the same seeded inputs
(bf16 values widened exactly for the oracle).  The same bar is applied to
each exported intermediate (Z, eta * Vhat, weight snapshots): they are bf16
roundings of exact values, so their error is about 1.5e-3 rms.

Small and ragged shapes are compared element by element over the whole
output here; the full-size workloads are compared whole in
test_parity_full_size.py.  Only a 262,144-token sequence is sampled: Z, Vhat
and first-chunk output rows entry by entry, the fast-weight state W_i at
every chunk boundary in every 256 x 256 block, and other output rows against
the identity O_[i] = Z_[i] W_i^T on the kernel's own bf16 operands.
"""
import numpy as np
import pytest
import torch

import oracle
from chunk_wise_weight_gb300 import config_inputs, ittt, make_inputs
from oracle import chunked

pytestmark = pytest.mark.gpu

REL_FRO = 5e-3
MAX_RATIO = 2e-2


def rel_fro(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_ratio(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def assert_parity(got, ref, what):
    rf, mr = rel_fro(got, ref), max_ratio(got, ref)
    print(f"parity {what}: rel_fro={rf:.3e} max_ratio={mr:.3e}")
    assert rf <= REL_FRO and mr <= MAX_RATIO, f"{what}: rel_fro={rf:.3e} max_ratio={mr:.3e}"


def to_device(inp, dev, w0_dtype=torch.bfloat16):
    g = {k: inp[k].to(dev, torch.bfloat16) for k in ("H", "X0", "W_gate", "W_up", "W_target")}
    g["W_down0"] = inp["W_down0"].to(dev, w0_dtype)
    g["conv_w"] = inp["conv_w"].to(dev, torch.float32)
    return g


def packed_slots(cu, C):
    """Snapshot slot of each packed document's first chunk, and the total."""
    base, g = [], 0
    for a, b in zip(cu, cu[1:]):
        base.append(g)
        g += -(-(b - a) // C)
    return base, g


def run(g, eta, C, *, pad_mode=0, out_dtype=torch.bfloat16, intermediates=False,
        state_in=None, want_state=False, fused_conv=False, dual=False, eta_tok=None,
        cu_seqlens=None, l2norm=False, single_cta=False):
    B, T, d = g["H"].shape
    f = g["W_gate"].shape[0]
    dev = g["H"].device
    if cu_seqlens is None:
        states, slots = B, -(-T // C)
    else:
        states, slots = len(cu_seqlens) - 1, packed_slots(cu_seqlens, C)[1]
    kw = {}
    if intermediates:
        kw["z_buf"] = torch.empty(B, T, f, dtype=torch.bfloat16, device=dev)
        kw["vhat_buf"] = torch.empty(B, T, d, dtype=torch.bfloat16, device=dev)
        if not dual:
            kw["snap_buf"] = torch.empty(B, slots, d, f, dtype=torch.bfloat16, device=dev)
    if want_state:
        kw["state_out"] = torch.empty(states, d, f, dtype=torch.float32, device=dev)
    if state_in is not None:
        kw["state_in"] = state_in
    out = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"],
                       None if state_in is not None else g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C, out_dtype=out_dtype, pad_mode=pad_mode,
                       fused_conv=fused_conv, dual=dual, eta_tok=eta_tok,
                       cu_seqlens=cu_seqlens, l2norm=l2norm, single_cta=single_cta, **kw)
    ittt.stream_status()
    res = {"O": out}
    res.update(kw)
    return res


def host(t):
    return t.detach().float().cpu().double().numpy()


# --------------------------------------------------------------------------
# Whole-output parity at sizes the oracle finishes in seconds
# --------------------------------------------------------------------------

SHAPES = [
    # B, T, d, f, C, eta
    (1, 256, 64, 256, 64, 0.05),     # the tiny named workload's shape
    (2, 512, 200, 584, 128, 0.05),   # ragged d (partial N tile) and f (odd pair)
    (1, 1024, 320, 1000, 256, 0.02), # several K blocks, ragged K tail in apply
    (3, 384, 136, 264, 192, 0.1),    # chunk not a multiple of the 128-row tile
    (1, 256, 64, 256, 256, 0.3),     # one chunk: no update at all
    (2, 640, 72, 136, 320, 0.07),    # tiny d and f, two chunks
]


@pytest.mark.parametrize("B,T,d,f,C,eta", SHAPES)
def test_full_parity_with_intermediates(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=100 + T + d)
    ref = oracle.forward(inp, eta, C, want_z=True, want_vhat=True, want_states=True)
    got = run(to_device(inp, cuda_device), eta, C, intermediates=True)
    assert_parity(host(got["z_buf"]), ref["Z"], "Z")
    assert_parity(host(got["vhat_buf"]), eta * ref["Vhat"], "eta * Vhat")
    n = T // C
    assert_parity(host(got["snap_buf"]), ref["states"][:, :n], "snapshots W_0..W_{n-1}")
    assert_parity(host(got["O"]), ref["O"], "O")


def test_tiny_named_workload(cuda_device):
    cfg, inp = config_inputs(0)
    ref = oracle.forward(inp, cfg["eta"], cfg["C"])
    got = run(to_device(inp, cuda_device), cfg["eta"], cfg["C"])
    assert_parity(host(got["O"]), ref["O"], "O")
    # Information only: error against the oracle on the unrounded fp32 inputs.
    _, raw = config_inputs(0, round_bf16=False)
    raw_ref = oracle.forward(raw, cfg["eta"], cfg["C"])
    print(f"vs unrounded fp32 inputs: rel_fro={rel_fro(host(got['O']), raw_ref['O']):.3e}")


@pytest.mark.parametrize("fused_conv", [False, True])
@pytest.mark.parametrize("pad_mode", [ittt.PAD_CHUNK, ittt.PAD_SEQUENCE])
def test_pad_modes(cuda_device, pad_mode, fused_conv):
    B, T, d, f, C, eta = 2, 512, 200, 384, 128, 0.05
    inp = make_inputs(B, T, d, f, seed=7)
    ref = oracle.forward(inp, eta, C, pad_mode=pad_mode, want_vhat=True)
    got = run(to_device(inp, cuda_device), eta, C, pad_mode=pad_mode, intermediates=True,
              fused_conv=fused_conv)
    assert_parity(host(got["vhat_buf"]), eta * ref["Vhat"], "eta * Vhat")
    assert_parity(host(got["O"]), ref["O"], "O")


@pytest.mark.parametrize("B,T,d,f,C,eta", SHAPES[:4])
def test_fused_and_split_conv_agree_bitwise(cuda_device, B, T, d, f, C, eta):
    """Both convolution variants round the same fp32 taps once: identical
    eta * Vhat and O."""
    g = to_device(make_inputs(B, T, d, f, seed=300 + d), cuda_device)
    a = run(g, eta, C, intermediates=True)
    b = run(g, eta, C, intermediates=True, fused_conv=True)
    assert torch.equal(a["vhat_buf"], b["vhat_buf"])
    assert torch.equal(a["O"], b["O"])


def test_fp32_output_and_fp32_initial_weight(cuda_device):
    B, T, d, f, C, eta = 1, 512, 192, 320, 128, 0.05
    inp = make_inputs(B, T, d, f, seed=8)
    inp["W_down0"] = inp["W_down0"] * 1.0  # fp32 values, not bf16-representable below
    inp["W_down0"] += torch.randn(d, f, generator=torch.Generator().manual_seed(3)) * 1e-4
    ref = oracle.forward(inp, eta, C, want_states=True)
    g = to_device(inp, cuda_device, w0_dtype=torch.float32)
    got = run(g, eta, C, out_dtype=torch.float32, intermediates=True)
    assert got["O"].dtype == torch.float32
    assert_parity(host(got["O"]), ref["O"], "O (fp32 out)")
    assert_parity(host(got["snap_buf"]), ref["states"][:, :T // C], "snapshots")


def test_state_out_and_streaming_continuation(cuda_device):
    """state_out returns W_n (after the last chunk's update); feeding it back
    as state_in continues the sequence exactly where it stopped (chunk-edge
    padding makes the split at a chunk boundary exact)."""
    B, T, d, f, C, eta = 2, 1024, 128, 256, 128, 0.03
    inp = make_inputs(B, T, d, f, seed=9)
    ref = oracle.forward(inp, eta, C, want_states=True)
    g = to_device(inp, cuda_device)
    half = T // 2
    first = {k: (v[:, :half].contiguous() if k in ("H", "X0") else v) for k, v in g.items()}
    second = {k: (v[:, half:].contiguous() if k in ("H", "X0") else v) for k, v in g.items()}
    a = run(first, eta, C, want_state=True)
    assert_parity(host(a["state_out"]), ref["states"][:, half // C], "state after first half")
    b = run(second, eta, C, state_in=a["state_out"], want_state=True)
    assert_parity(host(b["state_out"]), ref["states"][:, T // C], "final state")
    O = np.concatenate([host(a["O"]), host(b["O"])], axis=1)
    assert_parity(O, ref["O"], "O across two calls")


# --------------------------------------------------------------------------
# Partial last chunk and per-token learning rates
# --------------------------------------------------------------------------

PARTIAL = [
    # B, T, d, f, C, eta: the last chunk is the remainder T - (n-1) C
    (1, 640, 200, 584, 256, 0.05),   # chunks 256, 256, 128
    (2, 448, 136, 264, 192, 0.1),    # 192, 192, 64 (row tiles straddle chunks)
    (1, 192, 64, 256, 128, 0.2),     # 128, 64
    (2, 128, 72, 136, 256, 0.3),     # one partial chunk shorter than C
]


@pytest.mark.parametrize("B,T,d,f,C,eta", PARTIAL)
def test_partial_last_chunk(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=700 + T + d)
    ref = oracle.forward(inp, eta, C, want_z=True, want_vhat=True, want_states=True)
    got = run(to_device(inp, cuda_device), eta, C, intermediates=True, want_state=True)
    n = -(-T // C)
    assert_parity(host(got["vhat_buf"]), eta * ref["Vhat"], "eta * Vhat")
    assert_parity(host(got["snap_buf"]), ref["states"][:, :n], "snapshots")
    assert_parity(host(got["state_out"]), ref["states"][:, n], "state after the partial chunk")
    assert_parity(host(got["O"]), ref["O"], "O")


@pytest.mark.parametrize("fused_conv,dual", [(False, False), (True, False), (False, True)])
def test_per_token_rates(cuda_device, fused_conv, dual):
    B, T, d, f, C, eta = 2, 512, 200, 384, 128, 0.1
    inp = make_inputs(B, T, d, f, seed=801)
    rates = torch.rand(B, T, generator=torch.Generator().manual_seed(4)) + 0.25
    rates[0, 130:200] = 0.0
    ref = oracle.forward(inp, eta, C, want_vhat=True, want_states=True, eta_tok=rates)
    got = run(to_device(inp, cuda_device), eta, C, intermediates=True, fused_conv=fused_conv,
              dual=dual, eta_tok=rates.to(cuda_device))
    scaled = eta * rates.double().numpy()[:, :, None] * ref["Vhat"]
    assert_parity(host(got["vhat_buf"]), scaled, "eta * eta_tok * Vhat")
    if not dual:
        assert_parity(host(got["snap_buf"]), ref["states"][:, :T // C], "snapshots")
    assert_parity(host(got["O"]), ref["O"], "O")


def test_chunk_mean_update_through_token_rates(cuda_device):
    """The 1/C-scaled update (eta times the chunk's mean of Vhat_t^T Z_t, a
    variant the pages mention beside per-token rates) is the per-token rate
    1 / (length of t's chunk): the last, shorter chunk is averaged over its
    own length.  Against the oracle with the same rates, and with full
    chunks against the plain update at eta / C."""
    B, T, d, f, C, eta = 2, 456, 128, 320, 128, 0.5     # chunks 128, 128, 128, 72
    inp = make_inputs(B, T, d, f, seed=802)
    t = torch.arange(T)
    start = (t // C) * C
    length = torch.clamp(T - start, max=C).float()
    rates = (1.0 / length).expand(B, T).contiguous()
    ref = oracle.forward(inp, eta, C, want_states=True, eta_tok=rates)
    got = run(to_device(inp, cuda_device), eta, C, want_state=True, eta_tok=rates.to(cuda_device))
    assert_parity(host(got["O"]), ref["O"], "O (chunk-mean update)")
    assert_parity(host(got["state_out"]), ref["states"][:, -1], "final state (chunk-mean update)")
    full = oracle.forward(inp, eta / C, C, want_states=True)
    np.testing.assert_allclose(ref["states"][:, T // C], full["states"][:, T // C],
                               rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("B,T,d,f,C,eta", SHAPES[:4])
def test_single_cta_kernels(cuda_device, B, T, d, f, C, eta):
    """The single-CTA GEMMs (the fallback where CTA pairs cannot be resident)
    against the oracle, and against the default CTA-pair path."""
    inp = make_inputs(B, T, d, f, seed=1500 + T + d)
    ref = oracle.forward(inp, eta, C, want_states=True)
    g = to_device(inp, cuda_device)
    one = run(g, eta, C, intermediates=True, single_cta=True)
    assert_parity(host(one["snap_buf"]), ref["states"][:, :T // C], "snapshots (single CTA)")
    assert_parity(host(one["O"]), ref["O"], "O (single CTA)")
    # Same K order and fp32 accumulation: the two paths agree bit for bit.
    pair = run(g, eta, C, intermediates=True)
    for k in ("z_buf", "vhat_buf", "snap_buf", "O"):
        assert torch.equal(one[k], pair[k]), k


def test_apply_split_last_round(cuda_device):
    """The apply on CTA pairs runs a partial last round of t units (after at
    least two full rounds, 2t <= 76 pairs) as pieces over disjoint K ranges
    whose fp32 partials the last piece adds in piece order.  Here 160
    units (one 256-row tile per 256-token chunk, d = 256): the last 8 units
    (chunks 152..159) run as 4 pieces each.  Everything outside those chunks
    is bit-identical to the single-CTA path; inside, O differs from it only
    by the fp32 rounding of the other summation order, and the whole output
    is within the bar of the oracle."""
    B, T, d, f, C, eta = 1, 160 * 256, 256, 1024, 256, 0.02
    inp = make_inputs(B, T, d, f, seed=1777)
    ref = oracle.forward(inp, eta, C)
    g = to_device(inp, cuda_device)
    assert ittt.plan_form(B, T, d, f, C) == ittt.FORM_PRIMAL
    pair = run(g, eta, C)
    one = run(g, eta, C, single_cta=True)
    assert_parity(host(pair["O"]), ref["O"], "O (split last round)")
    split0 = 152 * 256
    assert torch.equal(pair["O"][:, :split0], one["O"][:, :split0])
    # Inside: the same products summed in another fp32 order, so the bf16
    # results differ by at most one unit in the last place -- where O is
    # not much smaller than its terms (elsewhere by an fp32 rounding of
    # the terms' scale, 2^-14 of max |O| bounds it here).
    a = pair["O"][:, split0:].double()
    b = one["O"][:, split0:].double()
    ulp = torch.exp2(torch.floor(torch.log2(b.abs().clamp_min(1e-30))) - 7)
    bound = ulp + 2.0 ** -14 * b.abs().max()
    err = (a - b).abs() - bound
    worst = int(torch.argmax(err))
    assert bool((err <= 0).all()), (
        f"split tiles: element {worst} pair {a.flatten()[worst].item()!r} "
        f"single {b.flatten()[worst].item()!r}")


# --------------------------------------------------------------------------
# Chunks and lengths that are not multiples of 64: the update masks the
# token lines past a chunk's end, the apply stores ragged tiles row by row
# --------------------------------------------------------------------------

RAGGED = [
    # B, T, d, f, C, eta
    (1, 250, 64, 256, 100, 0.05),    # chunks 100, 100, 50; T not a multiple of 64
    (2, 200, 72, 136, 48, 0.07),     # every chunk ends inside a 64-token stage
    (1, 77, 200, 584, 13, 0.03),     # 13-token chunks (one 16-token slice each)
    (2, 70, 64, 128, 1, 0.02),       # one token per chunk: per-token updates
    (1, 333, 136, 264, 160, 0.1),    # chunks 160, 160, 13
]


@pytest.mark.parametrize("B,T,d,f,C,eta", RAGGED)
def test_ragged_chunks(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=900 + T + C)
    ref = oracle.forward(inp, eta, C, want_z=True, want_vhat=True, want_states=True)
    got = run(to_device(inp, cuda_device), eta, C, intermediates=True, want_state=True)
    n = -(-T // C)
    assert_parity(host(got["z_buf"]), ref["Z"], "Z")
    assert_parity(host(got["vhat_buf"]), eta * ref["Vhat"], "eta * Vhat")
    assert_parity(host(got["snap_buf"]), ref["states"][:, :n], "snapshots")
    assert_parity(host(got["state_out"]), ref["states"][:, n], "final state")
    assert_parity(host(got["O"]), ref["O"], "O")
    o32 = run(to_device(inp, cuda_device), eta, C, out_dtype=torch.float32)["O"]
    assert_parity(host(o32), ref["O"], "O (fp32 out)")


EDGE = [
    # B, T, d, f, C, eta
    (1, 100, 8, 8, 7, 0.1),        # smallest widths: every TMA box exceeds its tensor
    (2, 33, 16, 24, 64, 0.2),      # chunk longer than the sequence: one partial chunk
    (3, 1, 64, 128, 1, 0.3),       # one token per sequence
    (1, 130, 24, 40, 2, 0.05),     # two-token chunks, widths below one 64-column box
]


@pytest.mark.parametrize("B,T,d,f,C,eta", EDGE)
def test_edge_shapes(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=1300 + T + d)
    ref = oracle.forward(inp, eta, C, want_states=True)
    got = run(to_device(inp, cuda_device), eta, C, want_state=True, intermediates=True)
    n = -(-T // C)
    assert_parity(host(got["snap_buf"]), ref["states"][:, :n], "snapshots")
    assert_parity(host(got["state_out"]), ref["states"][:, n], "final state")
    assert_parity(host(got["O"]), ref["O"], "O")
    # the default call (no snapshot buffer: W_0 read directly for chunk 0)
    plain = run(to_device(inp, cuda_device), eta, C)["O"]
    assert_parity(host(plain), ref["O"], "O (default call)")


def test_long_chunk_single_sequence(cuda_device):
    """A 2^17-token chunk: one chunk, O = Z W_0^T; the final state from one
    long contraction (sampled entries against the oracle)."""
    T, d, f, eta = 1 << 17, 64, 128, 1e-4
    inp = make_inputs(1, T, d, f, seed=1400)
    g = to_device(inp, cuda_device)
    got = run(g, eta, T, want_state=True, intermediates=True)
    rows = np.array([0, 1, T // 2, T - 1])
    assert_parity(host(got["O"][0][torch.as_tensor(rows)]),
                  oracle.first_chunk_rows(inp["H"][0], inp["W_gate"], inp["W_up"],
                                          inp["W_down0"], rows), "O rows")
    m, j = np.array([0, 5, d - 1]), np.array([0, 77, f - 1])
    ws = oracle.state_entries(inp["H"][0], inp["X0"][0], inp["W_gate"], inp["W_up"],
                              inp["W_down0"], inp["W_target"], inp["conv_w"], eta, T, m, j)
    assert_parity(host(got["state_out"][0][torch.as_tensor(m), torch.as_tensor(j)]), ws[:, 1],
                  "final state entries")


# --------------------------------------------------------------------------
# Packed documents (state reset at each document boundary)
# --------------------------------------------------------------------------

PACKED = [
    # cu_seqlens, d, f, C, eta
    ([0, 100, 356, 600], 72, 136, 64, 0.05),
    ([0, 1, 65, 130, 400], 200, 584, 128, 0.05),
    ([0, 37, 300, 301, 555, 700, 948, 1000, 1200, 1290], 64, 256, 96, 0.03),
    ([0, 512, 1024], 128, 256, 256, 0.03),   # whole chunks only
]


def _packed_inputs(cu, d, f, seed):
    inp = make_inputs(1, cu[-1], d, f, seed=seed)
    return inp


@pytest.mark.parametrize("cu,d,f,C,eta", PACKED)
def test_packed_documents(cuda_device, cu, d, f, C, eta):
    inp = _packed_inputs(cu, d, f, seed=950 + len(cu) + d)
    ref = oracle.forward_packed(inp, cu, eta, C, want_z=True, want_vhat=True, want_states=True)
    got = run(to_device(inp, cuda_device), eta, C, intermediates=True, want_state=True,
              cu_seqlens=cu)
    assert_parity(host(got["z_buf"])[0], ref["Z"], "Z")
    assert_parity(host(got["vhat_buf"])[0], eta * ref["Vhat"], "eta * Vhat")
    base, slots = packed_slots(cu, C)
    snap = host(got["snap_buf"])[0]
    want = np.concatenate([s[:-1] for s in ref["states"]])      # W_0..W_{n_k - 1} per document
    assert snap.shape[0] == slots == want.shape[0]
    assert_parity(snap, want, "snapshots")
    assert_parity(host(got["state_out"]), np.stack([s[-1] for s in ref["states"]]),
                  "final states")
    assert_parity(host(got["O"])[0], ref["O"], "O")


def test_packed_document_options(cuda_device):
    """Per-document initial states, per-token rates, sequence padding and
    fp32 output together."""
    cu, d, f, C, eta = [0, 150, 151, 420, 640], 128, 256, 128, 0.05
    inp = _packed_inputs(cu, d, f, seed=977)
    nd = len(cu) - 1
    w0 = torch.stack([inp["W_down0"] * (1.0 - 0.3 * k) for k in range(nd)])
    rates = torch.rand(1, cu[-1], generator=torch.Generator().manual_seed(5)) + 0.5
    pk = dict(inp)
    pk["W_down0"] = w0
    ref = oracle.forward_packed(pk, cu, eta, C, pad_mode=oracle.PAD_SEQUENCE, want_states=True,
                                eta_tok=rates)
    g = to_device(inp, cuda_device)
    got = run(g, eta, C, pad_mode=ittt.PAD_SEQUENCE, out_dtype=torch.float32,
              state_in=w0.to(cuda_device).contiguous(), want_state=True,
              eta_tok=rates.to(cuda_device), cu_seqlens=cu)
    assert_parity(host(got["O"])[0], ref["O"], "O")
    assert_parity(host(got["state_out"]), np.stack([s[-1] for s in ref["states"]]),
                  "final states")


def test_packed_equals_separate_calls_bitwise(cuda_device):
    """Each packed document gives bit for bit what a call on that document
    alone gives (same kernels, same per-row reduction order)."""
    cu, d, f, C, eta = [0, 200, 264, 700], 128, 256, 128, 0.05
    g = to_device(_packed_inputs(cu, d, f, seed=978), cuda_device)
    full = run(g, eta, C, cu_seqlens=cu)["O"]
    for a, b in zip(cu, cu[1:]):
        one = {k: (v[:, a:b].contiguous() if k in ("H", "X0") else v) for k, v in g.items()}
        assert torch.equal(run(one, eta, C)["O"][0], full[0, a:b])


# --------------------------------------------------------------------------
# Fast-weight L2 normalisation (one launch per chunk)
# --------------------------------------------------------------------------

L2 = [
    # B, T, d, f, C, eta
    (1, 512, 64, 256, 128, 0.05),
    (2, 640, 200, 584, 256, 0.05),     # ragged d, odd 256-column blocks, partial chunk
    (1, 333, 136, 264, 100, 0.1),      # chunks that end inside a stage
    (3, 384, 136, 1000, 192, 0.02),
]


L2_PAIRS = [
    # d a multiple of 256 and every chunk a multiple of 64 tokens: a regular
    # batch runs the walk with the state in TMEM on CTA pairs
    (2, 640, 256, 584, 128, 0.05),     # three 256-column blocks, chunks 128 x 5
    (1, 512, 512, 1000, 256, 0.02),    # two 256-row blocks, ragged d_ff
    (3, 512, 256, 9728, 128, 0.05),    # 38 column blocks: two groups of 38 pairs, 2 rounds
]


@pytest.mark.parametrize("B,T,d,f,C,eta", L2_PAIRS)
def test_l2norm_pairs_parity_and_single_cta_bitwise(cuda_device, B, T, d, f, C, eta):
    """The walk with the state in TMEM (regular batch on CTA pairs) against
    the oracle, and bit for bit against the walk with the state in HBM on
    single CTAs and on CTA pairs (forced by packing the same sequences as
    documents): all three sum the same partial sums in the same order."""
    inp = make_inputs(B, T, d, f, seed=1150 + T + d)
    ref = oracle.forward(inp, eta, C, want_states=True, l2norm=True)
    g = to_device(inp, cuda_device)
    got = run(g, eta, C, intermediates=True, want_state=True, l2norm=True)
    n = -(-T // C)
    assert_parity(host(got["snap_buf"]), ref["states"][:, :n], "normalised snapshots")
    assert_parity(host(got["state_out"]), ref["states"][:, n], "normalised final state")
    assert_parity(host(got["O"]), ref["O"], "O")
    one = run(g, eta, C, intermediates=True, want_state=True, l2norm=True, single_cta=True)
    assert_parity(host(one["O"]), ref["O"], "O (state in HBM, single CTAs)")
    cu = [b * T for b in range(B + 1)]
    pk = {k: v.reshape(1, B * T, d) if k in ("H", "X0") else v for k, v in g.items()}
    packed = run(pk, eta, C, intermediates=True, want_state=True, l2norm=True, cu_seqlens=cu)
    assert torch.equal(packed["O"].reshape(B, T, d), one["O"])
    assert torch.equal(packed["state_out"], one["state_out"])
    assert torch.equal(packed["snap_buf"].reshape(B, n, d, f), one["snap_buf"])
    for k in ("snap_buf", "state_out", "O"):
        assert torch.equal(one[k], got[k]), k


@pytest.mark.parametrize("B,T,d,f,C,eta", L2)
def test_l2norm_parity(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=1100 + T + d)
    ref = oracle.forward(inp, eta, C, want_states=True, l2norm=True)
    got = run(to_device(inp, cuda_device), eta, C, intermediates=True, want_state=True,
              l2norm=True)
    n = -(-T // C)
    assert_parity(host(got["snap_buf"]), ref["states"][:, :n], "normalised snapshots")
    assert_parity(host(got["state_out"]), ref["states"][:, n], "normalised final state")
    assert_parity(host(got["O"]), ref["O"], "O")
    # without state_out the last snapshot comes from the finalising kernel
    got2 = run(to_device(inp, cuda_device), eta, C, intermediates=True, l2norm=True)
    assert torch.equal(got2["snap_buf"], got["snap_buf"])
    assert torch.equal(got2["O"], got["O"])


def test_l2norm_packed_with_options(cuda_device):
    """Packed documents, per-document initial states (fp32), per-token
    rates and fp32 output with the normalised walk."""
    cu, d, f, C, eta = [0, 150, 151, 420, 700], 128, 256, 128, 0.05
    inp = _packed_inputs(cu, d, f, seed=1177)
    nd = len(cu) - 1
    w0 = torch.stack([inp["W_down0"] * (1.0 + 0.5 * k) for k in range(nd)])
    rates = torch.rand(1, cu[-1], generator=torch.Generator().manual_seed(6)) + 0.5
    pk = dict(inp)
    pk["W_down0"] = w0
    ref = oracle.forward_packed(pk, cu, eta, C, want_states=True, eta_tok=rates, l2norm=True)
    g = to_device(inp, cuda_device)
    got = run(g, eta, C, out_dtype=torch.float32, state_in=w0.to(cuda_device).contiguous(),
              want_state=True, eta_tok=rates.to(cuda_device), cu_seqlens=cu, l2norm=True,
              intermediates=True)
    snaps = np.concatenate([s[:-1] for s in ref["states"]])
    assert_parity(host(got["snap_buf"])[0], snaps, "normalised snapshots")
    assert_parity(host(got["state_out"]), np.stack([s[-1] for s in ref["states"]]),
                  "normalised final states")
    assert_parity(host(got["O"])[0], ref["O"], "O")


# --------------------------------------------------------------------------
# The dual schedule (scores Z Z^T instead of the fast-weight walk)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("B,T,d,f,C,eta", SHAPES)
def test_dual_form_parity(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=500 + T + d)
    ref = oracle.forward(inp, eta, C)
    got = run(to_device(inp, cuda_device), eta, C, dual=True)
    assert_parity(host(got["O"]), ref["O"], "O (dual)")


@pytest.mark.parametrize("B,T,d,f,C,eta", [
    (3, 320, 192, 320, 64, 0.05),     # last 256-row tile half past T; d < 256
    (2, 960, 320, 448, 192, 0.02),    # 256-row tiles straddle 192-token chunk edges
    (2, 1024, 512, 640, 128, 0.03),
])
def test_dual_form_pairs_match_single_cta(cuda_device, B, T, d, f, C, eta):
    """The dual apply on CTA pairs (256-row tiles sharing one scores range)
    against the oracle and against the single-CTA kernel: the extra scores
    a pair tile reads for its earlier rows are zeros, so both sum the same
    products in the same order."""
    inp = make_inputs(B, T, d, f, seed=900 + T + d)
    ref = oracle.forward(inp, eta, C)
    g = to_device(inp, cuda_device)
    pair = run(g, eta, C, dual=True)
    one = run(g, eta, C, dual=True, single_cta=True)
    assert_parity(host(pair["O"]), ref["O"], "O (dual, CTA pairs)")
    assert_parity(host(one["O"]), ref["O"], "O (dual, single CTA)")
    assert torch.equal(pair["O"], one["O"])


def test_dual_form_variants(cuda_device):
    """fp32 output, fp32 W_0, per-sequence initial state, fused conv."""
    B, T, d, f, C, eta = 2, 512, 192, 320, 128, 0.05
    inp = make_inputs(B, T, d, f, seed=17)
    ref = oracle.forward(inp, eta, C)
    g = to_device(inp, cuda_device, w0_dtype=torch.float32)
    got = run(g, eta, C, dual=True, out_dtype=torch.float32, fused_conv=True)
    assert_parity(host(got["O"]), ref["O"], "O (dual, fp32 out, fp32 W_0, fused conv)")
    st = torch.stack([g["W_down0"], -g["W_down0"]]).contiguous()
    binp = dict(inp)
    binp["W_down0"] = torch.stack([inp["W_down0"], -inp["W_down0"]])
    ref2 = oracle.forward(binp, eta, C)
    got2 = run(g, eta, C, dual=True, state_in=st)
    assert_parity(host(got2["O"]), ref2["O"], "O (dual, per-sequence W_0)")
    got3 = run(g, eta, C, state_in=st)
    assert_parity(host(got3["O"]), ref2["O"], "O (primal, per-sequence W_0)")


def test_dual_form_rejects_state_outputs(cuda_device):
    g = to_device(make_inputs(1, 256, 64, 256, seed=18), cuda_device)
    with pytest.raises(ittt.IttError) as e:
        run(g, 0.1, 64, dual=True, want_state=True)
    assert e.value.status == ittt.ERR_UNSUPPORTED


# --------------------------------------------------------------------------
# Structural properties, bit-exact on the GPU path
# --------------------------------------------------------------------------

def test_deterministic_and_plain_entry_point_identical(cuda_device):
    B, T, d, f, C, eta = 2, 512, 256, 512, 128, 0.05
    g = to_device(make_inputs(B, T, d, f, seed=10), cuda_device)
    o1 = run(g, eta, C)["O"]
    o2 = run(g, eta, C, intermediates=True)["O"]
    o3 = torch.empty_like(o1)
    ittt.forward_plain(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C, o3)
    ittt.stream_status()
    assert torch.equal(o1, o2) and torch.equal(o1, o3)


@pytest.mark.parametrize("which", ["H", "X0"])
@pytest.mark.parametrize("p", [0, 200, 255, 256, 511])
def test_causality_bitwise(cuda_device, which, p):
    """Changing H or X0 at token p leaves every output row t < p unchanged."""
    B, T, d, f, C, eta = 1, 768, 128, 256, 256, 0.05
    inp = make_inputs(B, T, d, f, seed=11)
    g = to_device(inp, cuda_device)
    base = run(g, eta, C)["O"]
    g2 = dict(g)
    g2[which] = g[which].clone()
    g2[which][0, p] += 2.0
    new = run(g2, eta, C)["O"]
    assert torch.equal(new[0, :p], base[0, :p])
    assert not torch.equal(new[0, p:], base[0, p:])


def test_batch_rows_independent_bitwise(cuda_device):
    B, T, d, f, C, eta = 3, 512, 128, 256, 128, 0.05
    g = to_device(make_inputs(B, T, d, f, seed=12), cuda_device)
    full = run(g, eta, C)["O"]
    for b in range(B):
        one = {k: (v[b:b + 1].contiguous() if k in ("H", "X0") else v) for k, v in g.items()}
        assert torch.equal(run(one, eta, C)["O"][0], full[b])


def test_eta_zero_is_gated_mlp(cuda_device):
    B, T, d, f, C = 1, 512, 128, 384, 128
    inp = make_inputs(B, T, d, f, seed=13)
    ref = oracle.forward(inp, 0.0, C)
    got = run(to_device(inp, cuda_device), 0.0, C)
    assert_parity(host(got["O"]), ref["O"], "O (eta = 0)")


def test_status_and_argument_errors_on_device(cuda_device):
    g = to_device(make_inputs(1, 256, 64, 256, seed=14), cuda_device)
    with pytest.raises(ittt.IttError) as e:
        ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                     g["conv_w"], 0.1, 0)
    assert e.value.status == ittt.ERR_INVALID_ARG
    with pytest.raises(ittt.IttError) as e:   # the fused conv needs 64-token multiples
        ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                     g["conv_w"], 0.1, 100, fused_conv=True)
    assert e.value.status == ittt.ERR_UNSUPPORTED
    ittt.stream_status()  # nothing recorded


def test_bounded_wait_times_out_and_context_survives(cuda_device):
    """A wait that nothing completes runs out after its limit: the kernel
    records the timeout, its other warp unwinds on the abort flag (the whole
    kernel lasts about one limit, not the other warp's four), the host reads
    ITTT_ERR_TIMEOUT once, and the library keeps working afterwards."""
    limit_ns = 20_000_000
    stream = torch.cuda.current_stream(cuda_device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    ittt.check_wait_timeout(limit_ns, stream)
    t1.record(stream)
    with pytest.raises(ittt.IttError) as e:
        ittt.stream_status(stream)
    assert e.value.status == ittt.ERR_TIMEOUT
    assert "bounded wait" in str(e.value)
    ms = t0.elapsed_time(t1)
    assert 0.9 * limit_ns / 1e6 <= ms < 2.5 * limit_ns / 1e6, ms
    ittt.stream_status(stream)  # the record was cleared
    B, T, d, f, C, eta = 1, 256, 64, 256, 64, 0.05
    inp = make_inputs(B, T, d, f, seed=19)
    got = run(to_device(inp, cuda_device), eta, C)
    assert_parity(host(got["O"]), oracle.forward(inp, eta, C)["O"], "O after a timeout")


# --------------------------------------------------------------------------
# Full-size named workloads: sampled entries against the oracle
# --------------------------------------------------------------------------

def _stratified(size, block, rng):
    """One random index inside every block of `block` consecutive indices."""
    starts = np.arange(0, size, block)
    return np.array([s + rng.integers(0, min(block, size - s)) for s in starts])


def _rows_differing(a, b):
    rows = (a != b).reshape(-1, a.shape[-1]).any(dim=1).nonzero().flatten()
    return f"{len(rows)} rows (first {rows[:6].tolist()})"


def _report_mismatch(g, eta, C, got, plain):
    """The plain call and the exporting call must agree bit for bit; when
    they do not, run both again and say which call and which stage was off
    before failing."""
    again = run(g, eta, C, intermediates=True)
    plain2 = torch.empty_like(plain)
    ittt.forward_plain(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C, plain2)
    ittt.stream_status()
    lines = [f"O plain vs export: {_rows_differing(plain, got['O'])}",
             f"O plain vs plain again: {_rows_differing(plain, plain2)}",
             f"O export vs export again: {_rows_differing(got['O'], again['O'])}",
             f"O plain again vs export again: {_rows_differing(plain2, again['O'])}"]
    for k in ("z_buf", "vhat_buf", "snap_buf"):
        lines.append(f"{k} export vs export again: {_rows_differing(got[k], again[k])}")
    pytest.fail("plain and exporting calls differ:\n  " + "\n  ".join(lines))


def _sampled_checks(index, device, dual=False, shape=None):
    """Sampled checks for sequences too long for a whole-output comparison.

    The fast-weight state is checked at every chunk boundary in every
    256 x 256 block of the [d, f] state: one row m per 256-row block and one
    column j per 256-column block (random offsets), all combinations, from
    the oracle's column-restricted prefix sum.  Z and eta * Vhat are sampled
    at chunk edges and at random; first-chunk output rows come from the
    oracle, later rows from the identity O_[i] = Z_[i] W_i^T on the kernel's
    own bf16 operands (a second, self-consistency check).
    """
    if shape is None:
        cfg, inp = config_inputs(index)
    else:
        B, T, d, f, C, eta = shape
        cfg = dict(B=B, T=T, d=d, f=f, C=C, eta=eta)
        inp = make_inputs(B, T, d, f, seed=index)
    B, T, d, f, C, eta = cfg["B"], cfg["T"], cfg["d"], cfg["f"], cfg["C"], cfg["eta"]
    n = T // C
    g = to_device(inp, device)
    got = run(g, eta, C, intermediates=True)
    plain = torch.empty_like(got["O"])
    ittt.forward_plain(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C, plain)
    ittt.stream_status()
    assert ittt.plan_form(B, T, d, f, C) == ittt.FORM_PRIMAL
    if not torch.equal(plain, got["O"]):
        _report_mismatch(g, eta, C, got, plain)
    rng = np.random.default_rng(1000 + index)
    for b in sorted({0, B - 1}):
        H, X0 = inp["H"][b], inp["X0"][b]
        # tokens at chunk edges and at random
        t = np.concatenate([[0, C - 1, C, T - 1], rng.integers(0, T, 60)])
        j = np.concatenate([[0, f - 1, f // 2, 1], rng.integers(0, f, 60)])
        m = np.concatenate([[0, d - 1, d // 2, 1], rng.integers(0, d, 60)])
        zg = host(got["z_buf"][b][torch.as_tensor(t), torch.as_tensor(j)])
        assert_parity(zg, oracle.z_entries(H, inp["W_gate"], inp["W_up"], t, j), f"Z[b={b}]")
        vg = host(got["vhat_buf"][b][torch.as_tensor(t), torch.as_tensor(m)])
        assert_parity(vg, eta * oracle.vhat_entries(X0, inp["conv_w"], inp["W_target"], C, t, m),
                      f"eta * Vhat[b={b}]")
        # fast-weight state: one entry in every 256 x 256 block, every boundary
        sm, sj = _stratified(d, 256, rng), _stratified(f, 256, rng)
        ws = chunked.state_grid(H, X0, inp["W_gate"], inp["W_up"], inp["W_down0"],
                                inp["W_target"], inp["conv_w"], eta, C, sm, sj)
        sg = host(got["snap_buf"][b][:, torch.as_tensor(sm)][:, :, torch.as_tensor(sj)])
        for i in range(n):
            assert_parity(sg[i], ws[i], f"snapshot {i} blocks [b={b}]")
        # first-chunk output rows, exactly from the oracle
        rows = np.array([0, 1, C // 2, C - 1])
        og = host(got["O"][b][torch.as_tensor(rows)])
        assert_parity(og, oracle.first_chunk_rows(H, inp["W_gate"], inp["W_up"],
                                                  inp["W_down0"], rows), f"O chunk 0 [b={b}]")
        # later rows: O_[i] = Z_[i] W_i^T on the kernel's own bf16 operands
        for tok in (C, T // 2 + 3, T - 1):
            i = tok // C
            z = host(got["z_buf"][b][tok])
            w = host(got["snap_buf"][b][i])
            assert_parity(host(got["O"][b][tok]), w @ z, f"O row {tok} [b={b}]")


def test_longest_sequence_sampled(cuda_device):
    """262,144 tokens in one sequence (64 chunks of 4096; Z alone is 5 GB and
    T * d_ff exceeds 2^31 elements): too long for a whole-output comparison
    (the named workloads and other widths are compared whole in
    test_parity_full_size.py), so the sampled checks above."""
    _sampled_checks(1700, cuda_device, shape=(1, 262144, 2560, 9728, 4096, 0.005))


# --------------------------------------------------------------------------
# Sequence sharding: folding a span (ITTT_FLAG_UPDATE_ONLY), the exclusive
# prefix of the spans' deltas (ittt_state_prefix), and the apply that reuses
# Z and eta * Vhat (ITTT_FLAG_REUSE_ZV); ranks emulated one after another
# on this GPU (no kernel waits on another)
# --------------------------------------------------------------------------

FOLD = [
    # B, T, d, f, C, eta
    (2, 512, 200, 584, 128, 0.05),   # CTA pairs: T a multiple of 64
    (1, 333, 136, 264, 160, 0.1),    # ragged T: single-CTA walk with masked K tail
    (3, 384, 64, 256, 384, 0.2),     # one chunk
]


@pytest.mark.parametrize("B,T,d,f,C,eta", FOLD)
def test_update_only_folds_every_chunk(cuda_device, B, T, d, f, C, eta):
    inp = make_inputs(B, T, d, f, seed=1800 + T)
    g = to_device(inp, cuda_device)
    rates = torch.rand(B, T, generator=torch.Generator().manual_seed(6)) + 0.5
    ref = oracle.forward(inp, eta, C, want_states=True, eta_tok=rates)
    zero = dict(inp, W_down0=torch.zeros(d, f))
    delta_ref = oracle.forward(zero, eta, C, want_states=True, eta_tok=rates)["states"][:, -1]
    start = torch.randn(B, d, f, generator=torch.Generator().manual_seed(7)) * 0.02
    start_ref = oracle.forward(dict(inp, W_down0=start), eta, C, want_states=True,
                               eta_tok=rates)["states"][:, -1]
    et = rates.to(cuda_device)
    plain = run(g, eta, C, intermediates=True, eta_tok=et)
    for w0, state_in, want in ((None, None, delta_ref), (g["W_down0"], None, ref["states"][:, -1]),
                               (None, start.to(cuda_device), start_ref)):
        st = torch.empty(B, d, f, dtype=torch.float32, device=cuda_device)
        z = torch.empty_like(plain["z_buf"])
        vh = torch.empty_like(plain["vhat_buf"])
        res = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], w0, g["W_target"],
                           g["conv_w"], eta, C, update_only=True, state_in=state_in,
                           state_out=st, z_buf=z, vhat_buf=vh, eta_tok=et)
        ittt.stream_status()
        assert res is None
        assert_parity(host(st), want, "folded state")
        # the producers are the forward's own: identical Z and eta * Vhat
        assert torch.equal(z, plain["z_buf"]) and torch.equal(vh, plain["vhat_buf"])


def test_update_only_packed_documents(cuda_device):
    cu = [0, 100, 356, 512]
    d, f, C, eta = 136, 264, 64, 0.05
    inp = make_inputs(1, 512, d, f, seed=1810)
    zero = dict(inp, W_down0=torch.zeros(d, f))
    ref = oracle.forward_packed(zero, cu, eta, C, want_states=True)
    g = to_device(inp, cuda_device)
    st = torch.empty(3, d, f, dtype=torch.float32, device=cuda_device)
    ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], None, g["W_target"], g["conv_w"],
                 eta, C, update_only=True, state_out=st, cu_seqlens=cu)
    ittt.stream_status()
    for k in range(3):
        assert_parity(host(st[k]), ref["states"][k][-1], f"document {k} folded")


@pytest.mark.parametrize("B,T,d,f,C,eta", SHAPES[:4] + [RAGGED[0]])
def test_reuse_zv_is_bitwise_the_forward(cuda_device, B, T, d, f, C, eta):
    """Given the Z and eta * Vhat a forward produced, the reusing call walks
    and applies the same operands: identical snapshots and output."""
    g = to_device(make_inputs(B, T, d, f, seed=1820 + T), cuda_device)
    a = run(g, eta, C, intermediates=True, want_state=True)
    snap = torch.empty_like(a["snap_buf"])
    st = torch.empty_like(a["state_out"])
    # the reusing call must not read H, X0 or the producer weights: poison them
    poisoned = {k: (torch.full_like(v, float("nan")) if k in ("H", "X0", "W_gate", "W_up",
                                                               "W_target", "conv_w") else v)
                for k, v in g.items()}
    O = ittt.forward(poisoned["H"], poisoned["X0"], poisoned["W_gate"], poisoned["W_up"],
                     g["W_down0"], poisoned["W_target"], poisoned["conv_w"], eta, C,
                     reuse_zv=True, z_buf=a["z_buf"], vhat_buf=a["vhat_buf"], snap_buf=snap,
                     state_out=st)
    ittt.stream_status()
    assert torch.equal(snap, a["snap_buf"])
    assert torch.equal(st, a["state_out"])
    assert torch.equal(O, a["O"])


@pytest.mark.parametrize("start", ["none", "bf16", "fp32", "per_state"])
def test_state_prefix_sums_in_order(cuda_device, start):
    """fp32 W_start + deltas[0] + ... + deltas[count-1], added in that order:
    bit for bit what numpy's sequential fp32 adds give."""
    R, S, d, f = 4, 3, 72, 136
    gen = torch.Generator().manual_seed(11)
    deltas = torch.randn(R, S, d, f, generator=gen) * torch.logspace(-3, 1, R)[:, None, None, None]
    w = {"none": None, "bf16": torch.randn(d, f, generator=gen).bfloat16(),
         "fp32": torch.randn(d, f, generator=gen), "per_state": torch.randn(S, d, f, generator=gen)}[start]
    dd = deltas.to(cuda_device)
    wd = None if w is None else w.to(cuda_device)
    for count in range(R + 1):
        got = ittt.state_prefix(wd, dd, count)
        ittt.stream_status()
        want = np.zeros((S, d, f), np.float32) if w is None else np.broadcast_to(
            w.float().numpy(), (S, d, f)).astype(np.float32)
        for k in range(count):
            want = want + deltas[k].numpy()
        assert np.array_equal(got.cpu().numpy(), want), count


SEQ_SHARDS = [
    # B, T, d, f, C, eta, ranks
    (2, 512, 200, 584, 128, 0.05, 2),
    (1, 1000, 136, 264, 128, 0.1, 3),   # 8 chunks, the last partial: spans 3, 3, 2
    (2, 384, 64, 256, 128, 0.2, 5),     # 3 chunks over 5 ranks: two empty spans
]


def _emulate_ranks(g, eta, C, ranks, eta_tok=None):
    """The sequence-sharded schedule with every rank's kernels run in turn on
    this GPU: fold each span, take the exclusive prefixes, apply each span."""
    from chunk_wise_weight_gb300.shard import CudaEngine, sequence_span
    eng = CudaEngine()
    B, T, d = g["H"].shape
    f = g["W_gate"].shape[0]
    spans = [sequence_span(T, C, ranks, r) for r in range(ranks)]
    deltas = torch.zeros(ranks, B, d, f, dtype=torch.float32, device=g["H"].device)
    keep = []
    for r, (a, b) in enumerate(spans):
        if b == a:
            keep.append(None)
            continue
        et = None if eta_tok is None else eta_tok[:, a:b].contiguous()
        delta, zv = eng.fold(g["H"][:, a:b].contiguous(), g["X0"][:, a:b].contiguous(),
                             g["W_gate"], g["W_up"], g["W_target"], g["conv_w"], eta, C,
                             eta_tok=et)
        deltas[r].copy_(delta)
        keep.append(zv)
    outs = []
    for r, (a, b) in enumerate(spans):
        if b == a:
            continue
        state_in = eng.prefix(g["W_down0"], deltas, r)
        outs.append(eng.apply(g["H"][:, a:b].contiguous(), g["X0"][:, a:b].contiguous(),
                              g["W_gate"], g["W_up"], g["W_target"], g["conv_w"], eta, C,
                              keep[r], state_in))
    final = eng.prefix(g["W_down0"], deltas, ranks)
    ittt.stream_status()
    return torch.cat(outs, dim=1), final


@pytest.mark.parametrize("B,T,d,f,C,eta,ranks", SEQ_SHARDS)
def test_sequence_sharded_matches_oracle(cuda_device, B, T, d, f, C, eta, ranks):
    inp = make_inputs(B, T, d, f, seed=1830 + T)
    rates = torch.rand(B, T, generator=torch.Generator().manual_seed(8)) + 0.5
    ref = oracle.forward(inp, eta, C, want_states=True, eta_tok=rates)
    g = to_device(inp, cuda_device)
    O, final = _emulate_ranks(g, eta, C, ranks, eta_tok=rates.to(cuda_device))
    assert_parity(host(O), ref["O"], f"O over {ranks} spans")
    assert_parity(host(final), ref["states"][:, -1], "state after the last span")


def test_sequence_parallel_forward_single_rank(cuda_device):
    """With no process group the sharded entry runs the whole sequence."""
    from chunk_wise_weight_gb300.shard import sequence_parallel_forward
    B, T, d, f, C, eta = 2, 512, 200, 584, 128, 0.05
    inp = make_inputs(B, T, d, f, seed=1840)
    ref = oracle.forward(inp, eta, C, want_states=True)
    g = to_device(inp, cuda_device)
    O, st = sequence_parallel_forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"],
                                      g["W_target"], g["conv_w"], eta, C, want_state=True)
    ittt.stream_status()
    assert_parity(host(O), ref["O"], "O")
    assert_parity(host(st), ref["states"][:, -1], "final state")


def test_sequence_sharded_full_size(cuda_device):
    """The 2 x 32k-token workload (d 2560, d_ff 9728, chunks of 2048) split
    into 4 spans of 4 chunks: the same output as the unsharded call up to
    the bf16 rounding of the snapshots (the deltas are summed in another
    order), and sampled states against the oracle."""
    cfg, inp = config_inputs(2)
    B, T, d, f, C, eta = cfg["B"], cfg["T"], cfg["d"], cfg["f"], cfg["C"], cfg["eta"]
    g = to_device(inp, cuda_device)
    whole = run(g, eta, C, want_state=True)
    O, final = _emulate_ranks(g, eta, C, 4)
    assert_parity(host(O), host(whole["O"]), "O, 4 spans vs one call")
    assert_parity(host(final), host(whole["state_out"]), "final state, 4 spans vs one call")
    rng = np.random.default_rng(1850)
    m, j = rng.integers(0, d, 12), rng.integers(0, f, 12)
    ws = oracle.state_entries(inp["H"][0], inp["X0"][0], inp["W_gate"], inp["W_up"],
                              inp["W_down0"], inp["W_target"], inp["conv_w"], eta, C, m, j)
    got = host(final[0][torch.as_tensor(m), torch.as_tensor(j)])
    assert_parity(got, ws[:, -1], "final state entries vs the oracle")


# --------------------------------------------------------------------------
# CUDA graphs: a forward with a caller workspace allocates nothing and
# synchronises nothing, so it can be captured once and replayed
# --------------------------------------------------------------------------

@pytest.mark.parametrize("variant", ["default", "l2norm", "fused_conv", "dual"])
def test_forward_captured_in_cuda_graph(cuda_device, variant):
    B, T, d, f, C, eta = 2, 512, 256, 584, 128, 0.05
    kw = {"l2norm": variant == "l2norm", "fused_conv": variant == "fused_conv",
          "dual": variant == "dual"}
    g = to_device(make_inputs(B, T, d, f, seed=1900), cuda_device)
    ws_bytes = ittt.workspace_bytes_ex(B, T, d, f, C, **kw)
    assert ws_bytes > 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_device)
    out = torch.empty(B, T, d, dtype=torch.bfloat16, device=cuda_device)

    def call():
        ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                     g["conv_w"], eta, C, out, workspace=ws, **kw)

    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(side):
        call()  # first call on the device: one-time set-up outside the capture
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    ittt.stream_status()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    out.zero_()
    for _ in range(3):
        graph.replay()
    ittt.stream_status()
    assert torch.equal(out, eager)
    # the graph reads the same buffers: new input values, new output
    g["H"].copy_(torch.flip(g["H"], dims=[1]))
    graph.replay()
    ittt.stream_status()
    want = torch.empty_like(out)
    ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                 g["conv_w"], eta, C, want, workspace=ws, **kw)
    ittt.stream_status()
    assert torch.equal(out, want)
    assert not torch.equal(out, eager)


# --------------------------------------------------------------------------
# Canaries: every buffer the library writes sits inside a larger allocation
# whose guard bytes before and after hold a sentinel; after the call the
# guards must be untouched (out-of-bounds writes on ragged shapes would show)
# --------------------------------------------------------------------------

GUARD = 4096  # bytes on each side (a multiple of 256: the views stay aligned)


def guarded(shape, dtype, device):
    """A tensor of `shape` inside a byte buffer with GUARD sentinel bytes on
    both sides; returns (view, check) where check() is True while the guards
    hold."""
    elem = torch.tensor([], dtype=dtype).element_size()
    n = int(np.prod(shape)) * elem
    raw = torch.full((n + 2 * GUARD,), 0xA5, dtype=torch.uint8, device=device)
    view = raw[GUARD:GUARD + n].view(dtype).view(shape)

    def check():
        return bool((raw[:GUARD] == 0xA5).all()) and bool((raw[GUARD + n:] == 0xA5).all())
    return view, check


CANARY = [
    # B, T, d, f, C, options
    (2, 333, 136, 264, 100, {}),                          # ragged chunks, single-CTA walk
    (1, 250, 200, 584, 128, {"want_state": True}),        # partial last chunk with state_out
    (2, 640, 72, 136, 320, {"out_dtype": torch.float32}), # fp32 output, masked stores
    (1, 512, 256, 584, 128, {"l2norm": True, "want_state": True}),
    (1, 600, 64, 256, 64, {"cu_seqlens": [0, 1, 130, 387, 600]}),
    (2, 256, 64, 256, 64, {"dual": True}),
]


@pytest.mark.parametrize("B,T,d,f,C,opts", CANARY)
def test_no_writes_outside_buffers(cuda_device, B, T, d, f, C, opts):
    opts = dict(opts)
    g = to_device(make_inputs(B, T, d, f, seed=2000 + T), cuda_device)
    cu = opts.pop("cu_seqlens", None)
    want_state = opts.pop("want_state", False)
    out_dtype = opts.pop("out_dtype", torch.bfloat16)
    states = B if cu is None else len(cu) - 1
    slots = -(-T // C) if cu is None else packed_slots(cu, C)[1]
    checks = []
    out, c = guarded((B, T, d), out_dtype, cuda_device)
    checks.append(("out", c))
    kw = {}
    kw["z_buf"], c = guarded((B, T, f), torch.bfloat16, cuda_device)
    checks.append(("z_buf", c))
    kw["vhat_buf"], c = guarded((B, T, d), torch.bfloat16, cuda_device)
    checks.append(("vhat_buf", c))
    if not opts.get("dual"):
        kw["snap_buf"], c = guarded((B, slots, d, f), torch.bfloat16, cuda_device)
        checks.append(("snap_buf", c))
    if want_state:
        kw["state_out"], c = guarded((states, d, f), torch.float32, cuda_device)
        checks.append(("state_out", c))
    ws_bytes = ittt.workspace_bytes_ex(B, T, d, f, C, cu_seqlens=cu, **opts, **kw)
    assert ws_bytes > 0
    kw["workspace"], c = guarded((ws_bytes,), torch.uint8, cuda_device)
    checks.append(("workspace", c))
    ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                 g["conv_w"], 0.05, C, out, cu_seqlens=cu, **opts, **kw)
    ittt.stream_status()
    for name, check in checks:
        assert check(), f"a kernel wrote outside {name}"
    # and the call did what it should: the output matches a plain call
    ref = torch.empty_like(out)
    ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                 g["conv_w"], 0.05, C, ref, cu_seqlens=cu, **opts)
    ittt.stream_status()
    assert torch.equal(out, ref)


def test_scratch_limit_on_device(cuda_device):
    B, T, d, f, C, eta = 1, 256, 64, 256, 64, 0.05
    g = to_device(make_inputs(B, T, d, f, seed=2100), cuda_device)
    need = ittt.workspace_bytes(B, T, d, f, C)
    out = torch.full((B, T, d), 7.0, dtype=torch.bfloat16, device=cuda_device)
    args = (g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"], g["conv_w"],
            eta, C, out)
    try:
        ittt.set_scratch_limit(need - 1)
        with pytest.raises(ittt.IttError) as err:
            ittt.forward(*args)
        assert err.value.status == ittt.ERR_OOM
        ittt.stream_status()
        assert bool((out == 7.0).all())                    # nothing ran
        ws = torch.empty(need, dtype=torch.uint8, device=cuda_device)
        ittt.forward(*args, workspace=ws)                  # caller scratch: not capped
        ittt.stream_status()
        first = out.clone()
        ittt.set_scratch_limit(need)                       # exactly enough
        ittt.forward(*args)
        ittt.stream_status()
        assert torch.equal(out, first)
    finally:
        ittt.set_scratch_limit(0)


def test_phase_events_may_be_partial(cuda_device):
    """NULL entries of the events array are skipped; the others bracket their
    phase."""
    B, T, d, f, C, eta = 1, 512, 256, 584, 128, 0.05
    g = to_device(make_inputs(B, T, d, f, seed=2200), cuda_device)
    n = len(ittt.PHASES)
    gi = ittt.PHASES.index("gateup")
    events = [None] * (2 * n)
    events[2 * gi] = torch.cuda.Event(enable_timing=True)
    events[2 * gi + 1] = torch.cuda.Event(enable_timing=True)
    out = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C, events=events)
    ittt.stream_status()
    assert events[2 * gi].elapsed_time(events[2 * gi + 1]) > 0.0
    ref = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C)
    ittt.stream_status()
    assert torch.equal(out, ref)


def test_forward_called_from_c(cuda_device, tmp_path):
    """A plain C99 program (tests/c_abi/forward_from_c.c) calls ittt_forward
    through the C-ABI on its own device buffers: its O equals, bit for bit,
    the same call made from Python."""
    import subprocess
    from test_abi import build_c_program
    exe = build_c_program(str(tmp_path / "forward_from_c"))
    B, T, d, f, C, eta = 2, 512, 256, 584, 128, 0.05
    g = to_device(make_inputs(B, T, d, f, seed=2300), cuda_device)
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(src, "wb") as fh:
        fh.write(np.array([B, T, d, f, C], np.int64).tobytes())
        fh.write(np.array([eta], np.float32).tobytes())
        for k in ("H", "X0", "W_gate", "W_up", "W_down0", "W_target"):
            fh.write(g[k].contiguous().view(torch.int16).cpu().numpy().tobytes())
        fh.write(g["conv_w"].contiguous().cpu().numpy().astype(np.float32).tobytes())
    r = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    got = torch.from_numpy(np.fromfile(dst, dtype=np.int16).reshape(B, T, d)).view(torch.bfloat16)
    ref = run(g, eta, C)["O"].cpu()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("l2norm,update_only,packed", [(False, False, False), (True, False, False),
                                                       (False, True, False), (False, False, True)])
def test_state_updated_in_place(cuda_device, l2norm, update_only, packed):
    """state_out may be state_in itself: a stream of calls continues from one
    fp32 state buffer, bit-identical to separate in and out buffers."""
    B, T, d, f, C, eta = 2, 512, 256, 584, 128, 0.05
    cu = None
    if packed:
        B, cu = 1, [0, 200, 384, 512]
    S = B if cu is None else len(cu) - 1
    g = to_device(make_inputs(B, T, d, f, seed=2400), cuda_device)
    start = (torch.randn(S, d, f, generator=torch.Generator().manual_seed(9)) * 0.02).to(cuda_device)
    kw = dict(l2norm=l2norm, update_only=update_only, cu_seqlens=cu)

    def call(state_in, state_out):
        return ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], None, g["W_target"],
                            g["conv_w"], eta, C, state_in=state_in, state_out=state_out, **kw)

    sep_out = torch.empty_like(start)
    o_sep = call(start.clone(), sep_out)
    buf = start.clone()
    o_in = call(buf, buf)
    ittt.stream_status()
    assert torch.equal(buf, sep_out)
    if not update_only:
        assert torch.equal(o_in, o_sep)
    # a second step continues from the updated buffer
    sep2 = torch.empty_like(start)
    call(sep_out.clone(), sep2)
    call(buf, buf)
    ittt.stream_status()
    assert torch.equal(buf, sep2)


def test_form_chosen_by_sequence_length(cuda_device):
    """Short sequences take the dual form by default (d 512, f 1024: below
    T = 853 tokens); both forms match the oracle, the default is the dual
    form bit for bit, and forcing the primal form gives the walk."""
    B, T, d, f, C, eta = 4, 512, 512, 1024, 128, 0.05
    assert ittt.plan_form(B, T, d, f, C) == ittt.FORM_DUAL
    inp = make_inputs(B, T, d, f, seed=2500)
    ref = oracle.forward(inp, eta, C)
    g = to_device(inp, cuda_device)
    args = (g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"], g["conv_w"],
            eta, C)
    auto = ittt.forward(*args)
    dual = ittt.forward(*args, dual=True)
    primal = ittt.forward(*args, primal=True)
    ittt.stream_status()
    assert torch.equal(auto, dual)
    assert_parity(host(auto), ref["O"], "O (dual form, chosen)")
    assert_parity(host(primal), ref["O"], "O (primal form, forced)")
    walk = run(g, eta, C, intermediates=True)["O"]   # snapshots requested: the walk
    assert torch.equal(primal, walk)
