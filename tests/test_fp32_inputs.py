"""fp32 inputs: H, X0, W_gate, W_up and W_target given as fp32 and never
rounded to bf16.  The library splits each value x into bf16 parts
hi = bf16(x), lo = bf16(x - hi) and forms every product of the gate/up and
target GEMMs as hi*hi + hi*lo + lo*hi over a concatenated K of 3 d, so Z and
eta * Vhat are the fp32-accurate products rounded once to bf16.

What the tests pin, on inputs drawn without rounding (so a bf16 rounding of
any input would show):

  * Z and eta * Vhat, exported through z_buf / vhat_buf, are within one bf16
    unit in the last place of the exact (fp64) products of the unrounded
    inputs, and equal the exact product rounded to bf16 for nearly every
    element (the few others sit within about 2^-16 relative of a rounding
    boundary).  The same layer with bf16-rounded inputs misses that by far,
    so a mode that silently rounded its inputs fails here.
  * O matches the fp64 oracle on the unrounded inputs within the layer's
    bar, and its error is below that of the bf16-input layer on the same
    values.
  * Regular batches, a ragged length with chunks that are not multiples of
    64 and widths that are not multiples of 64 (d = 200: a K block straddles
    the hi/lo segments), packed documents, per-token rates, the dual form,
    the normalised update, and two calls chained through the fp32 state.
"""
import numpy as np
import pytest
import torch

import oracle
from chunk_wise_weight_gb300 import ittt, make_inputs

REL_FRO = 5e-3
MAX_RATIO = 2e-2
# Fraction of elements allowed to differ from the exact product rounded to
# bf16 (those within ~2^-16 relative of a rounding boundary: ~1% expected
# at most).
MISROUND = 0.02


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    """bf16 unit in the last place at |x| (8 significand bits)."""
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7)


def _check_rounded(name, got, exact):
    """got (bf16 values, as fp64) against the exact fp64 products."""
    scale = np.sqrt(np.mean(exact ** 2))
    err = np.abs(got - exact)
    bound = _bf16_ulp(exact) + 1e-4 * scale
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), (
        f"{name}: element {np.unravel_index(worst, exact.shape)} got {got.flat[worst]!r}, "
        f"exact {exact.flat[worst]!r}, beyond one bf16 ulp")
    rounded = torch.from_numpy(exact).float().to(torch.bfloat16).double().numpy()
    frac = np.mean(got != rounded)
    assert frac <= MISROUND, f"{name}: {frac:.2%} of elements not the exact product rounded"
    return np.linalg.norm(got - exact) / np.linalg.norm(exact)


def _dev(inp, dev, dtype):
    t = {k: inp[k].to(dev, dtype) for k in ("H", "X0", "W_gate", "W_up", "W_target")}
    t["W_down0"] = inp["W_down0"].to(dev, torch.float32)
    t["conv_w"] = inp["conv_w"].to(dev, torch.float32)
    return t


def _run(t, eta, C, **kw):
    B, T, d = t["H"].shape
    f = t["W_gate"].shape[0]
    dev = t["H"].device
    z = torch.empty(B, T, f, dtype=torch.bfloat16, device=dev)
    vh = torch.empty(B, T, d, dtype=torch.bfloat16, device=dev)
    out = ittt.forward(t["H"], t["X0"], t["W_gate"], t["W_up"], t["W_down0"], t["W_target"],
                       t["conv_w"], eta, C, out_dtype=torch.float32, z_buf=z, vhat_buf=vh, **kw)
    ittt.stream_status()
    host = lambda x: x.double().cpu().numpy()  # noqa: E731
    return host(out), host(z), host(vh)


def _o_err(got, want):
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    mx = np.abs(got - want).max() / np.abs(want).max()
    return rel, mx


CASES = [
    # B, T, d, f, C, options
    (2, 1024, 256, 1024, 256, {}),
    (1, 1000, 200, 520, 192, {}),                    # ragged, d and f not multiples of 64
    (2, 512, 256, 1024, 128, {"dual": True}),
    (2, 768, 256, 768, 256, {"pad_mode": ittt.PAD_SEQUENCE, "rates": True}),
]


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,d,f,C,opt", CASES)
def test_fp32_inputs_match_unrounded_products(cuda_device, B, T, d, f, C, opt):
    opt = dict(opt)
    eta = 0.03
    inp = make_inputs(B, T, d, f, seed=500 + T + d, round_bf16=False)
    assert not torch.equal(inp["H"], inp["H"].to(torch.bfloat16).float())  # unrounded
    pad = opt.pop("pad_mode", ittt.PAD_CHUNK)
    kw = dict(pad_mode=pad, **opt)
    rates = kw.pop("rates", False)
    et_host = None
    if rates:
        g = torch.Generator().manual_seed(77)
        et_host = torch.rand(B, T, generator=g) * 1.5 + 0.25
        kw["eta_tok"] = et_host.to(cuda_device)
    want = oracle.forward(inp, eta, C, pad_mode=pad, want_z=True, want_vhat=True,
                          eta_tok=et_host)
    eta_v = eta * (et_host.double().numpy()[..., None] if rates else 1.0)

    o32, z32, v32 = _run(_dev(inp, cuda_device, torch.float32), eta, C, **kw)
    z_rel = _check_rounded("Z", z32, want["Z"])
    v_rel = _check_rounded("eta * Vhat", v32, eta_v * want["Vhat"])
    rel, mx = _o_err(o32, want["O"])
    assert rel <= REL_FRO and mx <= MAX_RATIO, f"O: rel={rel:.3e} max={mx:.3e}"

    # The same values rounded to bf16 first: Z and eta * Vhat then carry the
    # input rounding (several times the error), and O is no closer.
    o16, z16, v16 = _run(_dev(inp, cuda_device, torch.bfloat16), eta, C, **kw)
    z16_rel = np.linalg.norm(z16 - want["Z"]) / np.linalg.norm(want["Z"])
    v16_rel = np.linalg.norm(v16 - eta_v * want["Vhat"]) / np.linalg.norm(eta_v * want["Vhat"])
    assert z16_rel > 1.5 * z_rel, (z16_rel, z_rel)
    assert v16_rel > 1.5 * v_rel, (v16_rel, v_rel)
    assert rel < _o_err(o16, want["O"])[0]


@pytest.mark.gpu
def test_fp32_inputs_packed_documents(cuda_device):
    T, d, f, C, eta = 1500, 256, 768, 256, 0.03
    cu = [0, 300, 1000, 1500]
    inp = make_inputs(1, T, d, f, seed=909, round_bf16=False)
    want = oracle.forward_packed(inp, cu, eta, C, want_z=True, want_vhat=True)
    o32, z32, v32 = _run(_dev(inp, cuda_device, torch.float32), eta, C, cu_seqlens=cu)
    _check_rounded("Z", z32[0], want["Z"])
    _check_rounded("eta * Vhat", v32[0], eta * want["Vhat"])
    rel, mx = _o_err(o32[0], want["O"])
    assert rel <= REL_FRO and mx <= MAX_RATIO, f"O: rel={rel:.3e} max={mx:.3e}"


@pytest.mark.gpu
def test_fp32_inputs_plain_call_equals_export(cuda_device):
    """The plain ittt_forward entry point takes fp32 inputs too and gives the
    same O as the call that exports Z and eta * Vhat."""
    B, T, d, f, C, eta = 2, 512, 256, 512, 128, 0.05
    inp = make_inputs(B, T, d, f, seed=31, round_bf16=False)
    t = _dev(inp, cuda_device, torch.float32)
    o_exp, _, _ = _run(t, eta, C, primal=True)
    out = torch.empty(B, T, d, dtype=torch.float32, device=cuda_device)
    ittt.forward_plain(t["H"], t["X0"], t["W_gate"], t["W_up"], t["W_down0"], t["W_target"],
                       t["conv_w"], eta, C, out)
    ittt.stream_status()
    assert ittt.plan_form(B, T, d, f, C, fp32_inputs=True) == ittt.FORM_PRIMAL
    assert torch.equal(out.cpu().double(), torch.from_numpy(o_exp))


@pytest.mark.gpu
def test_fp32_inputs_l2_normalised_walk(cuda_device):
    """fp32 inputs with the normalised update: O within the bar against the
    oracle on the unrounded values, and closer than the same values rounded
    to bf16 first."""
    B, T, d, f, C, eta = 2, 1024, 256, 512, 128, 0.05
    inp = make_inputs(B, T, d, f, seed=77, round_bf16=False)
    want = oracle.forward(inp, eta, C, l2norm=True)["O"]
    errs = []
    for dt in (torch.float32, torch.bfloat16):
        t = _dev(inp, cuda_device, dt)
        out = ittt.forward(t["H"], t["X0"], t["W_gate"], t["W_up"], t["W_down0"], t["W_target"],
                           t["conv_w"], eta, C, out_dtype=torch.float32, l2norm=True)
        ittt.stream_status()
        errs.append(_o_err(out.double().cpu().numpy(), want))
    rel, mx = errs[0]
    assert rel <= REL_FRO and mx <= MAX_RATIO, f"O: rel={rel:.3e} max={mx:.3e}"
    assert rel < errs[1][0], (errs[0], errs[1])


@pytest.mark.gpu
def test_fp32_inputs_streaming_two_calls_equal_one(cuda_device):
    """fp32 inputs across two calls chained through state_out / state_in (a
    split at a chunk boundary): the final state matches the oracle, and O
    equals the single call's bit for bit (the same products, splits and
    walk)."""
    B, T, d, f, C, eta = 2, 1024, 256, 512, 128, 0.03
    inp = make_inputs(B, T, d, f, seed=78, round_bf16=False)
    ref = oracle.forward(inp, eta, C, want_states=True)
    t = _dev(inp, cuda_device, torch.float32)
    half = T // 2

    def call(H, X0, state_in=None):
        state = torch.empty(B, d, f, dtype=torch.float32, device=cuda_device)
        out = ittt.forward(H, X0, t["W_gate"], t["W_up"], t["W_down0"], t["W_target"],
                           t["conv_w"], eta, C, out_dtype=torch.float32, state_in=state_in,
                           state_out=state, primal=True)
        return out, state

    whole, s_whole = call(t["H"], t["X0"])
    a, s_a = call(t["H"][:, :half].contiguous(), t["X0"][:, :half].contiguous())
    b, s_b = call(t["H"][:, half:].contiguous(), t["X0"][:, half:].contiguous(), state_in=s_a)
    ittt.stream_status()
    assert torch.equal(torch.cat([a, b], dim=1), whole)
    assert torch.equal(s_b, s_whole)
    rel, mx = _o_err(s_b.double().cpu().numpy(), ref["states"][:, T // C])
    assert rel <= REL_FRO and mx <= MAX_RATIO, f"final state: rel={rel:.3e} max={mx:.3e}"
    rel, mx = _o_err(whole.double().cpu().numpy(), ref["O"])
    assert rel <= REL_FRO and mx <= MAX_RATIO, f"O: rel={rel:.3e} max={mx:.3e}"
