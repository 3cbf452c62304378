"""Whole-output parity at full size, through the C-ABI (libittt.so).

Every element of O, Z, eta * Vhat, every bf16 weight snapshot W_0..W_{n-1}
and the final fp32 fast-weight state is compared with the chunk-by-chunk
fp64 oracle (oracle/chunked.py: the sequential apply-then-update loop of
"[논문리뷰] In-Place Test-Time Training", Method §1 eq. (2)-(4), §2 eq.
(5)-(6), with float64 matrix products as its steps), at the full sizes of
the named workloads and of other layer widths.  The bar is the layer's:
relative Frobenius error <= 5e-3 and max elementwise error <= 2e-2 * max|ref|,
over each whole tensor and, for O, over every (sequence, chunk) block on its
own.

At these sizes every persistent kernel runs several rounds of units per CTA
pair (76 pairs on 152 SMs), so accumulator reuse across units, the update
walk's next-unit preload and the grouped gate/up raster are all exercised:

  workload (B x T, d/f, C)        gate/up units  apply units   update pair units
  1 x 8192, 2560/9728, 1024       32 x 76        320 (4.2 r)   190: 2 rounds + 38 pairs split into 76 halves
  2 x 32768, 2560/9728, 2048      256 x 76       2560 (33.7 r) 380: 5 rounds
  1 x 131072, 2560/9728, 4096     512 x 76       5120 (67.4 r) 190: 2 rounds + split
  8 x 16384, 2048/6144, 4096      512 x 48       4096 (53.9 r) 768: 10 rounds + 8 pairs split
  1 x 8100, 2560/9728, 1000       32 x 76        330 (4.3 r)   single-CTA walk (chunks not multiples of 64):
                                                                380 on 152 SMs: 2 rounds + 76 split

(gate/up: 256-row tiles x 128-column tiles of d_ff; apply: (chunk, 256-row
tile) x 256-column tiles of d; update: pairs of 256 x 256 state blocks,
d-block fastest.)  The call checked is the one bench.py times: a call without
exported intermediates gives the same O bit for bit.
"""
import time

import numpy as np
import pytest
import torch

from chunk_wise_weight_gb300 import config_inputs, ittt, make_inputs
from chunk_wise_weight_gb300.inputs import packed_offsets
from oracle import chunked

pytestmark = pytest.mark.gpu

REL_FRO = 5e-3
MAX_RATIO = 2e-2


class Err:
    """Running error of one tensor against the oracle, over many blocks."""

    def __init__(self, what):
        self.what, self.dd, self.rr, self.dmax, self.rmax = what, 0.0, 0.0, 0.0, 0.0

    def add(self, got, ref, block=None):
        diff = got - ref
        dd, rr = float((diff * diff).sum()), float((ref * ref).sum())
        dmax, rmax = float(np.abs(diff).max()), float(np.abs(ref).max())
        self.dd, self.rr = self.dd + dd, self.rr + rr
        self.dmax, self.rmax = max(self.dmax, dmax), max(self.rmax, rmax)
        if block is not None:
            rf, mr = (dd / max(rr, 1e-300)) ** 0.5, dmax / max(rmax, 1e-300)
            assert rf <= REL_FRO and mr <= MAX_RATIO, \
                f"{self.what} {block}: rel_fro={rf:.3e} max_ratio={mr:.3e}"

    def check(self):
        rf, mr = (self.dd / max(self.rr, 1e-300)) ** 0.5, self.dmax / max(self.rmax, 1e-300)
        print(f"parity {self.what}: rel_fro={rf:.3e} max_ratio={mr:.3e}")
        assert rf <= REL_FRO and mr <= MAX_RATIO, f"{self.what}: rel_fro={rf:.3e} max_ratio={mr:.3e}"
        return rf


def _rows_differing(a, b):
    rows = (a != b).reshape(-1, a.shape[-1]).any(dim=1).nonzero().flatten()
    return f"{len(rows)} rows (first {rows[:6].tolist()})"


def _host(t):
    return t.detach().double().cpu().numpy()


def _device_inputs(inp, dev):
    g = {k: inp[k].to(dev, torch.bfloat16) for k in ("H", "X0", "W_gate", "W_up", "W_target",
                                                     "W_down0")}
    g["conv_w"] = inp["conv_w"].to(dev, torch.float32)
    return g


def whole_output_parity(inp, eta, C, dev, *, pad_mode=0, eta_tok=None, l2norm=False, cu=None,
                        form="auto", expect_dual=None):
    """Run the layer with every intermediate exported and compare all of it
    with the oracle, sequence (or packed document) by sequence, chunk by
    chunk.  form: "auto" (the library's own choice, what bench.py runs),
    "primal" or "dual" (forced).  expect_dual: the choice "auto" must make
    (None: not checked).  Returns the relative Frobenius error of O."""
    t0 = time.time()
    g = _device_inputs(inp, dev)
    B, T, d = g["H"].shape
    f = g["W_gate"].shape[0]
    docs = [(b, 0, T) for b in range(B)] if cu is None else \
        [(0, a, e) for a, e in zip(cu, cu[1:])]
    slots, base = 0, []
    for _, a, e in docs:
        base.append(slots if cu is not None else 0)
        slots += -(-(e - a) // C)
    per_seq_slots = -(-T // C) if cu is None else slots
    et = None if eta_tok is None else eta_tok.to(dev, torch.float32)
    kw = dict(pad_mode=pad_mode, eta_tok=et, l2norm=l2norm, cu_seqlens=cu,
              primal=form == "primal", dual=form == "dual")
    plain = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                         g["conv_w"], eta, C, **kw)
    ittt.stream_status()
    plan = dict(pad_mode=pad_mode, l2norm=l2norm, cu_seqlens=cu, primal=kw["primal"],
                dual=kw["dual"])
    dual_chosen = ittt.plan_form(B, T, d, f, C, **plan) == ittt.FORM_DUAL
    if expect_dual is not None:
        assert dual_chosen == expect_dual
    kw["dual"], kw["primal"] = dual_chosen, not dual_chosen
    z = torch.empty(B, T, f, dtype=torch.bfloat16, device=dev)
    vh = torch.empty(B, T, d, dtype=torch.bfloat16, device=dev)
    bufs = dict(z_buf=z, vhat_buf=vh)
    if not dual_chosen:
        bufs["snap_buf"] = torch.empty(B, per_seq_slots, d, f, dtype=torch.bfloat16, device=dev)
        bufs["state_out"] = torch.empty(len(docs), d, f, dtype=torch.float32, device=dev)
    out = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"], g["W_target"],
                       g["conv_w"], eta, C, **kw, **bufs)
    ittt.stream_status()
    # The exporting call is the timed call's arithmetic, bit for bit.
    if not torch.equal(out, plain):
        again = ittt.forward(g["H"], g["X0"], g["W_gate"], g["W_up"], g["W_down0"],
                             g["W_target"], g["conv_w"], eta, C, **kw)
        ittt.stream_status()
        pytest.fail(f"exporting call differs from the plain call in {_rows_differing(out, plain)};"
                    f" plain again vs plain: {_rows_differing(again, plain)},"
                    f" plain again vs exporting: {_rows_differing(again, out)}")
    t_gpu = time.time() - t0

    errs = {k: Err(k) for k in ("O", "Z", "eta * Vhat", "snapshots", "final state")}
    w64 = chunked.weights64(inp)
    rates = None if eta_tok is None else eta_tok.reshape(B, T)
    for k, (b, a, e) in enumerate(docs):
        H, X0 = inp["H"][b, a:e], inp["X0"][b, a:e]
        for c in chunked.walk_sequence(H, X0, None, None, inp["W_down0"], None, inp["conv_w"],
                                       eta, C, pad_mode, None if rates is None else rates[b, a:e],
                                       l2norm, want_final=not dual_chosen, weights64=w64):
            lo, hi = a + c["lo"], a + c["hi"]
            where = f"[seq {b} doc {k} chunk {c['i']}]"
            errs["O"].add(_host(out[b, lo:hi]), c["O"], where)
            errs["Z"].add(_host(z[b, lo:hi]), c["Z"])
            # the exported target holds eta * eta_t * Vhat_t (rates folded in)
            r = 1.0 if rates is None else rates[b, lo:hi].double().numpy()[:, None]
            errs["eta * Vhat"].add(_host(vh[b, lo:hi]), eta * r * c["Vhat"])
            if not dual_chosen:
                errs["snapshots"].add(_host(bufs["snap_buf"][b, base[k] + c["i"]]), c["W"])
                if "W_next" in c:
                    errs["final state"].add(_host(bufs["state_out"][k]), c["W_next"])
    rf = errs["O"].check()
    errs["Z"].check()
    errs["eta * Vhat"].check()
    if not dual_chosen:
        errs["snapshots"].check()
        errs["final state"].check()
    print(f"gpu {t_gpu:.1f} s, oracle and comparison {time.time() - t0 - t_gpu:.1f} s")
    return rf


@pytest.mark.parametrize("index", [1, 2, 3, 4])
def test_named_workload_whole_output(cuda_device, index):
    """The four full-size named workloads (Qwen3-4B-shaped layer at 8k,
    2 x 32k and 128k tokens; the 8 x 16k pretraining batch), whole."""
    cfg, inp = config_inputs(index)
    whole_output_parity(inp, cfg["eta"], cfg["C"], cuda_device, expect_dual=False)


@pytest.mark.parametrize("shape,form", [
    ((1, 8192, 4096, 14336, 2048, 0.01), "auto"),    # Llama-3-8B-sized MLP: the walk
    ((2, 4096, 5120, 13824, 1024, 0.01), "auto"),    # Qwen2.5-14B-sized MLP: the dual form
    ((2, 4096, 5120, 13824, 1024, 0.01), "primal"),  # the same, walked (d_ff / 512 odd)
    ((2, 4096, 1024, 3072, 512, 0.02), "auto"),      # Qwen3-0.6B-sized MLP: the walk
])
def test_other_layer_widths_whole_output(cuda_device, shape, form):
    """Layer widths of other model sizes, in the form the library picks (by
    measured cost) and, where that is the dual form, walked as well."""
    B, T, d, f, C, eta = shape
    inp = make_inputs(B, T, d, f, seed=1600 + d)
    whole_output_parity(inp, eta, C, cuda_device, form=form)


def test_ragged_chunks_single_cta_whole_output(cuda_device):
    """Chunks of 1000 tokens (not a multiple of 64: the single-CTA walk with
    masked K blocks; apply tiles that end inside a chunk) and a 100-token
    last chunk, at the Qwen3-4B widths."""
    inp = make_inputs(1, 8100, 2560, 9728, seed=1650)
    whole_output_parity(inp, 0.01, 1000, cuda_device)


def test_per_token_rates_and_sequence_padding_whole_output(cuda_device):
    """Per-token learning rates ("[논문리뷰] Test-Time Training Done Right",
    per-token eta_i) and sequence-edge padding at 1 x 8192."""
    cfg, inp = config_inputs(1)
    rates = torch.rand(1, cfg["T"], generator=torch.Generator().manual_seed(4321)) + 0.5
    whole_output_parity(inp, cfg["eta"], cfg["C"], cuda_device, eta_tok=rates,
                        pad_mode=ittt.PAD_SEQUENCE)


def test_l2_normalised_walk_whole_output(cuda_device):
    """The normalised update rule (L2-Normalize(W - g) row by row, "[논문리뷰]
    Test-Time Training Done Right", Non-Linear Update of Fast-Weight) at
    1 x 8192, on CTA pairs (d a multiple of 256, chunks of 1024)."""
    cfg, inp = config_inputs(1)
    whole_output_parity(inp, cfg["eta"], cfg["C"], cuda_device, l2norm=True)


def test_packed_documents_whole_output(cuda_device):
    """The bench's packed-document mix: 2 x 32768 tokens in one row, ten
    documents of 664-15,801 tokens, the fast weight reset at every document
    (Method §3), chunks restarting at each document."""
    cfg, inp = config_inputs(2)
    T = cfg["B"] * cfg["T"]
    cu = packed_offsets(T, seed=2468)
    packed = dict(inp, H=inp["H"].reshape(1, T, -1), X0=inp["X0"].reshape(1, T, -1))
    whole_output_parity(packed, cfg["eta"], cfg["C"], cuda_device, cu=cu)


def test_dual_form_full_width_whole_output(cuda_device):
    """64 sequences of 256 tokens at the Qwen3-4B widths, where the library
    picks the dual form O_[i] = Z_[i] W_0^T + eta sum_{j<i} (Z_[i] Z_[j]^T)
    Vhat_[j] itself; compared with the walk of the oracle."""
    inp = make_inputs(64, 256, 2560, 9728, seed=1660)
    whole_output_parity(inp, 0.01, 64, cuda_device, expect_dual=True)
