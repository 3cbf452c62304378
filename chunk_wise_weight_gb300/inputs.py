"""Seeded synthetic inputs for the In-Place TTT fast-weight layer.

This module only draws random numbers: it holds none of the layer's
arithmetic, so both the CUDA path's tests and the fp64 oracle take their
inputs from here.

Workloads are shaped like the ones the In-Place TTT pages describe (a
Qwen3-4B-class gated MLP, contexts up to 128k tokens, chunk sizes 1k-4k);
the pages' models and datasets are not available, so every input is drawn
from fixed distributions:
    H, X0                ~ N(0, 1)
    W_gate, W_up, W_target ~ N(0, 1/d)
    W_down0              ~ N(0, 1/f)
    conv_w               ~ N(0, 1/3), shape [d, 3]
drawn in that order (H, X0, W_gate, W_up, W_down0, W_target, conv_w) in fp32
from a torch CPU generator, then rounded once to bf16 (round to nearest even)
so that the GPU path (bf16 in) and the oracle (fp64) see identical values.
"""
from __future__ import annotations

import math

import torch

# Named workloads: (batch, tokens, d_model, d_ff, chunk, eta, input dtype).
CONFIGS = [
    dict(name="tiny-d64-f256-T256-C64", B=1, T=256, d=64, f=256, C=64,
         eta=0.05, in_dtype="fp32"),
    dict(name="qwen3-4b-layer-T8k-C1024", B=1, T=8192, d=2560, f=9728, C=1024,
         eta=0.01, in_dtype="bf16"),
    dict(name="qwen3-4b-layer-B2-T32k-C2048", B=2, T=32768, d=2560, f=9728,
         C=2048, eta=0.01, in_dtype="bf16"),
    dict(name="qwen3-4b-layer-T128k-C4096", B=1, T=131072, d=2560, f=9728,
         C=4096, eta=0.005, in_dtype="bf16"),
    dict(name="pretrain-B8-T16k-d2048-f6144-C4096", B=8, T=16384, d=2048,
         f=6144, C=4096, eta=0.02, in_dtype="bf16"),
]

BASE_SEED = 1234
INPUT_NAMES = ("H", "X0", "W_gate", "W_up", "W_down0", "W_target", "conv_w")


def make_inputs(B: int, T: int, d: int, f: int, seed: int,
                round_bf16: bool = True) -> dict:
    """Draw one input set on the CPU: dict of float32 tensors.

    With round_bf16 (default) every value is exactly representable in bf16.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def draw(shape, std):
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if round_bf16:
            x = x.to(torch.bfloat16).to(torch.float32)
        return x

    out = {}
    out["H"] = draw((B, T, d), 1.0)
    out["X0"] = draw((B, T, d), 1.0)
    out["W_gate"] = draw((f, d), d ** -0.5)
    out["W_up"] = draw((f, d), d ** -0.5)
    out["W_down0"] = draw((d, f), f ** -0.5)
    out["W_target"] = draw((d, d), d ** -0.5)
    out["conv_w"] = draw((d, 3), 3 ** -0.5)
    return out


def config_inputs(index: int, round_bf16: bool = True) -> tuple[dict, dict]:
    """(config, inputs) for the named workload `index`, seed 1234 + index."""
    cfg = CONFIGS[index]
    inp = make_inputs(cfg["B"], cfg["T"], cfg["d"], cfg["f"],
                      BASE_SEED + index, round_bf16=round_bf16)
    return cfg, inp


def counted_flops(B: int, T: int, d: int, f: int, C: int) -> float:
    """Tensor-core FLOPs a call must do: gate/up (4df per token), target
    (2d^2), apply (2df) and the update of every chunk but the last (2df per
    token of chunks 0..n-2; the last chunk may be the partial remainder).
    Convolution and elementwise work are not counted."""
    n = -(-T // C)
    last = T - (n - 1) * C
    return float(B) * (T * (4 * d * f + 2 * d * d + 2 * d * f) + (T - last) * 2 * d * f)


def packed_offsets(total: int, seed: int, lo: int = 512, hi: int = 16384) -> list[int]:
    """Document offsets (cu_seqlens) for `total` tokens packed in one row.

    Lengths are drawn log-uniformly in [lo, hi] tokens (torch CPU generator,
    this seed) until the row is full; the last document takes the remainder.
    The pages give no document-length mix; this spreads lengths over the
    chunk sizes they use (a few hundred to many thousand tokens).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    cu = [0]
    while cu[-1] < total:
        u = float(torch.rand((), generator=g))
        n = int(round(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))))
        cu.append(min(total, cu[-1] + max(1, n)))
    return cu


def counted_flops_packed(cu_seqlens, d: int, f: int, C: int) -> float:
    """counted_flops summed over packed documents (each chunked on its own)."""
    return sum(counted_flops(1, b - a, d, f, C) for a, b in zip(cu_seqlens, cu_seqlens[1:]))
