"""ittt_forward_noalloc -- the forward for callers that cannot allocate
device memory while they run (a serving loop with a fixed, fully partitioned
memory budget; device memory owned by another framework's caching allocator;
a real-time path that forbids allocation after start-up).

It keeps its scratch in one fixed 64 MiB device array instead of allocating.
These tests check, on two calls in a row with different inputs (so nothing
the first call leaves in the shared scratch can stand in for the second):

  * that each output equals, bit for bit, the output of ittt_forward_ex in
    the primal form on the same inputs -- the two run the same kernels in
    the same order -- and matches the fp64 oracle within the layer's bar;
  * that the second call changes neither the device's free memory nor the
    memory PyTorch's caching allocator holds (nothing was allocated);
  * for a bf16 and an fp32 W_down0 (the fp32 one is first copied into the
    scratch's snapshot slot 0), bf16 and fp32 output, a partial last chunk,
    and chunks that are not multiples of 64 tokens (the single-CTA walk with
    masked K blocks);

and that work too large for the fixed array is refused before anything
runs.  This file is collected last, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from chunk_wise_weight_gb300 import build, ittt, make_inputs

REL_FRO = 5e-3
MAX_RATIO = 2e-2


def _entry():
    build.build()
    lib = ittt.load()
    fn = lib.ittt_forward_noalloc
    tp = ctypes.POINTER(ittt.Tensor)
    fn.argtypes = [tp, tp, tp, tp, tp, tp, tp, ctypes.c_float, ctypes.c_int64, tp,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, tensors, eta, chunk, out, stream):
    descs = [ittt.describe(t) for t in tensors] + [ittt.describe(out)]
    refs = [ctypes.byref(d) for d in descs]
    return fn(*refs[:7], ctypes.c_float(eta), ctypes.c_int64(chunk), refs[7],
              ctypes.c_void_p(stream))


CASES = [
    # W_down0 dtype, out dtype, T, chunk
    (torch.bfloat16, torch.bfloat16, 1024, 256),
    (torch.float32, torch.bfloat16, 1024, 256),   # W_0 copied into snapshot slot 0
    (torch.bfloat16, torch.float32, 1024, 256),   # fp32 output (no TMA store map)
    (torch.bfloat16, torch.bfloat16, 1000, 192),  # partial last chunk of 40 tokens
    (torch.bfloat16, torch.bfloat16, 1000, 200),  # chunks not multiples of 64: single-CTA walk
]


@pytest.mark.gpu
@pytest.mark.parametrize("w0_dtype,out_dtype,T,C", CASES)
def test_noalloc_matches_forward_on_two_calls_in_a_row(cuda_device, w0_dtype, out_dtype, T, C):
    fn = _entry()
    B, d, f, eta = 2, 256, 1024, 0.03
    stream = torch.cuda.current_stream(cuda_device)
    calls = []
    for seed in (21, 22):
        inp = make_inputs(B, T, d, f, seed=seed + T + C)
        g = [inp[k].to(cuda_device, torch.bfloat16) for k in ("H", "X0", "W_gate", "W_up")]
        g.append(inp["W_down0"].to(cuda_device, w0_dtype))
        g.append(inp["W_target"].to(cuda_device, torch.bfloat16))
        g.append(inp["conv_w"].to(cuda_device, torch.float32))
        ref = ittt.forward(*g, eta, C, out_dtype=out_dtype, primal=True)
        out = torch.full((B, T, d), float("nan"), dtype=out_dtype, device=cuda_device)
        calls.append((inp, g, ref, out))
    ittt.stream_status()
    torch.cuda.synchronize(cuda_device)

    # First call (on a fresh device it also does the one-time set-up).
    inp, g, ref, out = calls[0]
    assert _call(fn, g, eta, C, out, stream.cuda_stream) == ittt.OK, ittt.last_error()
    torch.cuda.synchronize(cuda_device)
    free_before = torch.cuda.mem_get_info(cuda_device)[0]
    reserved_before = torch.cuda.memory_reserved(cuda_device)
    # Second call, other inputs, straight after: no allocation anywhere.
    inp, g, ref, out = calls[1]
    assert _call(fn, g, eta, C, out, stream.cuda_stream) == ittt.OK, ittt.last_error()
    torch.cuda.synchronize(cuda_device)
    assert torch.cuda.mem_get_info(cuda_device)[0] == free_before
    assert torch.cuda.memory_reserved(cuda_device) == reserved_before
    ittt.stream_status()

    for k, (inp, g, ref, out) in enumerate(calls):
        # Same kernels, same order, same operands as the primal ittt_forward_ex.
        assert torch.equal(out, ref), f"call {k}: differs from ittt_forward_ex (primal)"
        want = oracle.forward(inp, eta, C)["O"]
        got = out.double().cpu().numpy()
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        mx = np.abs(got - want).max() / np.abs(want).max()
        assert rel <= REL_FRO and mx <= MAX_RATIO, f"call {k}: rel={rel:.3e} max={mx:.3e}"


def test_noalloc_refuses_work_beyond_its_fixed_scratch():
    """No GPU needed: the size check comes before any CUDA call."""
    fn = _entry()
    B, T, d, f = 1, 4096, 1024, 4096          # 8 MiB per chunk of snapshots...
    shapes = {"H": [B, T, d], "X0": [B, T, d], "W_gate": [f, d], "W_up": [f, d],
              "W_down0": [d, f], "W_target": [d, d], "conv_w": [d, 3], "out": [B, T, d]}
    descs = []
    for k, (name, shp) in enumerate(shapes.items()):
        t = ittt.Tensor()
        t.data = (k + 1) << 32                   # never dereferenced
        t.dtype = ittt.FP32 if name == "conv_w" else ittt.BF16
        t.ndim = len(shp)
        acc = 1
        for j in reversed(range(len(shp))):
            t.shape[j] = shp[j]
            t.stride[j] = acc
            acc *= shp[j]
        descs.append(t)
    refs = [ctypes.byref(t) for t in descs]
    status = fn(*refs[:7], ctypes.c_float(0.01), ctypes.c_int64(256), refs[7], None)
    assert status == ittt.ERR_UNSUPPORTED            # ...times 16 chunks: > 64 MiB
    assert "64 MiB" in ittt.last_error()
