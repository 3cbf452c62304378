"""ittt_forward_noalloc -- the forward for callers that cannot allocate
device memory while they run (a serving loop with a fixed, fully partitioned
memory budget; device memory owned by another framework's caching allocator;
a real-time path that forbids allocation after start-up).

It keeps its scratch in one fixed 64 MiB device array instead of allocating.
These tests check that it gives the output of ittt_forward on two calls in a
row (different inputs each time, so nothing left in the shared scratch by the
first call can stand in for the second), and that work too large for the
fixed array is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest
import torch

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


@pytest.mark.gpu
def test_noalloc_matches_forward_on_two_calls_in_a_row(cuda_device):
    fn = _entry()
    B, T, d, f, C, eta = 2, 1024, 256, 1024, 256, 0.03
    stream = torch.cuda.current_stream(cuda_device)
    for seed in (21, 22):
        inp = make_inputs(B, T, d, f, seed=seed)
        g = [inp[k].to(cuda_device, torch.bfloat16)
             for k in ("H", "X0", "W_gate", "W_up", "W_down0", "W_target")]
        g.append(inp["conv_w"].to(cuda_device, torch.float32))
        ref = torch.empty(B, T, d, dtype=torch.bfloat16, device=cuda_device)
        ittt.forward_plain(*g, eta, C, ref)
        out = torch.full((B, T, d), float("nan"), dtype=torch.bfloat16, device=cuda_device)
        status = _call(fn, g, eta, C, out, stream.cuda_stream)
        assert status == ittt.OK, ittt.last_error()
        ittt.stream_status()
        got = out.double().cpu().numpy()
        want = ref.double().cpu().numpy()
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        mx = np.abs(got - want).max() / np.abs(want).max()
        assert rel <= REL_FRO and mx <= MAX_RATIO, f"seed {seed}: rel={rel:.3e} max={mx:.3e}"


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
