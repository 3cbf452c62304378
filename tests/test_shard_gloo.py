"""The multi-rank path on CPU: two gloo ranks each run their share of a
batch (through the oracle, standing in for the GPU kernels) and the gathered
result equals the unsharded batch; timings reduce to the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunk_wise_weight_gb300.shard import max_over_ranks, shard_range


@pytest.mark.parametrize("total,world", [(4, 2), (5, 2), (1, 3), (8, 8), (7, 3)])
def test_shard_range_partitions(total, world):
    seen = []
    sizes = []
    for r in range(world):
        a, b = shard_range(total, world, r)
        seen.extend(range(a, b))
        sizes.append(b - a)
    assert seen == list(range(total))
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from chunk_wise_weight_gb300 import make_inputs
        inp = make_inputs(4, 8, 3, 5, seed=77)
        a, b = shard_range(4, world, rank)
        mine = dict(inp)
        mine["H"], mine["X0"] = inp["H"][a:b], inp["X0"][a:b]
        O = torch.from_numpy(oracle.forward(mine, 0.4, 4)["O"])
        parts = [torch.zeros(2, 8, 3, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(parts, O)
        slowest = max_over_ranks(float(rank + 1))
        if rank == 0:
            full = oracle.forward(inp, 0.4, 4)["O"]
            np.save(os.path.join(result_dir, "gathered.npy"), torch.cat(parts).numpy())
            np.save(os.path.join(result_dir, "full.npy"), full)
            np.save(os.path.join(result_dir, "slowest.npy"), np.array([slowest]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_batch(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    np.testing.assert_array_equal(np.load(tmp_path / "gathered.npy"), np.load(tmp_path / "full.npy"))
    assert float(np.load(tmp_path / "slowest.npy")[0]) == 2.0


def test_max_over_ranks_without_group():
    assert max_over_ranks(3.5) == 3.5


# --------------------------------------------------------------------------
# Sequence sharding: spans of whole chunks, fold, all-gather, prefix, apply
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,chunk,world", [(10, 3, 4), (4, 2, 3), (64, 16, 2), (70, 16, 3),
                                           (5, 8, 2), (96, 16, 6)])
def test_sequence_spans_are_whole_chunks(T, chunk, world):
    from chunk_wise_weight_gb300.shard import sequence_span
    spans = [sequence_span(T, chunk, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == T
    for (a, b), (c, _) in zip(spans, spans[1:]):
        assert b == c                                   # contiguous, in rank order
    nonempty = [(a, b) for a, b in spans if b > a]
    for a, b in nonempty:
        assert a % chunk == 0
    for a, b in nonempty[:-1]:
        assert (b - a) % chunk == 0                     # only the last may end mid-chunk
    n = -(-T // chunk)
    assert len(nonempty) == min(n, world)


class OracleEngine:
    """The three per-rank steps evaluated by the fp64 oracle (stands in for
    the GPU kernels on CPU ranks)."""

    def __init__(self, pad_mode=0):
        import oracle
        self.oracle = oracle

    def _span(self, H, X0, Wg, Wu, W0, Wt, cw):
        return dict(H=H, X0=X0, W_gate=Wg, W_up=Wu, W_down0=W0, W_target=Wt, conv_w=cw)

    def fold(self, H, X0, Wg, Wu, Wt, cw, eta, chunk, eta_tok=None):
        d, f = H.shape[2], Wg.shape[0]
        zero = torch.zeros(d, f)
        ref = self.oracle.forward(self._span(H, X0, Wg, Wu, zero, Wt, cw), eta, chunk,
                                  want_states=True, eta_tok=eta_tok)
        # what the kernels keep between the passes (Z and eta * Vhat) the
        # oracle recomputes: it keeps the span's per-token rates
        return torch.from_numpy(ref["states"][:, -1]), eta_tok

    def zeros(self, B, d, f, device):
        return torch.zeros(B, d, f, dtype=torch.float64)

    def prefix(self, W0, deltas, count):
        return W0.double() + deltas[:count].sum(0)

    def add(self, a, b):
        return a + b

    def apply(self, H, X0, Wg, Wu, Wt, cw, eta, chunk, zv, state_in, out=None):
        return torch.from_numpy(self.oracle.forward(
            self._span(H, X0, Wg, Wu, state_in.float(), Wt, cw), eta, chunk, eta_tok=zv)["O"])


def _seq_worker(rank, world, port, result_dir, T, chunk, exchange="allgather"):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from chunk_wise_weight_gb300 import make_inputs
        from chunk_wise_weight_gb300.shard import sequence_parallel_forward, sequence_span
        B, d, f, eta = 2, 6, 10, 0.3
        inp = make_inputs(B, T, d, f, seed=91)
        rates = torch.rand(B, T, generator=torch.Generator().manual_seed(5)) + 0.5
        a, b = sequence_span(T, chunk, world, rank)
        O, state = sequence_parallel_forward(
            inp["H"][:, a:b], inp["X0"][:, a:b], inp["W_gate"], inp["W_up"], inp["W_down0"],
            inp["W_target"], inp["conv_w"], eta, chunk, eta_tok=rates[:, a:b],
            engine=OracleEngine(), want_state=True, exchange=exchange)
        np.save(os.path.join(result_dir, f"O{rank}.npy"), O.double().numpy())
        np.save(os.path.join(result_dir, f"S{rank}.npy"), state.double().numpy())
        if rank == 0:
            import oracle
            ref = oracle.forward(inp, eta, chunk, want_states=True, eta_tok=rates)
            np.save(os.path.join(result_dir, "full.npy"), ref["O"])
            np.save(os.path.join(result_dir, "final.npy"), ref["states"][:, -1])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,T,chunk,exchange", [
    (2, 24, 4, "allgather"), (3, 26, 4, "allgather"), (3, 8, 4, "allgather"),
    (2, 24, 4, "scan"), (3, 26, 4, "scan"), (4, 32, 4, "scan"), (5, 38, 4, "scan"),
    (5, 12, 4, "scan")])
def test_gloo_ranks_shard_one_sequence(tmp_path, world, T, chunk, exchange):
    """Each rank folds its span, the deltas are all-gathered, each rank
    applies from the exclusive prefix: the spans' outputs concatenated equal
    the unsharded sequence, and the last rank's state is the final state.
    (26 tokens in chunks of 4 leave a partial last chunk; 8 tokens over
    three ranks leave the third with nothing.)"""
    mp.spawn(_seq_worker, args=(world, _free_port(), str(tmp_path), T, chunk, exchange),
             nprocs=world, join=True)
    O = np.concatenate([np.load(tmp_path / f"O{r}.npy") for r in range(world)], axis=1)
    full = np.load(tmp_path / "full.npy")
    assert O.shape == full.shape
    # the oracle takes fp32 starting states: agreement to fp32 rounding
    np.testing.assert_allclose(O, full, rtol=1e-5, atol=1e-5 * np.abs(full).max())
    np.testing.assert_allclose(np.load(tmp_path / f"S{world - 1}.npy"),
                               np.load(tmp_path / "final.npy"), rtol=1e-5, atol=1e-6)


def _misaligned_worker(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from chunk_wise_weight_gb300 import make_inputs
        from chunk_wise_weight_gb300.shard import sequence_parallel_forward
        inp = make_inputs(1, 12, 6, 10, seed=92)
        a, b = [(0, 6), (6, 12)][rank]        # 6 tokens: not a whole number of 4-token chunks
        try:
            sequence_parallel_forward(inp["H"][:, a:b], inp["X0"][:, a:b], inp["W_gate"],
                                      inp["W_up"], inp["W_down0"], inp["W_target"],
                                      inp["conv_w"], 0.3, 4, engine=OracleEngine())
            msg = "no error"
        except ValueError as e:
            msg = str(e)
        with open(os.path.join(result_dir, f"r{rank}.txt"), "w") as fh:
            fh.write(msg)
    finally:
        dist.destroy_process_group()


def test_gloo_ranks_reject_spans_off_chunk_edges(tmp_path):
    mp.spawn(_misaligned_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert "not a whole number" in (tmp_path / f"r{r}.txt").read_text()
