"""Sharding the layer across ranks (one process per GPU).

Batch sharding.  Each sequence carries its own fast-weight state that starts
from W_down0 (reset at document boundaries, "[논문리뷰] In-Place Test-Time
Training", Method §3), so sequences are independent units: a rank runs the
layer on its contiguous share of the batch and no tensor crosses ranks.  The
only cross-rank traffic is host-side bookkeeping: barriers and the max of
the ranks' timings.

Sequence sharding (context parallelism, Method §3 "Implementation Details":
per-chunk deltas in parallel, one prefix sum, then the apply).  Rank r owns
a contiguous span of whole chunks of every sequence.  The update is additive
and each chunk's delta depends on that chunk's tokens alone (the convolution
is zero-padded at chunk edges), so

  1. every rank folds its span into D_r = eta * sum_{i in span r}
     Vhat_[i]^T Z_[i] from a zero start, keeping Z and eta * Vhat;
  2. the ranks exchange the D_r: an all-gather of one [B, d, f] fp32 tensor
     per rank, or an exclusive scan by recursive doubling (ceil(log2 R) + 1
     point-to-point rounds of one tensor each instead of R - 1 received);
  3. rank r starts from W_down0 + D_0 + ... + D_{r-1} (an exclusive prefix)
     and runs the usual walk and apply over its span, reusing Z and eta*Vhat.

The exchange is the one data-path communication.  The work per token is the
single-GPU work plus one extra 2*d*f-FLOP contraction (step 1's fold).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_range(total: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of `rank`'s contiguous share of `total` units; shares
    differ by at most one unit and cover every unit exactly once."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def sequence_span(T: int, chunk: int, world: int, rank: int) -> tuple[int, int]:
    """Token span [start, stop) of `rank` when the chunks of a T-token
    sequence are shared out in contiguous runs: spans start on chunk
    boundaries, only the last non-empty span may end in a partial chunk, and
    ranks beyond the chunk count get an empty span."""
    if chunk <= 0 or T < 0:
        raise ValueError("bad T/chunk")
    n = -(-T // chunk)
    a, b = shard_range(n, world, rank)
    return min(a * chunk, T), min(b * chunk, T)


def max_over_ranks(value: float, device: torch.device | None = None) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank's);
    the value itself when no process group is running."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device: torch.device | None = None) -> None:
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


class CudaEngine:
    """The three per-rank steps of sequence sharding on the library's kernels."""

    def __init__(self, stream=None):
        from . import ittt
        self.ittt = ittt
        self.stream = stream

    def fold(self, H, X0, W_gate, W_up, W_target, conv_w, eta, chunk, eta_tok=None):
        """D = eta * sum_i Vhat_[i]^T Z_[i] over the span's chunks (zero
        start); returns (D [B,d,f] fp32, (Z, eta * Vhat))."""
        B, T, d = H.shape
        f = W_gate.shape[0]
        z = torch.empty(B, T, f, dtype=torch.bfloat16, device=H.device)
        vhat = torch.empty(B, T, d, dtype=torch.bfloat16, device=H.device)
        delta = torch.empty(B, d, f, dtype=torch.float32, device=H.device)
        self.ittt.forward(H, X0, W_gate, W_up, None, W_target, conv_w, eta, chunk,
                          stream=self.stream, update_only=True, state_out=delta, z_buf=z,
                          vhat_buf=vhat, eta_tok=eta_tok)
        return delta, (z, vhat)

    def zeros(self, B, d, f, device):
        return torch.zeros(B, d, f, dtype=torch.float32, device=device)

    def prefix(self, W_down0, deltas, count):
        """W_down0 + deltas[0] + ... + deltas[count-1] (fp32 [B,d,f])."""
        return self.ittt.state_prefix(W_down0, deltas, count, stream=self.stream)

    def add(self, a, b):
        """a + b for two fp32 [B,d,f] states (a first)."""
        return self.ittt.state_prefix(a, b.unsqueeze(0), 1, stream=self.stream)

    def apply(self, H, X0, W_gate, W_up, W_target, conv_w, eta, chunk, zv, state_in,
              out=None):
        z, vhat = zv
        return self.ittt.forward(H, X0, W_gate, W_up, None, W_target, conv_w, eta, chunk, out,
                                 stream=self.stream, state_in=state_in, reuse_zv=True, z_buf=z,
                                 vhat_buf=vhat)


def check_spans(T_r: int, chunk: int, world: int, group, device) -> None:
    """Every rank's span length, all-gathered: the spans must be whole chunks
    except the last non-empty one, and no non-empty span may follow an empty
    one (chunk edges are where the convolution pads and the prefix splits).
    Raises ValueError on every rank alike."""
    mine = torch.tensor([T_r], dtype=torch.int64, device=device)
    lens = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(lens, mine, group=group)
    lens = [int(t.item()) for t in lens]
    nonempty = [r for r, n in enumerate(lens) if n > 0]
    if nonempty and nonempty != list(range(len(nonempty))):
        raise ValueError(f"span lengths {lens}: a non-empty span follows an empty one")
    for r in nonempty[:-1]:
        if lens[r] % chunk != 0:
            raise ValueError(f"span lengths {lens}: span {r} is not a whole number of "
                             f"{chunk}-token chunks")


def exclusive_scan(delta, engine, world: int, rank: int, group=None):
    """(sum of the deltas of ranks < rank, sum of ranks <= rank) by recursive
    doubling: in round k each rank sends its running sum to rank + k and adds
    the one received from rank - k in front of its own (ranks in order), then
    one shift turns the inclusive sums into exclusive ones.  None stands for
    an empty sum (rank 0's exclusive prefix)."""
    incl = delta.contiguous()
    k = 1
    while k < world:
        ops, recv = [], None
        if rank + k < world:
            ops.append(dist.P2POp(dist.isend, incl, rank + k, group))
        if rank - k >= 0:
            recv = torch.empty_like(incl)
            ops.append(dist.P2POp(dist.irecv, recv, rank - k, group))
        for req in (dist.batch_isend_irecv(ops) if ops else []):
            req.wait()
        if recv is not None:
            incl = engine.add(recv, incl)
        k *= 2
    ops, excl = [], None
    if rank + 1 < world:
        ops.append(dist.P2POp(dist.isend, incl, rank + 1, group))
    if rank >= 1:
        excl = torch.empty_like(incl)
        ops.append(dist.P2POp(dist.irecv, excl, rank - 1, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return excl, incl


def sequence_parallel_forward(H, X0, W_gate, W_up, W_down0, W_target, conv_w, eta: float,
                              chunk: int, *, eta_tok=None, group=None, engine=None,
                              want_state: bool = False, exchange: str = "allgather"):
    """This rank's part of a sequence-sharded forward.

    H, X0 [B, T_r, d] (and eta_tok [B, T_r]) hold this rank's span of every
    sequence, as `sequence_span` assigns it: a multiple of `chunk` tokens
    except on the last non-empty span, possibly empty.  Every rank of
    `group` must call this together (the deltas are all-gathered).  Returns
    O [B, T_r, d] for the span and, with `want_state`, the fast weight after
    the span (on the last rank: after the whole sequence).  The convolution
    is zero-padded at chunk edges (the default pad mode), so no token crosses
    a span boundary.  `exchange`: "allgather" (the prefix adds the deltas in
    rank order) or "scan" (recursive doubling; the same sum in tree order).
    """
    if exchange not in ("allgather", "scan"):
        raise ValueError(f"exchange {exchange!r}")
    engine = engine or CudaEngine()
    if dist.is_available() and dist.is_initialized():
        world, rank = dist.get_world_size(group), dist.get_rank(group)
    else:
        world, rank = 1, 0
    B, T_r, d = H.shape
    f = W_gate.shape[0]
    if world > 1:
        check_spans(T_r, chunk, world, group, H.device)
    if T_r > 0:
        delta, zv = engine.fold(H, X0, W_gate, W_up, W_target, conv_w, eta, chunk,
                                eta_tok=eta_tok)
    else:
        delta, zv = engine.zeros(B, d, f, H.device), None
    if world > 1 and exchange == "scan":
        excl, incl = exclusive_scan(delta, engine, world, rank, group)
        state_in = (engine.prefix(W_down0, delta.unsqueeze(0), 0) if excl is None
                    else engine.prefix(W_down0, excl.unsqueeze(0), 1))
        after = lambda: engine.prefix(W_down0, incl.unsqueeze(0), 1)  # noqa: E731
    else:
        if world > 1:
            deltas = delta.new_empty((world,) + tuple(delta.shape))
            dist.all_gather(list(deltas.unbind(0)), delta, group=group)
        else:
            deltas = delta.unsqueeze(0)
        state_in = engine.prefix(W_down0, deltas, rank)
        after = lambda: engine.prefix(W_down0, deltas, rank + 1)  # noqa: E731
    if T_r > 0:
        O = engine.apply(H, X0, W_gate, W_up, W_target, conv_w, eta, chunk, zv, state_in)
    else:
        O = H.new_empty((B, 0, d))
    if want_state:
        return O, after()
    return O
