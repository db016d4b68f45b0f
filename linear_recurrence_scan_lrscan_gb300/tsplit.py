"""Sequence split across ranks: every rank holds one contiguous time segment
of all lanes, and one exchange of per-lane affine maps makes the ranks'
segment scans equal the whole-sequence scan.

This is the two-level decomposition of triton_training_scan.py
(_real_chunk_summary, _real_chunk_prefix, _real_chunk_replay and the reverse
mirror) with one chunk per rank:

  forward   1. each rank summarizes its segment as h -> P*h + Q (lrscan_summary);
            2. all-gather of the [2, B, D] fp32 maps (the only exchange);
            3. rank r composes the maps of ranks 0..r-1, in order, over the
               sequence's initial state: its incoming state h_in;
            4. each rank scans its segment from h_in (lrscan_fwd_state).
  backward  the same with the backward summary g -> P*g + Q of each segment
            (grad_last -> grad_h0), composed from the last rank down over the
            sequence's grad_last; each rank then runs lrscan_bwd_state with
            h0 = its h_in and grad_last = its incoming adjoint.  Rank 0's
            grad_h0 is the gradient of the sequence's initial state.

Composition order matters (maps compose as current ∘ accumulated, which is
associative but not commutative): forward, h_in = fold of h -> P_r*h + Q_r
over r = 0..rank-1; backward, over r = W-1..rank+1.  All arithmetic, the
composition included, is done by ``ops``: by default the CUDA library
(lrscan_summary, lrscan_compose_maps, lrscan_fwd_state, lrscan_bwd_state);
tests may pass any object with the same four methods.
"""
from __future__ import annotations

import torch


class LibraryOps:
    """Local segment work on this rank's GPU through the C ABI."""

    def summary(self, a, x, segment_pos, direction):
        from .lrscan import lrscan_summary
        P, Q = lrscan_summary(a, x, segment_pos=segment_pos, direction=direction)
        return torch.stack([P, Q])

    def compose(self, maps, rank, init, direction):
        from .lrscan import lrscan_compose_maps
        return lrscan_compose_maps(torch.stack(maps), rank, init, direction)

    def fwd_state(self, a, b, h0, segment_pos):
        from .lrscan import lrscan_fwd_state
        return lrscan_fwd_state(a, b, h0=h0, segment_pos=segment_pos)

    def bwd_state(self, a, out, grad_out, h0, segment_pos, grad_last):
        from .lrscan import lrscan_bwd_state
        return lrscan_bwd_state(a, out, grad_out, h0=h0, segment_pos=segment_pos, grad_last=grad_last)


def _rank(group) -> int:
    import torch.distributed as dist
    return dist.get_rank(group)


def all_gather_maps(local: torch.Tensor, group=None) -> list[torch.Tensor]:
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(out, local.contiguous(), group=group)
    return out


def tsplit_forward(a, b, *, h0=None, segment_pos=None, group=None, ops=None, gather=all_gather_maps, rank=None):
    """This rank's segment of the whole-sequence forward scan.

    a, b: [B, T_r, D] (this rank's time segment); h0: the sequence's initial
    state [B, D] fp32 (same on every rank) or None; segment_pos: this
    segment's [B, T_r] positions or None.  Returns (out, last, h_in): the
    segment's outputs, its final state (the sequence's on the last rank) and
    the state that entered it (needed by the backward).  `rank` defaults to
    the process's rank in `group`; `gather` to an all-gather over `group`."""
    ops = ops or LibraryOps()
    rank = _rank(group) if rank is None else rank
    maps = gather(ops.summary(a, b, segment_pos, "fwd"), group)
    h_in = ops.compose(maps, rank, h0, "fwd")
    out, last = ops.fwd_state(a, b, h_in, segment_pos)
    return out, last, h_in


def tsplit_backward(a, out, grad_out, *, h_in, segment_pos=None, grad_last=None, group=None, ops=None,
                    gather=all_gather_maps, rank=None):
    """This rank's segment of the whole-sequence backward scan; grad_last is
    the gradient at the sequence's final state (same on every rank) or None.
    Returns (grad_a, grad_b, grad_h0): grad_h0 of rank 0 is the gradient of
    the sequence's initial state."""
    ops = ops or LibraryOps()
    rank = _rank(group) if rank is None else rank
    maps = gather(ops.summary(a, grad_out, segment_pos, "bwd"), group)
    g_in = ops.compose(maps, rank, grad_last, "bwd")
    return ops.bwd_state(a, out, grad_out, h_in, segment_pos, g_in)
