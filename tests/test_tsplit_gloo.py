"""The sequence-split protocol across ranks (linear_recurrence_scan_lrscan_gb300.tsplit)
on CPU: world_size 2 and 3 `gloo` process groups, each rank holding one time
segment.  The local work is done by the oracle (fp64) through the protocol's
`ops` hook; the gathered segments must reproduce the oracle's whole-sequence
state-carrying scan (forward outputs and final state, backward gradients and
the initial-state gradient) to fp64 rounding."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """Local segment work by the CPU oracle (fp64)."""

    def __init__(self):
        import oracle
        self.o = oracle.default()

    @staticmethod
    def _np(t):
        return None if t is None else np.ascontiguousarray(t.numpy())

    def summary(self, a, x, segment_pos, direction):
        a, x, seg = self._np(a), self._np(x), self._np(segment_pos)
        B, T, D = a.shape
        if direction == "fwd":
            # P: the state reached from h0 = 1 with no input; Q: from h0 = 0
            _, P = self.o.fwd_state(a, np.zeros_like(a), "f64", h0=np.ones((B, D)), segment_pos=seg)
            _, Q = self.o.fwd_state(a, x, "f64", segment_pos=seg)
        else:
            z = np.zeros_like(a)
            _, _, P = self.o.bwd_state(a, z, z, "f64", segment_pos=seg, grad_last=np.ones((B, D)))
            _, _, Q = self.o.bwd_state(a, z, x, "f64", segment_pos=seg)
        return torch.from_numpy(np.stack([P, Q]))

    def compose(self, maps, rank, init, direction):
        W = len(maps)
        order = range(rank) if direction == "fwd" else range(W - 1, rank, -1)
        h = torch.zeros_like(maps[0][0]) if init is None else init.clone()
        for r in order:
            h = maps[r][0] * h + maps[r][1]
        return h

    def fwd_state(self, a, b, h0, segment_pos):
        out, last = self.o.fwd_state(self._np(a), self._np(b), "f64", h0=self._np(h0),
                                     segment_pos=self._np(segment_pos))
        return torch.from_numpy(out), torch.from_numpy(last)

    def bwd_state(self, a, out, grad_out, h0, segment_pos, grad_last):
        ga, gb, gh0 = self.o.bwd_state(self._np(a), self._np(out), self._np(grad_out), "f64", h0=self._np(h0),
                                       segment_pos=self._np(segment_pos), grad_last=self._np(grad_last))
        return torch.from_numpy(ga), torch.from_numpy(gb), torch.from_numpy(gh0)


def _problem(B=2, T=61, D=3):
    r = np.random.default_rng(5)
    a = r.uniform(0.6, 1.0, (B, T, D))
    b = r.standard_normal((B, T, D))
    g = r.standard_normal((B, T, D))
    h0 = r.standard_normal((B, D))
    gl = r.standard_normal((B, D))
    seg = np.ones((B, T), dtype=np.int32)
    seg[0, 0] = 0
    seg[0, 20] = 0
    seg[1, 33] = 0
    return a, b, g, h0, gl, seg


def _bounds(T, W):
    """Segment boundaries of W ranks (uneven on purpose)."""
    return [0, 7, 30, 45][:W] + [T]


def _rank_main(rank, world, port, result_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from linear_recurrence_scan_lrscan_gb300 import tsplit
        a, b, g, h0, gl, seg = _problem()
        cuts = _bounds(a.shape[1], world)
        lo, hi = cuts[rank], cuts[rank + 1]
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x))  # noqa: E731
        ops = OracleOps()
        sa, sb, sg, sseg = t(a[:, lo:hi]), t(b[:, lo:hi]), t(g[:, lo:hi]), t(seg[:, lo:hi])
        out, last, h_in = tsplit.tsplit_forward(sa, sb, h0=t(h0), segment_pos=sseg, ops=ops)
        ga, gb, gh0 = tsplit.tsplit_backward(sa, out, sg, h_in=h_in, segment_pos=sseg, grad_last=t(gl), ops=ops)
        np.savez(os.path.join(result_dir, f"r{rank}.npz"), out=out.numpy(), last=last.numpy(), ga=ga.numpy(),
                 gb=gb.numpy(), gh0=gh0.numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sequence_split_matches_whole_sequence(world, tmp_path, oracle_handle):
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    a, b, g, h0, gl, seg = _problem()
    out, last = oracle_handle.fwd_state(a, b, "f64", h0=h0, segment_pos=seg)
    ga, gb, gh0 = oracle_handle.bwd_state(a, out, g, "f64", h0=h0, segment_pos=seg, grad_last=gl)
    parts = [np.load(tmp_path / f"r{r}.npz") for r in range(world)]
    cat = lambda k: np.concatenate([p[k] for p in parts], axis=1)  # noqa: E731
    np.testing.assert_allclose(cat("out"), out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(parts[-1]["last"], last, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(cat("gb"), gb, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(cat("ga"), ga, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(parts[0]["gh0"], gh0, rtol=1e-12, atol=1e-12)
    # the protocol is not vacuous: without the exchange later segments differ
    alone, _ = oracle_handle.fwd_state(np.ascontiguousarray(a[:, 7:30]), np.ascontiguousarray(b[:, 7:30]), "f64",
                                       segment_pos=np.ascontiguousarray(seg[:, 7:30]))
    assert not np.allclose(alone, out[:, 7:30])


def _bench_rank(rank, world, port, result_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [1.0 + rank, 0.25 * (world - rank), 3.0]          # per-rank timings (ms)
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        value = bench.job_throughput(world, 1000, got[0])
        np.save(os.path.join(result_dir, f"b{rank}.npy"), np.array(got + [value]))
    finally:
        dist.destroy_process_group()


def test_bench_takes_the_slowest_rank(tmp_path):
    """The benchmark's multi-rank reduction: every rank ends with the slowest
    rank's times, and the job's value counts every rank's units over them."""
    world = 2
    mp.start_processes(_bench_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        got = np.load(tmp_path / f"b{r}.npy")
        assert got[:3].tolist() == [2.0, 0.5, 3.0]
        assert got[3] == pytest.approx(world * 1000 / 2.0e-3)
