"""The oracle over whole full-size tensors, on every host core.

Lanes (b, d) of the scan are independent, so the oracle's sequential forward
and backward can run on disjoint (batch row, lane slice) blocks in separate
processes and give exactly what one call over the whole tensor gives.  The
inputs and results live in shared memory; workers are spawn-started (a fork
after CUDA initialisation is unsafe), and each runs the oracle as it stands
on its blocks.  Test infrastructure only.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import sys
from concurrent.futures import ProcessPoolExecutor
from multiprocessing import shared_memory

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)


class Shared:
    """A numpy array in a named shared-memory block (owned by the creator)."""

    def __init__(self, shape, dtype, name=None):
        self.shape, self.dtype = tuple(shape), np.dtype(dtype)
        nbytes = max(1, int(np.prod(self.shape)) * self.dtype.itemsize)
        if name is None:
            self.shm = shared_memory.SharedMemory(create=True, size=nbytes)
            self.owner = True
        else:
            self.shm = shared_memory.SharedMemory(name=name)
            self.owner = False
        self.array = np.ndarray(self.shape, dtype=self.dtype, buffer=self.shm.buf)

    def spec(self):
        return (self.shm.name, self.shape, self.dtype.str)

    def close(self):
        self.array = None
        self.shm.close()
        if self.owner:
            self.shm.unlink()


def _blocks(B: int, D: int, T: int, jobs: int):
    """(b, d0, d1) blocks: about 4 per job, lane slices of at least 16."""
    per_row = max(1, min(D // 16 if D >= 16 else 1, -(-4 * jobs // max(1, B))))
    out = []
    for b in range(B):
        cuts = [D * i // per_row for i in range(per_row + 1)]
        out += [(b, cuts[i], cuts[i + 1]) for i in range(per_row) if cuts[i + 1] > cuts[i]]
    return out


def _worker(task):
    kind, dtype, specs, blocks = task
    if _ROOT not in sys.path:
        sys.path.insert(0, _ROOT)
    import oracle
    o = oracle.default()
    arrs = {k: Shared(s[1], s[2], name=s[0]) for k, s in specs.items()}
    try:
        A = {k: v.array for k, v in arrs.items()}
        for (b, d0, d1) in blocks:
            sl = np.s_[b:b + 1, :, d0:d1]
            if kind == "fwd":
                out, last = o.fwd(np.ascontiguousarray(A["a"][sl]), np.ascontiguousarray(A["b"][sl]), dtype)
                A["out"][sl] = out
                A["last"][b:b + 1, d0:d1] = last
            else:
                ga, gb = o.bwd(np.ascontiguousarray(A["a"][sl]), np.ascontiguousarray(A["out"][sl]),
                               np.ascontiguousarray(A["g"][sl]), dtype)
                A["ga"][sl] = ga
                A["gb"][sl] = gb
    finally:
        for v in arrs.values():
            v.close()
    return len(blocks)


class OraclePool:
    """Full-size oracle runs on `processes` spawn-started workers."""

    def __init__(self, processes: int | None = None):
        self.n = max(1, processes or min(32, os.cpu_count() or 1))
        self.pool = ProcessPoolExecutor(max_workers=self.n, mp_context=mp.get_context("spawn"))

    def close(self):
        self.pool.shutdown(wait=True)

    def _run(self, kind, dtype, ins: dict, outs: dict):
        shared = {}
        try:
            for k, x in ins.items():
                s = Shared(x.shape, x.dtype)
                s.array[...] = x
                shared[k] = s
            for k, (shape, dt) in outs.items():
                shared[k] = Shared(shape, dt)
            B, T, D = next(iter(ins.values())).shape
            blocks = _blocks(B, D, T, self.n)
            specs = {k: s.spec() for k, s in shared.items()}
            tasks = [(kind, dtype, specs, blocks[i::self.n]) for i in range(self.n) if blocks[i::self.n]]
            done = sum(self.pool.map(_worker, tasks))
            assert done == len(blocks)
            return {k: shared[k].array.copy() for k in outs}
        finally:
            for s in shared.values():
                s.close()

    def fwd(self, a: np.ndarray, b: np.ndarray, dtype: str):
        """The oracle's forward over the whole [B, T, D] tensors; ``(out, last)``."""
        B, T, D = a.shape
        r = self._run("fwd", dtype, {"a": a, "b": b},
                      {"out": (a.shape, a.dtype), "last": ((B, D), np.float32)})
        return r["out"], r["last"]

    def bwd(self, a: np.ndarray, out: np.ndarray, g: np.ndarray, dtype: str):
        """The oracle's backward over the whole tensors; ``(grad_a, grad_b)``."""
        r = self._run("bwd", dtype, {"a": a, "out": out, "g": g},
                      {"ga": (a.shape, a.dtype), "gb": (a.shape, a.dtype)})
        return r["ga"], r["gb"]
