"""Seeded synthetic inputs for the diagonal linear-recurrence scan.

This module only draws random numbers; it holds none of the scan's arithmetic,
so both the CUDA path and the CPU oracle can be fed from it.  Every tensor is
drawn in fp32 on the host with ``torch.Generator('cpu')`` and then stored in
the workload's storage dtype (round-to-nearest-even for bf16), so both sides
read the very same stored bits.

The five named workloads are the shapes and value distributions the scan is
measured on (all contiguous [B, T, D], D fastest):

  1  tiny fp32            B=1  T=64    D=256   a~U(0.80,0.999)  b,g~N(0,1)
  2  gated bf16           B=8  T=2048  D=2560  a=exp(-8*softplus(x)*r),
                                               x~N(0,1), r~U(0,1); b,g~N(0,1)
  3  long-sequence fp32   B=1  T=65536 D=2560  a~U(0.90,0.9999)  b,g~N(0,1)
                                               (chunk length 64)
  4  near-unit bf16       B=16 T=4096  D=4096  a~U(0.99,0.9999)  b~N(0,0.1^2)
                                               g~N(0,1)
  5  padded fp32          B=64 T=512   D=1024  valid length L_b~U{64..512};
                                               valid a~U(0.5,0.999), b,g~N(0,1);
                                               padded a=1, b=0, g=0

The decay of workload 2 is the RG-LRU style gate the first page's docstring
points to (RecurrentGemma); softplus(x) = log1p(exp(x)) is evaluated by
PyTorch on the host in fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED_BASE = 20260


@dataclass(frozen=True)
class Workload:
    cid: int
    name: str
    B: int
    T: int
    D: int
    dtype: str               # storage dtype: "f32" or "bf16"
    chunk: int | None = None
    padded: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def elements(self) -> int:
        return self.B * self.T * self.D

    @property
    def storage_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def describe(self) -> str:
        s = f"{self.name}: B={self.B} T={self.T} D={self.D} {self.dtype}"
        if self.chunk:
            s += f" chunk={self.chunk}"
        return s


WORKLOADS: dict[int, Workload] = {
    1: Workload(1, "tiny-fp32", 1, 64, 256, "f32"),
    2: Workload(2, "gated-bf16", 8, 2048, 2560, "bf16"),
    3: Workload(3, "long-seq-fp32", 1, 65536, 2560, "f32", chunk=64),
    4: Workload(4, "near-unit-bf16", 16, 4096, 4096, "bf16"),
    5: Workload(5, "padded-fp32", 64, 512, 1024, "f32", padded=True),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _uniform(gen, shape, lo, hi):
    return torch.empty(shape, dtype=torch.float32).uniform_(lo, hi, generator=gen)


def _normal(gen, shape, std=1.0):
    return torch.empty(shape, dtype=torch.float32).normal_(0.0, std, generator=gen)


def make_inputs(cid: int, *, B: int | None = None, T: int | None = None,
                D: int | None = None, seed: int | None = None) -> dict:
    """Draw (a, b, grad_out) for workload ``cid``; shape overrides keep its distributions.

    Returns a dict of CPU tensors in the storage dtype plus ``lengths`` (a
    [B] int64 tensor of valid lengths; T for unpadded workloads) and the
    ``workload`` record.
    """
    w = WORKLOADS[cid]
    B = w.B if B is None else B
    T = w.T if T is None else T
    D = w.D if D is None else D
    gen = torch.Generator("cpu").manual_seed(SEED_BASE + cid if seed is None else seed)
    shape = (B, T, D)
    lengths = torch.full((B,), T, dtype=torch.int64)
    if cid == 1:
        a = _uniform(gen, shape, 0.80, 0.999)
        b = _normal(gen, shape)
        g = _normal(gen, shape)
    elif cid == 2:
        x = _normal(gen, shape)
        r = _uniform(gen, shape, 0.0, 1.0)
        a = torch.exp(-8.0 * torch.nn.functional.softplus(x) * r)
        del x, r
        b = _normal(gen, shape)
        g = _normal(gen, shape)
    elif cid == 3:
        a = _uniform(gen, shape, 0.90, 0.9999)
        b = _normal(gen, shape)
        g = _normal(gen, shape)
    elif cid == 4:
        a = _uniform(gen, shape, 0.99, 0.9999)
        b = _normal(gen, shape, 0.1)
        g = _normal(gen, shape)
    elif cid == 5:
        lo = min(64, T)
        lengths = torch.randint(lo, T + 1, (B,), generator=gen, dtype=torch.int64)
        a = _uniform(gen, shape, 0.5, 0.999)
        b = _normal(gen, shape)
        g = _normal(gen, shape)
        pad = torch.arange(T)[None, :] >= lengths[:, None]          # [B, T]
        pad = pad[:, :, None].expand(shape)
        a[pad] = 1.0
        b[pad] = 0.0
        g[pad] = 0.0
    else:
        raise KeyError(cid)
    dt = TORCH_DTYPE[w.dtype]
    return {
        "a": a.to(dt).contiguous(),
        "b": b.to(dt).contiguous(),
        "grad_out": g.to(dt).contiguous(),
        "lengths": lengths,
        "workload": w,
        "shape": shape,
    }


def random_inputs(B: int, T: int, D: int, dtype: str = "f32", *, seed: int = 0,
                  a_lo: float = 0.5, a_hi: float = 0.999) -> dict:
    """Generic seeded case: a~U(a_lo,a_hi), b~N(0,1), grad_out~N(0,1)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    shape = (B, T, D)
    a = _uniform(gen, shape, a_lo, a_hi)
    b = _normal(gen, shape)
    g = _normal(gen, shape)
    dt = TORCH_DTYPE[dtype]
    return {"a": a.to(dt).contiguous(), "b": b.to(dt).contiguous(),
            "grad_out": g.to(dt).contiguous(),
            "lengths": torch.full((B,), T, dtype=torch.int64), "shape": shape}


# Complex scan workload (re/im planes).  The pages fix no complex workload
# sizes; this one has the shape and the decay magnitude of the gated bf16
# workload, with a uniformly random phase per (b, t, d).
COMPLEX_WORKLOAD = Workload(6, "complex-gated-bf16", 8, 2048, 2560, "bf16")


def make_complex_inputs(B: int | None = None, T: int | None = None, D: int | None = None, dtype: str | None = None,
                        *, seed: int | None = None) -> dict:
    """Draw the six planes (ar, ai, br, bi, go_r, go_i) of a complex scan:
    |a| = exp(-8*softplus(x)*r), x~N(0,1), r~U(0,1); arg a ~ U(-pi, pi);
    b and grad_out planes ~N(0,1).  Drawn in fp32, stored in `dtype`."""
    w = COMPLEX_WORKLOAD
    B = w.B if B is None else B
    T = w.T if T is None else T
    D = w.D if D is None else D
    dtype = w.dtype if dtype is None else dtype
    gen = torch.Generator("cpu").manual_seed(SEED_BASE + w.cid if seed is None else seed)
    shape = (B, T, D)
    x = _normal(gen, shape)
    r = _uniform(gen, shape, 0.0, 1.0)
    rad = torch.exp(-8.0 * torch.nn.functional.softplus(x) * r)
    del x, r
    ang = _uniform(gen, shape, -3.141592653589793, 3.141592653589793)
    planes = {"ar": rad * torch.cos(ang), "ai": rad * torch.sin(ang)}
    del rad, ang
    for k in ("br", "bi", "go_r", "go_i"):
        planes[k] = _normal(gen, shape)
    dt = TORCH_DTYPE[dtype]
    return {k: v.to(dt).contiguous() for k, v in planes.items()} | {"shape": shape, "workload": w}


# Generated-decay workload: the gated workload's shape, with the decay
# parametrized per token (eta) and per lane (nu_log) instead of stored.
GATED_WORKLOAD = Workload(7, "generated-decay-bf16", 8, 2048, 2560, "bf16")


def make_gated_inputs(B: int | None = None, T: int | None = None, D: int | None = None, dtype: str | None = None,
                      *, seed: int | None = None) -> dict:
    """eta ~ N(-1, 1) fp32 [B, T], nu_log ~ U(-2, 1) fp32 [D] (so decays spread
    over (0, 1) like the gated workload's), b and grad_out ~ N(0, 1) [B, T, D]
    in `dtype`."""
    w = GATED_WORKLOAD
    B = w.B if B is None else B
    T = w.T if T is None else T
    D = w.D if D is None else D
    dtype = w.dtype if dtype is None else dtype
    gen = torch.Generator("cpu").manual_seed(SEED_BASE + w.cid if seed is None else seed)
    eta = _normal(gen, (B, T)) - 1.0
    nu_log = _uniform(gen, (D,), -2.0, 1.0)
    b = _normal(gen, (B, T, D))
    g = _normal(gen, (B, T, D))
    dt = TORCH_DTYPE[dtype]
    return {"eta": eta.contiguous(), "nu_log": nu_log.contiguous(), "b": b.to(dt).contiguous(),
            "grad_out": g.to(dt).contiguous(), "shape": (B, T, D), "workload": w}


def to_numpy_storage(t: torch.Tensor):
    """CPU tensor -> numpy array as the oracle takes it (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def from_numpy_storage(x, dtype: str) -> torch.Tensor:
    """numpy storage array (bf16 as uint16 bits) -> CPU tensor of that dtype."""
    import numpy as np
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view("int16")).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))
