"""Host-buffer entry points (lrscan_fwd_host, lrscan_bwd_host,
lrscan_fwd_bwd_host): the operands live in host memory and the library
pipelines the copies with the kernels over batch-row chunks.

GPU tests compare them with the oracle (exactly on the sequential path,
whose order of operations is the oracle's) and with the device entry points
on the same tile variant (bit for bit: a lane's arithmetic does not depend on
which chunk of batch rows it was launched in).  The CPU tests cover what
needs no device: T == 0 and argument checks.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS, make_inputs, random_inputs
from parity_util import assert_close, assert_last_close, to_np


def test_no_steps_writes_zero_last_without_a_device():
    a = torch.empty((3, 0, 16))
    last = torch.full((3, 16), 7.0)
    out = torch.empty_like(a)
    L.lrscan_fwd_host(a, a, out=out, last=last)
    assert not last.any()
    ga, gb = torch.empty_like(a), torch.empty_like(a)
    L.lrscan_bwd_host(a, a, a, grad_a=ga, grad_b=gb)  # nothing to do


def test_host_argument_checks():
    a = torch.zeros((2, 4, 8))
    with pytest.raises(ValueError):
        L.lrscan_fwd_host(a, torch.zeros((2, 4, 9)), out=torch.empty_like(a), last=torch.empty(2, 8))
    with pytest.raises(ValueError):
        L.lrscan_fwd_host(a, a, out=torch.empty_like(a), last=torch.empty(2, 9))
    with pytest.raises(ValueError):
        L.lrscan_fwd_host(a, a.to(torch.bfloat16), out=torch.empty_like(a), last=torch.empty(2, 8))


gpu = pytest.mark.gpu


@pytest.fixture()
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    yield
    assert L.lrscan_sync_check() == 0


def _pinned(t):
    return t.contiguous().pin_memory()


@gpu
@pytest.mark.parametrize("dt,shape", [("f32", (5, 300, 200)), ("bf16", (3, 257, 1000)), ("f32", (1, 129, 16)),
                                      ("bf16", (7, 64, 40))])
def test_host_calls_match_the_oracle(_cuda, dt, shape):
    """Sequential path: exact; the oracle's forward output feeds the backward."""
    inp = random_inputs(*shape, dt, seed=900 + shape[0])
    a, b, g = (_pinned(inp[k]) for k in ("a", "b", "grad_out"))
    o = oracle.default()
    ref_out, ref_last = o.fwd(to_np(a), to_np(b), dt)
    out, last = L.lrscan_fwd_host(a, b, path="seq")
    assert_close(to_np(out), ref_out, dt, "out (host, seq)", exact=True)
    assert_last_close(last.numpy(), ref_last, "last (host, seq)", exact=True)
    out_ref_t = torch.from_numpy(np.ascontiguousarray(ref_out).view(np.int16)).view(torch.bfloat16) \
        if dt == "bf16" else torch.from_numpy(ref_out)
    ref_ga, ref_gb = o.bwd(to_np(a), ref_out, to_np(g), dt)
    ga, gb = L.lrscan_bwd_host(a, _pinned(out_ref_t), g, path="seq")
    assert_close(to_np(ga), ref_ga, dt, "grad_a (host, seq)", exact=True)
    assert_close(to_np(gb), ref_gb, dt, "grad_b (host, seq)", exact=True)
    # auto path (windowed tiles reassociate): tolerance
    out2, last2, ga2, gb2 = L.lrscan_fwd_bwd_host(a, b, g)
    assert_close(to_np(out2), ref_out, dt, "out (host, auto)", reassociated=True)
    assert_last_close(last2.numpy(), ref_last, "last (host, auto)")


def _window_variant(B, T, D, dt, name):
    v = 1
    while True:
        if L.lrscan_plan(B, T, D, dt, "fwd", path="window", tile_variant=v)["name"] == name:
            return v
        v += 1


@gpu
@pytest.mark.parametrize("pinned", [True, False])
def test_fwd_bwd_host_equals_device_calls_bit_for_bit(_cuda, pinned):
    """Same tile variant on the device: identical bits, whatever the chunking
    (B = 9 gives chunks of 3 rows) and whether the host memory is pinned."""
    B, T, D, dt = 9, 200, 320, "bf16"
    inp = random_inputs(B, T, D, dt, seed=910)
    hv = {k: (_pinned(inp[k]) if pinned else inp[k].contiguous()) for k in ("a", "b", "grad_out")}
    kw = dict(path="window", tile_variant=_window_variant(B, T, D, dt, "win_bf16_d32_s8_m5_n2"))
    out_h, last_h, ga_h, gb_h = L.lrscan_fwd_bwd_host(hv["a"], hv["b"], hv["grad_out"], **kw)
    ad, bd, gd = (inp[k].cuda() for k in ("a", "b", "grad_out"))
    out_d, last_d = L.lrscan_fwd(ad, bd, **kw)
    ga_d, gb_d = L.lrscan_bwd(ad, out_d, gd, **kw)
    assert L.lrscan_sync_check() == 0
    for name, h, d in (("out", out_h, out_d), ("grad_a", ga_h, ga_d), ("grad_b", gb_h, gb_d)):
        assert torch.equal(h.view(torch.int16), d.cpu().view(torch.int16)), name
    assert torch.equal(last_h, last_d.cpu())


@gpu
def test_host_unaligned_rows_and_single_row(_cuda):
    """D*2 not a multiple of 16 takes the plain path per chunk; B = 1 is one chunk."""
    for (B, T, D) in ((3, 50, 37), (1, 300, 64)):
        inp = random_inputs(B, T, D, "bf16", seed=920 + D)
        a, b, g = (_pinned(inp[k]) for k in ("a", "b", "grad_out"))
        o = oracle.default()
        ref_out, ref_last = o.fwd(to_np(a), to_np(b), "bf16")
        out, last, ga, gb = L.lrscan_fwd_bwd_host(a, b, g)
        assert_close(to_np(out), ref_out, "bf16", f"out {B, T, D}", reassociated=True)
        assert_last_close(last.numpy(), ref_last, f"last {B, T, D}")


@gpu
def test_host_full_size_workload_matches_device(_cuda):
    """The gated bf16 workload at full size through the host pipeline (chunks
    of ceil(B / 8) rows) against the device calls on the same tiles."""
    w = WORKLOADS[2]
    inp = make_inputs(2)
    a, b, g = (_pinned(inp[k]) for k in ("a", "b", "grad_out"))
    out_h, last_h, ga_h, gb_h = L.lrscan_fwd_bwd_host(a, b, g)
    ad, bd, gd = a.cuda(), b.cuda(), g.cuda()
    # the device calls below run the tiles the host call's chunks planned
    rows = -(-w.B // 8)
    pf = L.lrscan_plan(rows, w.T, w.D, w.dtype, "fwd")
    pb = L.lrscan_plan(rows, w.T, w.D, w.dtype, "bwd")
    kf = dict(path=pf["path"], tile_variant=pf["tile_variant"])
    kb = dict(path=pb["path"], tile_variant=pb["tile_variant"])
    out_d, last_d = L.lrscan_fwd(ad, bd, **kf)
    ga_d, gb_d = L.lrscan_bwd(ad, out_d, gd, **kb)
    assert L.lrscan_sync_check() == 0
    for name, h, d in (("out", out_h, out_d), ("grad_a", ga_h, ga_d), ("grad_b", gb_h, gb_d)):
        assert torch.equal(h.view(torch.int16), d.cpu().view(torch.int16)), name
    assert torch.equal(last_h, last_d.cpu())


@gpu
def test_host_call_reports_a_chunk_error_and_stays_usable(_cuda):
    """A chunk whose device call fails (the tiled path forced on rows that are
    not 16-byte multiples) stops the call with the error; the next call runs."""
    inp = random_inputs(4, 40, 37, "bf16", seed=930)
    a, b, g = (_pinned(inp[k]) for k in ("a", "b", "grad_out"))
    with pytest.raises(L.LrscanError):
        L.lrscan_fwd_bwd_host(a, b, g, path="seq")
    out, last = L.lrscan_fwd_host(a, b)
    ref_out, _ = oracle.default().fwd(to_np(a), to_np(b), "bf16")
    assert_close(to_np(out), ref_out, "bf16", "out after a failed call", reassociated=True)
