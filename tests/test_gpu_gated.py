"""GPU parity of the scan with generated decays exp(-exp(nu_log_d) exp(eta_t))
against the oracle.  The kernels use the hardware's fast exponential, so
every output is held to the tolerances of parity_util (fp32 rule, 2 bf16 ulps
with the near-cancellation clause); grad_eta and grad_nu_log are fp32 sums
compared with the fp32 rule against the oracle's double-accumulated sums."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import GATED_WORKLOAD, make_gated_inputs
from parity_util import bf16_beyond_ulps, assert_close, assert_last_close, assert_sum_close, bf16_bits_to_f32, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    yield
    assert L.lrscan_sync_check() == 0


def from_np(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))


def abs_terms(eta, nu_log, out, grad_out, dt):
    """sum|q| per token and per lane, q = grad_a * a * log a, from the fp64
    plain oracle on the materialized decays (the scale of the summed terms)."""
    w = (lambda x: bf16_bits_to_f32(x).astype(np.float64)) if dt == "bf16" else (lambda x: x.astype(np.float64))
    la = -np.exp(nu_log.astype(np.float64))[None, None, :] * np.exp(eta.astype(np.float64))[:, :, None]
    a = np.exp(la)
    ga, _ = oracle.default().bwd(a, w(out), w(grad_out), "f64")
    q = np.abs(ga * a * la)
    return q.sum(axis=2), q.sum(axis=(0, 1))


def check_gated(inp, dt, **kw):
    B, T, D = inp["shape"]
    eta, nu = inp["eta"].numpy(), inp["nu_log"].numpy()
    b, g = to_np(inp["b"]), to_np(inp["grad_out"])
    o = oracle.default()
    ref_out, ref_last = o.gated_fwd(eta, nu, b, dt)
    etad, nud = inp["eta"].cuda(), inp["nu_log"].cuda()
    out, last = L.lrscan_fwd_gated(etad, nud, inp["b"].cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    plan = L.lrscan_plan_gated(B, T, D, dt, "fwd", **kw)
    assert_close(to_np(out), ref_out, dt, f"out[{plan['name']}]", reassociated=True)
    assert_last_close(last.cpu().numpy(), ref_last, f"last[{plan['name']}]")
    ref_gb, ref_geta, ref_gnu = o.gated_bwd(eta, nu, ref_out, g, dt)
    gb, geta, gnu = L.lrscan_bwd_gated(etad, nud, from_np(ref_out, dt).cuda(), inp["grad_out"].cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    planb = L.lrscan_plan_gated(B, T, D, dt, "bwd", **kw)
    assert_close(to_np(gb), ref_gb, dt, f"grad_b[{planb['name']}]", reassociated=True)
    s_eta, s_nu = abs_terms(eta, nu, ref_out, g, dt)
    assert_sum_close(geta.cpu().numpy(), ref_geta, s_eta, f"grad_eta[{planb['name']}]")
    assert_sum_close(gnu.cpu().numpy(), ref_gnu, s_nu, f"grad_nu_log[{planb['name']}]")
    return plan, planb


SHAPES = [(3, 300, 200), (2, 77, 40), (1, 1, 8), (2, 257, 1000), (1, 33, 64)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_gated_every_variant_and_plain(dt, shape):
    B, T, D = shape
    inp = make_gated_inputs(B, T, D, dt, seed=700 + T)
    v = 1
    while True:
        try:
            L.lrscan_plan_gated(B, T, D, dt, path="seq", tile_variant=v)
        except L.LrscanError:
            break
        check_gated(inp, dt, path="seq", tile_variant=v)
        v += 1
    assert v > 2
    check_gated(inp, dt, path="plain")
    plan, planb = check_gated(inp, dt)
    assert plan["path"] == "seq" and planb["path"] == "seq" and planb["kernels"] == 2


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_gated_unaligned_rows_take_plain(dt):
    inp = make_gated_inputs(2, 90, 37, dt, seed=710)
    plan, planb = check_gated(inp, dt)
    assert plan["path"] == "plain" and planb["path"] == "plain"


def test_gated_empty_sequence():
    b = torch.empty((2, 0, 16), device="cuda")
    eta = torch.empty((2, 0), device="cuda")
    nu = torch.zeros(16, device="cuda")
    _, last = L.lrscan_fwd_gated(eta, nu, b)
    assert not last.any()
    _, geta, gnu = L.lrscan_bwd_gated(eta, nu, b, b)
    assert not gnu.any() and geta.numel() == 0


def test_gated_full_size():
    """The generated-decay workload at full size in the benchmark's launch
    configuration, every element: out and last of the forward; the backward
    runs on the oracle's forward output (so both sides read the same
    h_{t-1}): grad_b on every element, grad_eta on every token and
    grad_nu_log on every lane.  The decays come from a fast exponential, so
    this path agrees with the oracle to rounding (near-cancellation points
    allowed under the fp32 rule, and counted)."""
    w = GATED_WORKLOAD
    # the automatic plan on this shape: one warp per 16-lane slice, both directions
    for direction in ("fwd", "bwd"):
        assert L.lrscan_plan_gated(w.B, w.T, w.D, w.dtype, direction)["name"] == "gwarp_bf16_l16_r15"
    inp = make_gated_inputs()
    etad, nud = inp["eta"].cuda(), inp["nu_log"].cuda()
    out, last = L.lrscan_fwd_gated(etad, nud, inp["b"].cuda())
    assert L.lrscan_sync_check() == 0
    o = oracle.default()
    eta, nu = inp["eta"].numpy(), inp["nu_log"].numpy()
    ref_out, ref_last = o.gated_fwd(eta, nu, to_np(inp["b"]), w.dtype)
    out_n = to_np(out)
    del out
    print(f"[fullsize] gated out: beyond 2 bf16 ulps {bf16_beyond_ulps(out_n, ref_out)}", flush=True)
    assert_close(out_n, ref_out, w.dtype, "gated out, full size", reassociated=True)
    assert_last_close(last.cpu().numpy(), ref_last, "gated last, full size")
    g = to_np(inp["grad_out"])
    ref_gb, ref_geta, ref_gnu = o.gated_bwd(eta, nu, ref_out, g, w.dtype)
    gb, geta, gnu = L.lrscan_bwd_gated(etad, nud, from_np(ref_out, w.dtype).cuda(), inp["grad_out"].cuda())
    assert L.lrscan_sync_check() == 0
    gb_n = to_np(gb)
    print(f"[fullsize] gated grad_b: beyond 2 bf16 ulps {bf16_beyond_ulps(gb_n, ref_gb)}", flush=True)
    assert_close(gb_n, ref_gb, w.dtype, "gated grad_b, full size", reassociated=True)
    s_eta, s_nu = abs_terms(eta, nu, ref_out, g, w.dtype)
    assert_sum_close(geta.cpu().numpy(), ref_geta, s_eta, "gated grad_eta, full size")
    assert_sum_close(gnu.cpu().numpy(), ref_gnu, s_nu, "gated grad_nu_log, full size")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_gated_scan_autograd(dt):
    inp = make_gated_inputs(2, 150, 64, dt, seed=730)
    eta = inp["eta"].cuda().requires_grad_()
    nu = inp["nu_log"].cuda().requires_grad_()
    b = inp["b"].cuda().requires_grad_()
    out = L.gated_scan(eta, nu, b)
    (out.float() * inp["grad_out"].cuda().float()).sum().backward()
    o = oracle.default()
    ref_out, _ = o.gated_fwd(inp["eta"].numpy(), inp["nu_log"].numpy(), to_np(inp["b"]), dt)
    ref_gb, ref_geta, ref_gnu = o.gated_bwd(inp["eta"].numpy(), inp["nu_log"].numpy(), ref_out,
                                            to_np(inp["grad_out"]), dt)
    assert_close(to_np(b.grad), ref_gb, dt, "autograd grad_b", reassociated=True)
    s_eta, s_nu = abs_terms(inp["eta"].numpy(), inp["nu_log"].numpy(), ref_out, to_np(inp["grad_out"]), dt)
    assert_sum_close(eta.grad.cpu().numpy(), ref_geta, s_eta, "autograd grad_eta")
    assert_sum_close(nu.grad.cpu().numpy(), ref_gnu, s_nu, "autograd grad_nu_log")
