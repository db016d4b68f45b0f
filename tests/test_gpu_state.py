"""GPU parity of the state-carrying scan (initial state h0, segment resets,
gradient at the final state, gradient of the initial state) on every path and
tile variant, against the oracle's state-carrying functions.

Sequential paths are compared exactly; window and chunk paths re-associate the
recurrence and are held to the tolerances of parity_util.  A reset step's
grad_a must be +0 exactly (its decay is unused).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import random_inputs
from parity_util import assert_close, assert_last_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    yield
    assert L.lrscan_sync_check() == 0


def _dt(t):
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def from_np(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))


def segments(seed, B, T, p=0.05):
    """int32 [B, T] positions; zeros mark segment starts (row 0 starts at t=0,
    row 1 continues the initial state)."""
    r = np.random.default_rng(seed)
    starts = r.random((B, T)) < p
    starts[0, 0] = True
    if B > 1:
        starts[1, 0] = False
    seg = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        pos = 0
        for t in range(T):
            pos = 0 if starts[b, t] else pos + 1
            seg[b, t] = pos
    return seg


def state_inputs(B, T, D, dt, seed):
    inp = random_inputs(B, T, D, dt, seed=seed, a_lo=0.6, a_hi=1.0)
    r = np.random.default_rng(seed + 7)
    inp["h0"] = r.standard_normal((B, D)).astype(np.float32)
    inp["grad_last"] = r.standard_normal((B, D)).astype(np.float32)
    inp["seg"] = segments(seed + 9, B, T)
    return inp


def exact_plan(plan) -> bool:
    return bool(plan["exact"])


def check_state_case(inp, path=None, use=("h0", "seg", "grad_last"), want_grad_h0=True, **kw):
    a, b, g = inp["a"], inp["b"], inp["grad_out"]
    dt = _dt(a)
    B, T, D = a.shape
    h0 = inp["h0"] if "h0" in use else None
    seg = inp["seg"] if "seg" in use else None
    gl = inp["grad_last"] if "grad_last" in use else None
    o = oracle.default()
    ref_out, ref_last = o.fwd_state(to_np(a), to_np(b), dt, h0=h0, segment_pos=seg)
    plan = L.lrscan_plan(B, T, D, dt, "fwd", path=path, **kw)
    ex = exact_plan(plan)
    cu = lambda x: None if x is None else torch.from_numpy(x).cuda()  # noqa: E731
    out, last = L.lrscan_fwd_state(a.cuda(), b.cuda(), h0=cu(h0), segment_pos=cu(seg), path=path, **kw)
    assert L.lrscan_sync_check() == 0
    tag = f"{plan['name']} {'+'.join(use)}"
    assert_close(to_np(out), ref_out, dt, f"out[{tag}]", exact=ex, reassociated=not ex)
    assert_last_close(last.cpu().numpy(), ref_last, f"last[{tag}]", exact=ex)

    ref_ga, ref_gb, ref_gh0 = o.bwd_state(to_np(a), ref_out, to_np(g), dt, h0=h0, segment_pos=seg,
                                          grad_last=gl)
    planb = L.lrscan_plan(B, T, D, dt, "bwd", path=path, **kw)
    exb = exact_plan(planb)
    gh0 = torch.full((B, D), float("nan"), device="cuda") if want_grad_h0 else None
    ga, gb, gh0_out = L.lrscan_bwd_state(a.cuda(), from_np(ref_out, dt).cuda(), g.cuda(), h0=cu(h0),
                                         segment_pos=cu(seg), grad_last=cu(gl), grad_h0=gh0,
                                         want_grad_h0=want_grad_h0, path=path, **kw)
    assert L.lrscan_sync_check() == 0
    tagb = f"{planb['name']} {'+'.join(use)}"
    ga, gb = to_np(ga), to_np(gb)
    assert_close(gb, ref_gb, dt, f"grad_b[{tagb}]", exact=exb, reassociated=not exb)
    assert_close(ga, ref_ga, dt, f"grad_a[{tagb}]", exact=exb, reassociated=not exb)
    if seg is not None:
        zero = np.uint16(0) if dt == "bf16" else np.float32(0)
        at_reset = ga[seg == 0]
        assert (at_reset.view(np.uint16 if dt == "bf16" else np.uint32) == zero.view(
            np.uint16 if dt == "bf16" else np.uint32)).all(), f"grad_a at resets must be +0 [{tagb}]"
    if want_grad_h0:
        assert_last_close(gh0_out.cpu().numpy(), ref_gh0, f"grad_h0[{tagb}]", exact=exb)
    return plan, planb


SHAPES = {
    "f32": [(3, 300, 200), (2, 77, 36), (1, 1, 4), (2, 513, 1000)],
    "bf16": [(3, 300, 200), (2, 77, 40), (1, 1, 8), (2, 257, 1000)],
}


def _variants(path, dt):
    return list(range(1, L.lrscan_num_variants(path, dt) + 1))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape_i", range(4))
@pytest.mark.parametrize("path", ["seq", "window"])
def test_state_every_tile_variant(dt, shape_i, path):
    B, T, D = SHAPES[dt][shape_i]
    inp = state_inputs(B, T, D, dt, seed=300 + shape_i)
    for v in _variants(path, dt):
        check_state_case(inp, path=path, tile_variant=v)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["chunk", "plain", "auto"])
def test_state_other_paths(dt, path):
    for i, (B, T, D) in enumerate(SHAPES[dt]):
        inp = state_inputs(B, T, D, dt, seed=320 + i)
        if path == "chunk":
            for c in (16, 64):
                check_state_case(inp, path=path, chunk_len=c)
        else:
            check_state_case(inp, path=path)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("use", [("h0",), ("seg",), ("grad_last",), ("h0", "grad_last")])
@pytest.mark.parametrize("path", ["seq", "window", "chunk"])
def test_state_members_one_at_a_time(dt, use, path):
    inp = state_inputs(3, 300, 200, dt, seed=340)
    check_state_case(inp, path=path, use=use)
    check_state_case(inp, path=path, use=use, want_grad_h0=False)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_state_unaligned_rows_take_plain_kernels(dt):
    B, T, D = 2, 90, 37
    inp = state_inputs(B, T, D, dt, seed=350)
    plan, planb = check_state_case(inp)
    assert plan["path"] in ("plain", "chunk") and planb["path"] in ("plain", "chunk")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["seq", "window", "chunk", "plain"])
def test_prefill_then_continue_matches_one_call(dt, path):
    """Scanning a prefix and then the rest from its final state gives the
    one-call result (bit for bit on the sequential paths)."""
    B, T, D = 2, 300, 200
    inp = random_inputs(B, T, D, dt, seed=360, a_lo=0.6, a_hi=1.0)
    a, b = inp["a"].cuda(), inp["b"].cuda()
    out, last = L.lrscan_fwd_state(a, b, path=path)
    for T1 in (1, 129, 299):
        o1, l1 = L.lrscan_fwd_state(a[:, :T1].contiguous(), b[:, :T1].contiguous(), path=path)
        o2, l2 = L.lrscan_fwd_state(a[:, T1:].contiguous(), b[:, T1:].contiguous(), h0=l1, path=path)
        got = torch.cat([o1, o2], dim=1)
        if path in ("seq", "plain"):
            assert torch.equal(got, out) and torch.equal(l2, last), T1
        else:
            ref = oracle.default().fwd(to_np(inp["a"]), to_np(inp["b"]), _dt(inp["a"]))[0]
            assert_close(to_np(got), ref, _dt(inp["a"]), f"continued[{path}]", reassociated=True)
    assert L.lrscan_sync_check() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_state_empty_sequence(dt):
    B, D = 3, 64
    a = torch.empty((B, 0, D), dtype=torch.float32 if dt == "f32" else torch.bfloat16, device="cuda")
    h0 = torch.randn(B, D, device="cuda")
    gl = torch.randn(B, D, device="cuda")
    _, last = L.lrscan_fwd_state(a, a, h0=h0)
    assert torch.equal(last, h0)
    _, last = L.lrscan_fwd_state(a, a)
    assert not last.any()
    _, _, gh0 = L.lrscan_bwd_state(a, a, a, h0=h0, grad_last=gl)
    assert torch.equal(gh0, gl)
    _, _, gh0 = L.lrscan_bwd_state(a, a, a)
    assert not gh0.any()
    assert L.lrscan_sync_check() == 0


def test_state_absent_equals_plain_entry_points():
    """lrscan_*_state with no state is the plain scan, bit for bit."""
    inp = random_inputs(3, 300, 200, "bf16", seed=370, a_lo=0.6, a_hi=1.0)
    a, b, g = inp["a"].cuda(), inp["b"].cuda(), inp["grad_out"].cuda()
    o1, l1 = L.lrscan_fwd(a, b)
    o2, l2 = L.lrscan_fwd_state(a, b)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ga1, gb1 = L.lrscan_bwd(a, o1, g)
    ga2, gb2, _ = L.lrscan_bwd_state(a, o1, g)
    assert torch.equal(ga1, ga2) and torch.equal(gb1, gb2)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_scan_state_autograd(dt):
    B, T, D = 2, 150, 64
    inp = state_inputs(B, T, D, dt, seed=380)
    a = inp["a"].cuda().requires_grad_()
    b = inp["b"].cuda().requires_grad_()
    h0 = torch.from_numpy(inp["h0"]).cuda().requires_grad_()
    seg = torch.from_numpy(inp["seg"]).cuda()
    out, last = L.scan_state(a, b, h0=h0, segment_pos=seg)
    g = inp["grad_out"].cuda()
    gl = torch.from_numpy(inp["grad_last"]).cuda()
    ((out.float() * g.float()).sum() + (last * gl).sum()).backward()
    o = oracle.default()
    ref_out, _ = o.fwd_state(to_np(inp["a"]), to_np(inp["b"]), dt, h0=inp["h0"], segment_pos=inp["seg"])
    ref_ga, ref_gb, ref_gh0 = o.bwd_state(to_np(inp["a"]), ref_out, to_np(inp["grad_out"]), dt,
                                          h0=inp["h0"], segment_pos=inp["seg"], grad_last=inp["grad_last"])
    assert_close(to_np(a.grad), ref_ga, dt, "autograd grad_a", reassociated=True)
    assert_close(to_np(b.grad), ref_gb, dt, "autograd grad_b", reassociated=True)
    assert_last_close(h0.grad.cpu().numpy(), ref_gh0, "autograd grad_h0")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_state_on_the_grouped_chunk_prefix(dt):
    """h0 and grad_last enter through the grouped prefix's group-level scan."""
    inp = state_inputs(2, 40000, 8, dt, seed=390)
    plan, planb = check_state_case(inp, path="chunk", chunk_len=16, tile_variant=2)
    assert plan["kernels"] == 5 and planb["kernels"] == 5
