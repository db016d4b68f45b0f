"""GPU parity of the persistent chunk-streaming path (path "stream") against
the CPU oracle: forward and backward, both storage dtypes, every variant, on
shapes with ragged lane tiles, partial chunks, one-step sequences, and more
chunks than CTAs (so every CTA takes several tickets and looks back over
chunks published by others)."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import random_inputs
from parity_util import assert_close, assert_last_close, bf16_bits_to_f32, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    yield
    assert L.lrscan_sync_check() == 0


ORC = None


def orc():
    global ORC
    if ORC is None:
        ORC = oracle.default()
    return ORC


def from_np(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))


SHAPES = [(1, 1, 32), (1, 255, 32), (1, 256, 64), (1, 257, 64), (3, 700, 32), (2, 3001, 96), (1, 5000, 64),
          (2, 40000, 32), (1, 9, 8)]


def check(B, T, D, dt, variant, seed, a_lo=0.6):
    inp = random_inputs(B, T, D, dt, seed=seed, a_lo=a_lo, a_hi=1.0)
    a, b, g = inp["a"], inp["b"], inp["grad_out"]
    o = orc()
    ref_out, ref_last = o.fwd(to_np(a), to_np(b), dt)
    kw = dict(path="stream", tile_variant=variant)
    plan = L.lrscan_plan(B, T, D, dt, "fwd", **kw)
    assert plan["path"] == "stream" and not plan["exact"]
    out, last = L.lrscan_fwd(a.cuda(), b.cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    name = f"{plan['name']} B={B} T={T} D={D}"
    assert_close(to_np(out), ref_out, dt, f"out[{name}]", reassociated=True)
    assert_last_close(last.cpu().numpy(), ref_last, f"last[{name}]")
    if dt == "f32":
        assert np.array_equal(last.cpu().numpy(), to_np(out)[:, -1, :])
    ref_ga, ref_gb = o.bwd(to_np(a), ref_out, to_np(g), dt)
    ga, gb = L.lrscan_bwd(a.cuda(), from_np(ref_out, dt).cuda(), g.cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    assert_close(to_np(gb), ref_gb, dt, f"grad_b[{name}]", reassociated=True)
    assert_close(to_np(ga), ref_ga, dt, f"grad_a[{name}]", reassociated=True)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("shape_i", range(len(SHAPES)))
def test_stream_parity(dt, variant, shape_i):
    if variant > L.lrscan_num_variants("stream", dt):
        pytest.skip("no such variant for this dtype")
    B, T, D = SHAPES[shape_i]
    check(B, T, D, dt, variant, seed=900 + shape_i)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_stream_many_chunks_per_cta(dt):
    """More chunk tickets than CTAs (two 32-lane groups x 512 chunks of 512
    steps; bf16 forward: chunks of 1024): several per CTA."""
    B, T, D = 1, 1 << 18, 64
    plan = L.lrscan_plan(B, T, D, dt, "fwd", path="stream", tile_variant=1)
    chunk = plan["rows_per_window"] * plan["subchunks"]
    assert plan["ctas"] < 2 * (T // chunk)
    check(B, T, D, dt, 1, seed=950, a_lo=0.9)


STATE_SHAPES = [(1, 1, 32), (2, 3001, 96), (3, 700, 32), (1, 40000, 32), (1, 9, 8)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape_i", range(len(STATE_SHAPES)))
def test_stream_carried_state(dt, shape_i):
    """h0, segment resets (about one token in twenty starts a segment; batch
    row 0 starts one at t=0, row 1 continues h0), grad_last and grad_h0 on
    every stream variant, forward and backward against the oracle's state
    functions; grad_a is +0 at every reset."""
    from test_gpu_state import check_state_case, state_inputs
    B, T, D = STATE_SHAPES[shape_i]
    inp = state_inputs(B, T, D, dt, seed=960 + shape_i)
    for v in range(1, L.lrscan_num_variants("stream", dt) + 1):
        plan, planb = check_state_case(inp, path="stream", tile_variant=v)
        assert plan["path"] == "stream" and planb["path"] == "stream"


@pytest.mark.parametrize("use", [("h0",), ("seg",), ("grad_last",)])
def test_stream_state_members_one_at_a_time(use):
    from test_gpu_state import check_state_case, state_inputs
    inp = state_inputs(2, 5000, 64, "f32", seed=975)
    check_state_case(inp, path="stream", use=use)
    check_state_case(inp, path="stream", use=use, want_grad_h0=False)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_stream_carried_state(dt):
    """The complex chunk-streaming kernels with complex h0, segment resets
    (the forward's masks from the ticket warp, the backward's from per-tile
    loads), grad_last and grad_h0 = conj(a'_0) g_0, against the oracle's
    complex state functions: ragged lane tiles, partial chunks, one-step and
    many-chunk sequences, a reset at step 0; then each state member alone."""
    from test_gpu_complex import _cstate_inputs, check_cstate
    for i, (B, T, D) in enumerate([(1, 5000, 64), (2, 3001, 96), (1, 9, 8), (2, 40000, 32), (1, 700, 32)]):
        inp, h0, gl, seg = _cstate_inputs(B, T, D, dt, seed=990 + i)
        if i % 2:
            seg[:, 0] = 0  # a reset at step 0
        plan, planb = check_cstate(inp, dt, h0, gl, seg, path="stream")
        assert plan["path"] == "stream" and planb["path"] == "stream" and plan["name"].startswith("cstream_")
    # the automatic plan streams few lanes and long sequences with state too
    inp, h0, gl, seg = _cstate_inputs(1, 40000, 64, dt, seed=999)
    plan, planb = check_cstate(inp, dt, h0, gl, seg)
    assert plan["path"] == "stream" and planb["path"] == "stream"
    # one member at a time: h0 and grad_last only (no resets), resets only
    B, T, D = 1, 3000, 32
    inp, h0, gl, seg = _cstate_inputs(B, T, D, dt, seed=998)
    check_cstate(inp, dt, h0, gl, np.ones((B, T), dtype=np.int32), path="stream")
    zero = [np.zeros((B, D), dtype=np.float32)] * 2
    check_cstate(inp, dt, zero, zero, seg, path="stream")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_stream_in_cuda_graph(dt):
    """Captured into a graph (the workspace's ticket is zeroed and its maps and
    states refilled by captured memsets each call), replayed twice with new
    inputs: each replay against the oracle.  The captured backward reads its own static input
    (filled with the oracle's forward output before each replay)."""
    B, T, D = 1, 20000, 64
    kw = dict(path="stream")
    o = orc()
    static = {k: v.cuda() for k, v in random_inputs(B, T, D, dt, seed=970, a_lo=0.8, a_hi=1.0).items()
              if k in ("a", "b", "grad_out")}
    static["out_in"] = torch.empty_like(static["a"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        L.lrscan_fwd(static["a"], static["b"], **kw)  # outside capture: sizes the workspace
        L.lrscan_bwd(static["a"], static["out_in"], static["grad_out"], **kw)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out, last = L.lrscan_fwd(static["a"], static["b"], **kw)
        ga, gb = L.lrscan_bwd(static["a"], static["out_in"], static["grad_out"], **kw)
    for seed in (971, 972):
        fresh = random_inputs(B, T, D, dt, seed=seed, a_lo=0.8, a_hi=1.0)
        a_np = to_np(fresh["a"])
        ref_out, ref_last = o.fwd(a_np, to_np(fresh["b"]), dt)
        ref_ga, ref_gb = o.bwd(a_np, ref_out, to_np(fresh["grad_out"]), dt)
        for k in ("a", "b", "grad_out"):
            static[k].copy_(fresh[k].cuda())
        static["out_in"].copy_(from_np(ref_out, dt).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert L.lrscan_sync_check() == 0
        assert_close(to_np(out), ref_out, dt, f"out replay {seed}", reassociated=True)
        assert_last_close(last.cpu().numpy(), ref_last, f"last replay {seed}")
        assert_close(to_np(gb), ref_gb, dt, f"grad_b replay {seed}", reassociated=True)
        assert_close(to_np(ga), ref_ga, dt, f"grad_a replay {seed}", reassociated=True)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_stream_nan_inputs(dt):
    """NaNs whose bits are all ones (the workspace's "nothing published" word)
    in b, a and grad_out: the call ends without a timeout, the NaNs spread as
    in the oracle (from their step on, along their lane), and every other
    output agrees with it."""
    B, T, D = 1, 20000, 64
    inp = random_inputs(B, T, D, dt, seed=990, a_lo=0.8, a_hi=1.0)
    a_np, b_np, g_np = (np.array(to_np(inp[k])) for k in ("a", "b", "grad_out"))
    ones = np.array([0xFFFFFFFF], dtype=np.uint32).view(np.float32)[0] if dt == "f32" else np.uint16(0xFFFF)
    b_np[0, 7000, 5] = ones
    a_np[0, 12000, 40] = ones
    g_np[0, 15000, 20] = ones
    o = orc()
    ref_out, ref_last = o.fwd(a_np, b_np, dt)
    ref_ga, ref_gb = o.bwd(a_np, ref_out, g_np, dt)
    kw = dict(path="stream")
    out, last = L.lrscan_fwd(from_np(a_np, dt).cuda(), from_np(b_np, dt).cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    ga, gb = L.lrscan_bwd(from_np(a_np, dt).cuda(), from_np(ref_out, dt).cuda(), from_np(g_np, dt).cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    as_f32 = (lambda x: bf16_bits_to_f32(x)) if dt == "bf16" else (lambda x: x)
    for name, got, ref in (("out", to_np(out), ref_out), ("grad_b", to_np(gb), ref_gb), ("grad_a", to_np(ga), ref_ga)):
        assert np.isnan(as_f32(ref)).any(), name
        assert_close(got, ref, dt, name, reassociated=True)  # NaN pattern equal, the rest within tolerance
    assert np.array_equal(np.isnan(last.cpu().numpy()), np.isnan(ref_last))
