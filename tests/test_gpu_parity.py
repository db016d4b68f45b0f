"""GPU parity: every path of the CUDA library against the CPU oracle on the
same seeded inputs, element by element (tolerances in parity_util).

Small cases span several lane tiles, windows and chunks with ragged tails on
both axes, on every path and tile variant.  The named workloads at full size
(every element) are in test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS, make_inputs, random_inputs
from parity_util import assert_close, assert_last_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()  # loud failure if the library is missing
    yield
    assert L.lrscan_sync_check() == 0


ORC = None


def orc():
    global ORC
    if ORC is None:
        ORC = oracle.default()
    return ORC


def _dt(t):
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def exact_plan(plan) -> bool:
    """Paths whose every result is the sequential definition's own (the
    sequential and plain kernels, and the exact-walk windowed tiles)."""
    return bool(plan["exact"])


def gpu_fwd(a, b, **kw):
    ad, bd = a.cuda(), b.cuda()
    out, last = L.lrscan_fwd(ad, bd, **kw)
    assert L.lrscan_sync_check() == 0
    return to_np(out), last.cpu().numpy()


def gpu_bwd(a, out, g, **kw):
    ga, gb = L.lrscan_bwd(a.cuda(), out.cuda(), g.cuda(), **kw)
    assert L.lrscan_sync_check() == 0
    return to_np(ga), to_np(gb)


def from_np(x, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))


def check_case(inp, path=None, **kw):
    """Forward and backward of one case on one path, against the oracle."""
    a, b, g = inp["a"], inp["b"], inp["grad_out"]
    dt = _dt(a)
    B, T, D = a.shape
    o = orc()
    ref_out, ref_last = o.fwd(to_np(a), to_np(b), dt)
    plan = L.lrscan_plan(B, T, D, dt, "fwd", path=path, **kw)
    ex = exact_plan(plan)
    out, last = gpu_fwd(a, b, path=path, **kw)
    assert_close(out, ref_out, dt, f"out[{plan['name']}]", exact=ex, reassociated=not ex)
    assert_last_close(last, ref_last, f"last[{plan['name']}]", exact=ex)
    # the final state is the value stored at T-1 (before its storage rounding)
    if dt == "f32":
        assert np.array_equal(last, out[:, -1, :])
    # backward from the oracle's forward output (no expected value comes from the GPU)
    out_t = from_np(ref_out, dt)
    ref_ga, ref_gb = o.bwd(to_np(a), ref_out, to_np(g), dt)
    planb = L.lrscan_plan(B, T, D, dt, "bwd", path=path, **kw)
    exb = exact_plan(planb)
    ga, gb = gpu_bwd(a, out_t, g, path=path, **kw)
    assert_close(gb, ref_gb, dt, f"grad_b[{planb['name']}]", exact=exb, reassociated=not exb)
    assert_close(ga, ref_ga, dt, f"grad_a[{planb['name']}]", exact=exb, reassociated=not exb)
    return plan, planb


SMALL_SHAPES = {
    "f32": [(3, 300, 200), (2, 77, 36), (1, 1, 4), (1, 2, 8), (2, 513, 1000), (5, 129, 16)],
    "bf16": [(3, 300, 200), (2, 77, 40), (1, 1, 8), (2, 257, 1000), (4, 33, 24)],
}


def _variants(path, dt):
    return list(range(1, L.lrscan_num_variants(path, dt) + 1))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape_i", range(6))
@pytest.mark.parametrize("path", ["seq", "window"])
def test_tiled_paths_every_variant(dt, shape_i, path):
    shapes = SMALL_SHAPES[dt]
    if shape_i >= len(shapes):
        pytest.skip("no such shape")
    B, T, D = shapes[shape_i]
    inp = random_inputs(B, T, D, dt, seed=100 + shape_i, a_lo=0.6, a_hi=1.0)
    for v in _variants(path, dt):
        check_case(inp, path=path, tile_variant=v)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 32, 64, 128, 256, 512])
def test_chunked_path(dt, chunk):
    for i, (B, T, D) in enumerate(SMALL_SHAPES[dt]):
        inp = random_inputs(B, T, D, dt, seed=200 + i, a_lo=0.6, a_hi=1.0)
        check_case(inp, path="chunk", chunk_len=chunk)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_plain_path_and_unaligned_rows(dt):
    for i, (B, T, D) in enumerate(SMALL_SHAPES[dt] + [(2, 50, 3), (3, 70, 1), (2, 90, 13)]):
        inp = random_inputs(B, T, D, dt, seed=300 + i)
        check_case(inp, path="plain")
    # D whose rows are not 16-byte multiples: auto must take the plain path (exact)
    for (B, T, D) in [(2, 50, 3), (3, 70, 1), (2, 90, 13), (2, 1200, 6)]:
        inp = random_inputs(B, T, D, dt, seed=400 + D)
        plan, _ = check_case(inp)
        assert plan["path"] in ("plain", "chunk")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_unaligned_base_pointers(dt):
    """Tensors starting 1 element into an allocation: no bulk copies possible."""
    B, T, D = 2, 130, 64
    inp = random_inputs(B, T, D, dt, seed=7)
    o = orc()
    ref_out, ref_last = o.fwd(to_np(inp["a"]), to_np(inp["b"]), dt)
    n = B * T * D
    tdt = inp["a"].dtype
    bufs = [torch.zeros(n + 1, dtype=tdt, device="cuda") for _ in range(3)]
    a = bufs[0][1:].view(B, T, D)
    b = bufs[1][1:].view(B, T, D)
    out = bufs[2][1:].view(B, T, D)
    a.copy_(inp["a"].cuda())
    b.copy_(inp["b"].cuda())
    assert L.lrscan_plan(B, T, D, dt, "fwd", aligned=False)["path"] in ("plain", "chunk")
    _, last = L.lrscan_fwd(a, b, out)
    assert L.lrscan_sync_check() == 0
    assert_close(to_np(out), ref_out, dt, "out unaligned", exact=True)
    assert_last_close(last.cpu().numpy(), ref_last, exact=True)
    for path in ("chunk",):
        out.zero_()
        L.lrscan_fwd(a, b, out, path=path)
        assert L.lrscan_sync_check() == 0
        assert_close(to_np(out), ref_out, dt, f"out unaligned {path}", reassociated=True)


@pytest.mark.parametrize("path", [None, "seq", "window", "chunk", "plain"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_zero_decay_copies_b_bit_exactly(path, dt):
    inp = random_inputs(2, 200, 64, dt, seed=11)
    a = torch.zeros_like(inp["a"])
    out, last = gpu_fwd(a, inp["b"], path=path)
    assert np.array_equal(out, to_np(inp["b"]))


@pytest.mark.parametrize("path", [None, "seq", "window", "chunk", "plain"])
def test_unit_decay_integer_prefix_sums_exact(path):
    gen = torch.Generator().manual_seed(5)
    b = torch.randint(-8, 9, (2, 333, 48), generator=gen).float()
    a = torch.ones_like(b)
    out, last = gpu_fwd(a, b, path=path)
    assert np.array_equal(out, np.cumsum(b.numpy().astype(np.float64), axis=1).astype(np.float32))
    g = torch.randint(-8, 9, b.shape, generator=gen).float()
    ga, gb = gpu_bwd(a, torch.from_numpy(out), g, path=path)
    suffix = np.flip(np.cumsum(np.flip(g.numpy().astype(np.float64), 1), 1), 1)
    assert np.array_equal(gb, suffix.astype(np.float32))


def test_config1_all_paths():
    inp = make_inputs(1)
    check_case(inp)
    for path in ("seq", "window", "plain"):
        check_case(inp, path=path)
    for chunk in (16, 32, 64):
        check_case(inp, path="chunk", chunk_len=chunk)


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_named_workloads_reduced_size_all_paths(cid):
    """Each workload's value distributions at a size the oracle finishes fast."""
    w = WORKLOADS[cid]
    inp = make_inputs(cid, B=min(w.B, 3), T=min(w.T, 1000), D=min(w.D, 320))
    check_case(inp)
    for path in ("seq", "window", "plain"):
        check_case(inp, path=path)
    check_case(inp, path="chunk", chunk_len=w.chunk or 64)


def _check_padding(lengths, out, last, ga, gb, exact_carry):
    B = out.shape[0]
    for bb in range(B):
        n = int(lengths[bb])
        # padded gradients are exactly zero on every path
        assert not np.any(ga[bb, n:]) and not np.any(gb[bb, n:])
        # the stored last step is the final state on every path
        assert np.array_equal(last[bb], out[bb, -1])
        if exact_carry:
            assert np.array_equal(last[bb], out[bb, n - 1]), bb
            assert (out[bb, n:] == out[bb, n - 1][None, :]).all(), bb
        else:
            # identity steps change nothing; only one re-association point
            # (the next chunk boundary) may separate out[n-1] from the tail
            for d in range(out.shape[2]):
                assert len(np.unique(out[bb, n - 1:, d])) <= 2


@pytest.mark.parametrize("path", [None, "seq", "window", "chunk", "plain"])
def test_padding_identity_steps(path):
    inp = make_inputs(5, B=16, T=512, D=256)
    lengths = inp["lengths"].numpy()
    out, last = gpu_fwd(inp["a"], inp["b"], path=path)
    ga, gb = gpu_bwd(inp["a"], torch.from_numpy(out), inp["grad_out"], path=path)
    plan = L.lrscan_plan(16, 512, 256, "f32", "fwd", path=path)
    _check_padding(lengths, out, last, ga, gb, exact_carry=exact_plan(plan))


def test_empty_and_degenerate_shapes():
    # T == 0: last = h_{-1} = 0; nothing else touched
    for dt, tdt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        a = torch.empty(3, 0, 16, dtype=tdt, device="cuda")
        last = torch.full((3, 16), 7.0, device="cuda")
        L.lrscan_fwd(a, a, torch.empty_like(a), last)
        assert L.lrscan_sync_check() == 0
        assert not last.any()
        L.lrscan_bwd(a, a, a)
        z = torch.empty(0, 5, 16, dtype=tdt, device="cuda")
        L.lrscan_fwd(z, z)
        z = torch.empty(2, 5, 0, dtype=tdt, device="cuda")
        L.lrscan_fwd(z, z)
    assert L.lrscan_sync_check() == 0


@pytest.mark.parametrize("path", ["seq", "window", "chunk", "plain"])
def test_no_writes_outside_outputs(path):
    """Outputs placed between sentinel regions: ragged tails must not spill."""
    B, T, D = 3, 301, 40
    inp = random_inputs(B, T, D, "f32", seed=21)
    n = B * T * D
    pad = 4096
    sentinel = 12345.0
    buf = torch.full((3 * (n + 2 * pad),), sentinel, device="cuda")
    views = [buf[i * (n + 2 * pad) + pad: i * (n + 2 * pad) + pad + n].view(B, T, D) for i in range(3)]
    lastbuf = torch.full((B * D + 2 * pad,), sentinel, device="cuda")
    last = lastbuf[pad:pad + B * D].view(B, D)
    a, b, g = inp["a"].cuda(), inp["b"].cuda(), inp["grad_out"].cuda()
    L.lrscan_fwd(a, b, views[0], last, path=path)
    L.lrscan_bwd(a, views[0], g, views[1], views[2], path=path)
    assert L.lrscan_sync_check() == 0
    for i in range(3):
        base = i * (n + 2 * pad)
        assert (buf[base:base + pad] == sentinel).all()
        assert (buf[base + pad + n: base + 2 * pad + n] == sentinel).all()
    assert (lastbuf[:pad] == sentinel).all() and (lastbuf[pad + B * D:] == sentinel).all()


def test_non_default_stream_and_caller_workspace():
    inp = random_inputs(2, 3000, 64, "f32", seed=31)
    o = orc()
    ref_out, _ = o.fwd(to_np(inp["a"]), to_np(inp["b"]), "f32")
    s = torch.cuda.Stream()
    a, b = inp["a"].cuda(), inp["b"].cuda()
    need = L.lrscan_workspace_bytes(2, 3000, 64, 64)
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out, _ = L.lrscan_fwd(a, b, path="chunk", workspace=ws, stream=s)
    s.synchronize()
    assert L.lrscan_sync_check(stream=s) == 0
    assert_close(to_np(out), ref_out, "f32", "out caller workspace")
    small = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(L.LrscanError) as e:
        L.lrscan_fwd(a, b, path="chunk", workspace=small)
    assert e.value.code == L.LRSCAN_ENOMEM


def test_bounded_wait_gives_up_and_reports():
    """A wait that nothing will complete must expire, report, and leave the
    context usable (no trap, no hang)."""
    assert L.lrscan_sync_check() == 0
    rc = L.lrscan_selftest_wait_timeout(20_000_000)  # 20 ms
    assert rc == L.LRSCAN_ETIMEOUT
    assert L.lrscan_sync_check() == 0  # cleared by the read
    inp = random_inputs(1, 100, 32, "f32", seed=3)
    check_case(inp)


def test_autograd_wrapper_matches_direct_calls():
    inp = random_inputs(2, 400, 96, "f32", seed=41)
    a = inp["a"].cuda().requires_grad_(True)
    b = inp["b"].cuda().requires_grad_(True)
    g = inp["grad_out"].cuda()
    out = L.scan(a, b)
    out.backward(g)
    out2, _ = L.lrscan_fwd(a.detach(), b.detach())
    ga, gb = L.lrscan_bwd(a.detach(), out2, g)
    assert torch.equal(out, out2)
    assert torch.equal(a.grad, ga) and torch.equal(b.grad, gb)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape,chunk", [((2, 40000, 8), 16), ((1, 70001, 16), 32), ((1, 300001, 8), 512)])
def test_chunk_grouped_prefix(dt, shape, chunk):
    """The grouped chunk prefix (group maps, their prefix, per-group rescan;
    several groups and a ragged last group) against the oracle, forced and
    as the automatic choice, next to the flat prefix."""
    B, T, D = shape
    inp = random_inputs(B, T, D, dt, seed=600 + T, a_lo=0.9, a_hi=1.0)
    plan, planb = check_case(inp, path="chunk", chunk_len=chunk, tile_variant=2)
    assert plan["name"].endswith("_grouped") and plan["kernels"] == 5
    check_case(inp, path="chunk", chunk_len=chunk, tile_variant=1)
    auto = L.lrscan_plan(B, T, D, dt, "fwd", path="chunk", chunk_len=chunk)
    # automatic from 2,048 chunks per lane (586 chunks of 512 stay flat)
    assert auto["name"].endswith("_grouped") == (-(-T // chunk) >= 2048)
