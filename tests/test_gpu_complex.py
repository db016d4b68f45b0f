"""GPU parity of the complex diagonal scan (re/im planes) on every path and
tile variant, against the oracle's complex scan, and of the state-carrying
complex scan (h0, segment resets, grad_last, grad_h0) against the oracle's
complex state functions.  The sequential tiles and the plain kernels keep the
oracle's order of operations and are compared exactly; the windowed tiles and
the chunked path re-associate through complex affine maps and are held to the
tolerances of parity_util."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import COMPLEX_WORKLOAD, make_complex_inputs
from parity_util import assert_close, assert_last_close, bf16_beyond_ulps, to_np

pytestmark = pytest.mark.gpu

PLANES = ("ar", "ai", "br", "bi", "go_r", "go_i")


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


def check_complex(inp, dt, **kw):
    B, T, D = inp["shape"]
    np_in = {k: to_np(inp[k]) for k in PLANES}
    o = oracle.default()
    ref = o.cfwd(np_in["ar"], np_in["ai"], np_in["br"], np_in["bi"], dt)
    cu = {k: inp[k].cuda() for k in PLANES}
    got = L.lrscan_cfwd(cu["ar"], cu["ai"], cu["br"], cu["bi"], **kw)
    assert L.lrscan_sync_check() == 0
    plan = L.lrscan_plan_complex(B, T, D, dt, "fwd", **kw)
    tag = plan["name"]
    ex = bool(plan["exact"])  # windowed tiles and chunks re-associate through complex maps
    for name, g, r in zip(("out_r", "out_i"), got[:2], ref[:2]):
        assert_close(to_np(g), r, dt, f"{name}[{tag}]", exact=ex, reassociated=not ex)
    for name, g, r in zip(("last_r", "last_i"), got[2:], ref[2:]):
        assert_last_close(g.cpu().numpy(), r, f"{name}[{tag}]", exact=ex)
    # backward from the oracle's forward output
    out_r, out_i = from_np(ref[0], dt).cuda(), from_np(ref[1], dt).cuda()
    gref = o.cbwd(np_in["ar"], np_in["ai"], ref[0], ref[1], np_in["go_r"], np_in["go_i"], dt)
    ggot = L.lrscan_cbwd(cu["ar"], cu["ai"], out_r, out_i, cu["go_r"], cu["go_i"], **kw)
    assert L.lrscan_sync_check() == 0
    planb = L.lrscan_plan_complex(B, T, D, dt, "bwd", **kw)
    exb = bool(planb["exact"])
    for name, g, r in zip(("grad_ar", "grad_ai", "grad_br", "grad_bi"), ggot, gref):
        assert_close(to_np(g), r, dt, f"{name}[{planb['name']}]", exact=exb, reassociated=not exb)
    return plan, planb


SHAPES = [(3, 300, 200), (2, 77, 40), (1, 1, 8), (2, 257, 1000), (1, 33, 64)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_complex_every_variant(dt, shape):
    B, T, D = shape
    inp = make_complex_inputs(B, T, D, dt, seed=500 + T)
    n = 1
    while True:
        try:
            L.lrscan_plan_complex(B, T, D, dt, path="seq", tile_variant=n)
        except L.LrscanError:
            break
        check_complex(inp, dt, path="seq", tile_variant=n)
        n += 1
    assert n > 3
    check_complex(inp, dt, path="plain")
    plan, _ = check_complex(inp, dt)
    assert plan["path"] in ("seq", "window")


STREAM_SHAPES = [(1, 1, 32), (1, 255, 32), (1, 257, 64), (3, 700, 32), (2, 3001, 96), (1, 5000, 64),
                 (2, 40000, 32), (1, 9, 8)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", STREAM_SHAPES)
def test_complex_stream_path(dt, shape):
    """The persistent chunk-streaming kernel on the complex planes: ragged lane
    tiles, partial chunks, one-step sequences, several chunks per lane group,
    forward and backward against the oracle."""
    B, T, D = shape
    inp = make_complex_inputs(B, T, D, dt, seed=560 + T % 97)
    plan, planb = check_complex(inp, dt, path="stream")
    assert plan["path"] == "stream" and planb["path"] == "stream" and plan["name"].startswith("cstream_")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_stream_many_chunks_per_cta(dt):
    """More chunk tickets than CTAs (two lane groups x 512 forward chunks of
    512 steps), the automatic plan."""
    B, T, D = 1, 1 << 18, 64
    inp = make_complex_inputs(B, T, D, dt, seed=575)
    plan, planb = check_complex(inp, dt)
    assert plan["path"] == "stream" and planb["path"] == "stream" and plan["ctas"] < 2 * (T // 512)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_unaligned_takes_plain(dt):
    inp = make_complex_inputs(2, 90, 37, dt, seed=510)
    plan, planb = check_complex(inp, dt)
    assert plan["path"] == "plain" and planb["path"] == "plain"


def test_complex_empty_and_invalid():
    a = torch.empty((2, 0, 16), device="cuda")
    _, _, lr, li = L.lrscan_cfwd(a, a, a, a)
    assert not lr.any() and not li.any()
    x = torch.zeros((1, 4, 16), device="cuda")
    with pytest.raises(L.LrscanError):
        L.lrscan_cfwd(x, x, x, x, path="chunk", chunk_len=48)
    with pytest.raises(L.LrscanError):
        L.lrscan_cfwd(x, x, x, x, path="chunk", tile_variant=3)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 64, 512])
def test_complex_chunked_path(dt, chunk):
    """Complex chunk maps, their prefix and the replay on the small shapes
    (several chunks per lane, ragged tails, T shorter than a chunk)."""
    for i, (B, T, D) in enumerate(SHAPES):
        inp = make_complex_inputs(B, T, D, dt, seed=540 + i)
        plan, planb = check_complex(inp, dt, path="chunk", chunk_len=chunk)
        assert plan["path"] == "chunk" and planb["path"] == "chunk" and plan["name"].startswith(f"cchunk{chunk}_v")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_chunked_grouped_prefix_and_auto(dt):
    """Few lanes, long sequence (2,500 chunks of 16 per lane: five groups of
    512 maps, the last one ragged): the grouped prefix forced and as the
    automatic choice of the chunked path, the flat prefix forced, and the
    automatic plan (chunk streaming) against the oracle."""
    B, T, D = 1, 40000, 8
    inp = make_complex_inputs(B, T, D, dt, seed=550)
    plan, planb = check_complex(inp, dt, path="chunk", chunk_len=16, tile_variant=2)
    assert plan["name"].startswith("cchunk16_v") and plan["name"].endswith("_grouped") and planb["kernels"] == 5
    assert L.lrscan_plan_complex(B, T, D, dt, "fwd", path="chunk", chunk_len=16)["name"].endswith("_grouped")
    check_complex(inp, dt, path="chunk", chunk_len=16, tile_variant=1)
    plan, planb = check_complex(inp, dt)
    assert plan["path"] == "stream" and planb["path"] == "stream"


def test_complex_chunked_unaligned_rows():
    """The chunked kernels read one element per thread: any row alignment."""
    inp = make_complex_inputs(2, 3000, 37, "bf16", seed=560)
    plan, planb = check_complex(inp, "bf16", path="chunk", chunk_len=32)
    assert plan["path"] == "chunk"
    plan, _ = check_complex(inp, "bf16")
    assert plan["path"] == "chunk"  # few lanes, long enough: chunks also without alignment


def test_complex_full_size_every_element():
    """The complex workload at full size in the benchmark's launch
    configuration, every element of every plane against the oracle (the
    windowed tiles re-associate: near-cancellation points allowed under the
    fp32 rule, and counted); the backward reads the oracle's forward output,
    so both sides see the same h_{t-1}."""
    w = COMPLEX_WORKLOAD
    inp = make_complex_inputs()
    cu = {k: inp[k].cuda() for k in PLANES}
    got = L.lrscan_cfwd(cu["ar"], cu["ai"], cu["br"], cu["bi"])
    assert L.lrscan_sync_check() == 0
    o = oracle.default()
    ref = o.cfwd(*(to_np(inp[k]) for k in ("ar", "ai", "br", "bi")), w.dtype)
    ex = bool(L.lrscan_plan_complex(w.B, w.T, w.D, w.dtype, "fwd")["exact"])
    for name, g, r in zip(("out_r", "out_i"), got[:2], ref[:2]):
        gn = to_np(g)
        print(f"[fullsize] complex {name}: beyond 2 bf16 ulps {bf16_beyond_ulps(gn, r)}", flush=True)
        assert_close(gn, r, w.dtype, f"complex {name}, full size", exact=ex, reassociated=not ex)
    for name, g, r in zip(("last_r", "last_i"), got[2:], ref[2:]):
        assert_last_close(g.cpu().numpy(), r, f"complex {name}, full size", exact=ex)
    del got
    grads = L.lrscan_cbwd(cu["ar"], cu["ai"], from_np(ref[0], w.dtype).cuda(), from_np(ref[1], w.dtype).cuda(),
                          cu["go_r"], cu["go_i"])
    assert L.lrscan_sync_check() == 0
    gref = o.cbwd(*(to_np(inp[k]) for k in ("ar", "ai")), ref[0], ref[1],
                  *(to_np(inp[k]) for k in ("go_r", "go_i")), w.dtype)
    exb = bool(L.lrscan_plan_complex(w.B, w.T, w.D, w.dtype, "bwd")["exact"])
    for name, g, r in zip(("grad_ar", "grad_ai", "grad_br", "grad_bi"), grads, gref):
        gn = to_np(g)
        print(f"[fullsize] complex {name}: beyond 2 bf16 ulps {bf16_beyond_ulps(gn, r)}", flush=True)
        assert_close(gn, r, w.dtype, f"complex {name}, full size", exact=exb, reassociated=not exb)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_scan_autograd(dt):
    inp = make_complex_inputs(2, 150, 64, dt, seed=530)
    xs = [inp[k].cuda().requires_grad_() for k in ("ar", "ai", "br", "bi")]
    out_r, out_i = L.complex_scan(*xs)
    (out_r.float() * inp["go_r"].cuda().float() + out_i.float() * inp["go_i"].cuda().float()).sum().backward()
    o = oracle.default()
    np_in = {k: to_np(inp[k]) for k in PLANES}
    ref = o.cfwd(np_in["ar"], np_in["ai"], np_in["br"], np_in["bi"], dt)
    gref = o.cbwd(np_in["ar"], np_in["ai"], ref[0], ref[1], np_in["go_r"], np_in["go_i"], dt)
    for x, r in zip(xs, gref):
        assert_close(to_np(x.grad), r, dt, "complex autograd", reassociated=True)


# ------------------------------------------------ carried state and resets --
def _cstate_inputs(B, T, D, dt, seed):
    inp = make_complex_inputs(B, T, D, dt, seed=seed)
    r = np.random.default_rng(seed)
    h0 = [r.standard_normal((B, D)).astype(np.float32) for _ in range(2)]
    gl = [r.standard_normal((B, D)).astype(np.float32) for _ in range(2)]
    starts = r.random((B, T)) < 0.03
    seg = np.zeros((B, T), dtype=np.int32)
    for bb in range(B):
        pos = 0
        for t in range(T):
            pos = 0 if starts[bb, t] else (pos + 1 if t > 0 else 1)
            seg[bb, t] = pos
    return inp, h0, gl, seg


def check_cstate(inp, dt, h0, gl, seg, **kw):
    """Forward and backward with carried state against the oracle; the
    backward reads the oracle's forward output (both sides see the same
    h_{t-1})."""
    np_in = {k: to_np(inp[k]) for k in PLANES}
    o = oracle.default()
    ref = o.cfwd_state(np_in["ar"], np_in["ai"], np_in["br"], np_in["bi"], dt, h0=tuple(h0), segment_pos=seg)
    cu = {k: inp[k].cuda() for k in PLANES}
    th0 = tuple(torch.from_numpy(x).cuda() for x in h0)
    tgl = tuple(torch.from_numpy(x).cuda() for x in gl)
    tseg = torch.from_numpy(seg).cuda()
    got = L.lrscan_cfwd_state(cu["ar"], cu["ai"], cu["br"], cu["bi"], h0=th0, segment_pos=tseg, **kw)
    assert L.lrscan_sync_check() == 0
    B, T, D = inp["shape"]
    plan = L.lrscan_plan_complex(B, T, D, dt, "fwd", state=True, **kw)
    planb = L.lrscan_plan_complex(B, T, D, dt, "bwd", state=True, **kw)
    ex, exb = bool(plan["exact"]), bool(planb["exact"])
    for name, g, r in zip(("out_r", "out_i"), got[:2], ref[:2]):
        assert_close(to_np(g), r, dt, f"{name} (state) [{plan['name']}]", exact=ex, reassociated=not ex)
    for name, g, r in zip(("last_r", "last_i"), got[2:], ref[2:]):
        assert_last_close(g.cpu().numpy(), r, f"{name} (state) [{plan['name']}]", exact=ex)
    out_r, out_i = from_np(ref[0], dt).cuda(), from_np(ref[1], dt).cuda()
    gref = o.cbwd_state(np_in["ar"], np_in["ai"], ref[0], ref[1], np_in["go_r"], np_in["go_i"], dt, h0=tuple(h0),
                        segment_pos=seg, grad_last=tuple(gl))
    ggot = L.lrscan_cbwd_state(cu["ar"], cu["ai"], out_r, out_i, cu["go_r"], cu["go_i"], h0=th0, segment_pos=tseg,
                               grad_last=tgl, **kw)
    assert L.lrscan_sync_check() == 0
    for name, g, r in zip(("grad_ar", "grad_ai", "grad_br", "grad_bi"), ggot[:4], gref[:4]):
        assert_close(to_np(g), r, dt, f"{name} (state) [{planb['name']}]", exact=exb, reassociated=not exb)
    for name, g, r in zip(("grad_h0_r", "grad_h0_i"), ggot[4:], gref[4:]):
        assert_last_close(g.cpu().numpy(), r, f"{name} (state) [{planb['name']}]", exact=exb)
    # grad_a is exactly +0 at every segment start
    rs = np.broadcast_to((seg == 0)[..., None], ref[0].shape)
    for g in ggot[:2]:
        assert not to_np(g).view(np.uint16 if dt == "bf16" else np.uint32)[rs].any()
    return plan, planb


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [None, 16])
def test_complex_state_every_shape(dt, chunk):
    for i, (B, T, D) in enumerate(SHAPES):
        inp, h0, gl, seg = _cstate_inputs(B, T, D, dt, seed=570 + i)
        check_cstate(inp, dt, h0, gl, seg, path="chunk", chunk_len=chunk)
        check_cstate(inp, dt, h0, gl, seg)  # the automatic plan


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_state_every_tile_variant(dt):
    """Every tiled complex variant (sequential tiles bit for bit, windowed
    tiles to rounding) with h0, resets, grad_last and grad_h0, on shapes with
    ragged lane tiles and ragged last windows, against the oracle."""
    for i, (B, T, D) in enumerate([(3, 300, 200), (2, 77, 48), (1, 1, 16), (2, 1030, 96)]):
        inp, h0, gl, seg = _cstate_inputs(B, T, D, dt, seed=600 + i)
        if i % 2:
            seg[:, 0] = 0   # a reset at step 0
        n = 1
        while True:
            try:
                L.lrscan_plan_complex(B, T, D, dt, path="seq", tile_variant=n, state=True)
            except L.LrscanError:
                break
            check_cstate(inp, dt, h0, gl, seg, path="seq", tile_variant=n)
            n += 1
        assert n > 5


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_state_grouped_prefix_and_unaligned(dt):
    inp, h0, gl, seg = _cstate_inputs(1, 40000, 8, dt, seed=580)
    check_cstate(inp, dt, h0, gl, seg, chunk_len=16, tile_variant=2)  # five groups of 512 chunk maps
    check_cstate(inp, dt, h0, gl, seg, chunk_len=16, tile_variant=1)
    inp, h0, gl, seg = _cstate_inputs(2, 500, 37, dt, seed=581)      # rows not 16-byte aligned
    check_cstate(inp, dt, h0, gl, seg, chunk_len=32)


def test_complex_state_absent_equals_plain_and_empty():
    inp = make_complex_inputs(2, 300, 64, "f32", seed=590)
    cu = {k: inp[k].cuda() for k in PLANES}
    a = L.lrscan_cfwd(cu["ar"], cu["ai"], cu["br"], cu["bi"], path="chunk")
    b = L.lrscan_cfwd_state(cu["ar"], cu["ai"], cu["br"], cu["bi"], path="chunk")
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    ga = L.lrscan_cbwd(cu["ar"], cu["ai"], a[0], a[1], cu["go_r"], cu["go_i"], path="chunk")
    gb = L.lrscan_cbwd_state(cu["ar"], cu["ai"], a[0], a[1], cu["go_r"], cu["go_i"], path="chunk")
    for x, y in zip(ga, gb[:4]):
        assert torch.equal(x, y)
    # T == 0: last = h0, grad_h0 = grad_last
    e = torch.empty((2, 0, 16), device="cuda")
    h0 = (torch.randn(2, 16, device="cuda"), torch.randn(2, 16, device="cuda"))
    gl = (torch.randn(2, 16, device="cuda"), torch.randn(2, 16, device="cuda"))
    _, _, lr, li = L.lrscan_cfwd_state(e, e, e, e, h0=h0)
    assert torch.equal(lr, h0[0]) and torch.equal(li, h0[1])
    g = L.lrscan_cbwd_state(e, e, e, e, e, e, grad_last=gl)
    assert torch.equal(g[4], gl[0]) and torch.equal(g[5], gl[1])
    # the plain complex kernels carry no state
    x = torch.zeros((1, 64, 16), device="cuda")
    with pytest.raises(L.LrscanError):
        L.lrscan_cfwd_state(x, x, x, x, h0=(x[:, 0], x[:, 0]), path="plain")
    assert L.lrscan_sync_check() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_complex_scan_state_autograd(dt):
    """The autograd wrapper: gradients of Re(conj(go) h) + Re(conj(gl) last)
    to the decays, the inputs and h0 against the oracle."""
    B, T, D = 2, 300, 64
    inp, h0, gl, seg = _cstate_inputs(B, T, D, dt, seed=595)
    xs = [inp[k].cuda().requires_grad_() for k in ("ar", "ai", "br", "bi")]
    th0 = [torch.from_numpy(x).cuda().requires_grad_() for x in h0]
    tseg = torch.from_numpy(seg).cuda()
    out_r, out_i, last_r, last_i = L.complex_scan_state(*xs, h0=tuple(th0), segment_pos=tseg)
    go_r, go_i = inp["go_r"].cuda().float(), inp["go_i"].cuda().float()
    glr, gli = (torch.from_numpy(x).cuda() for x in gl)
    loss = (out_r.float() * go_r + out_i.float() * go_i).sum() + (last_r * glr + last_i * gli).sum()
    loss.backward()
    o = oracle.default()
    np_in = {k: to_np(inp[k]) for k in PLANES}
    ref = o.cfwd_state(np_in["ar"], np_in["ai"], np_in["br"], np_in["bi"], dt, h0=tuple(h0), segment_pos=seg)
    gref = o.cbwd_state(np_in["ar"], np_in["ai"], ref[0], ref[1], np_in["go_r"], np_in["go_i"], dt, h0=tuple(h0),
                        segment_pos=seg, grad_last=tuple(gl))
    for x, r in zip(xs, gref[:4]):
        assert_close(to_np(x.grad), r, dt, "complex state autograd", reassociated=True)
    for x, r in zip(th0, gref[4:]):
        assert_last_close(x.grad.cpu().numpy(), r, "grad h0 (autograd)")
