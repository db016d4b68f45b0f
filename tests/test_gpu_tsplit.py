"""GPU side of a sequence split across devices: the whole-sequence summary
(lrscan_summary) and the map composition (lrscan_compose_maps) against the
oracle, and the split protocol run as W simulated segments on one GPU (the
exchange replaced by the list of every segment's maps) against the oracle's
whole-sequence state-carrying scan."""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300 import tsplit
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


def _seg(B, T, seed):
    r = np.random.default_rng(seed)
    pos = np.ones((B, T), dtype=np.int32)
    pos[r.random((B, T)) < 0.02] = 0
    pos[0, 0] = 0
    return pos


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 300, 200), (2, 77, 37), (1, 1, 8)])
@pytest.mark.parametrize("with_seg", [False, True])
def test_summary_matches_oracle(dt, shape, with_seg):
    B, T, D = shape
    inp = random_inputs(B, T, D, dt, seed=400, a_lo=0.6, a_hi=1.0)
    a, b, g = (to_np(inp[k]) for k in ("a", "b", "grad_out"))
    seg = _seg(B, T, 401) if with_seg else None
    o = oracle.default()
    z = np.zeros_like(a)
    ones = np.ones((B, D), dtype=np.float32)
    segd = torch.from_numpy(seg).cuda() if with_seg else None
    P, Q = L.lrscan_summary(inp["a"].cuda(), inp["b"].cuda(), segment_pos=segd, direction="fwd")
    _, P_ref = o.fwd_state(a, z, dt, h0=ones, segment_pos=seg)
    _, Q_ref = o.fwd_state(a, b, dt, segment_pos=seg)
    assert_last_close(P.cpu().numpy(), P_ref, "P fwd", exact=True)
    assert_last_close(Q.cpu().numpy(), Q_ref, "Q fwd", exact=True)
    P, Q = L.lrscan_summary(inp["a"].cuda(), inp["grad_out"].cuda(), segment_pos=segd, direction="bwd")
    _, _, P_ref = o.bwd_state(a, z, z, dt, segment_pos=seg, grad_last=ones)
    _, _, Q_ref = o.bwd_state(a, z, g, dt, segment_pos=seg)
    assert_last_close(P.cpu().numpy(), P_ref, "P bwd", exact=True)
    assert_last_close(Q.cpu().numpy(), Q_ref, "Q bwd", exact=True)
    assert L.lrscan_sync_check() == 0


def test_summary_of_empty_sequence_is_identity():
    a = torch.empty((2, 0, 16), device="cuda")
    P, Q = L.lrscan_summary(a, a)
    assert torch.equal(P, torch.ones_like(P)) and not Q.any()


@pytest.mark.parametrize("W", [1, 2, 5])
def test_compose_maps_matches_oracle(W):
    B, D = 3, 50
    r = np.random.default_rng(410 + W)
    maps = np.stack([r.uniform(0.5, 1.0, (B, D)), r.standard_normal((B, D))], axis=0)[None].repeat(W, 0)
    maps = (maps * r.uniform(0.9, 1.1, maps.shape)).astype(np.float32)
    init = r.standard_normal((B, D)).astype(np.float32)
    md, idev = torch.from_numpy(maps).cuda(), torch.from_numpy(init).cuda()
    o = oracle.default()
    for rank in range(W):
        for direction, order in (("fwd", list(range(rank))), ("bwd", list(range(W - 1, rank, -1)))):
            got = L.lrscan_compose_maps(md, rank, idev, direction).cpu().numpy()
            if order:
                Ps = np.ascontiguousarray(np.stack([maps[k][0] for k in order], axis=1))
                Qs = np.ascontiguousarray(np.stack([maps[k][1] for k in order], axis=1))
                _, ref = o.fwd_state(Ps, Qs, "f32", h0=init)
            else:
                ref = init
            assert np.array_equal(got, ref), (rank, direction)
            none = L.lrscan_compose_maps(md, rank, None, direction).cpu().numpy()
            if not order:
                assert not none.any()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("cuts", [(0, 100, 300), (0, 1, 129, 250, 300)])
def test_split_protocol_simulated_segments(dt, cuts):
    B, T, D = 3, 300, 200
    inp = random_inputs(B, T, D, dt, seed=420, a_lo=0.6, a_hi=1.0)
    seg = _seg(B, T, 421)
    r = np.random.default_rng(422)
    h0 = r.standard_normal((B, D)).astype(np.float32)
    gl = r.standard_normal((B, D)).astype(np.float32)
    W = len(cuts) - 1
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    part = lambda t, k: t[:, cuts[k]:cuts[k + 1]].contiguous().cuda()  # noqa: E731
    ops = tsplit.LibraryOps()
    a_s = [part(inp["a"], k) for k in range(W)]
    b_s = [part(inp["b"], k) for k in range(W)]
    g_s = [part(inp["grad_out"], k) for k in range(W)]
    s_s = [dev(seg[:, cuts[k]:cuts[k + 1]]) for k in range(W)]
    fmaps = [ops.summary(a_s[k], b_s[k], s_s[k], "fwd") for k in range(W)]
    outs, lasts, hins = [], [], []
    for k in range(W):
        o_, l_, h_ = tsplit.tsplit_forward(a_s[k], b_s[k], h0=dev(h0), segment_pos=s_s[k], ops=ops,
                                           gather=lambda local, group: fmaps, rank=k)
        outs.append(o_), lasts.append(l_), hins.append(h_)
    bmaps = [ops.summary(a_s[k], g_s[k], s_s[k], "bwd") for k in range(W)]
    grads = [tsplit.tsplit_backward(a_s[k], outs[k], g_s[k], h_in=hins[k], segment_pos=s_s[k], grad_last=dev(gl),
                                    ops=ops, gather=lambda local, group: bmaps, rank=k) for k in range(W)]
    assert L.lrscan_sync_check() == 0
    o = oracle.default()
    a, b, g = (to_np(inp[k]) for k in ("a", "b", "grad_out"))
    ref_out, ref_last = o.fwd_state(a, b, dt, h0=h0, segment_pos=seg)
    ref_ga, ref_gb, ref_gh0 = o.bwd_state(a, ref_out, g, dt, h0=h0, segment_pos=seg, grad_last=gl)
    assert_close(to_np(torch.cat(outs, 1)), ref_out, dt, "split out", reassociated=True)
    assert_last_close(lasts[-1].cpu().numpy(), ref_last, "split last")
    assert_close(to_np(torch.cat([x[1] for x in grads], 1)), ref_gb, dt, "split grad_b", reassociated=True)
    assert_close(to_np(torch.cat([x[0] for x in grads], 1)), ref_ga, dt, "split grad_a", reassociated=True)
    assert_last_close(grads[0][2].cpu().numpy(), ref_gh0, "split grad_h0")
