"""CUDA graphs: the device entry points captured into a graph and replayed.

Each case runs the calls once on the capture stream (which sizes that
stream's library-owned workspace), captures them, writes new values into the
captured input buffers, replays, and compares the outputs bit for bit with
eager calls on the new values (same plans, same kernels).  A captured call
that would have to grow the workspace must fail before it enqueues anything;
that case runs in a child process so that nothing of it can leak into the
other tests.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import make_complex_inputs, make_gated_inputs, random_inputs

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    yield
    assert L.lrscan_sync_check() == 0


def _same(x, y, name):
    assert x.shape == y.shape and x.dtype == y.dtype, name
    if x.dtype in (torch.bfloat16, torch.float16):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), name
    else:
        assert torch.equal(x.view(torch.int32), y.view(torch.int32)), name


def _graph_replay_matches_eager(static: dict, run, fresh: dict):
    """run(static) -> tuple of outputs.  Capture it, refill `static` from
    `fresh`, replay, compare with run(fresh) issued eagerly."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(static)  # outside capture: sizes this stream's workspace
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        outs = run(static)
    for k, v in fresh.items():
        static[k].copy_(v)
    g.replay()
    torch.cuda.synchronize()
    ref = run({k: v.clone() for k, v in fresh.items()})
    torch.cuda.synchronize()
    assert L.lrscan_sync_check() == 0
    assert len(outs) == len(ref)
    for i, (o, r) in enumerate(zip(outs, ref)):
        if o is not None:
            _same(o, r, f"output {i}")
    # a second replay with other values: the graph holds no stale state
    for k, v in fresh.items():
        static[k].copy_(v.flip(1) if v.ndim == 3 else v)
    g.replay()
    torch.cuda.synchronize()
    ref2 = run({k: static[k].clone() for k in static})
    for i, (o, r) in enumerate(zip(outs, ref2)):
        if o is not None:
            _same(o, r, f"output {i} (second replay)")


def _real(B, T, D, dt, seed):
    inp = random_inputs(B, T, D, dt, seed=seed, a_lo=0.6, a_hi=1.0)
    return {k: inp[k].cuda() for k in ("a", "b", "grad_out")}


@pytest.mark.parametrize("dt,shape,kw", [
    ("bf16", (3, 300, 200), {}),                                  # automatic (windowed) tiles
    ("f32", (2, 1000, 96), {"path": "chunk", "chunk_len": 64}),   # chunked: library-owned workspace
    ("f32", (2, 257, 64), {"path": "seq"}),
])
def test_fwd_bwd_step_replays(dt, shape, kw):
    B, T, D = shape

    def run(x):
        out, last = L.lrscan_fwd(x["a"], x["b"], **kw)
        ga, gb = L.lrscan_bwd(x["a"], out, x["grad_out"], **kw)
        return out, last, ga, gb

    _graph_replay_matches_eager(_real(B, T, D, dt, 1000), run, _real(B, T, D, dt, 1001))


def _segments(B, T, seed):
    r = np.random.default_rng(seed)
    pos = np.zeros((B, T), dtype=np.int32)
    starts = r.random((B, T)) < 0.02
    for t in range(1, T):
        pos[:, t] = np.where(starts[:, t], 0, pos[:, t - 1] + 1)
    return torch.from_numpy(pos).cuda()


def test_state_step_replays():
    B, T, D, dt = 3, 300, 256, "bf16"

    def case(seed):
        x = _real(B, T, D, dt, seed)
        g = torch.Generator("cpu").manual_seed(seed)
        x["h0"] = torch.randn(B, D, generator=g).cuda()
        x["grad_last"] = torch.randn(B, D, generator=g).cuda()
        x["seg"] = _segments(B, T, seed)
        return x

    def run(x):
        out, last = L.lrscan_fwd_state(x["a"], x["b"], h0=x["h0"], segment_pos=x["seg"])
        ga, gb, gh0 = L.lrscan_bwd_state(x["a"], out, x["grad_out"], h0=x["h0"], segment_pos=x["seg"],
                                         grad_last=x["grad_last"])
        return out, last, ga, gb, gh0

    _graph_replay_matches_eager(case(1010), run, case(1011))


def test_complex_step_replays():
    B, T, D, dt = 2, 200, 64, "bf16"
    planes = ("ar", "ai", "br", "bi", "go_r", "go_i")

    def case(seed):
        inp = make_complex_inputs(B, T, D, dt, seed=seed)
        return {k: inp[k].cuda() for k in planes}

    def run(x):
        out_r, out_i, last_r, last_i = L.lrscan_cfwd(x["ar"], x["ai"], x["br"], x["bi"])
        grads = L.lrscan_cbwd(x["ar"], x["ai"], out_r, out_i, x["go_r"], x["go_i"])
        return (out_r, out_i, last_r, last_i, *grads)

    _graph_replay_matches_eager(case(1020), run, case(1021))


def test_complex_state_step_replays():
    """The state-carrying complex scan (chunked path, library-owned workspace)."""
    B, T, D, dt = 2, 300, 64, "bf16"
    planes = ("ar", "ai", "br", "bi", "go_r", "go_i")

    def case(seed):
        inp = make_complex_inputs(B, T, D, dt, seed=seed)
        x = {k: inp[k].cuda() for k in planes}
        g = torch.Generator("cpu").manual_seed(seed)
        for k in ("h0_r", "h0_i", "gl_r", "gl_i"):
            x[k] = torch.randn(B, D, generator=g).cuda()
        x["seg"] = _segments(B, T, seed)
        return x

    def run(x):
        out = L.lrscan_cfwd_state(x["ar"], x["ai"], x["br"], x["bi"], h0=(x["h0_r"], x["h0_i"]), segment_pos=x["seg"])
        g = L.lrscan_cbwd_state(x["ar"], x["ai"], out[0], out[1], x["go_r"], x["go_i"], h0=(x["h0_r"], x["h0_i"]),
                                segment_pos=x["seg"], grad_last=(x["gl_r"], x["gl_i"]))
        return (*out, *g)

    _graph_replay_matches_eager(case(1040), run, case(1041))


def test_generated_decay_step_replays():
    B, T, D, dt = 2, 300, 128, "bf16"

    def case(seed):
        inp = make_gated_inputs(B, T, D, dt, seed=seed)
        return {k: inp[k].cuda() for k in ("eta", "nu_log", "b", "grad_out")}

    def run(x):
        out, last = L.lrscan_fwd_gated(x["eta"], x["nu_log"], x["b"])
        gb, geta, gnu = L.lrscan_bwd_gated(x["eta"], x["nu_log"], out, x["grad_out"])
        return out, last, gb, geta, gnu

    _graph_replay_matches_eager(case(1030), run, case(1031))


_GROWTH_UNDER_CAPTURE = r"""
import torch
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
a = torch.rand(1, 4096, 64, device="cuda") * 0.5 + 0.4
b = torch.randn_like(a)
L.lrscan_fwd(a[:, :64].contiguous(), b[:, :64].contiguous(), path="chunk")  # first call, small workspace
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
try:
    with torch.cuda.graph(g, stream=s):
        L.lrscan_fwd(a, b, path="chunk")  # needs a larger workspace on the capture stream
except L.LrscanError as e:
    assert "stream capture" in str(e), str(e)
    print("refused")
else:
    raise SystemExit("the captured call grew the workspace")
out, last = L.lrscan_fwd(a, b, path="chunk")  # outside capture: grows and runs
ref, _ = L.lrscan_fwd(a, b, path="seq")
torch.cuda.synchronize()
assert L.lrscan_sync_check() == 0
assert torch.allclose(out, ref, rtol=1e-4, atol=1e-4)
print("ok")
"""


def test_workspace_growth_under_capture_is_refused():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", _GROWTH_UNDER_CAPTURE], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split() == ["refused", "ok"], r.stdout + r.stderr
