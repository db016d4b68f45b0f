"""GPU parity at full size: the named workloads 2-5 on the automatic plan
(the launch configuration the benchmark times), every element of every
output against the oracle, under the scan's stated tolerances with no
allowance: exact plans bit for bit, other bf16 outputs within 2 bf16 ulps of
the oracle, other fp32 outputs within 1e-4 (1 + |ref|).

The oracle runs over the whole tensors on every host core (disjoint lane
blocks in spawn-started processes, tests/oracle_pool.py).  The backward is fed
the oracle's own forward output, so each compared number depends on
oracle-side inputs only.  Workload 5 also checks the identity-padding
contract on the GPU's own forward and backward: its plans must be exact, so
the final state equals the state at the last valid token bit for bit.
"""
import numpy as np
import pytest
import torch

from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS, from_numpy_storage, make_inputs
from oracle_pool import OraclePool
from parity_util import assert_close, assert_last_close, bf16_beyond_ulps, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    p = OraclePool()
    yield p
    p.close()


def exact_plan(plan) -> bool:
    """Plans whose every result is the sequential definition's own."""
    return bool(plan["exact"])


def compare(got, ref, dt, what, exact):
    """Whole-tensor comparison, one batch row at a time (bounded host memory);
    prints the count of bf16 points beyond 2 ulps."""
    beyond = near = 0
    if dt == "bf16":
        for bb in range(got.shape[0]):
            n, m = bf16_beyond_ulps(got[bb:bb + 1], ref[bb:bb + 1])
            beyond, near = beyond + n, near + m
    print(f"[fullsize] {what}: {got.size} elements, exact={exact}, beyond 2 bf16 ulps: {beyond} "
          f"(of which within the fp32 rule: {near})", flush=True)
    for bb in range(got.shape[0]):
        assert_close(got[bb:bb + 1], ref[bb:bb + 1], dt, f"{what} row {bb}", exact=exact)
    return beyond


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_named_workload_full_size_every_element(cid, pool):
    w = WORKLOADS[cid]
    dt = w.dtype
    inp = make_inputs(cid)
    a, b, g = inp["a"], inp["b"], inp["grad_out"]
    plan = L.lrscan_plan(w.B, w.T, w.D, dt, "fwd")
    planb = L.lrscan_plan(w.B, w.T, w.D, dt, "bwd")
    exf, exb = exact_plan(plan), exact_plan(planb)
    ad, bd, gd = a.cuda(), b.cuda(), g.cuda()
    out, last = L.lrscan_fwd(ad, bd)
    assert L.lrscan_sync_check() == 0
    out_n, last_n = to_np(out), last.cpu().numpy()
    an, bn, gn = to_np(a), to_np(b), to_np(g)
    ref_out, ref_last = pool.fwd(an, bn, dt)
    compare(out_n, ref_out, dt, f"cfg{cid} out [{plan['name']}]", exf)
    assert_last_close(last_n, ref_last, f"cfg{cid} last [{plan['name']}]", exact=exf)

    ga, gb = L.lrscan_bwd(ad, from_numpy_storage(ref_out, dt).cuda(), gd)
    assert L.lrscan_sync_check() == 0
    ga_n, gb_n = to_np(ga), to_np(gb)
    del ga, gb
    ref_ga, ref_gb = pool.bwd(an, ref_out, gn, dt)
    compare(gb_n, ref_gb, dt, f"cfg{cid} grad_b [{planb['name']}]", exb)
    compare(ga_n, ref_ga, dt, f"cfg{cid} grad_a [{planb['name']}]", exb)

    if w.padded:
        # the padding contract on the GPU's own forward and backward; it is
        # bit-exact only on exact plans, so the plans must be exact
        assert exf and exb, (plan["name"], planb["name"])
        ga2, gb2 = L.lrscan_bwd(ad, out, gd)
        assert L.lrscan_sync_check() == 0
        lengths = inp["lengths"].numpy()
        ga2, gb2 = to_np(ga2), to_np(gb2)
        for bb in range(w.B):
            n = int(lengths[bb])
            assert not np.any(ga2[bb, n:]) and not np.any(gb2[bb, n:])
            assert np.array_equal(last_n[bb], out_n[bb, -1])
            assert np.array_equal(last_n[bb], out_n[bb, n - 1]), bb
            assert (out_n[bb, n:] == out_n[bb, n - 1][None, :]).all(), bb
