"""The chunked forward that allocates nothing (lrscan_fwd_chunk_noalloc).

Some callers cannot call cudaMalloc while they run -- code inside an
allocator or memory-pool callback, loops that ban allocation because it can
synchronize the device, hosts that give the library only pre-sized buffers.
For them the library keeps the chunked path's scratch in a fixed device
array.  This test calls that entry point through the C ABI and checks it
against the regular (allocating) entry point on the same inputs, on two
calls in a row with different shapes and dtypes, and checks that a problem
too large for the fixed scratch is refused before anything runs.

The file name puts it last in collection order; it depends on no other test.
"""
import numpy as np
import pytest
import torch

from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import random_inputs
from parity_util import assert_close, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20     # LRSCAN_NOALLOC_SCRATCH_BYTES in include/lrscan.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return L.lib()


def _noalloc(lib, a, b, chunk, stream):
    B, T, D = a.shape
    out = torch.empty_like(a)
    last = torch.empty((B, D), device=a.device, dtype=torch.float32)
    code = L.F32 if a.dtype == torch.float32 else L.BF16
    rc = lib.lrscan_fwd_chunk_noalloc(a.data_ptr(), b.data_ptr(), out.data_ptr(), last.data_ptr(),
                                      B, T, D, code, chunk, stream.cuda_stream)
    assert rc == L.LRSCAN_OK, (rc, lib.lrscan_last_error())
    return out, last


def test_noalloc_matches_the_allocating_chunked_forward_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream()
    cases = [(2, 3000, 256, "f32", 64), (3, 777, 136, "bf16", 32)]
    for (B, T, D, dt, chunk) in cases:
        inp = random_inputs(B, T, D, dt, seed=B * 1000 + T, a_lo=0.7, a_hi=1.0)
        a, b = inp["a"].cuda(), inp["b"].cuda()
        out_ref, last_ref = L.lrscan_fwd(a, b, path="chunk", chunk_len=chunk)
        out, last = _noalloc(lib, a, b, chunk, stream)
        assert L.lrscan_sync_check() == 0
        assert_close(to_np(out), to_np(out_ref), dt, f"no-alloc out {dt}", reassociated=True)
        assert_close(last.cpu().numpy(), last_ref.cpu().numpy(), "f32", f"no-alloc last {dt}")


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    # 2 * B * ceil(T/C) * D * 4 bytes = 64 MiB > 32 MiB: refused before any
    # launch, so the small buffers below are never read.
    x = torch.zeros(16, device="cuda")
    B, T, D, C = 1, 64 * 4096, 2048, 64
    assert 2 * B * (T // C) * D * 4 > SCRATCH_BYTES
    rc = lib.lrscan_fwd_chunk_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), None, B, T, D,
                                      L.F32, C, None)
    assert rc == L.LRSCAN_ENOMEM
    assert b"scratch" in lib.lrscan_last_error()
    assert L.lrscan_sync_check() == 0
