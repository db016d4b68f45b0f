"""The chunked forward that allocates nothing (lrscan_fwd_chunk_noalloc).

Some callers cannot call cudaMalloc while they run -- code inside an
allocator or memory-pool callback, loops that ban allocation because it can
synchronize the device, hosts that give the library only pre-sized buffers.
For them the library keeps the chunked path's scratch in a fixed device
array.  These tests call that entry point through the C ABI and check it
against the CPU oracle (the sequential definition) element by element, and
against the regular (allocating) entry point, on calls in a row with
different shapes, dtypes and chunk lengths, ragged sequence ends, without a
final-state output, with an empty sequence, and check that a problem too
large for the fixed scratch is refused before anything runs.

The file name puts it last in collection order; it depends on no other test.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_recurrence_scan_lrscan_gb300 import lrscan as L
from linear_recurrence_scan_lrscan_gb300.workloads import random_inputs
from parity_util import assert_close, assert_last_close, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20     # LRSCAN_NOALLOC_SCRATCH_BYTES in include/lrscan.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return L.lib()


def _noalloc(lib, a, b, chunk, stream, want_last=True):
    B, T, D = a.shape
    out = torch.full_like(a, 7.0)
    last = torch.full((B, D), 7.0, device=a.device, dtype=torch.float32) if want_last else None
    code = L.F32 if a.dtype == torch.float32 else L.BF16
    rc = lib.lrscan_fwd_chunk_noalloc(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                      last.data_ptr() if want_last else None, B, T, D, code, chunk,
                                      stream.cuda_stream)
    assert rc == L.LRSCAN_OK, (rc, lib.lrscan_last_error())
    return out, last


# (B, T, D, dtype, chunk_len): T not a multiple of the chunk length in most
# cases (a ragged last chunk); chunk_len 0 means the default 64
CASES = [(2, 3000, 256, "f32", 64), (3, 777, 136, "bf16", 32), (2, 1001, 64, "f32", 16),
         (1, 4099, 40, "bf16", 0), (4, 129, 24, "f32", 32), (2, 2050, 512, "bf16", 16)]


@pytest.mark.parametrize("want_last", [True, False])
def test_noalloc_matches_the_oracle_on_calls_in_a_row(lib, want_last):
    stream = torch.cuda.current_stream()
    o = oracle.default()
    for (B, T, D, dt, chunk) in CASES:
        inp = random_inputs(B, T, D, dt, seed=B * 1000 + T, a_lo=0.7, a_hi=1.0)
        a, b = inp["a"].cuda(), inp["b"].cuda()
        ref_out, ref_last = o.fwd(to_np(inp["a"]), to_np(inp["b"]), dt)
        out, last = _noalloc(lib, a, b, chunk, stream, want_last)
        assert L.lrscan_sync_check() == 0
        what = f"no-alloc {dt} B={B} T={T} D={D} C={chunk}"
        # the chunked forward re-associates: held to the scan's tolerances
        assert_close(to_np(out), ref_out, dt, f"{what} out", reassociated=True)
        if want_last:
            assert_last_close(last.cpu().numpy(), ref_last, f"{what} last")
            if dt == "f32":
                assert np.array_equal(last.cpu().numpy(), to_np(out)[:, -1, :])


def test_noalloc_matches_the_allocating_chunked_forward_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream()
    for (B, T, D, dt, chunk) in CASES[:2]:
        inp = random_inputs(B, T, D, dt, seed=B * 1000 + T, a_lo=0.7, a_hi=1.0)
        a, b = inp["a"].cuda(), inp["b"].cuda()
        out_ref, last_ref = L.lrscan_fwd(a, b, path="chunk", chunk_len=chunk or 64)
        out, last = _noalloc(lib, a, b, chunk, stream)
        assert L.lrscan_sync_check() == 0
        # both take the flat chunk prefix at these sizes: the same operations
        assert torch.equal(out, out_ref) and torch.equal(last, last_ref)


def test_noalloc_empty_sequence_zeroes_last(lib):
    for dt in (torch.float32, torch.bfloat16):
        a = torch.empty(3, 0, 16, dtype=dt, device="cuda")
        last = torch.full((3, 16), 7.0, device="cuda")
        code = L.F32 if dt == torch.float32 else L.BF16
        rc = lib.lrscan_fwd_chunk_noalloc(a.data_ptr(), a.data_ptr(), a.data_ptr(), last.data_ptr(), 3, 0, 16,
                                          code, 0, None)
        assert rc == L.LRSCAN_OK
        assert L.lrscan_sync_check() == 0
        assert not last.any()


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
