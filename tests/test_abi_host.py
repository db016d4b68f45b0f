"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point the header declares, rejects bad arguments before touching
a device, and the occupancy rule picks the expected paths."""
import ctypes
import os
import re

import pytest

from linear_recurrence_scan_lrscan_gb300 import lrscan as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lrscan.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lrscan_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    try:
        return L.lib()
    except L.LrscanUnavailable as e:
        pytest.fail(f"CUDA library not built: {e}")


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("lrscan_fwd", "lrscan_bwd", "lrscan_fwd_ex", "lrscan_bwd_ex", "lrscan_set_stream",
                     "lrscan_workspace_bytes", "lrscan_sync_check", "lrscan_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    for n in _declared():
        assert n in L.EXPORTS, f"binding does not declare {n}"


def test_version_and_strerror(lib):
    assert lib.lrscan_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.lrscan_strerror(code)
    assert L.strerror(-5) == "a bounded device wait timed out"


def _fwd(lib, a, b, out, last, B, T, D, dtype):
    return lib.lrscan_fwd(a, b, out, last, B, T, D, dtype)


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    p = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails validation
    assert _fwd(lib, p, p, p, None, 1, 8, 8, 7) == L.LRSCAN_EDTYPE
    assert _fwd(lib, p, p, p, None, -1, 8, 8, 0) == L.LRSCAN_EINVAL
    assert _fwd(lib, p, p, p, None, 1, -8, 8, 0) == L.LRSCAN_EINVAL
    assert _fwd(lib, p, p, p, None, 1, 8, -8, 1) == L.LRSCAN_EINVAL
    assert _fwd(lib, p, p, p, None, 1, 1 << 31, 8, 0) == L.LRSCAN_EINVAL          # T over int32
    assert _fwd(lib, p, p, p, None, 1 << 40, 1 << 20, 1 << 20, 0) == L.LRSCAN_EINVAL  # byte overflow
    assert _fwd(lib, None, p, p, None, 1, 8, 8, 0) == L.LRSCAN_EINVAL
    assert _fwd(lib, p, None, p, None, 1, 8, 8, 0) == L.LRSCAN_EINVAL
    assert _fwd(lib, p, p, None, None, 1, 8, 8, 0) == L.LRSCAN_EINVAL
    assert lib.lrscan_bwd(p, p, p, None, p, 1, 8, 8, 0) == L.LRSCAN_EINVAL
    assert lib.lrscan_bwd(p, p, p, p, p, 1, 8, 8, 3) == L.LRSCAN_EDTYPE


def test_wait_limit_has_a_floor(lib):
    """The device wait limit also bounds the kernels' drains of their own bulk
    copies, so limits under 1 ms are refused; the default (1 s) is restored."""
    assert lib.lrscan_set_wait_timeout_ns(0) == L.LRSCAN_EINVAL
    assert lib.lrscan_set_wait_timeout_ns(999_999) == L.LRSCAN_EINVAL
    assert lib.lrscan_set_wait_timeout_ns(1_000_000) == L.LRSCAN_OK
    assert lib.lrscan_set_wait_timeout_ns(1_000_000_000) == L.LRSCAN_OK


def test_empty_problems_are_noops(lib):
    # B == 0 or D == 0: nothing to do, NULL pointers allowed, no device needed
    assert _fwd(lib, None, None, None, None, 0, 8, 8, 0) == L.LRSCAN_OK
    assert _fwd(lib, None, None, None, None, 4, 8, 0, 1) == L.LRSCAN_OK
    assert lib.lrscan_bwd(None, None, None, None, None, 0, 5, 5, 0) == L.LRSCAN_OK
    assert lib.lrscan_bwd(None, None, None, None, None, 3, 0, 5, 0) == L.LRSCAN_OK


def test_workspace_bytes(lib):
    # two fp32 [B, ceil(T/C), D] buffers, each rounded up to 256 bytes
    pad = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # P and Q [B, Nc, D] plus the grouped prefix's PG and QG [B, ceil(Nc / 512), D]
    assert L.lrscan_workspace_bytes(1, 65536, 2560, 64) == 2 * 1024 * 2560 * 4 + 2 * 2 * 2560 * 4
    assert L.lrscan_workspace_bytes(2, 100, 3, 16) == 2 * pad(2 * 7 * 3 * 4) + 2 * pad(2 * 1 * 3 * 4)
    assert L.lrscan_workspace_bytes(1, 64, 8, 0) == L.lrscan_workspace_bytes(1, 64, 8, 64)
    assert L.lrscan_workspace_bytes(1, 64, 8, 48) == 0


EXPECTED_AUTO = {
    # workload: (forward tile, backward tile) the occupancy rule must pick
    2: ("win_bf16_d32_s8_m5_n2", "wfx_bf16_d32_s3_l16"),
    3: ("win_f32_d32_s31", "win_f32_d32_s16"),
    4: ("seq_bf16_d128_n3", "wfx_bf16_d64_s4_l16_v2"),
    5: ("seq_f32_d64_v1_n3", "xwin_f32_d64_s8"),
}
# which of those reproduce the sequential definition bit for bit
EXPECTED_EXACT = {2: (False, True), 3: (False, False), 4: (True, True), 5: (True, True)}


@pytest.mark.parametrize("cid", sorted(EXPECTED_AUTO))
def test_occupancy_rule_on_the_named_workloads(lib, cid):
    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS
    w = WORKLOADS[cid]
    for direction, want, exact in zip(("fwd", "bwd"), EXPECTED_AUTO[cid], EXPECTED_EXACT[cid]):
        p = L.lrscan_plan(w.B, w.T, w.D, w.dtype, direction)
        assert p["name"] == want, (cid, direction, p)
        assert p["exact"] == int(exact), (cid, direction, p)
        assert p["kernels"] == 1
        # every lane tile of the GPU-filling variants gets a CTA of its own
        assert p["ctas"] == w.B * -(-w.D // p["lanes_per_cta"])


def test_state_plans(lib):
    """Calls with carried state plan with their own backward list: the
    16-sub-chunk tiles at every lane count (the plain backward moves to the
    16-row tile above five CTAs per SM); forwards are shared."""
    from linear_recurrence_scan_lrscan_gb300.workloads import WORKLOADS
    for cid, want in ((2, "win_bf16_d32_s16_n4"), (4, "win_bf16_d32_s16_n2")):
        w = WORKLOADS[cid]
        assert L.lrscan_plan(w.B, w.T, w.D, w.dtype, "bwd", state=True)["name"] == want
        assert L.lrscan_plan(w.B, w.T, w.D, w.dtype, "fwd", state=True)["name"] == EXPECTED_AUTO[cid][0]
    w = WORKLOADS[4]
    assert L.lrscan_plan(w.B, w.T, w.D, w.dtype, "bwd")["name"] == EXPECTED_AUTO[4][1] == "wfx_bf16_d64_s4_l16_v2"


def test_fp32_forward_prefers_the_exact_sequential_path_when_lanes_fill_the_gpu(lib):
    for (B, T, D, dt) in [(64, 512, 1024, "f32"), (32, 1000, 4096, "f32")]:
        assert L.lrscan_plan(B, T, D, dt, "fwd")["path"] == "seq"


def test_bf16_forward_tiles(lib):
    """Few lanes: the high-residency window tile puts every CTA of the lane
    tiling on the GPU at once (5 per SM), the measured fastest bf16 forward
    there.  From two 128-lane tiles per SM: the exact sequential tile."""
    p = L.lrscan_plan(8, 2048, 2560, "bf16", "fwd")
    assert p["name"] == "win_bf16_d32_s8_m5_n2" and p["path"] == "window", p
    assert p["threads_per_cta"] == 8 * 16 + 32
    p = L.lrscan_plan(16, 4096, 4096, "bf16", "fwd")
    assert p["name"] == "seq_bf16_d128_n3" and p["path"] == "seq" and p["exact"] == 1, p


def test_exact_flag_of_every_tile_variant(lib):
    """Sequential tiles and the exact-walk window tiles report exact results;
    re-associating window tiles and the chunked path do not; plain kernels do."""
    for dt in ("f32", "bf16"):
        for path in ("seq", "window"):
            for v in range(1, L.lrscan_num_variants(path, dt) + 1):
                p = L.lrscan_plan(4, 512, 1024, dt, "fwd", path=path, tile_variant=v)
                want = path == "seq" or p["name"].startswith(("xwin_", "wfx_"))
                assert p["exact"] == int(want), p
        assert L.lrscan_plan(1, 1 << 16, 64, dt, "fwd", path="chunk")["exact"] == 0
        assert L.lrscan_plan(4, 512, 1024, dt, "fwd", path="plain")["exact"] == 1
        assert L.lrscan_plan_gated(4, 512, 1024, dt, "fwd", path="plain")["exact"] == 0


def test_occupancy_rule_few_lanes_long_sequence(lib):
    # 2^20 steps and only 64 fp32 lanes: both directions stream the chunks in
    # one pass (1,024 chunks of 512 steps per lane group), with or without
    # carried state; the chunked path's grouped prefix (512-step chunks
    # forward, 128 backward) when it is asked for
    for direction in ("fwd", "bwd"):
        for state in (False, True):
            p = L.lrscan_plan(1, 1 << 20, 64, "f32", direction, state=state)
            assert p["path"] == "stream" and p["name"] == "stream_f32_d32" and p["kernels"] == 1, p
            # bf16: the eight-warp 32-lane variant, with carried state and
            # resets the 64-lane tile
            q = L.lrscan_plan(1, 1 << 20, 64, "bf16", direction, state=state)
            want = "stream_bf16_d64" if state else "stream_bf16_d32"
            assert q["path"] == "stream" and q["name"] == want, q
    p = L.lrscan_plan(1, 1 << 20, 64, "f32", "fwd", path="chunk", state=True)
    assert p["path"] == "chunk" and p["kernels"] == 5 and p["name"].startswith("chunk512"), p
    assert p["name"].endswith("_grouped") and p["rows_per_window"] == 512
    assert p["workspace_bytes"] == L.lrscan_workspace_bytes(1, 1 << 20, 64, 512)
    p = L.lrscan_plan(1, 1 << 20, 64, "f32", "bwd", path="chunk", state=True)
    assert p["path"] == "chunk" and p["rows_per_window"] == 128 and p["name"].endswith("_grouped"), p
    # fp32 on 32-lane tiles (the forward in 256-step chunks from eight lane
    # groups); bf16 on the eight-warp 32-lane variant, except the forward from
    # four 64-lane groups (the 64-lane tile)
    want = {(1, 64, "bf16"): ("stream_bf16_d32", "stream_bf16_d32"),
            (8, 64, "f32"): ("stream_f32_d32_c256", "stream_f32_d32"),
            (1, 128, "f32"): ("stream_f32_d32", "stream_f32_d32"),
            (1, 256, "bf16"): ("stream_bf16_d64", "stream_bf16_d32"),
            (8, 64, "bf16"): ("stream_bf16_d64", "stream_bf16_d32")}
    for (B, D, dt), names in want.items():
        for direction, name in zip(("fwd", "bwd"), names):
            p = L.lrscan_plan(B, 1 << 18, D, dt, direction)
            lanes = 64 if "_d64" in name else 32
            assert p["path"] == "stream" and p["name"] == name and p["lanes_per_cta"] == lanes, (B, D, dt, p)
    # 32 chunks of 512 steps per lane group stream; fewer take the chunked path
    assert L.lrscan_plan(1, 16384, 64, "bf16", "fwd")["path"] == "stream"
    assert L.lrscan_plan(1, 8192, 64, "bf16", "fwd")["path"] == "chunk"
    # the chunked path's grouped prefix: too short for 2,048 chunks of 512, the
    # forward falls back to 256
    p = L.lrscan_plan(1, (1 << 19) + 1000, 64, "f32", "fwd", path="chunk")
    assert p["rows_per_window"] == 256 and p["name"].endswith("_grouped"), p
    # an explicit chunk length is kept
    p64 = L.lrscan_plan(1, 1 << 20, 64, "f32", "fwd", chunk_len=64)
    assert p64["rows_per_window"] == 64 and p64["name"].endswith("_grouped")
    flat = L.lrscan_plan(1, 1 << 20, 64, "f32", "fwd", path="chunk", tile_variant=1)
    assert flat["kernels"] == 3 and flat["workspace_bytes"] == 2 * 16384 * 64 * 4
    # few chunks per lane: the flat prefix
    p = L.lrscan_plan(1, 4096, 64, "f32", "fwd", path="chunk")
    assert p["kernels"] == 3 and not p["name"].endswith("_grouped")


def test_unaligned_rows_take_plain_loads(lib):
    p = L.lrscan_plan(4, 512, 1023, "f32", "fwd")          # D*4 not a multiple of 16
    assert p["path"] == "plain"
    p = L.lrscan_plan(4, 512, 1024, "bf16", "fwd", aligned=False)
    assert p["path"] == "plain"
    with pytest.raises(L.LrscanError):
        L.lrscan_plan(4, 512, 1023, "f32", "fwd", path="seq")   # TMA path cannot take it


def test_forced_paths_and_variants(lib):
    for path in ("seq", "window"):
        for dt in ("f32", "bf16"):
            n = L.lrscan_num_variants(path, dt)
            assert n >= 2
            names = set()
            for v in range(1, n + 1):
                p = L.lrscan_plan(8, 1000, 512, dt, "fwd", path=path, tile_variant=v)
                assert p["path"] == path and p["tile_variant"] == v
                names.add(p["name"])
            assert len(names) == n
            with pytest.raises(L.LrscanError):
                L.lrscan_plan(8, 1000, 512, dt, "fwd", path=path, tile_variant=n + 1)
    p = L.lrscan_plan(8, 1000, 512, "f32", "bwd", path="chunk", chunk_len=32)
    assert p["path"] == "chunk" and p["rows_per_window"] == 32
    with pytest.raises(L.LrscanError):
        L.lrscan_plan(8, 1000, 512, "f32", "bwd", path="chunk", chunk_len=48)
    with pytest.raises(L.LrscanError):
        L.lrscan_plan(8, 1000, 512, "f32", "bwd", path="chunk", chunk_len=1024)


def test_state_entry_points_validate_before_any_launch(lib):
    p = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails validation or is empty
    bad = L.State(h0=0x1002)      # not 4-byte aligned
    assert lib.lrscan_fwd_state(p, p, p, None, ctypes.byref(bad), 1, 8, 8, 0, None, None) == L.LRSCAN_EINVAL
    assert lib.lrscan_bwd_state(p, p, p, p, p, ctypes.byref(L.State(grad_h0=0x1001)), 1, 8, 8, 0, None,
                                None) == L.LRSCAN_EINVAL
    # the forward reads neither grad_last nor grad_h0
    fwd_only = L.State(grad_last=0x1003, grad_h0=0x1001)
    assert lib.lrscan_fwd_state(p, p, p, None, ctypes.byref(fwd_only), 0, 8, 8, 0, None, None) == L.LRSCAN_OK
    # empty batch or width: nothing to do, no device touched
    ok = L.State(h0=0x1000, segment_pos=0x2000, grad_last=0x3000, grad_h0=0x4000)
    for B, T, D in ((0, 8, 8), (2, 8, 0)):
        assert lib.lrscan_fwd_state(p, p, p, None, ctypes.byref(ok), B, T, D, 1, None, None) == L.LRSCAN_OK
        assert lib.lrscan_bwd_state(p, p, p, p, p, ctypes.byref(ok), B, T, D, 1, None, None) == L.LRSCAN_OK
    assert lib.lrscan_fwd_state(p, p, p, None, None, 1, 8, 8, 5, None, None) == L.LRSCAN_EDTYPE


def test_missing_library_fails_loudly_with_no_fallback(tmp_path):
    """Without liblrscan.so every entry point raises LrscanUnavailable: there
    is no CPU path to fall back to."""
    import subprocess
    import sys
    code = (
        "import torch\n"
        "from linear_recurrence_scan_lrscan_gb300 import lrscan as L\n"
        "a = torch.zeros(1, 4, 8)\n"
        "for call in (lambda: L.lrscan_plan(1, 4, 8, 'f32'),\n"
        "             lambda: L.lrscan_fwd_host(a, a, out=torch.empty_like(a), last=torch.empty(1, 8))):\n"
        "    try:\n"
        "        call()\n"
        "    except L.LrscanUnavailable:\n"
        "        continue\n"
        "    raise SystemExit('a call ran without the library')\n"
        "try:\n"
        "    L.lrscan_fwd(a, a)  # host tensors are refused: nothing computes on the CPU\n"
        "except (L.LrscanUnavailable, ValueError):\n"
        "    print('ok')\n")
    env = dict(os.environ, LRSCAN_LIBRARY=str(tmp_path / "absent.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.stdout, r.stderr)


def test_every_tile_variant_is_whole_warps(lib):
    """The tiled kernels' named barriers and mbarrier arrival counts take whole
    warps, so every variant of every table (real, carried-state, complex,
    generated-decay; both directions) must plan with a thread count that is a
    multiple of 32; the planner refuses an entry that is not."""
    B, T, D = 8, 1000, 512
    seen = 0
    for dt in ("f32", "bf16"):
        for direction in ("fwd", "bwd"):
            planners = [("real", lambda v, path: L.lrscan_plan(B, T, D, dt, direction, path=path, tile_variant=v)),
                        ("state", lambda v, path: L.lrscan_plan(B, T, D, dt, direction, path=path, tile_variant=v,
                                                                state=True)),
                        ("complex", lambda v, path: L.lrscan_plan_complex(B, T, D, dt, direction, path=path,
                                                                          tile_variant=v))]
            for what, plan in planners:
                for path in ("seq", "window"):
                    v = 1
                    while True:
                        try:
                            p = plan(v, path)
                        except L.LrscanError:
                            break
                        assert p["threads_per_cta"] % 32 == 0, (what, dt, direction, path, p)
                        seen += 1
                        v += 1
            v = 1
            while True:
                try:
                    p = L.lrscan_plan_gated(B, T, D, dt, direction, path="seq", tile_variant=v)
                except L.LrscanError:
                    break
                assert p["threads_per_cta"] % 32 == 0, ("gated", dt, direction, p)
                seen += 1
                v += 1
    assert seen > 40


def test_complex_chunked_plans(lib):
    """The complex scan's chunked path: automatic for few lanes (fewer than
    0.45 lane tiles of 32 per SM) and sequences too short to stream, or with
    an asked-for chunk length; twice the real path's scratch (re and
    im maps), flat or grouped prefix."""
    p = L.lrscan_plan_complex(1, 1 << 20, 64, "f32", "fwd", chunk_len=64)
    assert p["path"] == "chunk" and p["name"] == "cchunk64_v4_grouped" and p["kernels"] == 5, p
    assert L.lrscan_plan_complex(1, 8192, 64, "f32", "fwd")["path"] == "chunk"
    assert L.lrscan_plan_complex(1, 1 << 20, 64, "f32", "bwd", state=True)["path"] == "stream"
    assert L.lrscan_plan_complex(1, 1 << 20, 64, "f32", "bwd", state=True, chunk_len=64)["path"] == "chunk"
    assert p["workspace_bytes"] == 2 * L.lrscan_workspace_bytes(1, 1 << 20, 64, 64)
    flat = L.lrscan_plan_complex(1, 1 << 20, 64, "f32", "bwd", path="chunk", tile_variant=1)
    assert flat["kernels"] == 3 and flat["workspace_bytes"] == 4 * 16384 * 64 * 4
    p = L.lrscan_plan_complex(1, 1 << 20, 64, "bf16", "fwd", path="chunk", chunk_len=256)
    assert p["name"] == "cchunk256_v4_grouped" and p["rows_per_window"] == 256
    # enough lanes, or a short sequence: the tiled kernels
    assert L.lrscan_plan_complex(8, 2048, 2560, "bf16", "fwd")["path"] in ("seq", "window")
    assert L.lrscan_plan_complex(1, 500, 64, "f32", "fwd")["path"] in ("seq", "window")
    for bad in (dict(chunk_len=48), dict(tile_variant=3)):
        with pytest.raises(L.LrscanError):
            L.lrscan_plan_complex(1, 4096, 64, "f32", "fwd", path="chunk", **bad)


def test_complex_stream_plans(lib):
    """The complex scan streams few-lane long sequences: 32-lane tiles (fp32
    forward 256-step chunks of 16-row windows with four summary and four
    replay warps, backward 128-step chunks of 8-row windows with eight of
    each; bf16 twice the rows), and twice the real path's publication words
    (a complex map is two 64-bit words, a state one)."""
    pad = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for dt, rows, chunks in (("f32", (16, 8), (256, 128)), ("bf16", (32, 16), (512, 256))):
        for direction, r, chunk, warps in zip(("fwd", "bwd"), rows, chunks, (11, 19)):
            B, T, D = 1, 1 << 20, 64
            p = L.lrscan_plan_complex(B, T, D, dt, direction)
            assert p["path"] == "stream" and p["name"] == f"cstream_{dt}_d32" and p["exact"] == 0, p
            assert p["rows_per_window"] == r and p["subchunks"] * r == chunk and p["kernels"] == 1
            assert p["threads_per_cta"] == warps * 32 and p["smem_bytes"] <= 227 * 1024
            ng, nc = 2, T // chunk
            assert p["workspace_bytes"] == 256 + pad(ng * nc * 32 * 16) + pad(ng * nc * 32 * 8), p
            assert p["ctas"] == min(ng * nc, 152)
            q = L.lrscan_plan_complex(B, T, D, dt, direction, path="stream")
            assert q["name"] == p["name"]
    with pytest.raises(L.LrscanError):
        L.lrscan_plan_complex(1, 1 << 16, 64, "f32", "fwd", path="stream", tile_variant=2)
    with pytest.raises(L.LrscanError):
        L.lrscan_plan_complex(1, 1 << 16, 64, "f32", "fwd", path="stream", aligned=False)
    assert L.lrscan_plan_complex(1, 1 << 16, 64, "f32", "fwd", path="stream", state=True)["path"] == "stream"


def test_stream_plans(lib):
    """The persistent chunk-streaming path: four (bf16 32-lane tiles: eight)
    summary and as many replay warps, two scan warps and a ticket warp per
    CTA, one CTA per SM (no more than there are chunk tickets), 256- to
    1024-step chunks, its publication workspace (ticket, a map and a state per
    chunk and lane), and refusals where it cannot run."""
    pad = lambda x: (x + 255) // 256 * 256
    # name: {direction: (rows per window, windows per chunk, ring stages)}
    shapes = {"stream_f32_d32": {"fwd": (32, 16, 20), "bwd": (32, 8, 20)},
              "stream_f32_d32_c256": {"fwd": (32, 8, 20), "bwd": (32, 8, 20)},
              "stream_bf16_d32": {"fwd": (32, 32, 40), "bwd": (32, 16, 40)},
              "stream_bf16_d64": {"fwd": (32, 16, 24), "bwd": (32, 16, 20)},
              "stream_bf16_d64_c256": {"fwd": (32, 8, 24), "bwd": (32, 8, 20)}}
    warps = {"stream_bf16_d32": 19}
    for dt, names in (("f32", ("stream_f32_d32", "stream_f32_d32_c256")),
                      ("bf16", ("stream_bf16_d32", "stream_bf16_d64", "stream_bf16_d64_c256"))):
        assert L.lrscan_num_variants("stream", dt) == len(names)
        for v, name in enumerate(names, 1):
            for direction in ("fwd", "bwd"):
                rows, nwin, stages = shapes[name][direction]
                B, T, D = 1, 1 << 22, 64
                p = L.lrscan_plan(B, T, D, dt, direction, path="stream", tile_variant=v)
                assert p["path"] == "stream" and p["name"] == name and p["exact"] == 0, p
                assert p["rows_per_window"] == rows and p["subchunks"] == nwin and p["kernels"] == 1
                assert p["threads_per_cta"] == warps.get(name, 11) * 32 and p["stages"] == stages
                assert p["smem_bytes"] <= 227 * 1024
                dtl = p["lanes_per_cta"]
                ng, nc = B * -(-D // dtl), -(-T // (nwin * rows))
                assert p["workspace_bytes"] == 256 + pad(ng * nc * dtl * 8) + pad(ng * nc * dtl * 4)
                assert p["ctas"] == min(ng * nc, 152), p
    # a short sequence: no more CTAs than chunk tickets (2 rows x 2 lane tiles x 2 chunks)
    assert L.lrscan_plan(2, 1000, 64, "f32", "fwd", path="stream")["ctas"] == 2 * 2 * 2
    with pytest.raises(L.LrscanError):
        L.lrscan_plan(1, 1 << 16, 64, "f32", "fwd", path="stream", aligned=False)
    assert L.lrscan_plan(1, 1 << 16, 64, "f32", "fwd", path="stream", state=True)["path"] == "stream"
    with pytest.raises(L.LrscanError):
        L.lrscan_plan(1, 1 << 16, 64, "f32", "fwd", path="stream", tile_variant=3)
