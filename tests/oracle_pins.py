"""Pins that tie the CPU oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when that build disagrees with something the definition of the scan or plain
mathematics fixes: a hand-worked example, closed forms, exact rational brute
force, finite differences, adjoint identities, the IEEE rounding contract and
the padding contract.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on builds with planted mistakes and
checks that at least one of them fails for every mistake.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers --

def read_golden(name: str) -> dict[str, np.ndarray]:
    blocks: dict[str, list[list[float]]] = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                blocks[cur] = []
            else:
                blocks[cur].append([float(x) for x in line.split()])
    return {k: np.array(v, dtype=np.float64) for k, v in blocks.items()}


def _rng(seed):
    return np.random.default_rng(seed)


def _case(seed, B, T, D, lo=0.5, hi=0.999, dtype=np.float64):
    r = _rng(seed)
    a = r.uniform(lo, hi, (B, T, D)).astype(dtype)
    b = r.standard_normal((B, T, D)).astype(dtype)
    g = r.standard_normal((B, T, D)).astype(dtype)
    return a, b, g


# ------------------------------------------------------------ worked case --

def pin_golden_worked_example(o):
    """The hand-worked T=4, D=2 example, in every storage dtype, bit for bit."""
    gd = read_golden("hand_worked_T4_D2.txt")
    shape = (1, 4, 2)
    for dt in ("f64", "f32", "bf16"):
        if dt == "bf16":
            enc = lambda x: o.f32_to_bf16(x.astype(np.float32)).reshape(shape)  # noqa: E731
            dec = lambda x: o.bf16_to_f32(x).astype(np.float64)  # noqa: E731
        else:
            npdt = np.float64 if dt == "f64" else np.float32
            enc = lambda x, npdt=npdt: x.astype(npdt).reshape(shape)  # noqa: E731
            dec = lambda x: x.astype(np.float64)  # noqa: E731
        a, b, g = enc(gd["a"]), enc(gd["b"]), enc(gd["grad_out"])
        out, last = o.fwd(a, b, dt)
        assert np.array_equal(dec(out).reshape(4, 2), gd["out"]), (dt, "out")
        assert np.array_equal(last.astype(np.float64).reshape(1, 2), gd["last"]), (dt, "last")
        ga, gb = o.bwd(a, out, g, dt)
        assert np.array_equal(dec(gb).reshape(4, 2), gd["grad_b"]), (dt, "grad_b")
        assert np.array_equal(dec(ga).reshape(4, 2), gd["grad_a"]), (dt, "grad_a")


# ------------------------------------------------------------ closed forms --

def pin_unit_decay_is_prefix_sum(o):
    """a == 1: h is the running sum of b; g is the suffix sum of grad_out."""
    r = _rng(1)
    B, T, D = 2, 37, 5
    b = r.integers(-8, 9, (B, T, D)).astype(np.float64)
    g = r.integers(-8, 9, (B, T, D)).astype(np.float64)
    a = np.ones((B, T, D))
    for dt, npdt in (("f64", np.float64), ("f32", np.float32)):
        out, last = o.fwd(a.astype(npdt), b.astype(npdt), dt)
        assert np.array_equal(out.astype(np.float64), np.cumsum(b, axis=1)), dt
        assert np.array_equal(last.astype(np.float64), b.sum(axis=1)), dt
        ga, gb = o.bwd(a.astype(npdt), out, g.astype(npdt), dt)
        suffix = np.flip(np.cumsum(np.flip(g, axis=1), axis=1), axis=1)
        assert np.array_equal(gb.astype(np.float64), suffix), dt
        prev = np.concatenate([np.zeros((B, 1, D)), np.cumsum(b, axis=1)[:, :-1]], axis=1)
        assert np.array_equal(ga.astype(np.float64), suffix * prev), dt


def pin_zero_decay_is_identity(o):
    """a == 0: out = b, g = grad_out and grad_a_t = grad_out_t * b_{t-1}."""
    a0, b, g = _case(2, 3, 11, 4)
    a = np.zeros_like(a0)
    for dt, npdt in (("f64", np.float64), ("f32", np.float32)):
        bb, gg = b.astype(npdt), g.astype(npdt)
        out, last = o.fwd(a.astype(npdt), bb, dt)
        assert np.array_equal(out, bb), dt
        assert np.array_equal(last, bb[:, -1, :]), dt
        ga, gb = o.bwd(a.astype(npdt), out, gg, dt)
        assert np.array_equal(gb, gg), dt
        want = np.zeros_like(gg)
        want[:, 1:] = gg[:, 1:] * bb[:, :-1]
        assert np.array_equal(ga, want), dt


def pin_constant_decay_geometric(o):
    """a == c, b == 1: h_t = (1 - c^{t+1}) / (1 - c)."""
    T = 200
    for c in (0.3, 0.9, 0.999, -0.7):
        a = np.full((1, T, 1), c)
        b = np.ones((1, T, 1))
        out, last = o.fwd(a, b, "f64")
        t = np.arange(T)
        want = (1.0 - c ** (t + 1)) / (1.0 - c)
        np.testing.assert_allclose(out[0, :, 0], want, rtol=1e-12, atol=0)
        assert abs(last[0, 0] - want[-1]) <= 1e-12 * abs(want[-1])


def pin_constant_decay_direct_sum(o):
    """a == c, general b: h_t = sum_{s<=t} c^{t-s} b_s (direct O(T^2) sum)."""
    r = _rng(3)
    T, D, c = 64, 3, 0.93
    b = r.standard_normal((1, T, D))
    a = np.full_like(b, c)
    out, _ = o.fwd(a, b, "f64")
    for t in range(T):
        want = sum(c ** (t - s) * b[0, s] for s in range(t + 1))
        np.testing.assert_allclose(out[0, t], want, rtol=1e-12, atol=1e-13)


def pin_exact_rational_bruteforce(o):
    """Varying a, dyadic inputs: exact rational h_t = sum_s (prod_{u=s+1..t} a_u) b_s
    and exact gradients from their closed sums; the f64 oracle must match exactly."""
    r = _rng(4)
    B, T, D = 2, 7, 3
    a = r.integers(-8, 9, (B, T, D)) / 8.0
    b = r.integers(-16, 17, (B, T, D)) / 4.0
    g = r.integers(-16, 17, (B, T, D)) / 4.0
    out, last = o.fwd(a, b, "f64")
    ga, gb = o.bwd(a, out, g, "f64")
    for bb in range(B):
        for d in range(D):
            A = [Fraction(x) for x in a[bb, :, d]]
            Bv = [Fraction(x) for x in b[bb, :, d]]
            G = [Fraction(x) for x in g[bb, :, d]]

            def span(lo, hi):          # prod_{u=lo..hi} a_u (empty -> 1)
                p = Fraction(1)
                for u in range(lo, hi + 1):
                    p *= A[u]
                return p
            H = [sum(span(s + 1, t) * Bv[s] for s in range(t + 1)) for t in range(T)]
            # dL/db_s = sum_{t>=s} grad_out_t * prod_{u=s+1..t} a_u
            Gb = [sum(G[t] * span(s + 1, t) for t in range(s, T)) for s in range(T)]
            # dL/da_s = (dL/db_s) * h_{s-1}
            Ga = [Gb[s] * (H[s - 1] if s > 0 else 0) for s in range(T)]
            for t in range(T):
                assert Fraction(out[bb, t, d]) == H[t], ("h", bb, t, d)
                assert Fraction(gb[bb, t, d]) == Gb[t], ("grad_b", bb, t, d)
                assert Fraction(ga[bb, t, d]) == Ga[t], ("grad_a", bb, t, d)
            assert Fraction(last[bb, d]) == H[-1]


def pin_symbolic_small_T(o):
    """T <= 4: expand the recurrence symbolically, differentiate, evaluate."""
    import sympy as sp
    r = _rng(5)
    for T in (1, 2, 3, 4):
        av = sp.symbols(f"a0:{T}")
        bv = sp.symbols(f"b0:{T}")
        gv = sp.symbols(f"g0:{T}")
        h, hs = 0, []
        for t in range(T):
            h = av[t] * h + bv[t]
            hs.append(sp.expand(h))
        loss = sum(gv[t] * hs[t] for t in range(T))
        a = r.uniform(-1.2, 1.2, (1, T, 1))
        b = r.standard_normal((1, T, 1))
        g = r.standard_normal((1, T, 1))
        subs = {**{av[t]: a[0, t, 0] for t in range(T)},
                **{bv[t]: b[0, t, 0] for t in range(T)},
                **{gv[t]: g[0, t, 0] for t in range(T)}}
        out, _ = o.fwd(a, b, "f64")
        ga, gb = o.bwd(a, out, g, "f64")
        for t in range(T):
            assert abs(float(hs[t].subs(subs)) - out[0, t, 0]) <= 1e-12 * (1 + abs(out[0, t, 0]))
            dla = float(sp.diff(loss, av[t]).subs(subs))
            dlb = float(sp.diff(loss, bv[t]).subs(subs))
            assert abs(dla - ga[0, t, 0]) <= 1e-12 * (1 + abs(dla)), ("grad_a", T, t)
            assert abs(dlb - gb[0, t, 0]) <= 1e-12 * (1 + abs(dlb)), ("grad_b", T, t)


# ------------------------------------------------------------ derivatives --

def pin_finite_difference_jacobian(o):
    """Central differences of L = sum grad_out*h against the backward (fp64)."""
    a, b, g = _case(6, 2, 8, 3, lo=-0.95, hi=0.95)
    out, _ = o.fwd(a, b, "f64")
    ga, gb = o.bwd(a, out, g, "f64")
    eps = 1e-6

    def loss(aa, bb):
        h, _ = o.fwd(aa, bb, "f64")
        return float(np.sum(g * h))
    for idx in np.ndindex(a.shape):
        ap, am = a.copy(), a.copy()
        ap[idx] += eps
        am[idx] -= eps
        fd_a = (loss(ap, b) - loss(am, b)) / (2 * eps)
        bp, bm = b.copy(), b.copy()
        bp[idx] += eps
        bm[idx] -= eps
        fd_b = (loss(a, bp) - loss(a, bm)) / (2 * eps)
        assert abs(fd_a - ga[idx]) <= 1e-7 * (1 + abs(fd_a)), ("grad_a", idx, fd_a, ga[idx])
        assert abs(fd_b - gb[idx]) <= 1e-7 * (1 + abs(fd_b)), ("grad_b", idx, fd_b, gb[idx])


def pin_adjoint_dot_products(o):
    """<grad_out, J_b v> = <grad_b, v> and <grad_out, J_a u> = <grad_a, u>.

    The scan is linear in b, so J_b v = scan(a, v); the tangent of a in
    direction u is scan(a, u * h_{t-1})."""
    a, b, g = _case(7, 3, 50, 4)
    r = _rng(8)
    v = r.standard_normal(a.shape)
    u = r.standard_normal(a.shape)
    out, _ = o.fwd(a, b, "f64")
    ga, gb = o.bwd(a, out, g, "f64")
    jv, _ = o.fwd(a, v, "f64")
    lhs, rhs = np.sum(g * jv), np.sum(gb * v)
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(lhs))
    hprev = np.concatenate([np.zeros_like(out[:, :1]), out[:, :-1]], axis=1)
    ju, _ = o.fwd(a, u * hprev, "f64")
    lhs, rhs = np.sum(g * ju), np.sum(ga * u)
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(lhs))


def pin_linearity_in_b(o):
    a, b1, b2 = _case(9, 2, 40, 3)
    o1, _ = o.fwd(a, b1, "f64")
    o2, _ = o.fwd(a, b2, "f64")
    o3, _ = o.fwd(a, 2.5 * b1 - 0.75 * b2, "f64")
    np.testing.assert_allclose(o3, 2.5 * o1 - 0.75 * o2, rtol=1e-11, atol=1e-12)


def pin_reverse_scan_identity(o):
    """grad_b is the forward scan of reversed grad_out with decays shifted by one
    (A'_s = a_{T-s}, A'_0 = 0): bit for bit in fp32, because each reverse step
    is the same single-rounding fused step as a forward step."""
    a, _, g = _case(10, 3, 33, 5, dtype=np.float32)
    out = np.zeros_like(a)
    ga, gb = o.bwd(a, out, g, "f32")
    ra = np.zeros_like(a)
    ra[:, 1:] = np.flip(a, axis=1)[:, :-1]
    h, _ = o.fwd(ra, np.ascontiguousarray(np.flip(g, axis=1)), "f32")
    assert np.array_equal(np.flip(h, axis=1), gb)
    assert np.array_equal(ga, np.zeros_like(ga))


# ------------------------------------------------------ rounding contract --

def _f32_midpoint(x64: np.ndarray) -> np.ndarray:
    """True where a float64 value lies exactly halfway between two float32s."""
    lo = x64.astype(np.float32)
    other = np.nextafter(lo, np.where(x64 > lo, np.float32(np.inf), np.float32(-np.inf)))
    return (lo.astype(np.float64) + other.astype(np.float64)) / 2 == x64


def pin_f32_single_rounding_steps(o):
    """Every fp32 step is the correctly rounded value of a_t*h_{t-1} + b_t
    (and of a_{t+1}*g_{t+1} + grad_out_t), i.e. one fused rounding.

    The float64 evaluation of a*h (exact) + b can be off the exact value only
    where it lands exactly on an fp32 midpoint; such points are skipped."""
    a, b, g = _case(11, 2, 300, 16, lo=0.3, hi=1.05, dtype=np.float32)
    out, _ = o.fwd(a, b, "f32")
    prev = np.concatenate([np.zeros_like(out[:, :1]), out[:, :-1]], axis=1)
    exact = a.astype(np.float64) * prev.astype(np.float64) + b.astype(np.float64)
    ok = ~_f32_midpoint(exact)
    assert np.array_equal(out[ok], exact.astype(np.float32)[ok])
    ga, gb = o.bwd(a, out, g, "f32")
    nxt = np.concatenate([gb[:, 1:], np.zeros_like(gb[:, :1])], axis=1)
    anext = np.concatenate([a[:, 1:], np.zeros_like(a[:, :1])], axis=1)
    exact = anext.astype(np.float64) * nxt.astype(np.float64) + g.astype(np.float64)
    ok = ~_f32_midpoint(exact)
    assert np.array_equal(gb[ok], exact.astype(np.float32)[ok])
    prod = (gb.astype(np.float64) * prev.astype(np.float64))
    ok = ~_f32_midpoint(prod)
    assert np.array_equal(ga[ok], prod.astype(np.float32)[ok])


def pin_bf16_rne_against_torch(o):
    """fp32 -> bf16 narrowing is IEEE round-to-nearest-even, as torch's cast."""
    import torch
    r = _rng(12)
    vals = np.concatenate([
        r.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (r.standard_normal(5000) * 1e-38).astype(np.float32),      # subnormal range
        (r.standard_normal(5000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                  1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9,
                  -(1.0 + 2.0 ** -8), 2.0 ** -133, 2.0 ** -149, 65504.0],
                 dtype=np.float32),
    ])
    # exact halfway cases between neighbouring bf16 values
    base = (r.integers(0, 0x7f00, 4000).astype(np.uint32) << 16)
    half = (base | 0x8000).view(np.float32)
    vals = np.concatenate([vals, half, -half])
    mine = o.f32_to_bf16(vals)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    nan = o.f32_to_bf16(np.array([np.nan], dtype=np.float32))
    assert np.isnan(o.bf16_to_f32(nan)).all()
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    widened = o.bf16_to_f32(bits)
    ref_w = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    fin = np.isfinite(ref_w)
    assert np.array_equal(widened[fin], ref_w[fin])


def pin_bf16_storage_is_fp32_state(o):
    """bf16 storage changes only what is stored: the bf16 oracle equals the fp32
    oracle on widened inputs with its stores rounded to nearest even."""
    a, b, g = _case(13, 2, 97, 24, lo=0.8, hi=0.999, dtype=np.float32)
    a16, b16, g16 = o.f32_to_bf16(a), o.f32_to_bf16(b), o.f32_to_bf16(g)
    out16, last16 = o.fwd(a16, b16, "bf16")
    out32, last32 = o.fwd(o.bf16_to_f32(a16), o.bf16_to_f32(b16), "f32")
    assert np.array_equal(out16, o.f32_to_bf16(out32))
    assert np.array_equal(last16, last32)
    ga16, gb16 = o.bwd(a16, out16, g16, "bf16")
    ga32, gb32 = o.bwd(o.bf16_to_f32(a16), o.bf16_to_f32(out16), o.bf16_to_f32(g16), "f32")
    assert np.array_equal(ga16, o.f32_to_bf16(ga32))
    assert np.array_equal(gb16, o.f32_to_bf16(gb32))


# ------------------------------------------------- decomposition algebra --

def pin_chunked_equals_sequential(o):
    """The two-level decomposition reaches the sequential result: to rounding
    in fp64 for any chunk length (ragged last chunk included), bit for bit in
    fp32 forward when C = 1 or C >= T."""
    a, b, g = _case(14, 2, 150, 6, lo=0.6, hi=1.0)
    out, last = o.fwd(a, b, "f64")
    ga, gb = o.bwd(a, out, g, "f64")
    for C in (1, 7, 16, 64, 150, 400):
        co, cl = o.chunk_fwd(a, b, C, "f64")
        np.testing.assert_allclose(co, out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(cl, last, rtol=1e-12, atol=1e-12)
        cga, cgb = o.chunk_bwd(a, out, g, C, "f64")
        np.testing.assert_allclose(cgb, gb, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(cga, ga, rtol=1e-12, atol=1e-12)
    a32, b32 = a.astype(np.float32), b.astype(np.float32)
    out32, last32 = o.fwd(a32, b32, "f32")
    for C in (1, 150, 1000):
        co, cl = o.chunk_fwd(a32, b32, C, "f32")
        assert np.array_equal(co, out32), C
        assert np.array_equal(cl, last32), C


# ------------------------------------------------------------ padding ------

def pin_identity_padding_bit_exact(o):
    """Identity steps (a=1, b=0, grad_out=0) after a row's valid length carry
    the state bit for bit: last == out[L-1], out[t>=L] == out[L-1]; the
    gradients there are exactly zero."""
    r = _rng(15)
    B, T, D = 6, 40, 8
    a, b, g = _case(16, B, T, D, dtype=np.float32)
    L = r.integers(1, T + 1, B)
    L[0] = T
    for bb in range(B):
        a[bb, L[bb]:] = 1.0
        b[bb, L[bb]:] = 0.0
        g[bb, L[bb]:] = 0.0
    for dt in ("f32", "bf16"):
        aa, bb_, gg = (a, b, g) if dt == "f32" else (o.f32_to_bf16(a), o.f32_to_bf16(b),
                                                        o.f32_to_bf16(g))
        out, last = o.fwd(aa, bb_, dt)
        ga, gb = o.bwd(aa, out, gg, dt)
        for bb in range(B):
            n = L[bb]
            ref = out[bb, n - 1]
            assert np.array_equal(out[bb, n:], np.broadcast_to(ref, out[bb, n:].shape))
            if dt == "f32":
                assert np.array_equal(last[bb], ref)
            else:
                assert np.array_equal(o.f32_to_bf16(last[bb]), ref)
            dec = (lambda x: x) if dt == "f32" else o.bf16_to_f32
            assert not np.any(dec(gb[bb, n:]))      # +0 or -0 only
            assert not np.any(dec(ga[bb, n:]))


def pin_rows_are_independent(o):
    """Each batch row starts from h = 0: row results do not depend on the others."""
    a, b, g = _case(17, 4, 25, 3)
    out, last = o.fwd(a, b, "f64")
    ga, gb = o.bwd(a, out, g, "f64")
    for bb in range(4):
        o1, l1 = o.fwd(a[bb:bb + 1], b[bb:bb + 1], "f64")
        assert np.array_equal(o1[0], out[bb]) and np.array_equal(l1[0], last[bb])
        a1, b1 = o.bwd(a[bb:bb + 1], out[bb:bb + 1], g[bb:bb + 1], "f64")
        assert np.array_equal(a1[0], ga[bb]) and np.array_equal(b1[0], gb[bb])


def pin_empty_shapes(o):
    """Empty inputs are valid: no output, and last = h_{-1} = 0 when T == 0."""
    for shape in ((0, 5, 3), (2, 0, 3), (2, 5, 0)):
        a = np.zeros(shape)
        out, last = o.fwd(a, a, "f64")
        assert out.shape == shape and last.shape == (shape[0], shape[2])
        if shape[1] == 0:
            assert not np.any(last)
        o.bwd(a, a, a, "f64")


# ------------------------------------------- carried state and resets ----
# The state-carrying forms of the scan (initial state h0, segment resets
# where segment_pos == 0, gradient grad_last arriving at the final state,
# gradient grad_h0 of the initial state).

def _segments(seed, B, T, p=0.15, first=None):
    """int32 [B, T] segment positions with random segment starts (zeros)."""
    r = _rng(seed)
    starts = r.random((B, T)) < p
    if first is not None:
        starts[:, 0] = first
    seg = np.zeros((B, T), dtype=np.int32)
    for bb in range(B):
        pos = 0
        for t in range(T):
            pos = 0 if starts[bb, t] else pos + 1 if t > 0 else 1
            seg[bb, t] = pos
    return seg


def _state_case(seed, B, T, D, dtype):
    a, b, g = _case(seed, B, T, D, lo=0.6, hi=1.0, dtype=np.float32)
    r = _rng(seed + 1000)
    h0 = r.standard_normal((B, D)).astype(np.float32)
    gl = r.standard_normal((B, D)).astype(np.float32)
    return a, b, g, h0, gl


def _enc(o, dt, *xs):
    if dt == "bf16":
        return [o.f32_to_bf16(x) for x in xs]
    npdt = np.float64 if dt == "f64" else np.float32
    return [x.astype(npdt) for x in xs]


def _dec(o, dt, x):
    return o.bf16_to_f32(x).astype(np.float64) if dt == "bf16" else x.astype(np.float64)


def pin_state_absent_is_plain_scan(o):
    """No state, or a zero h0, no resets and a zero grad_last, gives the plain
    scan bit for bit; grad_h0 is then a_0 * g_0."""
    a, b, g, _, _ = _state_case(30, 2, 41, 5, np.float32)
    B, T, D = a.shape
    for dt in ("f32", "bf16", "f64"):
        aa, bb_, gg = _enc(o, dt, a, b, g)
        sdt = np.float64 if dt == "f64" else np.float32
        out, last = o.fwd(aa, bb_, dt)
        ga, gb = o.bwd(aa, out, gg, dt)
        for h0, seg, gl in ((None, None, None),
                            (np.zeros((B, D), sdt), np.arange(1, T + 1, dtype=np.int32)[None].repeat(B, 0),
                             np.zeros((B, D), sdt))):
            o2, l2 = o.fwd_state(aa, bb_, dt, h0=h0, segment_pos=seg)
            assert np.array_equal(o2, out) and np.array_equal(l2, last), dt
            ga2, gb2, gh0 = o.bwd_state(aa, out, gg, dt, h0=h0, segment_pos=seg, grad_last=gl)
            assert np.array_equal(ga2, ga) and np.array_equal(gb2, gb), dt
            want = _dec(o, dt, aa)[:, 0, :] * _dec(o, dt, gb)[:, 0, :] if dt != "bf16" else None
            if dt == "f64":
                assert np.array_equal(gh0, want)
            elif dt == "f32":
                assert np.array_equal(gh0, (a[:, 0, :].astype(np.float64) * gb[:, 0, :]).astype(np.float32))


def pin_state_prefill_continues_exactly(o):
    """Scanning a prefix, then the rest from the prefix's final state, equals
    one scan of the whole sequence bit for bit (forward, every dtype, with
    resets); the split backward (the suffix's grad_h0 fed to the prefix as
    grad_last) equals the whole backward to rounding."""
    a, b, g, h0, gl = _state_case(31, 3, 50, 4, np.float32)
    seg = _segments(32, 3, 50)
    for dt in ("f32", "bf16", "f64"):
        aa, bb_, gg = _enc(o, dt, a, b, g)
        sdt = np.float64 if dt == "f64" else np.float32
        hh, gll = h0.astype(sdt), gl.astype(sdt)
        out, last = o.fwd_state(aa, bb_, dt, h0=hh, segment_pos=seg)
        for T1 in (1, 17, 49):
            o1, l1 = o.fwd_state(np.ascontiguousarray(aa[:, :T1]), np.ascontiguousarray(bb_[:, :T1]), dt,
                                 h0=hh, segment_pos=np.ascontiguousarray(seg[:, :T1]))
            o2, l2 = o.fwd_state(np.ascontiguousarray(aa[:, T1:]), np.ascontiguousarray(bb_[:, T1:]), dt,
                                 h0=l1, segment_pos=np.ascontiguousarray(seg[:, T1:]))
            assert np.array_equal(np.concatenate([o1, o2], axis=1), out), (dt, T1)
            assert np.array_equal(l2, last), (dt, T1)
    a64, b64, g64 = (x.astype(np.float64) for x in (a, b, g))
    h064, gl64 = h0.astype(np.float64), gl.astype(np.float64)
    out, _ = o.fwd_state(a64, b64, "f64", h0=h064, segment_pos=seg)
    ga, gb, gh0 = o.bwd_state(a64, out, g64, "f64", h0=h064, segment_pos=seg, grad_last=gl64)
    for T1 in (1, 17, 49):
        sl1, sl2 = (slice(None), slice(None, T1)), (slice(None), slice(T1, None))
        c = np.ascontiguousarray
        _, l1 = o.fwd_state(c(a64[sl1]), c(b64[sl1]), "f64", h0=h064, segment_pos=c(seg[sl1]))
        ga2, gb2, gmid = o.bwd_state(c(a64[sl2]), c(out[sl2]), c(g64[sl2]), "f64", h0=l1,
                                     segment_pos=c(seg[sl2]), grad_last=gl64)
        ga1, gb1, g0 = o.bwd_state(c(a64[sl1]), c(out[sl1]), c(g64[sl1]), "f64", h0=h064,
                                   segment_pos=c(seg[sl1]), grad_last=gmid)
        np.testing.assert_allclose(np.concatenate([gb1, gb2], axis=1), gb, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(np.concatenate([ga1, ga2], axis=1), ga, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g0, gh0, rtol=1e-12, atol=1e-12)


def pin_state_segments_are_independent_sequences(o):
    """With resets, every segment is the plain scan of its own steps started
    from zero (the first one from h0 unless step 0 resets); in the backward the
    segments are independent too, grad_a is zero at a segment start, only the
    last segment sees grad_last and only the first one feeds grad_h0."""
    B, T, D = 4, 60, 3
    a, b, g, h0, gl = _state_case(33, B, T, D, np.float32)
    seg = _segments(34, B, T, p=0.1)
    seg[0, 0] = 0           # row 0 starts with a reset: h0 is ignored
    seg[1, 0] = 5           # row 1 continues h0
    for dt in ("f32", "bf16", "f64"):
        aa, bb_, gg = _enc(o, dt, a, b, g)
        sdt = np.float64 if dt == "f64" else np.float32
        hh, gll = h0.astype(sdt), gl.astype(sdt)
        out, last = o.fwd_state(aa, bb_, dt, h0=hh, segment_pos=seg)
        ga, gb, gh0 = o.bwd_state(aa, out, gg, dt, h0=hh, segment_pos=seg, grad_last=gll)
        for r in range(B):
            starts = [t for t in range(T) if seg[r, t] == 0]
            bounds = sorted(set([0] + starts + [T]))
            for k in range(len(bounds) - 1):
                lo, hi = bounds[k], bounds[k + 1]
                first = lo == 0 and seg[r, 0] != 0
                c = np.ascontiguousarray
                sa, sb, sg = c(aa[r:r + 1, lo:hi]), c(bb_[r:r + 1, lo:hi]), c(gg[r:r + 1, lo:hi])
                h_in = hh[r:r + 1] if first else None
                so, sl = o.fwd_state(sa, sb, dt, h0=h_in)
                assert np.array_equal(so, out[r:r + 1, lo:hi]), (dt, r, lo)
                if hi == T:
                    assert np.array_equal(sl, last[r:r + 1]), (dt, r)
                sga, sgb, sgh = o.bwd_state(sa, so, sg, dt, h0=h_in,
                                            grad_last=gll[r:r + 1] if hi == T else None)
                assert np.array_equal(sgb, gb[r:r + 1, lo:hi]), (dt, r, lo)
                # isolated segment: grad_a at its first step is g * 0 (+-0)
                assert np.array_equal(_dec(o, dt, sga), _dec(o, dt, ga[r:r + 1, lo:hi])), (dt, r, lo)
                if lo > 0 or not first:
                    assert _dec(o, dt, ga[r:r + 1, lo]).tolist() == [[0.0] * D]
                    assert not np.signbit(_dec(o, dt, ga[r:r + 1, lo])).any(), "+0 at a reset"
                if first:
                    assert np.array_equal(sgh, gh0[r:r + 1]), (dt, r)
            if seg[r, 0] == 0:
                assert np.array_equal(gh0[r], np.zeros(D)), (dt, r)


def pin_state_initial_state_closed_form(o):
    """a == c, b == 0: h_t = c^{t+1} h0, and with L = sum_t g_t h_t + gl h_{T-1}
    the initial-state gradient is sum_t g_t c^{t+1} + gl c^T; a reset at step r
    cuts both sums at r."""
    T = 40
    r = _rng(35)
    g = r.standard_normal((1, T, 1))
    for c in (0.9, -0.8, 1.0):
        a = np.full((1, T, 1), c)
        b = np.zeros((1, T, 1))
        h0 = np.array([[1.75]])
        gl = np.array([[-0.5]])
        out, last = o.fwd_state(a, b, "f64", h0=h0)
        t = np.arange(T)
        np.testing.assert_allclose(out[0, :, 0], c ** (t + 1) * 1.75, rtol=1e-12)
        np.testing.assert_allclose(last[0, 0], c ** T * 1.75, rtol=1e-12)
        _, _, gh0 = o.bwd_state(a, out, g, "f64", h0=h0, grad_last=gl)
        want = np.sum(g[0, :, 0] * c ** (t + 1)) - 0.5 * c ** T
        assert abs(gh0[0, 0] - want) <= 1e-12 * (1 + abs(want))
        for cut in (0, 13):
            seg = np.ones((1, T), dtype=np.int32)
            seg[0, cut] = 0
            out, last = o.fwd_state(a, b, "f64", h0=h0, segment_pos=seg)
            want_h = np.where(t < cut, c ** (t + 1) * 1.75, 0.0)
            np.testing.assert_allclose(out[0, :, 0], want_h, rtol=1e-12, atol=0)
            _, _, gh0 = o.bwd_state(a, out, g, "f64", h0=h0, segment_pos=seg, grad_last=gl)
            want = np.sum(g[0, :cut, 0] * c ** (t[:cut] + 1))
            assert abs(gh0[0, 0] - want) <= 1e-12 * (1 + abs(want)), (c, cut)


def pin_state_finite_difference_jacobian(o):
    """Central differences of L = sum grad_out*h + sum grad_last*h_{T-1} with
    an initial state and resets, against grad_a, grad_b and grad_h0 (fp64)."""
    B, T, D = 2, 9, 2
    a, b, g = _case(36, B, T, D, lo=-0.95, hi=0.95)
    r = _rng(37)
    h0 = r.standard_normal((B, D))
    gl = r.standard_normal((B, D))
    seg = np.ones((B, T), dtype=np.int32)
    seg[0, 4] = 0
    seg[1, 0] = 0
    seg[1, 6] = 0
    out, _ = o.fwd_state(a, b, "f64", h0=h0, segment_pos=seg)
    ga, gb, gh0 = o.bwd_state(a, out, g, "f64", h0=h0, segment_pos=seg, grad_last=gl)
    eps = 1e-6

    def loss(aa, bb, hh):
        h, last = o.fwd_state(aa, bb, "f64", h0=hh, segment_pos=seg)
        return float(np.sum(g * h) + np.sum(gl * last))
    for idx in np.ndindex(a.shape):
        for arr, grad, name in ((a, ga, "grad_a"), (b, gb, "grad_b")):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = (p, b, h0) if name == "grad_a" else (a, p, h0)
            args_m = (m, b, h0) if name == "grad_a" else (a, m, h0)
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * (1 + abs(fd)), (name, idx, fd, grad[idx])
    for idx in np.ndindex(h0.shape):
        p, m = h0.copy(), h0.copy()
        p[idx] += eps
        m[idx] -= eps
        fd = (loss(a, b, p) - loss(a, b, m)) / (2 * eps)
        assert abs(fd - gh0[idx]) <= 1e-7 * (1 + abs(fd)), ("grad_h0", idx, fd, gh0[idx])


def pin_state_symbolic_small_T(o):
    """T <= 3 with a symbolic initial state and every reset pattern: expand,
    differentiate, evaluate."""
    import sympy as sp
    import itertools
    r = _rng(38)
    for T in (1, 2, 3):
        av, bv, gv = sp.symbols(f"a0:{T}"), sp.symbols(f"b0:{T}"), sp.symbols(f"g0:{T}")
        h0s, gls = sp.symbols("h0 gl")
        for pattern in itertools.product((0, 1), repeat=T):
            h, hs = h0s, []
            for t in range(T):
                h = (0 if pattern[t] else av[t]) * h + bv[t]
                hs.append(sp.expand(h))
            loss = sum(gv[t] * hs[t] for t in range(T)) + gls * hs[-1]
            a = r.uniform(-1.2, 1.2, (1, T, 1))
            b = r.standard_normal((1, T, 1))
            g = r.standard_normal((1, T, 1))
            h0 = r.standard_normal((1, 1))
            gl = r.standard_normal((1, 1))
            seg = np.array([[0 if p else 7 for p in pattern]], dtype=np.int32)
            subs = {**{av[t]: a[0, t, 0] for t in range(T)}, **{bv[t]: b[0, t, 0] for t in range(T)},
                    **{gv[t]: g[0, t, 0] for t in range(T)}, h0s: h0[0, 0], gls: gl[0, 0]}
            out, _ = o.fwd_state(a, b, "f64", h0=h0, segment_pos=seg)
            ga, gb, gh0 = o.bwd_state(a, out, g, "f64", h0=h0, segment_pos=seg, grad_last=gl)
            close = lambda x, y: abs(x - y) <= 1e-12 * (1 + abs(x))  # noqa: E731
            for t in range(T):
                assert close(float(hs[t].subs(subs)), out[0, t, 0]), ("h", T, pattern, t)
                assert close(float(sp.diff(loss, av[t]).subs(subs)), ga[0, t, 0]), ("grad_a", T, pattern, t)
                assert close(float(sp.diff(loss, bv[t]).subs(subs)), gb[0, t, 0]), ("grad_b", T, pattern, t)
            assert close(float(sp.diff(loss, h0s).subs(subs)), gh0[0, 0]), ("grad_h0", T, pattern)


def pin_state_empty_sequence(o):
    """T == 0: the final state is h0 and the initial-state gradient is grad_last."""
    a = np.zeros((2, 0, 3))
    h0 = np.arange(6.0).reshape(2, 3)
    gl = -np.arange(6.0).reshape(2, 3)
    _, last = o.fwd_state(a, a, "f64", h0=h0)
    assert np.array_equal(last, h0)
    _, _, gh0 = o.bwd_state(a, a, a, "f64", h0=h0, grad_last=gl)
    assert np.array_equal(gh0, gl)
    _, _, gh0 = o.bwd_state(a, a, a, "f64")
    assert not np.any(gh0)


# ------------------------------------------------------- complex scan ----
# Complex a, b on separate re/im planes; the backward's adjoint carries
# conj(a_{t+1}) and grad_a = g * conj(h_{t-1}) (loss sum Re(conj(go) h)).

def _ccase(seed, B, T, D, rho=(0.5, 0.999), dtype=np.float64):
    r = _rng(seed)
    rad = r.uniform(*rho, (B, T, D))
    ang = r.uniform(-np.pi, np.pi, (B, T, D))
    ar, ai = (rad * np.cos(ang)).astype(dtype), (rad * np.sin(ang)).astype(dtype)
    br, bi, gr, gi = (r.standard_normal((B, T, D)).astype(dtype) for _ in range(4))
    return ar, ai, br, bi, gr, gi


def pin_complex_matches_numpy_complex(o):
    """Forward against numpy complex128 arithmetic; backward against the
    conjugate-transition adjoint evaluated in numpy complex128 (fp64)."""
    ar, ai, br, bi, gr, gi = _ccase(40, 2, 70, 3)
    out_r, out_i, last_r, last_i = o.cfwd(ar, ai, br, bi, "f64")
    a, b, go = ar + 1j * ai, br + 1j * bi, gr + 1j * gi
    h = np.zeros(a[:, 0].shape, complex)
    hs = []
    for t in range(a.shape[1]):
        h = a[:, t] * h + b[:, t]
        hs.append(h)
    hs = np.stack(hs, 1)
    np.testing.assert_allclose(out_r, hs.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out_i, hs.imag, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(last_r + 1j * last_i, hs[:, -1], rtol=1e-12, atol=1e-12)
    g_ar, g_ai, g_br, g_bi = o.cbwd(ar, ai, out_r, out_i, gr, gi, "f64")
    g = np.zeros_like(h)
    gs = np.zeros_like(hs)
    for t in range(a.shape[1] - 1, -1, -1):
        g = go[:, t] + (np.conj(a[:, t + 1]) * g if t + 1 < a.shape[1] else 0)
        gs[:, t] = g
    prev = np.concatenate([np.zeros_like(hs[:, :1]), hs[:, :-1]], axis=1)
    ga = gs * np.conj(prev)
    np.testing.assert_allclose(g_br + 1j * g_bi, gs, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g_ar + 1j * g_ai, ga, rtol=1e-12, atol=1e-12)


def pin_complex_constant_decay_geometric(o):
    """a == c (complex), b == 1: h_t = (1 - c^{t+1}) / (1 - c)."""
    T = 150
    for c in (0.9 * np.exp(0.3j), 0.999 * np.exp(-2.0j), -0.5 + 0.5j):
        ar = np.full((1, T, 1), c.real)
        ai = np.full((1, T, 1), c.imag)
        out_r, out_i, _, _ = o.cfwd(ar, ai, np.ones_like(ar), np.zeros_like(ar), "f64")
        want = (1 - c ** (np.arange(T) + 1)) / (1 - c)
        np.testing.assert_allclose(out_r[0, :, 0] + 1j * out_i[0, :, 0], want, rtol=1e-11, atol=1e-12)


def pin_complex_exact_rational(o):
    """Dyadic complex inputs: the fp64 forward and backward are exact, so they
    equal the rational evaluation of the recurrences term by term."""
    r = _rng(41)
    B, T, D = 1, 6, 2
    q = lambda n, s: r.integers(-n, n + 1, (B, T, D)) / s  # noqa: E731
    ar, ai, br, bi, gr, gi = q(4, 8.0), q(4, 8.0), q(8, 4.0), q(8, 4.0), q(8, 4.0), q(8, 4.0)
    out_r, out_i, _, _ = o.cfwd(ar, ai, br, bi, "f64")
    g_ar, g_ai, g_br, g_bi = o.cbwd(ar, ai, out_r, out_i, gr, gi, "f64")
    F = Fraction
    for d in range(D):
        A = [(F(ar[0, t, d]), F(ai[0, t, d])) for t in range(T)]
        Bv = [(F(br[0, t, d]), F(bi[0, t, d])) for t in range(T)]
        G = [(F(gr[0, t, d]), F(gi[0, t, d])) for t in range(T)]
        mul = lambda x, y: (x[0] * y[0] - x[1] * y[1], x[0] * y[1] + x[1] * y[0])  # noqa: E731
        conj = lambda x: (x[0], -x[1])  # noqa: E731
        add = lambda x, y: (x[0] + y[0], x[1] + y[1])  # noqa: E731
        H, h = [], (F(0), F(0))
        for t in range(T):
            h = add(mul(A[t], h), Bv[t])
            H.append(h)
        Gs, g = [None] * T, (F(0), F(0))
        for t in range(T - 1, -1, -1):
            g = add(G[t], mul(conj(A[t + 1]), g)) if t + 1 < T else G[t]
            Gs[t] = g
        for t in range(T):
            assert (F(out_r[0, t, d]), F(out_i[0, t, d])) == H[t], ("h", t, d)
            assert (F(g_br[0, t, d]), F(g_bi[0, t, d])) == Gs[t], ("grad_b", t, d)
            prev = conj(H[t - 1]) if t > 0 else (F(0), F(0))
            assert (F(g_ar[0, t, d]), F(g_ai[0, t, d])) == mul(Gs[t], prev), ("grad_a", t, d)


def pin_complex_finite_difference_jacobian(o):
    """Central differences of L = sum(go_r*h_r + go_i*h_i) against all four
    gradient planes (fp64)."""
    planes = list(_ccase(42, 1, 7, 2, rho=(0.4, 0.95)))
    gr, gi = planes[4], planes[5]
    out_r, out_i, _, _ = o.cfwd(*planes[:4], "f64")
    grads = o.cbwd(planes[0], planes[1], out_r, out_i, gr, gi, "f64")
    eps = 1e-6

    def loss(ps):
        hr, hi, _, _ = o.cfwd(*ps, "f64")
        return float(np.sum(gr * hr + gi * hi))
    for k in range(4):
        for idx in np.ndindex(planes[0].shape):
            p, m = [x.copy() for x in planes[:4]], [x.copy() for x in planes[:4]]
            p[k][idx] += eps
            m[k][idx] -= eps
            fd = (loss(p) - loss(m)) / (2 * eps)
            assert abs(fd - grads[k][idx]) <= 1e-7 * (1 + abs(fd)), (k, idx, fd, grads[k][idx])


def pin_complex_reduces_to_real_scans(o):
    """ai == 0: the real and imaginary planes are two independent real scans
    with the same decays (bit for bit in fp32 forward and for grad_b), and
    grad_ar is the sum of the two real grad_a."""
    ar, _, br, bi, gr, gi = _ccase(43, 2, 40, 5, dtype=np.float32)
    ar = np.abs(ar)
    z = np.zeros_like(ar)
    out_r, out_i, last_r, last_i = o.cfwd(ar, z, br, bi, "f32")
    rr, lr = o.fwd(ar, br, "f32")
    ri, li = o.fwd(ar, bi, "f32")
    assert np.array_equal(out_r, rr) and np.array_equal(out_i, ri)
    assert np.array_equal(last_r, lr) and np.array_equal(last_i, li)
    g_ar, g_ai, g_br, g_bi = o.cbwd(ar, z, out_r, out_i, gr, gi, "f32")
    gar, gbr = o.bwd(ar, rr, gr, "f32")
    gai, gbi = o.bwd(ar, ri, gi, "f32")
    assert np.array_equal(g_br, gbr) and np.array_equal(g_bi, gbi)
    np.testing.assert_allclose(g_ar, gar.astype(np.float64) + gai, rtol=1e-6, atol=1e-6)
    a64 = [x.astype(np.float64) for x in (ar, z, br, bi, gr, gi)]
    o_r, o_i, _, _ = o.cfwd(*a64[:4], "f64")
    _, g_ai64, _, _ = o.cbwd(a64[0], a64[1], o_r, o_i, a64[4], a64[5], "f64")
    # grad_ai = g_i h_r - g_r h_i of the two real problems
    _, gbr64 = o.bwd(a64[0], o_r, a64[4], "f64")
    _, gbi64 = o.bwd(a64[0], o_i, a64[5], "f64")
    pr = np.concatenate([np.zeros_like(o_r[:, :1]), o_r[:, :-1]], axis=1)
    pi = np.concatenate([np.zeros_like(o_i[:, :1]), o_i[:, :-1]], axis=1)
    np.testing.assert_allclose(g_ai64, gbi64 * pr - gbr64 * pi, rtol=1e-12, atol=1e-12)


def pin_complex_bf16_storage_is_fp32_state(o):
    """bf16 storage only rounds what is stored: the bf16 complex oracle equals
    the fp32 one on widened inputs with its stores rounded to nearest even."""
    planes = [o.f32_to_bf16(x) for x in _ccase(44, 2, 60, 8, dtype=np.float32)]
    w = [o.bf16_to_f32(x) for x in planes]
    r16 = o.cfwd(*planes[:4], "bf16")
    r32 = o.cfwd(*w[:4], "f32")
    for x16, x32 in zip(r16[:2], r32[:2]):
        assert np.array_equal(x16, o.f32_to_bf16(x32))
    assert np.array_equal(r16[2], r32[2]) and np.array_equal(r16[3], r32[3])
    g16 = o.cbwd(planes[0], planes[1], r16[0], r16[1], planes[4], planes[5], "bf16")
    g32 = o.cbwd(w[0], w[1], o.bf16_to_f32(r16[0]), o.bf16_to_f32(r16[1]), w[4], w[5], "f32")
    for x16, x32 in zip(g16, g32):
        assert np.array_equal(x16, o.f32_to_bf16(x32))


def pin_complex_identity_padding(o):
    """a = 1 + 0i, b = 0 after a row's valid length carries the state bit for bit."""
    ar, ai, br, bi, gr, gi = _ccase(45, 3, 30, 4, dtype=np.float32)
    L = [30, 11, 1]
    for bb, n in enumerate(L):
        ar[bb, n:], ai[bb, n:], br[bb, n:], bi[bb, n:] = 1.0, 0.0, 0.0, 0.0
        gr[bb, n:], gi[bb, n:] = 0.0, 0.0
    out_r, out_i, last_r, last_i = o.cfwd(ar, ai, br, bi, "f32")
    g = o.cbwd(ar, ai, out_r, out_i, gr, gi, "f32")
    for bb, n in enumerate(L):
        assert (out_r[bb, n:] == out_r[bb, n - 1]).all() and (out_i[bb, n:] == out_i[bb, n - 1]).all()
        assert np.array_equal(last_r[bb], out_r[bb, n - 1]) and np.array_equal(last_i[bb], out_i[bb, n - 1])
        for x in g:
            assert not np.any(x[bb, n:])


# ---------------------------------------------- generated (factorized) decay --
# a_{t,d} = exp(-exp(nu_log_d) * exp(eta_t)), rebuilt in the kernel from one
# value per token and one per lane; gradients flow to b, eta and nu_log.

def _gcase(seed, B, T, D, dtype=np.float64):
    r = _rng(seed)
    eta = r.uniform(-3.0, 1.0, (B, T)).astype(dtype)
    nu_log = r.uniform(-3.0, 0.5, (D,)).astype(dtype)
    b = r.standard_normal((B, T, D)).astype(dtype)
    g = r.standard_normal((B, T, D)).astype(dtype)
    return eta, nu_log, b, g


def _decay(eta, nu_log):
    return np.exp(-np.exp(nu_log)[None, None, :] * np.exp(eta)[:, :, None])


def pin_gated_equals_materialized_decay(o):
    """The generated-decay scan equals the plain scan of the materialized
    decays (numpy), and its parameter gradients equal the chain rule applied
    to the plain backward's grad_a: dL/dlog a = grad_a * a, d log a / d eta =
    d log a / d nu_log = log a."""
    eta, nu_log, b, g = _gcase(50, 2, 60, 5)
    a = _decay(eta, nu_log)
    out, last = o.gated_fwd(eta, nu_log, b, "f64")
    ref, ref_last = o.fwd(a, b, "f64")
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(last, ref_last, rtol=1e-12, atol=1e-13)
    gb, geta, gnu = o.gated_bwd(eta, nu_log, out, g, "f64")
    ga, rgb = o.bwd(a, out, g, "f64")
    np.testing.assert_allclose(gb, rgb, rtol=1e-12, atol=1e-13)
    q = ga * a * np.log(a)
    np.testing.assert_allclose(geta, q.sum(axis=2), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gnu, q.sum(axis=(0, 1)), rtol=1e-10, atol=1e-12)


def pin_gated_finite_difference(o):
    """Central differences of L = sum grad_out*h with respect to eta, nu_log
    and b against the backward (fp64)."""
    eta, nu_log, b, g = _gcase(51, 2, 7, 3)
    out, _ = o.gated_fwd(eta, nu_log, b, "f64")
    gb, geta, gnu = o.gated_bwd(eta, nu_log, out, g, "f64")
    eps = 1e-6

    def loss(e, n, bb):
        h, _ = o.gated_fwd(e, n, bb, "f64")
        return float(np.sum(g * h))
    for arr, grad, k in ((eta, geta, 0), (nu_log, gnu, 1), (b, gb, 2)):
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [eta, nu_log, b]
            args_m = [eta, nu_log, b]
            args_p[k], args_m[k] = p, m
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * (1 + abs(fd)), (k, idx, fd, grad[idx])


def pin_gated_zero_rate_is_prefix_sum(o):
    """nu = 0 (nu_log = -inf): every decay is exactly 1, h is the running sum
    of b, and the rate gradients vanish exactly."""
    r = _rng(52)
    B, T, D = 2, 30, 4
    b = r.integers(-8, 9, (B, T, D)).astype(np.float32)
    g = r.integers(-8, 9, (B, T, D)).astype(np.float32)
    eta = r.uniform(-2, 2, (B, T)).astype(np.float32)
    nu_log = np.full((D,), -np.inf, dtype=np.float32)
    out, last = o.gated_fwd(eta, nu_log, b, "f32")
    assert np.array_equal(out, np.cumsum(b, axis=1))
    gb, geta, gnu = o.gated_bwd(eta, nu_log, out, g, "f32")
    assert np.array_equal(gb, np.flip(np.cumsum(np.flip(g, axis=1), axis=1), axis=1))
    assert not np.any(geta) and not np.any(gnu)


def pin_gated_bf16_storage_is_fp32_state(o):
    """bf16 storage only rounds the stored tensors: the bf16 variant equals
    the fp32 one on widened inputs with its stores rounded."""
    eta, nu_log, b, g = _gcase(53, 2, 50, 8, dtype=np.float32)
    b16, g16 = o.f32_to_bf16(b), o.f32_to_bf16(g)
    out16, last16 = o.gated_fwd(eta, nu_log, b16, "bf16")
    out32, last32 = o.gated_fwd(eta, nu_log, o.bf16_to_f32(b16), "f32")
    assert np.array_equal(out16, o.f32_to_bf16(out32)) and np.array_equal(last16, last32)
    r16 = o.gated_bwd(eta, nu_log, out16, g16, "bf16")
    r32 = o.gated_bwd(eta, nu_log, o.bf16_to_f32(out16), o.bf16_to_f32(g16), "f32")
    assert np.array_equal(r16[0], o.f32_to_bf16(r32[0]))
    assert np.array_equal(r16[1], r32[1]) and np.array_equal(r16[2], r32[2])


# ------------------------------------------------ complex scan with state --
def _cstate_case(seed, B, T, D, dtype=np.float64):
    ar, ai, br, bi, gr, gi = _ccase(seed, B, T, D, dtype=dtype)
    r = _rng(seed + 2000)
    h0 = tuple(r.standard_normal((B, D)).astype(dtype) for _ in range(2))
    gl = tuple(r.standard_normal((B, D)).astype(dtype) for _ in range(2))
    return ar, ai, br, bi, gr, gi, h0, gl


def pin_cstate_absent_is_plain_complex(o):
    """No state, or a zero h0, no resets and a zero grad_last, gives the plain
    complex scan bit for bit (every dtype); grad_h0 is then conj(a_0) * g_0."""
    ar, ai, br, bi, gr, gi, _, _ = _cstate_case(60, 2, 33, 4, dtype=np.float32)
    B, T, D = ar.shape
    for dt in ("f32", "bf16", "f64"):
        planes = _enc(o, dt, ar, ai, br, bi, gr, gi)
        sdt = np.float64 if dt == "f64" else np.float32
        ref = o.cfwd(*planes[:4], dt)
        gref = o.cbwd(planes[0], planes[1], ref[0], ref[1], planes[4], planes[5], dt)
        zero = (np.zeros((B, D), sdt), np.zeros((B, D), sdt))
        noreset = np.arange(1, T + 1, dtype=np.int32)[None].repeat(B, 0)
        for h0, seg, gl in ((None, None, None), (zero, noreset, zero)):
            got = o.cfwd_state(*planes[:4], dt, h0=h0, segment_pos=seg)
            for x, y in zip(got, ref):
                assert np.array_equal(x, y), dt
            g = o.cbwd_state(planes[0], planes[1], ref[0], ref[1], planes[4], planes[5], dt, h0=h0,
                             segment_pos=seg, grad_last=gl)
            for x, y in zip(g[:4], gref):
                assert np.array_equal(x, y), dt
            if dt == "f64":
                a0 = planes[0][:, 0] + 1j * planes[1][:, 0]
                g0 = g[2][:, 0] + 1j * g[3][:, 0]
                want = np.conj(a0) * g0
                np.testing.assert_allclose(g[4], want.real, rtol=1e-13, atol=1e-13)
                np.testing.assert_allclose(g[5], want.imag, rtol=1e-13, atol=1e-13)


def pin_cstate_reduces_to_real_state_scan(o):
    """Zero imaginary parts everywhere (decays, inputs, h0, grad_last,
    grad_out): the real planes are the real state-carrying scan bit for bit in
    fp32, resets included, and every imaginary plane stays zero."""
    ar, _, br, _, gr, _, h0, gl = _cstate_case(61, 3, 45, 5, dtype=np.float32)
    ar = np.abs(ar)
    z = np.zeros_like(ar)
    zs = np.zeros_like(h0[0])
    seg = _segments(62, 3, 45, p=0.1)
    seg[0, 0] = 0
    out_r, out_i, last_r, last_i = o.cfwd_state(ar, z, br, z, "f32", h0=(h0[0], zs), segment_pos=seg)
    rr, lr = o.fwd_state(ar, br, "f32", h0=h0[0], segment_pos=seg)
    assert np.array_equal(out_r, rr) and np.array_equal(last_r, lr)
    assert not out_i.any() and not last_i.any()
    g = o.cbwd_state(ar, z, out_r, out_i, gr, z, "f32", h0=(h0[0], zs), segment_pos=seg, grad_last=(gl[0], zs))
    ga, gb, gh0 = o.bwd_state(ar, rr, gr, "f32", h0=h0[0], segment_pos=seg, grad_last=gl[0])
    assert np.array_equal(g[2], gb) and np.array_equal(g[0], ga) and np.array_equal(g[4], gh0)
    assert not g[1].any() and not g[3].any() and not g[5].any()


def pin_cstate_matches_numpy_complex(o):
    """fp64 against numpy complex128: the forward from h0 with a' = 0 at
    segment starts, and the adjoint with grad_last entering after the last
    step, conj(a'_{t+1}) transitions, grad_a = g conj(h_{t-1}) (0 at a reset)
    and grad_h0 = conj(a'_0) g_0."""
    B, T, D = 3, 57, 4
    ar, ai, br, bi, gr, gi, h0, gl = _cstate_case(63, B, T, D)
    seg = _segments(64, B, T, p=0.12)
    seg[2, 0] = 0
    a, b, go = ar + 1j * ai, br + 1j * bi, gr + 1j * gi
    rs = seg == 0
    ap = np.where(rs[..., None], 0, a)
    h = h0[0] + 1j * h0[1]
    hs = []
    for t in range(T):
        h = ap[:, t] * h + b[:, t]
        hs.append(h)
    hs = np.stack(hs, 1)
    out_r, out_i, last_r, last_i = o.cfwd_state(ar, ai, br, bi, "f64", h0=h0, segment_pos=seg)
    np.testing.assert_allclose(out_r + 1j * out_i, hs, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(last_r + 1j * last_i, hs[:, -1], rtol=1e-12, atol=1e-12)
    g = gl[0] + 1j * gl[1]
    gs = [None] * T
    nxt = np.ones((B, D), complex)  # a'_T = 1: grad_last enters the last step
    for t in range(T - 1, -1, -1):
        g = go[:, t] + np.conj(nxt) * g
        gs[t] = g
        nxt = ap[:, t]
    gs = np.stack(gs, 1)
    prev = np.concatenate([(h0[0] + 1j * h0[1])[:, None], hs[:, :-1]], axis=1)
    ga = np.where(rs[..., None], 0, gs * np.conj(prev))
    gh0 = np.conj(ap[:, 0]) * gs[:, 0]
    got = o.cbwd_state(ar, ai, out_r, out_i, gr, gi, "f64", h0=h0, segment_pos=seg, grad_last=gl)
    np.testing.assert_allclose(got[2] + 1j * got[3], gs, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[0] + 1j * got[1], ga, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[4] + 1j * got[5], gh0, rtol=1e-12, atol=1e-12)
    assert not got[0][rs].any() and not got[1][rs].any()


def pin_cstate_finite_difference(o):
    """Central differences of L = sum Re(conj(grad_out) h) + Re(conj(grad_last)
    last) on a tiny fp64 case with one reset: dL/dRe(h0) + i dL/dIm(h0) is
    grad_h0, and the same for a few decay and input entries."""
    B, T, D = 1, 6, 2
    ar, ai, br, bi, gr, gi, h0, gl = _cstate_case(65, B, T, D)
    seg = np.array([[1, 2, 0, 1, 2, 3]], dtype=np.int32)

    def loss(ar_, ai_, br_, bi_, h0_):
        o_r, o_i, l_r, l_i = o.cfwd_state(ar_, ai_, br_, bi_, "f64", h0=h0_, segment_pos=seg)
        return float((gr * o_r + gi * o_i).sum() + (gl[0] * l_r + gl[1] * l_i).sum())

    o_r, o_i, _, _ = o.cfwd_state(ar, ai, br, bi, "f64", h0=h0, segment_pos=seg)
    g_ar, g_ai, g_br, g_bi, gh_r, gh_i = o.cbwd_state(ar, ai, o_r, o_i, gr, gi, "f64", h0=h0, segment_pos=seg,
                                                      grad_last=gl)
    eps = 1e-6
    for k in range(2):
        for d in range(D):
            hp = [h0[0].copy(), h0[1].copy()]
            hm = [h0[0].copy(), h0[1].copy()]
            hp[k][0, d] += eps
            hm[k][0, d] -= eps
            fd = (loss(ar, ai, br, bi, tuple(hp)) - loss(ar, ai, br, bi, tuple(hm))) / (2 * eps)
            want = (gh_r if k == 0 else gh_i)[0, d]
            assert abs(fd - want) <= 1e-6 * (1 + abs(want)), (k, d, fd, want)
    for (t, d) in ((0, 0), (2, 1), (3, 0), (5, 1)):
        for name, arr, grad in (("ar", 0, g_ar), ("ai", 1, g_ai), ("br", 2, g_br), ("bi", 3, g_bi)):
            xs = [ar.copy(), ai.copy(), br.copy(), bi.copy()]
            xp = [x.copy() for x in xs]
            xm = [x.copy() for x in xs]
            xp[arr][0, t, d] += eps
            xm[arr][0, t, d] -= eps
            fd = (loss(*xp, h0) - loss(*xm, h0)) / (2 * eps)
            want = grad[0, t, d]
            assert abs(fd - want) <= 1e-6 * (1 + abs(want)), (name, t, d, fd, want)


def pin_cstate_empty_sequence_and_first_step_reset(o):
    """T == 0: the final state is h0 and the initial-state gradient is
    grad_last (zeros without them).  A reset at step 0 ignores h0 entirely:
    the outputs equal the scan without state and grad_h0 is exactly +0."""
    e = np.zeros((2, 0, 3))
    h0 = (np.arange(6.0).reshape(2, 3), -np.arange(6.0).reshape(2, 3) - 1)
    gl = (np.full((2, 3), 0.5), np.full((2, 3), -2.0))
    _, _, lr, li = o.cfwd_state(e, e, e, e, "f64", h0=h0)
    assert np.array_equal(lr, h0[0]) and np.array_equal(li, h0[1])
    g = o.cbwd_state(e, e, e, e, e, e, "f64", h0=h0, grad_last=gl)
    assert np.array_equal(g[4], gl[0]) and np.array_equal(g[5], gl[1])
    g = o.cbwd_state(e, e, e, e, e, e, "f64")
    assert not g[4].any() and not g[5].any()
    ar, ai, br, bi, gr, gi, h0, _ = _cstate_case(68, 2, 20, 3)
    seg = np.arange(20, dtype=np.int32)[None].repeat(2, 0)  # position 0 at step 0: a reset
    ref = o.cfwd(ar, ai, br, bi, "f64")
    got = o.cfwd_state(ar, ai, br, bi, "f64", h0=h0, segment_pos=seg)
    for x, y in zip(got, ref):
        assert np.array_equal(x, y)
    g = o.cbwd_state(ar, ai, ref[0], ref[1], gr, gi, "f64", h0=h0, segment_pos=seg)
    gref = o.cbwd(ar, ai, ref[0], ref[1], gr, gi, "f64")
    for x, y in zip(g[2:4], gref[2:4]):
        assert np.array_equal(x, y)
    assert not g[0][:, 0].any() and not g[1][:, 0].any()
    assert not g[4].any() and not g[5].any() and not np.signbit(g[4]).any()


def pin_cstate_prefill_continues_exactly(o):
    """A prefix, then the rest from the prefix's final state, equals one
    scan bit for bit (fp32 and fp64 forward, with resets); the split backward
    (the suffix's grad_h0 as the prefix's grad_last) equals the whole one to
    rounding (fp64)."""
    B, T, D = 2, 40, 3
    ar, ai, br, bi, gr, gi, h0, gl = _cstate_case(66, B, T, D)
    seg = _segments(67, B, T)
    c = np.ascontiguousarray
    for dt, npdt in (("f32", np.float32), ("f64", np.float64)):
        xs = [x.astype(npdt) for x in (ar, ai, br, bi)]
        hh = tuple(x.astype(npdt) for x in h0)
        ref = o.cfwd_state(*xs, dt, h0=hh, segment_pos=seg)
        for T1 in (1, 13, 39):
            p1 = o.cfwd_state(*[c(x[:, :T1]) for x in xs], dt, h0=hh, segment_pos=c(seg[:, :T1]))
            p2 = o.cfwd_state(*[c(x[:, T1:]) for x in xs], dt, h0=(p1[2], p1[3]), segment_pos=c(seg[:, T1:]))
            assert np.array_equal(np.concatenate([p1[0], p2[0]], 1), ref[0]), (dt, T1)
            assert np.array_equal(np.concatenate([p1[1], p2[1]], 1), ref[1]), (dt, T1)
            assert np.array_equal(p2[2], ref[2]) and np.array_equal(p2[3], ref[3]), (dt, T1)
    ref = o.cfwd_state(ar, ai, br, bi, "f64", h0=h0, segment_pos=seg)
    full = o.cbwd_state(ar, ai, ref[0], ref[1], gr, gi, "f64", h0=h0, segment_pos=seg, grad_last=gl)
    for T1 in (1, 13, 39):
        s1, s2 = (slice(None), slice(None, T1)), (slice(None), slice(T1, None))
        p1 = o.cfwd_state(c(ar[s1]), c(ai[s1]), c(br[s1]), c(bi[s1]), "f64", h0=h0, segment_pos=c(seg[s1]))
        b2 = o.cbwd_state(c(ar[s2]), c(ai[s2]), c(ref[0][s2]), c(ref[1][s2]), c(gr[s2]), c(gi[s2]), "f64",
                          h0=(p1[2], p1[3]), segment_pos=c(seg[s2]), grad_last=gl)
        b1 = o.cbwd_state(c(ar[s1]), c(ai[s1]), c(ref[0][s1]), c(ref[1][s1]), c(gr[s1]), c(gi[s1]), "f64",
                          h0=h0, segment_pos=c(seg[s1]), grad_last=(b2[4], b2[5]))
        for k in range(4):
            np.testing.assert_allclose(np.concatenate([b1[k], b2[k]], 1), full[k], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b1[4], full[4], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b1[5], full[5], rtol=1e-12, atol=1e-12)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
