"""CPU checks of the arithmetic shortcuts the NVFP4 kernels rely on.

The kernels take two decisions through cheaper fp32 sequences than the
oracle's exact ones; these tests replay those sequences in numpy (float32
steps, fused multiply-add emulated in float64, where the product is exact) over
every case that can matter, and compare with exact rational arithmetic:

1. block scale: e4m3(amax * fp32(1/6)) == e4m3(amax / 6) for every finite
   non-negative bf16 amax (torch's e4m3 conversion, saturating at 448);
2. e2m1 decision: q = fma(v, r_hi, v * r_lo) with r_hi ~ 1/s (the hardware
   reciprocal, allowed to be off by up to 2 ulp) and r_lo = r_hi * (1 - s*r_hi)
   rounds to the same e2m1 code as the exact v/s, for every e4m3 scale s, at
   every midpoint (ties) and on bf16 values around them.

4. the same quotient for the two-level contract, whose divisor is s * ts with
   ts a bf16 tensor scale (up to 12 significant bits): every pair of e4m3 and
   bf16 mantissas, at every tie and its bf16 neighbours.

And the fact the modfp8 kernels' decode rests on:

3. they convert e4m3 byte pairs to f16 pairs in hardware, then each f16 to
   fp32; that is exact only if every finite e4m3 value is an f16 value (the
   smallest e4m3 subnormal, 2^-9, is an f16 normal; 448 is far below the f16
   maximum).  The test checks the round trip e4m3 -> f16 -> fp32 against
   torch's float8_e4m3fn decoder for every finite code; the conversion itself
   runs in the GPU parity tests of the modfp8 producers.
"""
from fractions import Fraction

import numpy as np
import torch

F32 = np.float32


def _e4m3(vals: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(vals, dtype=np.float32)).clamp(max=448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_block_scale_by_multiplication_equals_division():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # every finite non-negative bf16
    amax = (bits << 16).view(np.float32)
    by_mul = _e4m3(amax * F32(1.0 / 6.0))
    exact = _e4m3((amax.astype(np.float64) / 6.0).astype(np.float32))
    assert np.array_equal(by_mul, exact)


def _fma32(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


MIDS = [Fraction(1, 4), Fraction(3, 4), Fraction(5, 4), Fraction(7, 4), Fraction(5, 2), Fraction(7, 2), Fraction(5)]
GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def _code_exact(v: Fraction, s: Fraction) -> int:
    q = abs(v) / s
    d = [abs(q - g) for g in GRID]
    best = min(d)
    c = [k for k, x in enumerate(d) if x == best]
    return c[0] if len(c) == 1 else [k for k in c if k % 2 == 0][0]


def _code_rne32(q: np.ndarray) -> np.ndarray:
    # nearest of the e2m1 grid, ties to even, on float32 quotients
    a = np.abs(q.astype(np.float64))
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    tie = (d == best)
    even = tie & (np.arange(8)[None, :] % 2 == 0)
    return np.where(tie.sum(axis=1) > 1, even.argmax(axis=1), tie.argmax(axis=1))


def test_e2m1_quotient_is_exact_at_midpoints_for_every_scale():
    scales = torch.arange(1, 0x7F, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for s in scales:
        s32 = F32(s)
        base = F32(1.0) / s32
        for ulps in (-2, -1, 0, 1, 2):
            rh = np.nextafter(base, F32(np.inf if ulps > 0 else -np.inf), dtype=np.float32) if ulps else base
            for _ in range(abs(ulps) - 1):
                rh = np.nextafter(rh, F32(np.inf if ulps > 0 else -np.inf), dtype=np.float32)
            rl = F32(rh * _fma32(np.array([-s32]), np.array([rh]), np.array([F32(1)]))[0])
            # ties and their bf16 neighbours, both signs
            vals = []
            for m in MIDS:
                v = float(m) * float(s)
                b = torch.tensor([v], dtype=torch.float64).float().to(torch.bfloat16)
                if float(b) != v:
                    continue  # not representable as a bf16 v: no tie possible
                bits = int(b.view(torch.int16))
                for k in (-1, 0, 1):
                    vals.append(torch.tensor([bits + k], dtype=torch.int16).view(torch.bfloat16).item())
            v = np.array(vals + [-x for x in vals], dtype=np.float32)
            q = _fma32(v, np.full_like(v, rh), (v * rl).astype(np.float32))
            got = _code_rne32(q)
            exp = np.array([_code_exact(Fraction(float(x)), Fraction(float(s))) for x in v])
            assert np.array_equal(got, exp), (s, ulps)


def test_every_finite_e4m3_value_is_an_f16_value():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    via_f16 = ref.astype(np.float16).astype(np.float32)
    assert np.array_equal(via_f16.view(np.uint32), ref.view(np.uint32))  # signs of zero included
    # the smallest subnormal 2^-9 and the largest normal 448 are among them
    assert ref[codes == 0x01][0] == 2.0**-9 and ref[codes == 0x7E][0] == 448.0
    assert np.all(np.abs(via_f16[ref != 0]) >= np.finfo(np.float16).tiny)  # f16 normals, not subnormals


def test_two_level_quotient_is_exact_for_every_divisor_mantissa():
    # divisor D = s * ts: e4m3 mantissas 1 + k/8 times bf16 mantissas 1 + m/128
    # (exponents only shift D and v together); exact codes from float64
    # comparisons of |v| with mid * D (exact: at most 3 + 12 + 8 bits)
    sm = np.arange(8, 16, dtype=np.float64) / 8
    tm = np.arange(128, 256, dtype=np.float64) / 128
    D = np.unique((sm[:, None] * tm[None, :]).reshape(-1))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    upper_even = np.array([False, True, False, True, False, True, False])  # upper neighbour's code is even

    def exact_code(v, d):
        a = np.abs(v)[:, None]
        th = mids[None, :] * d[:, None]
        up = (a > th) | ((a == th) & upper_even[None, :])
        return up.sum(axis=1)

    for ulps in (-2, -1, 0, 1, 2):
        d32 = D.astype(np.float32)
        assert np.array_equal(d32.astype(np.float64), D)          # exact in fp32
        rh = (F32(1.0) / d32).astype(np.float32)
        for _ in range(abs(ulps)):
            rh = np.nextafter(rh, F32(np.inf if ulps > 0 else -np.inf), dtype=np.float32)
        rl = (rh * _fma32(-d32, rh, np.ones_like(d32))).astype(np.float32)
        # candidate v: the bf16 values nearest mid * D and their neighbours
        tie = (mids[None, :] * D[:, None]).reshape(-1)
        dd = np.repeat(D, len(mids)).astype(np.float64)
        bits = torch.from_numpy(tie.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
        vs, ds, rhs, rls = [], [], [], []
        for k in (-1, 0, 1):
            b = torch.from_numpy((bits + k).astype(np.int16)).view(torch.bfloat16).double().numpy()
            vs.append(b); ds.append(dd)
            rhs.append(np.repeat(rh, len(mids))); rls.append(np.repeat(rl, len(mids)))
        v = np.concatenate(vs); v = np.concatenate([v, -v])
        d = np.concatenate(ds * 2)
        r_h = np.concatenate(rhs * 2); r_l = np.concatenate(rls * 2)
        v32 = v.astype(np.float32)
        assert np.array_equal(v32.astype(np.float64), v)
        q = _fma32(v32, r_h, (v32 * r_l).astype(np.float32))
        assert np.array_equal(_code_rne32(q), exact_code(v, d)), ulps


# ---------------------------------------------------------------------------
# two-level block scale: (amax / 6) / ts without IEEE divisions
# ---------------------------------------------------------------------------

def _rn32(x: Fraction) -> np.float32:
    """Round an exact rational to the nearest float32, ties to even (normal and
    subnormal range; no overflow in the cases below)."""
    f = np.float32(float(x))  # within one float32 ulp of x
    best = None
    for c in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        d = abs(Fraction(float(c)) - x)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(c).view(np.uint32)) & 1) == 0):
            best = (d, c)
    return np.float32(best[1])


def _fma_exact(a, b, c) -> np.float32:
    return _rn32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


INV6 = _rn32(Fraction(1, 6))


def _two_level_q_fast(amax: np.float32, ts: np.float32) -> np.float32:
    # the kernel's form: RN(amax / 6) and RN(q1 / ts) each from a product by the
    # correctly rounded reciprocal and one fused residual correction
    q = np.float32(amax * INV6)
    e = _fma_exact(np.float32(-6.0), q, amax)
    q1 = _fma_exact(e, INV6, q)
    rt = _rn32(Fraction(1) / Fraction(float(ts)))
    q = np.float32(q1 * rt)
    e = _fma_exact(-ts, q, q1)
    return _fma_exact(e, rt, q)


def _two_level_q_exact(amax: np.float32, ts: np.float32) -> np.float32:
    q1 = _rn32(Fraction(float(amax)) / 6)
    return _rn32(Fraction(float(q1)) / Fraction(float(ts)))


def test_two_level_scale_quotient_exact_for_every_significand_pair():
    # both operands are bf16 values: 8-bit significands; scaling by powers of
    # two commutes with the roundings in the normal range, so every pair of
    # significands at one exponent covers the kernel's fast path
    sig = [np.float32(m / 128.0) for m in range(128, 256)]
    for a in sig:
        for t in sig:
            assert _two_level_q_fast(a, t) == _two_level_q_exact(a, t), (a, t)


def test_two_level_scale_byte_on_random_bf16_pairs_across_the_range():
    # the e4m3 byte of fminf(q, 448) over bf16 pairs of every magnitude the fast
    # path takes (amax, ts >= 2^-100), overflow to the clamp included
    rng = np.random.default_rng(11)
    bits = rng.integers(0x0D80, 0x7F80, size=(6000, 2), dtype=np.uint32)  # from 2^-100 to the largest bf16
    for ab, tb in bits:
        a, t = (np.uint32(ab) << 16).view(np.float32), (np.uint32(tb) << 16).view(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            qf = _two_level_q_fast_safe(a, t)
        qe = _two_level_q_exact_big(a, t)
        assert _e4m3(np.fmin(np.float32(qf), np.float32(448.0))) == _e4m3(np.minimum(qe, 448.0)), (a, t)


def _two_level_q_fast_safe(amax, ts):
    # as _two_level_q_fast, with float32 overflow to inf as the hardware gives it
    # (the exact helpers above assume finite values)
    q = np.float32(amax * INV6)
    e = _fma_exact(np.float32(-6.0), q, amax)
    q1 = _fma_exact(e, INV6, q)
    rt = _rn32(Fraction(1) / Fraction(float(ts)))
    q = np.float32(q1 * rt)
    if not np.isfinite(q):
        return np.float32(np.nan)  # -ts * inf + q1 = -inf; -inf * rt + inf = NaN
    e = _fma_exact(-ts, q, q1)
    r = Fraction(float(e)) * Fraction(float(rt)) + Fraction(float(q))
    return np.float32(np.inf) if abs(r) > Fraction(float(np.finfo(np.float32).max)) else _rn32(r)


def _two_level_q_exact_big(amax, ts) -> float:
    q1 = _rn32(Fraction(float(amax)) / 6)
    r = Fraction(float(q1)) / Fraction(float(ts))
    return float("inf") if r > Fraction(float(np.finfo(np.float32).max)) else float(_rn32(r))
