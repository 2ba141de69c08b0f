"""Rows whose 4-bit codes sit exactly on rounding ties (test inputs only).

The store's code rule is clamp(rint_even(y / s), -8, 7) + 8 (round half to
even, after "feat(kvcache): add reliable quantized KV cache", whose PyTorch
reference rounds with torch.round; exact-scale blocks from its test-fix
commit: amax 8 -> scale 1).  Random data almost never lands on an exact half,
so these rows are built so that y / s is exactly k + 1/2 for every k in
-8 .. 7, where half-to-even, half-away-from-zero and truncation all disagree.

Unrotated rows (Q4_0): the values themselves, with an element of magnitude 8
per group so that s = fp16(8 / 8) = 1.

Rotated rows (Q4_HAD32): the store applies y = fl(fl-butterfly(x) * c) with
c = fp32(1/sqrt(32)).  A group is built from its butterfly output W, which has
two nonzero entries: W_a = +-2^j (the group maximum after the rotation, so
s = fp16(|W_a| c / 8)) and W_t, an fp32 value chosen so that fl(W_t * c) is
exactly h * s for the tie h.  The input is x = H W / 32 (H the +-1 Sylvester
matrix, H H = 32 I).  Every partial sum of the butterfly of x is
2^m / 32 * (+-W_a [.] +- W_t [.]), and W_t is picked so that W_a +- W_t is an
fp32 value, so the butterfly is exact and returns W.  Each group's tie is
checked here with numpy's fp32 arithmetic and scipy's Hadamard matrix, which
share nothing with the oracle or the CUDA library.

Nothing here encodes the rounding rule itself: the expected codes are the
literal table TIE_CODE below.
"""
import numpy as np
import scipy.linalg

C32 = np.float32(1.0 / np.sqrt(32.0))

# y / s -> stored code under round-half-to-even then the clamp to [-8, 7]
# (the code is q + 8): written out, one entry per half.
TIE_CODE = {
    0.5: 8, 1.5: 10, 2.5: 10, 3.5: 12, 4.5: 12, 5.5: 14, 6.5: 14, 7.5: 15,   # +7.5 rounds to 8, clamped to 7
    -0.5: 8, -1.5: 6, -2.5: 6, -3.5: 4, -4.5: 4, -5.5: 2, -6.5: 2, -7.5: 0,
}
HALVES = sorted(TIE_CODE)


def _half_away(h):
    return float(np.sign(h) * np.floor(abs(h) + 0.5))


def alternative_codes():
    """The codes two plausible wrong rules would store for the same ties
    (half away from zero, and truncation toward zero), both clamped."""
    away = {h: int(min(max(_half_away(h), -8), 7)) + 8 for h in HALVES}
    trunc = {h: int(min(max(np.trunc(h), -8), 7)) + 8 for h in HALVES}
    return away, trunc


def unrotated_rows(D=256):
    """Rows of the unrotated format: group G holds -8 (or +8) at one place, then
    the 16 halves, then zeros.  Returns (x [n, D] fp32, expected code per
    element [n, D], or -1 where the element is not a tie)."""
    ng = D // 32
    rows, exp = [], []
    for variant in range(4):
        x = np.zeros(D, np.float32)
        e = np.full(D, -1, np.int64)
        for G in range(ng):
            g = x[32 * G:32 * G + 32]
            eg = e[32 * G:32 * G + 32]
            a = (3 * G + variant) % 32
            g[a] = 8.0 if (G + variant) % 2 else -8.0       # amax 8 -> scale 1
            pos = [p for p in range(32) if p != a]
            order = np.roll(np.array(HALVES), G + 5 * variant)
            for p, h in zip(pos, order):
                g[p] = h
                eg[p] = TIE_CODE[h]
        rows.append(x)
        exp.append(e)
    return np.stack(rows), np.stack(exp)


def _ulp_neighbours(w, n=6):
    out = [np.float32(w)]
    up = dn = np.float32(w)
    for _ in range(n):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return out


def _rotated_group(j, sign_a, a, t, h):
    """The butterfly output W of one group (see the module text) with the tie h at
    index t, or None when no fp32 W_t near h s / c gives an exact tie."""
    wa = np.float32(sign_a * 2.0 ** j)
    ya = np.float32(wa * C32)
    s = np.float32(np.float16(np.float32(np.abs(ya)) / np.float32(8.0)))
    target = np.float32(h) * s                        # h has 4 significant bits, s 11: exact
    if float(target) != float(h) * float(s):
        return None
    for wt in _ulp_neighbours(np.float32(float(target) / float(C32))):
        if np.float32(wt * C32) != target:
            continue
        if abs(float(wt * C32)) >= abs(float(ya)):
            continue
        # W_a +- W_t must be fp32 values for the butterfly to stay exact
        if any(float(np.float32(float(wa) + sgn * float(wt))) != float(wa) + sgn * float(wt) for sgn in (1, -1)):
            continue
        W = np.zeros(32, np.float64)
        W[a], W[t] = float(wa), float(wt)
        return W
    return None


def rotated_rows(D=256, exponents=(-3, 0, 2, 4)):
    """Rows of the rotated format, one tie per group.  Returns (x [n, D] fp32,
    expected code per element [n, D] (-1 where not a tie), y [n, D] fp32 the
    rotated values, s [n, D // 32] the scales), every tie verified."""
    H = scipy.linalg.hadamard(32).astype(np.float64)
    ng = D // 32
    groups = []
    for j in exponents:
        for i, h in enumerate(HALVES):
            for attempt in range(32):
                a = (5 * i + attempt) % 32
                t = (a + 1 + 7 * attempt + i) % 32
                if t == a:
                    continue
                W = _rotated_group(j, 1 if (i + attempt) % 2 else -1, a, t, h)
                if W is not None:
                    groups.append((W, t, h))
                    break
    assert len(groups) >= 3 * len(HALVES), "too few exact ties found"
    while len(groups) % ng:
        groups.append(groups[len(groups) % ng])
    xs, es, ys, ss = [], [], [], []
    for r in range(len(groups) // ng):
        x = np.zeros(D, np.float32)
        e = np.full(D, -1, np.int64)
        y = np.zeros(D, np.float32)
        s = np.zeros(ng, np.float32)
        for G in range(ng):
            W, t, h = groups[r * ng + G]
            xg = H @ W / 32.0
            assert np.array_equal(xg.astype(np.float32).astype(np.float64), xg), "input not exact in fp32"
            assert np.array_equal(H @ xg, W), "butterfly not exact"
            yg = (W.astype(np.float32) * C32).astype(np.float32)
            sg = np.float32(np.float16(np.float32(np.abs(yg).max()) / np.float32(8.0)))
            assert float(yg[t]) / float(sg) == h          # the exact tie, in fp64 (no rounding)
            assert np.float32(yg[t] / sg) == np.float32(h)
            x[32 * G:32 * G + 32] = xg.astype(np.float32)
            e[32 * G + t] = TIE_CODE[h]
            y[32 * G:32 * G + 32] = yg
            s[G] = sg
        xs.append(x)
        es.append(e)
        ys.append(y)
        ss.append(s)
    return np.stack(xs), np.stack(es), np.stack(ys), np.stack(ss)


def near_tie_rows(D=256):
    """Unrotated rows whose quotients y / s sit within a few ulps of every
    half-integer k + 1/2 (k = -9 .. 8), for the scale 1 (group maximum 8) and
    the scale 0.8125 (group maximum 6.5, an exact fp16 value): y = the fp32
    value nearest (k + 1/2) s, then 1 .. 3 ulps either side.  Their codes
    depend on the last bit of the rounded quotient.  Returns x [n, D] fp32."""
    ng = D // 32
    vals = {1.0: [], 0.8125: []}
    for s in vals:
        for k in range(-9, 9):
            base = np.float32((k + 0.5) * s)
            up = dn = base
            cand = [base]
            for _ in range(3):
                up = np.nextafter(up, np.float32(np.inf))
                dn = np.nextafter(dn, np.float32(-np.inf))
                cand += [up, dn]
            vals[s] += [c for c in cand if abs(float(c)) <= 8.0 * s]
    groups = []
    for s, vs in vals.items():
        for i in range(0, len(vs), 31):
            g = np.zeros(32, np.float32)
            g[0] = np.float32(-8.0 * s)                      # the group maximum: s = fp16(8 s / 8) = s
            chunk = vs[i:i + 31]
            g[1:1 + len(chunk)] = chunk
            groups.append(g)
    while len(groups) % ng:
        groups.append(groups[len(groups) % ng])
    return np.stack(groups).reshape(-1, D)
