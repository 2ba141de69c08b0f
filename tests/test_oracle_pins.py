"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: library
conversions (numpy / torch / ml_dtypes), scipy's Hadamard matrix, closed
forms, brute force in numpy, and the figures the pages print
(tests/golden/page_figures.txt).  None of these tests needs a GPU.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle as O
from tests.conftest import golden

RNG = np.random.default_rng(20261202)


# --------------------------------------------------------------------------- fp16 / bf16

def _f16_candidates():
    x = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * np.float32(100.0),
        RNG.standard_normal(5000).astype(np.float32) * np.float32(1e-5),       # fp16 subnormals
        (RNG.standard_normal(5000) * 1e-8).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9, 2**-24, 2**-25, 3 * 2**-26], np.float32),
    ])
    # exact ties halfway between consecutive fp16 values
    h = RNG.integers(0, 0x7BFF, 4000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    return np.concatenate([x, mid, -mid])


def test_f16_rne_matches_numpy():
    x = _f16_candidates()
    ours = O.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_saturating_variant():
    x = np.array([65504.0, 65519.99, 65520.0, 1e30, -70000.0, np.inf], np.float32)
    got = O.f32_to_f16_bits(x, saturate=True)
    assert list(got) == [0x7BFF, 0x7BFF, 0x7BFF, 0x7BFF, 0xFBFF, 0x7BFF]


def test_f16_decode_matches_numpy():
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_bits_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_bf16_rne_matches_torch():
    x = np.concatenate([RNG.standard_normal(20000).astype(np.float32) * 37,
                        np.frombuffer(RNG.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32).tobytes(),
                                      np.float32)])
    x = x[np.isfinite(x)]
    ours = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------- e4m3

def _finite_codes():
    return np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)


def test_e4m3_table_from_definition():
    v = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    fig = golden("page_figures.txt")
    assert v[0x7E] == fig["fp8_max_finite"] == 448.0
    assert v[0x01] == 2.0**-9 and v[0x08] == 2.0**-6 and v[0x38] == 1.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                       # monotone
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign-magnitude
    assert math.copysign(1.0, v[0x80]) == -1.0            # -0
    # cross-check with torch's own e4m3 type
    ref = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fin = ~np.isnan(ref)
    assert np.array_equal(v[fin], ref[fin])


def test_e4m3_exhaustive_roundtrip():
    c = _finite_codes()
    vals = O.e4m3_to_f64(c).astype(np.float32)
    back = O.f32_to_e4m3(vals)
    assert np.array_equal(back, c)                       # includes -0 <-> 0x80


def test_e4m3_midpoints_round_to_even():
    pos = O.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    for sgn in (1.0, -1.0):
        for c in range(0x7E):
            mid = np.float32(sgn * (pos[c] + pos[c + 1]) / 2)       # exact in fp32
            assert float(mid) == sgn * (pos[c] + pos[c + 1]) / 2
            got = int(O.f32_to_e4m3(np.array([mid]))[0]) & 0x7F
            even = c if c % 2 == 0 else c + 1                      # includes binade carries
            assert got == even, (c, mid, got)
            up = np.nextafter(mid, np.float32(sgn * np.inf))
            dn = np.nextafter(mid, np.float32(0.0))
            assert int(O.f32_to_e4m3(np.array([up]))[0]) & 0x7F == c + 1
            assert int(O.f32_to_e4m3(np.array([dn]))[0]) & 0x7F == c


def test_e4m3_saturation_nan_and_zero():
    x = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e6, np.inf, -448.5, -np.inf, np.nan, -np.nan, 0.0, -0.0],
                 np.float32)
    got = list(O.f32_to_e4m3(x))
    assert got == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x00, 0x00, 0x00, 0x80]


def test_e4m3_matches_torch_in_range():
    x = np.concatenate([RNG.standard_normal(50000) * 40, RNG.standard_normal(20000) * 1e-2,
                        RNG.standard_normal(5000) * 1e-3]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = O.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_matches_ml_dtypes_in_range():
    ml = pytest.importorskip("ml_dtypes")
    x = (RNG.standard_normal(50000) * 60).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = O.f32_to_e4m3(x)
    ref = x.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------- Hadamard

def test_hadamard_matches_scipy_sylvester():
    Href = scipy.linalg.hadamard(32).astype(np.float64) / math.sqrt(32)
    cols = O.hadamard32_f64(np.eye(32).reshape(-1)).reshape(32, 32)   # row j = H e_j
    assert np.allclose(cols.T, Href, rtol=0, atol=1e-15)
    Hint = scipy.linalg.hadamard(32)
    assert np.array_equal(Hint @ Hint, 32 * np.eye(32, dtype=Hint.dtype))   # H is orthogonal, self-inverse


def test_hadamard_self_inverse_and_norm():
    x = RNG.standard_normal(32 * 64)
    y = O.hadamard32_f64(x)
    assert np.allclose(O.hadamard32_f64(y), x, rtol=0, atol=1e-13)
    assert np.allclose(np.linalg.norm(y.reshape(-1, 32), axis=1), np.linalg.norm(x.reshape(-1, 32), axis=1),
                       rtol=1e-14)


def test_fp32_butterfly_close_to_definition():
    x = (RNG.standard_normal(32 * 256) * 10).astype(np.float32)
    y32 = O.fwht32_f32(x).astype(np.float64)
    Href = scipy.linalg.hadamard(32).astype(np.float64) / math.sqrt(32)
    y64 = (x.astype(np.float64).reshape(-1, 32) @ Href.T).reshape(-1)
    scale = np.abs(x.reshape(-1, 32)).sum(1).repeat(32)
    assert np.all(np.abs(y32 - y64) <= 8 * 2.0**-24 * scale)
    assert O.rotation_constant() == np.float32(1 / np.sqrt(32))
    ones = O.fwht32_f32(np.ones(32, np.float32))
    assert ones[0] == np.float32(32) * np.float32(1 / np.sqrt(32)) and np.all(ones[1:] == 0)


# --------------------------------------------------------------------------- 4-bit rows

def _canon_codes(canon):
    """Unpack stored code bytes (groups in order, low nibble = even element) into integer codes."""
    return np.stack([canon & 0xF, canon >> 4], -1).reshape(-1).astype(np.int64)


def test_exact_scale_block_codes_equal_inputs():
    fig = golden("page_figures.txt")
    for trial in range(50):
        c = RNG.integers(-8, 8, 256)
        c.reshape(8, 32)[:, RNG.integers(0, 32)] = -8        # every group reaches |c| = 8 -> amax 8
        # x = H c, so the store's rotation gives back c (H is self-inverse)
        x = O.hadamard32_f64(c.astype(np.float64)).astype(np.float32)
        canon, sc = O.q4_quantize_row(x)
        assert np.all(O.f16_bits_to_f64(sc) == fig["exact_scale_scale"])
        assert np.array_equal(_canon_codes(canon), c + 8)


def test_q4_0_exact_scale_block_codes_equal_inputs():
    """Unrotated Q4_0 ("feat(kvcache): add reliable quantized KV cache", test fixes:
    an exact-scale block, amax 8.0 so that the scale is 1.0, has codes equal to
    the inputs): no rotation, so x itself is the code minus 8."""
    fig = golden("page_figures.txt")
    for trial in range(50):
        c = RNG.integers(-8, 8, 256)
        c.reshape(8, 32)[:, RNG.integers(0, 32)] = -8        # every group reaches |c| = 8 -> amax 8
        canon, sc = O.q4_quantize_row(c.astype(np.float32), rotate=False)
        assert np.all(O.f16_bits_to_f64(sc) == fig["exact_scale_scale"])
        assert np.array_equal(_canon_codes(canon), c + 8)
    # and the rotated form of the same input differs (the rotation is really skipped)
    canon_r, _ = O.q4_quantize_row(c.astype(np.float32), rotate=True)
    assert not np.array_equal(canon_r, canon)


def test_code_ties_round_half_to_even_and_clamp_unrotated():
    """Exact halves in exact-scale blocks ("feat(kvcache): add reliable quantized
    KV cache", test-fix commit: amax 8 -> scale 1.0; its PyTorch reference
    rounds with torch.round, half to even): y / s = k + 1/2 must store the even
    neighbour, and +7.5 (even neighbour 8) must clamp to 7.  The expected codes
    are a literal table; half-away-from-zero and truncation disagree with it on
    these inputs, so either mistake in the oracle fails here."""
    from tests import tie_rows
    x, exp = tie_rows.unrotated_rows()
    away, trunc = tie_rows.alternative_codes()
    assert any(away[h] != tie_rows.TIE_CODE[h] for h in tie_rows.HALVES)
    assert any(trunc[h] != tie_rows.TIE_CODE[h] for h in tie_rows.HALVES)
    for r in range(x.shape[0]):
        canon, sc = O.q4_quantize_row(x[r], rotate=False)
        assert np.all(O.f16_bits_to_f64(sc) == 1.0)
        codes = _canon_codes(canon)
        tie = exp[r] >= 0
        assert np.array_equal(codes[tie], exp[r][tie])
        amax = np.abs(x[r]) == 8.0
        assert np.array_equal(codes[amax], np.where(x[r][amax] > 0, 15, 0))   # +8 clamps to code 15, -8 is 0


def test_code_ties_round_half_to_even_through_the_rotation():
    """The same tie rule on the rotated path: inputs built so that the fp32
    butterfly is exact and one element per group lands on y / s = k + 1/2
    exactly (checked with numpy fp32 arithmetic and scipy's Hadamard matrix);
    the oracle's scale must be the fp16 value of amax / 8 and the tie codes the
    literal table."""
    from tests import tie_rows
    x, exp, y, s = tie_rows.rotated_rows()
    assert sorted({float(y[r][c] / s[r][c // 32]) for r, c in zip(*np.nonzero(exp >= 0))}) == tie_rows.HALVES
    for r in range(x.shape[0]):
        canon, sc = O.q4_quantize_row(x[r], rotate=True)
        assert np.array_equal(O.f16_bits_to_f64(sc), s[r].astype(np.float64))
        codes = _canon_codes(canon)
        tie = exp[r] >= 0
        assert np.array_equal(codes[tie], exp[r][tie])
        zero = y[r] == 0
        assert np.all(codes[zero] == 8)


def test_q4_0_attention_is_plain_attention_over_dequantized_rows():
    """Q4_0: out = softmax(sm q . K) V with K, V the dequantized unrotated rows, and
    those rows within one scale step of the inputs (half a step, except a
    positive maximum, whose code 8 is clamped to 7; the fp16 scale may round
    below amax / 8 by up to 2^-11 relative, hence the (1 + 2^-8) margin)."""
    Hk, Hq, D, ps, T = 1, 3, 64, 16, 40
    bt = np.array([2, 0, 3], np.int32)
    k = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
    c = O.Cache(O.Q4_0, Hk, D, ps, 4)
    _fill(c, k, v, bt, T)
    out = O.decode(c, q, [T], bt[None], 1 / 8)
    Kd = np.stack([O.q4_dequant_row(c.k[bt[j // ps], 0, j % ps], c.k_scale[bt[j // ps], 0, j % ps]) for j in range(T)])
    Vd = np.stack([O.q4_dequant_row(c.v[bt[j // ps], 0, j % ps], c.v_scale[bt[j // ps], 0, j % ps]) for j in range(T)])
    for h in range(Hq):
        assert np.allclose(out[0, h], _np_attention(q[0, h].astype(np.float64), Kd, Vd, 1 / 8), rtol=1e-12, atol=1e-12)
    step = np.repeat(np.stack([O.f16_bits_to_f64(c.k_scale[bt[j // ps], 0, j % ps]) for j in range(T)]), 32, 1)
    err = np.abs(Kd - k[:, 0].astype(np.float64))
    assert np.all(err <= step * (1 + 2.0**-8))              # fp16 scale may round below amax / 8
    assert np.mean(err <= 0.5 * step * 1.0001) > 0.95


def test_row_bytes_match_page_figures():
    fig = golden("page_figures.txt")
    canon, sc = O.q4_quantize_row(np.ones(256, np.float32))
    assert canon.nbytes + sc.nbytes == fig["q4_row_bytes_d256"]
    assert (canon.nbytes + sc.nbytes) * 4 * 2 * 16 == fig["q4_bytes_per_position_16_layers_4_heads"]
    assert 256 * 2 * 4 * 2 * 16 == fig["bf16_bytes_per_position_16_layers_4_heads"]
    assert (fig["q4_group_code_bytes"] + 2) / fig["q4_group_values"] == fig["q4_bytes_per_element"]
    c = O.Cache(O.FP8, 1, 512, 16, 1, rope_dim=64)
    per_tok = (c.k.nbytes + c.v.nbytes + c.k_scale.nbytes + c.v_scale.nbytes) // 16
    assert per_tok == fig["fp8_latent_bytes_per_token"]
    c4 = O.Cache(O.Q4, 4, 256, 16, 1)
    per_pos = (c4.k.nbytes + c4.v.nbytes + c4.k_scale.nbytes + c4.v_scale.nbytes) // 16
    assert per_pos * 16 == fig["q4_bytes_per_position_16_layers_4_heads"]


def test_quantize_roundtrip_bounds_and_scale():
    H = scipy.linalg.hadamard(32).astype(np.float64) / math.sqrt(32)
    for trial in range(200):
        x = (RNG.standard_normal(256) * RNG.choice([1e-3, 1.0, 30.0])).astype(np.float32)
        if trial % 7 == 0:
            x[RNG.integers(0, 256, 3)] *= 100
        canon, sc = O.q4_quantize_row(x)
        y = (x.astype(np.float64).reshape(8, 32) @ H.T)
        s = O.f16_bits_to_f64(sc)
        # scale = fp16(amax/8): within one fp16 rounding of the fp64 value
        amax = np.abs(y).max(1)
        assert np.all(np.abs(s - amax / 8) <= 2.0**-11 * amax / 8 + 1e-12)
        codes = _canon_codes(canon).reshape(8, 32)
        deq = (codes - 8) * s[:, None]
        err = np.abs(deq - y)
        ratio = y / s[:, None]
        inner = ratio <= 7.5
        assert np.all(err[inner] <= 0.5 * np.broadcast_to(s[:, None], err.shape)[inner] * (1 + 1e-5) + 1e-6)
        assert np.all(err <= 1.01 * s[:, None] + 1e-6)
        assert np.allclose(O.q4_dequant_row(canon, sc), deq.reshape(-1), rtol=0, atol=0)


def test_zero_row_and_tiny_scale():
    canon, sc = O.q4_quantize_row(np.zeros(256, np.float32))
    assert np.all(sc == 0) and np.all(_canon_codes(canon) == 8)
    canon, sc = O.q4_quantize_row(np.full(256, 1e-9, np.float32))   # amax/8 below the smallest fp16
    assert np.all(sc == 0) and np.all(_canon_codes(canon) == 8)


def test_signed_nibble_shift_form():
    # The test-fix commit of "feat(kvcache): add reliable quantized KV cache" checks the
    # arithmetic-shift sign extension in int32 semantics; the biased form code - 8
    # is the same number for every nibble.
    import ctypes
    for c in range(16):
        shifted = ctypes.c_int32(ctypes.c_int32((c ^ 8) << 28).value >> 28).value
        assert shifted == c - 8


def test_stored_layout_is_group_major():
    """Exact-scale rows whose element i of group G carries code (G + i) % 16: the
    stored row holds group G in bytes 16G .. 16G + 15, element 2b in the low and
    2b + 1 in the high nibble of byte b, and dequantising reads the same places."""
    for D in (32, 64, 256):
        NG = D // 32
        c = np.array([[(G + i) % 16 - 8 for i in range(32)] for G in range(NG)], np.int64)
        c[:, 31] = -8   # amax 8 in every group -> scale 1.0
        codes, sc = O.q4_quantize_row(c.reshape(-1).astype(np.float32), rotate=False)
        assert np.all(sc == 0x3C00)
        for G in range(NG):
            for b in range(16):
                assert codes[16 * G + b] == (c[G, 2 * b] + 8) | ((c[G, 2 * b + 1] + 8) << 4)
        assert np.array_equal(O.q4_dequant_row(codes, sc), c.reshape(-1).astype(np.float64))


# --------------------------------------------------------------------------- attention

def _np_attention(q, K, V, sm):
    s = sm * (K @ q)
    p = np.exp(s - s.max())
    return (p @ V) / p.sum()


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _fill(cache, k, v, block_table, seq_len):
    slots = np.array([block_table[j // cache.page_size] * cache.page_size + j % cache.page_size
                      for j in range(seq_len)], np.int32)
    O.store(cache, k, v, slots)


def test_brute_force_bf16_paged_gqa():
    """BF16 rows (no quantisation, no rotation): the oracle equals numpy softmax."""
    for T in (1, 2, 5, 8, 37):
        Hk, Hq, D, ps = 2, 6, 32, 4
        n_pages = (T + ps - 1) // ps + 3
        bt = RNG.permutation(n_pages)[: (T + ps - 1) // ps].astype(np.int32)
        k = _bf16_bits(RNG.standard_normal((T, Hk, D)))
        v = _bf16_bits(RNG.standard_normal((T, Hk, D)))
        q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
        c = O.Cache(O.BF16, Hk, D, ps, n_pages)
        _fill(c, k, v, bt, T)
        out = O.decode(c, q, [T], bt[None], 0.3)
        K, V = _bf16_vals(k), _bf16_vals(v)
        for h in range(Hq):
            ref = _np_attention(q[0, h].astype(np.float64), K[:, h // 3], V[:, h // 3], 0.3)
            assert np.allclose(out[0, h], ref, rtol=1e-13, atol=1e-13)


def test_q4_attention_is_rotated_space_attention():
    """Q4: out = H (softmax(sm (H q) . K_rot) V_rot) with K_rot, V_rot the dequantized rows."""
    H = scipy.linalg.hadamard(32).astype(np.float64) / math.sqrt(32)
    Hk, Hq, D, ps, T = 1, 3, 64, 16, 40
    n_pages = 4
    bt = np.array([2, 0, 3], np.int32)
    k = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
    c = O.Cache(O.Q4, Hk, D, ps, n_pages)
    _fill(c, k, v, bt, T)
    out = O.decode(c, q, [T], bt[None], 1 / 8)
    Kr = np.stack([O.q4_dequant_row(c.k[bt[j // ps], 0, j % ps], c.k_scale[bt[j // ps], 0, j % ps]) for j in range(T)])
    Vr = np.stack([O.q4_dequant_row(c.v[bt[j // ps], 0, j % ps], c.v_scale[bt[j // ps], 0, j % ps]) for j in range(T)])
    rot = lambda x: (x.reshape(-1, 32) @ H.T).reshape(-1)
    for h in range(Hq):
        o = _np_attention(rot(q[0, h].astype(np.float64)), Kr, Vr, 1 / 8)
        assert np.allclose(out[0, h], rot(o), rtol=1e-12, atol=1e-12)
    # dequantized rows are close to the rotated inputs (4-bit error bound)
    assert np.all(np.abs(Kr - np.stack([rot(r) for r in k[:, 0].astype(np.float64)])) <=
                  1.01 * np.repeat(np.stack([O.f16_bits_to_f64(c.k_scale[bt[j // ps], 0, j % ps]) for j in range(T)]), 32, 1))


def test_rotation_invariance_of_attention():
    """softmax(Hq . Hk) H(sum p Hv) == softmax(q . k) sum p v on unquantised data."""
    T, D = 300, 256
    K = RNG.standard_normal((T, D)) * 3
    V = RNG.standard_normal((T, D))
    q = RNG.standard_normal(D)
    rot = lambda x: O.hadamard32_f64(x.reshape(-1)).reshape(x.shape)
    a = _np_attention(q, K, V, 1 / 16)
    b = rot(_np_attention(rot(q), rot(K), rot(V), 1 / 16))
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T", [1, 2, 511, 512, 513, 1024, 1025, 4097])
def test_split_merge_equals_single_pass(T):
    Hk, Hq, D, ps = 1, 2, 32, 16
    n_pages = (T + ps - 1) // ps
    bt = np.arange(n_pages, dtype=np.int32)
    k = (RNG.standard_normal((T, Hk, D)) * 4).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
    c = O.Cache(O.Q4, Hk, D, ps, n_pages)
    _fill(c, k, v, bt, T)
    a = O.decode(c, q, [T], bt[None], 0.25, split=False)
    b = O.decode(c, q, [T], bt[None], 0.25, split=True)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12 * np.abs(a).max())


def test_closed_forms_one_key_and_equal_scores():
    D, ps = 64, 16
    c = O.Cache(O.Q4, 1, D, ps, 2)
    k = RNG.standard_normal((20, 1, D)).astype(np.float32)
    v = RNG.standard_normal((20, 1, D)).astype(np.float32)
    _fill(c, k, v, np.array([1, 0], np.int32), 20)
    q = RNG.standard_normal((1, 2, D)).astype(np.float32)
    out1 = O.decode(c, q, [1], np.array([[1, 0]], np.int32), 0.1)
    vrot = O.q4_dequant_row(c.v[1, 0, 0], c.v_scale[1, 0, 0])
    assert np.allclose(out1[0, 0], O.hadamard32_f64(vrot), rtol=0, atol=1e-14)   # one key -> its value
    qz = np.zeros((1, 2, D), np.float32)
    outm = O.decode(c, qz, [20], np.array([[1, 0]], np.int32), 0.1)
    Vr = np.stack([O.q4_dequant_row(c.v[[1, 0][j // ps], 0, j % ps], c.v_scale[[1, 0][j // ps], 0, j % ps])
                   for j in range(20)])
    assert np.allclose(outm[0, 1], O.hadamard32_f64(Vr.mean(0)), rtol=0, atol=1e-13)   # equal scores -> mean


def test_paged_equals_contiguous_and_store_is_row_local():
    Hk, Hq, D, ps, T = 2, 4, 64, 16, 100
    n_pages = 8
    k = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
    ident = np.arange(n_pages, dtype=np.int32)
    shuf = RNG.permutation(n_pages).astype(np.int32)
    c1, c2, c3 = (O.Cache(O.Q4, Hk, D, ps, n_pages) for _ in range(3))
    _fill(c1, k, v, ident, T)
    _fill(c2, k, v, shuf, T)
    a = O.decode(c1, q, [T], ident[None], 0.125)
    b = O.decode(c2, q, [T], shuf[None], 0.125)
    assert np.array_equal(a, b)
    for j in range(T):   # one token at a time ("resumed equals fresh")
        O.store(c3, k[j:j + 1], v[j:j + 1], np.array([j], np.int32))
    assert np.array_equal(c1.k, c3.k) and np.array_equal(c1.v_scale, c3.v_scale)


def test_gather_equals_dense_over_selected_rows():
    Hk, Hq, D, ps, T = 1, 2, 64, 16, 200
    c = O.Cache(O.Q4, Hk, D, ps, 13)
    bt = np.arange(13, dtype=np.int32)
    k = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
    _fill(c, k, v, bt, T)
    full = O.decode(c, q, [T], bt[None], 0.1)
    allsel = O.decode(c, q, [T], bt[None], 0.1, sel=np.arange(T, dtype=np.int32)[None])
    assert np.array_equal(full, allsel)
    sel = np.sort(RNG.choice(T, 37, replace=False)).astype(np.int32)
    c2 = O.Cache(O.Q4, Hk, D, ps, 3)
    _fill(c2, k[sel], v[sel], np.arange(3, dtype=np.int32), 37)
    a = O.decode(c, q, [T], bt[None], 0.1, sel=sel[None])
    b = O.decode(c2, q, [37], np.arange(3, dtype=np.int32)[None], 0.1)
    assert np.array_equal(a, b)


def test_prefill_row_equals_decode_at_its_position():
    Hk, Hq, D, ps = 1, 3, 64, 16
    depth, n_q = 40, 9
    T = depth + n_q
    c = O.Cache(O.Q4, Hk, D, ps, 4)
    bt = np.array([3, 1, 0, 2], np.int32)
    k = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    _fill(c, k, v, bt, T)
    q = RNG.standard_normal((n_q, Hq, D)).astype(np.float32)
    out = O.prefill(c, q, depth, bt, 0.125)
    for i in range(n_q):
        d = O.decode(c, q[i:i + 1], [depth + i + 1], bt[None], 0.125)
        assert np.array_equal(out[i], d[0])
    sub = O.prefill(c, q, depth, bt, 0.125, rows=[0, 8, 3])
    assert np.array_equal(sub, out[[0, 8, 3]])


def test_prefill_row_equals_decode_at_its_position_fp8():
    """The same for the fp8 latent rows: 576-wide queries, 512-wide outputs."""
    D, R, ps, Hq = 512, 64, 16, 2
    depth, n_q = 30, 5
    T = depth + n_q
    c = O.Cache(O.FP8, 1, D, ps, 3, rope_dim=R)
    bt = np.array([2, 0, 1], np.int32)
    rows = (RNG.standard_normal((T, D + R)) * np.exp(RNG.standard_normal((T, 1)))).astype(np.float32)
    slots = np.array([bt[j // ps] * ps + j % ps for j in range(T)], np.int32)
    assert O.store(c, rows, None, slots) == 0
    q = RNG.standard_normal((n_q, Hq, D + R)).astype(np.float32)
    out = O.prefill(c, q, depth, bt, 0.05)
    assert out.shape == (n_q, Hq, D)
    for i in range(n_q):
        d = O.decode(c, q[i:i + 1], [depth + i + 1], bt[None], 0.05)
        assert np.array_equal(out[i], d[0])


def test_empty_sequence_gives_zero():
    c = O.Cache(O.Q4, 1, 32, 16, 1)
    out = O.decode(c, np.ones((1, 1, 32), np.float32), [0], np.zeros((1, 1), np.int32), 1.0)
    assert np.all(out == 0)


def test_bad_block_table_is_reported():
    c = O.Cache(O.Q4, 1, 32, 16, 1)
    with pytest.raises(ValueError):
        O.decode(c, np.ones((1, 1, 32), np.float32), [5], np.array([[7]], np.int32), 1.0)


# --------------------------------------------------------------------------- fp8 latent rows

def test_fp8_row_encoding():
    for trial in range(100):
        x = (RNG.standard_normal(512) * np.exp(RNG.standard_normal())).astype(np.float32)
        codes, s = O.fp8_encode_row(x)
        amax = np.float32(np.abs(x).max())
        assert s == np.float32(amax / np.float32(448))
        inv = np.float32(448) / amax
        ref = torch.from_numpy(x * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes, ref)        # in range: torch's RNE cast is the same encoder
        deq = O.e4m3_to_f64(codes) * float(s)
        assert np.all(np.abs(deq - x) <= 2.0**-4 * np.abs(x) + 2.0**-10 * float(s) + 1e-30)
        assert O.e4m3_to_f64(codes).max() <= 448 and np.abs(O.e4m3_to_f64(codes)).max() == 448
    codes, s = O.fp8_encode_row(np.zeros(64, np.float32))
    assert s == 0 and np.all(codes == 0)
    tiny = np.full(64, 1e-40, np.float32)          # 448/amax overflows: guarded
    codes, s = O.fp8_encode_row(tiny)
    assert np.all(codes == 0) and s == np.float32(np.float32(1e-40) / np.float32(448))


def test_fp8_absorbed_attention_brute_force():
    T, Hq, D, R, ps = 50, 4, 64, 16, 16
    n_pages = 4
    rows = (RNG.standard_normal((T, D + R)) * np.exp(RNG.standard_normal((T, 1)))).astype(np.float32)
    c = O.Cache(O.FP8, 1, D, ps, n_pages, rope_dim=R)
    bt = np.array([2, 3, 0, 1], np.int32)
    slots = np.array([bt[j // ps] * ps + j % ps for j in range(T)], np.int32)
    O.store(c, rows, None, slots)
    q = RNG.standard_normal((1, Hq, D + R)).astype(np.float32)
    out = O.decode(c, q, [T], bt[None], 1 / math.sqrt(D + R))
    e4 = lambda b: torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    L = np.stack([e4(c.k[bt[j // ps], 0, j % ps]) * c.k_scale[bt[j // ps], 0, j % ps] for j in range(T)])
    Rr = np.stack([e4(c.v[bt[j // ps], 0, j % ps]) * c.v_scale[bt[j // ps], 0, j % ps] for j in range(T)])
    K = np.concatenate([L, Rr], 1)
    for h in range(Hq):
        ref = _np_attention(q[0, h].astype(np.float64), K, L, 1 / math.sqrt(D + R))
        assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-12)
    split = O.decode(c, q, [T], bt[None], 1 / math.sqrt(D + R), split=True)
    assert np.allclose(split, out, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- TQ4 (rotated int4 + codebook)

def _signs(n, seed):
    return np.random.default_rng(seed).integers(0, 2**32, n // 32, dtype=np.uint64).astype(np.uint32)


def _sign_vector(signs, n):
    return np.array([-1.0 if (signs[i // 32] >> (i % 32)) & 1 else 1.0 for i in range(n)])


def test_tq4_codebook_is_the_lloyd_max_quantizer_of_a_normal():
    """The 16 levels: +-M_m with M the fixed point of Lloyd's iteration for N(0,1)
    (centroids of the cells between midpoints), each rounded to fp16."""
    from scipy.stats import norm
    lv = O.tq4_levels()
    M = lv[:8]
    assert np.all(np.diff(M) > 0) and np.array_equal(lv[8:], -M)
    assert np.array_equal(M.astype(np.float16).astype(np.float64), M)
    L = np.linspace(-2.0, 2.0, 16)
    for _ in range(5000):
        t = np.concatenate([[-np.inf], (L[:-1] + L[1:]) / 2, [np.inf]])
        L = (norm.pdf(t[:-1]) - norm.pdf(t[1:])) / (norm.cdf(t[1:]) - norm.cdf(t[:-1]))
    star = L[8:]
    assert np.all(np.abs(M - star) <= 2.0**-11 * star)
    # its mean squared error on N(0,1): the Lloyd-Max figure for 16 levels
    x = np.random.default_rng(3).standard_normal(400000)
    q = np.sign(x) * M[np.clip(np.searchsorted((M[:-1] + M[1:]) / 2, np.abs(x)), 0, 7)]
    assert abs(np.mean((x - q) ** 2) - 0.0095) < 0.0003


def test_tq4_rotation_is_the_signed_walsh_hadamard_transform():
    """Forward: H (s * x) / sqrt(n) with scipy's Sylvester H; inverse undoes it; the
    store's fp32 butterfly equals the definition to fp32 rounding."""
    for n in (32, 64, 128, 256):
        s = _signs(n, n)
        sv = _sign_vector(s, n)
        H = scipy.linalg.hadamard(n) / math.sqrt(n)
        x = RNG.standard_normal(n)
        f = O.tq4_rotate_f64(x, s)
        assert np.allclose(f, H @ (sv * x), rtol=0, atol=1e-12)
        assert np.allclose(O.tq4_rotate_f64(f, s, inverse=True), x, rtol=0, atol=1e-12)
        y32 = O.tq4_rotate_f32(x.astype(np.float32), s)
        assert np.allclose(y32, H @ (sv * x.astype(np.float32).astype(np.float64)), rtol=0,
                           atol=1e-5 * np.abs(x).max())
    z = np.zeros(1, np.uint32)
    x = RNG.standard_normal(32)
    assert np.allclose(O.tq4_rotate_f64(x, z), scipy.linalg.hadamard(32) @ x / math.sqrt(32), atol=1e-12)


def test_tq4_codes_are_the_nearest_levels_at_radius_over_root_n():
    """Scale = ||x|| / sqrt(n) to fp16 rounding (the rotation keeps the radius);
    every code names the level nearest y / scale (brute force over 16 levels)."""
    lv = O.tq4_levels()
    for trial in range(60):
        n = (64, 128, 256)[trial % 3]
        s = _signs(n, 1000 + trial)
        x = (RNG.standard_normal(n) * RNG.choice([1e-3, 1.0, 50.0])).astype(np.float32)
        if trial % 5 == 0:
            x[RNG.integers(0, n, 3)] *= 40
        codes, sc = O.tq4_quantize_row(x, s)
        scale = float(np.array(sc, np.uint16).view(np.float16))
        radius = np.linalg.norm(x.astype(np.float64))
        assert abs(scale - radius / math.sqrt(n)) <= 2.0**-10 * radius / math.sqrt(n) + 1e-7
        c = np.stack([codes & 0xF, codes >> 4], -1).reshape(-1)
        y = O.tq4_rotate_f32(x, s).astype(np.float64)
        v = y / np.float64(np.float32(scale))
        best = np.argmin(np.abs(v[:, None] - lv[None, :]), 1)
        dist_c = np.abs(v - lv[c])
        dist_b = np.abs(v - lv[best])
        assert np.all(dist_c <= dist_b + 1e-6 * np.abs(v).max())


def test_tq4_distortion_matches_the_pages():
    """Rotated int4 + codebook reconstructs a row to rel-L2 ~0.096 at 4 bits
    ("Why rotated-int4"); 0.0975 is the Lloyd-Max figure for Gaussian coordinates.
    Outlier channels are spread by the rotation and change little."""
    fig = golden("page_figures.txt")
    for outliers in (False, True):
        errs = []
        for trial in range(120):
            n = 256
            s = _signs(n, 5000 + trial)
            x = RNG.standard_normal(n) * math.exp(RNG.standard_normal())
            if outliers:
                x[RNG.integers(0, n, 4)] *= 20
            x = x.astype(np.float32)
            codes, sc = O.tq4_quantize_row(x, s)
            rec = O.tq4_rotate_f64(O.tq4_dequant_row(codes, sc), s, inverse=True)
            errs.append(np.linalg.norm(rec - x) / np.linalg.norm(x))
        assert abs(np.mean(errs) - fig["tq4_rel_l2"]) < 0.008, np.mean(errs)


def test_tq4_zero_row():
    codes, sc = O.tq4_quantize_row(np.zeros(64, np.float32), _signs(64, 1))
    assert sc == 0 and np.all(codes == 0)
    assert np.all(O.tq4_dequant_row(codes, sc) == 0)


def test_tq4_attention_is_rotated_space_attention():
    """Decode over a TQ4 cache = softmax attention in the rotated space over the
    dequantised rows, output rotated back by the inverse transform (brute force
    in numpy with scipy's Hadamard)."""
    D, Hk, Hq, T, ps = 64, 2, 4, 45, 16
    s = _signs(D, 77)
    sv = _sign_vector(s, D)
    H = scipy.linalg.hadamard(D) / math.sqrt(D)
    npg = 4
    c = O.Cache(O.TQ4, Hk, D, ps, npg, signs=s)
    k = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    v = RNG.standard_normal((T, Hk, D)).astype(np.float32)
    bt = np.array([[2, 0, 3, 1]], np.int32)
    slots = np.array([bt[0, j // ps] * ps + j % ps for j in range(T)], np.int32)
    assert O.store(c, k, v, slots) == 0
    q = RNG.standard_normal((1, Hq, D)).astype(np.float32)
    out = O.decode(c, q, [T], bt, 0.2)
    for h in range(Hq):
        hk = h // (Hq // Hk)
        Kr = np.stack([O.tq4_dequant_row(c.k[bt[0, j // ps], hk, j % ps], c.k_scale[bt[0, j // ps], hk, j % ps])
                       for j in range(T)])
        Vr = np.stack([O.tq4_dequant_row(c.v[bt[0, j // ps], hk, j % ps], c.v_scale[bt[0, j // ps], hk, j % ps])
                       for j in range(T)])
        qr = H @ (sv * q[0, h].astype(np.float64))
        sc_ = 0.2 * (Kr @ qr)
        p = np.exp(sc_ - sc_.max())
        o = sv * (H @ ((p @ Vr) / p.sum()))
        assert np.allclose(out[0, h], o, rtol=0, atol=1e-12 * max(1.0, np.abs(o).max()))
