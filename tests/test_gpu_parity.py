"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Codes, scales and fp8 bytes must be bit-exact; attention outputs must satisfy
max|gpu - oracle| <= 2e-3 * max|oracle| per (sequence) output tensor [Hq, D]
(per query row for prefill), the oracle computing in fp64 over the same
quantised cache.  Sizes span several 16-key tiles, several 512-key
partitions and ragged tails.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from bit_quantized_kv_store_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_kv_store_gb300 import build
    build.build()
    from bit_quantized_kv_store_gb300 import _lib
    _lib.lib()
    return _lib


DEV = "cuda"


def bits_u16(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(got, ref, tol=TOL, what=""):
    got = np.asarray(got, np.float64)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert err <= tol * scale, f"{what}: max-abs error {err:.3g} > {tol} * {scale:.3g}"
    return err / scale


def make_cache_pair(K, fmt, Hk, D, ps, n_pages, rope=0, sign_seed=0):
    signs = synth.sign_mask(D, "tq4", sign_seed) if fmt == K.FMT_TQ4 else None
    g = K.Cache(fmt, Hk, D, ps, n_pages, device=DEV, rope_dim=rope, signs=signs)
    ofmt = {K.FMT_Q4_HAD32: O.Q4, K.FMT_BF16: O.BF16, K.FMT_FP8_ROW: O.FP8, K.FMT_Q4_0: O.Q4_0,
            K.FMT_TQ4: O.TQ4}[fmt]
    o = O.Cache(ofmt, Hk, D, ps, n_pages, rope_dim=rope,
                signs=None if signs is None else signs.numpy().view(np.uint32))
    return g, o


def to_np_in(t):
    """Host copy of an input tensor for the oracle (bf16 as uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return bits_u16(t)
    return t.cpu().numpy()


def check_planes_equal(g, o):
    assert np.array_equal(g.k.cpu().numpy().view(np.uint8) if g.k.dtype == torch.uint8 else bits_u16(g.k), o.k)
    assert np.array_equal(g.v.cpu().numpy().view(np.uint8) if g.v.dtype == torch.uint8 else bits_u16(g.v), o.v)
    if o.k_scale is not None:
        if g.k_scale.dtype == torch.float16:
            assert np.array_equal(bits_u16(g.k_scale), o.k_scale)
            assert np.array_equal(bits_u16(g.v_scale), o.v_scale)
        else:
            assert np.array_equal(g.k_scale.cpu().numpy().view(np.uint32), o.k_scale.view(np.uint32))
            assert np.array_equal(g.v_scale.cpu().numpy().view(np.uint32), o.v_scale.view(np.uint32))


def fill_sequence(K, g, o, k, v, bt_row, T, status=None):
    ps = g.page_size
    slots = np.array([bt_row[j // ps] * ps + j % ps for j in range(T)], np.int32)
    K.store(g, k.to(DEV), None if v is None else v.to(DEV), torch.from_numpy(slots).to(DEV), status=status)
    O.store(o, to_np_in(k), None if v is None else to_np_in(v), slots)


# --------------------------------------------------------------------------- store

@pytest.mark.parametrize("fmt", ["Q4_HAD32", "Q4_0"])
@pytest.mark.parametrize("reps", [40, 1])  # 40: > 256 rows, the row kernel; 1: the (row, group) kernel
def test_store_code_ties_round_half_to_even(K, fmt, reps):
    """Codes exactly on rounding ties (y / s = k + 1/2 for k = -8 .. 7, exact
    scales): both store kernels keep the even neighbour and clamp +7.5 to code
    15, bit-exact with the oracle and with the literal table of the expected
    codes."""
    from tests import tie_rows
    if fmt == "Q4_0":
        x, exp = tie_rows.unrotated_rows()
        gfmt = K.FMT_Q4_0
    else:
        x, exp, _, _ = tie_rows.rotated_rows()
        gfmt = K.FMT_Q4_HAD32
    x = np.tile(x, (reps, 1))
    exp = np.tile(exp, (reps, 1))
    n, D = x.shape
    ps = 16
    n_pages = (n + ps - 1) // ps
    g, o = make_cache_pair(K, gfmt, 1, D, ps, n_pages)
    kt = torch.from_numpy(x.reshape(n, 1, D))
    vt = torch.from_numpy(-x.reshape(n, 1, D))
    fill_sequence(K, g, o, kt, vt, np.arange(n_pages, dtype=np.int32), n)
    torch.cuda.synchronize()
    check_planes_equal(g, o)
    kb = g.k.cpu().numpy().reshape(-1, D // 2)[:n]
    codes = np.stack([kb & 15, kb >> 4], -1).reshape(n, D).astype(np.int64)
    tie = exp >= 0
    assert np.array_equal(codes[tie], exp[tie])


@pytest.mark.parametrize("reps", [200, 1])  # 200 rows x (K, V) > 256: the bulk kernel; 1: the (row, group) kernel
def test_store_codes_near_ties_bit_exact(K, reps):
    """Quotients y / s within 1 .. 3 ulps of every half-integer, for the scale 1
    and 0.8125 (unrotated rows, so y is the input): the code depends on the
    last bit of the IEEE-rounded quotient; both store kernels must match the
    oracle bit for bit."""
    from tests import tie_rows
    x = np.tile(tie_rows.near_tie_rows(), (reps, 1))
    n, D = x.shape
    ps = 16
    n_pages = (n + ps - 1) // ps
    g, o = make_cache_pair(K, K.FMT_Q4_0, 1, D, ps, n_pages)
    fill_sequence(K, g, o, torch.from_numpy(x.reshape(n, 1, D)), torch.from_numpy(-x.reshape(n, 1, D)),
                  np.arange(n_pages, dtype=np.int32), n)
    torch.cuda.synchronize()
    check_planes_equal(g, o)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [250, 20])  # large stores take the row kernel, small ones the (row, group) kernel
def test_store_q4_bit_exact(K, D, dtype, T):
    Hk, ps, n_pages = 3, 32, 9
    k = synth.outlier_normal((T, Hk, D), 4, 20.0, "cpu", D, "k").to(dtype)
    v = synth.heavy_tailed((T, Hk, D), "cpu", D, "v").to(dtype)
    g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, ps, n_pages)
    bt = synth.page_permutation(n_pages, D, "pages").numpy().astype(np.int32)
    fill_sequence(K, g, o, k, v, bt, T)
    torch.cuda.synchronize()
    check_planes_equal(g, o)


@pytest.mark.parametrize("fmt", ["Q4_HAD32", "Q4_0"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_store_q4_bulk_ragged_and_unaligned(K, fmt, D, dtype):
    """The bulk store (8 groups per warp): a row count that leaves the last warp
    and block part-empty, inputs that start off a 16-byte boundary (element
    loads instead of vector loads), negative slots (skipped) among valid ones;
    bit-exact with the oracle."""
    Hk, ps, T = 3, 16, 173
    n_pages = (T + ps - 1) // ps + 1
    gfmt = K.FMT_Q4_HAD32 if fmt == "Q4_HAD32" else K.FMT_Q4_0
    base_k = synth.outlier_normal((T + 1, Hk, D), 4, 20.0, "cpu", D, "uk").to(dtype).reshape(-1)
    base_v = synth.heavy_tailed((T + 1, Hk, D), "cpu", D, "uv").to(dtype).reshape(-1)
    for off in (0, 1):
        k = base_k[off:off + T * Hk * D].view(T, Hk, D)
        v = base_v[off:off + T * Hk * D].view(T, Hk, D)
        g, o = make_cache_pair(K, gfmt, Hk, D, ps, n_pages)
        slots = np.arange(T, dtype=np.int32)
        slots[::7] = -1                               # skipped tokens
        kd, vd = base_k.to(DEV)[off:off + T * Hk * D].view(T, Hk, D), base_v.to(DEV)[off:off + T * Hk * D].view(T, Hk, D)
        assert (kd.data_ptr() % 16 == 0) == (off == 0)
        K.store(g, kd, vd, torch.from_numpy(slots).to(DEV))
        O.store(o, to_np_in(k), to_np_in(v), slots)
        torch.cuda.synchronize()
        check_planes_equal(g, o)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [250, 20])
def test_store_q4_0_bit_exact(K, dtype, T):
    """The unrotated 4-bit format: codes and scales bit-exact with the oracle,
    through the row kernel (250 tokens) and the (row, group) kernel (20)."""
    Hk, D, ps, n_pages = 3, 256, 32, 9
    k = synth.outlier_normal((T, Hk, D), 4, 20.0, "cpu", D, "k0").to(dtype)
    v = synth.heavy_tailed((T, Hk, D), "cpu", D, "v0").to(dtype)
    g, o = make_cache_pair(K, K.FMT_Q4_0, Hk, D, ps, n_pages)
    bt = synth.page_permutation(n_pages, D, "pages0").numpy().astype(np.int32)
    fill_sequence(K, g, o, k, v, bt, T)
    torch.cuda.synchronize()
    check_planes_equal(g, o)


def test_store_q4_0_exact_scale_block(K):
    """Q4_0 exact-scale rows (amax 8 -> scale 1.0): the stored codes are the inputs
    plus 8, with no rotation in between."""
    Hk, D, ps = 1, 256, 16
    c = np.random.default_rng(5).integers(-8, 8, (3, Hk, D))
    c.reshape(3, 8, 32)[:, :, 0] = -8
    g = K.Cache(K.FMT_Q4_0, Hk, D, ps, 1, device=DEV)
    K.store(g, torch.from_numpy(c.astype(np.float32)).to(DEV), torch.from_numpy(c.astype(np.float32)).to(DEV),
            torch.arange(3, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(g.k_scale[0, 0, :3] == 1.0)
    # group G's codes sit at bytes 16G .. 16G + 15; bytes 2h, 2h + 1 hold elements
    # 32G + 4h .. + 3 (low nibble first)
    st = g.k[0, 0, :3].cpu().numpy()
    for G in range(8):
        for h in range(8):
            o_ = 16 * G + 2 * h
            got = [st[:, o_] & 15, st[:, o_] >> 4, st[:, o_ + 1] & 15, st[:, o_ + 1] >> 4]
            for j in range(4):
                assert np.array_equal(got[j], c[:, 0, 32 * G + 4 * h + j] + 8)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_store_tq4_bit_exact(K, D, dtype):
    """TQ4 rows: codes and the per-row fp16 scale bit-exact with the oracle
    (rotation, sum of squares, codebook decisions in the same fp32 order)."""
    Hk, ps, n_pages, T = 3, 32, 9, 250
    k = synth.outlier_normal((T, Hk, D), 4, 20.0, "cpu", D, "tk").to(dtype)
    v = synth.heavy_tailed((T, Hk, D), "cpu", D, "tv").to(dtype)
    g, o = make_cache_pair(K, K.FMT_TQ4, Hk, D, ps, n_pages, sign_seed=D)
    bt = synth.page_permutation(n_pages, D, "tpages").numpy().astype(np.int32)
    fill_sequence(K, g, o, k, v, bt, T)
    torch.cuda.synchronize()
    check_planes_equal(g, o)


def test_store_tq4_edge_rows(K):
    """Zero rows (scale 0, code 0), tiny rows (scale underflows), huge rows (scale
    saturates at 65504) and rows built on exact levels."""
    D, Hk = 256, 1
    rng = np.random.default_rng(9)
    rows = [np.zeros(D, np.float32), np.full(D, 1e-9, np.float32),
            (rng.standard_normal(D) * 1e7).astype(np.float32), (rng.standard_normal(D) * 1e-4).astype(np.float32)]
    for _ in range(6):
        rows.append(rng.standard_normal(D).astype(np.float32))
    x = torch.from_numpy(np.stack(rows)[:, None, :])
    g, o = make_cache_pair(K, K.FMT_TQ4, Hk, D, 16, 1, sign_seed=5)
    fill_sequence(K, g, o, x, x, np.array([0], np.int32), x.shape[0])
    torch.cuda.synchronize()
    check_planes_equal(g, o)
    assert bits_u16(g.k_scale)[0, 0, 0] == 0 and np.all(g.k[0, 0, 0].cpu().numpy() == 0)
    assert bits_u16(g.k_scale)[0, 0, 2] == 0x7BFF


@pytest.mark.parametrize("inverse", [False, True])
def test_tq4_rotate_matches_the_definition(K, inverse):
    D = 256
    signs = synth.sign_mask(D, "rot")
    c = K.Cache(K.FMT_TQ4, 1, D, 16, 1, device=DEV, signs=signs)
    x = synth.heavy_tailed((37, D), "cpu", "rotx", dtype=torch.float32)
    y = K.tq4_rotate(c, x.to(DEV), inverse=inverse).cpu().numpy()
    s = signs.numpy().view(np.uint32)
    for r in range(x.shape[0]):
        ref = O.tq4_rotate_f64(x[r].numpy(), s, inverse=inverse)
        assert np.abs(y[r] - ref).max() <= 1e-6 * np.abs(ref).max()


def test_store_q4_exact_scale_and_edge_rows(K):
    """Exact-scale rows (codes equal the inputs), zero rows, tiny rows, huge rows."""
    D, Hk = 256, 1
    rows = []
    rng = np.random.default_rng(5)
    for _ in range(8):
        c = rng.integers(-8, 8, D)
        c.reshape(8, 32)[:, 3] = -8
        rows.append(O.hadamard32_f64(c.astype(np.float64)).astype(np.float32))
    rows.append(np.zeros(D, np.float32))
    rows.append(np.full(D, 1e-9, np.float32))
    rows.append((rng.standard_normal(D) * 1e6).astype(np.float32))
    rows.append((rng.standard_normal(D) * 1e-5).astype(np.float32))
    x = torch.from_numpy(np.stack(rows)[:, None, :])
    T = x.shape[0]
    g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, 16, 1)
    fill_sequence(K, g, o, x, x, np.array([0], np.int32), T)
    torch.cuda.synchronize()
    check_planes_equal(g, o)
    assert np.all(bits_u16(g.k_scale)[0, 0, :8] == 0x3C00)   # scale 1.0


def test_store_skips_negative_and_flags_bad_slots(K):
    D, Hk, ps = 64, 2, 16
    g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, ps, 2)
    k = synth.normal((4, Hk, D), "cpu", "k")
    slots = torch.tensor([3, -1, 40, 17], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    K.store(g, k.to(DEV), k.to(DEV), slots.to(DEV), status=st)
    torch.cuda.synchronize()
    assert K.read_status(st) & K.DEV_BAD_SLOT
    assert O.store(o, k.numpy(), k.numpy(), slots.numpy()) == 1
    check_planes_equal(g, o)


def test_store_one_at_a_time_equals_batch(K):
    D, Hk, ps, T = 256, 4, 16, 70
    k = synth.heavy_tailed((T, Hk, D), "cpu", 7, "k")
    v = synth.heavy_tailed((T, Hk, D), "cpu", 7, "v")
    g1 = K.Cache(K.FMT_Q4_HAD32, Hk, D, ps, 5, device=DEV)
    g2 = K.Cache(K.FMT_Q4_HAD32, Hk, D, ps, 5, device=DEV)
    slots = torch.arange(T, dtype=torch.int32, device=DEV)
    K.store(g1, k.to(DEV), v.to(DEV), slots)
    for j in range(T):
        K.store(g2, k[j:j + 1].to(DEV), v[j:j + 1].to(DEV), slots[j:j + 1])
    torch.cuda.synchronize()
    assert torch.equal(g1.k, g2.k) and torch.equal(g1.v, g2.v)
    assert torch.equal(g1.k_scale.view(torch.int16), g2.k_scale.view(torch.int16))


def test_store_fp8_bit_exact(K):
    T, D, R, ps = 300, 512, 64, 16
    rows = synth.latent_rows(T, D + R, "cpu", "fp8")
    rows[5] = 0.0                       # zero row
    rows[6] = 1e-40                     # subnormal amax (448/amax overflows)
    rows[7, :D] = torch.linspace(-500, 500, D)
    g, o = make_cache_pair(K, K.FMT_FP8_ROW, 1, D, ps, 20, rope=R)
    bt = synth.page_permutation(20, "fp8pages").numpy().astype(np.int32)
    fill_sequence(K, g, o, rows, None, bt, T)
    torch.cuda.synchronize()
    check_planes_equal(g, o)


def test_store_bf16_bit_exact(K):
    T, Hk, D = 100, 4, 256
    k = synth.outlier_normal((T, Hk, D), 4, 20.0, "cpu", "bk")
    v = synth.outlier_normal((T, Hk, D), 4, 20.0, "cpu", "bv")
    g, o = make_cache_pair(K, K.FMT_BF16, Hk, D, 16, 7)
    fill_sequence(K, g, o, k, v, np.arange(7, dtype=np.int32), T)
    torch.cuda.synchronize()
    check_planes_equal(g, o)


def test_rotate_query(K):
    x = synth.heavy_tailed((5, 24, 256), "cpu", "rq")
    y = K.rotate_query(x.to(DEV)).cpu().numpy().astype(np.float64)
    ref = O.hadamard32_f64(x.float().numpy().astype(np.float64).reshape(-1)).reshape(y.shape)
    assert np.abs(y - ref).max() <= 1e-5 * np.abs(ref).max()
    xf = synth.normal((3, 64), "cpu", "rq2").to(DEV)
    K.rotate_query(xf, out=xf)   # in place
    assert np.allclose(xf.cpu().numpy(), O.hadamard32_f64(synth.normal((3, 64), "cpu", "rq2").numpy().astype(
        np.float64).reshape(-1)).reshape(3, 64), atol=1e-5)


def test_store_rotate_equals_store_then_rotate(K):
    """The fused launch writes the same cache bytes as the oracle's store and the
    same rotated queries as kvq_rotate_query, bit for bit; skipped slots and a
    bad slot behave as in kvq_store."""
    Hk, D, ps, n_pages = 4, 256, 16, 6
    for n_tok, qdt in ((1, torch.bfloat16), (32, torch.float32)):
        g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, ps, n_pages)
        k = synth.heavy_tailed((n_tok, Hk, D), "cpu", "sr", n_tok, "k").to(torch.bfloat16)
        v = synth.heavy_tailed((n_tok, Hk, D), "cpu", "sr", n_tok, "v").to(torch.bfloat16)
        slots = np.arange(n_tok, dtype=np.int32) * 3 % (n_pages * ps)
        if n_tok > 1:
            slots[1] = -1                  # skipped
            slots[2] = n_pages * ps + 5    # out of range: skipped, flagged
        q = synth.heavy_tailed((5, 24, D), "cpu", "srq", n_tok).to(qdt)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        qr = K.store_rotate(g, k.to(DEV), v.to(DEV), torch.from_numpy(slots).to(DEV), q.to(DEV), status=status)
        O.store(o, to_np_in(k), to_np_in(v), slots)
        check_planes_equal(g, o)
        assert torch.equal(qr, K.rotate_query(q.to(DEV)))
        assert (int(status.item()) != 0) == (n_tok > 1)


# --------------------------------------------------------------------------- decode

def decode_case(K, lens, Hk=4, Hq=24, D=256, ps=16, fmt=None, seed=0, dtype=torch.bfloat16, shuffle=True, gen="heavy"):
    fmt = K.FMT_Q4_HAD32 if fmt is None else fmt
    B = len(lens)
    pages_per = [(L + ps - 1) // ps for L in lens]
    n_pages = sum(pages_per) + 2
    max_pages = max(max(pages_per), 1)
    perm = synth.page_permutation(n_pages, seed, "perm").numpy().astype(np.int32) if shuffle else \
        np.arange(n_pages, dtype=np.int32)
    bt = np.zeros((B, max_pages), np.int32)
    off = 0
    for b, npg in enumerate(pages_per):
        bt[b, :npg] = perm[off:off + npg]
        off += npg
    g, o = make_cache_pair(K, fmt, Hk, D, ps, n_pages, sign_seed=seed)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        if gen == "heavy":
            k = synth.heavy_tailed((L, Hk, D), "cpu", seed, b, "k", dtype=dtype)
            v = synth.heavy_tailed((L, Hk, D), "cpu", seed, b, "v", dtype=dtype)
        else:
            k = synth.outlier_normal((L, Hk, D), 4, 20.0, "cpu", seed, b, "k").to(dtype)
            v = synth.outlier_normal((L, Hk, D), 4, 20.0, "cpu", seed, b, "v").to(dtype)
        fill_sequence(K, g, o, k, v, bt[b], L)
    if gen == "heavy":
        q = synth.heavy_tailed((B, Hq, D), "cpu", seed, "q", dtype=dtype)
    else:
        q = synth.outlier_normal((B, Hq, D), 4, 20.0, "cpu", seed, "q").to(dtype)
    return g, o, bt, q, max(max(lens), 1)


def run_decode(K, g, bt, q, lens, max_len, sm_scale, sel=None):
    B, Hq = q.shape[0], q.shape[1]
    ws = K.alloc_workspace(g, B, Hq, max_len, 0 if sel is None else sel.shape[1], device=DEV)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = K.decode(g, q.to(DEV), seq, torch.from_numpy(bt).to(DEV), max_len, sm_scale, ws,
                   sel=None if sel is None else torch.from_numpy(sel).to(DEV))
    torch.cuda.synchronize()
    return out.cpu().numpy(), ws


def test_decode_tiny_config(K):
    """1 sequence, 1024 keys, 4 KV / 24 query heads, head_dim 256, fp32 inputs with x20 outliers."""
    lens = [1024]
    g, o, bt, q, ml = decode_case(K, lens, dtype=torch.float32, gen="outlier", shuffle=False)
    torch.cuda.synchronize()
    check_planes_equal(g, o)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
    assert_close(out[0], ref[0], what="tiny decode")


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 127, 128, 129, 511, 512, 513, 1025, 4097])
def test_decode_lengths(K, T):
    g, o, bt, q, ml = decode_case(K, [T], seed=T)
    out, _ = run_decode(K, g, bt, q, [T], ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), [T], bt, 1 / 16)
    assert_close(out[0], ref[0], what=f"T={T}")


def test_decode_ragged_paged_batch(K):
    lens = [1, 700, 33, 2048, 1500, 0, 513, 3000]
    g, o, bt, q, ml = decode_case(K, lens, seed=11)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
    for b in range(len(lens)):
        if lens[b] == 0:
            assert np.all(out[b] == 0)
        else:
            assert_close(out[b], ref[b], what=f"seq {b}")


@pytest.mark.parametrize("Hk,Hq", [(1, 1), (2, 4), (1, 8), (8, 8), (3, 21)])
def test_decode_gqa_groups(K, Hk, Hq):
    lens = [900, 77]
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, seed=Hk * 100 + Hq)
    out, _ = run_decode(K, g, bt, q, lens, ml, 0.07)
    ref = O.decode(o, to_np_in(q), lens, bt, 0.07)
    for b in range(2):
        assert_close(out[b], ref[b], what=f"Hk={Hk} Hq={Hq} seq {b}")


@pytest.mark.parametrize("lens", [[1200, 530, 4100], [40000, 512, 38001, 39999, 20000]])
def test_decode_concurrent_equals_solo_and_deterministic(K, lens):
    """A batched sequence equals its solo decode bit for bit, for a small batch
    and for one whose grid (over two waves) is far larger than any of its
    sequences' alone."""
    g, o, bt, q, ml = decode_case(K, lens, seed=3)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    out2, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    assert np.array_equal(out, out2)
    for b in range(len(lens)):
        solo, _ = run_decode(K, g, bt[b:b + 1], q[b:b + 1], [lens[b]], lens[b], 1 / 16)
        assert np.array_equal(solo[0], out[b])


@pytest.mark.parametrize("Hk,Hq,L", [(4, 24, 100001), (4, 24, 78337), (8, 16, 40000), (2, 12, 160000)])
def test_decode_long_sequence_equals_batched(K, Hk, Hq, L):
    """One sequence whose grid is over one wave of four CTAs per SM (several
    waves, the last one partial) gives the same bits alone and next to a short
    sequence, and the same bits twice.  Partitions per KV head: 196 (the last of
    161 keys), 154 (the last of 1 key), 79 (8 KV heads: the last of 64 keys) and
    313 (2 KV heads: the last of 256 keys)."""
    lens = [L, 600]
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, seed=78)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    solo, _ = run_decode(K, g, bt[:1], q[:1], [L], L, 1 / 16)
    solo2, _ = run_decode(K, g, bt[:1], q[:1], [L], L, 1 / 16)
    assert np.array_equal(solo, solo2)
    assert np.array_equal(solo[0], out[0])


def test_decode_bad_page_in_a_late_wave(K):
    """A bad block-table entry in a partition of a later wave of a long
    sequence's decode: flagged, the sequence's outputs NaN, and the next decode
    unaffected."""
    L = 100001
    g, o, bt, q, ml = decode_case(K, [L], seed=79)
    good, _ = run_decode(K, g, bt, q, [L], L, 1 / 16)
    bad_bt = bt.copy()
    bad_bt[0, (170 * 512 + 40) // g.page_size] = -3  # partition 170 of 196 (KV head 3: CTA 758, in the second wave of 608)
    out, ws = run_decode(K, g, bad_bt, q, [L], L, 1 / 16)
    assert K.read_status(ws) & K.DEV_BAD_PAGE
    assert np.isnan(out[0]).all()
    again, _ = run_decode(K, g, bt, q, [L], L, 1 / 16)
    assert np.array_equal(again, good)


@pytest.mark.parametrize("L", [32769, 16383 + 200, 1337])
def test_decode_warp_specialised_equals_round_kernel(K, L):
    """A grid that fits in one wave of two CTAs per SM (the sequence alone) runs
    the warp-specialised kernel; next to a 40000-key sequence (79 partitions x 4
    KV heads x 2 sequences, over two CTAs per SM) it runs the round kernel.  The
    two give the same bits.  The last partition holds 1, 199 and 313 keys (tail
    rounds of 1, 5 and 4 tiles)."""
    lens = [L, 40000]
    g, o, bt, q, ml = decode_case(K, lens, seed=77)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    solo, _ = run_decode(K, g, bt[:1], q[:1], [L], L, 1 / 16)
    assert np.array_equal(solo[0], out[0])
    if L < 2000:
        ref = O.decode(o, to_np_in(q[:1]), [L], bt[:1], 1 / 16)
        assert_close(solo[0], ref[0], what=f"warp-specialised L={L}")


def _partials(ws, B, Hq, T, P_keys=512):
    """The status word and the partials (m, z, acc) of a 4-bit decode workspace
    ([256-byte header][m][z][acc], each area rounded up to 256 bytes, as the
    workspace-size test pins): the area after them is scratch (the fused
    merge's counters and block partials, or the queries a multi-wave decode
    rotated into it)."""
    n = B * Hq * max(1, -(-T // P_keys))
    r = lambda x: (x + 255) // 256 * 256
    return ws[:256 + 2 * r(4 * n) + r(4 * n * 256)].view(torch.int32)


def _clone_q4_cache(K, g):
    c = K.Cache(g.fmt, g.Hk, g.D, g.page_size, g.num_pages, device=DEV)
    for name in ("k", "v", "k_scale", "v_scale"):
        getattr(c, name).copy_(getattr(g, name))
    return c


@pytest.mark.parametrize("fmt", ["Q4_HAD32", "Q4_0"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lens", [[32769], [1], [512], [513], [1025, 9000, 700, 4097], [40000, 38001, 512, 20000],
                                  [100001]])
def test_decode_step_equals_store_rotate_decode(K, fmt, dtype, lens):
    """kvq_decode_step (store the new token inside the decode, rotate the query in
    the kernel) gives the same partials and the same cache planes, bit for bit, as
    kvq_store + kvq_rotate_query + kvq_decode_attn.  The new position falls at a
    partition's start (1, 513, 1025, 9000 -> 8999 = 17 * 512 + 295: mid), its end
    (512) and after a full partition (32769: a partition of one key); the first
    lists run the warp-specialised kernel on the unrotated query, the last two (a
    grid over two CTAs per SM) one rotation launch and then the round kernel (for
    the single 100001-key sequence, whose new position's partition 195 runs
    in the grid's second wave)."""
    f = K.FMT_Q4_HAD32 if fmt == "Q4_HAD32" else K.FMT_Q4_0
    g, o, bt, q, ml = decode_case(K, lens, fmt=f, seed=91, dtype=dtype)
    g2 = _clone_q4_cache(K, g)
    B, Hk, D = len(lens), g.Hk, g.D
    k_new = synth.heavy_tailed((B, Hk, D), "cpu", 91, "knew", dtype=dtype).to(DEV)
    v_new = synth.heavy_tailed((B, Hk, D), "cpu", 91, "vnew", dtype=dtype).to(DEV)
    qd = q.to(DEV)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    btd = torch.from_numpy(bt).to(DEV)
    ps = g.page_size
    slots = torch.tensor([int(bt[b, (L - 1) // ps]) * ps + (L - 1) % ps for b, L in enumerate(lens)],
                         dtype=torch.int32, device=DEV)
    ws1 = K.alloc_workspace(g, B, qd.shape[1], ml, device=DEV)
    ws2 = K.alloc_workspace(g, B, qd.shape[1], ml, device=DEV)
    K.decode_step(g, k_new, v_new, qd, seq, btd, ml, 1 / 16, ws1)
    K.store(g2, k_new, v_new, slots)
    qr = K.rotate_query(qd) if f == K.FMT_Q4_HAD32 else qd.float()
    K.decode_attn(g2, qr, seq, btd, ml, 1 / 16, ws2)
    torch.cuda.synchronize()
    for name in ("k", "v", "k_scale", "v_scale"):
        assert torch.equal(getattr(g, name).view(torch.uint8), getattr(g2, name).view(torch.uint8)), name
    assert torch.equal(_partials(ws1, B, qd.shape[1], ml), _partials(ws2, B, qd.shape[1], ml))
    if max(lens) < 2000:  # the merged rows against the oracle over the same cache
        out = torch.empty((B, qd.shape[1], D), dtype=torch.float32, device=DEV)
        K.merge(g, ws1, B, qd.shape[1], seq, ml, out)
        O.store(o, to_np_in(k_new.cpu()), to_np_in(v_new.cpu()), slots.cpu().numpy())
        ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
        for b in range(B):
            assert_close(out[b].cpu().numpy(), ref[b], what=f"decode_step seq {b}")


@pytest.mark.parametrize("Hk,Hq", [(2, 4), (3, 21), (8, 8), (1, 8)])
@pytest.mark.parametrize("lens", [[1025, 9000, 700], [100001]])
def test_decode_step_gqa_layouts(K, Hk, Hq, lens):
    """kvq_decode_step for other GQA layouts (groups of 2, 7, 1 and 8 heads):
    the cache planes and the partials bit-identical to kvq_store +
    kvq_rotate_query + kvq_decode_attn.  The cases' grids fall on both sides of
    one wave of two CTAs per SM (the warp-specialised kernel; or a rotation
    launch, then the round kernel, which stores the new token)."""
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, seed=93 + Hq)
    g2 = _clone_q4_cache(K, g)
    B, D = len(lens), g.D
    k_new = synth.heavy_tailed((B, Hk, D), "cpu", 93, "knew").to(DEV)
    v_new = synth.heavy_tailed((B, Hk, D), "cpu", 93, "vnew").to(DEV)
    qd = q.to(DEV)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    btd = torch.from_numpy(bt).to(DEV)
    ps = g.page_size
    slots = torch.tensor([int(bt[b, (L - 1) // ps]) * ps + (L - 1) % ps for b, L in enumerate(lens)],
                         dtype=torch.int32, device=DEV)
    ws1 = K.alloc_workspace(g, B, Hq, ml, device=DEV)
    ws2 = K.alloc_workspace(g, B, Hq, ml, device=DEV)
    K.decode_step(g, k_new, v_new, qd, seq, btd, ml, 1 / 16, ws1)
    K.store(g2, k_new, v_new, slots)
    K.decode_attn(g2, K.rotate_query(qd), seq, btd, ml, 1 / 16, ws2)
    torch.cuda.synchronize()
    for name in ("k", "v", "k_scale", "v_scale"):
        assert torch.equal(getattr(g, name).view(torch.uint8), getattr(g2, name).view(torch.uint8)), name
    assert torch.equal(_partials(ws1, B, Hq, ml), _partials(ws2, B, Hq, ml))


def test_decode_step_with_an_empty_sequence(K):
    """A sequence of length 0 in a decode step stores nothing and its outputs
    are zeros; the others' planes and partials equal kvq_store (slot -1 for the
    empty one: skipped) + kvq_rotate_query + kvq_decode_attn."""
    lens = [0, 700, 513]
    g, o, bt, q, ml = decode_case(K, lens, seed=95)
    g2 = _clone_q4_cache(K, g)
    B, Hk, D, Hq = len(lens), g.Hk, g.D, q.shape[1]
    k_new = synth.heavy_tailed((B, Hk, D), "cpu", 95, "knew").to(DEV)
    v_new = synth.heavy_tailed((B, Hk, D), "cpu", 95, "vnew").to(DEV)
    qd = q.to(DEV)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    btd = torch.from_numpy(bt).to(DEV)
    ps = g.page_size
    slots = torch.tensor([int(bt[b, (L - 1) // ps]) * ps + (L - 1) % ps if L > 0 else -1 for b, L in enumerate(lens)],
                         dtype=torch.int32, device=DEV)
    ws1 = K.alloc_workspace(g, B, Hq, ml, device=DEV)
    ws2 = K.alloc_workspace(g, B, Hq, ml, device=DEV)
    K.decode_step(g, k_new, v_new, qd, seq, btd, ml, 1 / 16, ws1)
    K.store(g2, k_new, v_new, slots)
    K.decode_attn(g2, K.rotate_query(qd), seq, btd, ml, 1 / 16, ws2)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=DEV)
    K.merge(g, ws1, B, Hq, seq, ml, out)
    torch.cuda.synchronize()
    for name in ("k", "v", "k_scale", "v_scale"):
        assert torch.equal(getattr(g, name).view(torch.uint8), getattr(g2, name).view(torch.uint8)), name
    assert torch.equal(_partials(ws1, B, Hq, ml), _partials(ws2, B, Hq, ml))
    assert K.read_status(ws1) == 0
    assert torch.count_nonzero(out[0]) == 0 and torch.isfinite(out[1:]).all()


def test_decode_step_bad_page_flags_and_stores_nothing(K):
    """A new position mapped to a page outside the pool: nothing is written, the
    decode flags KVQ_DEV_BAD_PAGE and the sequence's outputs are NaN."""
    lens = [700, 300]
    g, o, bt, q, ml = decode_case(K, lens, seed=92)
    before = [getattr(g, n).clone() for n in ("k", "v", "k_scale", "v_scale")]
    bt = bt.copy()
    bt[0, (lens[0] - 1) // g.page_size] = g.num_pages + 5
    B, Hk, D = 2, g.Hk, g.D
    k_new = synth.heavy_tailed((B, Hk, D), "cpu", 92, "knew").to(DEV)
    v_new = synth.heavy_tailed((B, Hk, D), "cpu", 92, "vnew").to(DEV)
    # the second sequence's new position is written (its page is good); compare the first's pages only
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ws = K.alloc_workspace(g, B, q.shape[1], ml, device=DEV)
    K.decode_step(g, k_new, v_new, q.to(DEV), seq, torch.from_numpy(bt).to(DEV), ml, 1 / 16, ws)
    out = torch.empty((B, q.shape[1], D), dtype=torch.float32, device=DEV)
    K.merge(g, ws, B, q.shape[1], seq, ml, out)
    torch.cuda.synchronize()
    assert K.read_status(ws) & K.DEV_BAD_PAGE
    assert torch.isnan(out[0]).all() and torch.isfinite(out[1]).all()
    pages0 = set(int(x) for x in bt[0, : (lens[0] + g.page_size - 1) // g.page_size] if 0 <= x < g.num_pages)
    for t0, name in zip(before, ("k", "v", "k_scale", "v_scale")):
        t1 = getattr(g, name)
        for pg in pages0:
            assert torch.equal(t0[pg], t1[pg]), name


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("Hk,Hq", [(4, 24), (2, 4), (3, 21)])
@pytest.mark.parametrize("lens", [[1500, 700], [40000, 38001]])
def test_decode_unrotated_query_equals_rotate_then_decode(K, dtype, Hk, Hq, lens):
    """The in-kernel query rotation gives the same partials, bit for bit (dense and
    gathered); the longer lengths make a dense grid of more than two CTAs per SM,
    which rotates in a launch of its own first."""
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, seed=500 + Hq, dtype=dtype)
    qd = q.to(DEV)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    btd = torch.from_numpy(bt).to(DEV)
    sel = torch.from_numpy(np.stack([synth.distinct_sorted(300, L, 5, b).numpy() for b, L in enumerate(lens)])
                           .astype(np.int32)).to(DEV)
    for s_ in (None, sel):
        n_sel = 0 if s_ is None else s_.shape[1]
        ws1 = K.alloc_workspace(g, 2, Hq, ml, n_sel, device=DEV)
        ws2 = K.alloc_workspace(g, 2, Hq, ml, n_sel, device=DEV)
        K.decode_attn(g, K.rotate_query(qd), seq, btd, ml, 1 / 16, ws1, sel=s_)
        K.decode_attn_unrotated(g, qd, seq, btd, ml, 1 / 16, ws2, sel=s_)
        torch.cuda.synchronize()
        T = ml if s_ is None else n_sel
        assert torch.equal(_partials(ws1, 2, Hq, T), _partials(ws2, 2, Hq, T))


def test_decode_gather(K):
    lens = [3000, 1800]
    g, o, bt, q, ml = decode_case(K, lens, seed=21)
    for n_sel in (1, 100, 512, 1300):
        sel = np.stack([synth.distinct_sorted(n_sel, L, 21, b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
        out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16, sel=sel)
        ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16, sel=sel)
        for b in range(2):
            assert_close(out[b], ref[b], what=f"gather n_sel={n_sel} seq {b}")


def test_decode_gather_solo_equals_batched(K):
    """A gather's partials do not depend on the kernel that runs it: one
    sequence's selection (8 partitions x 4 KV heads, a grid of one wave: the
    warp-specialised kernel) equals the same sequence's rows in a batch of ten
    (320 CTAs: the round kernel), bit for bit, for a full and a ragged
    selection."""
    lens = [5000 + 37 * b for b in range(10)]
    g, o, bt, q, ml = decode_case(K, lens, seed=24)
    for n_sel in (4096, 1300):
        sel = np.stack([synth.distinct_sorted(n_sel, L, 24, b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
        out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16, sel=sel)
        for b in (0, 7):
            solo, _ = run_decode(K, g, bt[b:b + 1], q[b:b + 1], [lens[b]], lens[b], 1 / 16, sel=sel[b:b + 1])
            assert np.array_equal(solo[0], out[b]), (n_sel, b)


def test_decode_gather_bad_index_and_bad_page(K):
    """A selected position outside its sequence (past its length, or negative)
    and a selected row on a page outside the pool: each is flagged, the
    sequence's outputs are NaN, and the other sequence matches the oracle.  The
    bad entries sit mid-partition (entry 700 of 1300: partition 1, tile 11),
    so the CTA's other rows are resolved and copied as usual."""
    lens = [3000, 1800]
    g, o, bt, q, ml = decode_case(K, lens, seed=22)
    n_sel = 1300
    sel = np.stack([synth.distinct_sorted(n_sel, L, 22, b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16, sel=sel)
    for bad_pos, flag in ((lens[0] + 7, K.DEV_BAD_INDEX), (-3, K.DEV_BAD_INDEX)):
        s1 = sel.copy()
        s1[0, 700] = bad_pos
        out, ws = run_decode(K, g, bt, q, lens, ml, 1 / 16, sel=s1)
        assert K.read_status(ws) & flag
        assert np.isnan(out[0]).all()
        assert_close(out[1], ref[1], what=f"healthy sequence next to a bad index {bad_pos}")
    bt2 = bt.copy()
    bt2[1, int(sel[1, 700]) // g.page_size] = g.num_pages + 3
    out, ws = run_decode(K, g, bt2, q, lens, ml, 1 / 16, sel=sel)
    assert K.read_status(ws) & K.DEV_BAD_PAGE
    assert np.isnan(out[1]).all()
    assert_close(out[0], ref[0], what="healthy sequence next to a bad page")


def test_decode_gather_at_the_limit(K):
    """4096 selected rows, the largest list the ABI accepts: eight full 512-entry
    partitions; the second sequence selects every one of its 4096 rows."""
    lens = [9000, 4096]
    g, o, bt, q, ml = decode_case(K, lens, seed=23)
    sel = np.stack([synth.distinct_sorted(4096, L, 23, b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
    assert np.array_equal(sel[1], np.arange(4096))
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16, sel=sel)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16, sel=sel)
    for b in range(2):
        assert_close(out[b], ref[b], what=f"gather n_sel=4096 seq {b}")


@pytest.mark.parametrize("lens", [[1], [17, 513], [1025, 3000]])
def test_decode_q4_0(K, lens):
    """The unrotated 4-bit format through the same decode kernel and merge (no
    rotation anywhere), against the oracle; also the unrotated-query entry point,
    which must leave the query as given."""
    g, o, bt, q, ml = decode_case(K, lens, fmt=K.FMT_Q4_0, seed=31)
    out, ws = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
    for b in range(len(lens)):
        assert_close(out[b], ref[b], what=f"Q4_0 seq {b}")
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ws2 = K.alloc_workspace(g, len(lens), q.shape[1], ml, device=DEV)
    K.decode_attn_unrotated(g, q.to(DEV), seq, torch.from_numpy(bt).to(DEV), ml, 1 / 16, ws2)
    torch.cuda.synchronize()
    assert torch.equal(ws, ws2)


def test_decode_q4_0_gather(K):
    lens = [2000, 700]
    g, o, bt, q, ml = decode_case(K, lens, fmt=K.FMT_Q4_0, seed=33)
    sel = np.stack([synth.distinct_sorted(300, L, 33, b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16, sel=sel)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16, sel=sel)
    for b in range(2):
        assert_close(out[b], ref[b], what=f"Q4_0 gather seq {b}")


# R rows of a GQA group of 6 fill ceil(6 R / 8) column tiles of one CTA (at most
# 4, i.e. 5 rows); more rows are cut into even slices: R = 1 .. 5 cover 1 .. 4
# tiles (R = 3 with dead columns), R = 6 two slices of 3, R = 8 two of 4, R = 20
# four of 5.  T0 = 510 puts the rows' ends on both sides of a partition edge.
@pytest.mark.parametrize("T0,R", [(1000, 4), (513, 3), (40, 8), (0, 2), (300, 1), (510, 5), (100, 6),
                                  (2000, 20), (4095, 2), (3000, 64)])   # 64: the maximum window (13 slices of 5 rows)
def test_decode_window_equals_plain_rows(K, T0, R):
    """A decode window (R draft rows of one sequence sharing its block table, row i
    attending keys 0 .. T0 + i) gives bit-identical partials and outputs to the
    plain batched decode of R sequences with those lengths and the block table
    repeated, and matches the oracle."""
    g, o, bt, _, _ = decode_case(K, [T0 + R], seed=40 + R)
    q = synth.heavy_tailed((R, 24, 256), "cpu", "win", T0, R)
    lens = [T0 + i + 1 for i in range(R)]
    ml = T0 + R
    dev_bt = torch.from_numpy(bt).to(DEV)
    ws_w = K.alloc_workspace(g, R, 24, ml, device=DEV)
    out_w = K.decode_window_causal(g, q.to(DEV), T0, dev_bt[0], 1 / 16, ws_w)
    bt_rep = np.repeat(bt, R, axis=0)
    out_p, ws_p = run_decode(K, g, bt_rep, q, lens, ml, 1 / 16)
    torch.cuda.synchronize()
    assert torch.equal(ws_w, ws_p)
    assert np.array_equal(out_w.cpu().numpy(), out_p)
    ref = O.decode(o, to_np_in(q), lens, bt_rep, 1 / 16)
    for i in range(R):
        assert_close(out_p[i], ref[i], what=f"window row {i}")


def test_decode_window_q4_0(K):
    """Windows over the unrotated 4-bit rows: the queries used as given, the rows
    bit-identical to the plain decode and close to the oracle."""
    T0, R = 900, 5
    g, o, bt, _, _ = decode_case(K, [T0 + R], fmt=K.FMT_Q4_0, seed=55)
    q = synth.heavy_tailed((R, 24, 256), "cpu", "win0")
    lens = [T0 + i + 1 for i in range(R)]
    ml = T0 + R
    dev_bt = torch.from_numpy(bt).to(DEV)
    ws_w = K.alloc_workspace(g, R, 24, ml, device=DEV)
    out_w = K.decode_window_causal(g, q.to(DEV), T0, dev_bt[0], 1 / 16, ws_w)
    out_p, _ = run_decode(K, g, np.repeat(bt, R, axis=0), q, lens, ml, 1 / 16)
    assert np.array_equal(out_w.cpu().numpy(), out_p)
    ref = O.decode(o, to_np_in(q), lens, np.repeat(bt, R, axis=0), 1 / 16)
    for i in range(R):
        assert_close(out_p[i], ref[i], what=f"Q4_0 window row {i}")


@pytest.mark.parametrize("Hk,Hq,R", [(1, 8, 4), (1, 8, 9), (3, 9, 7), (2, 2, 33)])
def test_decode_window_gqa_groups(K, Hk, Hq, R):
    """Windows over other GQA group sizes (8: 4 rows fill the 4 column tiles; 3:
    7 rows in 3 tiles; 1: 33 rows cut into two slices) equal the plain rows."""
    T0 = 700
    g, o, bt, _, _ = decode_case(K, [T0 + R], Hk=Hk, Hq=Hq, seed=70 + R)
    q = synth.heavy_tailed((R, Hq, 256), "cpu", "wing", Hq, R)
    lens = [T0 + i + 1 for i in range(R)]
    ml = T0 + R
    dev_bt = torch.from_numpy(bt).to(DEV)
    ws_w = K.alloc_workspace(g, R, Hq, ml, device=DEV)
    out_w = K.decode_window_causal(g, q.to(DEV), T0, dev_bt[0], 0.07, ws_w)
    out_p, _ = run_decode(K, g, np.repeat(bt, R, axis=0), q, lens, ml, 0.07)
    assert np.array_equal(out_w.cpu().numpy(), out_p)
    ref = O.decode(o, to_np_in(q[:2]), lens[:2], np.repeat(bt, 2, axis=0), 0.07)
    for i in range(2):
        assert_close(out_p[i], ref[i], what=f"window row {i}")


def test_decode_window_rows_in_any_order_and_bad_row(K):
    """Row lengths need not rise with the row index; a row whose length is out of
    range is flagged and comes out NaN while the other rows still equal their
    plain decodes."""
    lens = [900, 37, 1500, 512, 513]
    R = len(lens)
    g, o, bt, _, _ = decode_case(K, [max(lens)], seed=91)
    q = synth.heavy_tailed((R, 24, 256), "cpu", "winb")
    ml = max(lens)
    dev_bt = torch.from_numpy(bt).to(DEV)
    qr = K.rotate_query(q.to(DEV))
    for bad in (None, 3):
        ll = list(lens)
        if bad is not None:
            ll[bad] = ml + 1
        dl = torch.tensor(ll, dtype=torch.int32, device=DEV)
        ws = K.alloc_workspace(g, R, 24, ml, device=DEV)
        K.decode_window(g, qr, dl, dev_bt[0], ml, 1 / 16, ws)
        out = torch.empty((R, 24, 256), dtype=torch.float32, device=DEV)
        K.merge(g, ws, R, 24, dl, ml, out)
        out = out.cpu().numpy()
        good = [i for i in range(R) if i != bad]
        out_p, _ = run_decode(K, g, np.repeat(bt, len(good), axis=0), q[good], [lens[i] for i in good], ml, 1 / 16)
        assert np.array_equal(out[good], out_p)
        if bad is None:
            assert K.read_status(ws) == 0
        else:
            assert K.read_status(ws) & K.DEV_BAD_LENGTH
            assert np.isnan(out[bad]).all()


@pytest.mark.parametrize("T", [1, 15, 17, 129, 511, 513, 4097])
def test_decode_tq4_lengths(K, T):
    """TQ4 decode (query rotation, split-T partials with the codebook levels,
    merge and the inverse rotation) against the oracle."""
    g, o, bt, q, ml = decode_case(K, [T], fmt=K.FMT_TQ4, seed=500 + T)
    out, _ = run_decode(K, g, bt, q, [T], ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), [T], bt, 1 / 16)
    assert_close(out[0], ref[0], what=f"TQ4 T={T}")


@pytest.mark.parametrize("Hk,Hq", [(1, 8), (3, 21), (2, 2)])
def test_decode_tq4_gqa_batch(K, Hk, Hq):
    lens = [700, 45, 1100]
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, fmt=K.FMT_TQ4, seed=600 + Hq)
    out, _ = run_decode(K, g, bt, q, lens, ml, 0.07)
    ref = O.decode(o, to_np_in(q), lens, bt, 0.07)
    for b in range(len(lens)):
        assert_close(out[b], ref[b], what=f"TQ4 seq {b}")


def test_store_tq4_flags_bad_slots(K):
    D, Hk, ps = 64, 2, 16
    g, o = make_cache_pair(K, K.FMT_TQ4, Hk, D, ps, 2, sign_seed=2)
    k = synth.normal((4, Hk, D), "cpu", "tqbad")
    slots = torch.tensor([3, -1, 40, 17], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    K.store(g, k.to(DEV), k.to(DEV), slots.to(DEV), status=st)
    torch.cuda.synchronize()
    assert K.read_status(st) & K.DEV_BAD_SLOT
    assert O.store(o, k.numpy(), k.numpy(), slots.numpy()) == 1
    check_planes_equal(g, o)


def test_tq4_unsupported_paths_are_refused(K):
    g, o, bt, q, ml = decode_case(K, [100], fmt=K.FMT_TQ4, seed=3)
    ws = K.alloc_workspace(g, 1, 24, ml, 4, device=DEV)
    sel = torch.arange(4, dtype=torch.int32, device=DEV).reshape(1, 4)
    with pytest.raises(K.KvqError) as e:
        K.decode_attn(g, K.tq4_rotate(g, q.to(DEV)), torch.tensor([100], dtype=torch.int32, device=DEV),
                      torch.from_numpy(bt).to(DEV), ml, 1 / 16, ws, sel=sel)
    assert e.value.status == K.ERR_UNSUPPORTED
    with pytest.raises(K.KvqError):
        K.prefill_attn(g, q.to(DEV), 0, torch.from_numpy(bt[0]).to(DEV), 1 / 16)
    with pytest.raises(K.KvqError):
        K.decode_window(g, q.to(DEV).float(), torch.tensor([100], dtype=torch.int32, device=DEV),
                        torch.from_numpy(bt[0]).to(DEV), ml, 1 / 16, ws)


def test_decode_bad_page_and_length_are_flagged(K):
    lens = [600, 300]
    g, o, bt, q, ml = decode_case(K, lens, seed=4)
    bad = bt.copy()
    bad[0, 3] = 10_000
    out, ws = run_decode(K, g, bad, q, lens, ml, 1 / 16)
    assert K.read_status(ws) & K.DEV_BAD_PAGE
    assert np.isnan(out[0]).all()
    ref = O.decode(o, to_np_in(q[1:2]), [lens[1]], bt[1:2], 1 / 16)
    assert_close(out[1], ref[0], what="healthy sequence next to a bad one")
    out, ws = run_decode(K, g, bt, q, [600, 5000], ml, 1 / 16)   # length above max_seq_len
    assert K.read_status(ws) & K.DEV_BAD_LENGTH
    assert np.isnan(out[1]).all()


def test_bounded_wait_ends_with_timeout_status(K):
    """A copy wait that nothing completes gives up after its bound (~2 s) and
    reports KVQ_DEV_TIMEOUT; the context stays usable (a decode right after
    still matches the oracle)."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    K.selftest_wait_timeout(st)
    code = K.read_status(st)
    assert code & K.DEV_TIMEOUT
    assert time.time() - t0 < 30
    lens = [300]
    g, o, bt, q, ml = decode_case(K, lens, seed=13)
    out, ws = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    assert K.read_status(ws) == 0
    assert_close(out[0], O.decode(o, to_np_in(q), lens, bt, 1 / 16)[0], what="decode after the timeout")


@pytest.mark.parametrize("fmt", ["Q4", "Q4_0"])
def test_decode_merged_equals_decode_then_merge(K, fmt):
    """The fused decode + last-CTA merge: close to the two-launch path and to the
    oracle, for several sequences (one invalid, one empty), twice on the same
    workspace (the completion counters return to zero)."""
    f = K.FMT_Q4_HAD32 if fmt == "Q4" else K.FMT_Q4_0
    lens = [1500, 513, 40, 0, 2049]
    g, o, bt, q, ml = decode_case(K, lens, fmt=f, seed=77)
    qd = q.to(DEV)
    qr = K.rotate_query(qd) if f == K.FMT_Q4_HAD32 else qd.float()
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    dbt = torch.from_numpy(bt).to(DEV)
    ws = K.alloc_workspace(g, len(lens), 24, ml, device=DEV)
    ref2, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
    for _ in range(2):
        out = K.decode_merged(g, qr, seq, dbt, ml, 1 / 16, ws).cpu().numpy()
        assert K.read_status(ws) == 0
        for b, L in enumerate(lens):
            if L == 0:
                assert np.all(out[b] == 0)
                continue
            assert_close(out[b], ref[b], what=f"merged seq {b}")
            assert np.abs(out[b] - ref2[b]).max() <= 1e-5 * np.abs(ref2[b]).max()
    bad = torch.tensor([1500, 5000, 40, 0, 2049], dtype=torch.int32, device=DEV)
    out = K.decode_merged(g, qr, bad, dbt, ml, 1 / 16, ws).cpu().numpy()
    assert K.read_status(ws) & K.DEV_BAD_LENGTH
    assert np.isnan(out[1]).all()
    assert_close(out[0], ref[0], what="merged seq 0 next to an invalid one")


@pytest.mark.parametrize("Hk,Hq,lens", [(4, 4, [4500, 700]), (2, 6, [9000, 33]), (1, 8, [8193, 1]),
                                         (4, 32, [3000, 1200, 4097]), (8, 8, [40000, 2000]),
                                         (4, 32, [40000, 2000])])
def test_decode_merged_gqa_groups(K, Hk, Hq, lens):
    """The fused merge for GQA groups 1, 3, 8 (the fold's columns: 64 per head,
    up to four per thread) with lengths of one and several blocks of 8
    partitions; the last two cases' grids are over one wave (the multi-wave
    launch form).  Against the oracle and the two-launch path (to 1e-5)."""
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, seed=Hk * 100 + Hq + 7)
    qr = K.rotate_query(q.to(DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    dbt = torch.from_numpy(bt).to(DEV)
    ws = K.alloc_workspace(g, len(lens), Hq, ml, device=DEV)
    out = K.decode_merged(g, qr, seq, dbt, ml, 0.07, ws).cpu().numpy()
    assert K.read_status(ws) == 0
    ref2, _ = run_decode(K, g, bt, q, lens, ml, 0.07)
    ref = O.decode(o, to_np_in(q), lens, bt, 0.07)
    for b in range(len(lens)):
        assert_close(out[b], ref[b], what=f"merged Hk={Hk} Hq={Hq} seq {b}")
        assert np.abs(out[b] - ref2[b]).max() <= 1e-5 * np.abs(ref2[b]).max()


def test_decode_merged_blocks_batch_independent(K):
    """The fused merge's two levels (blocks of 8 partitions): lengths of 2 and 3
    blocks and one whose last block holds a single partition; each sequence's
    outputs against the oracle, equal bit for bit to the same sequence decoded
    alone (the tree depends only on partition indices), and run to run."""
    lens = [9000, 4097, 12800, 700]
    g, o, bt, q, ml = decode_case(K, lens, seed=91)
    qr = K.rotate_query(q.to(DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    dbt = torch.from_numpy(bt).to(DEV)
    ws = K.alloc_workspace(g, len(lens), 24, ml, device=DEV)
    out = K.decode_merged(g, qr, seq, dbt, ml, 1 / 16, ws).clone()
    again = K.decode_merged(g, qr, seq, dbt, ml, 1 / 16, ws)
    assert torch.equal(out, again)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
    for b, L in enumerate(lens):
        assert_close(out[b].cpu().numpy(), ref[b], what=f"merged blocks seq {b}")
        ws1 = K.alloc_workspace(g, 1, 24, L, device=DEV)
        solo = K.decode_merged(g, qr[b:b + 1].contiguous(), seq[b:b + 1].contiguous(),
                               dbt[b:b + 1].contiguous(), L, 1 / 16, ws1)
        assert torch.equal(solo[0], out[b]), f"seq {b}: batched != solo"


def test_decode_bf16_cache(K):
    lens = [1500, 513, 20]
    g, o, bt, q, ml = decode_case(K, lens, fmt=K.FMT_BF16, seed=8)
    torch.cuda.synchronize()
    check_planes_equal(g, o)
    out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16)
    for b in range(3):
        assert_close(out[b], ref[b], what=f"bf16 seq {b}")


@pytest.mark.parametrize("T", [1, 16, 17, 511, 513, 4097])
def test_decode_bf16_lengths(K, T):
    g, o, bt, q, ml = decode_case(K, [T], fmt=K.FMT_BF16, seed=300 + T)
    out, _ = run_decode(K, g, bt, q, [T], ml, 1 / 16)
    ref = O.decode(o, to_np_in(q), [T], bt, 1 / 16)
    assert_close(out[0], ref[0], what=f"bf16 T={T}")


@pytest.mark.parametrize("Hk,Hq", [(1, 8), (3, 21), (2, 2)])
def test_decode_bf16_gqa_groups(K, Hk, Hq):
    lens = [700, 45]
    g, o, bt, q, ml = decode_case(K, lens, Hk=Hk, Hq=Hq, fmt=K.FMT_BF16, seed=400 + Hq)
    out, _ = run_decode(K, g, bt, q, lens, ml, 0.07)
    ref = O.decode(o, to_np_in(q), lens, bt, 0.07)
    for b in range(2):
        assert_close(out[b], ref[b], what=f"bf16 Hk={Hk} Hq={Hq} seq {b}")


def test_decode_bf16_gather_and_bad_page(K):
    lens = [2600, 900]
    g, o, bt, q, ml = decode_case(K, lens, fmt=K.FMT_BF16, seed=41)
    for n_sel in (1, 100, 777):
        sel = np.stack([synth.distinct_sorted(n_sel, L, 41, b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
        out, _ = run_decode(K, g, bt, q, lens, ml, 1 / 16, sel=sel)
        ref = O.decode(o, to_np_in(q), lens, bt, 1 / 16, sel=sel)
        for b in range(2):
            assert_close(out[b], ref[b], what=f"bf16 gather n_sel={n_sel} seq {b}")
    bad = bt.copy()
    bad[0, 5] = 10_000
    out, ws = run_decode(K, g, bad, q, lens, ml, 1 / 16)
    assert K.read_status(ws) & K.DEV_BAD_PAGE
    assert np.isnan(out[0]).all()
    ref = O.decode(o, to_np_in(q[1:2]), [lens[1]], bt[1:2], 1 / 16)
    assert_close(out[1], ref[0], what="bf16 healthy sequence next to a bad one")


def test_decode_fp8_latent(K):
    D, R, ps, Hq = 512, 64, 16, 32
    lens = [1100, 40]
    n_pages = sum((L + ps - 1) // ps for L in lens) + 1
    g, o = make_cache_pair(K, K.FMT_FP8_ROW, 1, D, ps, n_pages, rope=R)
    perm = synth.page_permutation(n_pages, "fp8dec").numpy().astype(np.int32)
    mp = max((L + ps - 1) // ps for L in lens)
    bt = np.zeros((2, mp), np.int32)
    off = 0
    for b, L in enumerate(lens):
        npg = (L + ps - 1) // ps
        bt[b, :npg] = perm[off:off + npg]
        off += npg
        fill_sequence(K, g, o, synth.latent_rows(L, D + R, "cpu", "fp8dec", b), None, bt[b], L)
    torch.cuda.synchronize()
    check_planes_equal(g, o)
    q = synth.normal((2, Hq, D + R), "cpu", "fp8q")
    sm = 1 / math.sqrt(D + R)
    out, _ = run_decode(K, g, bt, q, lens, max(lens), sm)
    ref = O.decode(o, q.numpy(), lens, bt, sm)
    for b in range(2):
        assert_close(out[b], ref[b], what=f"fp8 seq {b}")
    sel = np.stack([synth.distinct_sorted(37, L, "fp8sel", b).numpy() for b, L in enumerate(lens)]).astype(np.int32)
    out, _ = run_decode(K, g, bt, q, lens, max(lens), sm, sel=sel)
    ref = O.decode(o, q.numpy(), lens, bt, sm, sel=sel)
    for b in range(2):
        assert_close(out[b], ref[b], what=f"fp8 gather seq {b}")


# --------------------------------------------------------------------------- prefill

def _fp8_prefill_case(K, depth, n_q, Hq=32, seed=0):
    D, R, ps = 512, 64, 16
    T = depth + n_q
    n_pages = (T + ps - 1) // ps + 1
    g, o = make_cache_pair(K, K.FMT_FP8_ROW, 1, D, ps, n_pages, rope=R)
    bt = synth.page_permutation(n_pages, "fp8pf", seed).numpy().astype(np.int32)
    fill_sequence(K, g, o, synth.latent_rows(T, D + R, "cpu", "fp8pf", seed), None, bt, T)
    q = synth.normal((n_q, Hq, D + R), "cpu", "fp8pfq", seed)
    return g, o, bt, q


@pytest.mark.parametrize("depth,n_q,Hq", [(0, 5, 32), (700, 6, 32), (1500, 3, 48), (3, 1, 16)])
def test_prefill_fp8_matches_oracle(K, depth, n_q, Hq):
    """fp8 latent prefill (one streaming CTA per row and 32 heads, the whole row one
    partition) against the oracle's causal prefill."""
    g, o, bt, q = _fp8_prefill_case(K, depth, n_q, Hq, seed=depth)
    sm = 1 / math.sqrt(576)
    out = K.prefill_attn_fp8(g, q.to(DEV), depth, torch.from_numpy(bt).to(DEV), sm).cpu().numpy()
    ref = O.prefill(o, q.numpy(), depth, bt, sm)
    for i in range(n_q):
        assert_close(out[i], ref[i], what=f"fp8 prefill row {i}")


def test_prefill_fp8_bad_page_is_flagged(K):
    """A block-table entry outside the pool: flagged in the workspace's status
    word; the rows that reach it come out NaN, the rows before it are intact."""
    depth, n_q, Hq = 60, 40, 32
    g, o, bt, q = _fp8_prefill_case(K, depth, n_q, Hq, seed=9)
    sm = 1 / math.sqrt(576)
    bad = bt.copy()
    bad[(depth + 20) // 16] = 10_000          # the page of key depth + 20 (page size 16)
    ws = torch.zeros(K.lib().kvq_prefill_fp8_workspace_size(g.ref, n_q, Hq), dtype=torch.uint8, device=DEV)
    out = K.prefill_attn_fp8(g, q.to(DEV), depth, torch.from_numpy(bad).to(DEV), sm, workspace=ws).cpu().numpy()
    assert K.read_status(ws) & K.DEV_BAD_PAGE
    first_bad = (depth + 20) // 16 * 16 - depth   # row i reads keys 0 .. depth + i
    assert np.isnan(out[n_q - 1]).all()
    ref = O.prefill(o, q.numpy(), depth, bt, sm, rows=list(range(first_bad)))
    for i in range(first_bad):
        assert_close(out[i], ref[i], what=f"fp8 prefill row {i} before the bad page")


def test_prefill_fp8_long_rows_equal_split_decode(K):
    """At 1M keys (past the pages' old 4096 / 8192 caps): the streaming prefill of
    the last rows equals the split-T decode + merge of the same rows."""
    D, R, ps, Hq = 512, 64, 64, 32
    n_q = 2
    T = (1 << 20) + n_q
    n_pages = (T + ps - 1) // ps
    g = K.Cache(K.FMT_FP8_ROW, 1, D, ps, n_pages, device=DEV, rope_dim=R)
    for s0 in range(0, T, 1 << 16):
        n = min(1 << 16, T - s0)
        K.store(g, synth.latent_rows(n, D + R, DEV, "fp8big", s0), None,
                torch.arange(s0, s0 + n, dtype=torch.int32, device=DEV))
    bt = torch.arange(n_pages, dtype=torch.int32, device=DEV)
    q = synth.normal((n_q, Hq, D + R), DEV, "fp8bigq")
    sm = 1 / math.sqrt(576)
    depth = T - n_q
    out = K.prefill_attn_fp8(g, q, depth, bt, sm)
    lens = torch.arange(depth + 1, T + 1, dtype=torch.int32, device=DEV)
    ws = K.alloc_workspace(g, n_q, Hq, T, device=DEV)
    ref = K.decode(g, q, lens, bt.reshape(1, -1).repeat(n_q, 1).contiguous(), T, sm, ws)
    torch.cuda.synchronize()
    for i in range(n_q):
        assert_close(out[i].cpu().numpy(), ref[i].cpu().numpy().astype(np.float64), tol=1e-4,
                     what=f"1M-key row {i}")


@pytest.mark.parametrize("depth,n_q", [(0, 20), (100, 37), (600, 150), (511, 1), (0, 1)])
def test_prefill(K, depth, n_q):
    Hk, Hq, D, ps = 4, 24, 256, 16
    T = depth + n_q
    n_pages = (T + ps - 1) // ps + 1
    g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, ps, n_pages)
    bt = synth.page_permutation(n_pages, "pf", depth).numpy().astype(np.int32)
    k = synth.heavy_tailed((T, Hk, D), "cpu", "pfk", depth)
    v = synth.heavy_tailed((T, Hk, D), "cpu", "pfv", depth)
    fill_sequence(K, g, o, k, v, bt, T)
    q = synth.heavy_tailed((n_q, Hq, D), "cpu", "pfq", depth)
    out = K.prefill_attn(g, q.to(DEV), depth, torch.from_numpy(bt).to(DEV), 1 / 16)
    torch.cuda.synchronize()
    ref = O.prefill(o, to_np_in(q), depth, bt, 1 / 16)
    got = out.cpu().numpy()
    for i in range(n_q):
        assert_close(got[i], ref[i], what=f"prefill row {i}")


def test_prefill_q4_0(K):
    """Prefill over the unrotated 4-bit format: the query and the output are used
    as given (no rotations), against the oracle."""
    Hk, Hq, D, ps, depth, n_q = 4, 24, 256, 16, 300, 70
    T = depth + n_q
    n_pages = (T + ps - 1) // ps + 1
    g, o = make_cache_pair(K, K.FMT_Q4_0, Hk, D, ps, n_pages)
    bt = synth.page_permutation(n_pages, "pf0", depth).numpy().astype(np.int32)
    k = synth.heavy_tailed((T, Hk, D), "cpu", "pfk0", depth)
    v = synth.heavy_tailed((T, Hk, D), "cpu", "pfv0", depth)
    fill_sequence(K, g, o, k, v, bt, T)
    q = synth.heavy_tailed((n_q, Hq, D), "cpu", "pfq0", depth)
    out = K.prefill_attn(g, q.to(DEV), depth, torch.from_numpy(bt).to(DEV), 1 / 16)
    torch.cuda.synchronize()
    ref = O.prefill(o, to_np_in(q), depth, bt, 1 / 16)
    got = out.cpu().numpy()
    for i in range(n_q):
        assert_close(got[i], ref[i], what=f"Q4_0 prefill row {i}")


@pytest.mark.parametrize("Hk,Hq,depth,n_q", [(2, 16, 70, 33), (3, 3, 200, 129), (1, 5, 0, 64)])
def test_prefill_gqa_groups(K, Hk, Hq, depth, n_q):
    D, ps = 256, 16
    T = depth + n_q
    n_pages = (T + ps - 1) // ps + 2
    g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, ps, n_pages)
    bt = synth.page_permutation(n_pages, "pfg", Hk, Hq).numpy().astype(np.int32)
    k = synth.heavy_tailed((T, Hk, D), "cpu", "pfgk", Hk, Hq)
    v = synth.heavy_tailed((T, Hk, D), "cpu", "pfgv", Hk, Hq)
    fill_sequence(K, g, o, k, v, bt, T)
    q = synth.outlier_normal((n_q, Hq, D), 4, 20.0, "cpu", "pfgq", Hk, Hq)   # fp32 queries
    out = K.prefill_attn(g, q.to(DEV), depth, torch.from_numpy(bt).to(DEV), 0.05)
    torch.cuda.synchronize()
    ref = O.prefill(o, q.numpy(), depth, bt, 0.05)
    got = out.cpu().numpy()
    for i in range(n_q):
        assert_close(got[i], ref[i], what=f"prefill Hk={Hk} Hq={Hq} row {i}")


def test_prefill_bad_page_is_flagged(K):
    Hk, Hq, D, ps, depth, n_q = 1, 6, 256, 16, 40, 10
    T = depth + n_q
    g, o = make_cache_pair(K, K.FMT_Q4_HAD32, Hk, D, ps, 4)
    bt = np.array([0, 1, 2, 3], np.int32)
    k = synth.normal((T, Hk, D), "cpu", "pbk")
    fill_sequence(K, g, o, k, k, bt, T)
    bad = bt.copy()
    bad[1] = 99
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q = synth.normal((n_q, Hq, D), "cpu", "pbq")
    out = K.prefill_attn(g, q.to(DEV), depth, torch.from_numpy(bad).to(DEV), 0.1, status=st)
    torch.cuda.synchronize()
    assert K.read_status(st) & K.DEV_BAD_PAGE
    assert np.isnan(out.cpu().numpy()).all()


def test_binding_refuses_strided_views(K):
    """A strided view would be read as if row-major: the binding refuses it."""
    q = torch.zeros((2, 24, 512), dtype=torch.float32, device=DEV)[:, :, ::2]
    with pytest.raises(ValueError):
        K.rotate_query(q)
    g = K.Cache(K.FMT_Q4_HAD32, 4, 256, 16, 2, device=DEV)
    g.k = g.k.transpose(0, 1)
    with pytest.raises(ValueError):
        g.refresh()
