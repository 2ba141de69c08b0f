"""GPU parity at the benchmark's full sizes, in the launch configurations
bench.py times, on outputs the oracle computes one by one.

The oracle is slow, so it evaluates samples: query heads 0 and 23 (of 24),
which read the first and the last KV head; the oracle's cache holds those two
KV heads only and sees a 2-head query whose GQA group is 1, so that head i
still reads its KV head.  Sampled sequences of the batch and sampled rows of
the prefill chunk likewise.  The inputs follow the benchmark's recipe (bf16,
5 % Student-t(3) x 10 channels), from the shared seeded generators.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from bit_quantized_kv_store_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
HK, HQ, D, PS = 4, 24, 256, 16
HEADS = [0, 23]     # sampled query heads
KV_HEADS = [0, 3]   # the KV heads they read (group of 6)
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


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    scale = np.abs(ref).max()
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref).max()
    assert err <= TOL * scale, f"{what}: max-abs error {err:.3g} > {TOL} * {scale:.3g}"


def fill(K, g, o, T, seed, tag, slots_of=None, oracle=True):
    """Store T tokens of one sequence in 64K-token chunks on both sides; slots_of
    maps positions to slots (identity by default)."""
    for s0 in range(0, T, 65536):
        n = min(65536, T - s0)
        k = synth.heavy_tailed((n, HK, D), DEV, seed, tag + "k", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), DEV, seed, tag + "v", s0, subset=(seed, "v"))
        pos = torch.arange(s0, s0 + n, dtype=torch.int32, device=DEV)
        slots = pos if slots_of is None else slots_of(pos)
        K.store(g, k, v, slots)
        if oracle:
            assert O.store(o, bits(k[:, KV_HEADS]), bits(v[:, KV_HEADS]), slots.cpu().numpy()) == 0


def signs_for(fmt, K, seed):
    return synth.sign_mask(D, seed, "full") if fmt == K.FMT_TQ4 else None


def pair(K, fmt, n_pages, seed):
    s = signs_for(fmt, K, seed)
    g = K.Cache(fmt, HK, D, PS, n_pages, device=DEV, signs=s)
    ofmt = {K.FMT_Q4_HAD32: O.Q4, K.FMT_TQ4: O.TQ4}[fmt]
    o = O.Cache(ofmt, len(KV_HEADS), D, PS, n_pages, signs=None if s is None else s.numpy().view(np.uint32))
    return g, o


def sampled(q):
    return bits(q[:, HEADS].contiguous())


@pytest.mark.parametrize("context,fmt", [(32768, "Q4"), (262144, "Q4"), (262144, "TQ4")])
def test_single_sequence_decode_full_size(K, context, fmt):
    """The decode step of the 32K / 262K benchmark rows (one sequence, T = N + 1
    keys, 16-token pages): rotation, split-T decode, merge (and rotation back)."""
    f = K.FMT_Q4_HAD32 if fmt == "Q4" else K.FMT_TQ4
    T = context + 1
    npg = (T + PS - 1) // PS
    g, o = pair(K, f, npg, 7)
    fill(K, g, o, T, 7, fmt)
    q = synth.heavy_tailed((1, HQ, D), DEV, 7, fmt + "q")
    bt = torch.arange(npg, dtype=torch.int32, device=DEV).reshape(1, -1)
    seq = torch.tensor([T], dtype=torch.int32, device=DEV)
    ws = K.alloc_workspace(g, 1, HQ, T, device=DEV)
    out = K.decode(g, q, seq, bt, T, 1 / 16, ws).cpu().numpy()
    assert K.read_status(ws) == 0
    ref = O.decode(o, sampled(q), [T], bt.cpu().numpy(), 1 / 16)
    assert_close(out[0, HEADS], ref[0], f"{fmt} decode at {context}")


def test_batched_ragged_decode_full_size(K):
    """The batched row: 32 sequences, lengths U{1024 .. 65536} + 1, 16-token pages
    from a seeded permutation; the shortest, a middle and the longest sequence
    checked against the oracle."""
    seed = 1234 + 3
    lens = synth.ragged_lengths(32, 1024, 65536, seed, "lens").tolist()
    T = [L + 1 for L in lens]
    pages = [(t + PS - 1) // PS for t in T]
    n_pages = sum(pages)
    perm = synth.page_permutation(n_pages, seed, "perm")
    bt = torch.zeros((32, max(pages)), dtype=torch.int32)
    off = 0
    for i, npg in enumerate(pages):
        bt[i, :npg] = perm[off:off + npg]
        off += npg
    order = sorted(range(32), key=lambda i: T[i])
    check = [order[0], order[16], order[-1]]
    g, o = pair(K, K.FMT_Q4_HAD32, n_pages, seed)
    btd = bt.to(DEV)
    for i, L in enumerate(T):
        fill(K, g, o, L, seed, f"b{i}", slots_of=lambda pos, i=i: (btd[i][pos // PS] * PS + pos % PS).to(torch.int32),
             oracle=i in check)
    q = synth.heavy_tailed((32, HQ, D), DEV, seed, "bq")
    seq = torch.tensor(T, dtype=torch.int32, device=DEV)
    ws = K.alloc_workspace(g, 32, HQ, max(T), device=DEV)
    out = K.decode(g, q, seq, btd, max(T), 1 / 16, ws).cpu().numpy()
    assert K.read_status(ws) == 0
    for i in check:
        ref = O.decode(o, sampled(q[i:i + 1]), [T[i]], bt[i:i + 1].numpy(), 1 / 16)
        assert_close(out[i, HEADS], ref[0], f"batched sequence {i} (T = {T[i]})")


def test_prefill_chunk_full_size(K):
    """The prefill row: a 4096-token chunk stored at depth 16384 and attended
    causally over the decoded slots; rows 0, 1, 2047, 4094, 4095 checked."""
    depth, n_q = 16384, 4096
    T = depth + n_q
    npg = (T + PS - 1) // PS
    g, o = pair(K, K.FMT_Q4_HAD32, npg, 11)
    fill(K, g, o, T, 11, "pf")
    q = synth.heavy_tailed((n_q, HQ, D), DEV, 11, "pfq")
    bt = torch.arange(npg, dtype=torch.int32, device=DEV)
    out = K.prefill_attn(g, q, depth, bt, 1 / 16).cpu().numpy()
    rows = [0, 1, 2047, 4094, 4095]
    ref = O.prefill(o, sampled(q), depth, bt.cpu().numpy(), 1 / 16, rows=rows)
    for r, i in enumerate(rows):
        assert_close(out[i, HEADS], ref[r], f"prefill row {i}")


def test_window_full_size_equals_plain_rows(K):
    """The window row: 4 draft rows at positions 262144 .. 262147 of one sequence
    equal the same rows decoded as 4 sequences, bit for bit."""
    R, T0 = 4, 262144
    T = T0 + R
    npg = (T + PS - 1) // PS
    g = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, npg, device=DEV)
    fill(K, g, None, T, 5, "w", oracle=False)
    q = synth.heavy_tailed((R, HQ, D), DEV, 5, "wq")
    bt = torch.arange(npg, dtype=torch.int32, device=DEV)
    ws_w = K.alloc_workspace(g, R, HQ, T, device=DEV)
    out_w = K.decode_window_causal(g, q, T0, bt, 1 / 16, ws_w)
    lens = torch.arange(T0 + 1, T + 1, dtype=torch.int32, device=DEV)
    ws_p = K.alloc_workspace(g, R, HQ, T, device=DEV)
    out_p = K.decode(g, q, lens, bt.reshape(1, -1).repeat(R, 1).contiguous(), T, 1 / 16, ws_p)
    torch.cuda.synchronize()
    assert torch.equal(out_w, out_p)


def test_fp8_latent_decode_full_size(K):
    """The fp8 rows: 262144 latent rows (512 + 64), 128 heads, split-T + merge,
    dense and over 2048 selected rows; 8 of the 128 heads checked (one KV head:
    every head reads it)."""
    Tf, Hf, DL, R = 262144, 128, 512, 64
    npg = Tf // PS
    g = K.Cache(K.FMT_FP8_ROW, 1, DL, PS, npg, device=DEV, rope_dim=R)
    o = O.Cache(O.FP8, 1, DL, PS, npg, rope_dim=R)
    for s0 in range(0, Tf, 65536):
        rows = synth.latent_rows(65536, DL + R, DEV, 21, "fp8", s0)
        slots = torch.arange(s0, s0 + 65536, dtype=torch.int32, device=DEV)
        K.store(g, rows, None, slots)
        assert O.store(o, rows.cpu().numpy(), None, slots.cpu().numpy()) == 0
    q = synth.normal((1, Hf, DL + R), DEV, 21, "fp8q")
    bt = torch.arange(npg, dtype=torch.int32, device=DEV).reshape(1, -1)
    seq = torch.tensor([Tf], dtype=torch.int32, device=DEV)
    ws = K.alloc_workspace(g, 1, Hf, Tf, device=DEV)
    sm = 1 / math.sqrt(DL + R)
    out = K.decode(g, q, seq, bt, Tf, sm, ws).cpu().numpy()
    heads = [0, 17, 40, 63, 64, 90, 101, 127]
    ref = O.decode(o, q[:, heads].cpu().numpy(), [Tf], bt.cpu().numpy(), sm)
    assert_close(out[0, heads], ref[0], "fp8 decode at 262144")
    # the gather row: 2048 selected absolute rows of the 262144 (split-T partials + merge)
    sel = synth.distinct_sorted(2048, Tf, 21, "sel").to(torch.int32).to(DEV).reshape(1, -1)
    wsg = K.alloc_workspace(g, 1, Hf, Tf, n_sel=2048, device=DEV)
    outg = K.decode(g, q, seq, bt, Tf, sm, wsg, sel=sel).cpu().numpy()
    refg = O.decode(o, q[:, heads].cpu().numpy(), [Tf], bt.cpu().numpy(), sm, sel=sel.cpu().numpy())
    assert_close(outg[0, heads], refg[0], "fp8 gather of 2048 rows at 262144")
