"""Full-size parity: the workloads the benchmark times, checked on sampled outputs.

Each case builds the cache on the GPU at full size with the benchmark's
recipes (heavy-tailed bf16 K/V, 16-token pages), runs the same entry points
the benchmark launches, and compares sampled outputs with the CPU oracle
computed one by one: codes and scales bit-exact for the sampled rows, and
attention within max|gpu - oracle| <= 2e-3 * max|oracle| per output tensor.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from bit_quantized_kv_store_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3
HK, HQ, D, PS = 4, 24, 256, 16


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_kv_store_gb300 import build
    build.build()
    from bit_quantized_kv_store_gb300 import _lib
    _lib.lib()
    return _lib


def bits16(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def close(got, ref, what):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref).max()
    assert err <= TOL * np.abs(ref).max(), f"{what}: {err:.3g} > {TOL} * {np.abs(ref).max():.3g}"


def one_head_oracle_cache(k_head, v_head, slots_np, n_pages):
    """An oracle cache holding one KV head (Hk = 1) for the sampled comparison."""
    oc = O.Cache(O.Q4, 1, D, PS, n_pages)
    O.store(oc, k_head[:, None, :], v_head[:, None, :], slots_np)
    return oc


def long_decode_case(K, context, seed, sample_kv_head):
    """One layer at `context` positions + the new token, identity page table,
    built like the benchmark; returns GPU output [1, 24, 256] and the oracle
    output for the 6 query heads of `sample_kv_head`."""
    dev = "cuda"
    T = context + 1
    n_pages = (T + PS - 1) // PS
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, n_pages, device=dev)
    ks, vs = [], []
    chunk = 32768
    for s0 in range(0, T, chunk):
        n = min(chunk, T - s0)
        k = synth.heavy_tailed((n, HK, D), dev, seed, "k", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), dev, seed, "v", s0, subset=(seed, "v"))
        K.store(c, k, v, torch.arange(s0, s0 + n, dtype=torch.int32, device=dev))
        ks.append(bits16(k[:, sample_kv_head]))
        vs.append(bits16(v[:, sample_kv_head]))
    q = synth.heavy_tailed((1, HQ, D), dev, seed, "q")
    bt = torch.arange(n_pages, dtype=torch.int32, device=dev).reshape(1, -1)
    seq = torch.tensor([T], dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, 1, HQ, T, device=dev)
    out = K.decode(c, q, seq, bt, T, 1 / math.sqrt(D), ws).cpu().numpy()
    kh, vh = np.concatenate(ks), np.concatenate(vs)
    oc = one_head_oracle_cache(kh, vh, np.arange(T, dtype=np.int32), n_pages)
    # the sampled head's planes must match the oracle's bit for bit
    assert np.array_equal(c.k[:, sample_kv_head].cpu().numpy(), oc.k[:, 0])
    assert np.array_equal(bits16(c.v_scale[:, sample_kv_head]), oc.v_scale[:, 0])
    grp = HQ // HK
    qh = bits16(q)[:, sample_kv_head * grp:(sample_kv_head + 1) * grp]
    ref = O.decode(oc, qh, [T], np.arange(n_pages, dtype=np.int32).reshape(1, -1), 1 / math.sqrt(D))
    return out[0, sample_kv_head * grp:(sample_kv_head + 1) * grp], ref[0]


def test_decode_32k_context(K):
    for kvh in (0, 3):
        got, ref = long_decode_case(K, 32768, 1235, kvh)
        close(got, ref, f"32K decode, KV head {kvh}")


def test_decode_262k_context(K):
    got, ref = long_decode_case(K, 262144, 1236, 2)
    close(got, ref, "262K decode, KV head 2")


def test_decode_bf16_32k_context(K):
    """The bf16 comparison cache at 32,769 keys: KV head 1 sampled against the oracle."""
    dev = "cuda"
    seed = 1240
    T = 32769
    n_pages = (T + PS - 1) // PS
    c = K.Cache(K.FMT_BF16, HK, D, PS, n_pages, device=dev)
    k = synth.heavy_tailed((T, HK, D), dev, seed, "k", subset=(seed, "k"))
    v = synth.heavy_tailed((T, HK, D), dev, seed, "v", subset=(seed, "v"))
    K.store(c, k, v, torch.arange(T, dtype=torch.int32, device=dev))
    q = synth.heavy_tailed((1, HQ, D), dev, seed, "q")
    bt = torch.arange(n_pages, dtype=torch.int32, device=dev).reshape(1, -1)
    seq = torch.tensor([T], dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, 1, HQ, T, device=dev)
    out = K.decode(c, q, seq, bt, T, 1 / 16, ws).cpu().numpy()
    oc = O.Cache(O.BF16, 1, D, PS, n_pages)
    O.store(oc, bits16(k[:, 1])[:, None], bits16(v[:, 1])[:, None], np.arange(T, dtype=np.int32))
    ref = O.decode(oc, bits16(q)[:, 6:12], [T], np.arange(n_pages, dtype=np.int32).reshape(1, -1), 1 / 16)
    close(out[0, 6:12], ref[0], "bf16 32K decode, KV head 1")


def test_batched_ragged_paged_decode_full_size(K):
    dev = "cuda"
    seed = 1237
    lens = synth.ragged_lengths(32, 1024, 65536, seed, "lens").tolist()
    T = [L + 1 for L in lens]
    pages = [(t + PS - 1) // PS for t in T]
    n_pages = sum(pages)
    perm = synth.page_permutation(n_pages, seed, "perm").numpy().astype(np.int32)
    bt = np.zeros((32, max(pages)), np.int32)
    off = 0
    for i, npg in enumerate(pages):
        bt[i, :npg] = perm[off:off + npg]
        off += npg
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, n_pages, device=dev)
    sample = [int(np.argmin(lens)), 7, int(np.argmax(lens))]
    kept = {}
    for i, t in enumerate(T):
        k = synth.heavy_tailed((t, HK, D), dev, seed, i, "k", subset=(seed, "k"))
        v = synth.heavy_tailed((t, HK, D), dev, seed, i, "v", subset=(seed, "v"))
        slots = torch.tensor([bt[i, j // PS] * PS + j % PS for j in range(t)], dtype=torch.int32, device=dev)
        K.store(c, k, v, slots)
        if i in sample:
            kept[i] = (bits16(k[:, 1]), bits16(v[:, 1]))
    q = synth.heavy_tailed((32, HQ, D), dev, seed, "q")
    seq = torch.tensor(T, dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, 32, HQ, max(T), device=dev)
    out = K.decode(c, q, seq, torch.from_numpy(bt).to(dev), max(T), 1 / 16, ws).cpu().numpy()
    qb = bits16(q)
    for i in sample:
        npg = pages[i]
        oc = one_head_oracle_cache(kept[i][0], kept[i][1], np.arange(T[i], dtype=np.int32), npg)
        ref = O.decode(oc, qb[i:i + 1, 6:12], [T[i]], np.arange(npg, dtype=np.int32).reshape(1, -1), 1 / 16)
        close(out[i, 6:12], ref[0], f"batched decode, sequence {i} (T={T[i]})")


def test_prefill_chunk_full_size(K):
    dev = "cuda"
    seed = 1238
    depth, nq = 16384, 4096
    Tp = depth + nq
    npg = (Tp + PS - 1) // PS
    bt = synth.page_permutation(npg, seed, "pf").numpy().astype(np.int32)
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, npg, device=dev)
    k = synth.heavy_tailed((Tp, HK, D), dev, seed, "k", subset=(seed, "k"))
    v = synth.heavy_tailed((Tp, HK, D), dev, seed, "v", subset=(seed, "v"))
    pos = np.arange(Tp)
    slots = torch.from_numpy((bt[pos // PS] * PS + pos % PS).astype(np.int32)).to(dev)
    K.store(c, k[:depth], v[:depth], slots[:depth])
    K.store(c, k[depth:], v[depth:], slots[depth:])
    q = synth.heavy_tailed((nq, HQ, D), dev, seed, "q")
    out = K.prefill_attn(c, q, depth, torch.from_numpy(bt).to(dev), 1 / 16).cpu().numpy()
    rows = [0, 1, 2047, nq - 1] + synth.distinct_sorted(4, nq, seed, "rows").tolist()
    kvh = 3
    oc = O.Cache(O.Q4, 1, D, PS, npg)
    O.store(oc, bits16(k[:, kvh])[:, None], bits16(v[:, kvh])[:, None], (bt[pos // PS] * PS + pos % PS).astype(np.int32))
    ref = O.prefill(oc, bits16(q)[:, 18:24], depth, bt, 1 / 16, rows=rows)
    for r, i in enumerate(rows):
        close(out[i, 18:24], ref[r], f"prefill row {i}")


def test_fp8_latent_full_size(K):
    dev = "cuda"
    seed = 1239
    Tf, Hf, DL, R = 262144, 128, 512, 64
    npg = Tf // PS
    c = K.Cache(K.FMT_FP8_ROW, 1, DL, PS, npg, device=dev, rope_dim=R)
    oc = O.Cache(O.FP8, 1, DL, PS, npg, rope_dim=R)
    for s0 in range(0, Tf, 65536):
        rows = synth.latent_rows(65536, DL + R, dev, seed, "fp8", s0)
        sl = np.arange(s0, s0 + 65536, dtype=np.int32)
        K.store(c, rows, None, torch.from_numpy(sl).to(dev))
        O.store(oc, rows.cpu().numpy(), None, sl)
    assert np.array_equal(c.k.cpu().numpy(), oc.k)
    assert np.array_equal(c.v.cpu().numpy(), oc.v)
    assert np.array_equal(c.k_scale.cpu().numpy().view(np.uint32), oc.k_scale.view(np.uint32))
    q = synth.normal((1, Hf, DL + R), dev, seed, "q")
    bt = torch.arange(npg, dtype=torch.int32, device=dev).reshape(1, -1)
    seq = torch.tensor([Tf], dtype=torch.int32, device=dev)
    sm = 1 / math.sqrt(DL + R)
    ws = K.alloc_workspace(c, 1, Hf, Tf, device=dev)
    out = K.decode(c, q, seq, bt, Tf, sm, ws).cpu().numpy()
    heads = [0, 77]
    ref = O.decode(oc, q.cpu().numpy()[:, heads], [Tf], bt.cpu().numpy(), sm)
    close(out[0, heads], ref[0], "fp8 dense decode, 262144 rows")
    sel = synth.distinct_sorted(2048, Tf, seed, "sel").numpy().astype(np.int32).reshape(1, -1)
    wsg = K.alloc_workspace(c, 1, Hf, Tf, n_sel=2048, device=dev)
    outg = K.decode(c, q, seq, bt, Tf, sm, wsg, sel=torch.from_numpy(sel).to(dev)).cpu().numpy()
    refg = O.decode(oc, q.cpu().numpy(), [Tf], bt.cpu().numpy(), sm, sel=sel)
    close(outg[0], refg[0], "fp8 gather of 2048 rows")
    sel4 = synth.distinct_sorted(4096, Tf, seed, "sel4").numpy().astype(np.int32).reshape(1, -1)
    ws4 = K.alloc_workspace(c, 1, Hf, Tf, n_sel=4096, device=dev)
    out4 = K.decode(c, q, seq, bt, Tf, sm, ws4, sel=torch.from_numpy(sel4).to(dev)).cpu().numpy()
    ref4 = O.decode(oc, q.cpu().numpy()[:, :8], [Tf], bt.cpu().numpy(), sm, sel=sel4)
    close(out4[0, :8], ref4[0], "fp8 gather of 4096 rows (the maximum)")


def test_decode_tq4_262k_context(K):
    """The TQ4 row at 262,145 keys: KV head 3 (query heads 18..23) against the
    oracle; the sampled head's codes and scales bit-exact."""
    dev = "cuda"
    seed = 1241
    T = 262145
    n_pages = (T + PS - 1) // PS
    signs = synth.sign_mask(D, seed, "tq4")
    c = K.Cache(K.FMT_TQ4, HK, D, PS, n_pages, device=dev, signs=signs)
    oc = O.Cache(O.TQ4, 1, D, PS, n_pages, signs=signs.numpy().view(np.uint32))
    kvh = 3
    for s0 in range(0, T, 65536):
        n = min(65536, T - s0)
        k = synth.heavy_tailed((n, HK, D), dev, seed, "k", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), dev, seed, "v", s0, subset=(seed, "v"))
        sl = np.arange(s0, s0 + n, dtype=np.int32)
        K.store(c, k, v, torch.from_numpy(sl).to(dev))
        O.store(oc, bits16(k[:, kvh])[:, None], bits16(v[:, kvh])[:, None], sl)
    assert np.array_equal(c.k[:, kvh].cpu().numpy(), oc.k[:, 0])
    assert np.array_equal(bits16(c.v_scale[:, kvh]), oc.v_scale[:, 0])
    q = synth.heavy_tailed((1, HQ, D), dev, seed, "q")
    bt = torch.arange(n_pages, dtype=torch.int32, device=dev).reshape(1, -1)
    seq = torch.tensor([T], dtype=torch.int32, device=dev)
    ws = K.alloc_workspace(c, 1, HQ, T, device=dev)
    out = K.decode(c, q, seq, bt, T, 1 / 16, ws).cpu().numpy()
    ref = O.decode(oc, bits16(q)[:, 18:24], [T], bt.cpu().numpy(), 1 / 16)
    close(out[0, 18:24], ref[0], "TQ4 262K decode, KV head 3")


def test_window_262k_equals_plain_rows(K):
    """The window row: 4 draft rows at positions 262144 .. 262147 of one sequence
    equal the same rows decoded as 4 sequences, bit for bit."""
    dev = "cuda"
    seed = 1242
    R, T0 = 4, 262144
    T = T0 + R
    n_pages = (T + PS - 1) // PS
    c = K.Cache(K.FMT_Q4_HAD32, HK, D, PS, n_pages, device=dev)
    for s0 in range(0, T, 65536):
        n = min(65536, T - s0)
        k = synth.heavy_tailed((n, HK, D), dev, seed, "k", s0, subset=(seed, "k"))
        v = synth.heavy_tailed((n, HK, D), dev, seed, "v", s0, subset=(seed, "v"))
        K.store(c, k, v, torch.arange(s0, s0 + n, dtype=torch.int32, device=dev))
    q = synth.heavy_tailed((R, HQ, D), dev, seed, "q")
    bt = torch.arange(n_pages, dtype=torch.int32, device=dev)
    ws_w = K.alloc_workspace(c, R, HQ, T, device=dev)
    out_w = K.decode_window_causal(c, q, T0, bt, 1 / 16, ws_w)
    lens = torch.arange(T0 + 1, T + 1, dtype=torch.int32, device=dev)
    ws_p = K.alloc_workspace(c, R, HQ, T, device=dev)
    out_p = K.decode(c, q, lens, bt.reshape(1, -1).repeat(R, 1).contiguous(), T, 1 / 16, ws_p)
    torch.cuda.synchronize()
    assert torch.equal(out_w, out_p)
