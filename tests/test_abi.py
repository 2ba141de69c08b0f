"""The C-ABI library loads, exports every entry point include/kvq.h declares,
and rejects bad host-side arguments before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT, golden

HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def K():
    from bit_quantized_kv_store_gb300 import build
    build.build()
    from bit_quantized_kv_store_gb300 import _lib
    _lib.lib()
    return _lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(K):
    names = declared_functions()
    assert len(names) >= 10
    L = K.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(K.SIGNATURES), "binding and header disagree"


def test_version_and_status_strings(K):
    L = K.lib()
    assert L.kvq_version() >= 100
    for s in (0, -1, -2, -3, -4):
        assert L.kvq_status_string(s)


def _desc(K, fmt=0, Hk=4, D=256, ps=16, pages=4, rope=0, ptr=4096):
    return K.CacheDesc(fmt, Hk, D, rope, ps, pages, ptr, ptr, ptr, ptr)


def test_host_validation_without_gpu(K):
    L = K.lib()
    d = _desc(K)
    dummy = ctypes.c_void_p(4096)
    # null cache / bad format / head_dim not a multiple of 32 / page size
    assert L.kvq_store(None, dummy, dummy, 0, 1, dummy, None, None) == K.ERR_INVALID_ARG
    assert L.kvq_store(ctypes.byref(_desc(K, fmt=7)), dummy, dummy, 0, 1, dummy, None, None) == K.ERR_INVALID_ARG
    assert L.kvq_store(ctypes.byref(_desc(K, D=48)), dummy, dummy, 0, 1, dummy, None, None) == K.ERR_UNSUPPORTED
    assert L.kvq_store(ctypes.byref(_desc(K, ps=8)), dummy, dummy, 0, 1, dummy, None, None) == K.ERR_UNSUPPORTED
    assert L.kvq_store(ctypes.byref(d), dummy, dummy, 5, 1, dummy, None, None) == K.ERR_INVALID_ARG   # dtype
    assert L.kvq_store(ctypes.byref(d), dummy, None, 0, 1, dummy, None, None) == K.ERR_INVALID_ARG    # v missing
    assert L.kvq_store(ctypes.byref(d), dummy, dummy, 0, -1, dummy, None, None) == K.ERR_INVALID_ARG  # n_tok
    assert L.kvq_store(ctypes.byref(d), dummy, dummy, 0, 0, dummy, None, None) == K.OK                # nothing to do
    fp8 = _desc(K, fmt=2, Hk=1, D=512, rope=64)
    assert L.kvq_store(ctypes.byref(fp8), dummy, dummy, 0, 1, dummy, None, None) == K.ERR_INVALID_ARG  # v must be NULL
    # unaligned planes
    assert L.kvq_store(ctypes.byref(_desc(K, ptr=4097)), dummy, dummy, 0, 1, dummy, None, None) == K.ERR_INVALID_ARG
    # rotation
    assert L.kvq_rotate_query(dummy, 0, dummy, 4, 40, None) == K.ERR_UNSUPPORTED
    assert L.kvq_rotate_query(dummy, 1, ctypes.c_void_p(4096), 4, 64, None) == K.ERR_INVALID_ARG  # in place needs f32
    # decode: group > 8, workspace too small, gather list too long, bad max_seq_len
    ws = L.kvq_decode_workspace_size(ctypes.byref(d), 2, 24, 1000, 0)
    assert ws > 0
    args = lambda Hq=24, msl=1000, sel=None, nsel=0, wsb=ws, mp=100: (
        ctypes.byref(d), dummy, 2, Hq, dummy, dummy, mp, msl, sel, nsel, ctypes.c_float(0.1), dummy, wsb, None)
    assert L.kvq_decode_attn(*args(Hq=40)) == K.ERR_UNSUPPORTED
    assert L.kvq_decode_attn(*args(wsb=ws - 1)) == K.ERR_WORKSPACE_TOO_SMALL
    assert L.kvq_decode_attn(*args(sel=dummy, nsel=5000)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_attn(*args(msl=100 * 16 + 1)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_attn(*args(Hq=25)) == K.ERR_INVALID_ARG   # not a multiple of Hk
    # merge: rotate_back only for the 4-bit format
    bf = _desc(K, fmt=1)
    assert L.kvq_merge(ctypes.byref(bf), dummy, 1 << 30, 1, 8, dummy, 100, 0, 1, dummy, None) == K.ERR_INVALID_ARG
    # prefill: only the 4-bit format
    assert L.kvq_prefill_attn(ctypes.byref(bf), dummy, 0, 4, 8, 0, dummy, 4, ctypes.c_float(0.1), dummy, None,
                              None) == K.ERR_UNSUPPORTED
    assert L.kvq_prefill_attn(ctypes.byref(d), dummy, 0, 100, 24, 0, dummy, 4, ctypes.c_float(0.1), dummy, None,
                              None) == K.ERR_INVALID_ARG   # chunk beyond the block table


def test_workspace_geometry(K):
    L = K.lib()
    d = _desc(K)
    for B, Hq, T in ((1, 24, 32769), (32, 24, 65537), (1, 24, 262145)):
        P = -(-T // 512)
        n = B * Hq * P
        r = lambda x: (x + 255) // 256 * 256
        nblk = -(-P // 8)
        nb = B * Hq * nblk
        # header, m and z, acc; then the fused merge's completion counters (per
        # (sequence, KV head), and per block of 8 partitions) and block partials
        assert L.kvq_decode_workspace_size(ctypes.byref(d), B, Hq, T, 0) == \
            256 + 2 * r(4 * n) + r(4 * n * 256) + r(4 * B * d.num_kv_heads * (1 + nblk)) + 2 * r(4 * nb) + \
            r(4 * nb * 256)


def test_plane_bytes_match_page_figures(K):
    L = K.lib()
    fig = golden("page_figures.txt")
    d = _desc(K, Hk=4, D=256, ps=16, pages=1)
    per_pos = sum(L.kvq_plane_bytes(ctypes.byref(d), p) for p in range(4)) // 16
    assert per_pos * 16 == fig["q4_bytes_per_position_16_layers_4_heads"]
    assert per_pos // (2 * 4) == fig["q4_row_bytes_d256"]
    b = _desc(K, fmt=1, Hk=4, D=256, ps=16, pages=1)
    assert sum(L.kvq_plane_bytes(ctypes.byref(b), p) for p in range(4)) // 16 * 16 == \
        fig["bf16_bytes_per_position_16_layers_4_heads"]
    f = _desc(K, fmt=2, Hk=1, D=512, ps=16, pages=1, rope=64)
    assert sum(L.kvq_plane_bytes(ctypes.byref(f), p) for p in range(4)) // 16 == fig["fp8_latent_bytes_per_token"]


def test_product_path_has_no_oracle_or_cpu_fallback():
    pkg = os.path.join(ROOT, "bit_quantized_kv_store_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "kvq_oracle" not in text, f


def _tq4_desc(K, D=256, signs=4096):
    return K.CacheDesc(4, 4, D, 0, 16, 4, 4096, 4096, 4096, 4096, signs)


def test_host_validation_of_the_other_entries(K):
    """Windows, the fused merge, unrotated queries, the fused decode step, TQ4,
    the fp8 prefill, the fused store + rotation and the no-allocation decode
    reject bad host arguments with their documented codes, before anything is
    enqueued."""
    L = K.lib()
    d = _desc(K)
    bf = _desc(K, fmt=1)
    fp8 = _desc(K, fmt=2, Hk=1, D=512, rope=64)
    dummy = ctypes.c_void_p(4096)
    f = ctypes.c_float(0.1)
    ws = L.kvq_decode_workspace_size(ctypes.byref(d), 4, 24, 1000, 0)
    # kvq_decode_window: 4-bit formats only, at most 64 rows, workspace size
    win = lambda c=d, rows=4, wsb=ws: (ctypes.byref(c), dummy, rows, 24, dummy, dummy, 100, 1000, f, dummy, wsb, None)
    assert L.kvq_decode_window(None, dummy, 4, 24, dummy, dummy, 100, 1000, f, dummy, ws, None) == K.ERR_INVALID_ARG
    assert L.kvq_decode_window(*win(c=bf)) == K.ERR_UNSUPPORTED
    assert L.kvq_decode_window(*win(rows=65)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_window(*win(wsb=ws - 1)) == K.ERR_WORKSPACE_TOO_SMALL
    # kvq_decode_merged: 4-bit only, an output, at most 8192 block weights per group
    mg = lambda c=d, out=dummy, msl=1000: (ctypes.byref(c), dummy, 1, 24, dummy, dummy, 100000, msl, f, dummy,
                                           1 << 40, out, None)
    assert L.kvq_decode_merged(*mg(c=fp8)) == K.ERR_UNSUPPORTED
    assert L.kvq_decode_merged(*mg(out=None)) == K.ERR_INVALID_ARG
    # 1366 blocks of 8 partitions x group 6 > 8192 block weights
    assert L.kvq_decode_merged(*mg(msl=(1365 * 8 + 1) * 512)) == K.ERR_UNSUPPORTED
    # kvq_decode_attn_unrotated: rotated 4-bit (or Q4_0) only, f32 / bf16 queries
    un = lambda c=d, qd=0, q=dummy: (ctypes.byref(c), q, qd, 2, 24, dummy, dummy, 100, 1000, None, 0, f, dummy, ws,
                                     None)
    assert L.kvq_decode_attn_unrotated(*un(c=bf)) == K.ERR_UNSUPPORTED
    assert L.kvq_decode_attn_unrotated(*un(qd=7)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_attn_unrotated(*un(q=None)) == K.ERR_INVALID_ARG
    # kvq_decode_step: Q4_HAD32 / Q4_0 only, f32 / bf16 rows and queries, all three inputs, workspace size
    ws2 = L.kvq_decode_workspace_size(ctypes.byref(d), 2, 24, 1000, 0)
    stp = lambda c=d, kn=dummy, vn=dummy, kd=0, q=dummy, qd=0, wsb=ws2: (
        ctypes.byref(c), kn, vn, kd, q, qd, 2, 24, dummy, dummy, 100, 1000, f, dummy, wsb, None)
    assert L.kvq_decode_step(None, *stp()[1:]) == K.ERR_INVALID_ARG
    assert L.kvq_decode_step(*stp(c=bf)) == K.ERR_UNSUPPORTED
    assert L.kvq_decode_step(*stp(c=_tq4_desc(K))) == K.ERR_UNSUPPORTED
    assert L.kvq_decode_step(*stp(kd=5)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_step(*stp(qd=5)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_step(*stp(kn=None)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_step(*stp(vn=None)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_step(*stp(q=None)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_step(*stp(wsb=ws2 - 1)) == K.ERR_WORKSPACE_TOO_SMALL
    # TQ4 caches: the sign mask is required and 4-byte aligned; head_dim 64 / 128 / 256
    one = ctypes.c_int32(0)
    st = lambda c: L.kvq_store(ctypes.byref(c), dummy, dummy, 0, 1, ctypes.byref(one), None, None)
    assert st(_tq4_desc(K, signs=None)) == K.ERR_INVALID_ARG
    assert st(_tq4_desc(K, signs=4098)) == K.ERR_INVALID_ARG
    assert st(_tq4_desc(K, D=96)) == K.ERR_UNSUPPORTED
    # kvq_tq4_rotate: TQ4 caches only; dtype; in place needs f32
    t = _tq4_desc(K)
    assert L.kvq_tq4_rotate(ctypes.byref(d), dummy, 0, dummy, 4, 24, None) == K.ERR_UNSUPPORTED
    assert L.kvq_tq4_rotate(ctypes.byref(t), dummy, 3, ctypes.c_void_p(8192), 4, 24, None) == K.ERR_INVALID_ARG
    assert L.kvq_tq4_rotate(ctypes.byref(t), dummy, 1, dummy, 4, 24, None) == K.ERR_INVALID_ARG
    # kvq_prefill_attn_fp8: fp8 latent rows, 16 | heads, the chunk inside the block table, workspace
    pw = L.kvq_prefill_fp8_workspace_size(ctypes.byref(fp8), 8, 128)
    assert pw > 0
    pf = lambda c=fp8, nq=8, hq=128, q0=0, mp=4, wsb=pw: (ctypes.byref(c), dummy, nq, hq, q0, dummy, mp, f, dummy,
                                                          wsb, dummy, None)
    assert L.kvq_prefill_attn_fp8(*pf(c=d)) == K.ERR_UNSUPPORTED
    assert L.kvq_prefill_attn_fp8(*pf(hq=24)) == K.ERR_UNSUPPORTED
    assert L.kvq_prefill_attn_fp8(*pf(nq=-1)) == K.ERR_INVALID_ARG
    assert L.kvq_prefill_attn_fp8(*pf(nq=0)) == K.OK
    assert L.kvq_prefill_attn_fp8(*pf(q0=60)) == K.ERR_INVALID_ARG    # rows 60..67 beyond 4 pages of 16
    assert L.kvq_prefill_attn_fp8(*pf(wsb=pw - 1)) == K.ERR_WORKSPACE_TOO_SMALL
    # kvq_store_rotate: dtypes, counts, pointers
    sr = lambda dt=0, qdt=0, n=1, qr=24, k=dummy, q=dummy, qo=ctypes.c_void_p(8192): (
        ctypes.byref(d), k, dummy, dt, n, dummy, None, q, qdt, qo, qr, None)
    assert L.kvq_store_rotate(*sr(dt=4)) == K.ERR_INVALID_ARG
    assert L.kvq_store_rotate(*sr(qdt=4)) == K.ERR_INVALID_ARG
    assert L.kvq_store_rotate(*sr(n=-1)) == K.ERR_INVALID_ARG
    assert L.kvq_store_rotate(*sr(k=None)) == K.ERR_INVALID_ARG
    assert L.kvq_store_rotate(*sr(q=None)) == K.ERR_INVALID_ARG
    assert L.kvq_store_rotate(*sr(qdt=1, qo=dummy)) == K.ERR_INVALID_ARG   # in place needs f32
    # kvq_decode_noalloc: a cache, a workspace that fits the static array, an output
    scratch = L.kvq_noalloc_scratch_bytes()
    assert scratch == 16 << 20
    na = lambda c=d, B=1, msl=1000, out=dummy: (ctypes.byref(c) if c else None, dummy, B, 24, dummy, dummy, 100000,
                                                msl, None, 0, f, 1, out, None, None)
    assert L.kvq_decode_noalloc(*na(c=None)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_noalloc(*na(B=64, msl=262145)) == K.ERR_WORKSPACE_TOO_SMALL
    assert L.kvq_decode_noalloc(*na(out=None)) == K.ERR_INVALID_ARG
    # every check of the decode and the merge comes before the status word is
    # cleared: with no GPU here, a call that got past them would fail with
    # KVQ_ERR_CUDA instead
    na_rb = lambda c, rb, q=dummy: (ctypes.byref(c), q, 1, 24, dummy, dummy, 100000, 1000, None, 0, f, rb, dummy,
                                    None, None)
    assert L.kvq_decode_noalloc(*na_rb(bf, 1)) == K.ERR_INVALID_ARG      # rotate_back on bf16 rows (merge's check)
    assert L.kvq_decode_noalloc(*na_rb(d, 1, q=None)) == K.ERR_INVALID_ARG
    assert L.kvq_decode_noalloc(*na_rb(d, 1, q=ctypes.c_void_p(4100))) == K.ERR_INVALID_ARG   # unaligned query
    assert L.kvq_decode_noalloc(ctypes.byref(d), dummy, 1, 24, dummy, None, 100000, 1000, None, 0, f, 1, dummy,
                                None, None) == K.ERR_INVALID_ARG   # no block table
    assert L.kvq_decode_noalloc(ctypes.byref(d), dummy, 1, 24, dummy, dummy, 10, 1000, None, 0, f, 1, dummy,
                                None, None) == K.ERR_INVALID_ARG   # 10 pages of 16 < 1000 keys
    assert L.kvq_decode_noalloc(ctypes.byref(d), dummy, 0, 24, None, None, 0, 0, None, 0, f, 1, None,
                                None, None) == K.OK                # nothing to do, nothing enqueued
    # status helpers
    assert L.kvq_selftest_wait_timeout(None, None) == K.ERR_INVALID_ARG
    assert L.kvq_read_status(None, dummy, None) == K.ERR_INVALID_ARG


def test_binding_refuses_host_memory(K):
    """The binding hands the kernels device addresses only: a host tensor or a
    host-resident cache is refused before any call."""
    import torch
    assert K._ptr(None) is None
    with pytest.raises(ValueError):
        K._ptr(torch.zeros(4))
    with pytest.raises(ValueError):
        K.Cache(K.FMT_Q4_HAD32, 4, 256, 16, 2, device="cpu")
