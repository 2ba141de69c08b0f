"""kvq_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a host application that owns every device allocation, a memory
pool that forbids new allocations, a latency-critical path that cannot pay for
cudaMalloc) cannot pass the workspace kvq_decode_attn needs; this entry point
keeps the split-T partials in the library's fixed device scratch array.  The
test calls it through the C ABI and compares it with the workspace-based
calls (kvq_decode_attn + kvq_merge) on the same inputs, twice in a row (the
second call sees the scratch array as the first left it).  It lives in a file
of its own that pytest collects last.
"""
import math

import numpy as np
import pytest
import torch

from bit_quantized_kv_store_gb300 import synth

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_kv_store_gb300 import build
    build.build()
    from bit_quantized_kv_store_gb300 import _lib
    _lib.lib()
    return _lib


def _problem(K, lens, seed):
    Hk, Hq, D, ps = 4, 24, 256, 16
    pages = [(L + ps - 1) // ps for L in lens]
    n_pages = sum(pages)
    perm = synth.page_permutation(n_pages, seed, "noalloc").numpy().astype(np.int32)
    bt = np.zeros((len(lens), max(pages)), np.int32)
    cache = K.Cache(K.FMT_Q4_HAD32, Hk, D, ps, n_pages, device="cuda")
    off = 0
    for b, L in enumerate(lens):
        bt[b, :pages[b]] = perm[off:off + pages[b]]
        off += pages[b]
        k = synth.heavy_tailed((L, Hk, D), "cuda", seed, b, "k")
        v = synth.heavy_tailed((L, Hk, D), "cuda", seed, b, "v")
        slots = torch.tensor([bt[b, j // ps] * ps + j % ps for j in range(L)], dtype=torch.int32, device="cuda")
        K.store(cache, k, v, slots)
    q = synth.heavy_tailed((len(lens), Hq, D), "cuda", seed, "q")
    return cache, torch.from_numpy(bt).cuda(), K.rotate_query(q), torch.tensor(lens, dtype=torch.int32,
                                                                               device="cuda")


def _reference(K, cache, qrot, seq, bt, ml, sm):
    B = qrot.shape[0]
    ws = K.alloc_workspace(cache, B, 24, ml, device="cuda")
    ref = torch.empty((B, 24, 256), dtype=torch.float32, device="cuda")
    K.decode_attn(cache, qrot, seq, bt, ml, sm, ws)
    K.merge(cache, ws, B, 24, seq, ml, ref)
    return ref, K.read_status(ws)


def test_noalloc_matches_workspace_path_twice(K):
    """Two calls in a row, the second one smaller (fewer sequences, shorter):
    it must not see the first call's partials, and each output must equal the
    workspace path's bit for bit (the same kernels on the same inputs)."""
    sm = 1 / math.sqrt(256)
    for call, (seed, lens) in enumerate(((31, [5000, 1300, 777]), (32, [700, 300]))):
        cache, bt, qrot, seq = _problem(K, lens, seed)
        ml = max(lens)
        ref, ref_status = _reference(K, cache, qrot, seq, bt, ml, sm)
        out = torch.full_like(ref, float("nan"))
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        K.decode_noalloc(cache, qrot, seq, bt, ml, sm, out, status=st)
        torch.cuda.synchronize()
        assert ref_status == 0 and K.read_status(st) == 0
        assert torch.isfinite(out).all(), f"call {call}"
        assert torch.equal(out, ref), f"call {call}"


def test_noalloc_reports_a_bad_page(K):
    """A block-table entry outside the pool: the status copy carries
    KVQ_DEV_BAD_PAGE, that sequence's rows come out NaN, the other sequence is
    unaffected and equal to the workspace path; a clean call right after has a
    clean status (the word is cleared per call)."""
    sm = 1 / math.sqrt(256)
    lens = [1500, 900]
    cache, bt, qrot, seq = _problem(K, lens, 33)
    bad = bt.clone()
    bad[1, 3] = cache.num_pages          # one past the pool
    ml = max(lens)
    ref, ref_status = _reference(K, cache, qrot, seq, bad, ml, sm)
    assert ref_status & K.DEV_BAD_PAGE
    out = torch.zeros_like(ref)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.decode_noalloc(cache, qrot, seq, bad, ml, sm, out, status=st)
    torch.cuda.synchronize()
    assert K.read_status(st) & K.DEV_BAD_PAGE
    assert torch.isnan(out[1]).all()
    assert torch.equal(out[0], ref[0])
    K.decode_noalloc(cache, qrot, seq, bt, ml, sm, out, status=st)
    torch.cuda.synchronize()
    assert K.read_status(st) == 0
    assert torch.isfinite(out).all()


def test_noalloc_rejects_problems_beyond_the_scratch(K):
    cache = K.Cache(K.FMT_Q4_HAD32, 4, 256, 16, 4, device="cuda")
    limit = K.lib().kvq_noalloc_scratch_bytes()
    assert limit == 16 << 20
    B, ml = 64, 65536   # 64 x 24 heads x 128 partitions x 1 KB partials >> 16 MiB
    assert K.workspace_size(cache, B, 24, ml) > limit
    q = torch.zeros((B, 24, 256), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(q)
    seq = torch.zeros(B, dtype=torch.int32, device="cuda")
    bt = torch.zeros((B, ml // 16), dtype=torch.int32, device="cuda")
    with pytest.raises(K.KvqError) as e:
        K.decode_noalloc(cache, q, seq, bt, ml, 0.1, out)
    assert e.value.status == K.ERR_WORKSPACE_TOO_SMALL
