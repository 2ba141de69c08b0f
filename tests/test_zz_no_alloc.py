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

TOL = 2e-3   # the attention tolerance used by the other parity tests


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


def test_noalloc_matches_workspace_path_twice(K):
    lens = [5000, 1300, 777]
    sm = 1 / math.sqrt(256)
    for call, seed in enumerate((31, 32)):   # two calls in a row, different inputs
        cache, bt, qrot, seq = _problem(K, lens, seed)
        ml = max(lens)
        ws = K.alloc_workspace(cache, len(lens), 24, ml, device="cuda")
        ref = torch.empty((len(lens), 24, 256), dtype=torch.float32, device="cuda")
        K.decode_attn(cache, qrot, seq, bt, ml, sm, ws)
        K.merge(cache, ws, len(lens), 24, seq, ml, ref)
        out = torch.full_like(ref, float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        K.decode_noalloc(cache, qrot, seq, bt, ml, sm, out, status=st)
        torch.cuda.synchronize()
        assert K.read_status(st) == 0
        r, o = ref.cpu().numpy().astype(np.float64), out.cpu().numpy().astype(np.float64)
        for b in range(len(lens)):
            assert np.isfinite(o[b]).all()
            assert np.abs(o[b] - r[b]).max() <= TOL * np.abs(r[b]).max(), f"call {call} seq {b}"


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
