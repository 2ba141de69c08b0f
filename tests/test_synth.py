"""The seeded input generators draw what their recipes say: the heavy-tailed
decode data (13 of 256 channels per head Student-t(3) x 10, the rest N(0,1),
one subset per head across chunked fills), the tiny-config outliers, the fp8
latent rows' log-normal row magnitudes, and the index generators.  Medians of
|x| are checked against their closed forms: 0.6745 for N(0,1) and
10 x 0.7649 for 10 t(3) (the t(3) quartile: tan(theta) / sqrt(3) = 0.7649 solves
the t(3) CDF at 3/4)."""
import math

import numpy as np
import torch

from bit_quantized_kv_store_gb300 import synth


def _t3_quartile():
    # CDF of t(3): 1/2 + (atan(u) + u / (1 + u^2)) / pi with u = x / sqrt(3); solve = 3/4 by bisection
    lo, hi = 0.0, 3.0
    for _ in range(100):
        mid = (lo + hi) / 2
        u = mid / math.sqrt(3)
        if 0.5 + (math.atan(u) + u / (1 + u * u)) / math.pi < 0.75:
            lo = mid
        else:
            hi = mid
    return lo


def test_heavy_tailed_channels():
    x = synth.heavy_tailed((6000, 4, 256), "cpu", "t", 1, dtype=torch.float32).numpy()
    med = np.median(np.abs(x), axis=0)                      # [heads, 256]
    heavy = med > 3.0
    assert (heavy.sum(1) == 13).all()                      # round(0.05 * 256) per head
    assert not np.array_equal(heavy[0], heavy[1])          # a subset per head
    q = _t3_quartile()
    assert abs(q - 0.7649) < 1e-3
    assert np.allclose(med[heavy], 10 * q, rtol=0.08)
    assert np.allclose(med[~heavy], 0.6745, rtol=0.06)


def test_heavy_tailed_subset_is_kept_across_chunks_and_seeded():
    a = synth.heavy_tailed((3000, 2, 256), "cpu", "L0", "k", 0, subset=("L0", "k"), dtype=torch.float32).numpy()
    b = synth.heavy_tailed((3000, 2, 256), "cpu", "L0", "k", 3000, subset=("L0", "k"), dtype=torch.float32).numpy()
    assert not np.array_equal(a, b)                        # other values ...
    ha = np.median(np.abs(a), axis=0) > 3.0
    hb = np.median(np.abs(b), axis=0) > 3.0
    assert np.array_equal(ha, hb)                          # ... the same heavy channels
    c = synth.heavy_tailed((3000, 2, 256), "cpu", "L0", "k", 0, subset=("L0", "k"), dtype=torch.float32).numpy()
    assert np.array_equal(a, c)                            # same keys, same tensor


def test_outlier_normal():
    x = synth.outlier_normal((5000, 3, 64), 4, 20.0, "cpu", "o").numpy()
    med = np.median(np.abs(x), axis=0)
    big = med > 5.0
    assert (big.sum(1) == 4).all()
    assert np.allclose(med[big], 20 * 0.6745, rtol=0.08)
    assert np.allclose(med[~big], 0.6745, rtol=0.08)


def test_latent_rows_have_log_normal_magnitudes():
    x = synth.latent_rows(4000, 576, "cpu", "lat").numpy().astype(np.float64)
    log_rms = np.log(np.sqrt((x * x).mean(1)))
    # rms of 576 N(0,1) values is ~1 (log ~0); the row factor exp(N(0,1)) sets the rest
    assert abs(log_rms.mean()) < 0.08 and abs(log_rms.std() - 1.0) < 0.06


def test_index_generators():
    L = synth.ragged_lengths(5000, 1024, 65536, "r").numpy()
    assert L.min() >= 1024 and L.max() <= 65536 and abs(L.mean() - (1024 + 65536) / 2) < 1000
    p = synth.page_permutation(777, "p").numpy()
    assert np.array_equal(np.sort(p), np.arange(777))
    s = synth.distinct_sorted(300, 1000, "s").numpy()
    assert len(np.unique(s)) == 300 and (np.diff(s) > 0).all() and s.min() >= 0 and s.max() < 1000
    assert np.array_equal(synth.distinct_sorted(64, 64, "s").numpy(), np.arange(64))
    w = synth.sign_mask(32 * 400, "m")
    assert w.dtype == torch.int32 and w.shape == (400,)
    bits = (w.numpy().astype(np.int64)[:, None] >> np.arange(32)) & 1
    assert abs(bits.mean() - 0.5) < 0.02
    assert 0.3 < bits[:, 31].mean() < 0.7                  # the sign bit carries a sign too
