"""Pins for the oracle's VSA pooling, scores and top-k (CPU only).

* Pooling: a constant cube pools to that constant; exactly summable data
  gives the exact mean; general data stays within the recursive-summation
  error bound of the exact mean; and a case built so that only the
  sequential token order gives the stated result pins the order reading.
* Scores: integer-valued inputs (exact in FP32) equal numpy's int64 matrix
  product; general inputs stay within gamma_D * sum |q||k| of the exact dot
  product; a case that only sequential, non-fused evaluation reproduces pins
  that reading.
* Top-k: equal to a brute-force rank count; ties go to the lower index;
  top-k = all returns every index; on data whose 64th/65th exact scores are
  farther apart than the FP32 error bound the FP32 selection equals the
  exact-arithmetic selection.
"""

import numpy as np

from oracle.vsa import cube_scores_fp32, pool_means_fp32, topk_blocks, vsa_select

U = 2.0 ** -24   # unit roundoff of FP32


def test_pool_constant_cube():
    x = np.full((2, 3 * 64, 8), 0.7, dtype=np.float16)
    m = pool_means_fp32(x, 64)
    assert m.shape == (2, 3, 8) and m.dtype == np.float32
    assert np.all(m == np.float32(np.float16(0.7)))


def test_pool_exactly_summable_equals_exact_mean():
    rng = np.random.default_rng(0)
    x = (rng.integers(-64, 64, (4, 256, 16)) / 16.0).astype(np.float16)
    m = pool_means_fp32(x, 64)
    exact = x.astype(np.float64).reshape(4, 4, 64, 16).sum(axis=2) / 64.0
    assert np.array_equal(m.astype(np.float64), exact)


def test_pool_within_summation_bound():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((3, 512, 32)) * 3).astype(np.float16)
    m = pool_means_fp32(x, 64).astype(np.float64)
    xd = x.astype(np.float64).reshape(3, 8, 64, 32)
    exact = xd.sum(axis=2) / 64.0
    bound = 63 * U / (1 - 63 * U) * np.abs(xd).sum(axis=2) / 64.0
    assert np.all(np.abs(m - exact) <= bound)


def test_pool_sequential_order():
    # 1.0 followed by 63 copies of 2^-24: each sequential FP32 addition
    # 1 + 2^-24 is a tie that rounds back to 1, so the sum is exactly 1.
    # Any other order (pairwise, reversed) accumulates the small terms first.
    x = np.full((64, 1), 2.0 ** -24, dtype=np.float16)
    x[0, 0] = 1.0
    assert pool_means_fp32(x, 64)[0, 0] == np.float32(1.0 / 64.0)
    y = x[::-1].copy()            # small terms first: their sum 63 * 2^-24 survives
    assert pool_means_fp32(y, 64)[0, 0] == np.float32((1.0 + 63 * 2.0 ** -24) / 64.0)


def test_scores_integer_inputs_match_int64_matmul():
    rng = np.random.default_rng(2)
    qi = rng.integers(-50, 50, (3, 20, 128))
    ki = rng.integers(-50, 50, (3, 30, 128))
    s = cube_scores_fp32(qi.astype(np.float32), ki.astype(np.float32))
    ref = np.einsum("hqd,hkd->hqk", qi, ki)
    assert np.array_equal(s.astype(np.int64), ref)


def test_scores_within_error_bound():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 16, 128)).astype(np.float32)
    k = rng.standard_normal((2, 24, 128)).astype(np.float32)
    s = cube_scores_fp32(q, k).astype(np.float64)
    qd, kd = q.astype(np.float64), k.astype(np.float64)
    exact = np.einsum("hqd,hkd->hqk", qd, kd)
    g = 128 * U / (1 - 128 * U)
    bound = g * np.einsum("hqd,hkd->hqk", np.abs(qd), np.abs(kd))
    assert np.all(np.abs(s - exact) <= bound)


def test_scores_sequential_unfused_order():
    # products: 1, then 127 products equal to 2^-25 (0.5 ulp of 1): sequential
    # FP32 adds round each tie back to 1; a fused or reordered sum would not.
    q = np.full((1, 128), 2.0 ** -13, dtype=np.float32)
    k = np.full((1, 128), 2.0 ** -12, dtype=np.float32)
    q[0, 0] = 1.0
    k[0, 0] = 1.0
    assert cube_scores_fp32(q, k)[0, 0] == np.float32(1.0)
    assert cube_scores_fp32(q[:, ::-1].copy(), k[:, ::-1].copy())[0, 0] > np.float32(1.0)


def _brute_topk(s, k):
    n = s.shape[-1]
    out = []
    for row in s.reshape(-1, n):
        rank = [(row > row[j]).sum() + (row[:j] == row[j]).sum() for j in range(n)]
        out.append(sorted(j for j in range(n) if rank[j] < k))
    return np.array(out).reshape(s.shape[:-1] + (k,))


def test_topk_matches_rank_count_random_and_ties():
    rng = np.random.default_rng(4)
    s = rng.standard_normal((3, 7, 40)).astype(np.float32)
    assert np.array_equal(topk_blocks(s, 9), _brute_topk(s, 9))
    t = rng.integers(0, 4, (3, 7, 40)).astype(np.float32)      # heavy ties
    assert np.array_equal(topk_blocks(t, 9), _brute_topk(t, 9))
    z = np.zeros((1, 2, 40), np.float32)
    assert np.array_equal(topk_blocks(z, 5)[0, 0], np.arange(5))
    assert np.array_equal(topk_blocks(s, 40)[1, 2], np.arange(40))


def test_duplicate_key_cubes_prefer_lower_index():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 8 * 64, 16)).astype(np.float16)
    k = rng.standard_normal((1, 1, 8 * 64, 16)).astype(np.float16)
    k[0, 0, 5 * 64:6 * 64] = k[0, 0, 2 * 64:3 * 64]           # cube 5 duplicates cube 2
    idx = vsa_select(q, k, 64, 8 - 1)
    for row in idx[0, 0]:
        # cubes 2 and 5 have identical scores: if only one is kept it is 2
        assert not (5 in row and 2 not in row)
    assert np.all(np.diff(idx, axis=-1) > 0)


def test_fp32_selection_equals_exact_selection_away_from_ties():
    rng = np.random.default_rng(6)
    q = (rng.standard_normal((2, 16 * 64, 32)) * 0.5 + 0.3).astype(np.float16)
    k = (rng.standard_normal((2, 96 * 64, 32)) * 0.5 + 0.3).astype(np.float16)
    idx = vsa_select(q, k, 64, 20)
    qd = q.astype(np.float64).reshape(2, 16, 64, 32).mean(axis=2)
    kd = k.astype(np.float64).reshape(2, 96, 64, 32).mean(axis=2)
    exact = np.einsum("hqd,hkd->hqk", qd, kd)
    checked = 0
    for h in range(2):
        for i in range(16):
            srt = np.sort(exact[h, i])[::-1]
            margin = srt[19] - srt[20]
            bound = 1e-5 * np.abs(qd[h, i]) @ np.abs(kd[h]).max(axis=0)
            if margin > 4 * bound:
                want = np.sort(np.argsort(-exact[h, i], kind="stable")[:20])
                assert np.array_equal(idx[h, i], want)
                checked += 1
    assert checked >= 24
