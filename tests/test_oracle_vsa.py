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


# ------------------------------------------------------------------ boundary cubes and prefix
import math  # noqa: E402

import pytest  # noqa: E402

from oracle import attention as A  # noqa: E402


def _valid_counts(nc, seed):
    rng = np.random.default_rng(seed)
    v = rng.integers(1, 65, nc)
    v[0] = 64
    return v


def test_partial_pool_equals_sequential_mean_of_real_tokens():
    rng = np.random.default_rng(20)
    nc, D = 5, 8
    x = rng.standard_normal((2, nc * 64, D)).astype(np.float16)
    val = _valid_counts(nc, 21)
    m = pool_means_fp32(x, 64, val)
    for b in range(2):
        for c in range(nc):
            for d in range(D):
                acc = np.float32(0.0)
                for t in range(val[c]):
                    acc = np.float32(acc + np.float32(x[b, c * 64 + t, d]))
                assert m[b, c, d] == np.float32(acc / np.float32(val[c]))


def _layout(prefix, nc, D, seed):
    rng = np.random.default_rng(seed)
    S = prefix + nc * 64
    q, k, v = (rng.standard_normal((1, 2, S, D)).astype(np.float16) for _ in range(3))
    return q, k, v, _valid_counts(nc, seed + 1)


def test_padding_contents_are_ignored():
    q, k, v, val = _layout(64, 6, 8, 22)
    idx = vsa_select(q, k, 64, 3, val, prefix=64)
    o, lse = A.vsa_sparse_attention(q, k, v, idx, 64, 0.4, valid=val, prefix=64)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for c in range(6):
        pad = slice(64 + c * 64 + val[c], 64 + (c + 1) * 64)
        q2[..., pad, :] = 7.0
        k2[..., pad, :] = -5.0
        v2[..., pad, :] = 100.0
    assert np.array_equal(vsa_select(q2, k2, 64, 3, val, prefix=64), idx)
    o2, lse2 = A.vsa_sparse_attention(q2, k2, v2, idx, 64, 0.4, valid=val, prefix=64)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def _brute_rows(q, k, v, scale, keys):
    out = []
    sc = float(np.float32(scale))
    for i, ks in keys:
        ws = [(j, math.exp(sc * sum(float(q[i, d]) * float(k[j, d]) for d in range(q.shape[1]))))
              for j in ks]
        tot = sum(w for _, w in ws)
        out.append([sum(w * float(v[j, d]) for j, w in ws) / tot for d in range(q.shape[1])])
    return np.array(out)


def _pin_prefix_and_partial(fn):
    q, k, v, val = _layout(64, 4, 4, 23)
    idx = np.array([[[0, 2], [1, 3], [0, 3], [2, 3]]] * 2)[None].astype(np.int32)
    o, lse = fn(q, k, v, idx, 64, 0.5, valid=val, prefix=64)
    real = [64 + c * 64 + t for c in range(4) for t in range(val[c])]
    ok = True
    for h in range(2):
        rows = [(i, list(range(64)) + real) for i in (0, 17, 63)]
        for c in range(4):
            sel = [64 + kc * 64 + t for kc in idx[0, h, c] for t in range(val[kc])]
            rows.append((64 + c * 64, sel))
            rows.append((64 + c * 64 + val[c] - 1, sel))
        want = _brute_rows(q[0, h], k[0, h], v[0, h], 0.5, rows)
        got = np.array([o[0, h, i] for i, _ in rows])
        ok &= np.allclose(got, want, rtol=1e-12, atol=1e-13)
        for c in range(4):                       # padding query slots
            pads = np.arange(64 + c * 64 + val[c], 64 + (c + 1) * 64)
            ok &= bool(np.all(o[0, h, pads] == 0)) and bool(np.all(np.isneginf(lse[0, h, pads])))
    return ok


def test_prefix_and_partial_cubes_brute_force():
    assert _pin_prefix_and_partial(A.vsa_sparse_attention)


def test_full_cubes_without_prefix_unchanged():
    q, k, v, _ = _layout(0, 4, 8, 24)
    idx = vsa_select(q, k, 64, 2)
    o1, l1 = A.vsa_sparse_attention(q, k, v, idx, 64, 0.3)
    o2, l2 = A.vsa_sparse_attention(q, k, v, idx, 64, 0.3, valid=np.full(4, 64), prefix=0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.array_equal(idx, vsa_select(q, k, 64, 2, np.full(4, 64)))


def _mutant_sparse(prefix_sees_video=True, mask_padding=True):
    def fn(q, k, v, idx, block, scale, valid=None, prefix=0):
        val = np.asarray(valid) if (valid is not None and mask_padding) else None
        o, lse = A.vsa_sparse_attention(q, k, v, idx, block, scale, valid=val, prefix=prefix)
        if not prefix_sees_video:
            for h in range(q.shape[1]):
                o[0, h, :prefix], lse[0, h, :prefix] = A.attention_rows(
                    q[0, h, :prefix], k[0, h, :prefix], v[0, h, :prefix], scale)
        return o, lse
    return fn


@pytest.mark.parametrize("name,fn", [
    ("padding keys not hidden", _mutant_sparse(mask_padding=False)),
    ("prefix queries see only the prefix", _mutant_sparse(prefix_sees_video=False)),
])
def test_planted_vsa_mistakes_are_caught(name, fn):
    assert not _pin_prefix_and_partial(fn), name


def test_planted_pool_by_block_is_caught():
    rng = np.random.default_rng(25)
    x = rng.standard_normal((1, 3 * 64, 4)).astype(np.float16)
    val = np.array([64, 40, 9])
    wrong = pool_means_fp32(x, 64, val) * val[None, :, None].astype(np.float32) / np.float32(64)
    assert not np.allclose(wrong, pool_means_fp32(x, 64, val))
