"""Pins for the oracle's VSA pooling, exact scores, top-k and coarse branch (CPU only).

* Pooling: a constant cube pools to that constant; exactly summable data
  gives the exact mean; general data stays within the recursive-summation
  error bound of the exact mean; and a case built so that only the
  sequential token order gives the stated result pins the order reading.
* The exact grid: pooled FP16 data over the whole FP16 range (huge values,
  subnormals, zeros, cancelling cubes, boundary counts) lies on the 2^-53
  grid the exact scores use, limb by limb equal to the value as a fraction.
* Exact scores: equal to sums of ``fractions.Fraction`` products on those
  extreme inputs; integer inputs equal numpy's int64 matrix product; a case
  that FP32 sequential scoring ranks the other way, and one that float64
  scoring cannot separate, are ranked by the exact value.
* Top-k: equal to a full sort by (exact score descending, index ascending)
  on random and tie-heavy inputs (duplicate, zero and constant cubes); a
  transposed selection is caught.
* Coarse branch: equal to a pure-Python softmax over Fraction-exact scores;
  scale 0 gives the mean pooled value, constant values give that constant,
  one key cube gives its pooled value; the gated combination leaves prefix
  and padding rows alone; a branch restricted to the selected cubes is caught.
"""

from fractions import Fraction
import math

import pytest

import numpy as np

from oracle.vsa import (coarse_attention, exact_scores, exact_scores_float, gated_output,
                        grid_limbs, pool_means_fp32, topk_blocks, topk_exact, vsa_select)

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


def _fraction_score(qv, kv):
    return sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qv, kv))


def _digits_value(parts, idx):
    top, d3, d2, d1, d0 = (int(p[idx]) for p in parts)
    return Fraction(top * 2 ** 92 + d3 * 2 ** 69 + d2 * 2 ** 46 + d1 * 2 ** 23 + d0, 2 ** 106)


def _pooled_extremes(seed):
    """Pooled FP16 data over the whole FP16 range: huge values, subnormals, zeros,
    cancelling cubes, boundary counts that are not powers of two."""
    rng = np.random.default_rng(seed)
    nc, D = 12, 128
    mag = 2.0 ** rng.integers(-24, 16, (nc * 64, D))
    x = (rng.choice([-1.0, 1.0], (nc * 64, D)) * mag * rng.uniform(1, 2, (nc * 64, D)))
    x = np.clip(x, -65504, 65504).astype(np.float16)
    x[:64] = 0                                        # an all-zero cube
    x[64:128:2] = -x[65:128:2]                        # a cube that nearly cancels
    counts = rng.integers(1, 65, nc)
    counts[3] = 64
    return x, counts


def test_pooled_means_lie_on_the_exact_grid():
    for seed in range(3):
        x, counts = _pooled_extremes(seed)
        m = pool_means_fp32(x[None], 64, counts)
        a0, a1, a2 = grid_limbs(m)
        back = (a0 + a1.astype(object) * 2 ** 23 + a2.astype(object) * 2 ** 46)
        for i in np.ndindex(m.shape):
            assert Fraction(int(back[i]), 2 ** 53) == Fraction(float(m[i]))
        assert np.all(np.abs(np.stack([a0, a1, a2])) < 2 ** 23)


def test_grid_limbs_rejects_values_off_the_grid():
    for bad in (2.0 ** -60, 2.0 ** 16, np.inf, np.nan):
        with pytest.raises(ValueError):
            grid_limbs(np.array([bad], np.float32))


def test_exact_scores_equal_fraction_sums():
    for seed in range(2):
        x, counts = _pooled_extremes(seed)
        y, _ = _pooled_extremes(seed + 10)
        qm = pool_means_fp32(x[None], 64, counts)
        km = pool_means_fp32(y[None], 64, counts)
        parts = exact_scores(qm, km)
        for i in range(qm.shape[1]):
            for j in range(km.shape[1]):
                assert _digits_value(parts, (0, i, j)) == _fraction_score(qm[0, i], km[0, j])
        assert np.all((parts[1] >= 0) & (parts[1] < 2 ** 23))


def test_exact_scores_integer_inputs_match_int64_matmul():
    rng = np.random.default_rng(2)
    qi = rng.integers(-50, 50, (3, 20, 128))
    ki = rng.integers(-50, 50, (3, 30, 128))
    s = exact_scores_float(qi.astype(np.float32), ki.astype(np.float32))
    ref = np.einsum("hqd,hkd->hqk", qi, ki)
    assert np.array_equal(s, ref.astype(np.float64))


def _brute_exact_topk(qm, km, topk):
    out = []
    for i in range(qm.shape[0]):
        sc = [(-_fraction_score(qm[i], km[j]), j) for j in range(km.shape[0])]
        out.append(sorted(j for _, j in sorted(sc)[:topk]))
    return np.array(out, dtype=np.int32)


def test_topk_exact_equals_full_sort_random_and_ties():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((6 * 64, 16)).astype(np.float16)
    k = rng.standard_normal((40 * 64, 16)).astype(np.float16)
    k[5 * 64:6 * 64] = k[2 * 64:3 * 64]                 # duplicate cube: exact tie
    k[7 * 64:9 * 64] = 0                                # zero cubes: exact ties
    k[20 * 64:21 * 64] = k[30 * 64:31 * 64]
    qm, km = pool_means_fp32(q, 64), pool_means_fp32(k, 64)
    for topk in (1, 9, 40):
        assert np.array_equal(topk_exact(qm, km, topk), _brute_exact_topk(qm, km, topk))
    const = np.full((3 * 64, 16), 0.5, np.float16)      # every score equal: lowest indices
    cm = pool_means_fp32(const, 64)
    assert np.array_equal(topk_exact(cm, cm, 2), [[0, 1]] * 3)


def test_exact_order_is_not_fp32_order():
    # key 1: products 1, 2^-25, 2^-25 (exact 1 + 2^-24); key 0: products 1, 2^-25
    # (exact 1 + 2^-25).  Sequential FP32 rounds both to 1.0 (a tie, so key 0),
    # the exact scores rank key 1 first.
    q = np.zeros((1, 128), np.float32)
    q[0, :3] = [1.0, 2.0 ** -13, 2.0 ** -13]
    k = np.zeros((2, 128), np.float32)
    k[0, :2] = [1.0, 2.0 ** -12]
    k[1, :3] = [1.0, 2.0 ** -12, 2.0 ** -12]
    assert np.array_equal(topk_exact(q, k, 1), [[1]])
    seq = np.float32(0)
    for d in range(128):
        seq = np.float32(seq + np.float32(q[0, d] * k[0, d]))
    assert seq == np.float32(1.0)


def test_planted_fp64_score_is_caught():
    # exact scores 2^10 + 2^-60 (key 1) and 2^10 (key 0): float64 cannot tell them
    # apart and would keep key 0 on the index tie-break.
    q = np.zeros((1, 128), np.float32)
    q[0, :2] = [2.0 ** 5, 2.0 ** -30]
    k = np.zeros((2, 128), np.float32)
    k[0, 0] = 2.0 ** 5
    k[1, :2] = [2.0 ** 5, 2.0 ** -30]
    fp64 = topk_blocks(np.einsum("qd,kd->qk", q.astype(np.float64), k.astype(np.float64)), 1)
    assert np.array_equal(fp64, [[0]])
    assert np.array_equal(topk_exact(q, k, 1), [[1]])


def test_planted_transposed_selection_is_caught():
    rng = np.random.default_rng(7)
    qm = pool_means_fp32(rng.standard_normal((5 * 64, 8)).astype(np.float16), 64)
    km = pool_means_fp32(rng.standard_normal((11 * 64, 8)).astype(np.float16), 64)
    want = _brute_exact_topk(qm, km, 3)
    assert np.array_equal(topk_exact(qm, km, 3), want)
    wrong = topk_exact(km, qm, 3)                        # ranks query cubes per key cube
    assert wrong.shape != want.shape or not np.array_equal(wrong, want)


def _brute_topk(s, k):
    n = s.shape[-1]
    out = []
    for row in s.reshape(-1, n):
        rank = [(row > row[j]).sum() + (row[:j] == row[j]).sum() for j in range(n)]
        out.append(sorted(j for j in range(n) if rank[j] < k))
    return np.array(out).reshape(s.shape[:-1] + (k,))


def test_topk_blocks_matches_rank_count_random_and_ties():
    rng = np.random.default_rng(4)
    s = rng.standard_normal((3, 7, 40)).astype(np.float32)
    assert np.array_equal(topk_blocks(s, 9), _brute_topk(s, 9))
    t = rng.integers(0, 4, (3, 7, 40)).astype(np.float32)      # heavy ties
    assert np.array_equal(topk_blocks(t, 9), _brute_topk(t, 9))


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


# ------------------------------------------------------------------ coarse branch
def _brute_coarse(qm, km, vm, scale):
    out = []
    sc = float(np.float32(scale))
    for i in range(qm.shape[0]):
        logits = [sc * float(_fraction_score(qm[i], km[j])) for j in range(km.shape[0])]
        mx = max(logits)
        w = [math.exp(x - mx) for x in logits]
        tot = sum(w)
        out.append([sum(w[j] * float(vm[j, d]) for j in range(len(w))) / tot
                    for d in range(vm.shape[1])])
    return np.array(out)


def test_coarse_attention_brute_force():
    rng = np.random.default_rng(30)
    q, k, v = (rng.standard_normal((1, 2, 7 * 64, 8)).astype(np.float16) for _ in range(3))
    counts = np.array([64, 10, 64, 33, 1, 64, 50])
    oc = coarse_attention(q, k, v, 64, 0.7, valid=counts)
    for h in range(2):
        qm, km, vm = (pool_means_fp32(x[0, h], 64, counts) for x in (q, k, v))
        assert np.allclose(oc[0, h], _brute_coarse(qm, km, vm, 0.7), rtol=1e-12, atol=1e-14)


def test_coarse_attention_special_cases():
    rng = np.random.default_rng(31)
    q, k, v = (rng.standard_normal((1, 1, 5 * 64, 8)).astype(np.float16) for _ in range(3))
    vm = pool_means_fp32(v[0, 0], 64).astype(np.float64)
    # scale 0: uniform weights over all key cubes -> the mean of the pooled values
    assert np.allclose(coarse_attention(q, k, v, 64, 0.0)[0, 0], vm.mean(axis=0)[None], atol=1e-15)
    # constant values: every output is that constant
    vc = np.full_like(v, 0.375)
    assert np.allclose(coarse_attention(q, k, vc, 64, 0.9), 0.375, atol=1e-15)
    # one key cube: the output is its pooled value
    one = coarse_attention(q, k[:, :, :64], v[:, :, :64], 64, 0.9)
    assert np.allclose(one[0, 0], np.broadcast_to(vm[0], (5, 8)), atol=1e-15)


def test_gated_output_layout():
    rng = np.random.default_rng(32)
    prefix, nc, D = 64, 3, 4
    S = prefix + nc * 64
    fine = rng.standard_normal((1, 1, S, D))
    counts = np.array([64, 20, 7])
    for c in range(nc):
        fine[:, :, prefix + c * 64 + counts[c]:prefix + (c + 1) * 64] = 0
    oc = rng.standard_normal((1, 1, nc, D))
    g = rng.standard_normal((1, 1, S, D))
    o = gated_output(fine, oc, g, 64, counts, prefix)
    assert np.array_equal(o[:, :, :prefix], fine[:, :, :prefix])
    for c in range(nc):
        r = prefix + c * 64
        assert np.allclose(o[0, 0, r:r + counts[c]], fine[0, 0, r:r + counts[c]] +
                           g[0, 0, r:r + counts[c]] * oc[0, 0, c], atol=0)
        assert np.all(o[0, 0, r + counts[c]:r + 64] == 0)
    assert np.array_equal(gated_output(fine, oc, np.zeros_like(g), 64, counts, prefix), fine)


def test_planted_coarse_over_selected_cubes_only_is_caught():
    rng = np.random.default_rng(33)
    q, k, v = (rng.standard_normal((1, 1, 6 * 64, 8)).astype(np.float16) for _ in range(3))
    oc = coarse_attention(q, k, v, 64, 0.5)
    idx = vsa_select(q, k, 64, 2)
    qm, km, vm = (pool_means_fp32(x[0, 0], 64) for x in (q, k, v))
    wrong = np.array([_brute_coarse(qm[i:i + 1], km[idx[0, 0, i]], vm[idx[0, 0, i]], 0.5)[0]
                      for i in range(6)])
    assert not np.allclose(wrong, oc[0, 0], atol=1e-6)


# ------------------------------------------------------------------ boundary cubes and prefix
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
