"""Pins for the oracle's attention (CPU only).

The oracle evaluates softmax attention with a max subtraction and numpy
matrix products.  These tests check it against other formulations and facts:

* brute force with pure-Python loops and ``math.exp`` without any max
  subtraction, including an explicit causal visibility loop;
* invariants: rows of weights sum to one (V = 1 gives O = 1), constant V
  gives V, joint key/value permutation, a common shift of every key, scale
  0 gives the mean of the visible values;
* causal special cases: with Q = KV row 0 returns v_0; the last real query
  sees every key and equals the dense row; Hq=6 / Hkv=1 equals six
  single-head calls on the shared K/V; padded rows are zero;
* block-sparse: selecting every cube equals dense, and the gather
  formulation equals a dense softmax with the unselected keys masked out;
* planted mistakes (an off-by-one causal mask, a dropped prefix offset, a
  transposed head mapping) each fail at least one of these pins.
"""

import math

import numpy as np
import pytest

from oracle import attention as A


def _rand(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float16)


def _brute(q, k, v, scale, visible):
    """Pure-Python softmax attention; exp of raw scores (inputs kept small)."""
    n, D = q.shape
    m = k.shape[0]
    o = np.zeros((n, D))
    lse = np.zeros(n)
    sc = float(np.float32(scale))
    for i in range(n):
        ws = []
        for j in range(m):
            if visible(i, j):
                s = sc * sum(float(q[i, d]) * float(k[j, d]) for d in range(D))
                ws.append((j, math.exp(s)))
        tot = sum(w for _, w in ws)
        for d in range(D):
            o[i, d] = sum(w * float(v[j, d]) for j, w in ws) / tot
        lse[i] = math.log(tot)
    return o, lse


def test_dense_brute_force():
    q, k, v = _rand((1, 2, 5, 8), 1), _rand((1, 2, 7, 8), 2), _rand((1, 2, 7, 8), 3)
    o, lse = A.dense_attention(q, k, v, 0.35)
    for h in range(2):
        ob, lb = _brute(q[0, h], k[0, h], v[0, h], 0.35, lambda i, j: True)
        assert np.allclose(o[0, h], ob, rtol=1e-12, atol=1e-13)
        assert np.allclose(lse[0, h], lb, rtol=1e-12, atol=1e-13)


def test_causal_brute_force():
    Q, KV, D = 6, 9, 8
    q, k, v = _rand((1, 2, Q, D), 4), _rand((1, 1, KV, D), 5), _rand((1, 1, KV, D), 6)
    q_real = 4
    o, lse = A.causal_prefill_attention(q, k, v, 0.3, q_real)
    prefix = KV - q_real
    for h in range(2):
        ob, lb = _brute(q[0, h, :q_real], k[0, 0], v[0, 0], 0.3, lambda i, j: j <= prefix + i)
        assert np.allclose(o[0, h, :q_real], ob, rtol=1e-12, atol=1e-13)
        assert np.allclose(lse[0, h, :q_real], lb, rtol=1e-12, atol=1e-13)
        assert np.all(o[0, h, q_real:] == 0) and np.all(np.isneginf(lse[0, h, q_real:]))


def test_weights_sum_to_one_and_constant_v():
    q, k = _rand((1, 1, 16, 32), 7, 2.0), _rand((1, 1, 40, 32), 8, 2.0)
    ones = np.ones((1, 1, 40, 32), dtype=np.float16)
    o, _ = A.dense_attention(q, k, ones, 0.2)
    assert np.max(np.abs(o - 1.0)) < 1e-12
    row = _rand((32,), 9)
    const = np.broadcast_to(row, (1, 1, 40, 32)).copy()
    o, _ = A.dense_attention(q, k, const, 0.2)
    assert np.max(np.abs(o - row.astype(np.float64))) < 1e-12


def test_joint_permutation_and_key_shift():
    q, k, v = _rand((1, 1, 10, 16), 10), _rand((1, 1, 30, 16), 11), _rand((1, 1, 30, 16), 12)
    o, lse = A.dense_attention(q, k, v, 0.25)
    p = np.random.default_rng(0).permutation(30)
    o2, lse2 = A.dense_attention(q, k[:, :, p], v[:, :, p], 0.25)
    assert np.allclose(o, o2, rtol=1e-12, atol=1e-13)
    u = np.random.default_rng(1).standard_normal(16)
    ks = k.astype(np.float64) + u          # every score of a row moves by scale * q_i . u
    o3, lse3 = A.dense_attention(q, ks, v, 0.25)
    assert np.allclose(o, o3, rtol=1e-10, atol=1e-11)
    shift = float(np.float32(0.25)) * (q[0, 0].astype(np.float64) @ u)
    assert np.allclose(lse3[0, 0], lse[0, 0] + shift, rtol=1e-10, atol=1e-10)


def test_scale_zero_gives_mean_of_visible_values():
    q, k, v = _rand((1, 1, 6, 8), 13), _rand((1, 1, 11, 8), 14), _rand((1, 1, 11, 8), 15)
    o, _ = A.dense_attention(q, k, v, 0.0)
    assert np.allclose(o[0, 0], v[0, 0].astype(np.float64).mean(axis=0)[None], atol=1e-13)
    o, _ = A.causal_prefill_attention(q, k, v, 0.0, 6)
    prefix = 11 - 6
    for i in range(6):
        want = v[0, 0, :prefix + i + 1].astype(np.float64).mean(axis=0)
        assert np.allclose(o[0, 0, i], want, atol=1e-13)


def _pin_row0(fn):
    q, k, v = _rand((1, 1, 12, 8), 20), _rand((1, 1, 12, 8), 21), _rand((1, 1, 12, 8), 22)
    o, _ = fn(q, k, v, 0.4, 12)                  # Q = KV: query 0 sees only key 0
    return np.allclose(o[0, 0, 0], v[0, 0, 0].astype(np.float64), atol=1e-14)


def _pin_last_row_dense(fn):
    q, k, v = _rand((1, 1, 8, 8), 23), _rand((1, 1, 20, 8), 24), _rand((1, 1, 20, 8), 25)
    o, _ = fn(q, k, v, 0.4, 8)                   # last real query sees all 20 keys
    od, _ = A.attention_rows(q[0, 0, 7:8], k[0, 0], v[0, 0], 0.4)
    return np.allclose(o[0, 0, 7], od[0], rtol=1e-12, atol=1e-13)


def _pin_gqa(fn):
    q, k, v = _rand((1, 6, 8, 8), 26), _rand((1, 2, 20, 8), 27), _rand((1, 2, 20, 8), 28)
    o, _ = fn(q, k, v, 0.4, 8)
    ok = True
    for h in range(6):
        kh = h // 3
        o1, _ = fn(q[:, h:h + 1], k[:, kh:kh + 1], v[:, kh:kh + 1], 0.4, 8)
        ok &= np.allclose(o[0, h], o1[0, 0], rtol=1e-12, atol=1e-13)
    return ok


def _pin_brute(fn):
    q, k, v = _rand((1, 1, 5, 4), 29), _rand((1, 1, 9, 4), 30), _rand((1, 1, 9, 4), 31)
    o, _ = fn(q, k, v, 0.5, 5)
    ob, _ = _brute(q[0, 0], k[0, 0], v[0, 0], 0.5, lambda i, j: j <= 4 + i)
    return np.allclose(o[0, 0], ob, rtol=1e-12, atol=1e-13)


PINS = [_pin_row0, _pin_last_row_dense, _pin_gqa, _pin_brute]


def test_causal_pins_hold_for_oracle():
    for pin in PINS:
        assert pin(A.causal_prefill_attention), pin.__name__


def _mutant(visible_rule, head_rule):
    def fn(q, k, v, scale, q_real):
        B, Hq, Qp, D = q.shape
        Hkv, KV = k.shape[1], k.shape[2]
        o = np.zeros((B, Hq, Qp, D))
        lse = np.zeros((B, Hq, Qp))
        for h in range(Hq):
            kh = head_rule(h, Hq, Hkv)
            r = np.arange(Qp)
            vis = visible_rule(np.arange(KV)[None, :], r[:, None], KV - q_real)
            o[0, h], lse[0, h] = A.attention_rows(q[0, h], k[0, kh], v[0, kh], scale, vis)
        return o, lse
    return fn


@pytest.mark.parametrize("name,mutant", [
    ("strict mask j < pos", _mutant(lambda j, i, p: j < p + i, lambda h, Hq, Hkv: h // (Hq // Hkv))),
    ("prefix offset dropped", _mutant(lambda j, i, p: j <= i, lambda h, Hq, Hkv: h // (Hq // Hkv))),
    ("head map h % Hkv", _mutant(lambda j, i, p: j <= p + i, lambda h, Hq, Hkv: h % Hkv)),
])
def test_planted_mistakes_are_caught(name, mutant):
    assert not all(pin(mutant) for pin in PINS), name


def test_vsa_all_cubes_equals_dense():
    B, H, block, nc, D = 1, 2, 8, 6, 16
    q, k, v = (_rand((B, H, nc * block, D), s) for s in (40, 41, 42))
    idx = np.tile(np.arange(nc, dtype=np.int32)[::-1], (B, H, nc, 1))
    o, lse = A.vsa_sparse_attention(q, k, v, idx, block, 0.25)
    od, lsed = A.dense_attention(q, k, v, 0.25)
    assert np.allclose(o, od, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, lsed, rtol=1e-12, atol=1e-13)


def test_vsa_gather_equals_masked_dense():
    B, H, block, nc, D, topk = 1, 2, 8, 10, 16, 3
    q, k, v = (_rand((B, H, nc * block, D), s) for s in (43, 44, 45))
    rng = np.random.default_rng(3)
    idx = np.sort(np.stack([[rng.choice(nc, topk, replace=False) for _ in range(nc)]
                            for _ in range(H)])[None], axis=-1).astype(np.int32)
    o, _ = A.vsa_sparse_attention(q, k, v, idx, block, 0.25)
    S = nc * block
    for h in range(H):
        vis = np.zeros((S, S), dtype=bool)
        for t in range(S):
            for c in idx[0, h, t // block]:
                vis[t, c * block:(c + 1) * block] = True
        om, _ = A.attention_rows(q[0, h], k[0, h], v[0, h], 0.25, vis)
        assert np.allclose(o[0, h], om, rtol=1e-12, atol=1e-13)


def test_sampled_rows_equal_full_evaluation():
    q, k, v = _rand((1, 3, 20, 8), 50), _rand((1, 1, 30, 8), 51), _rand((1, 1, 30, 8), 52)
    o, lse = A.causal_prefill_attention(q, k, v, 0.3, 18)
    rows = np.array([[2, 17], [0, 3], [1, 0], [2, 19]])
    os_, ls = A.causal_prefill_attention(q, k, v, 0.3, 18, rows=rows)
    for n, (h, i) in enumerate(rows):
        assert np.allclose(os_[n], o[0, h, i], rtol=1e-13, atol=1e-14)
        assert np.isclose(lse[0, h, i], ls[n], rtol=1e-13) or \
            (np.isneginf(ls[n]) and np.isneginf(lse[0, h, i]))


# ------------------------------------------------------------------ additive mask
def _brute_masked(q, k, v, scale, mask):
    """Pure-Python softmax(scale * q.k + mask) v; -inf entries are skipped."""
    n, D = q.shape
    m = k.shape[0]
    o = np.zeros((n, D))
    lse = np.zeros(n)
    sc = float(np.float32(scale))
    for i in range(n):
        ws = []
        for j in range(m):
            b = float(mask[i, j])
            if b == -math.inf:
                continue
            s = sc * sum(float(q[i, d]) * float(k[j, d]) for d in range(D)) + b
            ws.append((j, math.exp(s)))
        if not ws:
            lse[i] = -math.inf
            continue
        tot = sum(w for _, w in ws)
        for d in range(D):
            o[i, d] = sum(w * float(v[j, d]) for j, w in ws) / tot
        lse[i] = math.log(tot)
    return o, lse


def _mask(shape, seed, hide=0.2):
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(shape) * 1.5).astype(np.float16)
    m[rng.random(shape) < hide] = -np.inf
    return m


def test_masked_brute_force():
    q, k, v = _rand((1, 2, 5, 8), 60), _rand((1, 2, 9, 8), 61), _rand((1, 2, 9, 8), 62)
    mask = _mask((5, 9), 63)
    mask[2] = -np.inf                                   # one fully hidden row
    o, lse = A.dense_masked_attention(q, k, v, mask, 0.4)
    for h in range(2):
        ob, lb = _brute_masked(q[0, h], k[0, h], v[0, h], 0.4, mask)
        assert np.allclose(o[0, h], ob, rtol=1e-12, atol=1e-13)
        assert np.array_equal(np.isneginf(lse[0, h]), np.isneginf(lb))
        fin = np.isfinite(lb)
        assert np.allclose(lse[0, h][fin], lb[fin], rtol=1e-12, atol=1e-13)
    assert np.all(o[0, :, 2] == 0)


def test_mask_zero_equals_dense_and_inf_equals_visibility():
    q, k, v = _rand((1, 2, 6, 8), 64), _rand((1, 2, 11, 8), 65), _rand((1, 2, 11, 8), 66)
    o0, l0 = A.dense_masked_attention(q, k, v, np.zeros((6, 11), np.float16), 0.3)
    od, ld = A.dense_attention(q, k, v, 0.3)
    assert np.allclose(o0, od, rtol=1e-14, atol=1e-15) and np.allclose(l0, ld, rtol=1e-14)
    vis = np.random.default_rng(67).random((6, 11)) < 0.6
    vis[:, 0] = True
    om, lm = A.dense_masked_attention(q, k, v, np.where(vis, 0.0, -np.inf).astype(np.float16), 0.3)
    for h in range(2):
        ov, lv = A.attention_rows(q[0, h], k[0, h], v[0, h], 0.3, visible=vis)
        assert np.allclose(om[0, h], ov, rtol=1e-14, atol=1e-15)
        assert np.allclose(lm[0, h], lv, rtol=1e-14)


def test_mask_row_constant_shifts_lse_only():
    q, k, v = _rand((1, 1, 4, 8), 68), _rand((1, 1, 10, 8), 69), _rand((1, 1, 10, 8), 70)
    base = _mask((4, 10), 71, hide=0.0)
    shift = np.array([0.5, -1.25, 2.0, 0.0])[:, None]
    o1, l1 = A.dense_masked_attention(q, k, v, base, 0.3)
    o2, l2 = A.dense_masked_attention(q, k, v, (base.astype(np.float64) + shift), 0.3)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(l2[0, 0] - l1[0, 0], shift[:, 0], rtol=1e-12, atol=1e-12)


def test_mask_broadcast_per_head_slices():
    q, k, v = _rand((2, 3, 4, 8), 72), _rand((2, 3, 7, 8), 73), _rand((2, 3, 7, 8), 74)
    per_head = _mask((1, 3, 4, 7), 75)
    o, _ = A.dense_masked_attention(q, k, v, per_head, 0.5)
    for b in range(2):
        for h in range(3):
            oh, _ = A.dense_masked_attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                             v[b:b + 1, h:h + 1], per_head[0, h], 0.5)
            assert np.allclose(o[b, h], oh[0, 0], rtol=1e-14, atol=1e-15)
