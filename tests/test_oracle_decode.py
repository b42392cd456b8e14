"""Pins for the oracle's paged E4M3 decode attention (CPU only).

``oracle.decode.paged_decode_attention`` composes the bridge with causal
softmax attention.  These tests check it against facts that do not use it:

* brute force: a pure-Python walk over the page table, an E4M3 decode written
  from the bit fields, numpy's own double -> FP16 rounding and ``math.exp``
  softmax without a max subtraction;
* a single cached token (kv_len = nq = 1) returns that token's FP16 value;
* permuting the physical pages (and the table with them) changes nothing;
* bytes outside the live length (the rest of the last page, pages the
  table does not reach) change nothing;
* with an identity table, the new-token rows equal the causal prefill of the
  same positions over the bridged cache;
* planted mistakes (a query position off by one, the head map h % Hkv, a
  gather that ignores the page table, a dropped V scale) each fail a pin.
"""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import decode as DEC
from oracle import e4m3 as E
from oracle.fp16 import fp16_bits_to_f64


def _e4m3_scalar(byte):
    """E4M3 ("fn") from the bit fields: sign, 4-bit exponent (bias 7), 3-bit mantissa."""
    s, e, m = byte >> 7, (byte >> 3) & 15, byte & 7
    mag = m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def _case(B, Hq, Hkv, nq, D, ps, kv_lens, seed, max_pages=None, spare=2):
    """Small random decode problem with moderate codes (|value| < 8)."""
    rng = np.random.default_rng(seed)
    n_log = [-(-n // ps) for n in kv_lens]
    max_pages = max(n_log) + 1 if max_pages is None else max_pages
    P = sum(n_log) + spare
    exp_field = rng.integers(3, 10, size=(2, P, ps, Hkv, D))
    mant = rng.integers(0, 8, size=(2, P, ps, Hkv, D))
    sign = rng.integers(0, 2, size=(2, P, ps, Hkv, D))
    codes = ((sign << 7) | (exp_field << 3) | mant).astype(np.uint8)
    perm = rng.permutation(P)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, :n_log[b]] = perm[at:at + n_log[b]]
        at += n_log[b]
    q = (rng.standard_normal((B, Hq, nq, D)) * 0.5).astype(np.float16)
    return q, codes[0], codes[1], table, np.asarray(kv_lens, dtype=np.int32)


def _brute(q, kp, vp, table, kv_lens, ks, vs, scale):
    B, Hq, nq, D = q.shape
    ps, Hkv = kp.shape[1], kp.shape[2]
    group = Hq // Hkv
    sc = float(np.float32(scale))

    def tok(pages, b, t, h, s):
        page, slot = int(table[b][t // ps]), t % ps
        return [float(np.float16(_e4m3_scalar(int(pages[page, slot, h, d])) * s))
                for d in range(D)]

    o = np.zeros((B, Hq, nq, D))
    lse = np.zeros((B, Hq, nq))
    for b in range(B):
        n = int(kv_lens[b])
        for h in range(Hq):
            kh = h // group
            keys = [tok(kp, b, t, kh, float(np.float32(ks))) for t in range(n)]
            vals = [tok(vp, b, t, kh, float(np.float32(vs))) for t in range(n)]
            for i in range(nq):
                ws = [math.exp(sc * sum(float(q[b, h, i, d]) * keys[t][d] for d in range(D)))
                      for t in range(n - nq + i + 1)]
                tot = sum(ws)
                for d in range(D):
                    o[b, h, i, d] = sum(w * vals[t][d] for t, w in enumerate(ws)) / tot
                lse[b, h, i] = math.log(tot)
    return o, lse


def _pin_brute(fn):
    q, kp, vp, table, lens = _case(2, 4, 2, 2, 4, 4, (7, 10), 40)
    o, lse = fn(q, kp, vp, table, lens, 0.5, 0.25, 0.45)
    ob, lb = _brute(q, kp, vp, table, lens, 0.5, 0.25, 0.45)
    return np.allclose(o, ob, rtol=1e-12, atol=1e-13) and np.allclose(lse, lb, rtol=1e-12,
                                                                      atol=1e-13)


def _pin_single_token(fn):
    q, kp, vp, table, lens = _case(1, 3, 1, 1, 8, 4, (1,), 41)
    o, lse = fn(q, kp, vp, table, lens, 0.5, 0.125, 0.3)
    v0 = np.array([float(np.float16(_e4m3_scalar(int(c)) * 0.125))
                   for c in vp[table[0, 0], 0, 0]])
    return all(np.array_equal(o[0, h, 0], v0) for h in range(3))


def _pin_page_permutation(fn):
    q, kp, vp, table, lens = _case(2, 2, 1, 1, 8, 4, (9, 14), 42)
    o, lse = fn(q, kp, vp, table, lens, 1.0, 0.5, 0.3)
    perm = np.random.default_rng(43).permutation(kp.shape[0])     # new slot of old page p
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    o2, lse2 = fn(q, kp2, vp2, table2, lens, 1.0, 0.5, 0.3)
    return np.array_equal(o, o2) and np.array_equal(lse, lse2)


def _pin_live_length(fn):
    q, kp, vp, table, lens = _case(1, 2, 1, 2, 8, 4, (10,), 44, spare=3)
    o, lse = fn(q, kp, vp, table, lens, 1.0, 0.5, 0.3)
    kp2, vp2 = kp.copy(), vp.copy()
    last = table[0, (10 - 1) // 4]
    kp2[last, 10 % 4:] ^= 0x55                              # slots 10, 11 of the last page
    vp2[last, 10 % 4:] ^= 0x2A
    unused = np.setdiff1d(np.arange(kp.shape[0]), table[0][table[0] >= 0])
    kp2[unused] = 0x7E
    vp2[unused] = 0xFE
    o2, lse2 = fn(q, kp2, vp2, table, lens, 1.0, 0.5, 0.3)
    return np.array_equal(o, o2) and np.array_equal(lse, lse2)


def _pin_prefill_tail(fn):
    q, kp, vp, _, _ = _case(1, 6, 1, 3, 8, 4, (16,), 45, spare=0)
    table = np.arange(4, dtype=np.int32)[None]
    o, lse = fn(q, kp, vp, table, np.array([16]), 0.5, 0.25, 0.4)
    kb, vb = E.paged_e4m3_to_fp16(kp, vp, table[0], 16, 0.5, 0.25)
    k = fp16_bits_to_f64(kb).astype(np.float16)[None]      # FP16 values, exactly
    v = fp16_bits_to_f64(vb).astype(np.float16)[None]
    op, lp = A.causal_prefill_attention(q, k, v, 0.4, 3)
    return np.allclose(o, op, rtol=1e-12, atol=1e-13) and np.allclose(lse, lp, rtol=1e-12,
                                                                      atol=1e-13)


PINS = [_pin_brute, _pin_single_token, _pin_page_permutation, _pin_live_length, _pin_prefill_tail]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin_holds_for_oracle(pin):
    assert pin(DEC.paged_decode_attention)


def _mutant(pos_shift=0, head_rule=None, use_table=True, v_scale_on=True):
    def fn(q, kp, vp, table, kv_lens, ks, vs, scale):
        B, Hq, nq, D = q.shape
        Hkv = kp.shape[2]
        o = np.zeros((B, Hq, nq, D))
        lse = np.zeros((B, Hq, nq))
        for b in range(B):
            n = int(kv_lens[b])
            row = table[b] if use_table else np.arange(table.shape[1], dtype=np.int32)
            kb, vb = E.paged_e4m3_to_fp16(kp, vp, row, n, ks, vs if v_scale_on else 1.0)
            k, v = fp16_bits_to_f64(kb), fp16_bits_to_f64(vb)
            vis = np.arange(n)[None, :] <= (n - nq + pos_shift + np.arange(nq))[:, None]
            for h in range(Hq):
                kh = head_rule(h, Hq, Hkv) if head_rule else h // (Hq // Hkv)
                o[b, h], lse[b, h] = A.attention_rows(q[b, h], k[kh], v[kh], scale, vis)
        return o, lse
    return fn


@pytest.mark.parametrize("name,mutant", [
    ("query position one early", _mutant(pos_shift=-1)),
    ("head map h % Hkv", _mutant(head_rule=lambda h, Hq, Hkv: h % Hkv)),
    ("page table ignored", _mutant(use_table=False)),
    ("V scale dropped", _mutant(v_scale_on=False)),
])
def test_planted_mistakes_are_caught(name, mutant):
    assert not all(pin(mutant) for pin in PINS), name
