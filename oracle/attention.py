"""Fused attention O = softmax(scale * Q K^T + mask) V, float64 reference.

Test infrastructure only (see ``oracle/__init__.py``).

What is computed, per query row i (a row of Q), over its visible keys j:

    s_ij = scale * (q_i . k_j)
    w_ij = exp(s_ij - m_i) / sum_j' exp(s_ij' - m_i),   m_i = max_j s_ij
    o_i  = sum_j w_ij v_j
    lse_i = m_i + log(sum_j exp(s_ij - m_i))            (natural log-sum-exp)

The scale is the FP32 number the caller passes (the pages compute
1/sqrt(128) in double and store it in a float: FastVideo compare view,
minimax_h3_prefix.cu, ``prefix_forward``); the oracle uses that FP32 value
exactly.  Inputs are FP16 and are decoded exactly; everything after is
float64.  The GPU keeps FP32 accumulators and rounds P and O to FP16 ("FP32
QK/PV accumulation ... probabilities and final output retain FP16 storage":
"Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation); the
oracle does neither rounding, and the parity tolerance absorbs both.

Variants ("Integrate FP32 v37 prefill and exact E4M3 bridge", Implementation;
"Integrate H3 SM70 execution, metrics and VSA diagnostics", Purpose):

* dense      – every key visible (the D128 video-DiT heads); optionally an
               additive mask term (the "+ mask" of the formula).
* causal     – query head h reads KV head h // (Hq / Hkv) (shared-KV heads);
               query i of Q_real real queries sits at absolute position
               (KV - Q_real) + i and sees keys j <= that position.  Padded
               query rows (i >= Q_real) are defined as zero output with
               lse = -inf (the pages keep real-query causal offsets when
               queries are padded and say nothing about padded rows' values).
* block-sparse (VSA) – tokens are grouped in cubes of ``block`` consecutive
               tokens (cube-major order); query token i in cube c sees
               exactly the tokens of the key cubes listed in idx[c].

Rows can be evaluated for a sample of (batch*head, row) pairs, which is how
the large workloads are checked.
"""

import numpy as np


def _f64(x):
    return np.asarray(x).astype(np.float64)


def attention_rows(q, k, v, scale, visible=None, mask=None):
    """Softmax attention for a block of query rows against one key/value set.

    q: [n, D]; k, v: [m, D]; visible: optional bool [n, m]; mask: optional
    additive term [n, m] (the "+ mask" of the formula; -inf hides a key).
    Returns (o [n, D] float64, lse [n] float64).  A row with no visible key
    gets o = 0 and lse = -inf.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    sc = float(np.float32(scale))
    s = sc * (q @ k.T)
    if mask is not None:
        s = s + _f64(mask)
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(s - m_safe)
    l = w.sum(axis=1, keepdims=True)
    l_safe = np.where(l > 0, l, 1.0)
    o = (w @ v) / l_safe
    lse = m_safe[:, 0] + np.log(l_safe[:, 0])
    o[empty] = 0.0
    lse[empty] = -np.inf
    return o, lse


def _rows_by_head(rows, n_heads, n_rows):
    """Group (head, row) pairs by head; None means every row of every head."""
    if rows is None:
        return [(h, np.arange(n_rows)) for h in range(n_heads)]
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    return [(int(h), rows[rows[:, 0] == h, 1]) for h in np.unique(rows[:, 0])]


def _scatter(rows, groups, results, n_heads, n_rows, D):
    """Put per-head results back in the order the caller asked for."""
    if rows is None:
        o = np.zeros((n_heads, n_rows, D))
        lse = np.zeros((n_heads, n_rows))
        for (h, r), (oh, lh) in zip(groups, results):
            o[h, r] = oh
            lse[h, r] = lh
        return o, lse
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    o = np.zeros((len(rows), D))
    lse = np.zeros(len(rows))
    for (h, r), (oh, lh) in zip(groups, results):
        sel = np.nonzero(rows[:, 0] == h)[0]
        o[sel] = oh
        lse[sel] = lh
    return o, lse


def dense_attention(q, k, v, scale, rows=None):
    """Dense non-causal attention.

    q: [B][H][Sq][D]; k, v: [B][H][Skv][D] (FP16 arrays).
    rows: None (all rows; returns o [B][H][Sq][D], lse [B][H][Sq]) or an
    array of (b*H + h, i) pairs (returns o [n][D], lse [n]).
    """
    B, H, Sq, D = q.shape
    qf = q.reshape(B * H, Sq, D)
    kf = k.reshape(B * H, -1, D)
    vf = v.reshape(B * H, -1, D)
    groups = _rows_by_head(rows, B * H, Sq)
    results = [attention_rows(qf[h, r], kf[h], vf[h], scale) for h, r in groups]
    o, lse = _scatter(rows, groups, results, B * H, Sq, D)
    if rows is None:
        return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)
    return o, lse


def dense_masked_attention(q, k, v, mask, scale, rows=None):
    """Dense attention with an additive mask: softmax(scale * q.k + mask) v.

    q: [B][H][Sq][D]; k, v: [B][H][Skv][D] (FP16 arrays); mask: FP16 values
    broadcastable to [B][H][Sq][Skv] (e.g. [Sq][Skv] shared by every head).
    Entries equal to -inf hide a key; a row whose keys are all hidden gives
    o = 0, lse = -inf.  rows: as for ``dense_attention``.
    """
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    mk = np.broadcast_to(np.asarray(mask), (B, H, Sq, Skv)).reshape(B * H, Sq, Skv)
    qf = q.reshape(B * H, Sq, D)
    kf = k.reshape(B * H, -1, D)
    vf = v.reshape(B * H, -1, D)
    groups = _rows_by_head(rows, B * H, Sq)
    results = [attention_rows(qf[h, r], kf[h], vf[h], scale, mask=mk[h, r]) for h, r in groups]
    o, lse = _scatter(rows, groups, results, B * H, Sq, D)
    if rows is None:
        return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)
    return o, lse


def causal_prefill_attention(q, k, v, scale, q_real, rows=None):
    """Causal attention of the last Q_real positions with shared-KV heads.

    q: [B][Hq][Q_pad][D]; k, v: [B][Hkv][KV][D] (FP16 arrays), Hq % Hkv == 0.
    Query i < q_real is at absolute position (KV - q_real) + i and sees keys
    j <= that position; rows i >= q_real give o = 0, lse = -inf.
    rows: as for ``dense_attention`` with b*Hq + h as the head index.
    """
    B, Hq, Qp, D = q.shape
    Hkv, KV = k.shape[1], k.shape[2]
    group = Hq // Hkv
    prefix = KV - q_real
    qf = q.reshape(B * Hq, Qp, D)
    groups = _rows_by_head(rows, B * Hq, Qp)
    results = []
    for bh, r in groups:
        b, h = divmod(bh, Hq)
        kh = h // group
        pos = prefix + r                       # absolute positions of these queries
        visible = np.arange(KV)[None, :] <= pos[:, None]
        visible &= (r < q_real)[:, None]
        results.append(attention_rows(qf[bh, r], k[b, kh], v[b, kh], scale, visible))
    o, lse = _scatter(rows, groups, results, B * Hq, Qp, D)
    if rows is None:
        return o.reshape(B, Hq, Qp, D), lse.reshape(B, Hq, Qp)
    return o, lse


def vsa_sparse_attention(q, k, v, idx, block, scale, rows=None, valid=None, prefix=0):
    """Block-sparse attention over selected key cubes (the full VSA layout).

    q, k, v: [B][H][S][D] FP16.  Tokens [0, prefix) are prefix tokens (text or
    audio, not in cubes); tokens [prefix, S) are the video tokens in
    cube-major order, cube c = slots prefix + c*block .. + block - 1, of which
    the first valid[c] are real and the rest padding (valid None: full cubes).
    idx: int [B][H][(S - prefix)/block][topk], the key cubes each video query
    cube attends.

    * A prefix query (row < prefix) attends densely to every prefix token and
      every real video token ("prefix-dense queries").
    * A real video query in cube c attends exactly the real tokens of the
      cubes idx[b, h, c, :] (a gather of those keys, then ordinary softmax).
    * A padding query slot gives o = 0, lse = -inf.
    """
    B, H, S, D = q.shape
    nc = (S - prefix) // block
    val = np.full(nc, block, dtype=np.int64) if valid is None else np.asarray(valid, np.int64)
    qf = q.reshape(B * H, S, D)
    kf = k.reshape(B * H, S, D)
    vf = v.reshape(B * H, S, D)
    idxf = np.asarray(idx).reshape(B * H, nc, -1)
    real_video = np.concatenate([prefix + c * block + np.arange(val[c]) for c in range(nc)])
    all_keys = np.concatenate([np.arange(prefix), real_video]).astype(np.int64)
    groups = _rows_by_head(rows, B * H, S)
    results = []
    for bh, r in groups:
        o_h = np.zeros((len(r), D))
        l_h = np.full(len(r), -np.inf)
        pre = np.nonzero(r < prefix)[0]
        if pre.size:
            o_h[pre], l_h[pre] = attention_rows(qf[bh, r[pre]], kf[bh, all_keys], vf[bh, all_keys],
                                                scale)
        vid = np.nonzero(r >= prefix)[0]
        cubes = (r[vid] - prefix) // block
        slots = (r[vid] - prefix) % block
        for c in np.unique(cubes):
            sel = vid[(cubes == c) & (slots < val[c])]
            if sel.size == 0:
                continue
            toks = np.concatenate([prefix + kc * block + np.arange(val[kc])
                                   for kc in idxf[bh, c]]).astype(np.int64)
            o_c, l_c = attention_rows(qf[bh, r[sel]], kf[bh, toks], vf[bh, toks], scale)
            o_h[sel] = o_c
            l_h[sel] = l_c
        results.append((o_h, l_h))
    o, lse = _scatter(rows, groups, results, B * H, S, D)
    if rows is None:
        return o.reshape(B, H, S, D), lse.reshape(B, H, S)
    return o, lse
