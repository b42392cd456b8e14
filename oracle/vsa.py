"""VSA key-cube selection and the coarse (compression) branch.

Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix ("Integrate H3 SM70 execution, metrics and VSA
diagnostics", Purpose: top-k = 64, learned compression; FastVideo compare
view, minimax_h3_fusions/query_pool.py (``prepare_pooled_queries``),
minimax_h3_fusions/key_quant.py (``pool_quantize_smoothed_keys``) and
minimax_h3_fusions/kv_pool.py (``pool_quantize_prefix_kv``, which pools the
values of every tile as well)):

* tokens are grouped in cubes (tiles) of 64 consecutive tokens in tile order;
* a cube's pooled vector is the FP32 mean of its token vectors: an FP32 sum
  divided by the valid-token count with a correctly rounded division
  (``div_rn(total, count)``); queries, keys and values are pooled alike;
* each query cube keeps the ``topk`` key cubes whose pooled scores
  (pooled q . pooled k) are largest.

Readings where the pages are silent (each listed in the design notes):

* Summation order of the FP32 cube sum: sequential over the cube's tokens in
  token order, each addition rounded to FP32.
* Score: the EXACT dot product of the two FP32 pooled vectors (no rounding at
  all).  The pages fix the means' precision but not the score's, and the
  plainest quantity is the true dot product of those means.  Every product of
  two FP32 numbers is exact in FP64, and for pooled FP16 data every mean is an
  integer multiple of 2^-53 below 2^16 in magnitude (see ``grid_limbs``), so
  the score times 2^106 is an integer; it is computed exactly with integer
  limbs.
* Ties: the lower key-cube index wins; the selected set is reported in
  ascending key-cube order.
* Boundary cubes ("boundary handling"; the tile valid counts of the pages'
  pooling and block-list code): a cube holds ``valid[c]`` real tokens in its
  first slots and padding after them; pooling sums and divides by the real
  tokens only.  Prefix tokens (text/audio before the video tokens) are not
  in cubes and take no part in the selection.
* Coarse branch ("learned compression"; the pages pool V per tile but do not
  print the attention that consumes it): every query cube's pooled query
  attends, with the same softmax scale, over the pooled keys and pooled values
  of ALL key cubes of its head; the result is broadcast to the cube's real
  tokens and added to the fine (selected-cube) output through a gate the
  caller supplies (the learned part: o = o_fine + g * o_coarse, elementwise).
  Prefix tokens keep their dense output; padding query slots stay zero.
"""

import numpy as np


def pool_means_fp32(x, block, count=None):
    """FP32 cube means.  x: [..., S, D] FP16 (cube-major) -> [..., S/block, D] FP32.

    count: None (every cube full), or per-cube valid-token counts [S/block]
    (boundary cubes of a grid that the cube size does not divide: the valid
    tokens are the first ``count[c]`` slots of cube c, the rest is padding whose
    contents are ignored).  sum_t over the valid tokens is accumulated in token
    order with an FP32 rounding after every addition, then divided by the
    count with an FP32 correctly rounded division.
    """
    x = np.asarray(x)
    *lead, S, D = x.shape
    nc = S // block
    cnt = np.full(nc, block, dtype=np.int64) if count is None else np.asarray(count, np.int64)
    xs = x.reshape(*lead, nc, block, D).astype(np.float32)
    acc = np.zeros((*lead, nc, D), dtype=np.float32)
    for t in range(block):
        live = (t < cnt)[:, None]
        acc = np.where(live, np.add(acc, xs[..., t, :], dtype=np.float32), acc)
    return np.divide(acc, cnt.astype(np.float32)[:, None], dtype=np.float32)


# ------------------------------------------------------------------ exact scores
#
# Why every pooled mean sits on the grid 2^-53 * Z with |x| < 2^16: an FP16
# value is an integer multiple of 2^-24 below 2^16; an FP32 sum of such values
# rounds to a multiple of its own ulp, which is never finer than 2^-24 while
# the sum is a multiple of 2^-24, so the sum stays a multiple of 2^-24 (below
# 64 * 2^16).  A nonzero sum divided by a count <= 64 is at least 2^-30 in
# magnitude, a normal FP32 number whose 24-bit significand puts its last bit
# at 2^-53 or above.  So x * 2^53 is an integer M with |M| < 2^69: three
# limbs of 23 bits.

LIMB = 23
_MASK = (1 << LIMB) - 1
GRID_EXP = 53            # pooled means are integers times 2^-GRID_EXP
MAX_BITS = 69            # |x * 2^53| < 2^69


def grid_limbs(x):
    """FP32 array -> int64 limbs (a0, a1, a2) with x * 2^53 = a0 + a1 2^23 + a2 2^46.

    The limbs carry the sign of x (each |a_i| < 2^23).  Raises if a value is
    not finite, not an integer multiple of 2^-53, or not below 2^16 in
    magnitude, which pooled FP16 data never produces.

    Every step is exact in float64: x * 2^53 keeps x's 24 significant bits;
    floor and the subtraction of the floored high part only clear bits of a
    value that float64 holds, so each result is representable.
    """
    x = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("pooled means must be finite")
    M = x.astype(np.float64) * 2.0 ** GRID_EXP
    if not np.all(M == np.floor(M)):
        raise ValueError("a pooled mean is not a multiple of 2^-53")
    A = np.abs(M)
    if not np.all(A < 2.0 ** MAX_BITS):
        raise ValueError("a pooled mean is not below 2^16 in magnitude")
    a2 = np.floor(A / 2.0 ** (2 * LIMB))
    r = A - a2 * 2.0 ** (2 * LIMB)
    a1 = np.floor(r / 2.0 ** LIMB)
    a0 = r - a1 * 2.0 ** LIMB
    sgn = np.sign(M)
    return tuple((sgn * a).astype(np.int64) for a in (a0, a1, a2))


def exact_scores(qm, km):
    """Exact pooled scores.  qm: [..., Nq, D], km: [..., Nk, D] FP32.

    Returns (top, d3, d2, d1, d0), int64 arrays [..., Nq, Nk] with
        sum_d qm[d] km[d] * 2^106 = top 2^92 + d3 2^69 + d2 2^46 + d1 2^23 + d0,
    0 <= d_i < 2^23 and top signed: comparing these tuples lexicographically
    compares the exact scores.

    The nine limb products go through float64 matrix products: each limb is
    below 2^23 in magnitude, so a product is below 2^46 and a sum of D <= 128
    of them below 2^53, an integer that float64 holds exactly in any summation
    order.
    """
    qa = grid_limbs(qm)
    ka = grid_limbs(km)
    if np.asarray(qm).shape[-1] > 128:
        raise ValueError("head width above 128")
    c = [0] * 5                                 # limb position i + j
    for i in range(3):
        for j in range(3):
            p = np.matmul(qa[i].astype(np.float64), np.swapaxes(ka[j].astype(np.float64), -1, -2))
            c[i + j] = c[i + j] + p.astype(np.int64)
    digits = []
    carry = 0
    for pos in range(4):
        t = c[pos] + carry
        digits.append(t & _MASK)
        carry = t >> LIMB                       # floor division (arithmetic shift)
    top = c[4] + carry
    return top, digits[3], digits[2], digits[1], digits[0]


def exact_scores_float(qm, km):
    """The exact scores rounded to float64 (for display and coarse softmax checks)."""
    top, d3, d2, d1, d0 = exact_scores(qm, km)
    s = top.astype(np.float64) * 2.0 ** 92
    for d, p in ((d3, 69), (d2, 46), (d1, 23), (d0, 0)):
        s = s + d.astype(np.float64) * 2.0 ** p
    return s * 2.0 ** -106


def topk_exact(qm, km, topk):
    """The ``topk`` key cubes with the largest exact scores, ties to the lower
    index, in ascending order.  int32 [..., Nq, topk]."""
    top, d3, d2, d1, d0 = exact_scores(qm, km)
    idx = np.broadcast_to(np.arange(top.shape[-1], dtype=np.int64), top.shape)
    order = np.lexsort((idx, -d0, -d1, -d2, -d3, -top), axis=-1)
    return np.sort(order[..., :topk], axis=-1).astype(np.int32)


def topk_blocks(scores, topk):
    """The ``topk`` largest values per row of a plain score array, ties to the
    lower index, ascending.  scores: [..., Nq, Nk] -> int32 [..., Nq, topk]."""
    s = np.asarray(scores)
    order = np.argsort(-s, axis=-1, kind="stable")
    return np.sort(order[..., :topk], axis=-1).astype(np.int32)


def vsa_select(q, k, block, topk, valid=None, prefix=0):
    """Selection for every query cube.  q, k: [B][H][S][D] FP16; tokens
    [prefix, S) are the cube-major video tokens (S - prefix a multiple of
    block), valid the per-cube valid-token counts (None: full cubes).

    Returns idx int32 [B][H][(S - prefix)/block][topk].
    """
    qm = pool_means_fp32(np.asarray(q)[..., prefix:, :], block, valid)
    km = pool_means_fp32(np.asarray(k)[..., prefix:, :], block, valid)
    return topk_exact(qm, km, topk)


# ------------------------------------------------------------------ coarse branch
def coarse_attention(q, k, v, block, scale, valid=None, prefix=0):
    """Cube-level attention of the coarse branch, float64 from the FP32 means.

    q, k, v: [B][H][S][D] FP16.  For query cube i of a head:
        o_c[i] = sum_j softmax_j(scale * qm_i . km_j) vm_j
    over all key cubes j, with qm, km, vm the pages' FP32 cube means.
    Returns float64 [B][H][(S - prefix)/block][D].
    """
    qm = pool_means_fp32(np.asarray(q)[..., prefix:, :], block, valid).astype(np.float64)
    km = pool_means_fp32(np.asarray(k)[..., prefix:, :], block, valid).astype(np.float64)
    vm = pool_means_fp32(np.asarray(v)[..., prefix:, :], block, valid).astype(np.float64)
    s = float(np.float32(scale)) * np.matmul(qm, np.swapaxes(km, -1, -2))
    s = s - s.max(axis=-1, keepdims=True)
    w = np.exp(s)
    return np.matmul(w, vm) / w.sum(axis=-1, keepdims=True)


def gated_output(o_fine, o_coarse, gate, block, valid=None, prefix=0):
    """o = o_fine + gate * o_coarse[cube of the token] for real video tokens.

    o_fine: [B][H][S][D] (float), o_coarse: [B][H][NC][D], gate: [B][H][S][D].
    Prefix tokens keep o_fine; padding slots of boundary cubes stay as o_fine
    gives them (zero).  Returns float64 [B][H][S][D].
    """
    o = np.array(o_fine, dtype=np.float64, copy=True)
    S = o.shape[2]
    nc = (S - prefix) // block
    cnt = np.full(nc, block) if valid is None else np.asarray(valid)
    g = np.asarray(gate, dtype=np.float64)
    oc = np.asarray(o_coarse, dtype=np.float64)
    for c in range(nc):
        r0 = prefix + c * block
        r1 = r0 + int(cnt[c])
        o[:, :, r0:r1] += g[:, :, r0:r1] * oc[:, :, c:c + 1]
    return o
