"""VSA key-cube selection: cube mean pooling, cube scores, top-k.

Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix ("Integrate H3 SM70 execution, metrics and VSA
diagnostics", Purpose: top-k = 64; FastVideo compare view,
minimax_h3_fusions/query_pool.py (``prepare_pooled_queries``) and
minimax_h3_fusions/key_quant.py (``pool_quantize_smoothed_keys``)):

* tokens are grouped in cubes (tiles) of 64 consecutive tokens in tile order;
* a cube's pooled vector is the FP32 mean of its token vectors: an FP32 sum
  divided by the valid-token count with a correctly rounded division
  (``div_rn(total, count)``);
* each query cube keeps the ``topk`` key cubes whose pooled scores
  (pooled q . pooled k) are largest.

Readings where the pages are silent (each listed in the design notes):

* Summation order of the FP32 cube sum: sequential over the cube's tokens in
  token order, each addition rounded to FP32.
* Score precision and order: FP32, sequential over the head dimension d =
  0..D-1, each product rounded to FP32 and then added with an FP32 rounding
  (no fused multiply-add), starting from +0.  Selecting indices is an integer
  decision taken from floating point, so both sides must take it in the same
  precision and order; this is that order.
* Ties: the lower key-cube index wins; the selected set is reported in
  ascending key-cube order.
* Boundary cubes ("boundary handling"; the tile valid counts of the pages'
  pooling and block-list code): a cube holds ``valid[c]`` real tokens in its
  first slots and padding after them; pooling sums and divides by the real
  tokens only.  Prefix tokens (text/audio before the video tokens) are not
  in cubes and take no part in the selection.
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


def cube_scores_fp32(qm, km):
    """FP32 scores.  qm: [..., Nq, D], km: [..., Nk, D] FP32 -> [..., Nq, Nk] FP32.

    score = (((0 + q_0 k_0) + q_1 k_1) + ...) with every product and every
    sum rounded to FP32 (no fused multiply-add).
    """
    qm = np.asarray(qm, dtype=np.float32)
    km = np.asarray(km, dtype=np.float32)
    D = qm.shape[-1]
    acc = np.zeros(qm.shape[:-1] + (km.shape[-2],), dtype=np.float32)
    for d in range(D):
        prod = np.multiply(qm[..., :, None, d], km[..., None, :, d], dtype=np.float32)
        acc = np.add(acc, prod, dtype=np.float32)
    return acc


def topk_blocks(scores, topk):
    """The ``topk`` largest scores per row, ties to the lower index, ascending.

    scores: [..., Nq, Nk] -> int32 [..., Nq, topk].  A stable sort by
    decreasing score keeps equal scores in increasing index order, so the
    first ``topk`` entries are the selection; they are then sorted by index.
    """
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
    return topk_blocks(cube_scores_fp32(qm, km), topk)
