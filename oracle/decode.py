"""Attention of new query tokens over a paged E4M3 KV cache, float64.

Test infrastructure only (see ``oracle/__init__.py``).

The pages keep FP8 E4M3 KV caches in fixed-size pages for serving ("Integrate
FP32 v37 prefill and exact E4M3 bridge", Purpose and Implementation: the
exact E4M3 paged -> FP16 bridge; Validation: the E4M3 decode wave kernels and
the 256000-input decode).  A decode step attends the newest query tokens of
each sequence to everything cached so far.  The plainest reading, used here:

* the K and V values attention sees are exactly the bridge's FP16 values,
  RNE_fp16(decode(byte) * scale), gathered through the page table
  (``e4m3.paged_e4m3_to_fp16``);
* sequence b holds kv_len[b] tokens, the last nq of which are the new tokens,
  so query i (0 <= i < nq) sits at position kv_len[b] - nq + i and sees keys
  t <= that position (causal among the new tokens; nq = 1 is plain decode);
* query head h reads KV head h // (Hq / Hkv) (shared-KV heads);
* o and lse follow ``attention.attention_rows``: softmax(scale * q.k) v with
  the FP32 scale the caller passes, natural-log lse.
"""

import numpy as np

from .attention import attention_rows
from .e4m3 import paged_e4m3_to_fp16
from .fp16 import fp16_bits_to_f64


def paged_decode_attention(q, k_pages, v_pages, page_table, kv_lens, k_scale, v_scale, scale):
    """Decode attention over paged E4M3 caches.

    q          : FP16 [B][Hq][nq][D]
    k_pages    : uint8 [num_phys_pages][page_size][Hkv][D]  (v_pages alike)
    page_table : int [B][max_pages]; row b maps logical page p of sequence b
                 to a physical page (entries past ceil(kv_len/page_size) unused)
    kv_lens    : int [B], nq <= kv_lens[b] <= max_pages * page_size
    returns    : (o [B][Hq][nq][D], lse [B][Hq][nq]) float64
    """
    q = np.asarray(q)
    B, Hq, nq, D = q.shape
    Hkv = np.asarray(k_pages).shape[2]
    group = Hq // Hkv
    table = np.asarray(page_table)
    o = np.zeros((B, Hq, nq, D))
    lse = np.zeros((B, Hq, nq))
    for b in range(B):
        n = int(kv_lens[b])
        kb, vb = paged_e4m3_to_fp16(k_pages, v_pages, table[b], n, k_scale, v_scale)
        k = fp16_bits_to_f64(kb)                   # [Hkv][n][D]
        v = fp16_bits_to_f64(vb)
        pos = n - nq + np.arange(nq)               # absolute positions of the queries
        visible = np.arange(n)[None, :] <= pos[:, None]
        for h in range(Hq):
            o[b, h], lse[b, h] = attention_rows(q[b, h], k[h // group], v[h // group], scale,
                                                visible)
    return o, lse
