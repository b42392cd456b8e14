"""CPU oracle for the fused FP16 attention path — TEST INFRASTRUCTURE ONLY.

This package is the slow, plain, obviously-correct statement of what the GPU
library computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product path (the ``attention_fp16_flashattention_gb300`` package and its CUDA
library) never imports, links or calls anything here, and this package imports
nothing from the product path: the two share no code.

Arithmetic is float64 unless the pages fix another precision:

* ``fp16``      – IEEE binary16 decode / round-to-nearest-even encode.
* ``e4m3``      – FP8 E4M3 ("fn" variant) decode and the paged E4M3 -> FP16
                  bridge with a single rounding of the scaled value.
* ``attention`` – softmax(scale * Q K^T + mask) V for the dense, causal
                  (shared-KV heads, prefix offset) and block-sparse variants.
* ``decode``    – new query tokens attending to a paged E4M3 KV cache through
                  the bridge's FP16 values (causal among the new tokens).
* ``vsa``       – cube mean-pooling (FP32, as the pages fix), cube scores and
                  the top-k key-cube selection.

Every function cites the page and section it follows (the pages are the five
web pages on this subject: "Share SM70 projection, attention and row reduction
paths", "Generalize H3 SM70 execution and weight residency", "Integrate H3 SM70
execution, metrics and VSA diagnostics", "Integrate FP32 v37 prefill and exact
E4M3 bridge" and the FastVideo compare view "fasth3-spark-exact-perf").  Each
function is pinned by CPU tests in ``tests/test_oracle_*.py`` against closed
forms, invariants, library routines and brute force; no function here is
"parity unpinned".
"""

from . import fp16, e4m3, attention, decode, vsa  # noqa: F401
