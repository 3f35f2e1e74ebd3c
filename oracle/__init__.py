"""CPU oracle for the packed index-score + block top-k step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import, call or execute anything
in this package.  The product (the CUDA library and its Python binding) never
routes through it, and this package imports nothing from the product.

What it is: a plain, slow, obviously correct restatement of what the step
computes, in float64 numpy over the dequantised keys, one function per step of
the method, each citing the page passage it follows:

* ``formats``  - E4M3 / E2M1 decoding, round-to-nearest-even encoders, the
  NVFP4 per-16 quantiser (ROCm/ATOM #2745, Summary) and dequantisation.
* ``index``    - per-row causal-masked q.k scores, per-128-token block max
  (or log-sum-exp), forced init/local blocks and block top-k (sglang #45451,
  Modifications; sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring for
  EAGLE verify rows", Modifications 1 and Accuracy Tests), and the per-shard
  selection and merge of indexer context parallelism.

Pins (tests under ``-m "not gpu"``) tie it to facts outside itself: torch's own
float8_e4m3fn conversion, hand-worked NVFP4 groups, exhaustive bf16
representability of every e2m1 x E4M3 product, brute-force subset search for
the selection and pure-Python loops for the block maxima.

Parity status: every function here is pinned except the absolute score values
against the pages' own kernels, which print no scores ("parity unpinned" for
that comparison only).
"""
from . import formats, index  # noqa: F401
