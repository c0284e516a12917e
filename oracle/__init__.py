"""CPU oracle for compressed-KV-cache quantisation and decode attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call, link
or execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It is a plain, slow, fp64 restatement of what the pages define, written
without any blocking, fusion or reordering, so that it can be read against
the pages line by line. It shares no code with the CUDA library under
``quantised_kv_cache_gb300/``: the two sides only agree on the storage
format written out in ``include/tq.h`` and on the seeded counter generator
named there, and each implements both from their published definitions.

Sources (cited by title and section throughout):

* [TQ-stats] "Statistical Inference and Quality Measures of KV Cache
  Quantisations Inspired by TurboQuant" (D'Alberto), gist.science explainer,
  technical summary: "Theoretical framework", "Quantisation schemes",
  "Evaluation metrics", "Main contributions 1-4", "Results".
* [HeadQ] "HeadQ: Model-Visible Distortion and Score-Space Correction for
  KV-Cache Quantization", technical summary sections 2.1-3.
* [KIVI-geometry] "Your KV cache is not a bit problem but a geometry problem"
  (Goel): "What quantisation error is made of", "Keys", "Values",
  "The systems tax".
* [KVQuant++] "KVQuant++: attention-aware KV cache quantisation" forum post:
  "Codebook design", "Fast codebook lookup", "Rate-distortion performance",
  "Rotation-invariance guarantee", "Core innovation 5".

Functions whose parity has no independent pin say "parity unpinned" in their
docstring; at present that is only the 6D error frame in ``metrics.py``.
"""

from . import rng, codebook, rotation, turboquant, attention, kivi, metrics  # noqa: F401
