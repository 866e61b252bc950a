"""CPU oracle for paged fp8/fp6 decode attention — TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the
decode path computes. It exists to check the CUDA library, nothing else:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it. The product path
(``paged_fp8_decode_gb300``) never imports, calls or links it, and the
oracle imports nothing from the product path.

Sources (the mjolnir-kernel 0.1.0 pages):

* ``mjolnir/runner.py`` — ``tile_width``, ``T5DecodeRunner.slots`` /
  ``.plan`` (split plan, reduction rule), ``T5DecodeRunner.run`` (dynamic
  per-(sequence, KV head) e4m3 Q quantization, Q/O packing, ``q_mul`` /
  ``o_mul``), ``VariantKey`` comment on the packed fp6 format.
* ``mjolnir/backend.py`` — ``_install_fp6_scales`` (channel scales folded
  into Q and into the output), ``_t5_q_len`` (trailing zero-token padding
  requests), ``_seq_lens_cpu`` (planning on an upper bound; masking uses the
  true lengths in device memory).
* The package README ("A decode step", "fp6 (e2m3) KV in vLLM", "What it
  does") — causal vs. non-causal query blocks, the four steps of a decode
  step, split-KV partials merged by LSE.

Modules:

* :mod:`oracle.formats` — OCP e4m3 / e2m3 / e3m2 / e2m1 codecs, the fp6
  4-in-3 packing and the fp4 2-per-byte packing.
* :mod:`oracle.kvwrite` — the KV-cache write at ``slot_mapping`` (e4m3 with
  per-tensor / per-head scales, packed e2m3 / e3m2 / e2m1 with per-channel
  scales).
* :mod:`oracle.qquant`  — the Q quantization recipe (bit-exact target).
* :mod:`oracle.plan`    — ``tile_width``, ``slots`` and the split-KV plan
  (bit-exact target).
* :mod:`oracle.attention` — exact fp64 paged decode attention, split
  partials and the LSE merge.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values and properties fixed by the format definitions, the pages
and the mathematics (see each module's header). No function is unpinned.
"""

from . import attention, formats, plan, qquant  # noqa: F401
