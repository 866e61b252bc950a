"""KV-cache write at ``slot_mapping`` (oracle side).

Test infrastructure only (see :mod:`oracle`).

The step just before the decode path: the new tokens' K and V rows (bf16,
``[T, H_k, D]``) are quantized and scattered into the paged caches.

Sources:

* **e4m3 cache** -- the ``mjolnir/backend.py`` page routes the fp8 write to
  the serving engine's own cache write (``MjolnirImpl._write_kv``: key,
  value, the two caches, ``slot_mapping``, the cache dtype and the layer's
  ``_k_scale`` / ``_v_scale``). The pages do not print that kernel. Reading:
  ``code = e4m3(x / scale)`` with round-to-nearest-even and saturation (the
  conversion the pages use for Q, ``FP8_MAX = 448``), ``scale`` one value
  per tensor or one per KV head (the scale shapes the runner accepts,
  ``k_scale`` in ``T5DecodeRunner.run``).
* **e2m3 cache** -- ``MjolnirImpl.do_kv_cache_update`` calls the package's
  own packed write with the per-(KV head, channel) scales ``k_ch`` /
  ``v_ch`` of ``_install_fp6_scales``, the scales the cache is written
  with. Reading: ``code = e2m3(x / s[h, c])`` (round-to-nearest-even,
  saturating at 7.5), the row's codes packed 4 per 3 bytes
  (:func:`oracle.formats.fp6_pack_rows`).
* **e3m2 / e2m1 caches** -- the README names these formats beside e2m3 and
  gives no write for them. Reading: the e2m3 recipe with the format's own
  encoder (saturating at 28 / 6) and per-(KV head, channel) scales; e3m2 rows
  packed like e2m3 rows, e2m1 rows 2 codes per byte, low nibble first
  (:func:`oracle.formats.fp4_pack_rows`).
* **slots** -- ``slot_mapping[t]`` is the cache slot of token ``t``: page
  ``slot // page_size``, row ``slot % page_size`` (the paged layout of the
  decode path). Reading, as in the serving engine the backend plugs into: a
  negative slot marks a padding token, which writes nothing.

The division ``x / scale`` is IEEE float32 (the inputs are bf16, so their
float32 values are exact); the rounding to the cache format then starts from
that float32 quotient.

Pins (``tests/test_oracle_kvwrite.py``): padding slots write nothing and
untouched bytes stay as they were; rows whose values are representable
scaled codes are written exactly; every written row decodes to within half a
code step of ``x / scale``; writing the tokens in any order gives the same
cache; the packed rows unpack to the codes of the plain encoder.
"""

from __future__ import annotations

import numpy as np

from .formats import e2m1_encode, e2m3_encode, e3m2_encode, e4m3_encode, fp4_pack_rows, fp6_pack_rows

KV_E4M3, KV_E2M3, KV_E3M2, KV_E2M1 = 0, 1, 2, 3


def row_bytes(d: int, kv_format: int) -> int:
    """Bytes of one (token, KV head) row: ``d`` (e4m3), ``3d/4`` (e2m3,
    e3m2) or ``d/2`` (e2m1)."""
    if kv_format == KV_E4M3:
        return d
    return d // 2 if kv_format == KV_E2M1 else d * 3 // 4


def quantize_rows(x, scale, kv_format: int) -> np.ndarray:
    """Rows ``x`` ``[n, H_k, D]`` -> cache rows ``[n, H_k, row_bytes]``.

    ``scale``: e4m3 -- shape ``(1,)`` (per tensor) or ``(H_k,)`` (per head);
    e2m3 / e3m2 / e2m1 -- shape ``(H_k, D)`` (per head and channel).
    """
    x = np.asarray(x, dtype=np.float32)
    s = np.asarray(scale, dtype=np.float32)
    if kv_format == KV_E4M3:
        s = s.reshape(1, -1, 1) if s.size > 1 else s.reshape(1, 1, 1)
        y = (x / s).astype(np.float32)  # IEEE float32 quotient
        return e4m3_encode(y)
    y = (x / s.reshape(1, *s.shape)).astype(np.float32)
    if kv_format == KV_E2M3:
        return fp6_pack_rows(e2m3_encode(y))
    if kv_format == KV_E3M2:
        return fp6_pack_rows(e3m2_encode(y))
    if kv_format == KV_E2M1:
        return fp4_pack_rows(e2m1_encode(y))
    raise ValueError(kv_format)


def write_kv(key, value, k_pool, v_pool, slot_mapping, page_size: int, k_strides, v_strides,
             kv_format: int, k_scale, v_scale) -> None:
    """Scatter the quantized rows of every non-padding token into the pools.

    ``k_pool`` / ``v_pool``: flat ``uint8`` arrays, modified in place.
    ``*_strides``: byte strides ``(page, token, head)``; a row is contiguous.
    """
    key = np.asarray(key, dtype=np.float32)
    value = np.asarray(value, dtype=np.float32)
    n_tok, h_k, d = key.shape
    rb = row_bytes(d, kv_format)
    kq = quantize_rows(key, k_scale, kv_format)
    vq = quantize_rows(value, v_scale, kv_format)
    for t in range(n_tok):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue  # padding token
        page, row = slot // page_size, slot % page_size
        for pool, strides, q in ((k_pool, k_strides, kq), (v_pool, v_strides, vq)):
            for h in range(h_k):
                off = page * strides[0] + row * strides[1] + h * strides[2]
                pool[off:off + rb] = q[t, h]
