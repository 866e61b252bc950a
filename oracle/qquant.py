"""Dynamic per-(sequence, KV head) e4m3 quantization of Q (oracle side).

Test infrastructure only (see :mod:`oracle`).

Source: ``T5DecodeRunner.run`` on the ``mjolnir/runner.py`` page, the fp8-Q
branch of its "Q" block (the PyTorch path that the fused Triton pack
replaces), with ``FP8_MAX = 448`` from the top of that page. For request
``b`` and KV head ``g`` (``h_r = H_q / H_k`` query heads per KV head):

1. ``x[t, r, c] = float32(Q[b*ql + t, g*h_r + r, c])``, multiplied in float32
   by ``q_mul[g*h_r + r, c]`` when ``q_mul`` is given (fp6 KV: the K channel
   scales, ``k_mul`` of ``_install_fp6_scales`` on the ``mjolnir/backend.py``
   page);
2. ``amax = max |x|`` over ``t < ql, r < h_r, c < D``, clamped below at the
   float32 value of ``1e-6``;
3. ``scale = amax / 448`` (float32 division);
4. ``code[b, g, t*h_r + r, c] = e4m3(x / scale)`` with a float32 IEEE
   division and round-to-nearest-even (torch's ``.to(float8_e4m3fn)``);
5. ``q_descale[b, g] = scale``.

The packed row order ``t*h_r + r`` is the ``permute(0, 2, 1, 3, 4)`` of the
``(b, ql, h_k, h_r, d)`` view in the same block.

Pins (``tests/test_oracle_qquant.py``): the amax element maps to code
+-448; a constant Q gives 0x7E everywhere; every code is the nearest e4m3
value to ``x/scale`` (checked against the decode table, independent of the
encoder); the scale is the float32 quotient ``amax/448``; GQA row order.
"""

from __future__ import annotations

import numpy as np

from .formats import e4m3_encode

FP8_MAX = np.float32(448.0)
AMAX_FLOOR = np.float32(1e-6)


def quantize_q(q_f32, num_seqs: int, q_len: int, h_q: int, h_k: int, d: int, q_mul=None):
    """Quantize Q.

    ``q_f32``: float32 array ``[num_seqs*q_len, h_q, d]`` holding the bf16
    query values exactly. ``q_mul``: optional float32 ``[h_q, d]``.
    Returns ``(codes uint8 [B, h_k, q_len*h_r, d], descale float32 [B, h_k])``.
    """
    q = np.asarray(q_f32, dtype=np.float32)[: num_seqs * q_len]
    assert q.shape == (num_seqs * q_len, h_q, d)
    h_r = h_q // h_k
    x = q.copy()
    if q_mul is not None:
        x = (x * np.asarray(q_mul, dtype=np.float32).reshape(1, h_q, d)).astype(np.float32)
    x = x.reshape(num_seqs, q_len, h_k, h_r, d)
    amax = np.abs(x).max(axis=(1, 3, 4)).astype(np.float32)  # [B, h_k]
    amax = np.maximum(amax, AMAX_FLOOR)
    scale = (amax / FP8_MAX).astype(np.float32)
    y = (x / scale[:, None, :, None, None]).astype(np.float32)
    codes = e4m3_encode(y)  # [B, ql, h_k, h_r, d]
    codes = codes.transpose(0, 2, 1, 3, 4).reshape(num_seqs, h_k, q_len * h_r, d)
    return np.ascontiguousarray(codes), scale


def pack_q_rows(q_f32, num_seqs: int, q_len: int, h_q: int, h_k: int, d: int) -> np.ndarray:
    """The bf16-Q mode (``q_mode="bf16"`` of ``T5DecodeRunner``: Q unquantized):
    the query values themselves, in the same packed row order as the codes
    (``[B, h_k, q_len*h_r, d]``, row ``t*h_r + r``), as float64."""
    q = np.asarray(q_f32, dtype=np.float64)[: num_seqs * q_len]
    assert q.shape == (num_seqs * q_len, h_q, d)
    h_r = h_q // h_k
    x = q.reshape(num_seqs, q_len, h_k, h_r, d).transpose(0, 2, 1, 3, 4)
    return np.ascontiguousarray(x.reshape(num_seqs, h_k, q_len * h_r, d))

