"""Exact paged decode attention, split partials and the LSE merge (oracle side).

Test infrastructure only (see :mod:`oracle`).

What a decode step computes (README of the mjolnir-kernel package, "A decode
step", items 2-4, and ``T5DecodeRunner.run`` / ``_launch`` on the
``mjolnir/runner.py`` page), written out as its plain definition in float64:

for every request ``b`` with ``L = seq_lens[b] > 0``, KV head ``g``, packed
query row ``row = t*h_r + r`` (query token ``t < q_len``, query head
``h = g*h_r + r``):

* key ``j < L`` lives in page ``block_table[b][j // page_size]`` at slot
  ``j % page_size``; its K and V rows are dequantized codes times the K / V
  descale of ``(b, g)`` (per tensor, per KV head or per (request, KV head));
* ``s_j = softmax_scale * q_descale[b,g] * sum_c qcode[row,c] * k[j,c]``
  using the QUANTIZED Q codes (the kernel never sees bf16 Q);
* visible keys: causal -> ``j <= L - q_len + t`` (the query block is the last
  ``q_len`` tokens of the sequence); non-causal -> every ``j < L`` (each
  query token attends to all keys: README "What it does", the
  parallel-drafter block);
* ``O[row] = sum_j p_j v_j / sum_j p_j`` with ``p_j = exp(s_j - max s)``;
  then ``O[row, c] *= o_mul[h, c]`` when given (fp6 V channel scales,
  ``_install_fp6_scales`` on the ``mjolnir/backend.py`` page);
* ``lse[row] = max s + ln(sum_j p_j)``.

Readings where the pages are silent (each listed in the design notes):

* P is NOT rounded here: this is exact softmax attention. (The reference
  kernel rounds P to e4m3; the README "Tests" section says so.)
* Requests with ``seq_len == 0`` (trailing zero-token padding, ``_t5_q_len``
  on the backend page) produce no output at all: their rows stay NaN here and
  the GPU must leave them untouched.
* A causal row that sees no key (only possible when ``L < q_len``) yields
  zeros and ``lse = -inf``.
* ``softmax_scale`` is an input (the backend passes the layer's scale);
  the workloads use ``1/sqrt(D)``.

Split-KV (README item 4: a second kernel merges the split partials by their LSE): a chunk
``[a, e)`` of the keys yields ``m`` (max logit), ``l`` (sum of
``exp(s - m)``) and the normalised partial ``O~ = sum p v / l``; chunks merge
as ``O = sum_s w_s O~_s / sum_s w_s``, ``w_s = exp(m_s - M) * l_s``,
``M = max_s m_s``, empty chunks (``m = -inf``, ``l = 0``) weigh zero.

Pins (``tests/test_oracle_attention.py``): brute-force triple loop on tiny
inputs; paged == contiguous; page-permutation and HND/NHD-view invariance;
constant V returns V; a single key returns its V row; one query row reduces
to ``scipy.special.softmax(s) @ V``; the last causal row equals the
non-causal row; causal row ``t`` equals the non-causal result over the
prefix ``L - q_len + t + 1``; GQA heads with equal Q give equal O;
split + merge == unsplit for random partitions including empty chunks.
"""

from __future__ import annotations

import math

import numpy as np

from .formats import e2m1_decode, e2m3_decode, e3m2_decode, e4m3_decode, fp4_unpack_rows, fp6_unpack_rows

# packed (narrow) KV formats: codes per row are unpacked before decoding
_UNPACK = {"e2m3": fp6_unpack_rows, "e3m2": fp6_unpack_rows, "e2m1": fp4_unpack_rows}


def decode_codes(codes, kv_format: str) -> np.ndarray:
    if kv_format == "fp8":
        return e4m3_decode(codes)
    if kv_format == "e2m3":
        return e2m3_decode(codes)
    if kv_format == "e3m2":
        return e3m2_decode(codes)
    if kv_format == "e2m1":
        return e2m1_decode(codes)
    raise ValueError(kv_format)


def descale_at(ds, b: int, g: int) -> float:
    """K/V descale of (request b, KV head g): 1 element = per tensor,
    ``(h_k,)`` = per KV head, ``(B, h_k)`` = per (request, KV head)."""
    ds = np.asarray(ds, dtype=np.float64)
    if ds.size == 1:
        return float(ds.reshape(-1)[0])
    if ds.ndim == 1:
        return float(ds[g])
    return float(ds[b, g])


def to_bf16(x) -> np.ndarray:
    """Round float64 values to bfloat16 (8 significant bits), nearest-even.
    Returns float64 holding the bf16 values. Normal range only (decode
    outputs are far from bf16's subnormals and overflow)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def gather_unit(k_logical, v_logical, block_table, b: int, g: int, L: int, page_size: int,
                kv_format: str = "fp8"):
    """Codes of the first ``L`` keys of request ``b``, KV head ``g``.

    ``*_logical``: ``[num_pages, page_size, h_k, row_bytes]`` byte arrays
    (any strides: a transposed view of an HND or NHD buffer). e4m3 rows are
    one code per byte; packed e2m3 / e3m2 / e2m1 rows are unpacked here."""
    j = np.arange(L)
    pages = np.asarray(block_table)[b, j // page_size]
    slots_ = j % page_size
    kc, vc = k_logical[pages, slots_, g, :], v_logical[pages, slots_, g, :]
    if kv_format in _UNPACK:
        kc, vc = _UNPACK[kv_format](kc), _UNPACK[kv_format](vc)
    return kc, vc


def visible_mask(L: int, q_len: int, h_r: int, causal: bool) -> np.ndarray:
    """[n_q, L] boolean: may query row ``t*h_r + r`` see key ``j``?"""
    n_q = q_len * h_r
    t = np.arange(n_q) // h_r
    j = np.arange(L)
    if not causal:
        return np.ones((n_q, L), dtype=bool)
    return j[None, :] <= (L - q_len + t)[:, None]


def unit_logits(qcodes_bg, qdesc: float, kcodes, kdesc: float, kv_format: str, softmax_scale: float,
                q_values=False):
    """``q_values``: the rows are query values (bf16 mode), not e4m3 codes."""
    q = np.asarray(qcodes_bg, dtype=np.float64) if q_values else e4m3_decode(qcodes_bg) * float(qdesc)  # [n_q, d]
    k = decode_codes(kcodes, kv_format) * float(kdesc)  # [L, d]
    return softmax_scale * (q @ k.T)  # [n_q, L]


def softmax_rows(s, vis):
    """Per row: (m, l, p) with p = exp(s - m) on visible keys, 0 elsewhere."""
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    p = np.where(vis, np.exp(s - safe_m[:, None]), 0.0)
    return m, p.sum(axis=1), p


def decode_attention(q_codes, q_descale, k_logical, v_logical, k_descale, v_descale, block_table,
                     seq_lens, *, num_seqs: int, q_len: int, h_q: int, h_k: int, d: int,
                     page_size: int, kv_format: str, softmax_scale: float, causal: bool,
                     o_mul=None, units=None, q_values=False):
    """Full decode step.

    ``q_values`` (the runner's bf16 Q mode, Q left unquantized): ``q_codes`` holds the
    query values in the packed row order (:func:`oracle.qquant.pack_q_rows`)
    and ``q_descale`` is not used.

    Returns ``(out float64 [B*q_len, h_q, d], lse float64 [B, h_k, n_q])``;
    rows of requests with ``seq_len == 0`` (and of units not in ``units``
    when a subset is asked for) stay NaN.
    """
    h_r = h_q // h_k
    n_q = q_len * h_r
    out = np.full((num_seqs * q_len, h_q, d), np.nan)
    lse = np.full((num_seqs, h_k, n_q), np.nan)
    if units is None:
        units = [(b, g) for b in range(num_seqs) for g in range(h_k)]
    for b, g in units:
        L = int(seq_lens[b])
        if L <= 0:
            continue
        kc, vc = gather_unit(k_logical, v_logical, block_table, b, g, L, page_size, kv_format)
        s = unit_logits(q_codes[b, g], None if q_values else q_descale[b, g], kc, descale_at(k_descale, b, g),
                        kv_format, softmax_scale, q_values=q_values)
        vis = visible_mask(L, q_len, h_r, causal)
        m, l, p = softmax_rows(s, vis)
        v = decode_codes(vc, kv_format) * descale_at(v_descale, b, g)
        with np.errstate(invalid="ignore", divide="ignore"):
            o = np.where(l[:, None] > 0, (p @ v) / np.where(l > 0, l, 1.0)[:, None], 0.0)
            lse[b, g] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
        for row in range(n_q):
            t, r = divmod(row, h_r)
            h = g * h_r + r
            orow = o[row]
            if o_mul is not None:
                orow = orow * np.asarray(o_mul, dtype=np.float64)[h]
            out[b * q_len + t, h] = orow
    return out, lse


# ----------------------------------------------------------------------------
# split-KV partials and the LSE merge
# ----------------------------------------------------------------------------
def chunk_partial(s, vis, v, a: int, e: int):
    """Partial of keys ``[a, e)``: ``(m, l, O~)`` per row; empty -> (-inf, 0, 0)."""
    n_q = s.shape[0]
    if e <= a:
        return np.full(n_q, -np.inf), np.zeros(n_q), np.zeros((n_q, v.shape[1]))
    m, l, p = softmax_rows(s[:, a:e], vis[:, a:e])
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l[:, None] > 0, (p @ v[a:e]) / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return m, l, o


def merge_partials(ms, ls, os_):
    """LSE merge of split partials (lists over splits of per-row arrays)."""
    ms = np.stack(ms)  # [S, n_q]
    ls = np.stack(ls)
    os_ = np.stack(os_)  # [S, n_q, d]
    big_m = ms.max(axis=0)
    safe = np.where(np.isfinite(big_m), big_m, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - safe[None, :]), 0.0) * ls
    tot = w.sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(tot[:, None] > 0,
                     (w[:, :, None] * os_).sum(axis=0) / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
        lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    return o, lse


def effective_kv_bytes(seq_lens, h_k: int, d: int, kv_format: str) -> int:
    """Algorithmic KV bytes of one step: every valid token's K and V row of
    every KV head, read once (``kv_row_bytes`` = d bytes for e4m3, d*6/8 for
    packed e2m3, ``T5DecodeRunner.__init__``; d*6/8 for e3m2 and d/2 for
    e2m1 by the same count of bits)."""
    row = {"fp8": d, "e2m3": d * 6 // 8, "e3m2": d * 6 // 8, "e2m1": d // 2}[kv_format]
    return int(sum(int(x) for x in seq_lens)) * h_k * 2 * row


def brute_force_unit(qcodes_bg, qdesc, k_logical, v_logical, kdesc, vdesc, block_table, b, g, L,
                     page_size, kv_format, softmax_scale, q_len, h_r, causal):
    """Triple loop over rows, keys and channels, scalar math only; for the
    tiny pin cases."""
    from .formats import e2m1_value, e2m3_value, e3m2_value, e4m3_value

    dec = {"fp8": e4m3_value, "e2m3": e2m3_value, "e3m2": e3m2_value, "e2m1": e2m1_value}[kv_format]
    if kv_format in _UNPACK:  # unpack every page once, then index codes
        k_logical = _UNPACK[kv_format](k_logical)
        v_logical = _UNPACK[kv_format](v_logical)
    n_q, d = qcodes_bg.shape
    out = np.zeros((n_q, d))
    for row in range(n_q):
        t = row // h_r
        logits = []
        for j in range(L):
            if causal and j > L - q_len + t:
                continue
            page = int(block_table[b][j // page_size])
            acc = 0.0
            for c in range(d):
                acc += (e4m3_value(qcodes_bg[row, c]) * qdesc) * (dec(k_logical[page, j % page_size, g, c]) * kdesc)
            logits.append((j, softmax_scale * acc))
        if not logits:
            continue
        mx = max(x for _, x in logits)
        den = sum(math.exp(x - mx) for _, x in logits)
        for j, x in logits:
            page = int(block_table[b][j // page_size])
            w = math.exp(x - mx) / den
            for c in range(d):
                out[row, c] += w * dec(v_logical[page, j % page_size, g, c]) * vdesc
    return out
