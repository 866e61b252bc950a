"""Planted mistakes in the oracle, to show that its pins would catch them.

Each entry of ``PLANTS`` is one plausible slip in the oracle: a dropped term,
a wrong sign, bias, index or comparison, a transposed operand, a swapped byte
or nibble order. It also names the pin module that must catch it.
:func:`apply` installs the mistake by replacing attributes of the oracle's
modules. It is called only by ``tests/conftest.py`` in a child pytest process
that ``tests/test_oracle_pins_catch_mistakes.py`` starts with the environment
variable ``MJ_PLANT`` set, on the CPU. The regular test run never installs
one.
"""

from __future__ import annotations

import numpy as np

from oracle import attention as A
from oracle import formats as F
from oracle import kvwrite as W
from oracle import plan as P
from oracle import qquant as Q

ATTN = "test_oracle_attention.py"
FMT = "test_oracle_formats.py"
QQ = "test_oracle_qquant.py"
PLAN = "test_oracle_plan.py"
KVW = "test_oracle_kvwrite.py"


# ----------------------------------------------------------------------------
# attention: mask, logits, gather, softmax, merge, output placement
# ----------------------------------------------------------------------------
def _mask(strict: bool, row_index_mod: bool):
    def visible_mask(L, q_len, h_r, causal):
        n_q = q_len * h_r
        t = np.arange(n_q) % h_r if row_index_mod else np.arange(n_q) // h_r
        j = np.arange(L)
        if not causal:
            return np.ones((n_q, L), dtype=bool)
        lim = (L - q_len + t)[:, None]
        return j[None, :] < lim if strict else j[None, :] <= lim
    A.visible_mask = visible_mask


def _logits(drop: str):
    orig = A.unit_logits

    def unit_logits(qc, qd, kc, kd, fmt, ss, q_values=False):
        if drop == "k_descale":
            kd = 1.0
        elif drop == "q_descale" and qd is not None:
            qd = 1.0
        elif drop == "softmax_scale":
            ss = 1.0
        return orig(qc, qd, kc, kd, fmt, ss, q_values=q_values)
    A.unit_logits = unit_logits


def _gather(kind: str):
    unpack = A._UNPACK

    def gather_unit(kl, vl, bt, b, g, L, ps, kv_format="fp8"):
        j = np.arange(L)
        if kind == "page_slot":  # page from the slot, slot from the page index
            pages, slots_ = np.asarray(bt)[b, j % ps], j // ps
        else:
            pages, slots_ = np.asarray(bt)[b, j // ps], j % ps
        if kind == "k_for_v":  # V rows read from the K cache
            vl = kl
        kc, vc = kl[pages, slots_, g, :], vl[pages, slots_, g, :]
        if kv_format in unpack:
            kc, vc = unpack[kv_format](kc), unpack[kv_format](vc)
        return kc, vc
    A.gather_unit = gather_unit


def _softmax_ignores_mask():
    def softmax_rows(s, vis):
        m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
        safe_m = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(s - safe_m[:, None])
        return m, p.sum(axis=1), p
    A.softmax_rows = softmax_rows


def _merge(kind: str):
    def merge_partials(ms, ls, os_):
        ms, ls, os_ = np.stack(ms), np.stack(ls), np.stack(os_)
        big_m = ms.max(axis=0)
        safe = np.where(np.isfinite(big_m), big_m, 0.0)
        e = np.exp(safe[None, :] - ms) if kind == "sign" else np.exp(ms - safe[None, :])
        w = np.where(np.isfinite(ms), e, 0.0)
        if kind != "no_l":
            w = w * ls
        tot = w.sum(axis=0)
        with np.errstate(invalid="ignore", divide="ignore"):
            o = np.where(tot[:, None] > 0,
                         (w[:, :, None] * os_).sum(axis=0) / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
            lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        return o, lse
    A.merge_partials = merge_partials


def _chunk_inclusive():
    orig = A.chunk_partial

    def chunk_partial(s, vis, v, a, e):
        return orig(s, vis, v, a, min(e + 1, s.shape[1]))
    A.chunk_partial = chunk_partial


def _decode_wrap(kind: str):
    orig = A.decode_attention

    def decode_attention(q_codes, q_descale, k_logical, v_logical, k_descale, v_descale, *args, **kw):
        if kind == "v_descale_from_k":
            v_descale = k_descale
        if kind == "o_mul_dropped":
            kw["o_mul"] = None
        out, lse = orig(q_codes, q_descale, k_logical, v_logical, k_descale, v_descale, *args, **kw)
        if kind == "lse_log2":
            lse = lse / np.log(2.0)
        if kind == "gqa_head_order":  # head g*h_r + r written to r*h_k + g
            h_q, h_k = kw["h_q"], kw["h_k"]
            h_r = h_q // h_k
            perm = [(h % h_r) * h_k + h // h_r for h in range(h_q)]
            moved = np.full_like(out, np.nan)
            moved[:, perm] = out
            out = moved
        return out, lse
    A.decode_attention = decode_attention


def _descale_by_request():
    def descale_at(ds, b, g):
        ds = np.asarray(ds, dtype=np.float64)
        if ds.size == 1:
            return float(ds.reshape(-1)[0])
        if ds.ndim == 1:
            return float(ds[b % ds.shape[0]])
        return float(ds[b, g])
    A.descale_at = descale_at


# ----------------------------------------------------------------------------
# formats: codecs and packings
# ----------------------------------------------------------------------------
def _e4m3_bias8():
    table = F.E4M3_TABLE / 2.0
    F.e4m3_value = lambda code: float(table[int(code) & 0xFF])
    F.E4M3_TABLE = table
    F._E4M3_POS = table[:0x7F].copy()
    F.e4m3_decode = lambda codes: table[np.asarray(codes, dtype=np.uint8)]


def _e4m3_encode(kind: str):
    vals = F._E4M3_POS

    def e4m3_encode(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        i = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, len(vals) - 1)
        top = i >= len(vals) - 1
        j = np.minimum(i + 1, len(vals) - 1)
        twice, mid = 2.0 * a, vals[i] + vals[j]
        up = twice >= mid if kind == "ties_away" else (twice > mid) | ((twice == mid) & (i % 2 == 1))
        code = np.where(up, j, i)
        code = np.where(top, 0x7F if kind == "no_saturation" else 0x7E, code).astype(np.uint8)
        code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
        return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
    F.e4m3_encode = e4m3_encode


def _narrow_value(fmt: str):
    if fmt == "e2m3":  # subnormal step 1/4 instead of 1/8
        def value(code):
            code = int(code) & 0x3F
            sign = -1.0 if code & 0x20 else 1.0
            e, m = (code >> 3) & 0x3, code & 0x7
            return sign * (m / 4.0 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 1))
        F.e2m3_value = value
        F.E2M3_TABLE = np.array([value(c) for c in range(64)])
        F._E2M3_POS = F.E2M3_TABLE[:0x20].copy()
        F.e2m3_decode = lambda codes: F.E2M3_TABLE[np.asarray(codes, dtype=np.uint8) & 0x3F]
    elif fmt == "e3m2":  # exponent bias 4 instead of 3
        table = F.E3M2_TABLE / 2.0
        F.e3m2_value = lambda code: float(table[int(code) & 0x3F])
        F.E3M2_TABLE = table
        F.e3m2_decode = lambda codes: table[np.asarray(codes, dtype=np.uint8) & 0x3F]
    elif fmt == "e2m1":  # subnormal m instead of m/2
        def value(code):
            code = int(code) & 0xF
            sign = -1.0 if code & 0x8 else 1.0
            e, m = (code >> 1) & 0x3, code & 0x1
            return sign * (float(m) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))
        F.e2m1_value = value
        F.E2M1_TABLE = np.array([value(c) for c in range(16)])
        F.e2m1_decode = lambda codes: F.E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def _fp6_big_endian():
    unpack, pack = F.fp6_unpack_rows, F.fp6_pack_rows

    def swap(rows):
        rows = np.asarray(rows, dtype=np.uint8)
        g = rows.reshape(rows.shape[:-1] + (rows.shape[-1] // 3, 3))[..., ::-1]
        return np.ascontiguousarray(g).reshape(rows.shape)
    F.fp6_unpack_rows = lambda packed: unpack(swap(packed))
    F.fp6_pack_rows = lambda codes: swap(pack(codes))


def _fp4_high_nibble_first():
    unpack, pack = F.fp4_unpack_rows, F.fp4_pack_rows

    def swap(rows):
        rows = np.asarray(rows, dtype=np.uint8)
        return ((rows >> 4) | (rows << 4)).astype(np.uint8)
    F.fp4_unpack_rows = lambda packed: unpack(swap(packed))
    F.fp4_pack_rows = lambda codes: swap(pack(codes))


# ----------------------------------------------------------------------------
# Q quantization
# ----------------------------------------------------------------------------
def _qquant(kind: str):
    orig = Q.quantize_q
    if kind == "max_240":
        Q.FP8_MAX = np.float32(240.0)
        return
    if kind == "no_floor":
        Q.AMAX_FLOOR = np.float32(0.0)
        return

    def quantize_q(q_f32, num_seqs, q_len, h_q, h_k, d, q_mul=None):
        if kind == "q_mul_ignored":
            return orig(q_f32, num_seqs, q_len, h_q, h_k, d, None)
        if kind == "amax_first_token":  # the scale from token 0 of the block only
            h_r = h_q // h_k
            x = np.asarray(q_f32, dtype=np.float32)[: num_seqs * q_len].copy()
            if q_mul is not None:
                x = (x * np.asarray(q_mul, dtype=np.float32).reshape(1, h_q, d)).astype(np.float32)
            x = x.reshape(num_seqs, q_len, h_k, h_r, d)
            amax = np.maximum(np.abs(x[:, :1]).max(axis=(1, 3, 4)).astype(np.float32), Q.AMAX_FLOOR)
            scale = (amax / Q.FP8_MAX).astype(np.float32)
            codes = Q.e4m3_encode((x / scale[:, None, :, None, None]).astype(np.float32))
            codes = codes.transpose(0, 2, 1, 3, 4).reshape(num_seqs, h_k, q_len * h_r, d)
            return np.ascontiguousarray(codes), scale
        codes, scale = orig(q_f32, num_seqs, q_len, h_q, h_k, d, q_mul)
        if kind == "row_order":  # rows r*q_len + t instead of t*h_r + r
            h_r = h_q // h_k
            c = codes.reshape(num_seqs, h_k, q_len, h_r, d).transpose(0, 1, 3, 2, 4)
            codes = np.ascontiguousarray(c).reshape(num_seqs, h_k, q_len * h_r, d)
        return codes, scale
    Q.quantize_q = quantize_q


# ----------------------------------------------------------------------------
# plan
# ----------------------------------------------------------------------------
def _plan(kind: str):
    orig = P.plan_split_kv

    def plan_split_kv(seq_lens, num_seqs, q_len, h_q, h_k, sm_count, ctas_per_sm, max_splits, margin, pad_to,
                      fp8_q=True):
        if kind == "margin_dropped":
            return orig(seq_lens, num_seqs, q_len, h_q, h_k, sm_count, ctas_per_sm, max_splits, 0, pad_to, fp8_q)
        h_r = h_q // h_k
        s = P.slots(sm_count, ctas_per_sm, h_k, P.n_tiles(q_len, h_r, fp8_q))
        grown = [int(seq_lens[b]) + margin for b in range(num_seqs)]
        if kind == "tile_floor":
            t = [n // P.KV_TILE for n in grown]
        else:
            t = [-(-n // P.KV_TILE) if n > 0 else 0 for n in grown]
        red = max_splits > 1 and (num_seqs <= s if kind == "reduction_le" else num_seqs < s)
        work, n_splits = [], []
        if not red:
            chunk = max([1] + t)
            for b in range(num_seqs):
                work.append([b, 0, t[b], 0])
                n_splits.append(1)
        else:
            cands = range(max([1] + t), 0, -1) if kind == "largest_chunk" else range(1, max([1] + t) + 1)
            chunk = max([1] + t)
            for c in cands:
                if (sum(max(1, -(-tb // c)) for tb in t) <= s
                        and max([0] + [-(-tb // c) for tb in t]) <= max_splits):
                    chunk = c
                    break
            for b in range(num_seqs):
                ns = max(1, -(-t[b] // chunk))
                n_splits.append(ns)
                for sp in range(ns):
                    work.append([b, sp * chunk, min((sp + 1) * chunk, t[b]), sp])
        if len(work) > pad_to:
            raise ValueError("pad_to too small")
        work += [[0, 0, 0, 0] for _ in range(pad_to - len(work))]
        return P.Plan(work=work, n_splits=n_splits, chunk_tiles=chunk, with_reduction=red, slots=s,
                      num_work=pad_to)
    P.plan_split_kv = plan_split_kv


# ----------------------------------------------------------------------------
# KV-cache write
# ----------------------------------------------------------------------------
def _kvwrite(kind: str):
    orig_q = W.quantize_rows
    if kind == "scale_multiplied":
        def quantize_rows(x, scale, kv_format):
            s = np.asarray(scale, dtype=np.float32)
            return orig_q(x, (1.0 / s).astype(np.float32), kv_format)
        W.quantize_rows = quantize_rows
        return

    def write_kv(key, value, k_pool, v_pool, slot_mapping, page_size, k_strides, v_strides, kv_format,
                 k_scale, v_scale):
        key = np.asarray(key, dtype=np.float32)
        value = np.asarray(value, dtype=np.float32)
        n_tok, h_k, d = key.shape
        rb = W.row_bytes(d, kv_format)
        kq = W.quantize_rows(key, k_scale, kv_format)
        vq = W.quantize_rows(value, v_scale, kv_format)
        for t in range(n_tok):
            slot = int(slot_mapping[t])
            if kind == "padding_written":  # clamped to slot 0 instead of skipped
                slot = max(slot, 0)
            if slot < 0:
                continue
            if kind == "slot_swapped":
                page, row = slot % page_size, slot // page_size
            else:
                page, row = slot // page_size, slot % page_size
            for pool, strides, q in ((k_pool, k_strides, kq), (v_pool, v_strides, vq)):
                for h in range(h_k):
                    off = page * strides[0] + row * strides[1] + h * strides[2]
                    if off + rb <= pool.shape[0]:
                        pool[off:off + rb] = q[t, h]
    W.write_kv = write_kv



# ----------------------------------------------------------------------------
# second batch: causal flag, o_mul index, split partials, encoders' signs and
# ties, code bit order, plan helpers, Q division and scale, cache-write scales
# ----------------------------------------------------------------------------
def _causal_ignored():
    orig = A.visible_mask
    A.visible_mask = lambda L, q_len, h_r, causal: orig(L, q_len, h_r, False)


def _o_mul_by_kv_head():
    orig = A.decode_attention

    def decode_attention(*args, **kw):
        om = kw.get("o_mul")
        if om is not None:
            om = np.asarray(om)
            h_r = kw["h_q"] // kw["h_k"]
            kw["o_mul"] = om[np.arange(kw["h_q"]) // h_r]  # row g of a query-head array
        return orig(*args, **kw)
    A.decode_attention = decode_attention


def _chunk_unnormalised():
    def chunk_partial(s, vis, v, a, e):
        n_q = s.shape[0]
        if e <= a:
            return np.full(n_q, -np.inf), np.zeros(n_q), np.zeros((n_q, v.shape[1]))
        m, l, p = A.softmax_rows(s[:, a:e], vis[:, a:e])
        return m, l, p @ v[a:e]
    A.chunk_partial = chunk_partial


def _e4m3_sign_dropped():
    orig = F.e4m3_encode
    F.e4m3_encode = lambda x: orig(np.abs(np.asarray(x, dtype=np.float64)))


def _ties_away_encoder(pos_values, sign_bit):
    def encode(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        n = len(pos_values)
        i = np.clip(np.searchsorted(pos_values, a, side="right") - 1, 0, n - 1)
        j = np.minimum(i + 1, n - 1)
        code = np.where(2.0 * a >= pos_values[i] + pos_values[j], j, i)
        code = np.where(i >= n - 1, n - 1, code).astype(np.uint8)
        return np.where(np.signbit(x), code | sign_bit, code).astype(np.uint8)
    return encode


def _fp6_code_bits_reversed():
    unpack, pack = F.fp6_unpack_rows, F.fp6_pack_rows
    rev = np.array([int(f"{c:06b}"[::-1], 2) for c in range(64)], dtype=np.uint8)
    F.fp6_unpack_rows = lambda packed: rev[unpack(packed)]
    F.fp6_pack_rows = lambda codes: pack(rev[np.asarray(codes, dtype=np.uint8) & 0x3F])


def _plan_helper(kind: str):
    if kind == "tile_width_base_8":
        def tile_width(n_q, fp8_q):
            p = 1
            while p < n_q:
                p *= 2
            return max(8, min(32, p))
        P.tile_width = tile_width
    elif kind == "slots_ignore_row_tiles":
        P.slots = lambda sm_count, ctas_per_sm, h_k, n_row_tiles: max(1, (sm_count * ctas_per_sm) // h_k)


def _q_copy(kind: str):
    def quantize_q(q_f32, num_seqs, q_len, h_q, h_k, d, q_mul=None):
        h_r = h_q // h_k
        x = np.asarray(q_f32, dtype=np.float32)[: num_seqs * q_len].copy()
        if q_mul is not None:
            x = (x * np.asarray(q_mul, dtype=np.float32).reshape(1, h_q, d)).astype(np.float32)
        x = x.reshape(num_seqs, q_len, h_k, h_r, d)
        if kind == "amax_head0":
            amax = np.abs(x[:, :, :, :1]).max(axis=(1, 3, 4)).astype(np.float32)
        else:
            amax = np.abs(x).max(axis=(1, 3, 4)).astype(np.float32)
        if kind == "floor_on_scale":  # the floor applied to the scale itself
            scale = np.maximum((amax / Q.FP8_MAX).astype(np.float32), Q.AMAX_FLOOR)
        else:
            scale = (np.maximum(amax, Q.AMAX_FLOOR) / Q.FP8_MAX).astype(np.float32)
        sb = scale[:, None, :, None, None]
        if kind == "reciprocal":
            y = (x * (np.float32(1.0) / sb).astype(np.float32)).astype(np.float32)
        else:
            y = (x / sb).astype(np.float32)
        codes = Q.e4m3_encode(y).transpose(0, 2, 1, 3, 4).reshape(num_seqs, h_k, q_len * h_r, d)
        return np.ascontiguousarray(codes), scale
    Q.quantize_q = quantize_q


def _write_head0_scale():
    orig = W.quantize_rows

    def quantize_rows(x, scale, kv_format):
        s = np.asarray(scale, dtype=np.float32)
        if s.size > 1:  # every head takes head 0's scale(s)
            s = np.broadcast_to(s[:1], s.shape).copy()
        return orig(x, s, kv_format)
    W.quantize_rows = quantize_rows


def _write_e2m3_ties_away():
    W.e2m3_encode = _ties_away_encoder(F.E2M3_TABLE[:0x20].copy(), 0x20)


# ----------------------------------------------------------------------------
# third batch: bf16-Q rows, format dispatch, merge LSE, bf16 rounding, the
# bf16-Q tile width, write row bytes, the non-causal flag
# ----------------------------------------------------------------------------
def _pack_q_head_major():
    orig = Q.pack_q_rows

    def pack_q_rows(q_f32, num_seqs, q_len, h_q, h_k, d):
        rows = orig(q_f32, num_seqs, q_len, h_q, h_k, d)
        h_r = h_q // h_k
        r = rows.reshape(num_seqs, h_k, q_len, h_r, d).transpose(0, 1, 3, 2, 4)
        return np.ascontiguousarray(r).reshape(num_seqs, h_k, q_len * h_r, d)
    Q.pack_q_rows = pack_q_rows


def _e3m2_decoded_as_e2m3():
    orig = A.decode_codes
    A.decode_codes = lambda codes, kv_format: orig(codes, "e2m3" if kv_format == "e3m2" else kv_format)


def _merge_lse_log2():
    orig = A.merge_partials

    def merge_partials(ms, ls, os_):
        o, lse = orig(ms, ls, os_)
        return o, lse / np.log(2.0)
    A.merge_partials = merge_partials


def _bf16_truncates():
    def to_bf16(x):
        x = np.asarray(x, dtype=np.float64)
        m, e = np.frexp(x)
        return np.ldexp(np.trunc(m * 256.0), e - 8)
    A.to_bf16 = to_bf16


def _tile_width_bf16_as_fp8():
    orig = P.tile_width
    P.tile_width = lambda n_q, fp8_q: orig(n_q, True)


def _write_e2m1_row_as_fp6():
    orig = W.row_bytes
    W.row_bytes = lambda d, kv_format: d * 3 // 4 if kv_format == W.KV_E2M1 else orig(d, kv_format)


def _noncausal_as_causal():
    orig = A.visible_mask
    A.visible_mask = lambda L, q_len, h_r, causal: orig(L, q_len, h_r, True)


def _narrow_sign_dropped(name):
    orig = getattr(F, name)
    setattr(F, name, lambda x: orig(np.abs(np.asarray(x, dtype=np.float64))))


def _write_e3m2_with_e2m3_encoder():
    W.e3m2_encode = W.e2m3_encode

PLANTS = {
    # name: (install, pin module that must catch it)
    "causal_mask_strict": (lambda: _mask(True, False), ATTN),
    "causal_row_from_gqa_index": (lambda: _mask(False, True), ATTN),
    "k_descale_dropped": (lambda: _logits("k_descale"), ATTN),
    "q_descale_dropped": (lambda: _logits("q_descale"), ATTN),
    "softmax_scale_dropped": (lambda: _logits("softmax_scale"), ATTN),
    "page_and_slot_swapped": (lambda: _gather("page_slot"), ATTN),
    "v_rows_from_k_cache": (lambda: _gather("k_for_v"), ATTN),
    "softmax_ignores_mask": (_softmax_ignores_mask, ATTN),
    "merge_weight_without_l": (lambda: _merge("no_l"), ATTN),
    "merge_weight_sign": (lambda: _merge("sign"), ATTN),
    "chunk_end_inclusive": (_chunk_inclusive, ATTN),
    "v_descale_from_k": (lambda: _decode_wrap("v_descale_from_k"), ATTN),
    "o_mul_dropped": (lambda: _decode_wrap("o_mul_dropped"), ATTN),
    "lse_in_log2": (lambda: _decode_wrap("lse_log2"), ATTN),
    "gqa_head_order": (lambda: _decode_wrap("gqa_head_order"), ATTN),
    "head_descale_by_request": (_descale_by_request, ATTN),
    "e4m3_bias_8": (_e4m3_bias8, FMT),
    "e4m3_ties_away": (lambda: _e4m3_encode("ties_away"), FMT),
    "e4m3_no_saturation": (lambda: _e4m3_encode("no_saturation"), FMT),
    "e2m3_subnormal_step": (lambda: _narrow_value("e2m3"), FMT),
    "e3m2_bias_4": (lambda: _narrow_value("e3m2"), FMT),
    "e2m1_subnormal": (lambda: _narrow_value("e2m1"), FMT),
    "fp6_bytes_reversed": (_fp6_big_endian, FMT),
    "fp4_high_nibble_first": (_fp4_high_nibble_first, FMT),
    "q_max_240": (lambda: _qquant("max_240"), QQ),
    "q_amax_floor_dropped": (lambda: _qquant("no_floor"), QQ),
    "q_mul_ignored": (lambda: _qquant("q_mul_ignored"), QQ),
    "q_amax_first_token_only": (lambda: _qquant("amax_first_token"), QQ),
    "q_row_order": (lambda: _qquant("row_order"), QQ),
    "plan_margin_dropped": (lambda: _plan("margin_dropped"), PLAN),
    "plan_tiles_floor": (lambda: _plan("tile_floor"), PLAN),
    "plan_reduction_le": (lambda: _plan("reduction_le"), PLAN),
    "plan_largest_chunk": (lambda: _plan("largest_chunk"), PLAN),
    "write_scale_multiplied": (lambda: _kvwrite("scale_multiplied"), KVW),
    "write_slot_swapped": (lambda: _kvwrite("slot_swapped"), KVW),
    "write_padding_token": (lambda: _kvwrite("padding_written"), KVW),
    "causal_flag_ignored": (_causal_ignored, ATTN),
    "o_mul_row_by_kv_head": (_o_mul_by_kv_head, ATTN),
    "split_partial_not_normalised": (_chunk_unnormalised, ATTN),
    "e4m3_sign_dropped": (_e4m3_sign_dropped, FMT),
    "e2m3_ties_away": (lambda: setattr(F, "e2m3_encode", _ties_away_encoder(F._E2M3_POS, 0x20)), FMT),
    "fp6_code_bits_reversed": (_fp6_code_bits_reversed, FMT),
    "plan_tile_width_base_8": (lambda: _plan_helper("tile_width_base_8"), PLAN),
    "plan_slots_ignore_row_tiles": (lambda: _plan_helper("slots_ignore_row_tiles"), PLAN),
    "q_reciprocal_multiply": (lambda: _q_copy("reciprocal"), QQ),
    "q_amax_first_query_head_only": (lambda: _q_copy("amax_head0"), QQ),
    "q_floor_on_the_scale": (lambda: _q_copy("floor_on_scale"), QQ),
    "write_every_head_uses_head0_scale": (_write_head0_scale, KVW),
    "write_e2m3_ties_away": (_write_e2m3_ties_away, KVW),
    "bf16_q_rows_head_major": (_pack_q_head_major, ATTN),
    "e3m2_decoded_as_e2m3": (_e3m2_decoded_as_e2m3, ATTN),
    "merge_lse_in_log2": (_merge_lse_log2, ATTN),
    "bf16_rounding_truncates": (_bf16_truncates, ATTN),
    "plan_bf16_q_tile_width_as_fp8": (_tile_width_bf16_as_fp8, PLAN),
    "write_e2m1_row_bytes_as_fp6": (_write_e2m1_row_as_fp6, KVW),
    "noncausal_block_masked_as_causal": (_noncausal_as_causal, ATTN),
    "e3m2_sign_dropped": (lambda: _narrow_sign_dropped("e3m2_encode"), FMT),
    "e2m1_sign_dropped": (lambda: _narrow_sign_dropped("e2m1_encode"), FMT),
    "write_e3m2_rows_with_e2m3_encoder": (_write_e3m2_with_e2m3_encoder, KVW),
}


def apply(name: str) -> None:
    """Install the planted mistake ``name`` (see ``PLANTS``)."""
    PLANTS[name][0]()
