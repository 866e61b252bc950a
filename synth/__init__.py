"""Seeded synthetic decode workloads, shared by the tests, the benchmark and
the oracle checks.

This module draws random numbers and lays out buffers; it holds none of the
decode path's arithmetic (no Q quantization, no attention, no plan). It does
act as the KV-cache WRITER for its synthetic caches — the step that comes
before the decode path (a cache write at ``slot_mapping``) — so it rounds
N(0,1) values to the stored code format:

* e4m3 KV: ``torch``'s own ``float8_e4m3fn`` conversion of ``X / s`` with
  ``s = amax/448`` per tensor or per KV head;
* e2m3 KV: nearest of the 64 e2m3 values (ties to the even code) of
  ``X / s_c`` with static per-(KV head, channel) scales ``s_c = amax/7.5``,
  packed 4 codes per 3 bytes as a little-endian bitstream;
* e3m2 / e2m1 KV: the same with the format's largest value (28 / 6) in the
  scale; e3m2 rows packed like e2m3 rows, e2m1 rows 2 codes per byte (low
  nibble first).

Unused pool pages and the tail slots of each request's last page are
poisoned (e4m3 NaN ``0x7F``; the narrow formats have no NaN, so their
largest code: ``0x1F`` for e2m3 and e3m2, ``0x7`` for e2m1),
and unused block-table entries are ``-1``: a decode path that reads past a
request's last valid key shows up as NaN or as a wrong result.

Every array is host (numpy) memory; callers move it to the device.
The named workloads follow the shapes of the pages' target model
(Qwen3-8B: 32 query heads, 8 KV heads, head size 128) at the sizes of the
five benchmark configurations; :func:`make_case` builds any smaller case.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

E4M3_NAN = 0x7F
E2M3_POISON = 0x1F
E3M2_POISON = 0x1F
E2M1_POISON = 0x7
# the narrow (channel-scaled) KV formats: largest value, row bits per code
NARROW = {"e2m3": (7.5, 6), "e3m2": (28.0, 6), "e2m1": (6.0, 4)}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


# sub-stream ids
_S_Q, _S_K, _S_V, _S_LENS, _S_PAGES, _S_OUTLIER_K, _S_OUTLIER_V = range(7)


@dataclass
class Workload:
    name: str
    num_seqs: int  # requests, real + trailing padding
    q_len: int
    h_q: int
    h_k: int
    d: int
    page_size: int
    kv_format: str  # "fp8" | "e2m3" | "e3m2" | "e2m1"
    layout: str  # "HND" | "NHD"
    causal: bool
    seq_lens: np.ndarray  # int32 [B]; padding requests 0
    block_table: np.ndarray  # int32 [B, max_blocks]; unused entries -1
    num_pages: int
    q_bits: np.ndarray  # uint16 [B*q_len, h_q, d], bf16 bit patterns
    q_f32: np.ndarray  # float32 [B*q_len, h_q, d], the same values
    k_cache: np.ndarray  # uint8 physical buffer
    v_cache: np.ndarray
    kv_strides: tuple  # (page, token, head) byte strides of k_cache/v_cache
    row_bytes: int
    k_scale: np.ndarray  # float32: (1,) per tensor, (h_k,) per head
    v_scale: np.ndarray
    q_mul: np.ndarray | None = None  # float32 [h_q, d] (e2m3: K channel scales)
    o_mul: np.ndarray | None = None  # float32 [h_q, d] (e2m3: V channel scales)
    softmax_scale: float = 0.0
    meta: dict = field(default_factory=dict)

    @property
    def h_r(self) -> int:
        return self.h_q // self.h_k

    @property
    def n_q(self) -> int:
        return self.q_len * self.h_r

    def logical(self, which: str) -> np.ndarray:
        """``[num_pages, page_size, h_k, row_bytes]`` view of the K or V buffer."""
        buf = self.k_cache if which == "k" else self.v_cache
        if self.layout == "HND":
            return buf.transpose(0, 2, 1, 3)
        return buf


# ----------------------------------------------------------------------------
# synthetic cache writer
# ----------------------------------------------------------------------------
def _absmax(x: np.ndarray) -> float:
    return max(float(x.max()), -float(x.min())) if x.size else 0.0


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _e2m3_codes(x: np.ndarray) -> np.ndarray:
    """Nearest e2m3 code (ties to even) of float32 values with |x| <= 7.5.

    In [1, 7.5] e2m3 and e4m3 both carry 3 mantissa bits with normal
    exponents, so torch's e4m3 conversion rounds identically there and the
    e2m3 code is the e4m3 code with the exponent rebased (bias 7 -> bias 1).
    Below 1, e2m3 is the subnormal grid k/8 and the code is rint(8|x|)
    (ties to the even k, i.e. the even code)."""
    a = np.abs(x.astype(np.float32, copy=False))
    big = a >= 1.0
    c8 = _e4m3_codes(np.minimum(a, np.float32(7.5)))
    e4 = (c8 >> 3).astype(np.int16)
    hi = ((e4 - 6) << 3) | (c8 & 7)
    lo = np.rint(a * np.float32(8.0)).astype(np.int16)
    code = np.where(big, np.minimum(hi, 31), lo).astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x20), np.uint8(0))


def _e3m2_codes(x: np.ndarray) -> np.ndarray:
    """Nearest e3m2 code (ties to even) of float32 values, saturating at 28.

    In [0.25, 28] e3m2 and e5m2 both carry 2 mantissa bits with normal
    exponents, so torch's float8_e5m2 conversion rounds identically there and
    the e3m2 code is the e5m2 code with the exponent rebased (bias 15 -> 3).
    Below 0.25, e3m2 is the subnormal grid k/16 and the code is rint(16|x|)."""
    import torch

    a = np.minimum(np.abs(x.astype(np.float32, copy=False)), np.float32(28.0))
    c5 = torch.from_numpy(np.ascontiguousarray(a)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    hi = (((c5 >> 2).astype(np.int16) - 12) << 2) | (c5 & 3)
    lo = np.rint(a * np.float32(16.0)).astype(np.int16)
    code = np.where(a >= 0.25, hi, lo).astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x20), np.uint8(0))


def _e2m1_codes(x: np.ndarray) -> np.ndarray:
    """Nearest e2m1 code (ties to even) of float32 values, saturating at 6:
    per binade the code is its first code plus rint of the offset in steps
    (0.5 below 2, 1 in [2, 4), 2 in [4, 6]); rint's ties to even are the even
    codes."""
    a = np.minimum(np.abs(x.astype(np.float32, copy=False)), np.float32(6.0))
    code = np.where(a < 1.0, np.rint(2 * a),
                    np.where(a < 2.0, 2 + np.rint(2 * (a - 1)),
                             np.where(a < 4.0, 4 + np.rint(a - 2), 6 + np.rint((a - 4) / 2))))
    code = code.astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x8), np.uint8(0))


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """``[..., 2k]`` 4-bit codes -> ``[..., k]`` bytes, code 2j in the low nibble of byte j."""
    c = codes.astype(np.uint8).reshape(codes.shape[:-1] + (codes.shape[-1] // 2, 2))
    return (c[..., 0] | (c[..., 1] << 4)).astype(np.uint8)


def _narrow_rows(x: np.ndarray, kv_format: str) -> np.ndarray:
    """Scaled values -> packed rows of a narrow format."""
    if kv_format == "e2m3":
        return pack_e2m3(_e2m3_codes(x))
    if kv_format == "e3m2":
        return pack_e2m3(_e3m2_codes(x))
    return pack_e2m1(_e2m1_codes(x))


def pack_e2m3(codes: np.ndarray) -> np.ndarray:
    """``[..., 4k]`` 6-bit codes -> ``[..., 3k]`` bytes, little-endian bitstream."""
    n = codes.shape[-1]
    c = codes.astype(np.uint32).reshape(codes.shape[:-1] + (n // 4, 4))
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    b0 = (c0 | (c1 << 6)) & 0xFF
    b1 = ((c1 >> 2) | (c2 << 4)) & 0xFF
    b2 = ((c2 >> 4) | (c3 << 2)) & 0xFF
    out = np.stack([b0, b1, b2], axis=-1).astype(np.uint8)
    return out.reshape(codes.shape[:-1] + (n // 4 * 3,))


# ----------------------------------------------------------------------------
# builder
# ----------------------------------------------------------------------------
def make_case(*, name="case", num_seqs, q_len, h_q, h_k, d=128, page_size, seq_lens, layout="HND",
              kv_format="fp8", scale_mode="head", causal=True, pool_pages=None, seed=0,
              outlier_channels=0, outlier_gain=10.0, extra_block_cols=0, kv_values=None,
              q_values=None) -> Workload:
    """Build a seeded workload.

    ``seq_lens``: lengths of all ``num_seqs`` requests (0 = padding request).
    ``pool_pages``: pool size; default exactly the pages the requests use.
    Pages are drawn without replacement from the pool in a seeded random
    order. ``scale_mode``: "tensor" | "head" (e4m3) — the narrow formats
    (e2m3, e3m2, e2m1) always use per-(KV head, channel) scales folded into
    ``q_mul`` / ``o_mul``.
    ``kv_values``: optional ``(which, g, tok_req, tok_pos) -> float32 [n_tok, d]``
    giving the K ("k") or V ("v") values of KV head ``g`` for the valid
    tokens (request index and position of each) in place of N(0,1) draws;
    ``q_values``: optional float32 ``[num_seqs*q_len, h_q, d]`` in place of
    the N(0,1) Q (rounded to bf16 like it).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (num_seqs,)
    h_r = h_q // h_k
    pages_per = [math.ceil(int(L) / page_size) for L in seq_lens]
    need = sum(pages_per)
    pool = need if pool_pages is None else int(pool_pages)
    assert pool >= need
    pool = max(pool, 1)
    max_blocks = max([1] + pages_per) + extra_block_cols

    order = _rng(seed, _S_PAGES).permutation(pool)[:need].astype(np.int32)
    block_table = np.full((num_seqs, max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages_per):
        block_table[b, :n] = order[off:off + n]
        off += n

    # (page, slot) of every valid token, request-major
    tok_pages, tok_slots, tok_req, tok_pos = [], [], [], []
    for b, L in enumerate(seq_lens):
        j = np.arange(int(L))
        tok_pages.append(block_table[b, j // page_size])
        tok_slots.append(j % page_size)
        tok_req.append(np.full(int(L), b, dtype=np.int64))
        tok_pos.append(j)
    tok_pages = np.concatenate(tok_pages) if tok_pages else np.zeros(0, np.int32)
    tok_slots = np.concatenate(tok_slots) if tok_slots else np.zeros(0, np.int64)
    tok_req = np.concatenate(tok_req) if tok_req else np.zeros(0, np.int64)
    tok_pos = np.concatenate(tok_pos) if tok_pos else np.zeros(0, np.int64)
    n_tok = len(tok_pages)

    row_bytes = d if kv_format == "fp8" else d * NARROW[kv_format][1] // 8
    if layout == "HND":
        shape = (pool, h_k, page_size, row_bytes)
        strides = (h_k * page_size * row_bytes, row_bytes, page_size * row_bytes)
    elif layout == "NHD":
        shape = (pool, page_size, h_k, row_bytes)
        strides = (page_size * h_k * row_bytes, h_k * row_bytes, row_bytes)
    else:
        raise ValueError(layout)

    if kv_format == "fp8":
        poison_row = np.full(row_bytes, E4M3_NAN, dtype=np.uint8)
    elif kv_format == "e2m1":
        poison_row = pack_e2m1(np.full(d, E2M1_POISON, dtype=np.uint8))
    else:
        poison_row = pack_e2m3(np.full(d, E2M3_POISON if kv_format == "e2m3" else E3M2_POISON, dtype=np.uint8))

    # flat row index of (page, head g, slot) in the physical buffer
    def flat_rows(g):
        if layout == "HND":
            return (tok_pages.astype(np.int64) * h_k + g) * page_size + tok_slots
        return (tok_pages.astype(np.int64) * page_size + tok_slots) * h_k + g

    meta = {}
    caches, scales, chans = {}, {}, {}
    chunk = 1 << 16  # tokens per encode pass (bounds the temporaries)
    for which, stream, ostream in (("k", _S_K, _S_OUTLIER_K), ("v", _S_V, _S_OUTLIER_V)):
        buf = np.empty(shape, dtype=np.uint8)
        buf[...] = poison_row
        rows = buf.reshape(-1, row_bytes)
        per_head_scale = np.zeros(h_k, dtype=np.float32)
        ch_scale = np.zeros((h_k, d), dtype=np.float32)
        outl = [None] * h_k

        def draw(g):
            """KV head g's values: its own seeded streams (the heads draw in parallel)."""
            if kv_values is not None:
                return np.asarray(kv_values(which, g, tok_req, tok_pos), dtype=np.float32).reshape(n_tok, d)
            x = _rng(seed, 1000 * stream + g).standard_normal((n_tok, d), dtype=np.float32)
            if outlier_channels:
                ch = _rng(seed, 1000 * ostream + g).choice(d, size=outlier_channels, replace=False)
                x[:, ch] *= np.float32(outlier_gain)
                outl[g] = sorted(int(c) for c in ch)
            return x

        def encode(g, x, s_):
            """Scale and encode head g's rows in chunks and write them into the cache."""
            fr = flat_rows(g)
            for a in range(0, n_tok, chunk):
                xs_ = x[a:a + chunk] / s_
                codes = _e4m3_codes(xs_) if kv_format == "fp8" else _narrow_rows(xs_, kv_format)
                rows[fr[a:a + chunk]] = codes

        def head(g, tensor_scale=None):
            x = xs[g] if xs is not None else draw(g)
            if kv_format == "fp8":
                if tensor_scale is not None:
                    s_ = tensor_scale
                else:
                    s_ = np.float32((_absmax(x) if x.size else 1.0) / 448.0)
                    per_head_scale[g] = s_
            else:
                s_c = (np.maximum(x.max(axis=0), -x.min(axis=0)) if x.size
                       else np.ones(d, np.float32)).astype(np.float32)
                s_c = np.maximum(s_c / np.float32(NARROW[kv_format][0]), np.float32(1e-30))
                ch_scale[g] = s_c
                s_ = s_c[None, :]
            encode(g, x, s_)
            if xs is not None:
                xs[g] = None

        workers = max(1, min(h_k, os.cpu_count() or 1, 8))
        tensor_scale = np.float32(1.0)
        xs = None
        with ThreadPoolExecutor(max_workers=workers) as ex:
            if kv_format == "fp8" and scale_mode == "tensor":
                xs = list(ex.map(draw, range(h_k)))
                amax = max([_absmax(x) for x in xs] + [1e-30])
                tensor_scale = np.float32(amax / 448.0)
                list(ex.map(lambda g: head(g, tensor_scale), range(h_k)))
            else:
                list(ex.map(head, range(h_k)))
        if outlier_channels and kv_values is None:
            meta[f"{which}_outlier_channels"] = outl
        caches[which] = buf
        if kv_format == "fp8":
            scales[which] = (np.array([tensor_scale], dtype=np.float32) if scale_mode == "tensor"
                             else per_head_scale)
        else:
            scales[which] = np.ones(1, dtype=np.float32)
            chans[which] = ch_scale

    qrng = _rng(seed, _S_Q)
    q = qrng.standard_normal((num_seqs * q_len, h_q, d), dtype=np.float32)
    if q_values is not None:
        q = np.ascontiguousarray(q_values, dtype=np.float32).reshape(num_seqs * q_len, h_q, d)
    import torch

    qb = torch.from_numpy(q).to(torch.bfloat16)
    q_bits = qb.view(torch.int16).numpy().view(np.uint16).copy()
    q_f32 = qb.to(torch.float32).numpy().copy()

    q_mul = o_mul = None
    if kv_format in NARROW:
        q_mul = np.repeat(chans["k"], h_r, axis=0).astype(np.float32)
        o_mul = np.repeat(chans["v"], h_r, axis=0).astype(np.float32)

    return Workload(name=name, num_seqs=num_seqs, q_len=q_len, h_q=h_q, h_k=h_k, d=d,
                    page_size=page_size, kv_format=kv_format, layout=layout, causal=causal,
                    seq_lens=seq_lens, block_table=block_table, num_pages=pool, q_bits=q_bits,
                    q_f32=q_f32, k_cache=caches["k"], v_cache=caches["v"], kv_strides=strides,
                    row_bytes=row_bytes, k_scale=scales["k"], v_scale=scales["v"], q_mul=q_mul,
                    o_mul=o_mul, softmax_scale=1.0 / math.sqrt(d), meta=meta)


# ----------------------------------------------------------------------------
# the five benchmark configurations
# ----------------------------------------------------------------------------
def _uniform_lens(seed, n, lo, hi):
    return _rng(seed, _S_LENS).integers(lo, hi + 1, size=n).astype(np.int32)


def sink_case(*, name="sink", seq_lens, sink_pos, gap_binades=20.0, h_q=32, h_k=8, d=128, page_size=64,
              layout="NHD", seed=1020) -> Workload:
    """One dominant key per request (an attention sink) over many near-equal
    others, e4m3 KV with per-KV-head scales.

    Q = 1 + 0.05 N(0,1) (every channel near 1). The other keys' K rows are
    0.01 N(0,1), so their logits sit near 0 and close to one another; the
    sink's K row is the constant kappa = gap * ln 2 / sqrt(d), so with the
    softmax scale 1/sqrt(d) its logit is about ``gap_binades`` binades (gap *
    ln 2 nats) above the others for every query row. V: the others
    1 + 0.25 N(0,1), the sink -2 in every channel, so the output is a visible
    mix of the two whenever the others' share of the weight is not tiny.
    ``sink_pos[b]``: the sink's position in request b (negative: from the end).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = len(seq_lens)
    pos = np.array([int(p_) if p_ >= 0 else int(L) + int(p_) for p_, L in zip(sink_pos, seq_lens)], np.int64)
    kappa = np.float32(gap_binades * math.log(2.0) / math.sqrt(d))

    def kv_values(which, g, tok_req, tok_pos):
        rng = _rng(seed, 100 + 2 * g + (which == "v"))
        n = len(tok_req)
        is_sink = tok_pos == pos[tok_req]
        if which == "k":
            x = rng.standard_normal((n, d), dtype=np.float32) * np.float32(0.01)
            x[is_sink] = kappa
        else:
            x = np.float32(1.0) + rng.standard_normal((n, d), dtype=np.float32) * np.float32(0.25)
            x[is_sink] = np.float32(-2.0)
        return x

    q = np.float32(1.0) + np.float32(0.05) * _rng(seed, _S_Q).standard_normal((B, h_q, d), dtype=np.float32)
    w = make_case(name=name, num_seqs=B, q_len=1, h_q=h_q, h_k=h_k, d=d, page_size=page_size,
                  seq_lens=seq_lens, layout=layout, scale_mode="head", seed=seed, kv_values=kv_values,
                  q_values=q)
    w.meta["sink_pos"] = pos.tolist()
    w.meta["gap_binades"] = float(gap_binades)
    return w


def tiny(seed: int = 1001) -> Workload:
    """B=2, q_len=1, 8/2 heads, D=128, page 16, lens {37, 100}, e4m3 KV with one
    per-tensor scale each for K and V, HND, 10 pages in a seeded permutation."""
    return make_case(name="tiny", num_seqs=2, q_len=1, h_q=8, h_k=2, page_size=16,
                     seq_lens=[37, 100], layout="HND", scale_mode="tensor", seed=seed)


def qwen3_8b_decode(seed: int = 1002) -> Workload:
    """B=64, q_len=1, 32/8 heads, page 16, every length 4096, per-KV-head e4m3
    scales, HND, 16384 distinct pages drawn from a 20000-page pool."""
    return make_case(name="qwen3_8b_decode", num_seqs=64, q_len=1, h_q=32, h_k=8, page_size=16,
                     seq_lens=[4096] * 64, layout="HND", scale_mode="head", pool_pages=20000,
                     seed=seed)


def long_split(seed: int = 1003) -> Workload:
    """B=8, q_len=1, 32/8 heads, page 64, lengths uniform in [32768, 131072],
    per-KV-head e4m3 scales, NHD."""
    return make_case(name="long_split", num_seqs=8, q_len=1, h_q=32, h_k=8, page_size=64,
                     seq_lens=_uniform_lens(seed, 8, 32768, 131072), layout="NHD",
                     scale_mode="head", seed=seed)


def long_single(seed: int = 1013) -> Workload:
    """B=1, a single 131072-token sequence, otherwise as :func:`long_split`."""
    return make_case(name="long_single", num_seqs=1, q_len=1, h_q=32, h_k=8, page_size=64,
                     seq_lens=[131072], layout="NHD", scale_mode="head", seed=seed)


def spec_verify(causal: bool = True, seed: int = 1004) -> Workload:
    """B = 32 real + 8 trailing zero-token padding requests, q_len=4, page 32,
    lengths uniform in [1024, 16384], one per-tensor e4m3 scale, HND."""
    lens = np.concatenate([_uniform_lens(seed, 32, 1024, 16384), np.zeros(8, np.int32)])
    return make_case(name="spec_verify" + ("" if causal else "_noncausal"), num_seqs=40, q_len=4,
                     h_q=32, h_k=8, page_size=32, seq_lens=lens, layout="HND",
                     scale_mode="tensor", causal=causal, seed=seed)


def fp6_decode(seed: int = 1005) -> Workload:
    """B=128, q_len=1, 64/8 heads (GQA 8), page 128, every length 8192, packed
    e2m3 KV with 4 seeded x10 outlier channels per KV head (independently for
    K and V) and per-(KV head, channel) scales = amax/7.5, HND."""
    return make_case(name="fp6_decode", num_seqs=128, q_len=1, h_q=64, h_k=8, page_size=128,
                     seq_lens=[8192] * 128, layout="HND", kv_format="e2m3", outlier_channels=4,
                     seed=seed)


def fp6_e3m2_decode(seed: int = 1007) -> Workload:
    """:func:`fp6_decode` with packed e3m2 KV (largest 28; channel scales amax/28)."""
    return make_case(name="fp6_e3m2_decode", num_seqs=128, q_len=1, h_q=64, h_k=8, page_size=128,
                     seq_lens=[8192] * 128, layout="HND", kv_format="e3m2", outlier_channels=4,
                     seed=seed)


def fp4_decode(seed: int = 1008) -> Workload:
    """:func:`fp6_decode` with packed e2m1 KV (largest 6; channel scales amax/6):
    64-byte rows, 1.07 GB of KV."""
    return make_case(name="fp4_decode", num_seqs=128, q_len=1, h_q=64, h_k=8, page_size=128,
                     seq_lens=[8192] * 128, layout="HND", kv_format="e2m1", outlier_channels=4,
                     seed=seed)


def d256_decode(seed: int = 1006) -> Workload:
    """B=64, q_len=1, 16/8 heads (GQA 2), head size 256 (the head shape of
    Gemma-2/3-class models), page 16, every length 4096, per-KV-head e4m3
    scales, HND: 1.07 GB of KV, twice the Qwen3-8B batch's."""
    return make_case(name="d256_decode", num_seqs=64, q_len=1, h_q=16, h_k=8, d=256, page_size=16,
                     seq_lens=[4096] * 64, layout="HND", scale_mode="head", seed=seed)


WORKLOADS = {
    "tiny": tiny,
    "qwen3_8b_decode": qwen3_8b_decode,
    "long_split": long_split,
    "long_single": long_single,
    "spec_verify": spec_verify,
    "spec_verify_noncausal": lambda seed=1004: spec_verify(False, seed),
    "fp6_decode": fp6_decode,
    "d256_decode": d256_decode,
    "fp6_e3m2_decode": fp6_e3m2_decode,
    "fp4_decode": fp4_decode,
}


# ----------------------------------------------------------------------------
# inputs of the KV-cache write (mj_write_kv)
# ----------------------------------------------------------------------------
@dataclass
class WriteCase:
    name: str
    key_bf16: np.ndarray    # uint16 bf16 bits [T, h_k, d]
    value_bf16: np.ndarray
    key: np.ndarray         # float32 values of the bf16 inputs (exact)
    value: np.ndarray
    slots: np.ndarray       # int64 [T]; -1 = padding token
    k_pool: np.ndarray      # uint8, pre-filled with random bytes (written in place)
    v_pool: np.ndarray
    kv_strides: tuple       # byte strides (page, token, head)
    page_size: int
    num_pages: int
    kv_format: str          # "fp8" | "e2m3" | "e3m2" | "e2m1"
    k_scale: np.ndarray     # float32: [1] / [h_k] (fp8) or [h_k, d] (narrow formats)
    v_scale: np.ndarray
    scale_per_head: bool


def kv_write_case(*, name="write", num_tokens, h_k=8, d=128, page_size=16, num_pages, layout="HND",
                  kv_format="fp8", scale_mode="head", pad_every=0, outlier_channels=0, seed=0) -> WriteCase:
    """New K/V rows (N(0,1), rounded to bf16, optional x10 outlier channels),
    a slot for each token (distinct, random over the pool; every
    ``pad_every``-th token is padding, slot -1), pools pre-filled with random
    bytes, and scales: fp8 ``amax/448`` per tensor or per KV head, the narrow
    formats ``amax/max`` per (KV head, channel) (max 7.5 / 28 / 6)."""
    import torch

    rng = _rng(seed, 20)
    x = rng.standard_normal((2, num_tokens, h_k, d), dtype=np.float32)
    if outlier_channels:
        for s in range(2):
            for g in range(h_k):
                ch = rng.choice(d, outlier_channels, replace=False)
                x[s, :, g, ch] *= 10.0
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xf = (bits.astype(np.uint32) << 16).view(np.float32)  # exact float32 of the bf16 values
    cap = num_pages * page_size
    assert num_tokens <= cap
    slots = rng.permutation(cap)[:num_tokens].astype(np.int64)
    if pad_every:
        slots[pad_every - 1::pad_every] = -1
    rb = d if kv_format == "fp8" else d * NARROW[kv_format][1] // 8
    strides = (h_k * page_size * rb, rb, page_size * rb) if layout == "HND" else (page_size * h_k * rb, h_k * rb, rb)
    size = num_pages * page_size * h_k * rb
    k_pool = rng.integers(0, 256, size, dtype=np.uint8)
    v_pool = rng.integers(0, 256, size, dtype=np.uint8)
    live = slots >= 0
    scales = []
    for s in range(2):
        v = np.abs(xf[s][live]) if live.any() else np.ones((1, h_k, d), np.float32)
        if kv_format in NARROW:
            scales.append(np.maximum(v.max(axis=0), 1e-6).astype(np.float32) / np.float32(NARROW[kv_format][0]))
        elif scale_mode == "head":
            scales.append(np.maximum(v.max(axis=(0, 2)), 1e-6).astype(np.float32) / np.float32(448.0))
        else:
            scales.append(np.array([max(float(v.max()), 1e-6) / 448.0], dtype=np.float32))
    return WriteCase(name=name, key_bf16=bits[0], value_bf16=bits[1], key=xf[0], value=xf[1], slots=slots,
                     k_pool=k_pool, v_pool=v_pool, kv_strides=strides, page_size=page_size, num_pages=num_pages,
                     kv_format=kv_format, k_scale=scales[0], v_scale=scales[1],
                     scale_per_head=(kv_format == "fp8" and scale_mode == "head"))
