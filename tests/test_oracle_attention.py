"""Pins of the oracle's exact paged decode attention and of the LSE merge."""

import math

import numpy as np
import pytest
import scipy.special

import synth
from oracle import attention as A
from oracle import formats as F
from oracle.qquant import quantize_q


def _run(w, units=None, causal=None):
    codes, desc = quantize_q(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d, w.q_mul)
    out, lse = A.decode_attention(
        codes, desc, w.logical("k"), w.logical("v"), w.k_scale, w.v_scale, w.block_table,
        w.seq_lens, num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
        page_size=w.page_size, kv_format=w.kv_format, softmax_scale=w.softmax_scale,
        causal=w.causal if causal is None else causal, o_mul=w.o_mul, units=units)
    return codes, desc, out, lse


def _small(**kw):
    base = dict(num_seqs=3, q_len=1, h_q=4, h_k=2, d=128, page_size=16, seq_lens=[5, 33, 17],
                layout="HND", seed=11)
    base.update(kw)
    return synth.make_case(**base)


def _unit_scale(scale, g):
    """The K or V descale of KV head ``g``, read straight from the array the
    workload holds: one value for the whole tensor, or one per KV head.
    (Kept apart from the oracle's own lookup so that a wrong index there shows.)"""
    s = np.asarray(scale, dtype=np.float64).reshape(-1)
    return float(s[0]) if s.size == 1 else float(s[g])


@pytest.mark.parametrize("kv_format,q_len,causal,d", [("fp8", 1, True, 128), ("fp8", 3, True, 128),
                                                      ("fp8", 3, False, 128), ("e2m3", 2, True, 128),
                                                      ("fp8", 2, True, 256), ("e2m3", 1, False, 256),
                                                      ("e3m2", 2, True, 128), ("e2m1", 1, True, 128),
                                                      ("e2m1", 3, False, 256)])
def test_matches_brute_force(kv_format, q_len, causal, d):
    w = _small(kv_format=kv_format, q_len=q_len, causal=causal, seq_lens=[5, 21, 9], d=d,
               outlier_channels=0 if kv_format == "fp8" else 2)
    codes, desc, out, _ = _run(w)
    for b in range(w.num_seqs):
        for g in range(w.h_k):
            bf = A.brute_force_unit(codes[b, g], float(desc[b, g]), w.logical("k"), w.logical("v"),
                                    _unit_scale(w.k_scale, g), _unit_scale(w.v_scale, g),
                                    w.block_table, b, g, int(w.seq_lens[b]), w.page_size, w.kv_format,
                                    w.softmax_scale, w.q_len, w.h_r, causal)
            for row in range(w.n_q):
                t, r = divmod(row, w.h_r)
                o = out[b * w.q_len + t, g * w.h_r + r]
                want = bf[row] * (w.o_mul[g * w.h_r + r] if w.o_mul is not None else 1.0)
                np.testing.assert_allclose(o, want, rtol=1e-10, atol=1e-12)



def test_per_request_and_head_descales_match_brute_force():
    """Descales given per (request, KV head), a [B, H_k] array whose entries
    all differ: unit (b, g) must use entry [b, g]."""
    w = _small(seq_lens=[5, 21, 9], num_seqs=3, h_q=4, h_k=2)
    ks = np.array([[0.5, 0.75], [1.25, 2.0], [3.0, 0.375]]) * 0.01
    vs = np.array([[2.0, 0.25], [0.625, 1.5], [0.875, 4.0]]) * 0.01
    codes, desc = quantize_q(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d, w.q_mul)
    out, _ = A.decode_attention(codes, desc, w.logical("k"), w.logical("v"), ks, vs, w.block_table, w.seq_lens,
                                num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
                                page_size=w.page_size, kv_format=w.kv_format, softmax_scale=w.softmax_scale,
                                causal=w.causal)
    for b in range(w.num_seqs):
        for g in range(w.h_k):
            bf = A.brute_force_unit(codes[b, g], float(desc[b, g]), w.logical("k"), w.logical("v"), ks[b][g],
                                    vs[b][g], w.block_table, b, g, int(w.seq_lens[b]), w.page_size, w.kv_format,
                                    w.softmax_scale, w.q_len, w.h_r, w.causal)
            np.testing.assert_allclose(out[b, g * w.h_r:(g + 1) * w.h_r], bf, rtol=1e-10, atol=1e-12)

def test_paged_equals_contiguous_and_page_permutation():
    """The same tokens scattered over random pages of a larger pool, or laid
    out contiguously from page 0, give the same result."""
    w1 = _small(pool_pages=40, seed=5)
    w2 = _small(pool_pages=40, seed=5)
    bt = np.full_like(w2.block_table, -1)
    kc = np.zeros_like(w2.k_cache)
    vc = np.zeros_like(w2.v_cache)
    nxt = 0
    for b in range(w2.num_seqs):
        for j, p in enumerate(w2.block_table[b]):
            if p < 0:
                continue
            bt[b, j] = nxt
            kc[nxt] = w2.k_cache[p]
            vc[nxt] = w2.v_cache[p]
            nxt += 1
    w2.block_table, w2.k_cache, w2.v_cache = bt, kc, vc
    _, _, o1, l1 = _run(w1)
    _, _, o2, l2 = _run(w2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_hnd_and_nhd_views_agree():
    w1 = _small(layout="HND", seed=9)
    w2 = _small(layout="NHD", seed=9)
    np.testing.assert_array_equal(w1.logical("k"), w2.logical("k"))
    _, _, o1, _ = _run(w1)
    _, _, o2, _ = _run(w2)
    np.testing.assert_array_equal(o1, o2)


@pytest.mark.parametrize("d", [128, 256])
def test_constant_v_returns_v(d):
    w = _small(d=d)
    w.v_cache[...] = F.e4m3_encode(1.5)
    _, _, out, _ = _run(w)
    for b in range(w.num_seqs):
        for g in range(w.h_k):
            v = 1.5 * A.descale_at(w.v_scale, b, g)
            np.testing.assert_allclose(out[b, g * w.h_r:(g + 1) * w.h_r], v, rtol=1e-13)


def test_single_key_returns_its_v_row():
    w = _small(seq_lens=[1, 1, 1])
    _, _, out, _ = _run(w)
    for b in range(w.num_seqs):
        for g in range(w.h_k):
            p = w.block_table[b, 0]
            v = F.e4m3_decode(w.logical("v")[p, 0, g]) * A.descale_at(w.v_scale, b, g)
            for r in range(w.h_r):
                np.testing.assert_allclose(out[b, g * w.h_r + r], v, rtol=1e-13)


@pytest.mark.parametrize("d", [128, 256])
def test_one_row_is_scipy_softmax_times_v(d):
    w = _small(d=d)
    codes, desc, out, lse = _run(w)
    b, g = 1, 1
    L = int(w.seq_lens[b])
    kc, vc = A.gather_unit(w.logical("k"), w.logical("v"), w.block_table, b, g, L, w.page_size)
    q = F.e4m3_decode(codes[b, g, 0]) * float(desc[b, g])
    k = F.e4m3_decode(kc) * A.descale_at(w.k_scale, b, g)
    v = F.e4m3_decode(vc) * A.descale_at(w.v_scale, b, g)
    s = w.softmax_scale * (k @ q)
    np.testing.assert_allclose(out[b, g * w.h_r], scipy.special.softmax(s) @ v, rtol=1e-12)
    assert math.isclose(lse[b, g, 0], scipy.special.logsumexp(s), rel_tol=1e-12)


def test_causal_last_row_equals_noncausal_and_prefix_rule():
    w = _small(q_len=4, seq_lens=[9, 40, 23])
    _, _, oc, _ = _run(w, causal=True)
    _, _, on, _ = _run(w, causal=False)
    ql = w.q_len
    for b in range(w.num_seqs):
        np.testing.assert_array_equal(oc[b * ql + ql - 1], on[b * ql + ql - 1])
        assert not np.allclose(oc[b * ql], on[b * ql])
    # causal row t == non-causal result over the prefix L - q_len + t + 1
    codes, desc = quantize_q(w.q_f32, w.num_seqs, ql, w.h_q, w.h_k, w.d)
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        for t in range(ql):
            pre = L - ql + t + 1
            lens = np.array([pre if i == b else 0 for i in range(w.num_seqs)])
            o2, _ = A.decode_attention(codes, desc, w.logical("k"), w.logical("v"), w.k_scale,
                                       w.v_scale, w.block_table, lens, num_seqs=w.num_seqs,
                                       q_len=ql, h_q=w.h_q, h_k=w.h_k, d=w.d,
                                       page_size=w.page_size, kv_format="fp8",
                                       softmax_scale=w.softmax_scale, causal=False)
            np.testing.assert_allclose(oc[b * ql + t], o2[b * ql + t], rtol=1e-12, atol=1e-15)


def test_gqa_heads_with_equal_q_give_equal_o():
    w = _small()
    h_r = w.h_r
    for g in range(w.h_k):
        for r in range(1, h_r):
            w.q_f32[:, g * h_r + r] = w.q_f32[:, g * h_r]
    _, _, out, _ = _run(w)
    for g in range(w.h_k):
        for r in range(1, h_r):
            np.testing.assert_array_equal(out[:, g * h_r + r], out[:, g * h_r])


def test_padding_requests_write_nothing():
    w = _small(seq_lens=[7, 0, 0])
    _, _, out, lse = _run(w)
    assert np.all(np.isfinite(out[0]))
    assert np.all(np.isnan(out[1:])) and np.all(np.isnan(lse[1:]))


def test_split_merge_equals_unsplit():
    rng = np.random.default_rng(4)
    for trial in range(20):
        L = int(rng.integers(1, 300))
        n_q, d = int(rng.integers(1, 9)), 16
        s = rng.standard_normal((n_q, L)) * rng.uniform(0.1, 8)
        v = rng.standard_normal((L, d))
        vis = np.ones((n_q, L), bool)
        if trial % 3 == 0:
            vis = np.arange(L)[None, :] <= (L - n_q + np.arange(n_q))[:, None]
            vis[:, 0] = True
        m, l, o = A.chunk_partial(s, vis, v, 0, L)
        cuts = np.sort(rng.integers(0, L + 1, size=int(rng.integers(0, 6))))
        bounds = [0] + list(cuts) + [L, L]  # includes empty chunks
        parts = [A.chunk_partial(s, vis, v, a, e) for a, e in zip(bounds[:-1], bounds[1:])]
        om, lse = A.merge_partials([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
        np.testing.assert_allclose(om, o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, m + np.log(l), rtol=1e-12)


def test_bf16_rounding():
    assert A.to_bf16(1.0) == 1.0
    assert A.to_bf16(1.0 + 2 ** -9) == 1.0  # tie -> even
    assert A.to_bf16(1.0 + 3 * 2 ** -9) == 1.0 + 2 ** -7  # tie -> even (up)
    assert A.to_bf16(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    assert A.to_bf16(-3.0) == -3.0
    import torch
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(A.to_bf16(x.astype(np.float64)), ref)


# ----------------------------------------------------------------------------
# the bf16-Q mode (Q left unquantized)
# ----------------------------------------------------------------------------
def _run_bf16(w, units=None):
    from oracle.qquant import pack_q_rows

    qv = pack_q_rows(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d)
    return A.decode_attention(
        qv, None, w.logical("k"), w.logical("v"), w.k_scale, w.v_scale, w.block_table,
        w.seq_lens, num_seqs=w.num_seqs, q_len=w.q_len, h_q=w.h_q, h_k=w.h_k, d=w.d,
        page_size=w.page_size, kv_format=w.kv_format, softmax_scale=w.softmax_scale,
        causal=w.causal, o_mul=w.o_mul, units=units, q_values=True)


def test_bf16_q_row_order():
    from oracle.qquant import pack_q_rows

    B, ql, hq, hk, d = 2, 3, 6, 2, 4
    q = np.zeros((B * ql, hq, d))
    for tok in range(B * ql):
        for h in range(hq):
            q[tok, h] = 1000 * tok + 10 * h + np.arange(d) * 0.1  # the value names its place
    packed = pack_q_rows(q, B, ql, hq, hk, d)
    hr = hq // hk
    for b in range(B):
        for g in range(hk):
            for t in range(ql):
                for r in range(hr):
                    assert np.array_equal(packed[b, g, t * hr + r], q[b * ql + t, g * hr + r])


def test_bf16_q_mode_equals_fp8_mode_on_representable_q():
    # Q set to its own dequantised e4m3 codes: both modes see the same values
    w = _small(q_len=2, seq_lens=[7, 40, 19])
    codes, desc = quantize_q(w.q_f32, w.num_seqs, w.q_len, w.h_q, w.h_k, w.d, w.q_mul)
    deq = F.e4m3_decode(codes) * desc[:, :, None, None]  # [B, h_k, n_q, d]
    hr = w.h_r
    q = np.zeros_like(w.q_f32, dtype=np.float64)
    for b in range(w.num_seqs):
        for g in range(w.h_k):
            for row in range(w.n_q):
                t, r = divmod(row, hr)
                q[b * w.q_len + t, g * hr + r] = deq[b, g, row]
    w.q_f32 = q
    out_fp8 = _run(w)[2]
    out_bf16, _ = _run_bf16(w)
    np.testing.assert_allclose(out_bf16, out_fp8, rtol=1e-12, atol=1e-14)


def test_bf16_q_mode_matches_brute_force():
    w = _small(q_len=2, seq_lens=[6, 30, 11], causal=True)
    out, _ = _run_bf16(w)
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        for g in range(w.h_k):
            kc, vc = A.gather_unit(w.logical("k"), w.logical("v"), w.block_table, b, g, L, w.page_size)
            k = F.e4m3_decode(kc) * A.descale_at(w.k_scale, b, g)
            v = F.e4m3_decode(vc) * A.descale_at(w.v_scale, b, g)
            for t in range(w.q_len):
                for r in range(w.h_r):
                    qrow = np.asarray(w.q_f32[b * w.q_len + t, g * w.h_r + r], dtype=np.float64)
                    logits, vals = [], []
                    for j in range(L):
                        if j <= L - w.q_len + t:  # causal
                            logits.append(w.softmax_scale * float(qrow @ k[j]))
                            vals.append(v[j])
                    mx = max(logits)
                    wts = [math.exp(s - mx) for s in logits]
                    want = sum(wt * vv for wt, vv in zip(wts, vals)) / sum(wts)
                    np.testing.assert_allclose(out[b * w.q_len + t, g * w.h_r + r], want, rtol=1e-10, atol=1e-12)
