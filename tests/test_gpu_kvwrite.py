"""GPU parity of the KV-cache write (mj_write_kv) against the oracle.

Bit-exact: every byte of both pools -- the written rows and everything the
write must leave alone (padding tokens' would-be rows, all other slots).
"""

import numpy as np
import pytest

import synth
from oracle import kvwrite as OW

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


def _fmt(c):
    return OW.KV_E4M3 if c.kv_format == "fp8" else OW.KV_E2M3


def run_gpu_write(c, status_word=False):
    import torch

    import paged_fp8_decode_gb300 as mj

    dev = "cuda"
    key = torch.from_numpy(c.key_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    val = torch.from_numpy(c.value_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    slots = torch.from_numpy(c.slots).to(dev)
    kp = torch.from_numpy(c.k_pool.copy()).to(dev)
    vp = torch.from_numpy(c.v_pool.copy()).to(dev)
    ks = torch.from_numpy(np.ascontiguousarray(c.k_scale)).to(dev)
    vs = torch.from_numpy(np.ascontiguousarray(c.v_scale)).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev) if status_word else None
    fmt = mj.MJ_KV_E4M3 if c.kv_format == "fp8" else mj.MJ_KV_E2M3
    mj.mj_write_kv(key, val, slots, kp, vp, c.kv_strides, c.page_size, c.num_pages, fmt, ks, vs,
                   scale_per_head=c.scale_per_head, status=st)
    torch.cuda.synchronize()
    return kp.cpu().numpy(), vp.cpu().numpy(), (int(st.item()) if st is not None else None)


def run_oracle_write(c):
    kp, vp = c.k_pool.copy(), c.v_pool.copy()
    OW.write_kv(c.key, c.value, kp, vp, c.slots, c.page_size, c.kv_strides, c.kv_strides, _fmt(c),
                c.k_scale, c.v_scale)
    return kp, vp


SMALL = [
    dict(name="fp8_head_hnd", num_tokens=301, num_pages=40, page_size=16, layout="HND", kv_format="fp8",
         scale_mode="head", pad_every=7, seed=41),
    dict(name="fp8_tensor_nhd", num_tokens=257, num_pages=9, page_size=64, layout="NHD", kv_format="fp8",
         scale_mode="tensor", pad_every=5, seed=42),
    dict(name="fp8_one_token", num_tokens=1, num_pages=3, page_size=32, layout="HND", kv_format="fp8",
         scale_mode="head", seed=43),
    dict(name="e2m3_hnd", num_tokens=300, num_pages=5, page_size=128, layout="HND", kv_format="e2m3",
         outlier_channels=4, pad_every=9, seed=44),
    dict(name="e2m3_nhd", num_tokens=97, num_pages=12, page_size=16, layout="NHD", kv_format="e2m3",
         outlier_channels=4, pad_every=3, seed=45),
    # head size 256: 256-byte e4m3 rows, 192-byte packed e2m3 rows
    dict(name="fp8_d256_nhd", num_tokens=211, d=256, num_pages=30, page_size=16, layout="NHD", kv_format="fp8",
         scale_mode="head", pad_every=6, seed=50),
    dict(name="e2m3_d256_hnd", num_tokens=150, d=256, num_pages=4, page_size=64, layout="HND", kv_format="e2m3",
         outlier_channels=4, pad_every=8, seed=51),
]


@pytest.mark.parametrize("spec", SMALL, ids=[s["name"] for s in SMALL])
def test_write_bit_exact(spec):
    c = synth.kv_write_case(**spec)
    gk, gv, _ = run_gpu_write(c)
    ok, ov = run_oracle_write(c)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_write_saturates_and_keeps_signs():
    # rows scaled far past the format's range and tiny ones: saturation, signed zeros
    c = synth.kv_write_case(name="sat", num_tokens=64, num_pages=4, page_size=16, kv_format="fp8",
                            scale_mode="tensor", seed=46)
    c.k_scale = np.array([1e-4], np.float32)  # |x| / 1e-4 >> 448
    c.v_scale = np.array([1e6], np.float32)   # |x| / 1e6 rounds to (signed) zero
    gk, gv, _ = run_gpu_write(c)
    ok, ov = run_oracle_write(c)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    c2 = synth.kv_write_case(name="sat6", num_tokens=64, num_pages=4, page_size=16, kv_format="e2m3", seed=47)
    c2.k_scale = np.full_like(c2.k_scale, 1e-3)
    c2.v_scale = np.full_like(c2.v_scale, 1e5)
    gk, gv, _ = run_gpu_write(c2)
    ok, ov = run_oracle_write(c2)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_out_of_range_slot_is_skipped_and_reported():
    c = synth.kv_write_case(name="oob", num_tokens=20, num_pages=4, page_size=16, kv_format="fp8", seed=48)
    c.slots[5] = c.num_pages * c.page_size  # one past the pool
    gk, gv, status = run_gpu_write(c, status_word=True)
    c.slots[5] = -1  # the oracle's view: that token writes nothing
    ok, ov = run_oracle_write(c)
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)
    assert status == 1


@pytest.mark.parametrize("kv_format", ["fp8", "e2m3"])
def test_write_full_size_sampled(kv_format):
    """Bulk writes at the benchmark pools' sizes: every token of the Qwen3-8B
    decode batch (64 x 4096 tokens, 8 KV heads, page 16), and 65536 tokens
    into the fp6 configuration's pool (8192 pages of 128 tokens). The rows of
    4096 sampled tokens and a sample of untouched slots are checked."""
    import torch

    import paged_fp8_decode_gb300 as mj

    if kv_format == "fp8":
        spec = dict(num_tokens=64 * 4096, num_pages=64 * 256 + 64, page_size=16, kv_format="fp8",
                    scale_mode="head", pad_every=1000)
    else:
        spec = dict(num_tokens=65536, num_pages=8192, page_size=128, kv_format="e2m3",
                    outlier_channels=4, pad_every=1000)
    c = synth.kv_write_case(name="full_" + kv_format, seed=49, **spec)
    gk, gv, status = run_gpu_write(c, status_word=True)
    assert status == 0
    rng = np.random.default_rng(7)
    toks = rng.choice(c.key.shape[0], 4096, replace=False)
    fmt = _fmt(c)
    kq = OW.quantize_rows(c.key[toks], c.k_scale, fmt)
    vq = OW.quantize_rows(c.value[toks], c.v_scale, fmt)
    rb = OW.row_bytes(128, fmt)
    sp, stt, sh = c.kv_strides
    for i, t in enumerate(toks):
        s = int(c.slots[t])
        if s < 0:
            continue
        for g in range(c.key.shape[1]):
            off = (s // c.page_size) * sp + (s % c.page_size) * stt + g * sh
            assert np.array_equal(gk[off:off + rb], kq[i, g]) and np.array_equal(gv[off:off + rb], vq[i, g])
    # slots no token maps to keep their bytes
    used = np.zeros(c.num_pages * c.page_size, dtype=bool)
    used[c.slots[c.slots >= 0]] = True
    free = np.flatnonzero(~used)[:64 * c.page_size]
    for s in free[:: max(1, len(free) // 256)]:
        for g in range(c.key.shape[1]):
            off = (s // c.page_size) * sp + (s % c.page_size) * stt + g * sh
            assert np.array_equal(gk[off:off + rb], c.k_pool[off:off + rb])
    del torch, mj


@pytest.mark.parametrize("scale_bits", [0x3F800000, 0x40E00000, 0x40400000, 0x3DCCCCCD, 0x3FFFFFFF, 0x42EEEEEF,
                                        0x35800000, 0x4493E000, 0x3F7FFFFF, 0x3C23D70A])
def test_e4m3_write_every_bf16_value(scale_bits):
    """Every finite bf16 value through the e4m3 write with one scale: the
    codes must be those of the IEEE float32 quotient, rounded to nearest even
    and saturated (the oracle). The scales include 1, 7 (the hand-worked tie
    case of the Q quantization), 3, 0.1, the largest and the smallest
    significands (0x3FFFFFFF, 0x3F7FFFFF), and tiny and large values."""
    bits = np.arange(65536, dtype=np.uint32)
    finite = (bits & 0x7F80) != 0x7F80
    vals = bits[finite].astype(np.uint16)
    n = -(-vals.size // 128) * 128
    row = np.zeros(n, dtype=np.uint16)
    row[: vals.size] = vals
    kb = row.reshape(-1, 1, 128)
    vb = kb[::-1].copy()
    T = kb.shape[0]
    scale = np.array([scale_bits], dtype=np.uint32).view(np.float32)
    c = synth.WriteCase(name=f"every_bf16_{scale_bits:08x}", key_bf16=kb, value_bf16=vb,
                        key=(kb.astype(np.uint32) << 16).view(np.float32), value=(vb.astype(np.uint32) << 16).view(np.float32),
                        slots=np.arange(T, dtype=np.int64), k_pool=np.zeros(T * 128, np.uint8),
                        v_pool=np.zeros(T * 128, np.uint8), kv_strides=(16 * 128, 128, 16 * 128), page_size=16,
                        num_pages=T // 16 + 1, kv_format="fp8", k_scale=scale, v_scale=scale, scale_per_head=False)
    c.k_pool = np.zeros(c.num_pages * 16 * 128, np.uint8)
    c.v_pool = np.zeros(c.num_pages * 16 * 128, np.uint8)
    kp, vp, _ = run_gpu_write(c)
    okp, ovp = run_oracle_write(c)
    assert np.array_equal(kp, okp) and np.array_equal(vp, ovp)
