"""The C ABI on the host: the library loads, exports every declared symbol,
validates arguments before touching the device, and plans bit-identically
to the oracle. No GPU is needed (no call here reaches a kernel launch)."""

import ctypes
import os
import re

import numpy as np
import pytest

import paged_fp8_decode_gb300 as mj
from oracle import plan as OP

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_fp8_decode_gb300.build import build

    build()
    return mj.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "mj.h")).read()
    return re.findall(r"MJ_API\s+[\w\s\*]+?\b(mj_\w+)\s*\(", src)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11
    assert set(names) == set(mj.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.mj_status_string(code)
    assert mj.mj_version() == 100


def test_tile_width_and_slots_match_oracle(lib):
    for n_q in range(1, 80):
        assert mj.mj_tile_width(n_q) == OP.tile_width(n_q, True)
    for sm, cps, h_k, ql, h_q in [(152, 2, 8, 1, 32), (152, 4, 8, 4, 32), (20, 2, 8, 1, 32), (152, 2, 8, 1, 64),
                                  (152, 1, 2, 3, 32)]:
        assert mj.mj_slots(sm, cps, h_k, ql, h_q) == OP.slots(sm, cps, h_k, OP.n_tiles(ql, h_q // h_k))


@pytest.mark.parametrize("seed", range(60))
def test_plan_bit_identical_to_oracle(lib, seed):
    rng = np.random.default_rng(100 + seed)
    num_seqs = int(rng.integers(0, 40))
    lens = rng.integers(0, 200000 if seed % 3 == 0 else 5000, size=num_seqs).astype(np.int32)
    if num_seqs and seed % 4 == 0:
        lens[-min(3, num_seqs):] = 0
    h_k = int(rng.choice([1, 2, 4, 8]))
    h_q = h_k * int(rng.choice([1, 4, 8]))
    q_len = int(rng.integers(1, 6))
    sm, cps = int(rng.choice([20, 148, 152])), int(rng.integers(1, 5))
    max_splits = int(rng.choice([1, 2, 16, 64, 128]))
    margin = int(rng.integers(0, 5))
    s = OP.slots(sm, cps, h_k, OP.n_tiles(q_len, h_q // h_k))
    pad_to = max(s, num_seqs) + int(rng.integers(0, 3))
    ref = OP.plan_split_kv(lens, num_seqs, q_len, h_q, h_k, sm, cps, max_splits, margin, pad_to)
    got = mj.mj_plan_split_kv(lens, num_seqs, q_len, h_q, h_k, sm, cps, max_splits, margin, pad_to)
    assert got["slots"] == ref.slots
    assert got["with_reduction"] == ref.with_reduction
    assert got["chunk_tiles"] == ref.chunk_tiles
    assert np.array_equal(got["work"], np.array(ref.work, dtype=np.int32).reshape(pad_to, 4))
    assert list(got["n_splits"][:num_seqs]) == ref.n_splits


def test_plan_rejects_small_pad_to(lib):
    with pytest.raises(mj.MjError) as e:
        mj.mj_plan_split_kv(np.full(10, 100, np.int32), 10, 1, 32, 8, 152, 2, 16, 0, 5)
    assert e.value.status == mj.MJ_ERR_CAPACITY


def _valid_args():
    """A well-formed argument struct with fake (never dereferenced) 256-byte
    aligned addresses; each test breaks one thing and expects the host-side
    check to reject it before any launch."""
    a = mj.mj_decode_args()
    base = 1 << 40
    a.num_seqs, a.q_len, a.h_q, a.h_k, a.d, a.causal, a.softmax_scale = 2, 1, 8, 2, 128, 1, 0.088
    a.q_codes, a.q_descale = base, base + 0x1000
    a.kv_format, a.page_size, a.num_pages = 0, 16, 10
    a.k_cache, a.v_cache = base + 0x10000, base + 0x20000
    a.k_stride_page, a.k_stride_token, a.k_stride_head = 4096, 128, 2048
    a.v_stride_page, a.v_stride_token, a.v_stride_head = 4096, 128, 2048
    a.k_descale, a.v_descale = base + 0x2000, base + 0x2100
    a.descale_seq_stride, a.descale_head_stride = 0, 0
    a.block_table, a.block_table_stride, a.seq_lens = base + 0x3000, 8, base + 0x3100
    a.work, a.n_splits, a.num_work = base + 0x4000, base + 0x4100, 2
    a.with_reduction, a.chunk_tiles, a.max_splits, a.part_seqs = 0, 1, 16, 2
    a.out, a.out_tok_stride, a.out_head_stride = base + 0x5000, 1024, 128
    a.workspace, a.workspace_bytes = base + 0x8000, 256
    return a


@pytest.mark.parametrize("field,value,status", [
    ("d", 64, mj.MJ_ERR_UNSUPPORTED),
    ("d", 192, mj.MJ_ERR_UNSUPPORTED),
    ("d", 512, mj.MJ_ERR_UNSUPPORTED),
    ("page_size", 8, mj.MJ_ERR_UNSUPPORTED),
    ("kv_format", 7, mj.MJ_ERR_UNSUPPORTED),
    ("kv_format", 4, mj.MJ_ERR_UNSUPPORTED),
    ("h_q", 9, mj.MJ_ERR_INVALID_ARG),
    ("q_len", 0, mj.MJ_ERR_INVALID_ARG),
    ("q_codes", None, mj.MJ_ERR_INVALID_ARG),
    ("block_table", None, mj.MJ_ERR_INVALID_ARG),
    ("workspace", None, mj.MJ_ERR_INVALID_ARG),
    ("q_codes", (1 << 40) + 8, mj.MJ_ERR_ALIGNMENT),
    ("out", (1 << 40) + 0x5002, mj.MJ_ERR_ALIGNMENT),
    ("k_stride_token", 130, mj.MJ_ERR_ALIGNMENT),
    ("out_head_stride", 130, mj.MJ_ERR_ALIGNMENT),
    ("softmax_scale", 0.0, mj.MJ_ERR_INVALID_ARG),
    ("workspace_bytes", 16, mj.MJ_ERR_CAPACITY),
    ("impl", 9, mj.MJ_ERR_INVALID_ARG),
    ("out_dtype", 2, mj.MJ_ERR_UNSUPPORTED),
    ("q_mode", 3, mj.MJ_ERR_UNSUPPORTED),
])
def test_decode_args_rejected_on_host(lib, field, value, status):
    a = _valid_args()
    setattr(a, field, value)
    assert lib.mj_decode_attention(ctypes.byref(a), None) == status
    assert lib.mj_merge_lse(ctypes.byref(a), None) == status


@pytest.mark.parametrize("kv_format", [mj.MJ_KV_E2M3, mj.MJ_KV_E3M2, mj.MJ_KV_E2M1])
def test_packed_formats_need_32_byte_kv_alignment(lib, kv_format):
    a = _valid_args()
    a.kv_format = kv_format
    a.k_cache = (1 << 40) + 0x10010  # 16- but not 32-byte aligned
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_ALIGNMENT


@pytest.mark.parametrize("kv_format", [mj.MJ_KV_E3M2, mj.MJ_KV_E2M1])
def test_packed_formats_refuse_bf16_q(lib, kv_format):
    a = _valid_args()
    a.kv_format, a.q_mode, a.q_bf16 = kv_format, mj.MJ_Q_BF16, 1 << 40
    a.q_tok_stride, a.q_head_stride = 1024, 128
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_UNSUPPORTED


def test_reduction_needs_a_large_enough_workspace(lib):
    a = _valid_args()
    a.with_reduction = 1
    need = mj.mj_workspace_size(a.part_seqs, a.max_splits, a.q_len, a.h_q, a.h_k)
    a.workspace_bytes = need - 4
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_CAPACITY
    a.part_seqs = 1  # fewer than num_seqs
    a.workspace_bytes = need
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_INVALID_ARG


def test_workspace_size_formula(lib):
    n = mj.mj_workspace_size(38, 64, 1, 32, 8)
    assert n == 256 + 38 * 64 * 8 * 4 * (128 + 2) * 4
    n = mj.mj_workspace_size(38, 64, 1, 16, 8, 256)
    assert n == 256 + 38 * 64 * 8 * 2 * (256 + 2) * 4
    with pytest.raises(mj.MjError):
        mj.mj_workspace_size(38, 64, 1, 16, 8, 192)


def test_head_size_256_passes_the_host_checks(lib):
    """D = 256 is accepted: with no work rows the call validates and returns
    MJ_OK without launching anything (no device is touched)."""
    a = _valid_args()
    a.d = 256
    a.k_stride_page, a.k_stride_token, a.k_stride_head = 8192, 256, 4096
    a.v_stride_page, a.v_stride_token, a.v_stride_head = 8192, 256, 4096
    a.out_tok_stride, a.out_head_stride = 2048, 256
    a.num_work, a.impl = 0, 1  # nothing to launch; the CUDA-core path needs no driver query
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_OK
    assert lib.mj_merge_lse(ctypes.byref(a), None) == mj.MJ_OK  # no reduction: nothing to merge


def test_quantize_rejections(lib):
    f = lib.mj_quantize_q
    base = 1 << 40
    assert f(base, 4096, 128, 2, 1, 32, 8, 64, None, base, base, None) == mj.MJ_ERR_UNSUPPORTED
    assert f(base, 8192, 256, 2, 1, 32, 8, 384, None, base, base, None) == mj.MJ_ERR_UNSUPPORTED
    assert f(base, 4096, 128, 2, 1, 30, 8, 128, None, base, base, None) == mj.MJ_ERR_INVALID_ARG
    assert f(None, 4096, 128, 2, 1, 32, 8, 128, None, base, base, None) == mj.MJ_ERR_INVALID_ARG
    assert f(base + 2, 4096, 128, 2, 1, 32, 8, 128, None, base, base, None) == mj.MJ_ERR_ALIGNMENT
    assert f(base, 4096, 128, 0, 1, 32, 8, 128, None, None, None, None) == mj.MJ_OK  # empty batch: no-op


# ----------------------------------------------------------------------------
# mj_write_kv: host-side validation (every case is rejected before a launch)
# ----------------------------------------------------------------------------
def _valid_write_args():
    base = 1 << 40  # never dereferenced: every case below fails validation first
    a = mj.mj_write_kv_args()
    a.num_tokens, a.h_k, a.d = 4, 2, 128
    a.key, a.value = base, base + 0x1000
    a.key_tok_stride, a.key_head_stride = 256, 128
    a.value_tok_stride, a.value_head_stride = 256, 128
    a.slot_mapping = base + 0x2000
    a.kv_format, a.page_size, a.num_pages = 0, 16, 4
    a.k_cache, a.v_cache = base + 0x10000, base + 0x20000
    a.k_stride_page, a.k_stride_token, a.k_stride_head = 4096, 128, 2048
    a.v_stride_page, a.v_stride_token, a.v_stride_head = 4096, 128, 2048
    a.k_scale, a.v_scale, a.scale_per_head = base + 0x3000, base + 0x3100, 1
    return a


@pytest.mark.parametrize("field,value,status", [
    ("d", 64, mj.MJ_ERR_UNSUPPORTED),
    ("kv_format", 4, mj.MJ_ERR_UNSUPPORTED),
    ("page_size", 48, mj.MJ_ERR_UNSUPPORTED),
    ("num_tokens", -1, mj.MJ_ERR_INVALID_ARG),
    ("h_k", 0, mj.MJ_ERR_INVALID_ARG),
    ("key", None, mj.MJ_ERR_INVALID_ARG),
    ("slot_mapping", None, mj.MJ_ERR_INVALID_ARG),
    ("v_scale", None, mj.MJ_ERR_INVALID_ARG),
    ("key", (1 << 40) + 8, mj.MJ_ERR_ALIGNMENT),
    ("slot_mapping", (1 << 40) + 0x2004, mj.MJ_ERR_ALIGNMENT),
    ("key_head_stride", 132, mj.MJ_ERR_ALIGNMENT),
    ("k_stride_token", 120, mj.MJ_ERR_ALIGNMENT),
    ("v_stride_page", -16, mj.MJ_ERR_INVALID_ARG),
    ("k_scale", (1 << 40) + 0x3004, mj.MJ_ERR_ALIGNMENT),
])
def test_write_kv_args_rejected_on_host(lib, field, value, status):
    a = _valid_write_args()
    setattr(a, field, value)
    assert lib.mj_write_kv(ctypes.byref(a), None) == status


def test_write_kv_nothing_to_do(lib):
    a = _valid_write_args()
    a.num_tokens = 0
    a.key = a.value = a.slot_mapping = None  # nothing is read when there are no tokens
    assert lib.mj_write_kv(ctypes.byref(a), None) == mj.MJ_OK


def test_bf16_q_mode_host_checks(lib):
    a = _valid_args()
    a.q_mode, a.q_bf16 = mj.MJ_Q_BF16, None
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_INVALID_ARG
    a.q_bf16, a.q_tok_stride, a.q_head_stride = (1 << 40) + 0x9000, 4096, 132
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_ALIGNMENT
    a.q_head_stride = 128
    a.kv_format = mj.MJ_KV_E2M3  # e2m3 KV is fp8-Q only
    assert lib.mj_decode_attention(ctypes.byref(a), None) == mj.MJ_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(lib):
    """No CPU or library fallback: without libmj.so the binding raises."""
    saved = mj._lib
    try:
        mj._lib = None
        with pytest.raises(RuntimeError, match="no CPU or library fallback"):
            mj.load_library(os.path.join(ROOT, "no_such_dir", "libmj.so"))
    finally:
        mj._lib = saved


def test_product_path_never_imports_the_oracle():
    """The package (binding, step helpers, build, CUDA sources) names no
    oracle module, and importing it loads none."""
    pkg = os.path.join(ROOT, "paged_fp8_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b|#include\s+[<\"].*oracle", src, re.M), f
    import subprocess
    import sys

    code = ("import sys, paged_fp8_decode_gb300, paged_fp8_decode_gb300.step, paged_fp8_decode_gb300.build; "
            "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "[]"


def test_noalloc_rejects_oversized_plans_on_the_host(lib):
    """The allocation-free call checks its fixed scratch before touching the
    device: a plan whose partials exceed it is refused with MJ_ERR_CAPACITY."""
    a = mj.mj_decode_args()
    a.num_seqs, a.q_len, a.h_q, a.h_k, a.d = 8, 1, 32, 8, 128
    a.with_reduction, a.max_splits, a.part_seqs = 1, 64, 1000
    need = mj.mj_workspace_size(1000, 64, 1, 32, 8, 128)
    assert need > mj.NOALLOC_SCRATCH_BYTES
    assert lib.mj_decode_attention_noalloc(ctypes.byref(a), None) == mj.MJ_ERR_CAPACITY
    assert lib.mj_decode_attention_noalloc(None, None) == mj.MJ_ERR_INVALID_ARG


def test_wrappers_refuse_host_tensors_for_device_pointers(lib):
    """A CPU tensor's address means nothing to a kernel: the binding refuses it
    before calling into the library."""
    torch = pytest.importorskip("torch")
    q = torch.zeros(2, 32, 128, dtype=torch.bfloat16)
    codes = torch.zeros(2, 8, 4, 128, dtype=torch.uint8)
    desc = torch.zeros(2, 8, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mj.mj_quantize_q(q, 2, 1, 8, codes, desc)
    key = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    pool = torch.zeros(4 * 16 * 2 * 128, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mj.mj_write_kv(key, key, torch.zeros(4, dtype=torch.int64), pool, pool, (4096, 128, 2048), 16, 4, 0,
                       torch.ones(1), torch.ones(1))


def test_plan_refuses_buffers_it_would_overrun(lib):
    lens = np.full(8, 1000, np.int32)
    with pytest.raises(ValueError, match="num_seqs"):
        mj.mj_plan_split_kv(lens[:5], 8, 1, 32, 8, 152, 2, 16, 0, 64)
    with pytest.raises(ValueError, match="work_out"):
        mj.mj_plan_split_kv(lens, 8, 1, 32, 8, 152, 2, 16, 0, 64, work_out=np.zeros((63, 4), np.int32))
    with pytest.raises(ValueError, match="work_out"):
        mj.mj_plan_split_kv(lens, 8, 1, 32, 8, 152, 2, 16, 0, 64, work_out=np.zeros((64, 4), np.int64))
    with pytest.raises(ValueError, match="n_splits_out"):
        mj.mj_plan_split_kv(lens, 8, 1, 32, 8, 152, 2, 16, 0, 64, n_splits_out=np.zeros(7, np.int32))
    got = mj.mj_plan_split_kv(lens, 8, 1, 32, 8, 152, 2, 16, 0, 64, work_out=np.zeros((64, 4), np.int32),
                              n_splits_out=np.zeros(8, np.int32))
    assert got["with_reduction"] and sum(got["n_splits"]) <= got["slots"]


def test_plan_upload_validates_on_the_host(lib):
    """mj_plan_upload copies nothing for an empty plan and refuses missing
    or misaligned buffers before it enqueues anything."""
    base = 1 << 40  # never dereferenced: every case below returns before a copy
    f = lib.mj_plan_upload
    assert f(None, None, None, None, 0, 0, None) == mj.MJ_OK
    assert f(None, base, base, base, 64, 8, None) == mj.MJ_ERR_INVALID_ARG  # no host work buffer
    assert f(base, None, base, base, 64, 8, None) == mj.MJ_ERR_INVALID_ARG  # no host n_splits
    assert f(base, base, base, None, 64, 8, None) == mj.MJ_ERR_INVALID_ARG  # no device n_splits
    assert f(base, base, base + 4, base, 64, 8, None) == mj.MJ_ERR_ALIGNMENT
    assert f(base, base, base, base, -1, 8, None) == mj.MJ_ERR_INVALID_ARG


def test_decode_kernel_query(lib):
    """mj_decode_kernel validates like mj_decode_attention and reports the
    CUDA-core kernel when asked for it, without touching a device."""
    a = _valid_args()
    a.impl = mj.MJ_IMPL_SIMT
    v = ctypes.c_int(-1)
    assert lib.mj_decode_kernel(ctypes.byref(a), ctypes.byref(v)) == mj.MJ_OK and v.value == mj.MJ_IMPL_SIMT
    a.page_size = 24
    assert lib.mj_decode_kernel(ctypes.byref(a), ctypes.byref(v)) == mj.MJ_ERR_UNSUPPORTED
    assert lib.mj_decode_kernel(ctypes.byref(a), None) == mj.MJ_ERR_INVALID_ARG
