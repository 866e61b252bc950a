"""paged_fp8_decode_gb300 — Python binding of libmj (include/mj.h).

Paged decode attention over an e4m3 or packed e2m3 / e3m2 / e2m1 KV cache on GB300
(sm_103a). Every step of the path runs in the CUDA library; this module only
marshals arguments: torch tensors become device pointers and strides, torch
streams become ``cudaStream_t`` handles. The function names are the C names.

The library is built in-tree by :func:`paged_fp8_decode_gb300.build.build`.
There is no fallback: if ``libmj.so`` is missing or fails to load, every call
raises.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmj.so")

MJ_OK = 0
MJ_ERR_INVALID_ARG = -1
MJ_ERR_UNSUPPORTED = -2
MJ_ERR_ALIGNMENT = -3
MJ_ERR_CAPACITY = -4
MJ_ERR_CUDA = -5
MJ_ERR_DEVICE_CHECK = -6

MJ_KV_E4M3 = 0
MJ_KV_E2M3 = 1
MJ_KV_E3M2 = 2
MJ_KV_E2M1 = 3
KV_FORMATS = {"fp8": MJ_KV_E4M3, "e2m3": MJ_KV_E2M3, "e3m2": MJ_KV_E3M2, "e2m1": MJ_KV_E2M1}

MJ_Q_FP8 = 0
MJ_Q_BF16 = 1
MJ_Q_FP8_FUSED = 2

MJ_OUT_BF16 = 0
MJ_OUT_F16 = 1

MJ_IMPL_AUTO = 0
MJ_IMPL_SIMT = 1
MJ_IMPL_TCGEN05 = 2

KV_TILE = 128

# every symbol include/mj.h declares
EXPORTS = (
    "mj_status_string", "mj_version", "mj_tile_width", "mj_slots", "mj_plan_split_kv",
    "mj_quantize_q", "mj_workspace_size", "mj_workspace_init", "mj_workspace_status",
    "mj_decode_attention", "mj_merge_lse", "mj_decode_attention_noalloc", "mj_noalloc_status", "mj_write_kv",
    "mj_plan_upload", "mj_decode_kernel",
)

NOALLOC_SCRATCH_BYTES = 16 << 20


class MjError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} ({status})")
        self.status = status


class mj_decode_args(ctypes.Structure):
    """ctypes mirror of ``struct mj_decode_args`` (field order and types
    must match include/mj.h)."""

    _fields_ = [
        ("num_seqs", ctypes.c_int), ("q_len", ctypes.c_int), ("h_q", ctypes.c_int), ("h_k", ctypes.c_int),
        ("d", ctypes.c_int), ("causal", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("q_codes", ctypes.c_void_p), ("q_descale", ctypes.c_void_p),
        ("kv_format", ctypes.c_int), ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int64),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_stride_page", ctypes.c_int64), ("k_stride_token", ctypes.c_int64), ("k_stride_head", ctypes.c_int64),
        ("v_stride_page", ctypes.c_int64), ("v_stride_token", ctypes.c_int64), ("v_stride_head", ctypes.c_int64),
        ("k_descale", ctypes.c_void_p), ("v_descale", ctypes.c_void_p),
        ("descale_seq_stride", ctypes.c_int64), ("descale_head_stride", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int64), ("seq_lens", ctypes.c_void_p),
        ("work", ctypes.c_void_p), ("n_splits", ctypes.c_void_p), ("num_work", ctypes.c_int),
        ("with_reduction", ctypes.c_int), ("chunk_tiles", ctypes.c_int), ("max_splits", ctypes.c_int),
        ("part_seqs", ctypes.c_int),
        ("o_mul", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("out_tok_stride", ctypes.c_int64), ("out_head_stride", ctypes.c_int64), ("lse", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("impl", ctypes.c_int), ("kv_stages", ctypes.c_int), ("evict_first", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("q_mode", ctypes.c_int), ("q_bf16", ctypes.c_void_p),
        ("q_tok_stride", ctypes.c_int64), ("q_head_stride", ctypes.c_int64), ("q_mul", ctypes.c_void_p),
    ]


class mj_write_kv_args(ctypes.Structure):
    """ctypes mirror of ``struct mj_write_kv_args`` (include/mj.h)."""

    _fields_ = [
        ("num_tokens", ctypes.c_int), ("h_k", ctypes.c_int), ("d", ctypes.c_int),
        ("key", ctypes.c_void_p), ("value", ctypes.c_void_p),
        ("key_tok_stride", ctypes.c_int64), ("key_head_stride", ctypes.c_int64),
        ("value_tok_stride", ctypes.c_int64), ("value_head_stride", ctypes.c_int64),
        ("slot_mapping", ctypes.c_void_p),
        ("kv_format", ctypes.c_int), ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int64),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_stride_page", ctypes.c_int64), ("k_stride_token", ctypes.c_int64), ("k_stride_head", ctypes.c_int64),
        ("v_stride_page", ctypes.c_int64), ("v_stride_token", ctypes.c_int64), ("v_stride_head", ctypes.c_int64),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("scale_per_head", ctypes.c_int),
        ("status", ctypes.c_void_p),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmj.so (once). Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m paged_fp8_decode_gb300.build` "
                           "(the decode path has no CPU or library fallback)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.mj_status_string.restype = ctypes.c_char_p
    lib.mj_status_string.argtypes = [i32]
    lib.mj_version.argtypes = []
    lib.mj_tile_width.argtypes = [i32]
    lib.mj_slots.argtypes = [i32, i32, i32, i32, i32]
    lib.mj_plan_split_kv.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp,
                                     ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.mj_quantize_q.argtypes = [vp, i64, i64, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.mj_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.mj_workspace_init.argtypes = [vp, sz, vp]
    lib.mj_workspace_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.mj_decode_attention.argtypes = [ctypes.POINTER(mj_decode_args), vp]
    lib.mj_merge_lse.argtypes = [ctypes.POINTER(mj_decode_args), vp]
    lib.mj_decode_attention_noalloc.argtypes = [ctypes.POINTER(mj_decode_args), vp]
    lib.mj_noalloc_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.mj_plan_upload.argtypes = [vp, vp, vp, vp, i32, i32, vp]
    lib.mj_decode_kernel.argtypes = [ctypes.POINTER(mj_decode_args), ctypes.POINTER(ctypes.c_int)]
    lib.mj_write_kv.argtypes = [ctypes.POINTER(mj_write_kv_args), vp]
    _lib = lib
    return lib


def _check(fn: str, status: int) -> int:
    if status != MJ_OK:
        text = load_library().mj_status_string(status).decode()
        raise MjError(fn, status, text)
    return status


def _ptr(t) -> int | None:
    """Device pointer of a CUDA tensor (None -> NULL). A tensor in host memory
    is refused: its address handed to a kernel would fault, or on a host the
    GPU can address, silently read the wrong memory."""
    if t is None:
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"expected a CUDA tensor for a device pointer, got {getattr(t, 'device', type(t).__name__)}")
    return int(t.data_ptr())


def _host_int32(a, n: int, what: str) -> int:
    """Address of a contiguous int32 host buffer of at least ``n`` elements
    (numpy array or CPU tensor); anything smaller would be overrun."""
    import numpy as np

    if isinstance(a, np.ndarray):
        ok = a.dtype == np.int32 and a.flags.c_contiguous and a.size >= n
        addr = a.ctypes.data
    else:
        import torch

        ok = (not a.is_cuda) and a.dtype == torch.int32 and a.is_contiguous() and a.numel() >= n
        addr = int(a.data_ptr())
    if not ok:
        raise ValueError(f"{what}: need a contiguous int32 host buffer of at least {n} elements")
    return addr


def _stream(stream) -> int | None:
    """cudaStream_t of a torch.cuda.Stream (None -> the current stream)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) or None


# ----------------------------------------------------------------------------
# the C calls
# ----------------------------------------------------------------------------
def mj_version() -> int:
    return load_library().mj_version()


def mj_tile_width(n_q: int) -> int:
    return load_library().mj_tile_width(int(n_q))


def mj_slots(sm_count: int, ctas_per_sm: int, h_k: int, q_len: int, h_q: int) -> int:
    return load_library().mj_slots(int(sm_count), int(ctas_per_sm), int(h_k), int(q_len), int(h_q))


def mj_plan_split_kv(seq_lens_host, num_seqs: int, q_len: int, h_q: int, h_k: int, sm_count: int,
                     ctas_per_sm: int, max_splits: int, margin: int, pad_to: int, work_out=None,
                     n_splits_out=None) -> dict:
    """Host plan. ``seq_lens_host``: int32 numpy array / CPU tensor.
    ``work_out`` / ``n_splits_out``: optional int32 host buffers (numpy or
    pinned CPU tensors) to write into; otherwise numpy arrays are returned."""
    import numpy as np

    lib = load_library()
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32).reshape(-1)[:num_seqs])
    if lens.size != num_seqs:
        raise ValueError(f"seq_lens_host holds {lens.size} lengths, num_seqs is {num_seqs}")
    if work_out is None:
        work_out = np.zeros((max(0, pad_to), 4), dtype=np.int32)
    if n_splits_out is None:
        n_splits_out = np.zeros(max(1, num_seqs), dtype=np.int32)
    work_addr = _host_int32(work_out, 4 * max(0, pad_to), "work_out")
    nsplit_addr = _host_int32(n_splits_out, num_seqs, "n_splits_out")

    chunk, red, slots = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check("mj_plan_split_kv", lib.mj_plan_split_kv(
        lens.ctypes.data if num_seqs else None, num_seqs, q_len, h_q, h_k, sm_count, ctas_per_sm,
        max_splits, margin, pad_to, work_addr, nsplit_addr, ctypes.byref(chunk),
        ctypes.byref(red), ctypes.byref(slots)))
    return {"work": work_out, "n_splits": n_splits_out, "chunk_tiles": chunk.value,
            "with_reduction": bool(red.value), "slots": slots.value, "num_work": pad_to}


def mj_plan_upload(work_host, n_splits_host, work_dev, n_splits_dev, pad_to: int, num_seqs: int, stream=None):
    """Copy a host plan (pinned int32 CPU tensors) into the fixed device plan
    buffers on ``stream`` (one asynchronous copy per buffer)."""
    import torch

    for t, n, what in ((work_dev, 4 * pad_to, "work_dev"), (n_splits_dev, num_seqs, "n_splits_dev")):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() < n:
            raise ValueError(f"{what}: a contiguous int32 device buffer of at least {n} elements is required")
    _check("mj_plan_upload", load_library().mj_plan_upload(
        _host_int32(work_host, 4 * pad_to, "work_host"), _host_int32(n_splits_host, num_seqs, "n_splits_host"),
        _ptr(work_dev), _ptr(n_splits_dev), pad_to, num_seqs, _stream(stream)))


def mj_decode_kernel(args: mj_decode_args) -> int:
    """The kernel mj_decode_attention runs for ``args``: MJ_IMPL_TCGEN05 or MJ_IMPL_SIMT."""
    v = ctypes.c_int(0)
    _check("mj_decode_kernel", load_library().mj_decode_kernel(ctypes.byref(args), ctypes.byref(v)))
    return v.value


def mj_quantize_q(q, num_seqs: int, q_len: int, h_k: int, q_codes, q_descale, q_mul=None, stream=None):
    """``q``: bf16 tensor ``[>= num_seqs*q_len, h_q, d]`` (any token/head
    strides, channel stride 1)."""
    h_q, d = int(q.shape[1]), int(q.shape[2])
    assert q.stride(2) == 1
    _check("mj_quantize_q", load_library().mj_quantize_q(
        _ptr(q), q.stride(0), q.stride(1), num_seqs, q_len, h_q, h_k, d, _ptr(q_mul), _ptr(q_codes),
        _ptr(q_descale), _stream(stream)))


def mj_workspace_size(part_seqs: int, max_splits: int, max_q_len: int, h_q: int, h_k: int, d: int = 128) -> int:
    n = ctypes.c_size_t(0)
    _check("mj_workspace_size", load_library().mj_workspace_size(part_seqs, max_splits, max_q_len, h_q, h_k, d,
                                                                 ctypes.byref(n)))
    return n.value


def mj_workspace_init(workspace, stream=None):
    _check("mj_workspace_init", load_library().mj_workspace_init(_ptr(workspace), workspace.numel(),
                                                                 _stream(stream)))


def mj_workspace_status(workspace, stream=None) -> int:
    """Read and clear the device status word (synchronises). 0 = clean."""
    v = ctypes.c_uint32(0)
    st = load_library().mj_workspace_status(_ptr(workspace), _stream(stream), ctypes.byref(v))
    if st not in (MJ_OK, MJ_ERR_DEVICE_CHECK):
        _check("mj_workspace_status", st)
    return v.value


def mj_decode_attention(args: mj_decode_args, stream=None):
    _check("mj_decode_attention", load_library().mj_decode_attention(ctypes.byref(args), _stream(stream)))


def mj_merge_lse(args: mj_decode_args, stream=None):
    _check("mj_merge_lse", load_library().mj_merge_lse(ctypes.byref(args), _stream(stream)))


def mj_decode_attention_noalloc(args: mj_decode_args, stream=None):
    """Decode + merge with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory; see
    include/mj.h)."""
    _check("mj_decode_attention_noalloc",
           load_library().mj_decode_attention_noalloc(ctypes.byref(args), _stream(stream)))


def mj_noalloc_status(stream=None) -> int:
    """Read and clear the status word of the allocation-free call's scratch on
    the current device (synchronises). 0 = clean."""
    v = ctypes.c_uint32(0)
    st = load_library().mj_noalloc_status(_stream(stream), ctypes.byref(v))
    if st not in (MJ_OK, MJ_ERR_DEVICE_CHECK):
        _check("mj_noalloc_status", st)
    return v.value


def mj_write_kv(key, value, slot_mapping, k_cache, v_cache, kv_strides, page_size: int, num_pages: int,
                kv_format: int, k_scale, v_scale, scale_per_head: bool = False, status=None, stream=None):
    """Quantize K/V rows into the paged caches at ``slot_mapping``.

    ``key`` / ``value``: bf16 ``[T, h_k, d]`` (any token/head strides, channel
    stride 1). ``slot_mapping``: int64 ``[T]`` (negative = padding).
    ``k_cache`` / ``v_cache``: uint8 pools; ``kv_strides``: byte strides
    ``(page, token, head)`` shared by both. ``k_scale`` / ``v_scale``:
    float32 -- e4m3 ``[1]`` or ``[h_k]`` (``scale_per_head``), the packed formats
    ``[h_k, d]``. ``status``: optional int32/uint32 device word."""
    assert key.stride(2) == 1 and value.stride(2) == 1
    a = mj_write_kv_args()
    a.num_tokens, a.h_k, a.d = int(key.shape[0]), int(key.shape[1]), int(key.shape[2])
    a.key, a.value = _ptr(key), _ptr(value)
    a.key_tok_stride, a.key_head_stride = key.stride(0), key.stride(1)
    a.value_tok_stride, a.value_head_stride = value.stride(0), value.stride(1)
    a.slot_mapping = _ptr(slot_mapping)
    a.kv_format, a.page_size, a.num_pages = int(kv_format), int(page_size), int(num_pages)
    a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
    a.k_stride_page, a.k_stride_token, a.k_stride_head = (int(x) for x in kv_strides)
    a.v_stride_page, a.v_stride_token, a.v_stride_head = (int(x) for x in kv_strides)
    a.k_scale, a.v_scale = _ptr(k_scale), _ptr(v_scale)
    a.scale_per_head = 1 if scale_per_head else 0
    a.status = _ptr(status)
    _check("mj_write_kv", load_library().mj_write_kv(ctypes.byref(a), _stream(stream)))


from .step import DecodeStep  # noqa: E402,F401
