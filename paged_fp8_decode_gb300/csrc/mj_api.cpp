// Host side of the C ABI (include/mj.h): argument validation, the split-KV
// plan, workspace layout, and kernel launches. Nothing here allocates,
// synchronises (except mj_workspace_status, documented as a debugging aid)
// or reads device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "mj_internal.h"

namespace {

using mj::DecodeParams;

constexpr int kVersion = 100;  // 0.1.0

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int next_pow2(int n) {
  int p = 1;
  while (p < n) p *= 2;
  return p;
}

int n_row_tiles(int n_q) { return int(ceil_div(n_q, mj_tile_width(n_q))); }

int status_of(cudaError_t e) { return e == cudaSuccess ? MJ_OK : MJ_ERR_CUDA; }

bool page_size_ok(int ps) { return ps == 16 || ps == 32 || ps == 64 || ps == 128; }

// Validate a decode argument struct and derive the kernel parameters.
int make_params(const mj_decode_args* a, DecodeParams* p) {
  if (!a) return MJ_ERR_INVALID_ARG;
  if (a->num_seqs < 0 || a->q_len < 1 || a->h_k < 1 || a->h_q < 1 || a->h_q % a->h_k) return MJ_ERR_INVALID_ARG;
  if (!mj::head_dim_ok(a->d)) return MJ_ERR_UNSUPPORTED;
  if (!mj::kv_format_ok(a->kv_format)) return MJ_ERR_UNSUPPORTED;
  if (!page_size_ok(a->page_size)) return MJ_ERR_UNSUPPORTED;
  if (a->num_pages < 1 || a->num_work < 0 || a->block_table_stride < 0) return MJ_ERR_INVALID_ARG;
  if (a->impl < MJ_IMPL_AUTO || a->impl > MJ_IMPL_TCGEN05) return MJ_ERR_INVALID_ARG;
  if (!(a->softmax_scale > 0.f) || !std::isfinite(a->softmax_scale)) return MJ_ERR_INVALID_ARG;
  if (a->q_mode != MJ_Q_FP8 && a->q_mode != MJ_Q_BF16 && a->q_mode != MJ_Q_FP8_FUSED) return MJ_ERR_UNSUPPORTED;
  const bool bf16_q = a->q_mode != MJ_Q_FP8;  // the call reads bf16 Q
  if (a->q_mode == MJ_Q_BF16 && a->kv_format != MJ_KV_E4M3) return MJ_ERR_UNSUPPORTED;  // packed KV is fp8-Q only
  if (a->q_mul && !aligned(a->q_mul, 16)) return MJ_ERR_ALIGNMENT;
  const void* q0 = bf16_q ? a->q_bf16 : a->q_codes;
  const void* q1 = bf16_q ? a->q_bf16 : a->q_descale;
  const void* need[] = {q0, q1, a->k_cache,  a->v_cache, a->k_descale, a->v_descale,
                        a->block_table, a->seq_lens, a->work, a->n_splits, a->out, a->workspace};
  for (const void* ptr : need)
    if (!ptr) return MJ_ERR_INVALID_ARG;
  if (bf16_q) {
    if (a->q_tok_stride < 0 || a->q_head_stride < 0) return MJ_ERR_INVALID_ARG;
    if (a->q_tok_stride % 8 || a->q_head_stride % 8) return MJ_ERR_ALIGNMENT;
  }
  const uintptr_t kv_align = a->kv_format == MJ_KV_E4M3 ? 16 : 32;
  const void* a16[] = {q0, q1, a->block_table, a->seq_lens, a->work,
                       a->n_splits, a->out, a->workspace};
  for (const void* ptr : a16)
    if (!aligned(ptr, 16)) return MJ_ERR_ALIGNMENT;
  if (!aligned(a->k_cache, kv_align) || !aligned(a->v_cache, kv_align)) return MJ_ERR_ALIGNMENT;
  if ((a->o_mul && !aligned(a->o_mul, 16)) || (a->lse && !aligned(a->lse, 4))) return MJ_ERR_ALIGNMENT;
  if (!aligned(a->k_descale, 4) || !aligned(a->v_descale, 4)) return MJ_ERR_ALIGNMENT;
  const int64_t kvs[] = {a->k_stride_page, a->k_stride_token, a->k_stride_head,
                         a->v_stride_page, a->v_stride_token, a->v_stride_head};
  for (int64_t s : kvs) {
    if (s < 0) return MJ_ERR_INVALID_ARG;
    if (s % 16) return MJ_ERR_ALIGNMENT;
  }
  if (a->out_tok_stride < 0 || a->out_head_stride < 0 || a->descale_seq_stride < 0 || a->descale_head_stride < 0)
    return MJ_ERR_INVALID_ARG;
  if (a->out_tok_stride % 8 || a->out_head_stride % 8) return MJ_ERR_ALIGNMENT;
  if (a->out_dtype != MJ_OUT_BF16 && a->out_dtype != MJ_OUT_F16) return MJ_ERR_UNSUPPORTED;

  const int h_r = a->h_q / a->h_k;
  const int n_q = a->q_len * h_r;
  if (a->with_reduction) {
    if (a->max_splits < 1 || a->part_seqs < a->num_seqs || a->chunk_tiles < 1) return MJ_ERR_INVALID_ARG;
    size_t need_bytes = 0;
    int st = mj_workspace_size(a->part_seqs, a->max_splits, a->q_len, a->h_q, a->h_k, a->d, &need_bytes);
    if (st != MJ_OK) return st;
    if (a->workspace_bytes < need_bytes) return MJ_ERR_CAPACITY;
  } else if (a->workspace_bytes < mj::kWsHeader) {
    return MJ_ERR_CAPACITY;
  }

  DecodeParams& q = *p;
  std::memset(&q, 0, sizeof(q));
  q.num_seqs = a->num_seqs;
  q.q_len = a->q_len;
  q.h_q = a->h_q;
  q.h_k = a->h_k;
  q.h_r = h_r;
  q.n_q = n_q;
  q.d = a->d;
  q.causal = a->causal ? 1 : 0;
  q.kv_format = a->kv_format;
  q.page_size = a->page_size;
  q.row_bytes = mj::kv_row_bytes(a->kv_format, a->d);
  q.num_pages = a->num_pages;
  q.tw = mj_tile_width(n_q);
  q.n_row_tiles = n_row_tiles(n_q);
  q.q_codes = a->q_codes;
  q.q_descale = a->q_descale;
  q.q_mode = a->q_mode;
  q.q_mul = a->q_mode == MJ_Q_FP8_FUSED ? a->q_mul : nullptr;
  q.q_bf16 = static_cast<const uint16_t*>(a->q_bf16);
  q.q_ts = a->q_tok_stride;
  q.q_hs = a->q_head_stride;
  q.k_cache = static_cast<const uint8_t*>(a->k_cache);
  q.v_cache = static_cast<const uint8_t*>(a->v_cache);
  q.k_sp = a->k_stride_page;
  q.k_st = a->k_stride_token;
  q.k_sh = a->k_stride_head;
  q.v_sp = a->v_stride_page;
  q.v_st = a->v_stride_token;
  q.v_sh = a->v_stride_head;
  q.k_descale = a->k_descale;
  q.v_descale = a->v_descale;
  q.ds_seq = a->descale_seq_stride;
  q.ds_head = a->descale_head_stride;
  q.block_table = a->block_table;
  q.bt_stride = a->block_table_stride;
  q.seq_lens = a->seq_lens;
  q.work = a->work;
  q.n_splits = a->n_splits;
  q.num_work = a->num_work;
  q.with_reduction = a->with_reduction ? 1 : 0;
  q.chunk_tiles = std::max(1, a->chunk_tiles);
  q.max_splits = std::max(1, a->max_splits);
  q.part_seqs = a->part_seqs;
  // Widened narrow codes are the true values over kv_widen_factor.
  const float fmt = mj::kv_widen_factor(a->kv_format);
  q.qk_scale_log2 = a->softmax_scale * 1.4426950408889634f * fmt;
  q.v_fmt = fmt;
  q.o_mul = a->o_mul;
  q.out = static_cast<uint16_t*>(a->out);
  q.out_f16 = a->out_dtype == MJ_OUT_F16 ? 1 : 0;
  q.out_ts = a->out_tok_stride;
  q.out_hs = a->out_head_stride;
  q.lse = a->lse;
  char* ws = static_cast<char*>(a->workspace);
  q.status = reinterpret_cast<uint32_t*>(ws);
  const int64_t rows = int64_t(std::max(0, a->part_seqs)) * q.max_splits * a->h_k * n_q;
  q.o_part = reinterpret_cast<float*>(ws + mj::kWsHeader);
  q.m_part = q.o_part + rows * a->d;
  q.l_part = q.m_part + rows;
  q.kv_stages = a->kv_stages;
  q.evict_first = a->evict_first;
  return MJ_OK;
}

}  // namespace

extern "C" {

const char* mj_status_string(int status) {
  switch (status) {
    case MJ_OK: return "ok";
    case MJ_ERR_INVALID_ARG: return "invalid argument";
    case MJ_ERR_UNSUPPORTED: return "unsupported configuration";
    case MJ_ERR_ALIGNMENT: return "alignment requirement not met";
    case MJ_ERR_CAPACITY: return "caller buffer too small";
    case MJ_ERR_CUDA: return "CUDA runtime error";
    case MJ_ERR_DEVICE_CHECK: return "a kernel recorded an anomaly";
    default: return "unknown status";
  }
}

int mj_version(void) { return kVersion; }

int mj_tile_width(int n_q) { return std::max(16, std::min(32, next_pow2(std::max(1, n_q)))); }

int mj_slots(int sm_count, int ctas_per_sm, int h_k, int q_len, int h_q) {
  if (sm_count < 1 || ctas_per_sm < 1 || h_k < 1 || q_len < 1 || h_q < h_k) return 1;
  const int n_q = q_len * (h_q / h_k);
  return std::max(1, (sm_count * ctas_per_sm) / (h_k * n_row_tiles(n_q)));
}

int mj_plan_split_kv(const int32_t* seq_lens_host, int num_seqs, int q_len, int h_q, int h_k,
                     int sm_count, int ctas_per_sm, int max_splits, int margin, int pad_to,
                     int32_t* work_host, int32_t* n_splits_host, int* chunk_tiles,
                     int* with_reduction, int* slots_out) {
  const mj::NvtxRange range("mj_plan_split_kv");
  if (num_seqs < 0 || q_len < 1 || h_k < 1 || h_q < 1 || h_q % h_k || sm_count < 1 || ctas_per_sm < 1 ||
      max_splits < 1 || margin < 0 || pad_to < 0)
    return MJ_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!seq_lens_host || !n_splits_host)) return MJ_ERR_INVALID_ARG;
  if (pad_to > 0 && !work_host) return MJ_ERR_INVALID_ARG;
  const int s = mj_slots(sm_count, ctas_per_sm, h_k, q_len, h_q);
  if (pad_to < std::max(s, num_seqs)) return MJ_ERR_CAPACITY;
  for (int b = 0; b < num_seqs; ++b)
    if (seq_lens_host[b] < 0) return MJ_ERR_INVALID_ARG;

  auto tiles = [&](int b) -> int64_t {
    const int64_t L = int64_t(seq_lens_host[b]) + margin;
    return L > 0 ? ceil_div(L, mj::kKvTile) : 0;
  };
  const bool red = max_splits > 1 && num_seqs < s;
  int64_t max_t = 0;
  for (int b = 0; b < num_seqs; ++b) max_t = std::max(max_t, tiles(b));

  int64_t chunk = std::max<int64_t>(1, max_t);
  if (red) {
    // Smallest c with sum_b max(1, ceil(t_b/c)) <= slots and
    // max_b ceil(t_b/c) <= max_splits. Both sides fall monotonically with c
    // and c = max(1, max_t) always qualifies (num_seqs < slots), so a binary
    // search finds the same c as a linear scan.
    auto fits = [&](int64_t c) {
      int64_t items = 0, widest = 0;
      for (int b = 0; b < num_seqs; ++b) {
        const int64_t n = ceil_div(tiles(b), c);
        items += std::max<int64_t>(1, n);
        widest = std::max(widest, n);
      }
      return items <= s && widest <= max_splits;
    };
    int64_t lo = 1, hi = std::max<int64_t>(1, max_t);
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (fits(mid))
        hi = mid;
      else
        lo = mid + 1;
    }
    chunk = lo;
  }
  if (chunk > INT32_MAX) return MJ_ERR_INVALID_ARG;

  int64_t row = 0;
  for (int b = 0; b < num_seqs; ++b) {
    const int64_t t = tiles(b);
    const int64_t ns = red ? std::max<int64_t>(1, ceil_div(t, chunk)) : 1;
    n_splits_host[b] = int32_t(ns);
    for (int64_t sp = 0; sp < ns; ++sp) {
      if (row >= pad_to) return MJ_ERR_CAPACITY;
      const int64_t tb = red ? sp * chunk : 0;
      const int64_t te = red ? std::min((sp + 1) * chunk, t) : t;
      if (te > INT32_MAX) return MJ_ERR_INVALID_ARG;
      int32_t* w = work_host + 4 * row;
      w[0] = b;
      w[1] = int32_t(tb);
      w[2] = int32_t(te);
      w[3] = int32_t(sp);
      ++row;
    }
  }
  for (; row < pad_to; ++row) std::memset(work_host + 4 * row, 0, 4 * sizeof(int32_t));
  if (chunk_tiles) *chunk_tiles = int(chunk);
  if (with_reduction) *with_reduction = red ? 1 : 0;
  if (slots_out) *slots_out = s;
  return MJ_OK;
}

int mj_plan_upload(const int32_t* work_host, const int32_t* n_splits_host, int32_t* work_dev, int32_t* n_splits_dev,
                   int pad_to, int num_seqs, void* stream) {
  const mj::NvtxRange range("mj_plan_upload");
  if (pad_to < 0 || num_seqs < 0) return MJ_ERR_INVALID_ARG;
  if ((pad_to > 0 && (!work_host || !work_dev)) || (num_seqs > 0 && (!n_splits_host || !n_splits_dev)))
    return MJ_ERR_INVALID_ARG;
  if ((work_dev && !aligned(work_dev, 16)) || (n_splits_dev && !aligned(n_splits_dev, 16))) return MJ_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one copy per buffer
  if (pad_to > 0) {
    const cudaError_t e =
        cudaMemcpyAsync(work_dev, work_host, size_t(pad_to) * 4 * sizeof(int32_t), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return MJ_ERR_CUDA;
  }
  if (num_seqs > 0) {
    const cudaError_t e =
        cudaMemcpyAsync(n_splits_dev, n_splits_host, size_t(num_seqs) * sizeof(int32_t), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return MJ_ERR_CUDA;
  }
  return MJ_OK;
}

int mj_decode_kernel(const mj_decode_args* args, int* impl) {
  if (!impl) return MJ_ERR_INVALID_ARG;
  DecodeParams p;
  const int st = make_params(args, &p);
  if (st != MJ_OK) return st;
  if (args->impl == MJ_IMPL_SIMT) {
    *impl = MJ_IMPL_SIMT;
    return MJ_OK;
  }
  const bool tc = mj::decode_tc_supported(p);
  if (!tc && args->impl == MJ_IMPL_TCGEN05) return MJ_ERR_UNSUPPORTED;
  *impl = tc ? MJ_IMPL_TCGEN05 : MJ_IMPL_SIMT;
  return MJ_OK;
}

int mj_quantize_q(const void* q, int64_t q_tok_stride, int64_t q_head_stride, int num_seqs, int q_len,
                  int h_q, int h_k, int d, const float* q_mul, uint8_t* q_codes, float* q_descale,
                  void* stream) {
  const mj::NvtxRange range("mj_quantize_q");
  if (num_seqs < 0 || q_len < 1 || h_k < 1 || h_q < 1 || h_q % h_k) return MJ_ERR_INVALID_ARG;
  if (!mj::head_dim_ok(d)) return MJ_ERR_UNSUPPORTED;
  if (num_seqs == 0) return MJ_OK;
  if (!q || !q_codes || !q_descale) return MJ_ERR_INVALID_ARG;
  if (q_tok_stride < 0 || q_head_stride < 0) return MJ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(q_codes, 16) || !aligned(q_descale, 4) || (q_mul && !aligned(q_mul, 16)))
    return MJ_ERR_ALIGNMENT;
  mj::QuantParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.q_ts = q_tok_stride;
  p.q_hs = q_head_stride;
  p.num_seqs = num_seqs;
  p.q_len = q_len;
  p.h_q = h_q;
  p.h_k = h_k;
  p.h_r = h_q / h_k;
  p.n_q = q_len * p.h_r;
  p.d = d;
  p.q_mul = q_mul;
  p.codes = q_codes;
  p.descale = q_descale;
  return status_of(mj::launch_quantize_q(p, static_cast<cudaStream_t>(stream)));
}

int mj_write_kv(const mj_write_kv_args* a, void* stream) {
  const mj::NvtxRange range("mj_write_kv");
  if (!a) return MJ_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->h_k < 1 || a->num_pages < 0) return MJ_ERR_INVALID_ARG;
  if (!mj::head_dim_ok(a->d)) return MJ_ERR_UNSUPPORTED;
  if (!mj::kv_format_ok(a->kv_format)) return MJ_ERR_UNSUPPORTED;
  if (a->page_size != 16 && a->page_size != 32 && a->page_size != 64 && a->page_size != 128)
    return MJ_ERR_UNSUPPORTED;
  if (a->num_tokens == 0) return MJ_OK;
  if (int64_t(a->num_tokens) * a->h_k >= (int64_t(1) << 31)) return MJ_ERR_INVALID_ARG;
  if (!a->key || !a->value || !a->slot_mapping || !a->k_cache || !a->v_cache || !a->k_scale || !a->v_scale)
    return MJ_ERR_INVALID_ARG;
  const int64_t el[] = {a->key_tok_stride, a->key_head_stride, a->value_tok_stride, a->value_head_stride};
  const int64_t by[] = {a->k_stride_page, a->k_stride_token, a->k_stride_head,
                        a->v_stride_page, a->v_stride_token, a->v_stride_head};
  for (int64_t v : el)
    if (v < 0) return MJ_ERR_INVALID_ARG;
  for (int64_t v : by)
    if (v < 0) return MJ_ERR_INVALID_ARG;
  for (int64_t v : el)
    if (v % 8) return MJ_ERR_ALIGNMENT;
  for (int64_t v : by)
    if (v % 16) return MJ_ERR_ALIGNMENT;
  if (!aligned(a->key, 16) || !aligned(a->value, 16) || !aligned(a->slot_mapping, 8) || !aligned(a->k_cache, 16) ||
      !aligned(a->v_cache, 16) || !aligned(a->k_scale, 16) || !aligned(a->v_scale, 16) ||
      (a->status && !aligned(a->status, 4)))
    return MJ_ERR_ALIGNMENT;
  return status_of(mj::launch_write_kv(*a, static_cast<cudaStream_t>(stream)));
}

int mj_workspace_size(int part_seqs, int max_splits, int max_q_len, int h_q, int h_k, int d, size_t* bytes) {
  if (!bytes || part_seqs < 0 || max_splits < 1 || max_q_len < 1 || h_k < 1 || h_q < 1 || h_q % h_k)
    return MJ_ERR_INVALID_ARG;
  if (!mj::head_dim_ok(d)) return MJ_ERR_UNSUPPORTED;
  const int64_t rows = int64_t(part_seqs) * max_splits * h_k * int64_t(max_q_len) * (h_q / h_k);
  *bytes = mj::kWsHeader + size_t(rows) * (size_t(d) + 2) * sizeof(float);
  return MJ_OK;
}

int mj_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  const mj::NvtxRange range("mj_workspace_init");
  if (!workspace || workspace_bytes < mj::kWsHeader) return MJ_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return MJ_ERR_ALIGNMENT;
  return status_of(cudaMemsetAsync(workspace, 0, mj::kWsHeader, static_cast<cudaStream_t>(stream)));
}

int mj_workspace_status(void* workspace, void* stream, uint32_t* device_status) {
  const mj::NvtxRange range("mj_workspace_status");
  if (!workspace || !device_status) return MJ_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return MJ_ERR_CUDA;
  *device_status = v;
  return v ? MJ_ERR_DEVICE_CHECK : MJ_OK;
}

int mj_decode_attention(const mj_decode_args* args, void* stream) {
  const mj::NvtxRange range("mj_decode_attention");
  DecodeParams p;
  int st = make_params(args, &p);
  if (st != MJ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (args->impl != MJ_IMPL_SIMT) {
    bool unsupported = false;
    const cudaError_t e = mj::launch_decode_tc(p, s, &unsupported);
    if (!unsupported) return status_of(e);
    if (args->impl == MJ_IMPL_TCGEN05) return MJ_ERR_UNSUPPORTED;
  }
  // The CUDA-core kernel tiles query rows by the smallest power of two that
  // holds them (at least 4, at most 32).
  p.tw = std::max(4, std::min(32, next_pow2(p.n_q)));
  p.n_row_tiles = int(ceil_div(p.n_q, p.tw));
  return status_of(mj::launch_decode_simt(p, s));
}

int mj_merge_lse(const mj_decode_args* args, void* stream) {
  const mj::NvtxRange range("mj_merge_lse");
  DecodeParams p;
  int st = make_params(args, &p);
  if (st != MJ_OK) return st;
  return status_of(mj::launch_merge(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
