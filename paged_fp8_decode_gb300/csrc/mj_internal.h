// Internal definitions shared by the host ABI layer (mj_api.cpp) and the
// kernels. Not part of the public ABI: see include/mj.h.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/mj.h"

namespace mj {

// An NVTX range over an exported call (header-only NVTX: a few instructions
// when no tool is attached), so that a profiler timeline shows which call
// enqueued which kernels.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kKvTile = 128;   // tokens per KV tile (the plan's unit)
constexpr int kMaxHeadDim = 256;
// Supported head sizes: 128 and 256 (the runner page's T5DecodeRunner asserts
// head_size % 128 == 0; its kernels are built per head size).
inline bool head_dim_ok(int d) { return d == 128 || d == 256; }
constexpr int kMaxRowTile = 32;

// Widening factor of a cache format: the kernels widen a narrow code to an
// e4m3 code worth value / factor (e2m3, e2m1: 2^-6; e3m2: 2^-4; e4m3: 1).
__host__ __device__ constexpr float kv_widen_factor(int kv_format) {
  return kv_format == MJ_KV_E3M2 ? 16.f : (kv_format == MJ_KV_E4M3 ? 1.f : 64.f);
}

// Bytes of one (token, KV head) row of a cache format.
__host__ __device__ constexpr int kv_row_bytes(int kv_format, int d) {
  return kv_format == MJ_KV_E4M3 ? d : (kv_format == MJ_KV_E2M1 ? d / 2 : d * 3 / 4);
}

inline bool kv_format_ok(int f) { return f >= MJ_KV_E4M3 && f <= MJ_KV_E2M1; }

// Workspace layout: a 256-byte header (status word at offset 0), then the
// split partials o_part [rows][d], m_part [rows], l_part [rows].
constexpr size_t kWsHeader = 256;

// Status bits a kernel may OR into the workspace status word.
constexpr uint32_t kStatusBadPage = 1u;
constexpr uint32_t kStatusTimeout = 2u;
constexpr uint32_t kStatusBadPlan = 4u;

// Everything a decode / merge launch needs, by value (kernel parameter).
struct DecodeParams {
  int num_seqs, q_len, h_q, h_k, h_r, n_q, d;
  int causal;
  int kv_format, page_size, row_bytes;
  int64_t num_pages;
  int tw, n_row_tiles;  // query rows per CTA, row tiles per (request, head)
  int first_wave;       // tensor-core kernel: CTAs resident at once on the device

  const uint8_t* q_codes;
  const float* q_descale;
  int q_mode;               // mj_q_mode: 0 codes, 1 bf16 as is, 2 bf16 quantized in the kernel
  const uint16_t* q_bf16;
  int64_t q_ts, q_hs;       // element strides of q_bf16
  const float* q_mul;       // q_mode 2: nullable [h_q][d]
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  int64_t k_sp, k_st, k_sh, v_sp, v_st, v_sh;  // byte strides (page, token, head)
  const float* k_descale;
  const float* v_descale;
  int64_t ds_seq, ds_head;

  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;

  const int32_t* work;
  const int32_t* n_splits;
  int num_work, with_reduction, chunk_tiles, max_splits, part_seqs;

  // logits in the log2 domain: t = (q_code . k_code) * q_descale * k_descale * qk_scale_log2
  float qk_scale_log2;  // softmax_scale * log2(e) * (format factor of K)
  float v_fmt;          // format factor of V (64 for widened e2m3, else 1)

  const float* o_mul;
  uint16_t* out;  // bf16 (or fp16) bits
  int out_f16;    // 1: out holds fp16
  int64_t out_ts, out_hs;
  float* lse;

  uint32_t* status;
  float* o_part;
  float* m_part;
  float* l_part;

  int kv_stages;
  int evict_first;
  int tma_head_inner;  // tensor-core kernel: head dimension is the TMA's dim 1
};

// Index of a partial row: ((b*max_splits + s)*h_k + g)*n_q + row.
__host__ __device__ inline int64_t part_index(const DecodeParams& p, int b, int s, int g, int row) {
  return ((int64_t(b) * p.max_splits + s) * p.h_k + g) * p.n_q + row;
}

__host__ __device__ inline float kv_descale(const float* ds, int64_t seq_stride, int64_t head_stride,
                                            int b, int g) {
  return ds[int64_t(b) * seq_stride + int64_t(g) * head_stride];
}

struct QuantParams {
  const uint16_t* q;
  int64_t q_ts, q_hs;
  int num_seqs, q_len, h_q, h_k, h_r, n_q, d;
  const float* q_mul;
  uint8_t* codes;
  float* descale;
};

cudaError_t launch_quantize_q(const QuantParams& p, cudaStream_t stream);
cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_write_kv(const mj_write_kv_args& a, cudaStream_t stream);
// Tensor-core kernel; sets *unsupported (and launches nothing) when the
// arguments are outside its envelope.
cudaError_t launch_decode_tc(DecodeParams p, cudaStream_t stream, bool* unsupported);
// Whether the tensor-core kernel takes these arguments (launches nothing).
bool decode_tc_supported(const DecodeParams& p);

}  // namespace mj
