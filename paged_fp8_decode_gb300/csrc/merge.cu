// mj_merge_lse kernel: combine split-KV partials by log-sum-exp.
//
// README of the mjolnir-kernel package, "A decode step" item 4: a small
// second kernel combines the split-KV partials by LSE. A partial row holds
// the split's normalised output O~ (float32, d channels), its max logit m
// (log2 domain) and its sum l = sum 2^(t - m). For request b, KV head g and
// query row: M = max_s m_s, w_s = 2^(m_s - M) l_s, O = sum w_s O~_s / sum w_s.
// Splits that start at or past seq_lens[b] (a plan made from an upper bound)
// and rows with no visible key in a split (m = -inf, l = 0) weigh zero; the
// exponent is never formed from two infinities.
#include "mj_device.cuh"
#include "mj_internal.h"

namespace mj {

namespace {

__global__ void __launch_bounds__(kHeadDim) merge_kernel(DecodeParams p) {
  const int b = blockIdx.x, g = blockIdx.y, c = threadIdx.x;
  const int ns = min(p.n_splits[b], p.max_splits);
  if (ns <= 1) return;  // single split: the decode kernel wrote the output directly
  const int L = p.seq_lens[b];
  if (L <= 0) return;
  const int64_t span = int64_t(p.chunk_tiles) * kKvTile;
  const int live = int(min(int64_t(ns), (int64_t(L) + span - 1) / span));  // splits with >= 1 key

  const float vd = kv_descale(p.v_descale, p.ds_seq, p.ds_head, b, g) * p.v_fmt;
  for (int row = 0; row < p.n_q; ++row) {
    float M = -INFINITY;
    for (int s = 0; s < live; ++s) M = fmaxf(M, p.m_part[part_index(p, b, s, g, row)]);
    float acc = 0.f, wsum = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < live; ++s) {
        const int64_t idx = part_index(p, b, s, g, row);
        const float ms = p.m_part[idx];
        if (ms == -INFINITY) continue;
        const float wgt = fast_exp2(ms - M) * p.l_part[idx];
        acc = fmaf(wgt, p.o_part[idx * kHeadDim + c], acc);
        wsum += wgt;
      }
    }
    const int tq = row / p.h_r, rr = row % p.h_r, h = g * p.h_r + rr;
    float val = wsum > 0.f ? acc / wsum * vd : 0.f;
    if (p.o_mul) val *= p.o_mul[int64_t(h) * kHeadDim + c];
    p.out[int64_t(b * p.q_len + tq) * p.out_ts + int64_t(h) * p.out_hs + c] = float_to_bf16_bits(val);
    if (p.lse && c == 0)
      p.lse[(int64_t(b) * p.h_k + g) * p.n_q + row] = wsum > 0.f ? (M + fast_log2(wsum)) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
  if (!p.with_reduction || p.num_seqs == 0) return cudaSuccess;
  dim3 grid(p.num_seqs, p.h_k);
  merge_kernel<<<grid, kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mj
