// mj_merge_lse kernel: combine split-KV partials by log-sum-exp.
//
// README of the mjolnir-kernel package, "A decode step" item 4: the split
// partials are merged by their log-sum-exp in a kernel of their own. A
// partial row holds the split's normalised output O~ (float32, d channels),
// its max logit m (log2 domain) and its sum l = sum 2^(t - m). For request b,
// KV head g and query row: M = max_s m_s, w_s = 2^(m_s - M) l_s, O = sum w_s O~_s / sum w_s.
// Splits that start at or past seq_lens[b] (a plan made from an upper bound)
// and rows with no visible key in a split (m = -inf, l = 0) weigh zero; the
// exponent is never formed from two infinities.
//
// One CTA per (request, KV head, query row), one thread per channel (D = 128
// or 256): the split weights are computed by as many threads in parallel,
// and the channel sums read the partials with independent, coalesced loads.
#include "mj_device.cuh"
#include "mj_internal.h"

namespace mj {

namespace {

// D threads (one per channel): 4 warps for D = 128, 8 for D = 256
template <int D>
__global__ void __launch_bounds__(D) merge_kernel(DecodeParams p) {
  constexpr int kWarps = D / 32;
  extern __shared__ float wsh[];  // weights of the live splits
  __shared__ float red[kWarps];
  // launched with programmatic stream serialization: the partials are the
  // preceding decode grid's output
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, g = blockIdx.y, row = blockIdx.z, c = threadIdx.x;
  const int warp = c >> 5, lane = c & 31;
  const int ns = min(p.n_splits[b], p.max_splits);
  if (ns <= 1) return;  // single split: the decode kernel wrote the output directly
  const int L = p.seq_lens[b];
  if (L <= 0) return;
  const int64_t span = int64_t(p.chunk_tiles) * kKvTile;
  const int live = int(min(int64_t(ns), (int64_t(L) + span - 1) / span));  // splits with >= 1 key

  // each thread loads the (m, l) of its first two splits once (any further
  // ones, beyond 2 D splits, twice): max logit over the live splits
  float ml[2] = {-INFINITY, -INFINITY}, ll[2] = {0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = c + k * D;
    if (s < live) {
      const int64_t idx = part_index(p, b, s, g, row);
      ml[k] = p.m_part[idx];
      ll[k] = p.l_part[idx];
    }
  }
  float mloc = fmaxf(ml[0], ml[1]);
  for (int s = c + 2 * D; s < live; s += D) mloc = fmaxf(mloc, p.m_part[part_index(p, b, s, g, row)]);
  mloc = warp_max(mloc);
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w2 = 1; w2 < kWarps; ++w2) M = fmaxf(M, red[w2]);
  __syncthreads();

  // split weights
  auto weight = [&](float ms, float ls) { return (M == -INFINITY || ms == -INFINITY) ? 0.f : fast_exp2(ms - M) * ls; };
  float wloc = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = c + k * D;
    if (s < live) {
      const float wgt = weight(ml[k], ll[k]);
      wsh[s] = wgt;
      wloc += wgt;
    }
  }
  for (int s = c + 2 * D; s < live; s += D) {
    const int64_t idx = part_index(p, b, s, g, row);
    const float wgt = weight(p.m_part[idx], p.l_part[idx]);
    wsh[s] = wgt;
    wloc += wgt;
  }
  wloc = warp_sum(wloc);
  if (lane == 0) red[warp] = wloc;
  __syncthreads();
  float wsum = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2) wsum += red[w2];

  // weighted channel sum: eight independent loads in flight per thread
  const float* op = p.o_part + part_index(p, b, 0, g, row) * D + c;
  const int64_t split_stride = int64_t(p.h_k) * p.n_q * D;  // part_index step per split
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int s = 0;
  for (; s + 8 <= live; s += 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = fmaf(wsh[s + k], op[int64_t(s + k) * split_stride], a[k]);
  }
  for (; s < live; ++s) a[0] = fmaf(wsh[s], op[int64_t(s) * split_stride], a[0]);
  const float acc = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));

  const int tq = row / p.h_r, h = g * p.h_r + row % p.h_r;
  const float vd = kv_descale(p.v_descale, p.ds_seq, p.ds_head, b, g) * p.v_fmt;
  float val = wsum > 0.f ? acc / wsum * vd : 0.f;
  if (p.o_mul) val *= p.o_mul[int64_t(h) * D + c];
  p.out[int64_t(b * p.q_len + tq) * p.out_ts + int64_t(h) * p.out_hs + c] = float_to_out_bits(val, p.out_f16);
  if (p.lse && c == 0)
    p.lse[(int64_t(b) * p.h_k + g) * p.n_q + row] = wsum > 0.f ? (M + fast_log2(wsum)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
  if (!p.with_reduction || p.num_seqs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_seqs, p.h_k, p.n_q);
  cfg.blockDim = dim3(p.d);
  cfg.dynamicSmemBytes = size_t(p.max_splits) * sizeof(float);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.d == 256 ? cudaLaunchKernelEx(&cfg, merge_kernel<256>, p) : cudaLaunchKernelEx(&cfg, merge_kernel<128>, p);
}

}  // namespace mj
