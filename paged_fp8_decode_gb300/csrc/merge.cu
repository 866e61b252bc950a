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
// or 256), or four when the grid is smaller than the GPU: the split weights
// are computed by as many threads in parallel, and the channel sums read the
// partials with independent, coalesced loads.
#include <atomic>

#include "mj_device.cuh"
#include "mj_internal.h"

namespace mj {

namespace {

// kGroups x D threads: thread t takes channel t % D of the splits
// s = t / D (mod kGroups), so each thread reads 1 / kGroups of the splits'
// partials and the kGroups sums meet in shared memory. Four groups shorten
// each CTA's chain of loads when the grid is too small to fill the GPU (a
// few long requests split many ways); one group keeps the many small CTAs of
// a large batch cheap to schedule.
template <int D, int kGroups>
__global__ void __launch_bounds__(kGroups * D) merge_kernel(DecodeParams p) {
  constexpr int kThreads = kGroups * D;
  constexpr int kWarps = kThreads / 32;
  extern __shared__ float wsh[];  // weights of the live splits
  __shared__ float red[kWarps];
  __shared__ float part[kGroups > 1 ? kGroups - 1 : 1][D];  // groups 1 .. kGroups-1: their channel sums
  // launched with programmatic stream serialization: the partials are the
  // preceding decode grid's output
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, g = blockIdx.y, row = blockIdx.z, t = threadIdx.x;
  const int c = t % D, grp = t / D;
  const int warp = t >> 5, lane = t & 31;
  const int ns = min(p.n_splits[b], p.max_splits);
  if (ns <= 1) return;  // single split: the decode kernel wrote the output directly
  const int L = p.seq_lens[b];
  if (L <= 0) return;
  const int64_t span = int64_t(p.chunk_tiles) * kKvTile;
  const int live = int(min(int64_t(ns), (int64_t(L) + span - 1) / span));  // splits with >= 1 key

  // thread t loads the (m, l) of split t (and of t + kThreads ..., if any):
  // max logit over the live splits
  float m0 = -INFINITY, l0 = 0.f;
  if (t < live) {
    const int64_t idx = part_index(p, b, t, g, row);
    m0 = p.m_part[idx];
    l0 = p.l_part[idx];
  }
  float mloc = m0;
  for (int s = t + kThreads; s < live; s += kThreads) mloc = fmaxf(mloc, p.m_part[part_index(p, b, s, g, row)]);
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
  if (t < live) {
    wsh[t] = weight(m0, l0);
    wloc = wsh[t];
  }
  for (int s = t + kThreads; s < live; s += kThreads) {
    const int64_t idx = part_index(p, b, s, g, row);
    wsh[s] = weight(p.m_part[idx], p.l_part[idx]);
    wloc += wsh[s];
  }
  wloc = warp_sum(wloc);
  if (lane == 0) red[warp] = wloc;
  __syncthreads();
  float wsum = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2) wsum += red[w2];

  // weighted channel sum over this group's splits (grp, grp + kGroups, ...),
  // eight independent loads in flight per thread
  const float* op = p.o_part + part_index(p, b, 0, g, row) * D + c;
  const int64_t split_stride = int64_t(p.h_k) * p.n_q * D;  // part_index step per split
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int s = grp;
  for (; s + 7 * kGroups < live; s += 8 * kGroups) {
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = fmaf(wsh[s + k * kGroups], op[int64_t(s + k * kGroups) * split_stride], a[k]);
  }
  for (; s < live; s += kGroups) a[0] = fmaf(wsh[s], op[int64_t(s) * split_stride], a[0]);
  float acc = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  if constexpr (kGroups > 1) {
    if (grp > 0) part[grp - 1][c] = acc;
    __syncthreads();
    if (grp > 0) return;
#pragma unroll
    for (int k = 0; k < kGroups - 1; ++k) acc += part[k][c];
  }

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
  // four thread groups per CTA when the grid is smaller than the GPU
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<int> sm_count[64];  // per device, looked up once (host threads may race)
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  const bool wide = int64_t(p.num_seqs) * p.h_k * p.n_q < sms;
  cfg.blockDim = dim3((wide ? 4 : 1) * p.d);
  cfg.dynamicSmemBytes = size_t(p.max_splits) * sizeof(float);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.d == 256)
    return wide ? cudaLaunchKernelEx(&cfg, merge_kernel<256, 4>, p) : cudaLaunchKernelEx(&cfg, merge_kernel<256, 1>, p);
  return wide ? cudaLaunchKernelEx(&cfg, merge_kernel<128, 4>, p) : cudaLaunchKernelEx(&cfg, merge_kernel<128, 1>, p);
}

}  // namespace mj
