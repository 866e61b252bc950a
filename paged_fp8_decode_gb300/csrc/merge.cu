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
// Two shapes. When the (request, KV head, query row) units are fewer than the
// SMs (a few long requests split many ways), one CTA per unit with four
// threads per channel: the split weights are computed by as many threads in
// parallel, and with a plan of at most 64 splits every partial the CTA may
// need is requested at once, before the split count is known, and those past
// the live splits are masked off afterwards. Otherwise one warp per unit,
// eight units per CTA, each lane holding four channels: the whole grid is
// resident at once, the weights need no block barrier (warp shuffles), and the
// first four splits' partials are requested with the split count.
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
// a large batch cheap to schedule. kSpec > 0 (four groups, max_splits <=
// kSpec * kGroups): the loads of the splits' (m, l) and of this thread's
// kSpec partial channels are issued together, right after the wait, for
// every split the workspace holds; the ones at or past the live count are
// uninitialised memory and never reach the arithmetic (selected off, not
// multiplied by zero).
template <int D, int kGroups, int kSpec>
__global__ void __launch_bounds__(kGroups * D) merge_kernel(DecodeParams p) {
  constexpr int kThreads = kGroups * D;
  constexpr int kWarps = kThreads / 32;
  static_assert(kSpec == 0 || kSpec * kGroups <= kThreads, "one (m, l) per thread");
  extern __shared__ float wsh[];  // weights of the live splits
  __shared__ float red[kWarps];
  __shared__ float part[kGroups > 1 ? kGroups - 1 : 1][D];  // groups 1 .. kGroups-1: their channel sums
  // launched with programmatic stream serialization: the partials are the
  // preceding decode grid's output. The trigger lets the next kernel on the
  // stream (the next step's decode, which waits for this grid before it reads
  // anything) launch and run its set-up on the SMs these few CTAs leave free.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, g = blockIdx.y, row = blockIdx.z, t = threadIdx.x;
  const int c = t % D, grp = t / D;
  const int warp = t >> 5, lane = t & 31;
  const float* op = p.o_part + part_index(p, b, 0, g, row) * D + c;
  const int64_t split_stride = int64_t(p.h_k) * p.n_q * D;  // part_index step per split
  // the epilogue's constants, loaded with the partials
  const int tq = row / p.h_r, h = g * p.h_r + row % p.h_r;
  const float vd = kv_descale(p.v_descale, p.ds_seq, p.ds_head, b, g) * p.v_fmt;
  const float om = p.o_mul ? p.o_mul[int64_t(h) * D + c] : 1.f;

  float m0 = -INFINITY, l0 = 0.f;
  float ov[kSpec > 0 ? kSpec : 1];
  if constexpr (kSpec > 0) {
    if (t < p.max_splits) {
      const int64_t idx = part_index(p, b, t, g, row);
      m0 = p.m_part[idx];
      l0 = p.l_part[idx];
    }
#pragma unroll
    for (int k = 0; k < kSpec; ++k) {
      const int s = grp + k * kGroups;
      ov[k] = s < p.max_splits ? op[int64_t(s) * split_stride] : 0.f;
    }
  }
  const int ns = min(p.n_splits[b], p.max_splits);
  if (ns <= 1) return;  // single split: the decode kernel wrote the output directly
  const int L = p.seq_lens[b];
  if (L <= 0) return;
  const int64_t span = int64_t(p.chunk_tiles) * kKvTile;
  const int live = int(min(int64_t(ns), (int64_t(L) + span - 1) / span));  // splits with >= 1 key

  // thread t holds the (m, l) of split t (and reads those of t + kThreads ...,
  // if any): max logit over the live splits
  if constexpr (kSpec > 0) {
    if (t >= live) {
      m0 = -INFINITY;
      l0 = 0.f;
    }
  } else if (t < live) {
    const int64_t idx = part_index(p, b, t, g, row);
    m0 = p.m_part[idx];
    l0 = p.l_part[idx];
  }
  float mloc = m0;
  if constexpr (kSpec == 0)
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
  if constexpr (kSpec == 0) {
    for (int s = t + kThreads; s < live; s += kThreads) {
      const int64_t idx = part_index(p, b, s, g, row);
      wsh[s] = weight(p.m_part[idx], p.l_part[idx]);
      wloc += wsh[s];
    }
  }
  wloc = warp_sum(wloc);
  if (lane == 0) red[warp] = wloc;
  __syncthreads();
  float wsum = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2) wsum += red[w2];

  // weighted channel sum over this group's splits (grp, grp + kGroups, ...)
  float acc;
  if constexpr (kSpec > 0) {
    float a[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kSpec; ++k) {
      const int s = grp + k * kGroups;
      if (s < live) a[k & 1] = fmaf(wsh[s], ov[k], a[k & 1]);
    }
    acc = a[0] + a[1];
  } else {
    // eight independent loads in flight per thread
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int s = grp;
    for (; s + 7 * kGroups < live; s += 8 * kGroups) {
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = fmaf(wsh[s + k * kGroups], op[int64_t(s + k * kGroups) * split_stride], a[k]);
    }
    for (; s < live; s += kGroups) a[0] = fmaf(wsh[s], op[int64_t(s) * split_stride], a[0]);
    acc = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  }
  if constexpr (kGroups > 1) {
    if (grp > 0) part[grp - 1][c] = acc;
    __syncthreads();
    if (grp > 0) return;
#pragma unroll
    for (int k = 0; k < kGroups - 1; ++k) acc += part[k][c];
  }

  float val = wsum > 0.f ? acc / wsum * vd : 0.f;
  if (p.o_mul) val *= om;
  p.out[int64_t(b * p.q_len + tq) * p.out_ts + int64_t(h) * p.out_hs + c] = float_to_out_bits(val, p.out_f16);
  if (p.lse && c == 0)
    p.lse[(int64_t(b) * p.h_k + g) * p.n_q + row] = wsum > 0.f ? (M + fast_log2(wsum)) * kLn2 : -INFINITY;
}

// One warp per unit (b, g, row), kRows units per CTA. Lane l holds channels
// 4l .. 4l + 3 of each 128-channel half. The (m, l) of splits 0 .. 31 sit in
// lanes 0 .. 31; a split's weight reaches every lane by shuffle. The first
// kPre splits' partials (uninitialised memory where past the live count, and
// never used there) are loaded before the split count is known.
template <int D, int kRows>
__global__ void __launch_bounds__(32 * kRows) merge_rows_kernel(DecodeParams p) {
  constexpr int kV = D / 128;  // float4 per lane
  constexpr int kPre = 4;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t unit = int64_t(blockIdx.x) * kRows + (threadIdx.x >> 5);
  if (unit >= int64_t(p.num_seqs) * p.h_k * p.n_q) return;
  const int row = int(unit % p.n_q);
  const int g = int((unit / p.n_q) % p.h_k);
  const int b = int(unit / (int64_t(p.n_q) * p.h_k));
  const float4* op = reinterpret_cast<const float4*>(p.o_part + part_index(p, b, 0, g, row) * D) + lane;
  const int64_t split_stride = int64_t(p.h_k) * p.n_q * (D / 4);  // in float4
  const int tq = row / p.h_r, h = g * p.h_r + row % p.h_r;

  float m0 = -INFINITY, l0 = 0.f;
  if (lane < p.max_splits) {
    const int64_t idx = part_index(p, b, lane, g, row);
    m0 = p.m_part[idx];
    l0 = p.l_part[idx];
  }
  float4 pre[kPre][kV];
#pragma unroll
  for (int k = 0; k < kPre; ++k)
#pragma unroll
    for (int v = 0; v < kV; ++v)
      pre[k][v] = k < p.max_splits ? op[int64_t(k) * split_stride + v * 32] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float vd = kv_descale(p.v_descale, p.ds_seq, p.ds_head, b, g) * p.v_fmt;
  float4 om[kV];
#pragma unroll
  for (int v = 0; v < kV; ++v)
    om[v] = p.o_mul ? reinterpret_cast<const float4*>(p.o_mul + int64_t(h) * D)[lane + 32 * v] : make_float4(1.f, 1.f, 1.f, 1.f);
  const int ns = min(p.n_splits[b], p.max_splits);
  if (ns <= 1) return;  // single split: the decode kernel wrote the output directly
  const int L = p.seq_lens[b];
  if (L <= 0) return;
  const int64_t span = int64_t(p.chunk_tiles) * kKvTile;
  const int live = int(min(int64_t(ns), (int64_t(L) + span - 1) / span));  // splits with >= 1 key

  // max logit over the live splits
  if (lane >= live) m0 = -INFINITY;
  float M = m0;
  for (int s = lane + 32; s < live; s += 32) M = fmaxf(M, p.m_part[part_index(p, b, s, g, row)]);
  M = warp_max(M);
  auto weight = [&](float ms, float ls) { return (M == -INFINITY || ms == -INFINITY) ? 0.f : fast_exp2(ms - M) * ls; };

  float4 acc[kV];
#pragma unroll
  for (int v = 0; v < kV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](float w, const float4& o, int v) {
    acc[v].x = fmaf(w, o.x, acc[v].x);
    acc[v].y = fmaf(w, o.y, acc[v].y);
    acc[v].z = fmaf(w, o.z, acc[v].z);
    acc[v].w = fmaf(w, o.w, acc[v].w);
  };
  // splits 0 .. 31: weight in lane s
  const float w0 = lane < live ? weight(m0, l0) : 0.f;
  float wsum = w0;
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const float wk = __shfl_sync(0xFFFFFFFFu, w0, k);
    if (k < live)
#pragma unroll
      for (int v = 0; v < kV; ++v) add(wk, pre[k][v], v);
  }
  const int n0 = min(live, 32);
#pragma unroll 4
  for (int s = kPre; s < n0; ++s) {
    const float ws = __shfl_sync(0xFFFFFFFFu, w0, s);
#pragma unroll
    for (int v = 0; v < kV; ++v) add(ws, op[int64_t(s) * split_stride + v * 32], v);
  }
  // splits 32 and up, 32 at a time
  for (int base = 32; base < live; base += 32) {
    const int s = base + lane;
    float wl = 0.f;
    if (s < live) {
      const int64_t idx = part_index(p, b, s, g, row);
      wl = weight(p.m_part[idx], p.l_part[idx]);
    }
    wsum += wl;
    const int n = min(live - base, 32);
    for (int j = 0; j < n; ++j) {
      const float ws = __shfl_sync(0xFFFFFFFFu, wl, j);
#pragma unroll
      for (int v = 0; v < kV; ++v) add(ws, op[int64_t(base + j) * split_stride + v * 32], v);
    }
  }
  wsum = warp_sum(wsum);

  auto fin = [&](float a) { return wsum > 0.f ? a / wsum * vd : 0.f; };
  uint16_t* out = p.out + int64_t(b * p.q_len + tq) * p.out_ts + int64_t(h) * p.out_hs;
#pragma unroll
  for (int v = 0; v < kV; ++v) {
    float x0 = fin(acc[v].x), x1 = fin(acc[v].y), x2 = fin(acc[v].z), x3 = fin(acc[v].w);
    if (p.o_mul) {
      x0 *= om[v].x;
      x1 *= om[v].y;
      x2 *= om[v].z;
      x3 *= om[v].w;
    }
    uint2 packed;
    packed.x = uint32_t(float_to_out_bits(x0, p.out_f16)) | (uint32_t(float_to_out_bits(x1, p.out_f16)) << 16);
    packed.y = uint32_t(float_to_out_bits(x2, p.out_f16)) | (uint32_t(float_to_out_bits(x3, p.out_f16)) << 16);
    *reinterpret_cast<uint2*>(out + 4 * lane + 128 * v) = packed;
  }
  if (p.lse && lane == 0)
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
  const int64_t units = int64_t(p.num_seqs) * p.h_k * p.n_q;
  const bool wide = units < sms;
  constexpr int kRows = 8;
  if (wide) {
    cfg.blockDim = dim3(4 * p.d);
    cfg.dynamicSmemBytes = size_t(p.max_splits) * sizeof(float);
  } else {
    if ((units + kRows - 1) / kRows > INT32_MAX) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(unsigned((units + kRows - 1) / kRows));
    cfg.blockDim = dim3(32 * kRows);
    cfg.dynamicSmemBytes = 0;
  }
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // four groups and at most 64 splits: all loads in one round
  const bool spec = p.max_splits <= 64;
  if (!wide)
    return p.d == 256 ? cudaLaunchKernelEx(&cfg, merge_rows_kernel<256, kRows>, p)
                      : cudaLaunchKernelEx(&cfg, merge_rows_kernel<128, kRows>, p);
  if (p.d == 256)
    return spec ? cudaLaunchKernelEx(&cfg, merge_kernel<256, 4, 16>, p) : cudaLaunchKernelEx(&cfg, merge_kernel<256, 4, 0>, p);
  return spec ? cudaLaunchKernelEx(&cfg, merge_kernel<128, 4, 16>, p) : cudaLaunchKernelEx(&cfg, merge_kernel<128, 4, 0>, p);
}

}  // namespace mj
