// mj_quantize_q kernel: dynamic per-(request, KV head) e4m3 quantization of Q.
//
// Follows the fp8-Q branch of the "Q" block of T5DecodeRunner.run
// (mjolnir/runner.py page): x = float(q) [* q_mul]; amax over the request's
// q_len x h_r x d values of KV head g, clamped at 1e-6; scale = amax/448;
// code = e4m3_rne(x/scale); packed row t*h_r + r. Every step is float32 with
// round-to-nearest (explicit __fmul_rn / __fdiv_rn: no contraction, no
// approximate division), so the codes and scales are bit-identical to the
// float32 recipe.
#include <cuda_fp8.h>

#include "mj_device.cuh"
#include "mj_internal.h"

namespace mj {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float load_x(const QuantParams& p, int b, int g, int i) {
  const int per_tok = p.h_r * p.d;
  const int t = i / per_tok;
  const int r = (i / p.d) % p.h_r;
  const int c = i % p.d;
  const int h = g * p.h_r + r;
  const int64_t off = int64_t(b * p.q_len + t) * p.q_ts + int64_t(h) * p.q_hs + c;
  float x = bf16_bits_to_float(p.q[off]);
  if (p.q_mul) x = __fmul_rn(x, p.q_mul[int64_t(h) * p.d + c]);
  return x;
}

__global__ void __launch_bounds__(kThreads) quantize_q_kernel(QuantParams p) {
  // The decode kernel that follows waits for this grid before it reads Q
  // (griddepcontrol.wait); let it start its KV streaming right away.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int g = blockIdx.y;
  const int n = p.q_len * p.h_r * p.d;

  float amax = 0.f;
  for (int i = threadIdx.x; i < n; i += kThreads) amax = fmaxf(amax, fabsf(load_x(p, b, g, i)));
  amax = warp_max(amax);
  __shared__ float red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  amax = fmaxf(amax, 1e-6f);
  const float scale = __fdiv_rn(amax, 448.0f);

  uint8_t* codes = p.codes + (int64_t(b) * p.h_k + g) * p.n_q * p.d;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const float y = __fdiv_rn(load_x(p, b, g, i), scale);
    const int t = i / (p.h_r * p.d);
    const int r = (i / p.d) % p.h_r;
    const int c = i % p.d;
    codes[int64_t(t * p.h_r + r) * p.d + c] =
        static_cast<uint8_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
  }
  if (threadIdx.x == 0) p.descale[int64_t(b) * p.h_k + g] = scale;
}

}  // namespace

cudaError_t launch_quantize_q(const QuantParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  dim3 grid(p.num_seqs, p.h_k);
  quantize_q_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mj
