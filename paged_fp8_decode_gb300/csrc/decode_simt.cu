// CUDA-core variant of mj_decode_attention.
//
// One CTA (4 warps) per (work row, KV head, query-row tile). Each warp walks
// 32-key blocks of the work row's key range; lane j owns key j of the block
// for S = Q.K^T (the whole K row through 16-byte loads) and channels
// 128*h + 4*lane .. 128*h + 4*lane+3 of each 128-channel half h for
// O += P.V (coalesced 128-byte V reads per key and half). The
// online softmax runs per warp in the log2 domain; the four warps' (m, l, O)
// are merged in shared memory at the end. Keys at or past the request's
// device seq_len are never read, so stale or poisoned page tails cannot leak
// into the result.
//
// This is the generic path: any row tile up to 32 (16 with D = 256), any
// strides, e4m3 or packed e2m3 / e3m2 / e2m1, D = 128 or 256, e4m3 Q codes or
// bf16 Q as is.
// The tensor-core kernel is the fast path.
#include <cuda_fp8.h>

#include "mj_device.cuh"
#include "mj_internal.h"

namespace mj {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

// Four 6-bit (e2m3 / e3m2) or 4-bit (e2m1) codes, one per byte, widened to
// e4m3 codes (value / kv_widen_factor).
__device__ __forceinline__ uint32_t widen4_codes(uint32_t four_codes, int kv_format) {
  if (kv_format == MJ_KV_E2M3) return e2m3x4_to_e4m3x4(four_codes);
  if (kv_format == MJ_KV_E3M2) return e3m2x4_to_e4m3x4(four_codes);
  return e2m1x4_to_e4m3x4(four_codes);
}

// Codes 16*i .. 16*i+15 of one K row as floats (e4m3: bytes 16i..16i+15;
// e2m3 / e3m2: packed bytes 12i..12i+11, e2m1: bytes 8i..8i+7, widened to e4m3).
__device__ __forceinline__ void load_k16(const uint8_t* row, int kv_format, int i, float k[16]) {
  if (kv_format == MJ_KV_E4M3) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + i);
    e4m3x4_to_float(v.x, k + 0);
    e4m3x4_to_float(v.y, k + 4);
    e4m3x4_to_float(v.z, k + 8);
    e4m3x4_to_float(v.w, k + 12);
  } else if (kv_format == MJ_KV_E2M1) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(row) + i);
    e4m3x4_to_float(e2m1x4_to_e4m3x4(spread4x4(v.x & 0xFFFFu)), k + 0);
    e4m3x4_to_float(e2m1x4_to_e4m3x4(spread4x4(v.x >> 16)), k + 4);
    e4m3x4_to_float(e2m1x4_to_e4m3x4(spread4x4(v.y & 0xFFFFu)), k + 8);
    e4m3x4_to_float(e2m1x4_to_e4m3x4(spread4x4(v.y >> 16)), k + 12);
  } else {
    const uint32_t* r32 = reinterpret_cast<const uint32_t*>(row) + 3 * i;
    const uint32_t w0 = __ldg(r32), w1 = __ldg(r32 + 1), w2 = __ldg(r32 + 2);
    const uint32_t g0 = w0 & 0xFFFFFFu;
    const uint32_t g1 = __funnelshift_r(w0, w1, 24) & 0xFFFFFFu;
    const uint32_t g2 = __funnelshift_r(w1, w2, 16) & 0xFFFFFFu;
    const uint32_t g3 = w2 >> 8;
    e4m3x4_to_float(widen4_codes(spread6x4(g0), kv_format), k + 0);
    e4m3x4_to_float(widen4_codes(spread6x4(g1), kv_format), k + 4);
    e4m3x4_to_float(widen4_codes(spread6x4(g2), kv_format), k + 8);
    e4m3x4_to_float(widen4_codes(spread6x4(g3), kv_format), k + 12);
  }
}

// Channels 4*j .. 4*j+3 of one V row.
__device__ __forceinline__ void load_v4(const uint8_t* row, int kv_format, int j, float v[4]) {
  if (kv_format == MJ_KV_E4M3) {
    e4m3x4_to_float(__ldg(reinterpret_cast<const uint32_t*>(row) + j), v);
  } else if (kv_format == MJ_KV_E2M1) {
    const uint32_t h = __ldg(reinterpret_cast<const uint16_t*>(row) + j);
    e4m3x4_to_float(e2m1x4_to_e4m3x4(spread4x4(h)), v);
  } else {
    const uint8_t* p = row + 3 * j;
    const uint32_t g = uint32_t(__ldg(p)) | (uint32_t(__ldg(p + 1)) << 8) | (uint32_t(__ldg(p + 2)) << 16);
    e4m3x4_to_float(widen4_codes(spread6x4(g), kv_format), v);
  }
}

template <int NR, int D>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeParams p) {
  constexpr int DH = D / 128;  // 128-channel halves; thread / lane work repeats per half
  __shared__ __align__(16) float qs[NR][D];  // Q rows, later the O accumulator
  __shared__ float ps[kWarps][32][NR];              // P of each warp's 32-key block
  __shared__ float red_m[kWarps][NR], red_l[kWarps][NR];
  __shared__ int page_of[kWarps][32];

  const int g = blockIdx.y;
  const int4 w = reinterpret_cast<const int4*>(p.work)[blockIdx.x];
  const int b = w.x;
  if (w.z <= w.y || b < 0 || b >= p.num_seqs) return;
  if (p.with_reduction && (w.w < 0 || w.w >= p.max_splits || b >= p.part_seqs)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadPlan);
    return;
  }
  const int L = p.seq_lens[b];
  if (L <= 0) return;
  const int64_t k0 = int64_t(w.y) * kKvTile;
  const int64_t k1 = min(int64_t(w.z) * kKvTile, int64_t(L));
  if (k1 <= k0) return;
  const int r0 = blockIdx.z * p.tw;
  const int nr = min(p.tw, p.n_q - r0);
  if (nr <= 0) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Q of this row tile -> shared floats (rows >= nr are zero): the e4m3
  // codes (row t*h_r + r of the packed tile), the bf16 Q as is (token t,
  // query head g*h_r + r), or that bf16 Q quantized here with mj_quantize_q's
  // recipe (q_mul, amax over all q_len*h_r rows of (b, g), amax/448, e4m3
  // round-to-nearest-even satfinite; IEEE float32 steps throughout).
  float qd = 1.f;  // descale of the staged Q values
  const uint8_t* qrow = p.q_codes + ((int64_t(b) * p.h_k + g) * p.n_q + r0) * D;
  auto q_in = [&](int rr, int c) {  // bf16 Q of packed row rr, channel c (times q_mul)
    const int tq = rr / p.h_r, h = g * p.h_r + rr % p.h_r;
    float x = bf16_bits_to_float(p.q_bf16[int64_t(b * p.q_len + tq) * p.q_ts + int64_t(h) * p.q_hs + c]);
    if (p.q_mul) x = __fmul_rn(x, p.q_mul[int64_t(h) * D + c]);
    return x;
  };
  if (p.q_mode == MJ_Q_FP8_FUSED) {
    // 128 threads, channels tid + 128*h; the tile's rows once, into
    // registers; the rows of (b, g) outside the tile only count towards the amax
    float xr[DH][NR];
    float am = 0.f;
#pragma unroll
    for (int hh = 0; hh < DH; ++hh) {
      const int c = tid + 128 * hh;
#pragma unroll
      for (int r = 0; r < NR; ++r) xr[hh][r] = r < nr ? q_in(r0 + r, c) : 0.f;
#pragma unroll
      for (int r = 0; r < NR; ++r) am = fmaxf(am, fabsf(xr[hh][r]));
      for (int rr = 0; rr < p.n_q; ++rr)
        if (rr < r0 || rr >= r0 + nr) am = fmaxf(am, fabsf(q_in(rr, c)));
    }
    am = warp_max(am);
    if (lane == 0) red_m[warp][0] = am;
    __syncthreads();
    am = fmaxf(fmaxf(red_m[0][0], red_m[1][0]), fmaxf(red_m[2][0], red_m[3][0]));
    qd = __fdiv_rn(fmaxf(am, 1e-6f), 448.0f);
#pragma unroll
    for (int hh = 0; hh < DH; ++hh) {
#pragma unroll
      for (int row = 0; row < NR; ++row) {
        float v = 0.f;
        if (row < nr) {
          __nv_fp8_e4m3 code;
          code.__x = __nv_cvt_float_to_fp8(__fdiv_rn(xr[hh][row], qd), __NV_SATFINITE, __NV_E4M3);
          v = float(code);
        }
        qs[row][tid + 128 * hh] = v;
      }
    }
  } else {
    for (int i = tid; i < NR * D / 4; i += kThreads) {
      const int row = i / (D / 4), c4 = i % (D / 4);
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (row < nr) {
        if (p.q_mode == MJ_Q_BF16) {
          const int rr = r0 + row, tq = rr / p.h_r, h = g * p.h_r + rr % p.h_r;
          const uint2 u = *reinterpret_cast<const uint2*>(p.q_bf16 + int64_t(b * p.q_len + tq) * p.q_ts +
                                                          int64_t(h) * p.q_hs + 4 * c4);
          v[0] = __uint_as_float(u.x << 16);
          v[1] = __uint_as_float(u.x & 0xFFFF0000u);
          v[2] = __uint_as_float(u.y << 16);
          v[3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
          e4m3x4_to_float(reinterpret_cast<const uint32_t*>(qrow + row * D)[c4], v);
        }
      }
      *reinterpret_cast<float4*>(&qs[row][4 * c4]) = make_float4(v[0], v[1], v[2], v[3]);
    }
    if (p.q_mode == MJ_Q_FP8) qd = p.q_descale[int64_t(b) * p.h_k + g];
  }
  __syncthreads();

  const float kd = kv_descale(p.k_descale, p.ds_seq, p.ds_head, b, g);
  const float scale = qd * kd * p.qk_scale_log2;
  const int64_t causal_base = int64_t(L) - p.q_len;  // query t sees key j iff j <= L - q_len + t

  float m[NR], l[NR], o[NR][4 * DH];  // o[r][4h + e]: channel 128h + 4*lane + e
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < 4 * DH; ++e) o[r][e] = 0.f;
  }

  const int64_t kbase_head = int64_t(g) * p.k_sh;
  const int64_t vbase_head = int64_t(g) * p.v_sh;
  const int32_t* bt = p.block_table + int64_t(b) * p.bt_stride;

  for (int64_t kb = k0 + int64_t(warp) * 32; kb < k1; kb += kWarps * 32) {
    const int64_t key = kb + lane;
    const bool valid = key < k1;
    int page = 0;
    bool page_ok = false;
    if (valid) {
      page = bt[key / p.page_size];
      page_ok = page >= 0 && int64_t(page) < p.num_pages;
      if (!page_ok) atomicOr(p.status, kStatusBadPage);
    }
    page_of[warp][lane] = page_ok ? page : -1;

    float t[NR];
    if (page_ok) {
      const int slot = int(key % p.page_size);
      const uint8_t* krow = p.k_cache + int64_t(page) * p.k_sp + int64_t(slot) * p.k_st + kbase_head;
      float acc[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) acc[r] = 0.f;
#pragma unroll 1
      for (int i = 0; i < D / 16; ++i) {
        float kf[16];
        load_k16(krow, p.kv_format, i, kf);
#pragma unroll
        for (int c = 0; c < 16; c += 4) {
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            const float4 q4 = *reinterpret_cast<const float4*>(&qs[r][16 * i + c]);
            acc[r] = fmaf(q4.x, kf[c], acc[r]);
            acc[r] = fmaf(q4.y, kf[c + 1], acc[r]);
            acc[r] = fmaf(q4.z, kf[c + 2], acc[r]);
            acc[r] = fmaf(q4.w, kf[c + 3], acc[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const int tq = (r0 + r) / p.h_r;
        const bool vis = r < nr && (!p.causal || key <= causal_base + tq);
        t[r] = vis ? acc[r] * scale : -INFINITY;
      }
    } else {
#pragma unroll
      for (int r = 0; r < NR; ++r) t[r] = -INFINITY;
    }

#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float mx = warp_max(t[r]);
      const float m_new = fmaxf(m[r], mx);
      float alpha, pr;
      if (m_new == -INFINITY) {
        alpha = 1.f;
        pr = 0.f;
      } else {
        alpha = fast_exp2(m[r] - m_new);
        pr = fast_exp2(t[r] - m_new);
      }
      m[r] = m_new;
      l[r] = l[r] * alpha + pr;
#pragma unroll
      for (int e = 0; e < 4 * DH; ++e) o[r][e] *= alpha;
      ps[warp][lane][r] = pr;
    }
    __syncwarp();

    const int nkeys = int(min(int64_t(32), k1 - kb));
    for (int kk = 0; kk < nkeys; ++kk) {
      const int pg = page_of[warp][kk];
      if (pg < 0) continue;
      const int slot = int((kb + kk) % p.page_size);
      const uint8_t* vrow = p.v_cache + int64_t(pg) * p.v_sp + int64_t(slot) * p.v_st + vbase_head;
      float v[4 * DH];
#pragma unroll
      for (int hh = 0; hh < DH; ++hh) load_v4(vrow, p.kv_format, 32 * hh + lane, v + 4 * hh);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const float pr = ps[warp][kk][r];
#pragma unroll
        for (int e = 0; e < 4 * DH; ++e) o[r][e] = fmaf(pr, v[e], o[r][e]);
      }
    }
    __syncwarp();
  }

  // ---- merge the four warps ------------------------------------------------
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const float ls = warp_sum(l[r]);
    if (lane == 0) {
      red_m[warp][r] = m[r];
      red_l[warp][r] = ls;
    }
  }
  __syncthreads();  // also: every warp is done reading qs

  float f[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float M = red_m[0][r];
#pragma unroll
    for (int w2 = 1; w2 < kWarps; ++w2) M = fmaxf(M, red_m[w2][r]);
    f[r] = (m[r] == -INFINITY) ? 0.f : fast_exp2(m[r] - M);
  }
  for (int w2 = 0; w2 < kWarps; ++w2) {
    if (warp == w2) {
#pragma unroll
      for (int r = 0; r < NR; ++r) {
#pragma unroll
        for (int hh = 0; hh < DH; ++hh) {
          float4* dst = reinterpret_cast<float4*>(&qs[r][128 * hh + 4 * lane]);
          float4 cur = (w2 == 0) ? make_float4(0.f, 0.f, 0.f, 0.f) : *dst;
          cur.x = fmaf(o[r][4 * hh + 0], f[r], cur.x);
          cur.y = fmaf(o[r][4 * hh + 1], f[r], cur.y);
          cur.z = fmaf(o[r][4 * hh + 2], f[r], cur.z);
          cur.w = fmaf(o[r][4 * hh + 3], f[r], cur.w);
          *dst = cur;
        }
      }
    }
    __syncthreads();
  }

  const bool direct = !p.with_reduction || p.n_splits[b] <= 1;
  const float vd = kv_descale(p.v_descale, p.ds_seq, p.ds_head, b, g) * p.v_fmt;
  for (int r = 0; r < nr; ++r) {
    float M = red_m[0][r];
    for (int w2 = 1; w2 < kWarps; ++w2) M = fmaxf(M, red_m[w2][r]);
    float Lt = 0.f;
    if (M != -INFINITY)
      for (int w2 = 0; w2 < kWarps; ++w2)
        if (red_m[w2][r] != -INFINITY) Lt += red_l[w2][r] * fast_exp2(red_m[w2][r] - M);
    const int row = r0 + r;
#pragma unroll
    for (int hh = 0; hh < DH; ++hh) {
      const int c = tid + 128 * hh;  // 128 threads, channels c
      const float on = Lt > 0.f ? qs[r][c] / Lt : 0.f;
      if (direct) {
        const int tq = row / p.h_r, rr = row % p.h_r, h = g * p.h_r + rr;
        float val = on * vd;
        if (p.o_mul) val *= p.o_mul[int64_t(h) * D + c];
        p.out[int64_t(b * p.q_len + tq) * p.out_ts + int64_t(h) * p.out_hs + c] = float_to_out_bits(val, p.out_f16);
        if (p.lse && c == 0)
          p.lse[(int64_t(b) * p.h_k + g) * p.n_q + row] = Lt > 0.f ? (M + fast_log2(Lt)) * kLn2 : -INFINITY;
      } else {
        const int64_t idx = part_index(p, b, w.w, g, row);
        p.o_part[idx * D + c] = on;
        if (c == 0) {
          p.m_part[idx] = Lt > 0.f ? M : -INFINITY;
          p.l_part[idx] = Lt;
        }
      }
    }
  }
}

template <int D>
void launch_rows_simt(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  if (p.tw <= 4)
    decode_simt_kernel<4, D><<<grid, kThreads, 0, stream>>>(p);
  else if (p.tw <= 8)
    decode_simt_kernel<8, D><<<grid, kThreads, 0, stream>>>(p);
  else if (p.tw <= 16)
    decode_simt_kernel<16, D><<<grid, kThreads, 0, stream>>>(p);
  else if constexpr (D == 128)
    decode_simt_kernel<32, D><<<grid, kThreads, 0, stream>>>(p);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams& p0, cudaStream_t stream) {
  if (p0.num_work == 0) return cudaSuccess;
  DecodeParams p = p0;
  if (p.d == 256 && p.tw > 16) {
    // D = 256 keeps 16 rows per CTA (the O accumulator stays in registers):
    // a 32-row tile of the plan becomes two CTAs' worth of rows
    p.tw = 16;
    p.n_row_tiles = (p.n_q + 15) / 16;
  }
  dim3 grid(p.num_work, p.h_k, p.n_row_tiles);
  if (p.d == 256)
    launch_rows_simt<256>(p, grid, stream);
  else
    launch_rows_simt<128>(p, grid, stream);
  return cudaGetLastError();
}

}  // namespace mj
