// mj_write_kv kernel: quantize the new tokens' K/V rows into the paged caches.
//
// The write that precedes a decode step (MjolnirImpl.do_kv_cache_update on
// the mjolnir/backend.py page): token t's row of KV head g goes to page
// slot / page_size, row slot % page_size; code = fmt(x / scale), with one
// scale per tensor or per KV head (e4m3) or per (KV head, channel) (packed
// e2m3, the channel scales of _install_fp6_scales; e3m2 and e2m1 likewise).
// The quotient is IEEE
// float32 (__fdiv_rn) and the rounding to the cache format is to nearest,
// ties to even, saturating, so the bytes are identical to that recipe.
//
// HBM-bound: each thread reads one 16-byte chunk of bf16 of K and of V
// (8 channels; two chunks for the packed formats) and writes their codes once.
// Consecutive threads take consecutive chunks of a row, and rows of
// consecutive heads and tokens, so both the loads and the stores are
// coalesced.
#include <cuda_fp8.h>

#include <algorithm>

#include <atomic>

#include "mj_device.cuh"
#include "mj_internal.h"

namespace mj {

namespace {

constexpr int kThreads = 256;

// e2m3 code of y: round to nearest, ties to even, saturating at 7.5; the
// sign bit (bit 5) follows the sign of y. Magnitudes below 1 are subnormal
// multiples of 1/8; at or above 1 each binade [2^e, 2^(e+1)) has 8 steps of
// 2^e / 8. The scalings by powers of two are exact, so the only rounding is
// the one __float2uint_rn (to nearest even) does; a mantissa that rounds up
// to 8 carries into the next binade's code, which is the correct result.
__device__ __forceinline__ uint32_t e2m3_code(float y) {
  const float a = fminf(fabsf(y), 7.5f);
  uint32_t c;
  if (a < 1.0f) {
    c = __float2uint_rn(a * 8.0f);  // 0 .. 8 (8 = 1.0, the first normal)
  } else {
    const int e = a >= 4.0f ? 2 : (a >= 2.0f ? 1 : 0);
    const float m = a * __int_as_float((127 - e) << 23);  // a / 2^e, in [1, 2)
    c = (uint32_t(e + 1) << 3) + __float2uint_rn((m - 1.0f) * 8.0f);
  }
  return c | (signbit(y) ? 0x20u : 0u);
}

// e3m2 code of y: round to nearest, ties to even, saturating at 28; sign bit
// 5. Below 0.25 the subnormal grid is k/16; each binade [2^e, 2^(e+1)),
// e = -2 .. 4, has 4 steps of 2^e / 4 (code (e + 3) * 4 + step). As in
// e2m3_code the scalings are exact and __float2uint_rn is the one rounding.
__device__ __forceinline__ uint32_t e3m2_code(float y) {
  const float a = fminf(fabsf(y), 28.0f);
  uint32_t c;
  if (a < 0.25f) {
    c = __float2uint_rn(a * 16.0f);  // 0 .. 4 (4 = 0.25, the first normal)
  } else {
    const int e = (__float_as_int(a) >> 23) - 127;          // floor(log2 a), -2 .. 4
    const float m = a * __int_as_float((127 - e) << 23);    // a / 2^e, in [1, 2)
    c = (uint32_t(e + 3) << 2) + __float2uint_rn((m - 1.0f) * 4.0f);
  }
  return c | (signbit(y) ? 0x20u : 0u);
}

// e2m1 code of y: round to nearest, ties to even, saturating at 6; sign bit 3.
// Below 1 the grid is k/2; binades [1, 2), [2, 4), [4, 8) have 2 steps each.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fminf(fabsf(y), 6.0f);
  uint32_t c;
  if (a < 1.0f) {
    c = __float2uint_rn(a * 2.0f);  // 0 .. 2 (2 = 1.0)
  } else {
    const int e = a >= 4.0f ? 2 : (a >= 2.0f ? 1 : 0);
    const float m = a * __int_as_float((127 - e) << 23);  // a / 2^e, in [1, 2)
    c = (uint32_t(e + 1) << 1) + __float2uint_rn((m - 1.0f) * 2.0f);
  }
  return c | (signbit(y) ? 0x8u : 0u);
}

__device__ __forceinline__ void bf16x8_to_float(uint4 v, float x[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

struct WriteParams {
  const uint16_t* key;
  const uint16_t* value;
  int64_t k_ts, k_hs, v_ts, v_hs;
  const int64_t* slots;
  int num_tokens, h_k, d;
  int page_size;
  int64_t num_slots;  // num_pages * page_size
  uint8_t* k_cache;
  uint8_t* v_cache;
  int64_t k_sp, k_st, k_sh, v_sp, v_st, v_sh;
  const float* k_scale;
  const float* v_scale;
  int scale_per_head;
  uint32_t* status;
};

// Quantize one loaded chunk (CH channels of a K or V row) and store its codes.
// e4m3: in[0] holds 8 channels; the packed formats: in[0..1] hold 16.
template <int F>
__device__ __forceinline__ void quantize_store(const uint4* in, const float* scale, uint8_t* dst, int c) {
  if constexpr (F == MJ_KV_E4M3) {
    float x[8];
    bf16x8_to_float(in[0], x);
    const float s = scale[0];
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[4 * k], s), __fdiv_rn(x[4 * k + 1], s)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(x[4 * k + 2], s), __fdiv_rn(x[4 * k + 3], s)), __NV_SATFINITE, __NV_E4M3);
      w[k] = uint32_t(lo) | (uint32_t(hi) << 16);
    }
    *reinterpret_cast<uint2*>(dst + c * 8) = make_uint2(w[0], w[1]);
  } else if constexpr (F == MJ_KV_E2M1) {
    // 16 codes, code k at bits [4k, 4k + 4) of 8 little-endian bytes
    float x[16];
    bf16x8_to_float(in[0], x);
    bf16x8_to_float(in[1], x + 8);
    const float4* sc = reinterpret_cast<const float4*>(scale + c * 16);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 s4 = sc[q];
      const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int idx = 4 * q + k;
        w[idx >> 3] |= e2m1_code(__fdiv_rn(x[idx], sv[k])) << (4 * (idx & 7));
      }
    }
    *reinterpret_cast<uint2*>(dst + c * 8) = make_uint2(w[0], w[1]);
  } else {
    float x[16];
    bf16x8_to_float(in[0], x);
    bf16x8_to_float(in[1], x + 8);
    const float4* sc = reinterpret_cast<const float4*>(scale + c * 16);
    // code k of the chunk at bits [6k, 6k + 6) of a 96-bit little-endian group
    uint64_t lo = 0, hi = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 s4 = sc[q];
      const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int idx = 4 * q + k, bit = 6 * idx;
        const float q6 = __fdiv_rn(x[idx], sv[k]);
        const uint64_t code = F == MJ_KV_E2M3 ? e2m3_code(q6) : e3m2_code(q6);
        if (bit < 64) {
          lo |= code << bit;
          if (bit + 6 > 64) hi |= code >> (64 - bit);
        } else {
          hi |= code << (bit - 64);
        }
      }
    }
    uint32_t* d32 = reinterpret_cast<uint32_t*>(dst + c * 12);
    d32[0] = uint32_t(lo);
    d32[1] = uint32_t(lo >> 32);
    d32[2] = uint32_t(hi);
  }
}

// One work item per (token, head, chunk of CH channels), K and V: CH = 8 for
// e4m3 (8 codes = 8 bytes), 16 for the packed formats (16 codes = 12 bytes,
// or 8 for e2m1). A thread takes
// U items a stride apart and issues all their loads before any store, so
// enough bytes are in flight to cover the memory latency (the stores may
// alias the inputs as far as the compiler knows, so it would not reorder
// them itself). The row index (token, head) fits in 32 bits (checked on the
// host).
template <int F, int D>
__global__ void __launch_bounds__(kThreads) write_kv_kernel(WriteParams p) {
  constexpr bool PK = F != MJ_KV_E4M3;  // packed (channel-scaled) format
  constexpr int CH = PK ? 16 : 8;
  constexpr int NCH = D / CH;  // chunks per row
  constexpr int NV = CH / 8;          // 16-byte loads per chunk of one side
  constexpr int U = PK ? 2 : 4;       // items per thread per round
  const uint64_t total = uint64_t(uint32_t(p.num_tokens) * uint32_t(p.h_k)) * NCH;
  const uint64_t stride = uint64_t(gridDim.x) * kThreads;
  for (uint64_t base = uint64_t(blockIdx.x) * kThreads + threadIdx.x; base < total; base += U * stride) {
    uint4 kin[U][NV], vin[U][NV];
    int64_t slot[U];
    int tok[U], head[U], chunk[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t i = base + u * stride;
      slot[u] = -1;
      if (i < total) {
        const uint32_t row = uint32_t(i / NCH);
        chunk[u] = int(i % NCH);
        tok[u] = int(row / uint32_t(p.h_k));
        head[u] = int(row - uint32_t(tok[u]) * uint32_t(p.h_k));
        slot[u] = p.slots[tok[u]];
        const uint4* ks = reinterpret_cast<const uint4*>(p.key + tok[u] * p.k_ts + head[u] * p.k_hs + chunk[u] * CH);
        const uint4* vs =
            reinterpret_cast<const uint4*>(p.value + tok[u] * p.v_ts + head[u] * p.v_hs + chunk[u] * CH);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          kin[u][v] = ks[v];
          vin[u][v] = vs[v];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (slot[u] < 0) continue;  // padding token (or no item)
      if (slot[u] >= p.num_slots) {
        if (p.status && chunk[u] == 0 && head[u] == 0) atomicOr(p.status, kStatusBadPage);
        continue;
      }
      const int g = head[u];
      const int64_t page = slot[u] / p.page_size, prow = slot[u] % p.page_size;
      const int s_idx = PK ? g * D : (p.scale_per_head ? g : 0);
      quantize_store<F>(kin[u], p.k_scale + s_idx, p.k_cache + page * p.k_sp + prow * p.k_st + g * p.k_sh,
                           chunk[u]);
      quantize_store<F>(vin[u], p.v_scale + s_idx, p.v_cache + page * p.v_sp + prow * p.v_st + g * p.v_sh,
                           chunk[u]);
    }
  }
}

template <int D>
void launch_format(int kv_format, unsigned nb, const WriteParams& p, cudaStream_t stream) {
  switch (kv_format) {
    case MJ_KV_E2M3: write_kv_kernel<MJ_KV_E2M3, D><<<nb, kThreads, 0, stream>>>(p); break;
    case MJ_KV_E3M2: write_kv_kernel<MJ_KV_E3M2, D><<<nb, kThreads, 0, stream>>>(p); break;
    case MJ_KV_E2M1: write_kv_kernel<MJ_KV_E2M1, D><<<nb, kThreads, 0, stream>>>(p); break;
    default: write_kv_kernel<MJ_KV_E4M3, D><<<nb, kThreads, 0, stream>>>(p); break;
  }
}

}  // namespace

cudaError_t launch_write_kv(const mj_write_kv_args& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  WriteParams p;
  p.key = static_cast<const uint16_t*>(a.key);
  p.value = static_cast<const uint16_t*>(a.value);
  p.k_ts = a.key_tok_stride;
  p.k_hs = a.key_head_stride;
  p.v_ts = a.value_tok_stride;
  p.v_hs = a.value_head_stride;
  p.slots = a.slot_mapping;
  p.num_tokens = a.num_tokens;
  p.h_k = a.h_k;
  p.d = a.d;
  p.page_size = a.page_size;
  p.num_slots = a.num_pages * a.page_size;
  p.k_cache = static_cast<uint8_t*>(a.k_cache);
  p.v_cache = static_cast<uint8_t*>(a.v_cache);
  p.k_sp = a.k_stride_page;
  p.k_st = a.k_stride_token;
  p.k_sh = a.k_stride_head;
  p.v_sp = a.v_stride_page;
  p.v_st = a.v_stride_token;
  p.v_sh = a.v_stride_head;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.scale_per_head = a.scale_per_head;
  p.status = a.status;
  const bool packed = a.kv_format != MJ_KV_E4M3;
  const int64_t work = int64_t(a.num_tokens) * a.h_k * (a.d / (packed ? 16 : 8));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // SM count per device, looked up once (host threads may race)
  static std::atomic<int> sm_count[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  // enough blocks to fill every SM (8 x 256 threads each), fewer for small writes
  const int64_t blocks = std::min<int64_t>((work + kThreads - 1) / kThreads, int64_t(sms) * 8);
  if (a.d == 256)
    launch_format<256>(a.kv_format, unsigned(blocks), p, stream);
  else
    launch_format<128>(a.kv_format, unsigned(blocks), p, stream);
  return cudaGetLastError();
}

}  // namespace mj
