#pragma once

// The tcgen05 decode kernel template and its launch helpers, shared by the
// translation units that instantiate it (decode_tc_*.cu: one per cache
// format / head size, compiled in parallel) and by decode_tc.cu, which holds
// the host-side checks, the tensor maps and the dispatch.
//
// Tensor-core variant of mj_decode_attention for sm_103a: TMA page streaming
// into a shared-memory ring, tcgen05.mma (kind f8f6f4, e4m3 x e4m3 -> f32) with
// accumulators in tensor memory, online softmax on CUDA cores.
//
// The README of the mjolnir-kernel package ("A decode step", item 3) describes
// the shape of this design for Jetson Thor: pages arrive by TMA in a
// shared-memory ring (evicted first from L2), the tensor cores keep the
// scores and the output in TMEM, and warpgroups do the softmax. This kernel is
// written for GB300 from that description:
//
// * One CTA per (work row, KV head, query-row tile); 7 warps (10 with packed
//   e2m3 / e3m2 / e2m1 KV):
//     warps 0, 6 TMA producers of the K and the V tiles: block-table lookups
//                (32 entries per warp load), one 4-D tensor-map load per
//                (page, head, 128-channel sub-tile) into the ring;
//     warp 1     TMEM allocation and the single-thread MMA issuer;
//     warps 2-5  softmax warpgroup: thread x owns TMEM lane x, i.e. key x of a
//                128-key tile for S and channel x (of each 128-channel half)
//                for O;
//     warps 7-9  packed KV only: widen each landed V tile to e4m3.
// * The ring alternates K and V tiles of 128 keys x D bytes (D / 128 sub-tiles
//   of 128 keys x 128 bytes), 128-byte swizzled by the TMA so that
//   tcgen05.mma reads them directly.
// * Both products are issued "keys as M" so that M = 128 fills the tensor
//   core even for a handful of query rows:
//     S^T[key][row] = K[key][:] . Q[row][:]       A = K tile (K-major), B = Q tile
//     O^T[d][col]  += V^T[d][key] . P^T[key][col] A = V tile (MN-major), B = P tile
// * P = 2^(t - m + 8) (at most 2^8.6) is written as four e4m3 terms in
//   separate N columns of the same PV product: pair A, hi = e4m3(p) and
//   lo = e4m3(p - hi), and, where p < 1/4, pair B, the same split of what
//   pair A left, (p - hi - lo) * 2^10; the epilogue adds pair B's columns
//   times 2^-10. Every p is then carried to within max(2^-8 p, 2^-20), so
//   keys far below the row's max keep their weight (pair A alone would round
//   everything 18 binades below the max to zero). l sums the p themselves.
//   The factor 2^8 cancels in O / l.
// * Keys at or past the device seq_len are masked by select on S; in a
//   request's last, partial tile the V producer warp also zeroes the V rows
//   past the end before the PV product (page tails may hold NaN codes, and
//   0 * NaN would reach O through the MMA).
// * The launch may overlap the preceding kernel (programmatic dependent
//   launch). Before its wait for that kernel, the producer warps ask L2 for
//   the CTA's first KV tiles (a prefetch returns no data, so a guess made
//   from inputs not yet final costs traffic, never correctness); a grid that
//   does not split lets the next kernel launch early in turn.
// * Every wait is bounded (2 s); a timeout raises a status bit and the CTA
//   unwinds, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cstddef>
#include <mutex>
#include <type_traits>

#include "mj_device.cuh"
#include "mj_internal.h"
#include "tc_ptx.cuh"

namespace mj {

namespace {

constexpr int kThreadsTc = 224;      // e4m3 KV: 7 warps
// packed KV (e2m3, e3m2, e2m1): + 3 V-widening warps (7-9). With warps 2-5 on the four SM
// sub-partitions, the widening work then spreads over three of them rather
// than two (two CTAs per SM keep at most five warps per sub-partition either
// way, so the register budget is the same).
constexpr int kThreadsTcFp6 = 320;
constexpr int kConvThreads = kThreadsTcFp6 - 7 * 32;
constexpr int kConvWarp0 = 7;
constexpr int kSoftmaxWarp0 = 2;     // warps 2-5: softmax warpgroup
constexpr int kVProducerWarp = 6;
// tiles a CTA asks L2 for before the programmatic-launch wait: more in the
// first wave, whose CTAs can start while the preceding kernel still runs (16
// when the grid is at most two waves, else 8), unless a split grid runs in
// several waves (measured: a deeper prefetch then costs the later waves more
// than it gives the first)
constexpr int kPrefetchTiles = 4, kPrefetchTilesFirstWave = 8, kPrefetchTilesShortGrid = 16;
constexpr int kTileBytes = kKvTile * 128;  // 128 keys x 128 bytes
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct TcSmem {
  // offsets (bytes) from the 1024-aligned dynamic shared-memory base
  uint32_t ring, q, p0, p1, ctrl, total;
};

// Shared-memory bytes of one 128-channel sub-tile of the Q tile (nqk rows).
__host__ __device__ constexpr uint32_t q_sub_bytes(int nqk) { return uint32_t((nqk * 128 + 1023) / 1024) * 1024u; }

// nsb: S / P buffers in flight (P buffer j at p0 + j * (p1 - p0)); dh: 128-channel
// sub-tiles per row (D / 128): a ring entry holds dh 16 KB sub-tiles, the Q
// tile dh sub-tiles of q_sub_bytes(nqk).
__host__ __device__ inline TcSmem tc_smem_layout(int stages, int nqk, int npv, int nsb, int dh) {
  TcSmem s;
  s.ring = 0;
  s.q = stages * dh * kTileBytes;
  s.p0 = s.q + dh * q_sub_bytes(nqk);
  s.p1 = s.p0 + ((npv * 128 + 1023) / 1024) * 1024;
  s.ctrl = s.p0 + nsb * (s.p1 - s.p0);
  s.total = s.ctrl + 3072;
  return s;
}

// control block inside the ctrl region
struct Ctrl {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t s_full[4];
  uint64_t p_full[4];
  uint64_t o_full[4];
  uint64_t red_bar[2];  // the 4 softmax warps have posted their row maxima (or their bound)
  uint64_t row_bar[2];  // ... their row maxima, after a bound exchange that did not settle
  uint64_t sum_bar;     // ... their row sums
  uint64_t drain;       // MMA drain after an abort
  uint64_t q_ready;     // the softmax warps have written the Q tile
  uint64_t vconv[16];   // packed KV: V tile of ring slot s widened to e4m3
  uint64_t v_tail;      // e4m3 KV: the last, partial V tile has its rows past the end zeroed
  uint32_t tmem_base;
  int abort;
  alignas(16) float red[2][4][32];  // per-tile row maxima of the 4 softmax warps (read as float4)
  alignas(16) float bound[2][4];    // per softmax warp: max over its rows and keys of (tile max - m_ref)
  alignas(16) float lsum[4][32];    // row sums of the 4 softmax warps
  float alpha[4][32];               // per softmax warp: the rescale factors of the current tiles
  float qamax[2][4];                // bf16 Q: per softmax warp, |x| max and |residual| max
};
static_assert(sizeof(Ctrl) <= 3072, "control block");
static_assert(offsetof(Ctrl, red) % 16 == 0 && offsetof(Ctrl, lsum) % 16 == 0 && offsetof(Ctrl, bound) % 16 == 0,
              "float4 access to red/lsum/bound");

// Reduce NR per-lane values over the 32 lanes of a warp, one row per lane
// group: a reduce-scatter (each step halves the rows a lane keeps and
// exchanges the other half) followed by a butterfly over the lanes that share
// a row. Row r ends up in lanes r*(32/NR) .. r*(32/NR) + 32/NR - 1. This takes
// NR - 1 + log2(32/NR) shuffles instead of 5*NR for independent butterflies.
template <int NR, bool MAX>
__device__ __forceinline__ float rs_reduce(float (&v)[NR], int lane) {
#pragma unroll
  for (int c = NR, m = 16; c > 1; c >>= 1, m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < c / 2; ++j) {
      const float send = upper ? v[j] : v[c / 2 + j];
      const float keep = upper ? v[c / 2 + j] : v[j];
      const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, m);
      v[j] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int m = 16 / NR; m > 0; m >>= 1) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, r, m);
    r = MAX ? fmaxf(r, o) : r + o;
  }
  return r;
}

__device__ __forceinline__ uint32_t p_byte_offset(int n, int key) {
  // P^T tile: row n (a B-matrix column), 128 keys, K-major, 128-byte swizzle
  return uint32_t(n) * 128u + ((uint32_t((key >> 4) ^ (n & 7))) << 4) + uint32_t(key & 15);
}

// Widen the 16 packed e2m3 codes of a 16-byte shared-memory chunk (12 bytes of
// little-endian bitstream, 4 bytes of padding, as TMA's 16U6_ALIGN16B type
// stores them) to 16 e4m3 codes worth 2^-6 times the e2m3 values: per code,
// the 5 magnitude bits keep their place and the sign moves from bit 5 to bit 7
// (an e2m3 code read as e4m3 with a zero-extended exponent is exactly 2^-6
// times its value, subnormals included). Every resulting code is finite.
__device__ __forceinline__ uint32_t widen4(uint32_t g) {
  // code k of g sits at bits [6k, 6k + 6): magnitude -> byte k bits 0-4, sign -> bit 7
  return (g & 0x1Fu) | ((g << 2) & 0x1F80u) | ((g << 4) & 0x1F8000u) | ((g << 6) & 0x1F800000u) |
         ((g << 8) & 0x80000000u);
}

// e3m2: the same 16U6_ALIGN16B chunk; each code widened to an e4m3 code worth
// 2^-4 times its value (the 5 magnitude bits move up one place, the sign to
// bit 7). e2m1: TMA's 16U4_ALIGN16B type stores 16 codes in the first 8 bytes
// of the chunk (code k at bits [4k, 4k + 4)) and 8 bytes of padding; each code
// is widened to an e4m3 code worth 2^-6 times its value.
template <int KF>
__device__ __forceinline__ uint4 widen_chunk(uint4 in) {
  uint4 o;
  if constexpr (KF == MJ_KV_E2M3) {
    o.x = widen4(in.x);
    o.y = widen4(__funnelshift_r(in.x, in.y, 24));
    o.z = widen4(__funnelshift_r(in.y, in.z, 16));
    o.w = widen4(in.z >> 8);
  } else if constexpr (KF == MJ_KV_E3M2) {
    o.x = e3m2x4_to_e4m3x4(spread6x4(in.x & 0xFFFFFFu));
    o.y = e3m2x4_to_e4m3x4(spread6x4(__funnelshift_r(in.x, in.y, 24) & 0xFFFFFFu));
    o.z = e3m2x4_to_e4m3x4(spread6x4(__funnelshift_r(in.y, in.z, 16) & 0xFFFFFFu));
    o.w = e3m2x4_to_e4m3x4(spread6x4(in.z >> 8));
  } else {
    o.x = e2m1x4_to_e4m3x4(spread4x4(in.x & 0xFFFFu));
    o.y = e2m1x4_to_e4m3x4(spread4x4(in.x >> 16));
    o.z = e2m1x4_to_e4m3x4(spread4x4(in.y & 0xFFFFu));
    o.w = e2m1x4_to_e4m3x4(spread4x4(in.y >> 16));
  }
  return o;
}

// kind::f8f6f4 operand type of a cache format's codes (instruction
// descriptor field): e4m3 0, e2m3 3, e3m2 4, e2m1 5.
__host__ __device__ constexpr uint32_t mma_kv_type(int kf) {
  return kf == MJ_KV_E2M3 ? 3u : (kf == MJ_KV_E3M2 ? 4u : (kf == MJ_KV_E2M1 ? 5u : 0u));
}

// TMEM columns a kernel instance uses: its S buffers (NQK columns each, two
// or four of them) and its D / 128 O accumulators (NPV columns each); and the
// power of two it allocates. An instance that needs all 512 columns must run
// alone on its SM (launch_tc sizes its shared memory so that it does).
__host__ __device__ constexpr int tc_nsb(int /*nr*/) { return 4; }  // S buffers in flight
// P buffers in shared memory: one per S buffer, except at 8 and 16 rows
// (tile pairs), where two (one pair) leave room for a 6-entry ring at two
// CTAs per SM at 8 rows and shrink the footprint at 16; the softmax then
// writes a pair's P only once the PV products of the pair before it are
// complete.
__host__ __device__ constexpr int tc_npb(int nr) { return (nr == 8 || nr == 16) ? 2 : tc_nsb(nr); }
__host__ __device__ constexpr int tc_tmem_cols_used(int nqk, int npv, int nr, int d) {
  return tc_nsb(nr) * nqk + (d / 128) * npv;
}
__host__ __device__ constexpr uint32_t tc_tmem_alloc_cols(int cols) {
  return cols <= 64 ? 64u : (cols <= 128 ? 128u : (cols <= 256 ? 256u : 512u));
}

// QM, how Q arrives (mj_q_mode): 0 e4m3 codes from mj_quantize_q; 1 bf16 Q
// as is, represented as two e4m3 terms per value; 2 bf16 Q quantized here
// with mj_quantize_q's recipe (see the Q staging in the softmax warps).
// D, the head size (128 or 256): a K or V row of D channels is DH = D / 128
// sub-tiles of 128 bytes; QK accumulates over the sub-tiles and PV runs once
// per sub-tile into its own O accumulator (channel 128 * dh + lane).
// KF, the cache format (mj_kv_format): e4m3, or packed e2m3 / e3m2 / e2m1,
// whose K tiles the MMA reads as they land and whose V tiles warps 7-9 widen
// to e4m3 first.
template <int NQK, int NPV, int NR, int KF, int QM = 0, int D = 128>
__global__ void __launch_bounds__(KF != MJ_KV_E4M3 ? kThreadsTcFp6 : kThreadsTc, (NR <= 16 ? 2 : 1))
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     DecodeParams p) {
  constexpr int DH = D / 128;
  constexpr uint32_t kEntry = DH * kTileBytes;  // one ring entry: a K or V tile
  constexpr uint32_t kQSub = q_sub_bytes(NQK);
  // P columns: term k (A hi, A lo, B hi, B lo) of row r at column k * NR + r
  static_assert(NPV == 4 * NR && NR <= NQK && NR >= 4 && (NR & (NR - 1)) == 0, "row tile");
  constexpr bool PK = KF != MJ_KV_E4M3;  // a packed (narrow) format: no NaN codes, V widened
  static_assert(QM != 1 || (!PK && 2 * NR <= NQK), "bf16 Q: e4m3 KV, hi and lo rows in the Q tile");
  static_assert((D == 128 || D == 256) && (!PK || D == 128), "head size (packed formats: 128)");
  // TP tiles per softmax iteration; NSB S and P buffers let QK run up to
  // NSB - 1 tiles ahead of PV, so the softmax of a tile never waits for
  // the QK product of the next.
  constexpr int TP = (NR <= 8 || (NR == 16 && QM != 1 && !PK)) ? 2 : 1;
  constexpr int NSB = tc_nsb(NR);
  static_assert(NSB >= 2 * TP, "S / P buffers");
  constexpr int NPB = tc_npb(NR);  // P buffers: P_j in buffer j % NPB
  static_assert(NPB % TP == 0 && NPB >= TP && NPB <= NSB, "P buffers");
  // TMEM: NSB S buffers (NQK columns each), DH O accumulators (NPV columns each)
  constexpr int kCols = tc_tmem_cols_used(NQK, NPV, NR, D);
  constexpr uint32_t kTmemCols = tc_tmem_alloc_cols(kCols);
  static_assert(kCols <= 512, "TMEM columns");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int stages = p.kv_stages;

  const TcSmem lay = tc_smem_layout(stages, NQK, NPV, NPB, DH);
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem + lay.ctrl);
  const uint32_t ring_addr = tc::smem_u32(smem + lay.ring);
  const uint32_t q_addr = tc::smem_u32(smem + lay.q);
  const uint32_t p_stride = lay.p1 - lay.p0;  // P buffer j at p0 + j * p_stride

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- set-up: barriers, TMEM, Q tile ------------------------------------
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.empty[s]), 1);
    }
    for (int s = 0; s < NSB; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.s_full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.p_full[s]), 128);
      tc::mbar_init(tc::smem_u32(&ctl.o_full[s]), 1);
    }
    for (int s = 0; s < 2; ++s) tc::mbar_init(tc::smem_u32(&ctl.red_bar[s]), 4);
    for (int s = 0; s < 2; ++s) tc::mbar_init(tc::smem_u32(&ctl.row_bar[s]), 4);
    tc::mbar_init(tc::smem_u32(&ctl.sum_bar), 4);
    tc::mbar_init(tc::smem_u32(&ctl.drain), 1);
    tc::mbar_init(tc::smem_u32(&ctl.q_ready), 128);
    tc::mbar_init(tc::smem_u32(&ctl.v_tail), 1);
    if (PK)
      for (int s = 0; s < stages; ++s) tc::mbar_init(tc::smem_u32(&ctl.vconv[s]), kConvThreads);
    ctl.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmap_k);
    tc::prefetch_tmap(&tmap_v);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&ctl.tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort = &ctl.abort;

  // The launch may overlap the end of the preceding kernel on the stream
  // (programmatic dependent launch): the set-up above reads nothing that
  // kernel writes. With bf16 Q (as is, or quantized here) that kernel may
  // have written anything read below (seq_lens, the KV cache, the plan), so
  // every thread waits for it here. With fp8 codes the preceding kernel is
  // mj_quantize_q, which wrote only the Q codes and descales: only the
  // softmax warps wait, before they read them.
  //
  // Before that wait, the two TMA producer warps ask L2 for the first
  // kPrefetchTiles tiles of the CTA's work row (its K and its V pages, the
  // lanes taking every 32nd page; more in the first wave of a grid without
  // a split or of one wave): HBM streams them while the preceding kernel
  // finishes, and a CTA that starts later has them requested before it has
  // read seq_lens.
  // A prefetch hands nothing to the SM, and L2 is where the preceding
  // kernel's writes land, so it cannot return stale data: the work row and
  // block-table entries it is aimed with are only a guess (read before the
  // wait, bounds-checked), and everything is read again after it.
  if constexpr (QM != 0) {
    if (warp == 0 || warp == kVProducerWarp) {
      const int4 wp = reinterpret_cast<const int4*>(p.work)[blockIdx.x / unsigned(p.h_k)];
      const int gp = int(blockIdx.x % unsigned(p.h_k));
      if (blockIdx.y == 0 && wp.z > wp.y && wp.x >= 0 && wp.x < p.num_seqs) {
        const int ppt = kKvTile / p.page_size;
        const int64_t grid = int64_t(gridDim.x) * gridDim.y;
        const bool deep = int64_t(blockIdx.x) + int64_t(gridDim.x) * blockIdx.y < p.first_wave &&
                          (!p.with_reduction || grid <= p.first_wave);
        const int depth = !deep ? kPrefetchTiles
                                : (grid <= 2 * int64_t(p.first_wave) ? kPrefetchTilesShortGrid : kPrefetchTilesFirstWave);
        const int n = min(depth, wp.z - wp.y) * ppt;  // pages
        const CUtensorMap* map = warp == 0 ? &tmap_k : &tmap_v;
        for (int k = lane; k < n; k += 32) {
          const int64_t e = int64_t(wp.y) * ppt + k;  // block-table entry of the page
          if (e >= p.bt_stride) break;
          const int pg = p.block_table[int64_t(wp.x) * p.bt_stride + e];
          if (pg >= 0 && int64_t(pg) < p.num_pages) {
#pragma unroll
            for (int dh = 0; dh < DH; ++dh) {
              if (p.tma_head_inner)
                tc::tma_prefetch_4d(map, 128 * dh, gp, 0, pg);
              else
                tc::tma_prefetch_4d(map, 128 * dh, 0, gp, pg);
            }
          }
        }
      }
    }
    // With no split (no merge kernel follows), the next kernel on the stream
    // may launch now: its CTAs take the SMs this grid's last CTAs leave and
    // run their set-up and prefetches meanwhile. (After a split the merge's
    // CTAs would sit on those SMs instead, and the step is slower.)
    if (!p.with_reduction) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc::grid_dependency_wait();
  }

  // CTA x = (work row, KV head) with the head fastest: the CTAs that run
  // together stream the same requests' pages (with token-major layouts the
  // heads of a page interleave, so they share DRAM rows). A CTA with
  // nothing to do (an empty work row, a padding request, a split past the
  // end, no rows in its tile) goes straight to the teardown.
  const int g = int(blockIdx.x % unsigned(p.h_k));
  const int4 w = reinterpret_cast<const int4*>(p.work)[blockIdx.x / unsigned(p.h_k)];
  const int b = w.x;
  bool active = w.z > w.y && b >= 0 && b < p.num_seqs;
  if (active && p.with_reduction && (w.w < 0 || w.w >= p.max_splits || b >= p.part_seqs)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadPlan);
    active = false;
  }
  const int L = active ? p.seq_lens[b] : 0;
  const int64_t k0 = int64_t(w.y) * kKvTile;
  const int64_t k1 = min(int64_t(w.z) * kKvTile, int64_t(L));
  const int r0 = blockIdx.y * p.tw;
  const int nr = min(min(p.tw, p.n_q - r0), NR);
  active = active && L > 0 && k1 > k0 && nr > 0;
  const int ntiles = active ? int((k1 - k0 + kKvTile - 1) / kKvTile) : 0;
  // the last tile ends before k0 + ntiles * 128: its V rows past the end get zeroed
  const bool last_partial = k0 + int64_t(ntiles) * kKvTile > k1;

  // TMEM columns: S buffer j % NSB at [(j % NSB) NQK, ...), the O accumulators
  // after them (sub-tile dh at tO + dh * NPV)
  auto tS = [&](int j) { return tmem + uint32_t((j % NSB) * NQK); };
  const uint32_t tO = tmem + uint32_t(NSB * NQK);
  // barrier slot and phase parity of tile j's S / P / O events
  auto bs = [&](int j) { return j % NSB; };
  auto bp = [&](int j) { return uint32_t(j / NSB) & 1u; };

  if (active) {
    if (warp == 0 || warp == kVProducerWarp) {
      // ======================= TMA producers ==================================
      // warp 0 loads the K tiles (ring entries u = 2i), warp kVProducerWarp the
      // V tiles (u = 2i + 1), concurrently: a CTA's TMA issue rate, not HBM,
      // bounds small-page streaming, and two issuing warps double it.
      const int half = warp == 0 ? 0 : 1;
      const CUtensorMap* map = half ? &tmap_v : &tmap_k;
      const uint64_t pol = p.evict_first ? tc::l2_policy_evict_first() : tc::l2_policy_evict_normal();
      const int ps = p.page_size;
      const int ppt = kKvTile / ps;
      const int64_t first_page = k0 / ps;
      const int64_t npages = (k1 + ps - 1) / ps - first_page;
      const int32_t* bt = p.block_table + int64_t(b) * p.bt_stride + first_page;
      const uint32_t page_bytes = uint32_t(ps) * 128u;                 // shared-memory footprint
      const uint32_t page_tx = uint32_t(ps) * uint32_t(p.row_bytes);  // bytes the copy delivers
      int64_t batch = -1;
      int entry = -1;
      bool ok = true;
      int issued = 0;  // tiles whose load this warp issued
      for (int i = 0; i < ntiles && ok; ++i) {
        // lane j < nvalid issues the load of page j of tile i (one page id per lane)
        const int nvalid = int(min(int64_t(ppt), npages - int64_t(i) * ppt));
        const int64_t e0 = int64_t(i) * ppt;
        if (batch < 0 || e0 + nvalid > batch + 32) {
          batch = e0;
          entry = (e0 + lane < npages) ? bt[e0 + lane] : -1;
        }
        const int pg = __shfl_sync(0xFFFFFFFFu, entry, int(e0 - batch) + (lane & 7));
        if (half == 0 && lane < nvalid && (pg < 0 || int64_t(pg) >= p.num_pages)) atomicOr(p.status, kStatusBadPage);
        const int u = 2 * i + half;
        const int slot = u % stages;
        const uint32_t round = uint32_t(u / stages);
        const uint32_t full = tc::smem_u32(&ctl.full[slot]);
        if (lane == 0) {
          ok = tc::mbar_wait(tc::smem_u32(&ctl.empty[slot]), (round & 1u) ^ 1u, abort, kWaitLimitNs);
          if (ok) tc::mbar_arrive_expect_tx(full, uint32_t(nvalid) * page_tx);
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (ok && lane < nvalid) {
          // sub-tile dh: channels 128 dh .. 128 dh + 127 (x = 128 dh bytes, 16-byte aligned)
#pragma unroll
          for (int dh = 0; dh < DH; ++dh) {
            const uint32_t dst = ring_addr + uint32_t(slot) * kEntry + uint32_t(dh) * kTileBytes + uint32_t(lane) * page_bytes;
            if (p.tma_head_inner)
              tc::tma_load_4d(dst, map, full, 128 * dh, g, 0, pg, pol);
            else
              tc::tma_load_4d(dst, map, full, 128 * dh, 0, g, pg, pol);
          }
        }
        if (ok) ++issued;
        __syncwarp();
      }
      if (!PK && half == 1 && ok && last_partial) {
        // Last, partial V tile: zero its rows past the end (page tails and
        // stale ring contents may hold NaN codes, and 0 * NaN would reach O
        // through the PV product), then release it to the MMA issuer. This warp
        // may wait on the slot's full barrier: its own wait on the slot's empty
        // barrier showed that the previous occupant has landed and been consumed.
        const int u = 2 * (ntiles - 1) + 1;
        const int slot = u % stages;
        if (lane == 0) ok = tc::mbar_wait(tc::smem_u32(&ctl.full[slot]), uint32_t(u / stages) & 1u, abort, kWaitLimitNs);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (ok) {
          const int first_dead = int(k1 - (k0 + int64_t(ntiles - 1) * kKvTile));  // rows >= this are past the end
#pragma unroll
          for (int dh = 0; dh < DH; ++dh) {
            uint4* tile = reinterpret_cast<uint4*>(smem + lay.ring + slot * kEntry + dh * kTileBytes);
            for (int c = first_dead * 8 + lane; c < kKvTile * 8; c += 32) tile[c] = make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.v_tail));
        }
      }
      if (!ok && lane == 0) {
        // abort: wait (bounded) for this warp's loads still in flight before the CTA exits
        const uint64_t t0 = tc::globaltimer_ns();
        for (int i = max(0, issued - stages); i < issued; ++i) {
          const int u = 2 * i + half;
          while (!tc::mbar_try_wait(tc::smem_u32(&ctl.full[u % stages]), uint32_t(u / stages) & 1u) &&
                 tc::globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    } else if (PK && warp >= kConvWarp0) {
      // ======================= V widening (packed KV) ===========================
      // Each V tile is widened in place, chunk by chunk, once its load lands.
      const int ct = tid - kConvWarp0 * 32;  // 0 .. kConvThreads - 1
      bool ok = true;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int u = 2 * i + 1;
        const int slot = u % stages;
        ok = tc::mbar_wait(tc::smem_u32(&ctl.full[slot]), uint32_t(u / stages) & 1u, abort, kWaitLimitNs);
        if (!ok) break;
        uint4* tile = reinterpret_cast<uint4*>(smem + lay.ring + slot * kEntry);
#pragma unroll 4
        for (int k = ct; k < kTileBytes / 16; k += kConvThreads) tile[k] = widen_chunk<KF>(tile[k]);
        tc::fence_async_smem();
        tc::mbar_arrive(tc::smem_u32(&ctl.vconv[slot]));
      }
    } else if (warp == 1) {
      // ======================= MMA issuer ======================================
      if (lane == 0) {
        // K is read in its own format straight from the packed TMA layout
        // (kind::f8f6f4 mixes an e2m3 / e3m2 / e2m1 A with the e4m3 Q); V
        // always arrives as e4m3.
        constexpr uint32_t idesc_qk = tc::idesc_e4m3(128, NQK, false, false) | (mma_kv_type(KF) << 7);
        // PV: A = V tile (MN-major), B = P (MN-major, no swizzle: [key][16 columns] blocks)
        constexpr uint32_t idesc_pv = tc::idesc_e4m3(128, NPV, true, true);
        const uint64_t qdesc = tc::smem_desc(q_addr, 16, 1024, tc::kSwizzle128B);
        // Event loop: issue QK_nq as soon as K tile nq has landed (at most one
        // tile ahead of PV: two S buffers), and PV_np as soon as P_np is
        // written and V tile np has landed. Neither product waits behind the
        // other's operands.
        bool ok = tc::mbar_wait(tc::smem_u32(&ctl.q_ready), 0, abort, kWaitLimitNs);
        int nq = 0, np = 0;
        uint64_t t_idle = 0;
        while (ok && np < ntiles) {
          bool progressed = false;
          if (nq < ntiles && nq <= np + NSB - 1) {
            const int u = 2 * nq;
            const int slot = u % stages;
            if (tc::mbar_test_wait(tc::smem_u32(&ctl.full[slot]), uint32_t(u / stages) & 1u)) {
              tc::tc_fence_after();
#pragma unroll
              for (int dh = 0; dh < DH; ++dh) {
                const uint64_t kdesc = tc::smem_desc(ring_addr + uint32_t(slot) * kEntry + uint32_t(dh) * kTileBytes, 16,
                                                     1024, tc::kSwizzle128B);
                const uint64_t qd = qdesc + uint64_t((uint32_t(dh) * kQSub) >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // 128 channels of the sub-tile in steps of 32 bytes
                  tc::umma_f8f6f4(tS(nq), kdesc + uint64_t(2 * k), qd + uint64_t(2 * k), idesc_qk, dh > 0 || k > 0);
              }
              tc::umma_commit(tc::smem_u32(&ctl.s_full[bs(nq)]));
              tc::umma_commit(tc::smem_u32(&ctl.empty[slot]));
              ++nq;
              progressed = true;
            }
          }
          if (np < nq) {
            const int u = 2 * np + 1;
            const int slot = u % stages;
            // V tile ready: widened (packed), tail-zeroed (last partial e4m3 tile, a
            // one-shot barrier), else landed
            const bool tail = !PK && last_partial && np == ntiles - 1;
            const uint32_t vbar = tc::smem_u32(PK ? &ctl.vconv[slot] : (tail ? &ctl.v_tail : &ctl.full[slot]));
            const uint32_t vpar = tail ? 0u : uint32_t(u / stages) & 1u;
            if (tc::mbar_test_wait(tc::smem_u32(&ctl.p_full[bs(np)]), bp(np)) && tc::mbar_test_wait(vbar, vpar)) {
              tc::tc_fence_after();
              // P, MN-major without swizzle: 8-key core groups 128 B apart (LBO),
              // 16-column blocks 2 KB apart (SBO)
              const uint64_t pdesc =
                  tc::smem_desc(tc::smem_u32(smem + lay.p0) + uint32_t(np % NPB) * p_stride, 128, 2048, 0);
#pragma unroll
              for (int dh = 0; dh < DH; ++dh) {
                const uint64_t vdesc = tc::smem_desc(ring_addr + uint32_t(slot) * kEntry + uint32_t(dh) * kTileBytes,
                                                     kTileBytes, 1024, tc::kSwizzle128B);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // K = 128 keys in steps of 32 (32 rows x 128 B of V, 32 x 16 B of P)
                  tc::umma_f8f6f4(tO + uint32_t(dh * NPV), vdesc + uint64_t(256 * k), pdesc + uint64_t(32 * k), idesc_pv,
                                  (np > 0 || k > 0));
              }
              tc::umma_commit(tc::smem_u32(&ctl.o_full[bs(np)]));
              tc::umma_commit(tc::smem_u32(&ctl.empty[slot]));
              ++np;
              progressed = true;
            }
          }
          if (progressed) {
            t_idle = 0;
          } else {
            const uint64_t now = tc::globaltimer_ns();
            if (t_idle == 0) {
              t_idle = now;
            } else if (now - t_idle > kWaitLimitNs || *abort) {
              *abort = 1;
              ok = false;
              break;
            }
            // back off: this warp shares its SM sub-partition with a softmax
            // warp, whose issue slots a tight polling loop would take
            __nanosleep(64);
          }
        }
        if (!ok) {
          // abort: wait (bounded) until every MMA issued so far has completed
          tc::umma_commit(tc::smem_u32(&ctl.drain));
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(tc::smem_u32(&ctl.drain), 0) && tc::globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    } else {
      // ======================= softmax warpgroup ===============================
      // Q codes and descales come from the preceding grid (mj_quantize_q) when
      // it is launched just before: wait for it here only, so that the TMA
      // producers stream KV meanwhile.
      tc::grid_dependency_wait();
      const int xq = tid - kSoftmaxWarp0 * 32;
      float sc_hi = 0.f, sc_lo = 0.f;  // bf16 Q: logit scales of its hi and lo terms
      float sq = 1.f;                  // Q quantized here: its descale
      // max over the 128 softmax threads (the four softmax warps always reach this barrier)
      auto block_max = [&](float v, int slot) {
        v = warp_max(v);
        if (lane == 0) ctl.qamax[slot][warp & 3] = v;
        tc::named_bar_sync(1, 128);
        return fmaxf(fmaxf(ctl.qamax[slot][0], ctl.qamax[slot][1]), fmaxf(ctl.qamax[slot][2], ctl.qamax[slot][3]));
      };
      // Q tile: DH sub-tiles (channels 128 dh ..) of [NQK rows][128 B], K-major,
      // 128-byte swizzle: byte c of row r in sub-tile c >> 7, 16-byte chunk
      // ((c & 127) >> 4) ^ (r & 7)
      auto q_off = [&](int r, int c) {
        return lay.q + uint32_t(c >> 7) * kQSub + uint32_t(r * 128 + ((((c & 127) >> 4) ^ (r & 7)) << 4) + (c & 15));
      };
      // zero rows r_from .. NQK-1 of every sub-tile
      auto zero_rows = [&](int r_from) {
        for (int i = xq; i < (NQK - r_from) * 8 * DH; i += 128) {
          const int dh = i / ((NQK - r_from) * 8), j = i % ((NQK - r_from) * 8);
          *reinterpret_cast<uint4*>(smem + lay.q + dh * kQSub + r_from * 128 + j * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      };
      if constexpr (QM == 0) {
        // Q codes rows r0 .. r0+nr-1 into the Q tile; other rows 0
        const uint8_t* qsrc = p.q_codes + ((int64_t(b) * p.h_k + g) * p.n_q + r0) * D;
        for (int i = xq; i < NQK * 8 * DH; i += 128) {
          const int r = i / (8 * DH), c = (i % (8 * DH)) * 16;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (r < nr) v = *reinterpret_cast<const uint4*>(qsrc + r * D + c);
          *reinterpret_cast<uint4*>(smem + q_off(r, c)) = v;
        }
      } else if constexpr (QM == 2) {
        // mj_quantize_q's recipe, in the kernel: x = bf16 Q (times q_mul), the
        // scale from the amax over all q_len*h_r rows of (b, g), then e4m3
        // round-to-nearest-even satfinite, every step an IEEE float32 operation,
        // so the codes and the descale are the ones that call writes. Thread xq
        // takes channels xq + 128 dh of every row.
        auto q_in = [&](int rr, int c) {
          const int tq = rr / p.h_r, h = g * p.h_r + rr % p.h_r;
          float v = bf16_bits_to_float(p.q_bf16[int64_t(b * p.q_len + tq) * p.q_ts + int64_t(h) * p.q_hs + c]);
          if (p.q_mul) v = __fmul_rn(v, p.q_mul[int64_t(h) * D + c]);
          return v;
        };
        // the tile's rows once, into registers (independent loads); the rows of
        // (b, g) outside the tile only count towards the amax
        float xr[DH][NR];
        float am = 0.f;
#pragma unroll
        for (int dh = 0; dh < DH; ++dh) {
          const int c = xq + 128 * dh;
#pragma unroll
          for (int r = 0; r < NR; ++r) xr[dh][r] = r < nr ? q_in(r0 + r, c) : 0.f;
#pragma unroll
          for (int r = 0; r < NR; ++r) am = fmaxf(am, fabsf(xr[dh][r]));
          for (int rr = 0; rr < p.n_q; ++rr)
            if (rr < r0 || rr >= r0 + nr) am = fmaxf(am, fabsf(q_in(rr, c)));
        }
        sq = __fdiv_rn(fmaxf(block_max(am, 0), 1e-6f), 448.0f);
#pragma unroll
        for (int dh = 0; dh < DH; ++dh) {
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            uint8_t code = 0;
            if (r < nr) code = __nv_cvt_float_to_fp8(__fdiv_rn(xr[dh][r], sq), __NV_SATFINITE, __NV_E4M3);
            smem[q_off(r, xq + 128 * dh)] = code;
          }
        }
        zero_rows(NR);  // the rows past the tile
      } else {
        // bf16 Q as two e4m3 terms: hi = e4m3(x / s_hi) with s_hi = amax/448,
        // lo = e4m3((x - hi*s_hi) / s_lo) with s_lo = (max |residual|)/448.
        // hi fills rows 0 .. NR-1 of the Q tile and lo rows NR .. 2NR-1, so one
        // QK product gives both terms; the logit is s_hi*S_hi + s_lo*S_lo.
        // Thread xq owns EPT consecutive channels of one row (NR x D values
        // over 128 threads; EPT divides 128, so they share one sub-tile).
        constexpr int EPT = NR * DH;
        const int row = (xq * EPT) / D, c0 = (xq * EPT) % D;
        float xv[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) xv[e] = 0.f;
        if (row < nr) {
          const int rr = r0 + row, tq = rr / p.h_r, h = g * p.h_r + rr % p.h_r;
          const uint16_t* src = p.q_bf16 + int64_t(b * p.q_len + tq) * p.q_ts + int64_t(h) * p.q_hs + c0;
#pragma unroll
          for (int e = 0; e < EPT; e += 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(src + e);
            xv[e] = __uint_as_float(u.x << 16);
            xv[e + 1] = __uint_as_float(u.x & 0xFFFF0000u);
            xv[e + 2] = __uint_as_float(u.y << 16);
            xv[e + 3] = __uint_as_float(u.y & 0xFFFF0000u);
          }
        }
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) am = fmaxf(am, fabsf(xv[e]));
        const float s_hi = __fdiv_rn(fmaxf(block_max(am, 0), 1e-6f), 448.f);
        uint32_t hw[EPT / 4];
        float rm = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; e += 2) {
          const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(xv[e], s_hi), __fdiv_rn(xv[e + 1], s_hi)), __NV_SATFINITE, __NV_E4M3);
          const float2 hv = e4m3x2_to_float2(h2);
          xv[e] -= hv.x * s_hi;  // the residual
          xv[e + 1] -= hv.y * s_hi;
          rm = fmaxf(rm, fmaxf(fabsf(xv[e]), fabsf(xv[e + 1])));
          if ((e & 3) == 0)
            hw[e / 4] = uint32_t(h2);
          else
            hw[e / 4] |= uint32_t(h2) << 16;
        }
        const float rmax = block_max(rm, 1);
        const float s_lo = rmax > 0.f ? __fdiv_rn(rmax, 448.f) : 1.f;
        uint32_t lw[EPT / 4];
#pragma unroll
        for (int e = 0; e < EPT; e += 2) {
          const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(xv[e], s_lo), __fdiv_rn(xv[e + 1], s_lo)), __NV_SATFINITE, __NV_E4M3);
          if ((e & 3) == 0)
            lw[e / 4] = uint32_t(l2);
          else
            lw[e / 4] |= uint32_t(l2) << 16;
        }
        // 4 codes per word (c is a multiple of 4: one 16-byte chunk)
#pragma unroll
        for (int e = 0; e < EPT; e += 4) {
          const int c = c0 + e;
          *reinterpret_cast<uint32_t*>(smem + q_off(row, c)) = hw[e / 4];
          *reinterpret_cast<uint32_t*>(smem + q_off(NR + row, c)) = lw[e / 4];
        }
        zero_rows(2 * NR);  // the rows past the two terms
        const float kq = kv_descale(p.k_descale, p.ds_seq, p.ds_head, b, g) * p.qk_scale_log2;
        sc_hi = s_hi * kq;
        sc_lo = s_lo * kq;
      }
      tc::fence_async_smem();
      tc::mbar_arrive(tc::smem_u32(&ctl.q_ready));
      const int qd = warp & 3;          // TMEM lane quadrant of this warp
      const int x = qd * 32 + lane;     // key of the tile (S) / channel (O)
      const uint32_t lane_off = uint32_t(qd * 32) << 16;
      const float kd = kv_descale(p.k_descale, p.ds_seq, p.ds_head, b, g);
      // bf16 Q as two terms: the logits are formed when S is read (scale 1 below)
      const float scale =
          QM == 1 ? 1.f : (QM == 2 ? sq : p.q_descale[int64_t(b) * p.h_k + g]) * kd * p.qk_scale_log2;
      // last visible key of each row (query token t sees keys j <= L - q_len + t)
      int lim[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r)
        lim[r] = r < nr ? (p.causal ? L - p.q_len + (r0 + r) / p.h_r : INT_MAX) : -1;
      const int lim_min = lim[0];  // the tile's first row has the smallest limit

      // m_ref: the reference max each row's P is scaled by; it only moves when a
      // tile's max exceeds it by more than kTau (log2 units), and then O (kept
      // in TMEM across tiles) is rescaled in place. P = 2^(t - m_ref + 8) stays
      // <= 2^(8 + kTau) < 448, so every e4m3 term of P stays finite.
      constexpr float kTau = 0.6f;
      float m_ref[NR], l_part[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        m_ref[r] = -INFINITY;
        l_part[r] = 0.f;
      }
      bool ok = true;
      constexpr int kGroup = 32 / NR;  // lanes that share a row after rs_reduce
      const int my_row = lane / kGroup;
      constexpr bool kBound = NR >= 8;  // the single-bound check before the per-row maxima
      int xr = 0;                       // per-row exchanges so far (kBound; the same count in every thread)
      // P buffers whose pair-B blocks may hold nonzero codes in this thread's
      // chunk (bit j: buffer j); at first every buffer (shared memory starts
      // with arbitrary contents)
      uint32_t b_dirty = (1u << NPB) - 1u;
      constexpr int kSmallBudget = 8 / TP;  // iterations whose weights below 1/4 went with pair A alone
      int n_small = 0;

      // TP tiles per iteration: with few rows, the two S buffers are processed
      // together (256 keys), so the row-max reduction, the cross-warp exchange
      // and the fences are paid once per pair and the two tiles' arithmetic
      // interleaves.
      for (int i = 0; i < ntiles; i += TP) {
        const int nt = min(TP, ntiles - i);
        float s[TP][NR];  // S columns of the real rows only
#pragma unroll
        for (int a = 0; a < TP; ++a) {
          if (a < nt) {
            ok = ok && tc::mbar_wait(tc::smem_u32(&ctl.s_full[bs(i + a)]), bp(i + a), abort, kWaitLimitNs);
          }
        }
        if (!ok) break;
        tc::tc_fence_after();
        if constexpr (QM != 1) {
#pragma unroll
          for (int a = 0; a < TP; ++a) {
            if (a < nt) {
              tc::tmem_ld_cols<NR>(tS(i + a) + lane_off, s[a]);
            } else {
#pragma unroll
              for (int c = 0; c < NR; ++c) s[a][c] = -INFINITY;
            }
          }
          tc::tmem_wait_ld();
        } else {
          // columns 0 .. NR-1: the hi term's products, NR .. 2NR-1: the lo term's
          float s2[TP][2 * NR];
#pragma unroll
          for (int a = 0; a < TP; ++a)
            if (a < nt) tc::tmem_ld_cols<2 * NR>(tS(i + a) + lane_off, s2[a]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int a = 0; a < TP; ++a)
#pragma unroll
            for (int c = 0; c < NR; ++c) s[a][c] = a < nt ? fmaf(s2[a][NR + c], sc_lo, s2[a][c] * sc_hi) : -INFINITY;
        }

        int key[TP];
        bool valid[TP];
#pragma unroll
        for (int a = 0; a < TP; ++a) {
          key[a] = int(k0) + (i + a) * kKvTile + x;
          valid[a] = a < nt && key[a] < int(k1);
        }
        // Every key of the iteration visible to every row (the common case:
        // no tile past the end, no causal limit inside): no per-row masks.
        // Rows past nr then see S = 0 (their Q rows are zero); their P only
        // reaches O columns that are never written out.
        const int64_t it_end = k0 + int64_t(i + nt) * kKvTile;  // one past the iteration's last key
        const bool all_vis = nt == TP && it_end <= k1 && it_end - 1 <= int64_t(lim_min);
        float tmp[NR];
        if (all_vis) {
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            float v = s[0][r] * scale;
#pragma unroll
            for (int a = 1; a < TP; ++a) v = fmaxf(v, s[a][r] * scale);
            tmp[r] = v;
          }
        } else {
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            float v = -INFINITY;
#pragma unroll
            for (int a = 0; a < TP; ++a)
              v = fmaxf(v, (valid[a] && key[a] <= lim[r]) ? s[a][r] * scale : -INFINITY);
            tmp[r] = v;
          }
        }
        const int xi = i / TP;  // exchange sequence number
        bool rescale = false;
        // With 8 or more rows, one bound first: the largest (tile max - m_ref)
        // over the rows and keys of the four warps. A row's reference only
        // moves when its tile max exceeds it by more than kTau, so a bound
        // <= kTau (the common case once the references have settled) skips the
        // per-row reductions. A row with no visible key so far gives
        // -inf - -inf = NaN, which fmaxf drops; its first visible key gives +inf.
        bool settled = false;
        if constexpr (kBound) {
          float dmax = -INFINITY;
#pragma unroll
          for (int r = 0; r < NR; ++r) dmax = fmaxf(dmax, tmp[r] - m_ref[r]);
          dmax = warp_max(dmax);
          if (lane == 0) ctl.bound[xi & 1][qd] = dmax;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.red_bar[xi & 1]));
          ok = tc::mbar_wait(tc::smem_u32(&ctl.red_bar[xi & 1]), uint32_t(xi >> 1) & 1u, abort, kWaitLimitNs);
          if (!ok) break;
          const float4 bd = *reinterpret_cast<const float4*>(&ctl.bound[xi & 1][0]);
          settled = fmaxf(fmaxf(bd.x, bd.y), fmaxf(bd.z, bd.w)) <= kTau;  // the same in every thread
        }
        if (!settled) {
          // per-row maxima over the four warps: exchange number xe (counted
          // apart from the bound exchanges when there are both)
          const int xe = kBound ? xr++ : xi;
          const uint32_t xbar = tc::smem_u32(kBound ? &ctl.row_bar[xe & 1] : &ctl.red_bar[xe & 1]);
          const float wmax = rs_reduce<NR, true>(tmp, lane);
          if (lane % kGroup == 0) ctl.red[xe & 1][qd][my_row] = wmax;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(xbar);
          ok = tc::mbar_wait(xbar, uint32_t(xe >> 1) & 1u, abort, kWaitLimitNs);
          if (!ok) break;

          // new reference maxima (the same decision in every thread)
#pragma unroll
          for (int r = 0; r < NR; r += 4) {
            const float4 a = *reinterpret_cast<const float4*>(&ctl.red[xe & 1][0][r]);
            const float4 b4 = *reinterpret_cast<const float4*>(&ctl.red[xe & 1][1][r]);
            const float4 c4 = *reinterpret_cast<const float4*>(&ctl.red[xe & 1][2][r]);
            const float4 d4 = *reinterpret_cast<const float4*>(&ctl.red[xe & 1][3][r]);
            const float tm[4] = {fmaxf(fmaxf(a.x, b4.x), fmaxf(c4.x, d4.x)), fmaxf(fmaxf(a.y, b4.y), fmaxf(c4.y, d4.y)),
                                 fmaxf(fmaxf(a.z, b4.z), fmaxf(c4.z, d4.z)), fmaxf(fmaxf(a.w, b4.w), fmaxf(c4.w, d4.w))};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float alpha = 1.f;
              if (tm[j] > m_ref[r + j] + kTau) {  // false for -inf tiles
                alpha = fast_exp2(m_ref[r + j] - tm[j]);  // 0 when m_ref = -inf
                rescale |= m_ref[r + j] != -INFINITY;
                m_ref[r + j] = tm[j];
                l_part[r + j] *= alpha;
              }
              // the O rescale below reads the factors back from shared memory
              if (lane == 0) ctl.alpha[qd][r + j] = alpha;
            }
          }
        }

        // p = 2^(t - m_ref + 8) of every (key, row) of the iteration, in place
        // of s; 0 where the row does not see the key. pmin: the smallest
        // weight of a visible key (for the pair-B budget below).
        float pmin = INFINITY;
        {
          float c8[NR];
#pragma unroll
          for (int r = 0; r < NR; ++r) c8[r] = 8.f - m_ref[r];
          if (all_vis) {
#pragma unroll
            for (int a = 0; a < TP; ++a)
#pragma unroll
              for (int r = 0; r < NR; ++r) {
                s[a][r] = fast_exp2(fmaf(s[a][r], scale, c8[r]));
                pmin = fminf(pmin, s[a][r]);
              }
          } else {
#pragma unroll
            for (int a = 0; a < TP; ++a)
#pragma unroll
              for (int r = 0; r < NR; ++r) {
                const bool vis = valid[a] && key[a] <= lim[r] && m_ref[r] != -INFINITY;
                s[a][r] = vis ? fast_exp2(fmaf(s[a][r], scale, c8[r])) : 0.f;
                pmin = fminf(pmin, vis ? s[a][r] : INFINITY);
              }
          }
        }
        // Pair A alone is within 2^-8 p of every p >= 1/4 and within 2^-10 of
        // every smaller one. A thread lets up to kSmallBudget of its
        // iterations with a weight below 1/4 (the smallest nonzero one tells)
        // go with pair A alone: that is at most TP kSmallBudget = 8 such keys
        // per row and thread, 1024 per row, 2^-10 each against a row sum of at
        // least 2^8: 2^-8 of it. Past that budget its warp adds pair B to every
        // iteration that holds small weights. Typical rows (keys within 10
        // binades of their max, bar a few) never pay for pair B; long rows far
        // below one dominant key do.
        const int small = pmin < 0.25f ? 1 : 0;
        const bool need_b = __any_sync(0xFFFFFFFFu, n_small + small > kSmallBudget);
        if (!need_b) n_small += small;

        // This key's column of P^T: term k of row r at byte k * NR + r (k: A hi,
        // A lo, B hi, B lo) of 16-column block (byte / 16), the key's 16-byte
        // chunk in it. Pair A is hi = e4m3(p), lo = e4m3(p - hi); pair B the
        // same split of (p - hi - lo) * 2^10 where p < 1/4, else 0. (One body,
        // instantiated with and without pair B.) With 8 or more rows pair B has
        // blocks of its own: without pair B only pair A's blocks are stored,
        // and pair B's are cleared only where this thread's chunk of the buffer
        // may still hold nonzero codes (b_dirty).
        auto make_p = [&](auto with_b) {
          constexpr bool WB = decltype(with_b)::value;
#pragma unroll
          for (int a = 0; a < TP; ++a) {
            if (a >= nt) break;
            uint32_t words[NPV / 4];
#pragma unroll
            for (int w2 = 0; w2 < NPV / 4; ++w2) words[w2] = 0u;
#pragma unroll
            for (int r = 0; r < NR; r += 2) {
              const float x0 = s[a][r], x1 = s[a][r + 1];
              const __nv_fp8x2_storage_t hi2 = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
              const float2 hf = e4m3x2_to_float2(hi2);
              const float d0 = x0 - hf.x, d1 = x1 - hf.y;  // exact
              const __nv_fp8x2_storage_t lo2 = __nv_cvt_float2_to_fp8x2(make_float2(d0, d1), __NV_SATFINITE, __NV_E4M3);
              const int sh = (r % 4) * 8;  // the pair's two bytes in their word
              words[r / 4] |= uint32_t(hi2) << sh;
              words[(NR + r) / 4] |= uint32_t(lo2) << sh;
              if constexpr (WB) {
                // pair B: what pair A left of p (exact), times 2^10, where p < 1/4
                const float2 lf = e4m3x2_to_float2(lo2);
                const float y0 = x0 < 0.25f ? (d0 - lf.x) * 1024.f : 0.f;
                const float y1 = x1 < 0.25f ? (d1 - lf.y) * 1024.f : 0.f;
                const __nv_fp8x2_storage_t bh2 = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
                const float2 bhf = e4m3x2_to_float2(bh2);
                const __nv_fp8x2_storage_t bl2 =
                    __nv_cvt_float2_to_fp8x2(make_float2(y0 - bhf.x, y1 - bhf.y), __NV_SATFINITE, __NV_E4M3);
                words[(2 * NR + r) / 4] |= uint32_t(bh2) << sh;
                words[(3 * NR + r) / 4] |= uint32_t(bl2) << sh;
              }
              // l sums the weights themselves; O gets them to within
              // max(2^-8 p, 2^-20) each
              l_part[r] += x0;
              l_part[r + 1] += x1;
            }
            uint8_t* pt = smem + lay.p0 + ((i + a) % NPB) * p_stride;
            constexpr int kBlkA = NR >= 8 ? NPV / 32 : NPV / 16;  // blocks always stored
#pragma unroll
            for (int bk = 0; bk < kBlkA; ++bk)
              *reinterpret_cast<uint4*>(pt + bk * 2048 + x * 16) =
                  make_uint4(words[4 * bk], words[4 * bk + 1], words[4 * bk + 2], words[4 * bk + 3]);
            if constexpr (kBlkA < NPV / 16) {
              const uint32_t bit = 1u << ((i + a) % NPB);
              if (WB || (b_dirty & bit)) {
#pragma unroll
                for (int bk = kBlkA; bk < NPV / 16; ++bk)
                  *reinterpret_cast<uint4*>(pt + bk * 2048 + x * 16) =
                      make_uint4(words[4 * bk], words[4 * bk + 1], words[4 * bk + 2], words[4 * bk + 3]);
                b_dirty = WB ? (b_dirty | bit) : (b_dirty & ~bit);
              }
            }
          }
        };
        if constexpr (NPB < NSB) {
          // this pair's P buffers last held the pair before the previous one:
          // wait until the MMAs have read them (the commit after PV_{i-1}
          // covers every earlier product)
          if (i >= NPB) {
            ok = tc::mbar_wait(tc::smem_u32(&ctl.o_full[bs(i - 1)]), bp(i - 1), abort, kWaitLimitNs);
            if (!ok) break;
          }
        }
        if (need_b)
          make_p(std::true_type{});
        else
          make_p(std::false_type{});
        if (rescale) {
          // O holds the PV sums up to tile i-1, scaled by the old references:
          // wait for the last of them and rescale O in TMEM before PV_i (which
          // waits for p_full, signalled below). Done after P is written, when
          // S no longer occupies registers.
          ok = tc::mbar_wait(tc::smem_u32(&ctl.o_full[bs(i - 1)]), bp(i - 1), abort, kWaitLimitNs);
          if (!ok) break;
          __syncwarp();  // lane 0's factors
          tc::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DH * NPV; c += 16) {
            float v[16];
            tc::tmem_ld16(tO + lane_off + c, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= ctl.alpha[qd][((c + j) % NPV) % NR];  // column k * NR + r: row r
            tc::tmem_st16(tO + lane_off + c, v);
          }
          tc::tmem_wait_st();
        }

        tc::fence_async_smem();
        tc::tc_fence_before();
#pragma unroll
        for (int a = 0; a < TP; ++a)
          if (a < nt) tc::mbar_arrive(tc::smem_u32(&ctl.p_full[bs(i + a)]));
        if (!ok) break;
      }
      // the final O: wait for the last PV product; o_acc[dh][r] is channel
      // 128 dh + x: pair A's two columns of row r plus 2^-10 times pair B's
      float o_acc[DH][NR];
#pragma unroll
      for (int dh = 0; dh < DH; ++dh)
#pragma unroll
        for (int r = 0; r < NR; ++r) o_acc[dh][r] = 0.f;
      ok = ok && tc::mbar_wait(tc::smem_u32(&ctl.o_full[bs(ntiles - 1)]), bp(ntiles - 1), abort, kWaitLimitNs);
      if (ok) {
        tc::tc_fence_after();
#pragma unroll
        for (int dh = 0; dh < DH; ++dh) {
          float ob[NR];  // pair B's sum
#pragma unroll
          for (int r = 0; r < NR; ++r) ob[r] = 0.f;
#pragma unroll
          for (int c = 0; c < NPV; c += 16) {
            float v[16];
            tc::tmem_ld16(tO + lane_off + dh * NPV + c, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c + j;
              if (col < 2 * NR)
                o_acc[dh][col % NR] += v[j];
              else
                ob[col % NR] += v[j];
            }
          }
#pragma unroll
          for (int r = 0; r < NR; ++r) o_acc[dh][r] = fmaf(ob[r], 1.f / 1024.f, o_acc[dh][r]);
        }
      }

      // ---- epilogue --------------------------------------------------------
      {
        float tmp[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) tmp[r] = l_part[r];
        const float wsum = rs_reduce<NR, false>(tmp, lane);
        if (lane % kGroup == 0) ctl.lsum[qd][my_row] = wsum;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.sum_bar));
      ok = ok && tc::mbar_wait(tc::smem_u32(&ctl.sum_bar), 0, abort, kWaitLimitNs);
      if (ok) {
        const bool direct = !p.with_reduction || p.n_splits[b] <= 1;
        const float vd = kv_descale(p.v_descale, p.ds_seq, p.ds_head, b, g) * p.v_fmt;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (r >= nr) break;
          const float lr = ctl.lsum[0][r] + ctl.lsum[1][r] + ctl.lsum[2][r] + ctl.lsum[3][r];
          const int row = r0 + r;
          const int tq = row / p.h_r, h = g * p.h_r + row % p.h_r;
          const int64_t idx = direct ? 0 : part_index(p, b, w.w, g, row);
#pragma unroll
          for (int dh = 0; dh < DH; ++dh) {
            const int ch = 128 * dh + x;
            const float on = lr > 0.f ? o_acc[dh][r] / lr : 0.f;
            if (direct) {
              float val = on * vd;
              if (p.o_mul) val *= p.o_mul[int64_t(h) * D + ch];
              p.out[int64_t(b * p.q_len + tq) * p.out_ts + int64_t(h) * p.out_hs + ch] = float_to_out_bits(val, p.out_f16);
            } else {
              p.o_part[idx * D + ch] = on;
            }
          }
          if (x == 0) {
            if (direct) {
              if (p.lse)
                p.lse[(int64_t(b) * p.h_k + g) * p.n_q + row] =
                    lr > 0.f ? (m_ref[r] + fast_log2(lr) - 8.f) * kLn2 : -INFINITY;
            } else {
              p.m_part[idx] = lr > 0.f ? m_ref[r] : -INFINITY;
              p.l_part[idx] = lr * (1.f / 256.f);
            }
          }
        }
      }
    }
  }  // active

  // ---- teardown ------------------------------------------------------------
  if (*abort && tid == 0) atomicOr(p.status, kStatusTimeout);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}


constexpr int kMaxDynSmem = 227 * 1024;  // per-block opt-in limit of sm_100-class GPUs
constexpr int kSmemPerSm = 228 * 1024;   // shared memory of one SM (each block also takes 1 KB)
constexpr int kMaxDevices = 64;

template <int NQK, int NPV, int NR, int KF, int QM, int D>
cudaError_t launch_tc(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p0, cudaStream_t stream) {
  DecodeParams p = p0;
  // the ring depth the shared memory holds (even, at least 2)
  auto smem_bytes = [&](int stages) {
    return int(tc_smem_layout(stages, NQK, NPV, tc_npb(NR), D / 128).total) + 1024;
  };
  if (p.kv_stages <= 0) {
    // default: the deepest ring up to 6 entries that keeps two CTAs per SM
    // (one for the 32-row tiles, whose registers allow only one)
    p.kv_stages = 6;
    if (NR <= 16)
      while (p.kv_stages > 2 && 2 * (smem_bytes(p.kv_stages) + 1024) > kSmemPerSm) p.kv_stages -= 2;
  }
  while (p.kv_stages > 2 && smem_bytes(p.kv_stages) > kMaxDynSmem) p.kv_stages -= 2;
  int bytes = smem_bytes(p.kv_stages);
  // An instance that allocates all 512 TMEM columns must be alone on its SM:
  // a second CTA's allocation would wait for the first to finish. Asking for
  // more than half of the SM's shared memory guarantees that.
  constexpr uint32_t kTmemCols = tc_tmem_alloc_cols(tc_tmem_cols_used(NQK, NPV, NR, D));
  if (kTmemCols == 512 && bytes <= kSmemPerSm / 2) bytes = kSmemPerSm / 2 + 1024;
  // The dynamic shared-memory limit is an attribute of the kernel on each
  // device: raise it once per device (atomically: host threads may race).
  static std::atomic<int> configured[kMaxDevices];  // largest size set so far, per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int have = configured[dev].load(std::memory_order_acquire);
  if (bytes > have) {
    e = cudaFuncSetAttribute(decode_tc_kernel<NQK, NPV, NR, KF, QM, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
    if (e != cudaSuccess) return e;
    while (bytes > have && !configured[dev].compare_exchange_weak(have, bytes, std::memory_order_acq_rel)) {
    }
  }
  // CTAs resident at once (the first wave), looked up once per device and
  // shared-memory size
  static std::atomic<int64_t> first_wave[kMaxDevices];  // (bytes << 32) | CTAs
  int64_t fw = first_wave[dev].load(std::memory_order_acquire);
  if ((fw >> 32) != int64_t(bytes)) {
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_tc_kernel<NQK, NPV, NR, KF, QM, D>,
                                                      KF != MJ_KV_E4M3 ? kThreadsTcFp6 : kThreadsTc, size_t(bytes));
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    fw = (int64_t(bytes) << 32) | int64_t(per_sm) * sms;
    first_wave[dev].store(fw, std::memory_order_release);
  }
  p.first_wave = int(fw & 0xFFFFFFFFll);
  cudaLaunchConfig_t cfg = {};
  if (int64_t(p.num_work) * p.h_k > INT32_MAX || p.n_row_tiles > 65535) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(unsigned(p.num_work) * unsigned(p.h_k), unsigned(p.n_row_tiles));
  cfg.blockDim = dim3(KF != MJ_KV_E4M3 ? kThreadsTcFp6 : kThreadsTc);
  cfg.dynamicSmemBytes = size_t(bytes);
  cfg.stream = stream;
  // Programmatic dependent launch: the grid may start before the preceding
  // kernel on the stream has finished; the kernel waits for it
  // (griddepcontrol.wait) before it reads anything that kernel may have
  // written (with fp8 Q codes, whose writer mj_quantize_q must precede it
  // directly, only before it reads the codes).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<NQK, NPV, NR, KF, QM, D>, mk, mv, p);
}

// The kernel instance for the row tile (the plan's tile width, 16 or 32
// rows; fewer rows take the 4- or 8-row variants). With bf16 Q as two terms
// the Q tile holds two rows (hi, lo) per query row. P takes 4 columns per
// row (two pairs of e4m3 terms).
template <int KF, int QM, int D = 128>
cudaError_t launch_rows(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream) {
  constexpr int K = QM == 1 ? 2 : 1;
  if (p.tw <= 16) {
    if (p.n_q <= 4) return launch_tc<16, 16, 4, KF, QM, D>(mk, mv, p, stream);
    if (p.n_q <= 8) return launch_tc<16, 32, 8, KF, QM, D>(mk, mv, p, stream);
    return launch_tc<16 * K, 64, 16, KF, QM, D>(mk, mv, p, stream);
  }
  return launch_tc<32 * K, 128, 32, KF, QM, D>(mk, mv, p, stream);
}

// packed KV takes fp8 Q only: codes, or quantized here
template <int KF>
cudaError_t launch_packed(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream) {
  return p.q_mode == MJ_Q_FP8_FUSED ? launch_rows<KF, 2>(mk, mv, p, stream) : launch_rows<KF, 0>(mk, mv, p, stream);
}

}  // namespace

// Per-variant launchers, each defined in its own translation unit: the row-tile
// and Q-mode dispatch (launch_rows) for one cache format and head size.
cudaError_t launch_tc_e4m3_d128(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_tc_e4m3_d256(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_tc_e2m3(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_tc_e3m2(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_tc_e2m1(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t stream);

}  // namespace mj
