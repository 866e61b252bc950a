// Host side of the tcgen05 decode path: its envelope (tc_supported), the
// 4-D tensor maps of the K and V caches, and the dispatch to the per-variant
// launchers (decode_tc_*.cu). The kernel is in decode_tc_kernel.cuh.
#include "decode_tc_kernel.cuh"

namespace mj {

namespace {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 4-D byte tensor (row, token, head, page) of one K or V cache; the smaller of
// the token / head strides goes to dimension 1 (a box extent of 1 in the head
// dimension leaves the shared-memory layout [token][128 B] either way).
bool encode_kv_map(CUtensorMap* map, const void* base, const DecodeParams& p, int64_t sp, int64_t st, int64_t sh,
                   bool head_inner) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t sh_eff = p.h_k == 1 ? (head_inner ? 32 : sp) : sh;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  dims[0] = cuuint64_t(p.d);  // channels (e4m3 bytes, or packed codes); a box is 128 of them
  box[0] = 128;
  if (head_inner) {
    dims[1] = cuuint64_t(p.h_k);
    dims[2] = cuuint64_t(p.page_size);
    strides[0] = cuuint64_t(sh_eff);
    strides[1] = cuuint64_t(st);
    box[1] = 1;
    box[2] = cuuint32_t(p.page_size);
  } else {
    dims[1] = cuuint64_t(p.page_size);
    dims[2] = cuuint64_t(p.h_k);
    strides[0] = cuuint64_t(st);
    strides[1] = cuuint64_t(sh_eff);
    box[1] = cuuint32_t(p.page_size);
    box[2] = 1;
  }
  dims[3] = cuuint64_t(p.num_pages);
  strides[2] = cuuint64_t(sp);
  box[3] = 1;
  // e4m3: one byte per element. Packed formats (D = 128 only): 16U6_ALIGN16B
  // (e2m3, e3m2) keeps 16 codes in 12 bytes and lands each group in a 16-byte
  // shared-memory chunk (4 bytes of padding); 16U4_ALIGN16B (e2m1) keeps 16
  // codes in 8 bytes and lands them in the first half of a 16-byte chunk.
  // tcgen05.mma reads either chunk as its 16 codes; dims[0] counts codes.
  const CUtensorMapDataType dt = p.kv_format == MJ_KV_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : p.kv_format == MJ_KV_E2M1 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
                                                             : CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B;
  const CUresult r = fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const DecodeParams& p) {
  if (p.q_mode == MJ_Q_BF16 && p.kv_format != MJ_KV_E4M3) return false;
  if (p.kv_format != MJ_KV_E4M3) {
    if (p.d != 128) return false;  // packed formats: D = 128 only
    // the packed TMA types want 32-byte aligned strides (and base, checked
    // by the ABI for the packed formats)
    const int64_t st[] = {p.k_sp, p.k_st, p.k_sh, p.v_sp, p.v_st, p.v_sh};
    for (int64_t v : st)
      if (v % 32) return false;
  }
  if (p.n_q > 32 && p.tw != 32) return false;
  if (p.num_pages > INT32_MAX || p.h_k > 65535) return false;
  const int64_t sm[] = {p.k_sp, p.v_sp};
  for (int64_t s : sm)
    if (s == 0) return false;
  if (!encode_fn()) return false;
  return true;
}

int tc_max_stages() { return 13; }

namespace {

// The tensor-core kernel's preconditions and its two tensor maps; false when
// the arguments are outside its envelope.
bool tc_prepare(DecodeParams& p, CUtensorMap* mk, CUtensorMap* mv) {
  if (!tc_supported(p)) return false;
  p.tma_head_inner = (p.k_sh < p.k_st) ? 1 : 0;
  if (((p.v_sh < p.v_st) ? 1 : 0) != p.tma_head_inner) return false;
  return encode_kv_map(mk, p.k_cache, p, p.k_sp, p.k_st, p.k_sh, p.tma_head_inner) &&
         encode_kv_map(mv, p.v_cache, p, p.v_sp, p.v_st, p.v_sh, p.tma_head_inner);
}

}  // namespace

bool decode_tc_supported(const DecodeParams& p0) {
  DecodeParams p = p0;
  CUtensorMap mk, mv;
  return tc_prepare(p, &mk, &mv);
}

cudaError_t launch_decode_tc(DecodeParams p, cudaStream_t stream, bool* unsupported) {
  *unsupported = false;
  CUtensorMap mk, mv;
  if (!tc_prepare(p, &mk, &mv)) {
    *unsupported = true;
    return cudaSuccess;
  }
  // kv_stages <= 0: the launcher picks the default depth for the instance
  if (p.kv_stages > tc_max_stages()) p.kv_stages = tc_max_stages();
  // The ring depth is always even, so that K tiles (ring entries u = 2i) and
  // V tiles (u = 2i + 1) never share a slot. Every waiter on full[slot] must
  // know that the slot's previous occupant has landed: a phase-parity wait
  // for the k-th use of a barrier passes wrongly while use k - 1 is still
  // pending. With K-only and V-only slots the previous occupant of a K (V)
  // slot is an earlier K (V) tile that the MMA issuer (or the V-widening
  // warps) has already consumed in order. With an odd depth a K slot's
  // previous occupant is a V tile, which the issuer's look-ahead QK probe (up
  // to three tiles ahead of PV) can reach before it has landed.
  if (p.kv_stages > 0 && (p.kv_stages & 1)) p.kv_stages = p.kv_stages > 2 ? p.kv_stages - 1 : 2;
  if (p.num_work == 0) return cudaSuccess;
  // row tile = the plan's tile width (16 or 32 rows)
  if (p.kv_format != MJ_KV_E4M3) {
    // K enters the MMA as true values (no widening factor); V is widened in
    // shared memory and keeps the factor in v_fmt.
    p.qk_scale_log2 *= 1.0f / kv_widen_factor(p.kv_format);
    if (p.kv_format == MJ_KV_E2M3) return launch_tc_e2m3(mk, mv, p, stream);
    if (p.kv_format == MJ_KV_E3M2) return launch_tc_e3m2(mk, mv, p, stream);
    return launch_tc_e2m1(mk, mv, p, stream);
  }
  return p.d == 256 ? launch_tc_e4m3_d256(mk, mv, p, stream) : launch_tc_e4m3_d128(mk, mv, p, stream);
}

}  // namespace mj
