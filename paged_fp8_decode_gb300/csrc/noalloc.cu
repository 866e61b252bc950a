// mj_decode_attention_noalloc: decode + merge for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving engine that
// reserves nearly all of HBM for its KV-cache pool up front and forbids later
// cudaMalloc calls, or a plugin living inside a host framework whose own
// caching allocator owns device memory (a raw cudaMalloc/cudaFree there
// bypasses that allocator and synchronises the device). For them, this entry
// point keeps the split-KV partials in a fixed array compiled into the
// library instead of a caller workspace.
//
// The array is file-scope `static __device__`, so every GPU that loads the
// library holds its MJ_NOALLOC_SCRATCH_BYTES until the process exits. In host
// code its name is only a host-side stand-in for the device symbol; the
// device address is looked up once per device with cudaGetSymbolAddress (with
// that device current) and passed to the kernels. The lookup, and the zeroing
// of the status header (enqueued on the caller's stream, ahead of that call's
// kernels), happen on the first call on each device, which should therefore
// come before any stream capture. All calls share the one array, so calls
// whose kernels overlap on the GPU (different streams, concurrent threads)
// race on it; issue them in order on one stream. mj_noalloc_status reads and
// clears the status word the kernels record anomalies in.
#include <cuda_runtime.h>

#include <mutex>

#include "mj_internal.h"

namespace {

constexpr size_t kScratchBytes = MJ_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once:
// the first call on a device also zeroes the header on `stream`).
int scratch_on_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MJ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MJ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return MJ_ERR_CUDA;
    // the status word (header) is the only part that must start at zero;
    // the partials are always written before they are read within a call.
    // Zeroed on the caller's stream, so that it is ordered before this
    // call's kernels whatever kind of stream that is.
    if (cudaMemsetAsync(ptr, 0, mj::kWsHeader, stream) != cudaSuccess) return MJ_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return MJ_OK;
}

}  // namespace

extern "C" int mj_decode_attention_noalloc(const mj_decode_args* args, void* stream) {
  const mj::NvtxRange range("mj_decode_attention_noalloc");
  if (!args) return MJ_ERR_INVALID_ARG;
  size_t need = mj::kWsHeader;
  if (args->with_reduction) {
    const int st =
        mj_workspace_size(args->part_seqs, args->max_splits, args->q_len, args->h_q, args->h_k, args->d, &need);
    if (st != MJ_OK) return st;
  }
  if (need > kScratchBytes) return MJ_ERR_CAPACITY;  // the plan needs more than the fixed array holds
  void* scratch = nullptr;
  int st = scratch_on_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (st != MJ_OK) return st;
  mj_decode_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kScratchBytes;
  st = mj_decode_attention(&a, stream);
  if (st != MJ_OK) return st;
  return mj_merge_lse(&a, stream);
}

extern "C" int mj_noalloc_status(void* stream, uint32_t* device_status) {
  if (!device_status) return MJ_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (st != MJ_OK) return st;
  return mj_workspace_status(scratch, stream, device_status);
}
