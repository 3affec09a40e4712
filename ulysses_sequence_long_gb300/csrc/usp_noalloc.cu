// usp_noalloc.cu — document boundaries from position_ids without a caller
// workspace.
//
// usp_cu_seqlens_from_position_ids needs a small device workspace for its
// per-block scan states.  Some callers cannot provide one: code that may
// not call cudaMalloc (or any allocator) on its path — for example a runtime
// whose device memory is entirely pre-reserved by another allocator, or a
// plugin interface that hands the library only its input and output pointers.
// For them this entry point keeps that scratch in a fixed, file-scope device
// array instead, and allocates nothing.
//
// The array is `kScratchInts` int32 (64 KiB) and covers B*S up to
// kMaxTokens = 2^24 tokens; every GPU that loads the library holds it until
// the process exits.  All calls share it: two calls whose kernels overlap on
// the GPU (different streams, or different host threads) race on it, so
// callers must order such calls.  Nothing in it needs to start at zero: the
// first of the scan's two kernels resets every block state and the counter
// the second one uses, so whatever a previous call left there never matters.
#include <cuda_runtime.h>
#include <stdint.h>

#include "usp_internal.h"

namespace {

constexpr int kMaxTokens = 1 << 24;
constexpr int kScratchInts = 16384;  // 64 KiB
static_assert(usp::cu_seqlens_ws_bytes_for(kMaxTokens) <= sizeof(int32_t) * kScratchInts,
              "the fixed scratch must hold the scan's workspace for kMaxTokens positions");

static __device__ __align__(256) int32_t g_scan_scratch[kScratchInts];

// Device address of g_scan_scratch on the current device.  In host code the
// name g_scan_scratch is only a host-side stand-in, not a device address, so
// it is looked up with the device current, on every call: a cached address
// would go stale if the caller reset the device between calls.
int scratch_for_current_device(int32_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scan_scratch) != cudaSuccess || p == nullptr) return USP_ERR_CUDA;
  *out = static_cast<int32_t*>(p);
  return USP_OK;
}

}  // namespace

extern "C" int usp_cu_seqlens_from_position_ids_noalloc(const int32_t* pos, int B, int S, int P,
                                                        int32_t* cu_seqlens, int32_t* n_docs, int32_t* max_len,
                                                        int32_t* dev_status, usp_stream_t stream) {
  if (pos == nullptr || cu_seqlens == nullptr || n_docs == nullptr || max_len == nullptr) return USP_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || P <= 0) return USP_ERR_INVALID_ARG;
  if (S % P != 0) return USP_ERR_INDIVISIBLE;
  if (static_cast<int64_t>(B) * S > kMaxTokens) return USP_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (usp::cu_seqlens_ws_bytes(B, S) > sizeof(int32_t) * static_cast<size_t>(kScratchInts))
    return USP_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != USP_OK) return rc;
  return usp::launch_cu_seqlens(pos, B, S, P, cu_seqlens, n_docs, max_len, scratch, dev_status,
                                reinterpret_cast<cudaStream_t>(stream));
}
