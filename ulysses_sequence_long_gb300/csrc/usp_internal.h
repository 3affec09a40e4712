// usp_internal.h — host-side declarations shared by the library's translation
// units (launchers behind the C entry points of include/usp.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/usp.h"

namespace usp {

// SM count of the current device (cached per device).
int device_sm_count();

// Records a CUDA error of the last launch as USP_ERR_CUDA.
int check_launch();

// Exact unsigned 32-bit division by a runtime constant (multiply-high and
// shift, Granlund & Montgomery 1994, "Division by invariant integers using
// multiplication", round-up variant).
struct FastDiv {
  uint32_t d, m, s;
  FastDiv() : d(1), m(0), s(0) {}
  explicit FastDiv(uint32_t div) : d(div) {
    s = 0;
    while ((1ull << s) < div) ++s;
    m = static_cast<uint32_t>(((1ull << 32) * ((1ull << s) - div)) / div + 1);
  }
#ifdef __CUDACC__
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    uint32_t hi = __umulhi(n, m);
    return static_cast<uint32_t>((static_cast<uint64_t>(hi) + n) >> s);
  }
#endif
};

// Ps sequence shards, Ph head blocks (Ps = Ph = P: the Ulysses exchange;
// Ps = ring*ulysses, Ph = ulysses: the exchange of the ring x Ulysses hybrid).
int launch_relayout(const void* src, void* dst, int B, int S, int H, int D, int Ps, int Ph, int elem_bytes,
                    bool to_head, cudaStream_t st);
int launch_relayout_qkv(const void* const src[3], void* const dst[3], const int H[3], int B, int S, int D, int Ps,
                        int Ph, int elem_bytes, cudaStream_t st);
int launch_ring_fwd_merge(const usp_attn_params& p, const void* o_step, const float* lse_step, float* o_acc,
                          float* lse_acc, void* o, float* lse, int flags, cudaStream_t st);
int launch_ring_grad_accumulate(const void* g_step, float* g_acc, void* g_out, size_t n, int flags, cudaStream_t st);
// Document-boundary scan: at most one block per kScanChunk positions, and its
// workspace (a 256-byte header holding the block ticket, then one 64-bit state
// per block).
constexpr int kScanChunk = 32768;
constexpr size_t kScanHeaderBytes = 256;
constexpr size_t cu_seqlens_ws_bytes_for(long long tokens) {
  return kScanHeaderBytes +
         (8 * static_cast<size_t>(tokens > kScanChunk ? (tokens + kScanChunk - 1) / kScanChunk : 1) + 255) / 256 * 256;
}
int launch_cu_seqlens(const int32_t* pos, int B, int S, int P, int32_t* cu, int32_t* n_docs, int32_t* max_len,
                      int32_t* ws, int32_t* status, cudaStream_t st);
size_t cu_seqlens_ws_bytes(int B, int S);

int launch_attn_fwd(const usp_attn_params& p, const void* q, const void* k, const void* v, void* o, float* lse,
                    int32_t* status, cudaStream_t st);
int launch_attn_bwd(const usp_attn_params& p, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, void* dq, void* dk, void* dv, float* dsinks, void* ws,
                    size_t ws_bytes, int32_t* status, cudaStream_t st);
size_t attn_bwd_ws_bytes(const usp_attn_params& p);
size_t attn_bwd_ds_bytes(const usp_attn_params& p);  // stored-dS blocks (0: no such path for the shape)
int launch_attn_bwd_preprocess(const usp_attn_params& p, const void* o, const float* lse, const void* dO, float* dsinks,
                               void* ws, int32_t* status, cudaStream_t st);
int launch_attn_bwd_dkdv(const usp_attn_params& p, const void* q, const void* k, const void* v, const float* lse,
                         const void* dO, void* dk, void* dv, const void* ws, size_t ws_bytes, int32_t* status,
                         cudaStream_t st);
int launch_attn_bwd_dq(const usp_attn_params& p, const void* q, const void* k, const void* v, const float* lse,
                       const void* dO, void* dq, const void* ws, size_t ws_bytes, int32_t* status, cudaStream_t st);

}  // namespace usp
