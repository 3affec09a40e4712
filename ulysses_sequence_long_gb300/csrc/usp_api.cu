// usp_api.cu — the extern "C" entry points of include/usp.h: argument checks,
// workspace carving, tensor-map encoding and dispatch to the kernels.  No
// entry point allocates device memory or synchronises the stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "usp_attn_common.cuh"
#include "usp_internal.h"

namespace usp {

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> g(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

int check_launch() { return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA; }

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_head_tmap(CUtensorMap* m, const void* base, int P, int BS, int H, int D, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return USP_ERR_CUDA;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(BS),
                        static_cast<cuuint64_t>(P)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(BS) * H * D * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? USP_OK : USP_ERR_CUDA;
}

// Tensor map of a seq-layout bf16 tensor [P][B][Sl][H][D]: dims {D, H, Sl, B, P},
// box {64, 1, rows, 1, 1}; a box of `rows` tokens must lie in one shard of one row.
int make_seq_tmap(CUtensorMap* m, const void* base, int P, int B, int Sl, int H, int D, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return USP_ERR_CUDA;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(Sl),
                        static_cast<cuuint64_t>(B), static_cast<cuuint64_t>(P)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                           static_cast<cuuint64_t>(Sl) * H * D * 2, static_cast<cuuint64_t>(B) * Sl * H * D * 2};
  cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? USP_OK : USP_ERR_CUDA;
}

int make_stats_tmap(CUtensorMap* m, const void* base, int BS, int pitch, int rows, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return USP_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(BS), 2, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch) * 4, static_cast<cuuint64_t>(pitch) * 8};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_rows), 2, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? USP_OK : USP_ERR_CUDA;
}

// Tensor map of the stored dS blocks, bf16 [n_blocks][128 keys][64 queries]:
// dims {64, 128, n_blocks}, box {64, 128, 2} (the two 64-query blocks of one
// 128-row query tile, stored next to each other), 128-byte swizzle.
int make_ds_tmap(CUtensorMap* m, const void* base, long long n_blocks) {
  auto fn = encode_fn();
  if (fn == nullptr) return USP_ERR_CUDA;
  cuuint64_t dims[3] = {64, 128, static_cast<cuuint64_t>(n_blocks)};
  cuuint64_t strides[2] = {128, 128 * 128};
  cuuint32_t box[3] = {64, 128, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? USP_OK : USP_ERR_CUDA;
}

// The same blocks as store targets of one compute warp: box {64, 32, 1} (the
// 64 query columns of 32 key rows, 128-byte rows), 128-byte swizzle.
int make_ds_store_tmap(CUtensorMap* m, void* base, long long n_blocks) {
  auto fn = encode_fn();
  if (fn == nullptr) return USP_ERR_CUDA;
  cuuint64_t dims[3] = {64, 128, static_cast<cuuint64_t>(n_blocks)};
  cuuint64_t strides[2] = {128, 128 * 128};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS ? USP_OK : USP_ERR_CUDA;
}

}  // namespace usp

using namespace usp;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Ps sequence shards, Ph head blocks (Ps = Ph = P for the Ulysses exchange).
// H % Ph == 0: H/Ph heads per block.  H < Ph with Ph % H == 0: every head is
// replicated on Ph/H blocks (the head-layout tensor is Ph/H times larger); the
// exchange back then sums the replicas, which needs bf16 elements.
int check_relayout_args(const void* a, const void* b, int B, int S, int H, int D, int Ps, int Ph, int eb,
                        bool to_head) {
  if (a == nullptr || b == nullptr) return USP_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || H <= 0 || D <= 0 || Ps <= 0 || Ph <= 0) return USP_ERR_INVALID_ARG;
  if (eb != 1 && eb != 2 && eb != 4 && eb != 8) return USP_ERR_INVALID_ARG;
  const bool replicated = H < Ph;
  if ((replicated ? Ph % H : H % Ph) != 0 || S % Ps != 0) return USP_ERR_INDIVISIBLE;
  if (replicated && !to_head && eb != 2) return USP_ERR_UNSUPPORTED;
  const uint64_t hpr = replicated ? 1 : static_cast<uint64_t>(H / Ph);
  uint64_t run = hpr * D * eb;
  if (run % 16 != 0 || !aligned16(a) || !aligned16(b)) return USP_ERR_ALIGNMENT;
  uint64_t seq_vec = static_cast<uint64_t>(B) * S * H * D * eb / 16;
  uint64_t head_vec = static_cast<uint64_t>(Ph) * B * S * hpr * D * eb / 16;
  if (head_vec >= (1ull << 32) || static_cast<uint64_t>(Ph) * B * S >= (1ull << 32)) return USP_ERR_UNSUPPORTED;
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  const uint64_t bytes_a = (to_head ? seq_vec : head_vec) * 16, bytes_b = (to_head ? head_vec : seq_vec) * 16;
  if (pa < pb + bytes_b && pb < pa + bytes_a) return USP_ERR_INVALID_ARG;  // buffers overlap
  return USP_OK;
}

// ring x ulysses shards; 0 when the product is not a positive int
int hybrid_shards(int ring, int ulysses) {
  if (ring <= 0 || ulysses <= 0) return 0;
  const int64_t ps = static_cast<int64_t>(ring) * ulysses;
  return ps > (1 << 30) ? 0 : static_cast<int>(ps);
}

int check_attn_params(const usp_attn_params* p) {
  if (p == nullptr) return USP_ERR_INVALID_ARG;
  if (p->B <= 0 || p->S <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->P <= 0) return USP_ERR_INVALID_ARG;
  if (p->cu_seqlens == nullptr || p->n_docs == nullptr) return USP_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return USP_ERR_INVALID_ARG;
  if (p->window_left < -1) return USP_ERR_UNSUPPORTED;
  if (!(p->softmax_scale >= 0.f) || isinf(p->softmax_scale)) return USP_ERR_INVALID_ARG;
  // query heads split over the ranks; key/value heads either split too or,
  // when there are fewer of them than ranks, are replicated P/Hkv times
  if (p->Hq % p->P != 0 || p->Hq % p->Hkv != 0 || p->S % p->P != 0) return USP_ERR_INDIVISIBLE;
  if (p->Hkv >= p->P ? p->Hkv % p->P != 0 : p->P % p->Hkv != 0) return USP_ERR_INDIVISIBLE;
  if (p->D != 64 && p->D != 128) return USP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->B) * p->S >= (1ll << 30)) return USP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->P) * p->B * p->S * p->Hq * p->D >= (1ll << 40)) return USP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->B) * p->S * p->Hq >= (1ll << 31)) return USP_ERR_UNSUPPORTED;  // 32-bit row counters
  if (p->Hq > 1024) return USP_ERR_UNSUPPORTED;  // the preprocess stages 32 tokens x Hq row sums in shared memory
  if (p->io_layout != USP_IO_HEAD && p->io_layout != USP_IO_SEQ && p->io_layout != USP_IO_SEQ_KV_HEAD)
    return USP_ERR_INVALID_ARG;
  // ring x Ulysses step: the kernels' 256-row blocks never straddle a super-chunk
  if (p->ring < 0) return USP_ERR_INVALID_ARG;
  const int ring = p->ring > 1 ? p->ring : 1;
  if (ring > 1) {
    if (p->ring_step < 0 || p->ring_step >= ring) return USP_ERR_INVALID_ARG;
    if (p->S % ring != 0 || (p->S / ring) % 256 != 0) return USP_ERR_UNSUPPORTED;
  } else if (p->ring_step != 0) {
    return USP_ERR_INVALID_ARG;
  }
  // a head group of the backward passes (fused layout only)
  if (p->head_count < 0 || p->head_first < 0) return USP_ERR_INVALID_ARG;
  if (p->head_count == 0 && p->head_first != 0) return USP_ERR_INVALID_ARG;
  if (p->head_count > 0) {
    if (p->io_layout != USP_IO_SEQ) return USP_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(p->head_first) + p->head_count > p->Hkv) return USP_ERR_INVALID_ARG;
  }
  // fused exchanges: tiles of 128 tokens must never straddle a sequence shard
  // (P shards, P*ring for the hybrid)
  if (p->io_layout != USP_IO_HEAD &&
      (p->S % (static_cast<int64_t>(p->P) * ring) != 0 || (p->S / (p->P * ring)) % 128 != 0))
    return USP_ERR_UNSUPPORTED;
  return USP_OK;
}

}  // namespace

extern "C" {

const char* usp_status_string(int s) {
  switch (s) {
    case USP_OK: return "USP_OK";
    case USP_ERR_INVALID_ARG: return "USP_ERR_INVALID_ARG: null pointer, bad size or flag, or overlapping buffers";
    case USP_ERR_INDIVISIBLE: return "USP_ERR_INDIVISIBLE: sp size must divide S and the heads, Hkv must divide Hq";
    case USP_ERR_UNSUPPORTED: return "USP_ERR_UNSUPPORTED: head dim, element size or problem size not supported";
    case USP_ERR_ALIGNMENT: return "USP_ERR_ALIGNMENT: pointers and contiguous runs must be 16-byte aligned";
    case USP_ERR_BAD_SEQLENS: return "USP_ERR_BAD_SEQLENS: cu_seqlens does not describe the gathered sequence";
    case USP_ERR_BAD_POSITIONS: return "USP_ERR_BAD_POSITIONS: negative position id";
    case USP_ERR_TIMEOUT: return "USP_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    case USP_ERR_CUDA: return "USP_ERR_CUDA: CUDA call or launch failed";
    case USP_ERR_WORKSPACE: return "USP_ERR_WORKSPACE: workspace missing, misaligned or too small";
    default: return "USP_ERR_UNKNOWN";
  }
}

int usp_version(void) { return 100; }

int usp_relayout_fwd(const void* x_seq, void* x_head, int B, int S, int H, int D, int P, int eb,
                     usp_stream_t stream) {
  int rc = check_relayout_args(x_seq, x_head, B, S, H, D, P, P, eb, true);
  if (rc != USP_OK) return rc;
  return launch_relayout(x_seq, x_head, B, S, H, D, P, P, eb, true, reinterpret_cast<cudaStream_t>(stream));
}

int usp_relayout_bwd(const void* x_head, void* x_seq, int B, int S, int H, int D, int P, int eb,
                     usp_stream_t stream) {
  int rc = check_relayout_args(x_head, x_seq, B, S, H, D, P, P, eb, false);
  if (rc != USP_OK) return rc;
  return launch_relayout(x_head, x_seq, B, S, H, D, P, P, eb, false, reinterpret_cast<cudaStream_t>(stream));
}

static int relayout_qkv(const void* q_seq, const void* k_seq, const void* v_seq, void* q_head, void* k_head,
                        void* v_head, int B, int S, int Hq, int Hkv, int D, int Ps, int Ph, int eb,
                        usp_stream_t stream) {
  int rc;
  if (Hq % Ph != 0) return USP_ERR_INDIVISIBLE;  // query heads are never replicated
  if ((rc = check_relayout_args(q_seq, q_head, B, S, Hq, D, Ps, Ph, eb, true)) != USP_OK) return rc;
  if ((rc = check_relayout_args(k_seq, k_head, B, S, Hkv, D, Ps, Ph, eb, true)) != USP_OK) return rc;
  if ((rc = check_relayout_args(v_seq, v_head, B, S, Hkv, D, Ps, Ph, eb, true)) != USP_OK) return rc;
  const void* src[3] = {q_seq, k_seq, v_seq};
  void* dst[3] = {q_head, k_head, v_head};
  int H[3] = {Hq, Hkv, Hkv};
  return launch_relayout_qkv(src, dst, H, B, S, D, Ps, Ph, eb, reinterpret_cast<cudaStream_t>(stream));
}

int usp_relayout_fwd_qkv(const void* q_seq, const void* k_seq, const void* v_seq, void* q_head, void* k_head,
                         void* v_head, int B, int S, int Hq, int Hkv, int D, int P, int eb, usp_stream_t stream) {
  return relayout_qkv(q_seq, k_seq, v_seq, q_head, k_head, v_head, B, S, Hq, Hkv, D, P, P, eb, stream);
}

int usp_hybrid_relayout_fwd(const void* x_seq, void* x_head, int B, int S, int H, int D, int ring, int ulysses,
                            int eb, usp_stream_t stream) {
  const int ps = hybrid_shards(ring, ulysses);
  if (ps == 0) return USP_ERR_INVALID_ARG;
  int rc = check_relayout_args(x_seq, x_head, B, S, H, D, ps, ulysses, eb, true);
  if (rc != USP_OK) return rc;
  return launch_relayout(x_seq, x_head, B, S, H, D, ps, ulysses, eb, true, reinterpret_cast<cudaStream_t>(stream));
}

int usp_hybrid_relayout_bwd(const void* x_head, void* x_seq, int B, int S, int H, int D, int ring, int ulysses,
                            int eb, usp_stream_t stream) {
  const int ps = hybrid_shards(ring, ulysses);
  if (ps == 0) return USP_ERR_INVALID_ARG;
  int rc = check_relayout_args(x_head, x_seq, B, S, H, D, ps, ulysses, eb, false);
  if (rc != USP_OK) return rc;
  return launch_relayout(x_head, x_seq, B, S, H, D, ps, ulysses, eb, false, reinterpret_cast<cudaStream_t>(stream));
}

int usp_hybrid_relayout_fwd_qkv(const void* q_seq, const void* k_seq, const void* v_seq, void* q_head,
                                void* k_head, void* v_head, int B, int S, int Hq, int Hkv, int D, int ring,
                                int ulysses, int eb, usp_stream_t stream) {
  const int ps = hybrid_shards(ring, ulysses);
  if (ps == 0) return USP_ERR_INVALID_ARG;
  return relayout_qkv(q_seq, k_seq, v_seq, q_head, k_head, v_head, B, S, Hq, Hkv, D, ps, ulysses, eb, stream);
}

// ---- one real rank's side of the exchanges: send buffers for an all-to-all
// between processes and the receive buffers back into the rank's layouts.
// All four are the relayout kernel with one side of the permutation trivial:
// Ps = 1 sequence shard and Ph = P head blocks (the rank's own shard split by
// destination), or Ps = P shards (one per source rank) and Ph = 1 block.
static int a2a_heads_per_rank(int H, int P) { return H >= P ? H / P : 1; }

int usp_a2a_pack_seq_to_head(const void* x_local, void* send, int B, int S_local, int H, int D, int P, int eb,
                             usp_stream_t stream) {
  int rc = check_relayout_args(x_local, send, B, S_local, H, D, 1, P, eb, true);
  if (rc != USP_OK) return rc;
  return launch_relayout(x_local, send, B, S_local, H, D, 1, P, eb, true, reinterpret_cast<cudaStream_t>(stream));
}

int usp_a2a_unpack_seq_to_head(const void* recv, void* x_head, int B, int S_local, int H, int D, int P, int eb,
                               usp_stream_t stream) {
  if (H <= 0 || P <= 0 || S_local <= 0) return USP_ERR_INVALID_ARG;
  if (H >= P ? H % P != 0 : P % H != 0) return USP_ERR_INDIVISIBLE;
  if (static_cast<int64_t>(S_local) * P >= (1ll << 31)) return USP_ERR_UNSUPPORTED;
  const int hpr = a2a_heads_per_rank(H, P), S = S_local * P;
  int rc = check_relayout_args(recv, x_head, B, S, hpr, D, P, 1, eb, true);
  if (rc != USP_OK) return rc;
  return launch_relayout(recv, x_head, B, S, hpr, D, P, 1, eb, true, reinterpret_cast<cudaStream_t>(stream));
}

int usp_a2a_pack_head_to_seq(const void* x_head, void* send, int B, int S_local, int H, int D, int P, int eb,
                             usp_stream_t stream) {
  if (H <= 0 || P <= 0 || S_local <= 0) return USP_ERR_INVALID_ARG;
  if (H >= P ? H % P != 0 : P % H != 0) return USP_ERR_INDIVISIBLE;
  if (static_cast<int64_t>(S_local) * P >= (1ll << 31)) return USP_ERR_UNSUPPORTED;
  const int hpr = a2a_heads_per_rank(H, P), S = S_local * P;
  int rc = check_relayout_args(x_head, send, B, S, hpr, D, P, 1, eb, false);
  if (rc != USP_OK) return rc;
  return launch_relayout(x_head, send, B, S, hpr, D, P, 1, eb, false, reinterpret_cast<cudaStream_t>(stream));
}

int usp_a2a_unpack_head_to_seq(const void* recv, void* x_local, int B, int S_local, int H, int D, int P, int eb,
                               usp_stream_t stream) {
  int rc = check_relayout_args(recv, x_local, B, S_local, H, D, 1, P, eb, false);
  if (rc != USP_OK) return rc;
  return launch_relayout(recv, x_local, B, S_local, H, D, 1, P, eb, false, reinterpret_cast<cudaStream_t>(stream));
}

size_t usp_cu_seqlens_workspace_bytes(int B, int S) {
  if (B <= 0 || S <= 0) return 0;
  return cu_seqlens_ws_bytes(B, S);
}

int usp_cu_seqlens_from_position_ids(const int32_t* pos, int B, int S, int P, int32_t* cu_seqlens, int32_t* n_docs,
                                     int32_t* max_len, void* ws, size_t ws_bytes, int32_t* dev_status,
                                     usp_stream_t stream) {
  if (pos == nullptr || cu_seqlens == nullptr || n_docs == nullptr || max_len == nullptr) return USP_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || P <= 0) return USP_ERR_INVALID_ARG;
  if (S % P != 0) return USP_ERR_INDIVISIBLE;
  if (static_cast<int64_t>(B) * S >= 0x7FFFFFFFll) return USP_ERR_UNSUPPORTED;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 15u) || ws_bytes < cu_seqlens_ws_bytes(B, S))
    return USP_ERR_WORKSPACE;
  return launch_cu_seqlens(pos, B, S, P, cu_seqlens, n_docs, max_len, static_cast<int32_t*>(ws), dev_status,
                           reinterpret_cast<cudaStream_t>(stream));
}

int usp_attn_fwd(const usp_attn_params* params, const void* q, const void* k, const void* v, void* o, float* lse,
                 int32_t* dev_status, usp_stream_t stream) {
  int rc = check_attn_params(params);
  if (rc != USP_OK) return rc;
  if (params->head_count != 0) return USP_ERR_INVALID_ARG;  // head groups are for the dK/dV and dQ passes
  // a ring step leaves the sink out; usp_ring_fwd_merge adds it once at the last step
  if (params->ring > 1 && params->sinks != nullptr) return USP_ERR_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr) return USP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return USP_ERR_ALIGNMENT;
  return launch_attn_fwd(*params, q, k, v, o, lse, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

size_t usp_attn_bwd_fast_workspace_bytes(const usp_attn_params* params) {
  if (check_attn_params(params) != USP_OK) return 0;
  const size_t ds = attn_bwd_ds_bytes(*params);
  return ds == 0 ? 0 : attn_bwd_ws_bytes(*params) + ds;
}

size_t usp_attn_bwd_workspace_bytes(const usp_attn_params* params) {
  if (check_attn_params(params) != USP_OK) return 0;
  return attn_bwd_ws_bytes(*params);
}

int usp_attn_bwd(const usp_attn_params* params, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, void* dq, void* dk, void* dv, float* dsinks, void* ws,
                 size_t ws_bytes, int32_t* dev_status, usp_stream_t stream) {
  int rc = check_attn_params(params);
  if (rc != USP_OK) return rc;
  if (params->head_count != 0) return USP_ERR_INVALID_ARG;  // head groups are for the dK/dV and dQ passes
  if (params->io_layout == USP_IO_SEQ_KV_HEAD) return USP_ERR_UNSUPPORTED;  // a forward-only layout
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr || dO == nullptr ||
      dq == nullptr || dk == nullptr || dv == nullptr)
    return USP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return USP_ERR_ALIGNMENT;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < attn_bwd_ws_bytes(*params))
    return USP_ERR_WORKSPACE;
  return launch_attn_bwd(*params, q, k, v, o, lse, dO, dq, dk, dv, params->sinks ? dsinks : nullptr, ws, ws_bytes,
                         dev_status, reinterpret_cast<cudaStream_t>(stream));
}

int usp_attn_bwd_preprocess(const usp_attn_params* params, const void* o, const float* lse, const void* dO,
                            float* dsinks, void* ws, size_t ws_bytes, int32_t* dev_status, usp_stream_t stream) {
  int rc = check_attn_params(params);
  if (rc != USP_OK) return rc;
  if (params->head_count != 0) return USP_ERR_INVALID_ARG;  // head groups are for the dK/dV and dQ passes
  if (params->io_layout == USP_IO_SEQ_KV_HEAD) return USP_ERR_UNSUPPORTED;  // a forward-only layout
  if (o == nullptr || lse == nullptr || dO == nullptr) return USP_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(lse) || !aligned16(dO)) return USP_ERR_ALIGNMENT;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < attn_bwd_ws_bytes(*params))
    return USP_ERR_WORKSPACE;
  return launch_attn_bwd_preprocess(*params, o, lse, dO, params->sinks ? dsinks : nullptr, ws, dev_status,
                                    reinterpret_cast<cudaStream_t>(stream));
}

int usp_attn_bwd_dkdv(const usp_attn_params* params, const void* q, const void* k, const void* v, const float* lse,
                      const void* dO, void* dk, void* dv, const void* ws, size_t ws_bytes, int32_t* dev_status,
                      usp_stream_t stream) {
  int rc = check_attn_params(params);
  if (rc != USP_OK) return rc;
  if (params->io_layout == USP_IO_SEQ_KV_HEAD) return USP_ERR_UNSUPPORTED;  // a forward-only layout
  if (q == nullptr || k == nullptr || v == nullptr || lse == nullptr || dO == nullptr || dk == nullptr ||
      dv == nullptr)
    return USP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dO) || !aligned16(dk) ||
      !aligned16(dv))
    return USP_ERR_ALIGNMENT;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < attn_bwd_ws_bytes(*params))
    return USP_ERR_WORKSPACE;
  return launch_attn_bwd_dkdv(*params, q, k, v, lse, dO, dk, dv, ws, ws_bytes, dev_status,
                              reinterpret_cast<cudaStream_t>(stream));
}

int usp_attn_bwd_dq(const usp_attn_params* params, const void* q, const void* k, const void* v, const float* lse,
                    const void* dO, void* dq, const void* ws, size_t ws_bytes, int32_t* dev_status,
                    usp_stream_t stream) {
  int rc = check_attn_params(params);
  if (rc != USP_OK) return rc;
  if (params->io_layout == USP_IO_SEQ_KV_HEAD) return USP_ERR_UNSUPPORTED;  // a forward-only layout
  if (q == nullptr || k == nullptr || v == nullptr || lse == nullptr || dO == nullptr || dq == nullptr)
    return USP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dO) || !aligned16(dq))
    return USP_ERR_ALIGNMENT;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < attn_bwd_ws_bytes(*params))
    return USP_ERR_WORKSPACE;
  return launch_attn_bwd_dq(*params, q, k, v, lse, dO, dq, ws, ws_bytes, dev_status,
                            reinterpret_cast<cudaStream_t>(stream));
}

int usp_ring_fwd_merge(const usp_attn_params* params, const void* o_step, const float* lse_step, float* o_acc,
                       float* lse_acc, void* o, float* lse, int flags, usp_stream_t stream) {
  int rc = check_attn_params(params);
  if (rc != USP_OK) return rc;
  if (params->head_count != 0) return USP_ERR_INVALID_ARG;  // head groups are for the dK/dV and dQ passes
  if (flags & ~(USP_RING_FIRST | USP_RING_LAST)) return USP_ERR_INVALID_ARG;
  const bool first = flags & USP_RING_FIRST, last = flags & USP_RING_LAST;
  if (o_step == nullptr || lse_step == nullptr) return USP_ERR_INVALID_ARG;
  if ((!first || !last) && (o_acc == nullptr || lse_acc == nullptr)) return USP_ERR_INVALID_ARG;
  if (last && (o == nullptr || lse == nullptr)) return USP_ERR_INVALID_ARG;
  if (!aligned16(o_step) || (o_acc && !aligned16(o_acc)) || (o && !aligned16(o))) return USP_ERR_ALIGNMENT;
  if (static_cast<uint64_t>(params->P) * params->B * params->S * (params->Hq / params->P) * (params->D / 8) >=
      (1ull << 32))
    return USP_ERR_UNSUPPORTED;
  return launch_ring_fwd_merge(*params, o_step, lse_step, o_acc, lse_acc, o, lse, flags,
                               reinterpret_cast<cudaStream_t>(stream));
}

int usp_ring_grad_accumulate(const void* g_step, float* g_acc, void* g_out, size_t n, int flags,
                             usp_stream_t stream) {
  if (flags & ~(USP_RING_FIRST | USP_RING_LAST)) return USP_ERR_INVALID_ARG;
  const bool first = flags & USP_RING_FIRST, last = flags & USP_RING_LAST;
  if (g_step == nullptr || ((!first || !last) && g_acc == nullptr) || (last && g_out == nullptr))
    return USP_ERR_INVALID_ARG;
  if (n % 8 != 0) return USP_ERR_ALIGNMENT;
  if (!aligned16(g_step) || (g_acc && !aligned16(g_acc)) || (g_out && !aligned16(g_out))) return USP_ERR_ALIGNMENT;
  if (n / 8 >= (1ull << 32)) return USP_ERR_UNSUPPORTED;
  return launch_ring_grad_accumulate(g_step, g_acc, g_out, n, flags, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
