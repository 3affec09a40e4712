// usp_attn_bwd.cu — attention backward (placeholder until the kernels land).
#include "usp_attn_common.cuh"
#include "usp_internal.h"

namespace usp {
size_t attn_bwd_ws_bytes(const usp_attn_params& p) {
  size_t rows = static_cast<size_t>(p.B) * p.S * p.Hq;
  return (rows * sizeof(float) + 255) / 256 * 256;
}
int launch_attn_bwd(const usp_attn_params&, const void*, const void*, const void*, const void*, const float*,
                    const void*, void*, void*, void*, float*, void*, int32_t*, cudaStream_t) {
  return USP_ERR_UNSUPPORTED;
}
}  // namespace usp
