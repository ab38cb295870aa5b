// Device code shared by the tensor-core and CUDA-core Newton-Schulz paths.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace muon {

// Last-iteration output of element (r, c) of the n x m short-side result.
__device__ __forceinline__ void ns_last_store(const NsParams& p, int gm, int n, int m, int r, int c, float o,
                                           float s_apply) {
  const size_t idx = (p.flags[gm] & NS_TALL) ? (size_t)c * n + r : (size_t)r * m + c;
  if (p.dst_mode == 0) {
    if (p.dst_dtype == MUON_DTYPE_BF16) reinterpret_cast<bf16*>(p.dst[gm])[idx] = __float2bfloat16_rn(o);
    else reinterpret_cast<float*>(p.dst[gm])[idx] = o;
  } else {
    if (p.dst_dtype == MUON_DTYPE_BF16) {
      bf16* W = reinterpret_cast<bf16*>(p.dst[gm]);
      const float w = __bfloat162float(W[idx]);
      W[idx] = __float2bfloat16_rn(w - p.eta * (s_apply * o + p.lam * w));
    } else {
      float* W = reinterpret_cast<float*>(p.dst[gm]);
      const float w = W[idx];
      W[idx] = w - p.eta * (s_apply * o + p.lam * w);
    }
  }
}

}  // namespace muon
