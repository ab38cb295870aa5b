// Device helpers shared by the Muon kernels: dtype conversion, 4-wide vector
// loads/stores, fixed-order reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace muon {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------
// scalar conversion
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// 4 consecutive elements <-> float[4]; the pointer must be aligned to 4 elements
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld4(const float* p, float v[4]) {
  float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ld4(const bf16* p, float v[4]) {
  uint2 x = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(x.x << 16);
  v[1] = __uint_as_float(x.x & 0xFFFF0000u);
  v[2] = __uint_as_float(x.y << 16);
  v[3] = __uint_as_float(x.y & 0xFFFF0000u);
}
// streaming (read-once) variants
__device__ __forceinline__ void ld4_stream(const float* p, float v[4]) {
  float4 x = __ldcs(reinterpret_cast<const float4*>(p));
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ld4_stream(const bf16* p, float v[4]) {
  uint2 x = __ldcs(reinterpret_cast<const uint2*>(p));
  v[0] = __uint_as_float(x.x << 16);
  v[1] = __uint_as_float(x.x & 0xFFFF0000u);
  v[2] = __uint_as_float(x.y << 16);
  v[3] = __uint_as_float(x.y & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}
__device__ __forceinline__ void st4(float* p, const float v[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st4(bf16* p, const float v[4]) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
}

// Packed 4-element loads: the raw registers as loaded, converted later.  Kernels
// issue every raw load of a thread first and convert afterwards, so that a
// thread's DRAM requests are all in flight together rather than one round trip
// per chunk.
template <typename T> struct Raw4;
template <> struct Raw4<float> { using type = float4; };
template <> struct Raw4<bf16> { using type = uint2; };
__device__ __forceinline__ float4 ldraw(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ uint2 ldraw(const bf16* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ float4 ldraw_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ uint2 ldraw_stream(const bf16* p) { return __ldcs(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ void cvt4(const float4& r, float v[4]) { v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w; }
__device__ __forceinline__ void cvt4(const uint2& r, float v[4]) {
  v[0] = __uint_as_float(r.x << 16);
  v[1] = __uint_as_float(r.x & 0xFFFF0000u);
  v[2] = __uint_as_float(r.y << 16);
  v[3] = __uint_as_float(r.y & 0xFFFF0000u);
}

// element-wise (unaligned / ragged) access
template <typename T> __device__ __forceinline__ float ld1(const T* p) { return to_f32(*p); }
template <typename T> __device__ __forceinline__ void st1(T* p, float v) { *p = from_f32<T>(v); }

// ---------------------------------------------------------------------------
// fixed-order reductions (deterministic)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the block; every thread gets the result.  `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();  // protect `red` from a previous use
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nwarps) ? red[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

__device__ __forceinline__ float inv_norm_from_sumsq(float ss) {
  // An exactly zero line or matrix gives a zero direction (no epsilon).  Any other
  // sum is divided through as it is: NaN stays NaN and Inf gives 0, so a non-finite
  // momentum propagates into the direction as the division M/||M|| defines it.
  return ss == 0.f ? 0.f : 1.0f / sqrtf(ss);
}

}  // namespace muon
