// AdamW for the parameters Muon does not update (biases, normalisation weights,
// out-of-block parameters; "Scaling Muon for Diffusion Transformers", summary
// page: these stay on AdamW, with an auxiliary group at LR 1e-4).
//
// One multi-tensor launch: every parameter of the list is cut into 4096-element
// blocks; each thread updates 4-element chunks with fp32 math:
//   m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g^2;
//   p <- p - lr*( (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + wd*p ).
// Bandwidth-bound: reads p, g, m, v and writes p, m, v.
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace muon {
namespace {

constexpr int ADAMW_MAX_PARAMS = 256;
constexpr int ADAMW_CHUNK = 4096;

struct AdamwEntry {
  void* P;
  const void* G;
  float* m;
  float* v;
  long long numel;
  int block_begin;
  int vec;
};
struct AdamwParams {
  AdamwEntry e[ADAMW_MAX_PARAMS];
  int n;
  int total_blocks;
  float lr, beta1, beta2, eps, wd;
  float omb1, omb2;    // 1 - beta1, 1 - beta2, formed in double precision on the host
  float inv_bc1;       // 1 / (1 - beta1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
};
static_assert(sizeof(AdamwParams) < 32000, "AdamwParams too large");

__device__ __forceinline__ float adamw_one(float& p, float g, float& m, float& v, const AdamwParams& q) {
  m = q.beta1 * m + q.omb1 * g;
  v = q.beta2 * v + q.omb2 * g * g;
  const float denom = sqrtf(v) * q.inv_sqrt_bc2 + q.eps;
  p = p - q.lr * ((m * q.inv_bc1) / denom + q.wd * p);
  return p;
}

// Elements i .. i+3 (those below numel) one at a time.
template <typename PT, typename GT>
__device__ __forceinline__ void adamw_tail(PT* P, const GT* G, const AdamwEntry& e, long long i, const AdamwParams& q) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (i + j < e.numel) {
      float p = ld1(P + i + j), m = e.m[i + j], v = e.v[i + j];
      adamw_one(p, ld1(G + i + j), m, v, q);
      st1(P + i + j, p);
      e.m[i + j] = m;
      e.v[i + j] = v;
    }
  }
}

template <typename PT, typename GT>
__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamwParams q) {
  int lo = 0, hi = q.n - 1;
  const int b = blockIdx.x;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (q.e[mid].block_begin <= b) lo = mid; else hi = mid - 1;
  }
  const AdamwEntry& e = q.e[lo];
  const long long e0 = (long long)(b - e.block_begin) * ADAMW_CHUNK;
  PT* P = reinterpret_cast<PT*>(e.P);
  const GT* G = reinterpret_cast<const GT*>(e.G);
  constexpr int KC = ADAMW_CHUNK / (256 * 4);
  if (e.vec) {
    // all loads of the block first, then the updates: one DRAM round trip per thread
    typename Raw4<PT>::type pr[KC];
    typename Raw4<GT>::type gr[KC];
    float4 mr[KC], vr[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const long long i = e0 + (long long)(k * 256 + threadIdx.x) * 4;
      if (i + 4 <= e.numel) {
        pr[k] = ldraw(P + i);
        gr[k] = ldraw_stream(G + i);
        mr[k] = ldraw(e.m + i);
        vr[k] = ldraw(e.v + i);
      }
    }
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const long long i = e0 + (long long)(k * 256 + threadIdx.x) * 4;
      if (i + 4 <= e.numel) {
        float p[4], g[4], m[4], v[4];
        cvt4(pr[k], p);
        cvt4(gr[k], g);
        cvt4(mr[k], m);
        cvt4(vr[k], v);
#pragma unroll
        for (int j = 0; j < 4; ++j) adamw_one(p[j], g[j], m[j], v[j], q);
        st4(P + i, p);
        st4(e.m + i, m);
        st4(e.v + i, v);
      } else {
        adamw_tail(P, G, e, i, q);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < KC; ++k) adamw_tail(P, G, e, e0 + (long long)(k * 256 + threadIdx.x) * 4, q);
  }
}

bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }
size_t dt_size(int dt) { return dt == MUON_DTYPE_BF16 ? 2 : 4; }

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" int muon_adamw_step(const muon_adamw_param* params, int n, int64_t t, float lr, double beta1,
                               double beta2, float eps, float weight_decay, muon_stream_t stream) {
  if (n < 0 || t < 1) return MUON_ERR_INVALID;
  if (n == 0) return MUON_OK;
  if (!params) return MUON_ERR_INVALID;
  if (!(beta1 >= 0.0 && beta1 < 1.0 && beta2 >= 0.0 && beta2 < 1.0 && eps >= 0.f)) return MUON_ERR_INVALID;
  const int p_dt = params[0].p_dtype, g_dt = params[0].g_dtype;
  for (int i = 0; i < n; ++i) {
    const muon_adamw_param& a = params[i];
    if (a.numel < 0) return MUON_ERR_INVALID;
    if (a.p_dtype != p_dt || a.g_dtype != g_dt) return MUON_ERR_UNSUPPORTED;
    if ((p_dt != MUON_DTYPE_F32 && p_dt != MUON_DTYPE_BF16) || (g_dt != MUON_DTYPE_F32 && g_dt != MUON_DTYPE_BF16))
      return MUON_ERR_UNSUPPORTED;
    if (a.numel == 0) continue;
    if (!a.P || !a.G || !a.m || !a.v) return MUON_ERR_INVALID;
    if (!is_aligned(a.P, dt_size(p_dt)) || !is_aligned(a.G, dt_size(g_dt)) || !is_aligned(a.m, 4) ||
        !is_aligned(a.v, 4))
      return MUON_ERR_INVALID;
  }
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3)
    return MUON_ERR_NO_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static thread_local AdamwParams q;
  const double bc1 = 1.0 - std::pow(beta1, (double)t);
  const double bc2 = 1.0 - std::pow(beta2, (double)t);
  int i = 0;
  while (i < n) {
    std::memset(&q, 0, sizeof(q));
    q.lr = lr;
    q.beta1 = (float)beta1;
    q.beta2 = (float)beta2;
    q.omb1 = (float)(1.0 - beta1);
    q.omb2 = (float)(1.0 - beta2);
    q.eps = eps;
    q.wd = weight_decay;
    q.inv_bc1 = (float)(1.0 / bc1);
    q.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
    int j = 0, blocks = 0;
    for (; i < n && j < ADAMW_MAX_PARAMS; ++i) {
      const muon_adamw_param& a = params[i];
      if (a.numel == 0) continue;
      AdamwEntry& e = q.e[j++];
      e.P = a.P;
      e.G = a.G;
      e.m = a.m;
      e.v = a.v;
      e.numel = a.numel;
      e.block_begin = blocks;
      e.vec = is_aligned(a.P, 4 * dt_size(p_dt)) && is_aligned(a.G, 4 * dt_size(g_dt)) && is_aligned(a.m, 16) &&
              is_aligned(a.v, 16);
      const long long nb = (a.numel + ADAMW_CHUNK - 1) / ADAMW_CHUNK;
      if ((long long)blocks + nb >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
      blocks += (int)nb;
    }
    q.n = j;
    q.total_blocks = blocks;
    if (j == 0) continue;
    const bool pb = p_dt == MUON_DTYPE_BF16, gb = g_dt == MUON_DTYPE_BF16;
    if (pb && gb) adamw_kernel<bf16, bf16><<<blocks, 256, 0, s>>>(q);
    else if (pb && !gb) adamw_kernel<bf16, float><<<blocks, 256, 0, s>>>(q);
    else if (!pb && gb) adamw_kernel<float, bf16><<<blocks, 256, 0, s>>>(q);
    else adamw_kernel<float, float><<<blocks, 256, 0, s>>>(q);
    if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
