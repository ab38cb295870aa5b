// Single-pass RowNorm step for tall matrices (A > B), whose RowNorm lines are
// the B columns ("Scaling Muon for Diffusion Transformers", distributed-
// implementation paragraph: tall matrices reduce per-column norm scalars).
//
// A thread-block cluster of CL CTAs owns one strip of CW columns of one matrix;
// CTA k of the cluster owns rows [k*slab, (k+1)*slab).  Each CTA streams its slab
// once: M <- mu*M + G is stored to global memory and kept in shared memory,
// and per-column sums of squares are reduced inside the CTA.  After a cluster
// barrier every CTA adds the CL column partials from its peers' shared memory
// in rank order (the same order everywhere, so the result is deterministic), and
// then applies W <- W - eta*(s*M/||column|| + lambda*W) from shared memory.
// HBM traffic: G 2 + M 4 + M 4 + W 2 + W 2 = 14 bytes per element (bf16 W/G),
// against 18 for the two-pass form that reads M and W again.
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace muon {

namespace {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;\n" ::
          : "memory");
}
// Load a float from the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float dsmem_ld(const float* local, uint32_t rank) {
  const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

template <typename WT, typename GT, int CW, int CL, int NT>
__global__ void __launch_bounds__(NT, 2) cols_cluster_kernel(const __grid_constant__ ColsParams p) {
  constexpr int TPR = CW / 4;       // threads per row (4 columns each)
  constexpr int RPI = NT / TPR;     // rows per pass of the CTA
  constexpr int UNROLL = 4;
  extern __shared__ __align__(16) float sm[];
  float* slabM = sm;                                  // [slab][CW]
  float* red = sm + (size_t)p.slab_max * CW;          // [NT/32][CW]
  float* colpart = red + (NT / 32) * CW;              // [CW]
  float* inv = colpart + CW;                          // [CW]

  const int unit = blockIdx.x / CL;
  const uint32_t rank = cluster_ctarank();
  int lo = 0, hi = p.nmat - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.mat[mid].unit_begin <= unit) lo = mid; else hi = mid - 1;
  }
  const ColsMat& mt = p.mat[lo];
  const int A = mt.rows, B = mt.cols;
  const int c0 = (unit - mt.unit_begin) * CW;
  const int slab = (A + CL - 1) / CL;
  const int r0 = (int)rank * slab;
  const int r1 = min(A, r0 + slab);
  const int tcol = (threadIdx.x % TPR) * 4;
  const int trow = threadIdx.x / TPR;
  const bool colok = c0 + tcol < B;  // B % 4 == 0: a 4-column chunk is wholly in or out
  float* __restrict__ Mg = mt.M;
  const GT* __restrict__ Gg = reinterpret_cast<const GT*>(mt.G);
  WT* __restrict__ Wg = reinterpret_cast<WT*>(mt.W);

  // ---- pass over the slab: momentum, store, column sums of squares
  float cs[4] = {0.f, 0.f, 0.f, 0.f};
  for (int rb = r0 + trow; rb < r1; rb += RPI * UNROLL) {
    float v[UNROLL][4];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) {
        const size_t off = (size_t)r * B + c0 + tcol;
        float g[4];
        ld4(Mg + off, v[u]);
        ld4_stream(Gg + off, g);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[u][j] = p.mu * v[u][j] + g[j];
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) {
        st4(Mg + (size_t)r * B + c0 + tcol, v[u]);
        st4(slabM + (size_t)(r - r0) * CW + tcol, v[u]);
#pragma unroll
        for (int j = 0; j < 4; ++j) cs[j] = fmaf(v[u][j], v[u][j], cs[j]);
      }
    }
  }
  // lanes tcol, tcol + TPR, ... of a warp share columns: fixed-order tree
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int o = TPR; o < 32; o <<= 1) cs[j] += __shfl_xor_sync(0xffffffffu, cs[j], o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane < TPR) {
#pragma unroll
    for (int j = 0; j < 4; ++j) red[warp * CW + tcol + j] = cs[j];
  }
  __syncthreads();
  if (threadIdx.x < CW) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) t += red[w * CW + threadIdx.x];
    colpart[threadIdx.x] = t;
  }
  // ---- cluster: add the CL slab partials in rank order
  cluster_sync_all();
  if (threadIdx.x < CW) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < CL; ++q) t += dsmem_ld(&colpart[threadIdx.x], (uint32_t)q);
    inv[threadIdx.x] = inv_norm_from_sumsq(t);
  }
  __syncthreads();

  // ---- apply from shared memory
  float iv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) iv[j] = inv[tcol + j];
  for (int rb = r0 + trow; rb < r1; rb += RPI * UNROLL) {
    float w[UNROLL][4];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) ld4(Wg + (size_t)r * B + c0 + tcol, w[u]);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) {
        float m[4], o[4];
        ld4(slabM + (size_t)(r - r0) * CW + tcol, m);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = w[u][j] - p.eta * (mt.scale * (m[j] * iv[j]) + p.lam * w[u][j]);
        st4(Wg + (size_t)r * B + c0 + tcol, o);
      }
    }
  }
  // peers may still be reading this CTA's colpart
  cluster_sync_all();
}

constexpr int kCL = 16;
constexpr int kNT = 512;

template <int CW>
size_t cols_smem_bytes(int slab_max) {
  return (size_t)slab_max * CW * 4 + (size_t)(kNT / 32) * CW * 4 + 2 * CW * 4;
}

template <typename WT, typename GT, int CW>
cudaError_t launch_cols_t(const ColsParams& p, cudaStream_t s) {
  auto kern = cols_cluster_kernel<WT, GT, CW, kCL, kNT>;
  const size_t smem = cols_smem_bytes<CW>(p.slab_max);
  static std::mutex mu;
  static std::map<int, bool> configured;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!configured[dev]) {
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess) return e;
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, COLS_MAX_SMEM)) != cudaSuccess)
        return e;
      configured[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.total_units * kCL, 1, 1);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidClusterSize;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CW>
cudaError_t launch_cols_cw(int w_dt, int g_dt, const ColsParams& p, cudaStream_t s) {
  const bool wb = w_dt == MUON_DTYPE_BF16, gb = g_dt == MUON_DTYPE_BF16;
  if (wb && gb) return launch_cols_t<bf16, bf16, CW>(p, s);
  if (wb && !gb) return launch_cols_t<bf16, float, CW>(p, s);
  if (!wb && gb) return launch_cols_t<float, bf16, CW>(p, s);
  return launch_cols_t<float, float, CW>(p, s);
}

}  // namespace

int cols_cluster_size() { return kCL; }

// Widest strip (32 or 16 columns) whose slab fits the shared-memory budget; 0 if none.
int cols_strip_width(int max_rows) {
  const int slab = (max_rows + kCL - 1) / kCL;
  if (cols_smem_bytes<32>(slab) <= COLS_SMEM_TARGET) return 32;
  if (cols_smem_bytes<16>(slab) <= COLS_MAX_SMEM) return 16;
  return 0;
}

cudaError_t launch_cols(int w_dt, int g_dt, int cw, const ColsParams& p, cudaStream_t s) {
  if (p.total_units <= 0) return cudaSuccess;
  if (cw == 32) return launch_cols_cw<32>(w_dt, g_dt, p, s);
  if (cw == 16) return launch_cols_cw<16>(w_dt, g_dt, p, s);
  return cudaErrorInvalidValue;
}

}  // namespace muon
