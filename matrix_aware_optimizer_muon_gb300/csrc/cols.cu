// Single-pass RowNorm step for tall matrices (A > B), whose RowNorm lines are
// the B columns ("Scaling Muon for Diffusion Transformers", distributed-
// implementation paragraph: tall matrices reduce per-column norm scalars).
// Selected by MUON_DEBUG_TALL_CLUSTER; the default tall path is tall.cu, whose
// row-contiguous passes reach higher DRAM efficiency than these 32-column strips.
//
// A thread-block cluster of CL CTAs owns one strip of CW columns of one matrix;
// CTA k of the cluster owns rows [k*slab, (k+1)*slab).  Each CTA streams its slab
// once: M <- mu*M + G is kept in shared memory (and written back to global memory
// in the second phase), and per-column sums of squares are reduced inside the
// CTA.  After a cluster
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
// Cluster barrier whose arrival releases this thread's prior writes (used after
// the column partials are written to shared memory; no global stores are
// outstanding then, so the release is cheap).
__device__ __forceinline__ void cluster_sync_release() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;\n" ::
          : "memory");
}
// Cluster barrier that orders nothing: it only keeps every CTA's shared memory
// alive until its peers have finished reading it (those reads completed before
// the peers arrived, since their values were already used).
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile(
      "barrier.cluster.arrive.relaxed.aligned;\n"
      "barrier.cluster.wait.aligned;\n" ::
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
  constexpr int UNROLL1 = sizeof(GT) == 2 ? 6 : 4;   // rows of M and G in flight per thread
  constexpr int UNROLL2 = sizeof(WT) == 2 ? 12 : 6;  // rows of W in flight per thread
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

  // ---- pass over the slab: momentum, store, column sums of squares.
  // Raw (packed) loads of UNROLL1 rows are issued before any use.
  float cs[4] = {0.f, 0.f, 0.f, 0.f};
  for (int rb = r0 + trow; rb < r1; rb += RPI * UNROLL1) {
    float4 mr[UNROLL1];
    typename Raw4<GT>::type gr[UNROLL1];
#pragma unroll
    for (int u = 0; u < UNROLL1; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) {
        const size_t off = (size_t)r * B + c0 + tcol;
        mr[u] = *reinterpret_cast<const float4*>(Mg + off);
        gr[u] = ldraw_stream(Gg + off);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL1; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) {
        float g[4], v[4];
        cvt4(gr[u], g);
        v[0] = p.mu * mr[u].x + g[0];
        v[1] = p.mu * mr[u].y + g[1];
        v[2] = p.mu * mr[u].z + g[2];
        v[3] = p.mu * mr[u].w + g[3];
        st4(slabM + (size_t)(r - r0) * CW + tcol, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) cs[j] = fmaf(v[j], v[j], cs[j]);
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
  cluster_sync_release();
  if (threadIdx.x < CW) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < CL; ++q) t += dsmem_ld(&colpart[threadIdx.x], (uint32_t)q);
    if (rank == 0 && c0 + (int)threadIdx.x < B) note_nonfinite(p.status, t);
    inv[threadIdx.x] = inv_norm_from_sumsq(t);
  }
  __syncthreads();
  if (mt.nz && rank == 0 && threadIdx.x < 32) {   // telemetry: nonzero columns of this strip
    const int c = threadIdx.x;
    const unsigned nzb = __ballot_sync(0xffffffffu, c < CW && c0 + c < B && inv[c < CW ? c : 0] > 0.f);
    if (threadIdx.x == 0 && nzb) atomicAdd(mt.nz, __popc(nzb));
  }

  // ---- apply from shared memory
  float iv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) iv[j] = inv[tcol + j];
  for (int rb = r0 + trow; rb < r1; rb += RPI * UNROLL2) {
    typename Raw4<WT>::type wr[UNROLL2];
#pragma unroll
    for (int u = 0; u < UNROLL2; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) wr[u] = ldraw(Wg + (size_t)r * B + c0 + tcol);
    }
#pragma unroll
    for (int u = 0; u < UNROLL2; ++u) {
      const int r = rb + u * RPI;
      if (r < r1 && colok) {
        float w[4], m[4], o[4];
        cvt4(wr[u], w);
        ld4(slabM + (size_t)(r - r0) * CW + tcol, m);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = w[j] - p.eta * (mt.scale * (m[j] * iv[j]) + p.lam * w[j]);
        st4(Mg + (size_t)r * B + c0 + tcol, m);
        st4(Wg + (size_t)r * B + c0 + tcol, o);
      }
    }
  }
  // peers may still be reading this CTA's colpart
  cluster_sync_relaxed();
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

// Widest strip (32 or 16 columns) whose slab of fp32 momentum fits the
// shared-memory budget; 0 if none.  (The slab holds no G or W.)
int cols_strip_width(int max_rows, int /*stage_elem_bytes*/) {
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
