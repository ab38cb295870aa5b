// Newton-Schulz-5 GEMMs in fp32 on the CUDA cores (the fp32 NS5 mode).
//
// Same three products as the tensor-core path (S = X X^T; B = b S + c S S;
// X <- a X + B X, Eq. (2) of the "Muon is Scalable" notes, section 2.1) with the
// same fused epilogues, but every operand and intermediate stays fp32.  Outputs
// are computed on dense 64 x 64 tiles; S and S*S come out exactly symmetric
// because element (i, j) and element (j, i) accumulate the same products in the
// same order.
#include "common.cuh"
#include "internal.h"
#include "ns_common.cuh"

namespace muon {

constexpr int SB = 64, SK = 32;

__global__ void __launch_bounds__(256) ns_simt_kernel(const __grid_constant__ NsParams p) {
  __shared__ float As[SK][SB + 4];
  __shared__ float Bs[SK][SB + 4];
  const int t = blockIdx.x;
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= t) ++g;
  const NsGroup& G = p.g[g];
  const int lt = t - G.tile_begin;
  const int mat = lt / G.tiles_per_mat;
  const int rr = lt - mat * G.tiles_per_mat;
  const int tm = rr / G.ntiles, tn = rr - tm * G.ntiles;
  const int kind = p.kind;
  const int n = G.n, m = G.m;
  const int gm = G.mat_base + mat;

  const float* A;
  const float* B;
  int lda, ldb, K, ncols;
  if (kind == GEMM_GRAM) {
    A = reinterpret_cast<const float*>(G.opA) + (size_t)mat * G.stride_nm;
    B = A;
    lda = ldb = G.ld_m;
    K = m;
    ncols = n;
  } else if (kind == GEMM_POLY) {
    A = reinterpret_cast<const float*>(G.opA) + (size_t)mat * G.stride_nn;
    B = A;
    lda = ldb = G.ld_n;
    K = n;
    ncols = n;
  } else {
    A = reinterpret_cast<const float*>(G.opA) + (size_t)mat * G.stride_nn;
    B = reinterpret_cast<const float*>(G.opB) + (size_t)mat * G.stride_nm;
    lda = G.ld_n;
    ldb = G.ld_m;
    K = n;
    ncols = m;
  }

  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int row0 = tm * SB, col0 = tn * SB;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // Operand slices of SK columns of K: the next slice is loaded into registers while
  // the current one is multiplied out of shared memory (one barrier pair per slice).
  constexpr int PER = SB * SK / 256;   // elements of each operand per thread and slice
  float ra[PER], rb[PER];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int e = tid + q * 256;
      {
        const int i = e / SK, k = e - (e / SK) * SK;
        const int row = row0 + i;
        ra[q] = (row < n && k0 + k < K) ? A[(size_t)row * lda + k0 + k] : 0.f;
      }
      if (kind == GEMM_UPDATE) {
        const int k = e / SB, j = e - (e / SB) * SB;
        const int col = col0 + j;
        rb[q] = (k0 + k < K && col < ncols) ? B[(size_t)(k0 + k) * ldb + col] : 0.f;
      } else {
        const int j = e / SK, k = e - (e / SK) * SK;
        const int col = col0 + j;
        rb[q] = (col < ncols && k0 + k < K) ? B[(size_t)col * ldb + k0 + k] : 0.f;
      }
    }
  };
  load(0);
  for (int k0 = 0; k0 < K; k0 += SK) {
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int e = tid + q * 256;
      As[e - (e / SK) * SK][e / SK] = ra[q];
      if (kind == GEMM_UPDATE) Bs[e / SB][e - (e / SB) * SB] = rb[q];
      else Bs[e - (e / SK) * SK][e / SK] = rb[q];
    }
    __syncthreads();
    if (k0 + SK < K) load(k0 + SK);   // in flight during the products below
#pragma unroll
    for (int k = 0; k < SK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  const float inv = p.inv_norm ? p.inv_norm[gm] : 1.f;
  const float s_apply = p.rms_match * sqrtf((float)m);
  float osq = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= n) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = col0 + tx * 4 + j;
      if (c >= ncols) continue;
      float v = acc[i][j];
      if (kind == GEMM_GRAM) {
        if (p.first_iter) v *= inv * inv;
        reinterpret_cast<float*>(G.out)[(size_t)mat * G.stride_nn + (size_t)r * G.ld_n + c] = v;
      } else if (kind == GEMM_POLY) {
        const float s = reinterpret_cast<const float*>(G.epi_in)[(size_t)mat * G.stride_nn + (size_t)r * G.ld_n + c];
        reinterpret_cast<float*>(G.out)[(size_t)mat * G.stride_nn + (size_t)r * G.ld_n + c] = p.b * s + p.c * v;
      } else {
        const float x = reinterpret_cast<const float*>(G.epi_in)[(size_t)mat * G.stride_nm + (size_t)r * G.ld_m + c];
        const float sc = p.first_iter ? inv : 1.f;
        const float o = sc * (p.a * x + v);
        osq = fmaf(o, o, osq);
        if (p.last_iter && p.dst_mode != 2) ns_last_store(p, gm, n, m, r, c, o, s_apply);
        else reinterpret_cast<float*>(G.out)[(size_t)mat * G.stride_nm + (size_t)r * G.ld_m + c] = o;
      }
    }
  }
  if (kind == GEMM_UPDATE && p.last_iter && p.osq_part) {   // one partial per 64 x 64 tile
    __shared__ float red[32];
    const float t = block_sum(osq, red);
    if (threadIdx.x == 0) p.osq_part[blockIdx.x] = t;
  }
}

cudaError_t launch_ns_simt(const NsParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  ns_simt_kernel<<<p.total_tiles, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace muon
