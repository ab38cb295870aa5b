// Bandwidth-bound kernels of the Muon step.
//
//  * ew_tile_kernel: one pass over 64 x 128 tiles of M (and G, W) doing any
//    combination of: momentum M <- mu*M + G ("Muon is Scalable" notes, section
//    2.1, Eq. (1)); per-tile sum of squares for ||M||_F (section 2.1, X0 = M/||M||_F);
//    the bf16/fp32 copy X~ of M on the short-side orientation that feeds the
//    Newton-Schulz GEMMs; per-tile line partial sums for RowNorm; and the second
//    RowNorm pass W <- W - eta*(s*M/||line|| + lambda*W) (Eq. (4) with the
//    Periodic Row-wise scale).
//  * rows_kernel: the whole RowNorm step for a wide/square matrix in one pass:
//    one CTA per row keeps the row in registers (momentum, row norm, apply);
//    rows_wide_kernel: the same for rows of 6145..12288 columns, shaped for two
//    CTAs per SM.
//  * apply_kernel: W <- W - eta*(s*U + lambda*W) from a given direction U.
//  * fro_final_kernel / line_final_kernel: fixed-order reductions of partials.
//
// Every reduction has a fixed order, so results are bit-reproducible.
#include "common.cuh"
#include "internal.h"

// Target four-element chunks per thread of the one-row-per-CTA RowNorm kernel.
#ifndef MUON_ROWS_CPT
#define MUON_ROWS_CPT 3
#endif

namespace muon {

template <typename T, int N>
struct alignas(16) Arr { T v[N]; };

__device__ __forceinline__ int find_mat_ew(const EwParams& p, int t) {
  int lo = 0, hi = p.nmat - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.mat[mid].tile_begin <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The refresh step's momentum pass (modes with EW_XT) is held to three CTAs per SM:
// measured 13% faster on the 1.3B set than at the two its registers would allow.
template <typename WT, typename GT, typename XT, int MODE>
__global__ void __launch_bounds__(EW_THREADS, (MODE & EW_XT) ? 3 : 1)
ew_tile_kernel(const __grid_constant__ EwParams p) {
  constexpr bool kMom = (MODE & EW_MOMENTUM) != 0;
  constexpr bool kFro = (MODE & EW_FRO) != 0;
  constexpr bool kXT = (MODE & EW_XT) != 0;
  constexpr bool kLine = (MODE & EW_LINEPART) != 0;
  constexpr bool kApply = (MODE & EW_APPLY_LINE) != 0;
  constexpr bool kR = (MODE & EW_WRITE_R) != 0;
  constexpr int RPT = TILE_R / (EW_THREADS / 32);  // rows per thread = 8

  __shared__ float red[32];

  const int t = blockIdx.x;
  const int mi = find_mat_ew(p, t);
  const EwMat& mt = p.mat[mi];
  const int lt = t - mt.tile_begin;
  const int tr = lt / mt.tiles_c;
  const int tc = lt - tr * mt.tiles_c;
  const int r0 = tr * TILE_R, c0 = tc * TILE_C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = mt.rows, cols = mt.cols;
  const int cb = c0 + lane * 4;
  const bool vec = mt.vec && (cb + 4 <= cols);
  float* __restrict__ Mp = mt.M;

  float v[RPT][4];
  float w[kApply ? RPT : 1][4];
  float inv_col[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (kApply || kR) {
    if (mt.tall) {
#pragma unroll
      for (int j = 0; j < 4; ++j) inv_col[j] = (cb + j < cols) ? mt.line_inv[cb + j] : 0.f;
    }
  }

  // ---- load (and momentum) ----
  if (vec) {
    // every row's loads are issued before any is used: one DRAM round trip per tile
    float4 mr[RPT];
    typename Raw4<GT>::type gr[kMom ? RPT : 1];
    typename Raw4<WT>::type wr[kApply ? RPT : 1];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + warp + (EW_THREADS / 32) * i;
      const size_t off = (size_t)r * (size_t)cols + (size_t)cb;
      if (r < rows) {
        mr[i] = ldraw(Mp + off);
        if constexpr (kMom) gr[i] = ldraw_stream(reinterpret_cast<const GT*>(mt.G) + off);
        if constexpr (kApply) wr[i] = ldraw(reinterpret_cast<const WT*>(mt.W) + off);
      }
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + warp + (EW_THREADS / 32) * i;
      if (r < rows) {
        cvt4(mr[i], v[i]);
        if constexpr (kMom) {
          float g[4];
          cvt4(gr[i], g);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[i][j] = p.mu * v[i][j] + g[j];
        }
        if constexpr (kApply) cvt4(wr[i], w[i]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[i][j] = 0.f;
          if constexpr (kApply) w[i][j] = 0.f;
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + warp + (EW_THREADS / 32) * i;
      const bool rok = r < rows;
      const size_t off = (size_t)r * (size_t)cols + (size_t)cb;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = rok && (cb + j < cols);
        float m = ok ? Mp[off + j] : 0.f;
        if constexpr (kMom) {
          if (ok) m = p.mu * m + ld1(reinterpret_cast<const GT*>(mt.G) + off + j);
        }
        v[i][j] = m;
        if constexpr (kApply) w[i][j] = ok ? ld1(reinterpret_cast<const WT*>(mt.W) + off + j) : 0.f;
      }
    }
  }

  // ---- store momentum ----
  if constexpr (kMom) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + warp + (EW_THREADS / 32) * i;
      if (r >= rows) continue;
      const size_t off = (size_t)r * (size_t)cols + (size_t)cb;
      if (vec) {
        st4(Mp + off, v[i]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (cb + j < cols) Mp[off + j] = v[i][j];
      }
    }
  }

  // ---- per-tile sum of squares (Frobenius partial) ----
  if constexpr (kFro) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(v[i][j], v[i][j], ss);
    ss = block_sum(ss, red);
    if (threadIdx.x == 0) mt.part[lt] = ss;
  }

  // ---- line partials ----
  if constexpr (kLine) {
    if (mt.tall) {
      // columns are the lines: sum over this tile's 64 rows, fixed order
      __shared__ float colred[EW_THREADS / 32][TILE_C];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) s = fmaf(v[i][j], v[i][j], s);
        colred[warp][lane * 4 + j] = s;
      }
      __syncthreads();
      if (threadIdx.x < TILE_C) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < EW_THREADS / 32; ++k) s += colred[k][threadIdx.x];
        const int c = c0 + threadIdx.x;
        if (c < cols) mt.line_part[(size_t)tr * cols + c] = s;
      }
    } else {
      // rows are the lines: sum over this tile's 128 columns
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) s = fmaf(v[i][j], v[i][j], s);
        s = warp_sum(s);
        const int r = r0 + warp + (EW_THREADS / 32) * i;
        if (lane == 0 && r < rows) mt.line_part[(size_t)tc * rows + r] = s;
      }
    }
  }

  // ---- RowNorm output or apply ----
  if constexpr (kApply || kR) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = r0 + warp + (EW_THREADS / 32) * i;
      if (r >= rows) continue;
      const float inv_row = mt.tall ? 0.f : mt.line_inv[r];
      float u[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) u[j] = v[i][j] * (mt.tall ? inv_col[j] : inv_row);
      const size_t off = (size_t)r * (size_t)cols + (size_t)cb;
      if constexpr (kR) {
        float* R = reinterpret_cast<float*>(mt.aux);
        if (vec) st4(R + off, u);
        else {
#pragma unroll
          for (int j = 0; j < 4; ++j) if (cb + j < cols) R[off + j] = u[j];
        }
      }
      if constexpr (kApply) {
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = w[i][j] - p.eta * (mt.scale * u[j] + p.lam * w[i][j]);
        WT* Wp = reinterpret_cast<WT*>(mt.W);
        if (vec) st4(Wp + off, o);
        else {
#pragma unroll
          for (int j = 0; j < 4; ++j) if (cb + j < cols) st1(Wp + off + j, o[j]);
        }
      }
    }
  }

  // ---- X~ on the short-side orientation ----
  if constexpr (kXT) {
    XT* X = reinterpret_cast<XT*>(mt.aux);
    const int ld = mt.ld_aux;
    if (!mt.tall) {
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = r0 + warp + (EW_THREADS / 32) * i;
        if (r >= rows) continue;
        const size_t off = (size_t)r * ld + cb;
        if (cb + 4 <= cols) st4(X + off, v[i]);
        else {
#pragma unroll
          for (int j = 0; j < 4; ++j) if (cb + j < cols) st1(X + off + j, v[i][j]);
        }
      }
    } else {
      // X~ = M^T: stage the tile transposed in shared memory, then write rows of X~.
      constexpr int PAD = 2;
      __shared__ XT tb[TILE_C][TILE_R + PAD];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int rl = warp + (EW_THREADS / 32) * i;
#pragma unroll
        for (int j = 0; j < 4; ++j) tb[lane * 4 + j][rl] = from_f32<XT>(v[i][j]);
      }
      __syncthreads();
      const int rr = r0 + 2 * lane;  // this lane's two M rows = two X~ columns
#pragma unroll 4
      for (int k = 0; k < TILE_C / (EW_THREADS / 32); ++k) {
        const int cl = warp + (EW_THREADS / 32) * k;
        const int c = c0 + cl;
        if (c >= cols) continue;
        XT* dst = X + (size_t)c * ld + rr;
        if (rr + 1 < rows) {
          if constexpr (sizeof(XT) == 2) {
            // rr is even and ld a multiple of 8: one 4-byte store of the pair
            *reinterpret_cast<__nv_bfloat162*>(dst) = *reinterpret_cast<const __nv_bfloat162*>(&tb[cl][2 * lane]);
          } else {
            dst[0] = tb[cl][2 * lane];
            dst[1] = tb[cl][2 * lane + 1];
          }
        } else if (rr < rows) {
          dst[0] = tb[cl][2 * lane];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// single-pass RowNorm step, rows of a wide/square matrix
// ---------------------------------------------------------------------------
__device__ __forceinline__ int find_mat_rows(const RowsParams& p, int t) {
  int lo = 0, hi = p.nmat - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.mat[mid].row_begin <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename WT, typename GT, int CPT>
__global__ void __launch_bounds__(1024)
rows_kernel(const __grid_constant__ RowsParams p) {
  __shared__ float red[32];
  const int rg = blockIdx.x;
  const RowsMat& mt = p.mat[find_mat_rows(p, rg)];
  const int r = rg - mt.row_begin;
  const int cols = mt.cols;
  const size_t base = (size_t)r * (size_t)cols;
  float* __restrict__ Mp = mt.M + base;
  const GT* __restrict__ Gp = reinterpret_cast<const GT*>(mt.G) + base;
  WT* __restrict__ Wp = reinterpret_cast<WT*>(mt.W) + base;

  float v[CPT][4], w[CPT][4];
  float ss = 0.f;
  if (mt.vec) {
    // every chunk's loads are issued before any is used: one DRAM round trip per row
    float4 mr[CPT];
    typename Raw4<GT>::type gr[CPT];
    typename Raw4<WT>::type wr[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      const int c = (threadIdx.x + k * blockDim.x) * 4;
      if (c + 4 <= cols) {
        mr[k] = ldraw(Mp + c);
        gr[k] = ldraw_stream(Gp + c);
        wr[k] = ldraw(Wp + c);
      }
    }
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      const int c = (threadIdx.x + k * blockDim.x) * 4;
      float g[4];
      if (c + 4 <= cols) {
        cvt4(mr[k], v[k]);
        cvt4(gr[k], g);
        cvt4(wr[k], w[k]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[k][j] = g[j] = w[k][j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[k][j] = p.mu * v[k][j] + g[j];
        ss = fmaf(v[k][j], v[k][j], ss);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      const int c = (threadIdx.x + k * blockDim.x) * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = c + j < cols;
        v[k][j] = ok ? p.mu * Mp[c + j] + ld1(Gp + c + j) : 0.f;
        w[k][j] = ok ? ld1(Wp + c + j) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(v[k][j], v[k][j], ss);
    }
  }
  const float sst = block_sum(ss, red);
  if (threadIdx.x == 0) note_nonfinite(p.status, sst);
  const float inv = inv_norm_from_sumsq(sst);
  if (mt.nz && threadIdx.x == 0 && inv > 0.f) atomicAdd(mt.nz, 1);   // telemetry: nonzero rows
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 4;
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = w[k][j] - p.eta * (mt.scale * (v[k][j] * inv) + p.lam * w[k][j]);
    if (mt.vec && c + 4 <= cols) {
      st4(Mp + c, v[k]);
      st4(Wp + c, o);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c + j < cols) { Mp[c + j] = v[k][j]; st1(Wp + c + j, o[j]); }
    }
  }
}

// Rows of 6145..12288 columns: 512 threads with 4-6 four-element chunks each, at
// most 64 registers a thread (the 1024-thread bound), so two CTAs per SM and one
// row's reduction and stores overlap another's loads.  The general kernel above
// takes up to 1024 threads here, one CTA per SM (measured 5.7 against 7.1 TB/s on
// 2560 x 10240 matrices).  The element-load path is a kernel of its own
// (kVec = false), so that its registers do not count against the vector path.
//
// RowNorm of one row with cols % 4 != 0 or unaligned bases: element loads.
template <typename WT, typename GT, int CPT>
__device__ __forceinline__ void rows_scalar(float* __restrict__ Mp, const GT* __restrict__ Gp, WT* __restrict__ Wp,
                                         int cols, float scale, int* nz, float mu, float eta, float lam,
                                         float* red, unsigned int* status) {
  float v[CPT][4], w[CPT][4];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = c + j < cols;
      v[k][j] = ok ? mu * Mp[c + j] + ld1(Gp + c + j) : 0.f;
      w[k][j] = ok ? ld1(Wp + c + j) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) ss = fmaf(v[k][j], v[k][j], ss);
  }
  const float sst = block_sum(ss, red);
  if (threadIdx.x == 0) note_nonfinite(status, sst);
  const float inv = inv_norm_from_sumsq(sst);
  if (nz && threadIdx.x == 0 && inv > 0.f) atomicAdd(nz, 1);   // telemetry: nonzero rows
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = (threadIdx.x + k * blockDim.x) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c + j < cols) {
        Mp[c + j] = v[k][j];
        st1(Wp + c + j, w[k][j] - eta * (scale * (v[k][j] * inv) + lam * w[k][j]));
      }
  }
}

// kVec: every matrix of the launch has vec set (cols % 4 == 0, aligned bases).
template <typename WT, typename GT, int CPT, bool kVec>
__global__ void __launch_bounds__(1024)
rows_wide_kernel(const __grid_constant__ RowsParams p) {
  __shared__ float red[32];
  const int rg = blockIdx.x;
  const RowsMat& mt = p.mat[find_mat_rows(p, rg)];
  const int r = rg - mt.row_begin;
  const int cols = mt.cols;
  const size_t base = (size_t)r * (size_t)cols;
  float* __restrict__ Mp = mt.M + base;
  const GT* __restrict__ Gp = reinterpret_cast<const GT*>(mt.G) + base;
  WT* __restrict__ Wp = reinterpret_cast<WT*>(mt.W) + base;

  float ss = 0.f;
  if constexpr (kVec) {
    // Every chunk's loads are issued before any is used: one DRAM round trip per
    // row.  The raw registers start at zero and only the loads are conditional, so
    // the conversions below run unconditionally and no load can be moved down to
    // a use under the same bound (which serialises the round trips).
    float v[CPT][4], w[CPT][4];
    {
      float4 mr[CPT] = {};
      typename Raw4<GT>::type gr[CPT] = {};
      typename Raw4<WT>::type wr[CPT] = {};
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const int c = (threadIdx.x + k * blockDim.x) * 4;
        if (c + 4 <= cols) {
          mr[k] = ldraw(Mp + c);
          gr[k] = ldraw_stream(Gp + c);
          wr[k] = ldraw(Wp + c);
        }
      }
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        float g[4];
        cvt4(mr[k], v[k]);
        cvt4(gr[k], g);
        cvt4(wr[k], w[k]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[k][j] = p.mu * v[k][j] + g[j];
          ss = fmaf(v[k][j], v[k][j], ss);
        }
      }
    }
    const float sst = block_sum(ss, red);
    if (threadIdx.x == 0) note_nonfinite(p.status, sst);
    const float inv = inv_norm_from_sumsq(sst);
    if (mt.nz && threadIdx.x == 0 && inv > 0.f) atomicAdd(mt.nz, 1);   // telemetry: nonzero rows
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      const int c = (threadIdx.x + k * blockDim.x) * 4;
      if (c + 4 <= cols) {   // cols % 4 == 0 here: a chunk is whole or past the row
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = w[k][j] - p.eta * (mt.scale * (v[k][j] * inv) + p.lam * w[k][j]);
        st4(Mp + c, v[k]);
        st4(Wp + c, o);
      }
    }
  } else {
    rows_scalar<WT, GT, CPT>(Mp, Gp, Wp, cols, mt.scale, mt.nz, p.mu, p.eta, p.lam, red, p.status);
  }
}

// ---------------------------------------------------------------------------
// apply from a given direction
// ---------------------------------------------------------------------------
template <typename WT, typename UT>
__global__ void __launch_bounds__(256)
apply_kernel(const __grid_constant__ ApplyParams p) {
  int lo = 0, hi = p.nmat - 1;
  const int b = blockIdx.x;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.mat[mid].block_begin <= b) lo = mid; else hi = mid - 1;
  }
  const ApplyMat& mt = p.mat[lo];
  const long long e0 = (long long)(b - mt.block_begin) * APPLY_CHUNK;
  WT* Wp = reinterpret_cast<WT*>(mt.W);
  const UT* Up = reinterpret_cast<const UT*>(mt.U);
  constexpr int KC = APPLY_CHUNK / (256 * 4);
  if (mt.vec) {
    // all loads of the block first, then the updates: one DRAM round trip per thread
    typename Raw4<WT>::type wr[KC];
    typename Raw4<UT>::type ur[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const long long e = e0 + (long long)(k * 256 + threadIdx.x) * 4;
      if (e + 4 <= mt.numel) {
        wr[k] = ldraw(Wp + e);
        ur[k] = ldraw_stream(Up + e);
      }
    }
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const long long e = e0 + (long long)(k * 256 + threadIdx.x) * 4;
      if (e + 4 <= mt.numel) {
        float w[4], u[4], o[4];
        cvt4(wr[k], w);
        cvt4(ur[k], u);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = w[j] - p.eta * (mt.scale * u[j] + p.lam * w[j]);
        st4(Wp + e, o);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (e + j < mt.numel) {
            const float w = ld1(Wp + e + j), u = ld1(Up + e + j);
            st1(Wp + e + j, w - p.eta * (mt.scale * u + p.lam * w));
          }
        }
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const long long e = e0 + (long long)(k * 256 + threadIdx.x) * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (e + j < mt.numel) {
          const float w = ld1(Wp + e + j), u = ld1(Up + e + j);
          st1(Wp + e + j, w - p.eta * (mt.scale * u + p.lam * w));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// fixed-order finalisers
// ---------------------------------------------------------------------------
__device__ __forceinline__ double block_sum_f64(double v, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (warp == 0) {
    t = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  }
  return t;
}

// One CTA per matrix: ||M_i||^2 = sum of the matrix's tile partials (fixed order).
__global__ void __launch_bounds__(256)
fro_final_kernel(const __grid_constant__ FroFinalParams p) {
  __shared__ double red[32];
  const int i = blockIdx.x;
  const int b = p.begin[i], e = p.begin[i] + p.count[i];
  double s = 0.0;
  for (int t = b + threadIdx.x; t < e; t += blockDim.x) s += (double)p.part[t];
  s = block_sum_f64(s, red);
  if (threadIdx.x == 0) {
    const int o = p.out_index[i];
    const float ss = (float)s;
    note_nonfinite(p.status, ss);
    if (p.fro_sq) p.fro_sq[o] = ss;
    if (p.inv_norm) p.inv_norm[o] = inv_norm_from_sumsq(ss);
    if (p.fro) p.fro[o] = sqrtf(ss);
  }
}

// One thread per line: inv[l] = 1/sqrt(sum over the partial rows), fixed order.
__global__ void __launch_bounds__(256)
line_final_kernel(const __grid_constant__ LineFinalParams p) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= p.total_lines) return;
  int lo = 0, hi = p.nmat - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.mat[mid].line_begin <= g) lo = mid; else hi = mid - 1;
  }
  const LineFinalMat& mt = p.mat[lo];
  const int l = g - mt.line_begin;
  double s = 0.0;
  for (int q = 0; q < mt.parts; ++q) s += (double)mt.part[(size_t)q * mt.lines + l];
  note_nonfinite(p.status, (float)s);
  const float inv = inv_norm_from_sumsq((float)s);
  mt.inv[l] = inv;
  if (mt.nz && inv > 0.f) atomicAdd(mt.nz, 1);   // telemetry: nonzero lines
}

// One CTA per matrix: sum of the O^2 partials (fixed order) -> RMS(O) and the
// Eq. (6) scale rms_match / RMS(O) (zero for a zero output).
__global__ void __launch_bounds__(256)
osq_final_kernel(const __grid_constant__ OsqFinalParams p) {
  __shared__ double red[32];
  const int i = blockIdx.x;
  const long long b = p.begin[i];
  double s = 0.0;
  for (int t = threadIdx.x; t < p.count[i]; t += blockDim.x) s += (double)p.part[b + t];
  s = block_sum_f64(s, red);
  if (threadIdx.x == 0) {
    const int o = p.out_index[i];
    const double r = p.numel[i] > 0 ? sqrt(s / p.numel[i]) : 0.0;
    if (p.rms_out) p.rms_out[o] = (float)r;
    if (p.scale_out) p.scale_out[o] = r > 0.0 ? (float)(p.rms_match / r) : 0.f;
  }
}

// RMS of a RowNorm direction: every nonzero line has unit norm, so RMS^2 = nz / (A*B).
__global__ void nz_rms_kernel(const __grid_constant__ NzRmsParams p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.nmat) return;
  const int o = p.out_index[i];
  p.rms_out[o] = p.numel[i] > 0 ? (float)sqrt((double)p.nz[o] / p.numel[i]) : 0.f;
}

// 8 consecutive bf16 values <-> float[8]; the pointer is 16-byte aligned
__device__ __forceinline__ void load_bf16x8(const bf16* p, float v[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    v[2 * h] = __uint_as_float(w[h] << 16);
    v[2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void store_bf16x8(bf16* p, const float v[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// W <- W - eta*(scale*O + lambda*W) for O kept in the workspace on the short side
// (n x m, leading dimension ld).  64 x 64 tiles of O pass through shared memory so
// that a tall W (m x n, W[c][r] = update of O[r][c]) is read and written along its
// rows too.
// Element idx of a 64 x 64 tile of O (n x m) and the W element it updates:
// W is n x m (wide; consecutive idx walk a row of W and of O) or m x n (tall;
// consecutive idx walk a row of W, a column of O).
__device__ __forceinline__ void applyws_coords(bool tall, int idx, int r0, int c0, int n, int m, int& rr,
                                               int& cc, size_t& widx) {
  if (!tall) {
    rr = idx / APPLYWS_TILE;
    cc = idx % APPLYWS_TILE;
    widx = (size_t)(r0 + rr) * m + (c0 + cc);
  } else {
    cc = idx / APPLYWS_TILE;
    rr = idx % APPLYWS_TILE;
    widx = (size_t)(c0 + cc) * n + (r0 + rr);
  }
}

template <typename WT, typename OT>
__global__ void __launch_bounds__(256)
apply_ws_kernel(const __grid_constant__ ApplyWsParams p) {
  __shared__ float t[APPLYWS_TILE][APPLYWS_TILE + 1];
  int lo = 0, hi = p.nmat - 1;
  const int b = blockIdx.x;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.mat[mid].tile_begin <= b) lo = mid; else hi = mid - 1;
  }
  const ApplyWsMat& mt = p.mat[lo];
  const int lt = b - mt.tile_begin;
  const int tr = lt / mt.tiles_c, tc = lt - tr * mt.tiles_c;
  const int r0 = tr * APPLYWS_TILE, c0 = tc * APPLYWS_TILE;
  const int n = mt.n, m = mt.m;
  const OT* O = reinterpret_cast<const OT*>(mt.O);
  const bf16* L = reinterpret_cast<const bf16*>(mt.O_lo);
  constexpr int PER = APPLYWS_TILE * APPLYWS_TILE / 256;   // elements per thread (256 threads)
  constexpr bool kBf16 = sizeof(WT) == 2 && sizeof(OT) == 2;
  if constexpr (kBf16) {
    // O (and its residual) as 8-element vectors: lane v takes row v / 8 of the tile,
    // columns (v % 8) * 8 .. + 7 (rows of O are 16-byte aligned: ld is a multiple of 8)
    float f[PER / 8][8];
#pragma unroll
    for (int q = 0; q < PER / 8; ++q) {
      const int v = threadIdx.x + q * 256;
      const int r = r0 + (v >> 3), c = c0 + (v & 7) * 8;
      const size_t off = (size_t)r * mt.ld + c;
      if (mt.ovec && r < n && c + 8 <= m) {
        float lo[8];
        load_bf16x8(O + off, f[q]);
        if (L) {
          load_bf16x8(L + off, lo);
#pragma unroll
          for (int k = 0; k < 8; ++k) f[q][k] += lo[k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          f[q][k] = 0.f;
          if (r < n && c + k < m) f[q][k] = to_f32(O[off + k]) + (L ? __bfloat162float(L[off + k]) : 0.f);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < PER / 8; ++q) {
      const int v = threadIdx.x + q * 256;
#pragma unroll
      for (int k = 0; k < 8; ++k) t[v >> 3][(v & 7) * 8 + k] = f[q][k];
    }
  } else {
    float ov[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int idx = threadIdx.x + q * 256;
      const int r = r0 + idx / APPLYWS_TILE, c = c0 + idx % APPLYWS_TILE;
      ov[q] = 0.f;
      if (r < n && c < m) {
        const size_t off = (size_t)r * mt.ld + c;
        ov[q] = to_f32(O[off]);
        if (L) ov[q] += __bfloat162float(L[off]);
      }
    }
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int idx = threadIdx.x + q * 256;
      t[idx / APPLYWS_TILE][idx % APPLYWS_TILE] = ov[q];
    }
  }
  __syncthreads();
  const float sc = p.scale[mt.scale_index];
  WT* W = reinterpret_cast<WT*>(mt.W);
  if constexpr (kBf16) {
    if (mt.vec) {
      // W in its own orientation as 8-element row segments: lane v takes W row v / 8 of
      // the tile and W columns (v % 8) * 8 .. + 7 (a wide W row is an O row; a tall W
      // row is an O column, read from the tile transposed)
      float wv[PER / 8][8];
      bool ok[PER / 8];
      size_t widx[PER / 8];
#pragma unroll
      for (int q = 0; q < PER / 8; ++q) {
        const int v = threadIdx.x + q * 256;
        const int a = v >> 3, e = (v & 7) * 8;
        if (!mt.tall) {
          ok[q] = r0 + a < n && c0 + e + 8 <= m;
          widx[q] = (size_t)(r0 + a) * m + (c0 + e);
        } else {
          ok[q] = c0 + a < m && r0 + e + 8 <= n;
          widx[q] = (size_t)(c0 + a) * n + (r0 + e);
        }
        if (ok[q]) load_bf16x8(W + widx[q], wv[q]);
      }
#pragma unroll
      for (int q = 0; q < PER / 8; ++q) {
        const int v = threadIdx.x + q * 256;
        const int a = v >> 3, e = (v & 7) * 8;
        if (ok[q]) {
          float o[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float u = mt.tall ? t[e + k][a] : t[a][e + k];
            o[k] = wv[q][k] - p.eta * (sc * u + p.lam * wv[q][k]);
          }
          store_bf16x8(W + widx[q], o);
        } else {
          // ragged edge of the matrix: element by element
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = mt.tall ? e + k : a, cc = mt.tall ? a : e + k;
            if (r0 + rr < n && c0 + cc < m) {
              const size_t wi = mt.tall ? (size_t)(c0 + cc) * n + (r0 + rr) : (size_t)(r0 + rr) * m + (c0 + cc);
              const float w = ld1(W + wi);
              st1(W + wi, w - p.eta * (sc * t[rr][cc] + p.lam * w));
            }
          }
        }
      }
      return;
    }
  }
  // every element's W load is issued before the first store (one DRAM round trip)
  float wv[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int idx = threadIdx.x + q * 256;
    int rr, cc;
    size_t widx;
    applyws_coords(mt.tall, idx, r0, c0, n, m, rr, cc, widx);
    wv[q] = (r0 + rr < n && c0 + cc < m) ? ld1(W + widx) : 0.f;
  }
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int idx = threadIdx.x + q * 256;
    int rr, cc;
    size_t widx;
    applyws_coords(mt.tall, idx, r0, c0, n, m, rr, cc, widx);
    if (r0 + rr < n && c0 + cc < m) st1(W + widx, wv[q] - p.eta * (sc * t[rr][cc] + p.lam * wv[q]));
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <typename WT, typename GT, typename XT>
static cudaError_t launch_ew_t(int mode, const EwParams& p, cudaStream_t s) {
  const dim3 grid(p.total_tiles), block(EW_THREADS);
  switch (mode) {
#define MUON_EW_CASE(M) \
  case (M): ew_tile_kernel<WT, GT, XT, (M)><<<grid, block, 0, s>>>(p); break;
    MUON_EW_CASE(EW_MOMENTUM)
    MUON_EW_CASE(EW_MOMENTUM | EW_FRO)
    MUON_EW_CASE(EW_MOMENTUM | EW_FRO | EW_XT)
    MUON_EW_CASE(EW_FRO | EW_XT)
    MUON_EW_CASE(EW_FRO)
    MUON_EW_CASE(EW_MOMENTUM | EW_LINEPART)
    MUON_EW_CASE(EW_LINEPART)
    MUON_EW_CASE(EW_APPLY_LINE)
    MUON_EW_CASE(EW_WRITE_R)
#undef MUON_EW_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_ew(int mode, int w_dt, int g_dt, int x_dt, const EwParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const bool wb = w_dt == MUON_DTYPE_BF16, gb = g_dt == MUON_DTYPE_BF16, xb = x_dt == MUON_DTYPE_BF16;
  if (wb && gb) return xb ? launch_ew_t<bf16, bf16, bf16>(mode, p, s) : launch_ew_t<bf16, bf16, float>(mode, p, s);
  if (wb && !gb) return xb ? launch_ew_t<bf16, float, bf16>(mode, p, s) : launch_ew_t<bf16, float, float>(mode, p, s);
  if (!wb && gb) return xb ? launch_ew_t<float, bf16, bf16>(mode, p, s) : launch_ew_t<float, bf16, float>(mode, p, s);
  return xb ? launch_ew_t<float, float, bf16>(mode, p, s) : launch_ew_t<float, float, float>(mode, p, s);
}

template <typename WT, typename GT>
static cudaError_t launch_rows_t(int max_cols, const RowsParams& p, cudaStream_t s) {
  // At most 3-4 four-element chunks per thread keeps registers low and many
  // threads resident; rows up to 16384 columns use at most 1024 threads.
  const int chunks = (max_cols + 3) / 4;
  // 6145..12288 columns (8192 for fp32 W and G, whose five- and six-chunk kernels
  // spill): rows_wide_kernel, 512 threads
  if (chunks > 3 * 512 && chunks <= (sizeof(WT) + sizeof(GT) == 8 ? 4 : 6) * 512) {
    bool vec = true;
    for (int i = 0; i < p.nmat; ++i) vec = vec && p.mat[i].vec;
    const dim3 grid(p.total_rows), block(512);
    if (chunks <= 4 * 512) {
      if (vec) rows_wide_kernel<WT, GT, 4, true><<<grid, block, 0, s>>>(p);
      else rows_wide_kernel<WT, GT, 4, false><<<grid, block, 0, s>>>(p);
    } else if (chunks <= 5 * 512) {
      if (vec) rows_wide_kernel<WT, GT, 5, true><<<grid, block, 0, s>>>(p);
      else rows_wide_kernel<WT, GT, 5, false><<<grid, block, 0, s>>>(p);
    } else {
      if (vec) rows_wide_kernel<WT, GT, 6, true><<<grid, block, 0, s>>>(p);
      else rows_wide_kernel<WT, GT, 6, false><<<grid, block, 0, s>>>(p);
    }
    return cudaGetLastError();
  }
  int T = ((chunks + MUON_ROWS_CPT - 1) / MUON_ROWS_CPT + 31) / 32 * 32;
  T = T < 64 ? 64 : (T > 1024 ? 1024 : T);
  const int cpt = (chunks + T - 1) / T;
  const dim3 grid(p.total_rows), block(T);
  switch (cpt) {
#define MUON_ROWS_CASE(C) \
  case (C): rows_kernel<WT, GT, (C)><<<grid, block, 0, s>>>(p); break;
    MUON_ROWS_CASE(1) MUON_ROWS_CASE(2) MUON_ROWS_CASE(3) MUON_ROWS_CASE(4)
#undef MUON_ROWS_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_rows(int w_dt, int g_dt, int max_cols, const RowsParams& p, cudaStream_t s) {
  if (p.total_rows <= 0) return cudaSuccess;
  if (max_cols > ROWS_MAX_COLS) return cudaErrorInvalidValue;
  const bool wb = w_dt == MUON_DTYPE_BF16, gb = g_dt == MUON_DTYPE_BF16;
  if (wb && gb) return launch_rows_t<bf16, bf16>(max_cols, p, s);
  if (wb && !gb) return launch_rows_t<bf16, float>(max_cols, p, s);
  if (!wb && gb) return launch_rows_t<float, bf16>(max_cols, p, s);
  return launch_rows_t<float, float>(max_cols, p, s);
}

cudaError_t launch_apply(int w_dt, int u_dt, const ApplyParams& p, cudaStream_t s) {
  if (p.total_blocks <= 0) return cudaSuccess;
  const dim3 grid(p.total_blocks), block(256);
  const bool wb = w_dt == MUON_DTYPE_BF16, ub = u_dt == MUON_DTYPE_BF16;
  if (wb && ub) apply_kernel<bf16, bf16><<<grid, block, 0, s>>>(p);
  else if (wb && !ub) apply_kernel<bf16, float><<<grid, block, 0, s>>>(p);
  else if (!wb && ub) apply_kernel<float, bf16><<<grid, block, 0, s>>>(p);
  else apply_kernel<float, float><<<grid, block, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fro_final(const FroFinalParams& p, cudaStream_t s) {
  if (p.nmat <= 0) return cudaSuccess;
  fro_final_kernel<<<p.nmat, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_osq_final(const OsqFinalParams& p, cudaStream_t s) {
  if (p.nmat <= 0) return cudaSuccess;
  osq_final_kernel<<<p.nmat, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_nz_rms(const NzRmsParams& p, cudaStream_t s) {
  if (p.nmat <= 0) return cudaSuccess;
  nz_rms_kernel<<<(p.nmat + 127) / 128, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_apply_ws(int w_dt, int o_dt, const ApplyWsParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const bool wb = w_dt == MUON_DTYPE_BF16, ob = o_dt == MUON_DTYPE_BF16;
  if (wb && ob) apply_ws_kernel<bf16, bf16><<<p.total_tiles, 256, 0, s>>>(p);
  else if (wb && !ob) apply_ws_kernel<bf16, float><<<p.total_tiles, 256, 0, s>>>(p);
  else if (!wb && ob) apply_ws_kernel<float, bf16><<<p.total_tiles, 256, 0, s>>>(p);
  else apply_ws_kernel<float, float><<<p.total_tiles, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_line_final(const LineFinalParams& p, cudaStream_t s) {
  if (p.total_lines <= 0) return cudaSuccess;
  line_final_kernel<<<(p.total_lines + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace muon
