// Newton-Schulz-5 GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One iteration of Eq. (2) of the "Muon is Scalable for LLM Training" notes
// (section 2.1), X <- a X + b (X X^T) X + c (X X^T)^2 X, is computed in the
// factored form
//     S = X X^T               (GEMM_GRAM,   n x n, symmetric: upper tiles only)
//     B = b S + c S S         (GEMM_POLY,   n x n, symmetric: upper tiles only)
//     X <- a X + B X          (GEMM_UPDATE, n x m)
// with bf16 operands, fp32 accumulation in tensor memory, and every output
// rounded to bf16.  The first iteration folds X0 = M/||M||_F into the epilogues
// (S scaled by 1/||M||^2, X by 1/||M||), so the momentum is never normalised in
// a separate pass.  In the last iteration the UPDATE epilogue either writes O or
// applies W <- W - eta*(0.2*sqrt(max(A, B))*O + lambda*W) (Eq. (4)/(7)) directly.
//
// Two kernel forms share the roles and the epilogue:
//   ns_tc_pair_kernel (default): 2-CTA clusters (tcgen05 cta_group::2) on 256 x 256
//               tiles, each CTA staging half of A and half of B (32 KB a K step);
//   ns_tc_kernel: one CTA per 128 x 256 tile (48 KB a K step).
// Both are persistent (one CTA per SM), 320 threads:
//   warp 0      TMA producer (one lane): mbarrier ring of A and B tiles, 128-byte
//               swizzle;
//   warp 1      TMEM allocator and MMA issuer (one lane; in the pair form only the
//               even CTA issues): tcgen05.mma kind::f16, K = 16, two 256-column
//               fp32 accumulators so the epilogue of tile i overlaps the MMAs of i+1;
//   warps 2..9  epilogue, two per TMEM lane quarter, each draining 128 of the
//               256 columns: tcgen05.ld of the accumulator rows, fused combine,
//               global stores (symmetric outputs are written with their mirror).
// Tiles of all same-shape matrices (and of several shape groups) form one flat
// list that CTAs (or clusters) walk with a stride.  Every mbarrier wait is bounded
// in time; on expiry the kernel records MUON_DEV_TIMEOUT in the status word, all
// roles stop, in-flight copies and MMAs are drained (again bounded) and TMEM is
// freed before exit.
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "ns_common.cuh"

namespace muon {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half of the columns
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int EPI_CHUNKS = BN / 32 / (NUM_EPI_WARPS / 4);  // 32-column chunks per epilogue warp
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;   // mbarriers, the TMEM address and the abort flag
constexpr int SMEM_LIMIT = 227 * 1024;
// Dynamic shared memory of a launch: the operand ring, the 1 KB alignment slack of the
// swizzled ring, the barriers.
constexpr int smem_bytes(int stage_bytes, int stages) { return stages * stage_bytes + 1024 + BAR_BYTES; }

struct Tile {
  int g, mat, tm, tn;
};

__device__ __forceinline__ Tile decode(const NsParams& p, int t) {
  Tile ti;
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= t) ++g;
  const NsGroup& G = p.g[g];
  int lt = t - G.tile_begin;
  ti.g = g;
  ti.mat = lt / G.tiles_per_mat;
  int r = lt - ti.mat * G.tiles_per_mat;
  if (p.kind == GEMM_UPDATE) {
    ti.tn = r / G.mtiles;
    ti.tm = r - ti.tn * G.mtiles;
  } else {
    // upper-triangle tiles of the n x n output: column block tn holds row
    // blocks 0 .. min(2*tn+1, mtiles-1)
    int tn = 0;
    while (true) {
      const int cnt = min(2 * tn + 2, G.mtiles);
      if (r < cnt) break;
      r -= cnt;
      ++tn;
    }
    ti.tn = tn;
    ti.tm = r;
  }
  return ti;
}

// Bounded wait on an mbarrier phase.  Returns false on timeout (recorded in the
// status word and the CTA's abort flag) or, when honor_abort, if another role
// already aborted.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             const NsParams& p, bool honor_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      if (p.status) atomicOr(p.status, DEV_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    reinterpret_cast<uint4*>(dst)[q] = u;
  }
}

// 256-bit global accesses (32-byte aligned): a row-per-lane chunk of 64 bytes in two
// instructions instead of four, so half the L1 requests for the same bytes.
__device__ __forceinline__ void ld_v8(const void* src, uint32_t* w) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(src));
}
__device__ __forceinline__ void st_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void ld_v8x2(const void* src, uint32_t* w) {
  ld_v8(src, w);
  ld_v8(reinterpret_cast<const uint8_t*>(src) + 32, w + 8);
}
__device__ __forceinline__ void store_bf16x32_v8(bf16* dst, const float (&v)[32]) {
  uint32_t w[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) w[h] = pack_bf16x2(v[2 * h], v[2 * h + 1]);
  st_v8(dst, w);
  st_v8(reinterpret_cast<uint8_t*>(dst) + 32, w + 8);
}
__device__ __forceinline__ void load_bf16x32(const bf16* src, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * q + 2 * h] = __uint_as_float(w[h] << 16);
      v[8 * q + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
    }
  }
}

// Global inputs of one epilogue chunk (32 consecutive columns of one row),
// loaded one chunk ahead so that the loads overlap the previous chunk's work.
// Only full, vector-aligned chunks are prefetched; ragged chunks at a matrix
// edge load element by element in epi_finish.
struct ChunkIn {
  uint32_t w[32];
  bool ok;
};

__device__ __forceinline__ void ld_u4x4(const void* src, uint32_t* w) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[q];
    w[4 * q] = u.x; w[4 * q + 1] = u.y; w[4 * q + 2] = u.z; w[4 * q + 3] = u.w;
  }
}
__device__ __forceinline__ void unpack_bf16x32(const uint32_t* w, float (&v)[32]) {
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    v[2 * h] = __uint_as_float(w[h] << 16);
    v[2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void epi_prefetch(const NsParams& p, const NsGroup& G, const Tile& ti, int r, int c0,
                                             ChunkIn& in) {
  in.ok = false;
  const int n = G.n, m = G.m;
  const int gm = G.mat_base + ti.mat;
  if (p.kind == GEMM_GRAM) return;
  if (p.kind == GEMM_POLY) {
    if (r >= n || c0 + 32 > n || r > c0 + 31) return;
    ld_v8x2(reinterpret_cast<const bf16*>(G.epi_in) + (size_t)ti.mat * G.stride_nn + (size_t)r * G.ld_n + c0, in.w);
    in.ok = true;
    return;
  }
  if (r >= n || c0 + 32 > m) return;
  if (p.first_iter) {
    const float* Mp = p.msrc[gm];
    if (p.flags[gm] & NS_TALL) {
#pragma unroll
      for (int j = 0; j < 32; ++j) in.w[j] = __float_as_uint(Mp[(size_t)(c0 + j) * n + r]);
    } else if (p.flags[gm] & NS_MVEC8) {
      const float* src = Mp + (size_t)r * m + c0;
#pragma unroll
      for (int q = 0; q < 4; ++q) ld_v8(src + 8 * q, in.w + 8 * q);
    } else if (p.flags[gm] & NS_MVEC) {
      const float4* src = reinterpret_cast<const float4*>(Mp + (size_t)r * m + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = src[q];
        in.w[4 * q] = __float_as_uint(f.x); in.w[4 * q + 1] = __float_as_uint(f.y);
        in.w[4 * q + 2] = __float_as_uint(f.z); in.w[4 * q + 3] = __float_as_uint(f.w);
      }
    } else {
      return;
    }
    in.ok = true;
    return;
  }
  const size_t off = (size_t)ti.mat * G.stride_nm + (size_t)r * G.ld_m + c0;
  if (!p.fold_a) ld_v8x2(reinterpret_cast<const bf16*>(G.epi_in) + off, in.w);
  if (G.lo_in) {
    ld_v8x2(reinterpret_cast<const bf16*>(G.lo_in) + off, in.w + 16);
  } else if (p.last_iter && p.dst_mode == 1 && p.dst_dtype == MUON_DTYPE_BF16) {
    if (p.flags[gm] & NS_WVEC8) {
      ld_v8x2(reinterpret_cast<const bf16*>(p.dst[gm]) + (size_t)r * m + c0, in.w + 16);
    } else if (p.flags[gm] & NS_WVEC) {
      ld_u4x4(reinterpret_cast<const bf16*>(p.dst[gm]) + (size_t)r * m + c0, in.w + 16);
    } else if (p.flags[gm] & NS_TALL) {
      // tall W (m x n): W[c][r]; consecutive lanes read consecutive r
      const unsigned short* Wt = reinterpret_cast<const unsigned short*>(p.dst[gm]) + r;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        in.w[16 + h] = (uint32_t)Wt[(size_t)(c0 + 2 * h) * n] | ((uint32_t)Wt[(size_t)(c0 + 2 * h + 1) * n] << 16);
    }
  }
  in.ok = true;
}

// Combine and store 32 consecutive columns [c0, c0+32) of row r of one tile.
template <bool kOsq>
__device__ __forceinline__ void epi_finish(const NsParams& p, const NsGroup& G, const Tile& ti, int r, int c0,
                                           float (&v)[32], const ChunkIn& in, float& osq) {
  const int n = G.n, m = G.m;
  const int gm = G.mat_base + ti.mat;
  if (p.kind == GEMM_UPDATE) {
    if (r >= n || c0 >= m) return;
    const float sc = p.first_iter ? p.inv_norm[gm] : 1.0f;
    const bool full = c0 + 32 <= m;
    float x[32];
    if (p.fold_a) {
      // a*X_hi is already in the accumulator ((B + aI) X_hi); the residual X_lo,
      // where it is carried, adds a*X_lo here
      if (G.lo_in && in.ok) {
        unpack_bf16x32(in.w + 16, x);
      } else if (G.lo_in) {
        const bf16* Lin = reinterpret_cast<const bf16*>(G.lo_in) + (size_t)ti.mat * G.stride_nm + (size_t)r * G.ld_m;
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = (c0 + j < m) ? __bfloat162float(Lin[c0 + j]) : 0.f;
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = 0.f;
      }
    } else if (in.ok && p.first_iter) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(in.w[j]);
    } else if (in.ok) {
      unpack_bf16x32(in.w, x);
      if (G.lo_in) {
        float l[32];
        unpack_bf16x32(in.w + 16, l);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] += l[j];
      }
    } else if (p.first_iter) {
      // a*X0 from the fp32 momentum itself (X0 = M on the short side), ragged edge
      const float* Mp = p.msrc[gm];
      const bool tall = p.flags[gm] & NS_TALL;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        x[j] = (c0 + j < m) ? (tall ? Mp[(size_t)(c0 + j) * n + r] : Mp[(size_t)r * m + c0 + j]) : 0.f;
    } else {
      const size_t off = (size_t)ti.mat * G.stride_nm + (size_t)r * G.ld_m;
      const bf16* Xin = reinterpret_cast<const bf16*>(G.epi_in) + off;
      const bf16* Lin = G.lo_in ? reinterpret_cast<const bf16*>(G.lo_in) + off : nullptr;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        x[j] = (c0 + j < m) ? __bfloat162float(Xin[c0 + j]) + (Lin ? __bfloat162float(Lin[c0 + j]) : 0.f) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = sc * (p.a * x[j] + v[j]);
    if (kOsq && p.last_iter) {   // sum of squares of the output O (telemetry, Eq. (6))
#pragma unroll
      for (int j = 0; j < 32; ++j) osq = (c0 + j < m) ? fmaf(v[j], v[j], osq) : osq;
    }
    if (p.last_iter && p.dst_mode == 2 && (p.flags[gm] & NS_TALL)) {
      // O of a tall matrix kept for Eq. (6) in W's orientation (m x n, leading
      // dimension n, in this matrix's slot of the output buffers): consecutive lanes
      // write consecutive elements, and the apply pass needs no transpose
      const size_t base = (size_t)ti.mat * G.stride_nm + r;
      bf16* Ot = reinterpret_cast<bf16*>(G.out) + base;
      bf16* Lt = G.lo_out ? reinterpret_cast<bf16*>(G.lo_out) + base : nullptr;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < m) {
          const bf16 h = __float2bfloat16_rn(v[j]);
          Ot[(size_t)(c0 + j) * n] = h;
          if (Lt) Lt[(size_t)(c0 + j) * n] = __float2bfloat16_rn(v[j] - __bfloat162float(h));
        }
    } else if (!p.last_iter || p.dst_mode == 2) {
      const size_t off = (size_t)ti.mat * G.stride_nm + (size_t)r * G.ld_m + c0;
      bf16* Xout = reinterpret_cast<bf16*>(G.out) + off;
      bf16* Lout = G.lo_out ? reinterpret_cast<bf16*>(G.lo_out) + off : nullptr;
      float lo[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) lo[j] = v[j] - __bfloat162float(__float2bfloat16_rn(v[j]));
      if (full) {
        store_bf16x32_v8(Xout, v);
        if (Lout) store_bf16x32_v8(Lout, lo);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < m) {
            Xout[j] = __float2bfloat16_rn(v[j]);
            if (Lout) Lout[j] = __float2bfloat16_rn(lo[j]);
          }
      }
    } else {
      const float s_apply = p.rms_match * sqrtf((float)m);
      if (in.ok && p.dst_mode == 1 && p.dst_dtype == MUON_DTYPE_BF16 && (p.flags[gm] & NS_WVEC)) {
        // wide bf16 W: W[r][c0..c0+31] as 32- or 16-byte vectors
        float w[32];
        unpack_bf16x32(in.w + 16, w);
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = w[j] - p.eta * (s_apply * v[j] + p.lam * w[j]);
        bf16* Wr = reinterpret_cast<bf16*>(p.dst[gm]) + (size_t)r * m + c0;
        if (p.flags[gm] & NS_WVEC8) store_bf16x32_v8(Wr, w);
        else store_bf16x32(Wr, w);
      } else if (p.dst_mode == 0 && p.dst_dtype == MUON_DTYPE_BF16 && full && (p.flags[gm] & NS_WVEC)) {
        // bf16 O output, wide: row r of O, 32 consecutive columns as 32- or 16-byte vectors
        bf16* Or = reinterpret_cast<bf16*>(p.dst[gm]) + (size_t)r * m + c0;
        if (p.flags[gm] & NS_WVEC8) store_bf16x32_v8(Or, v);
        else store_bf16x32(Or, v);
      } else if (in.ok && p.dst_mode == 1 && p.dst_dtype == MUON_DTYPE_BF16 && (p.flags[gm] & NS_TALL)) {
        // tall bf16 W: element (r, c) of the short-side result is W[c][r]
        float w[32];
        unpack_bf16x32(in.w + 16, w);
        bf16* Wt = reinterpret_cast<bf16*>(p.dst[gm]) + r;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          Wt[(size_t)(c0 + j) * n] = __float2bfloat16_rn(w[j] - p.eta * (s_apply * v[j] + p.lam * w[j]));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < m) ns_last_store(p, gm, n, m, r, c0 + j, v[j], s_apply);
      }
    }
    return;
  }

  // symmetric n x n outputs: element (r, c) with r <= c is written at (r, c) and (c, r)
  if (r >= n || c0 >= n) return;
  if (r > c0 + 31) return;  // whole chunk below the diagonal
  if (p.kind == GEMM_GRAM) {
    const float sc = p.first_iter ? p.inv_norm[gm] * p.inv_norm[gm] : 1.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= sc;
  } else {
    float s[32];
    if (in.ok) {
      unpack_bf16x32(in.w, s);
    } else {
      const bf16* S = reinterpret_cast<const bf16*>(G.epi_in) + (size_t)ti.mat * G.stride_nn + (size_t)r * G.ld_n;
#pragma unroll
      for (int j = 0; j < 32; ++j) s[j] = (c0 + j < n) ? __bfloat162float(S[c0 + j]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = p.b * s[j] + p.c * v[j];
    if (p.fold_a) {   // B + a*I
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += (c0 + j == r) ? p.a : 0.f;
    }
  }
  bf16* out = reinterpret_cast<bf16*>(G.out) + (size_t)ti.mat * G.stride_nn;
  if (r <= c0 && c0 + 32 <= n) {
    store_bf16x32_v8(out + (size_t)r * G.ld_n + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) out[(size_t)(c0 + j) * G.ld_n + r] = __float2bfloat16_rn(v[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int c = c0 + j;
      if (c < n && r <= c) {
        const bf16 h = __float2bfloat16_rn(v[j]);
        out[(size_t)r * G.ld_n + c] = h;
        out[(size_t)c * G.ld_n + r] = h;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// CTA-pair form (tcgen05 cta_group::2): a 2-CTA cluster computes a 256 x 256 output
// tile.  The even CTA issues every MMA (M = 256, N = 256, K = 16); each CTA stages
// its own 128 rows of A and 128 columns (N) of B per K step, 32 KB a stage instead
// of 48, so four stages hold as many K steps in flight as the one-CTA form's four in
// two thirds of the shared memory, and each CTA's tensor memory receives its 128 rows of the tile, drained by its own
// epilogue warps exactly as in the one-CTA form.
//   full[s]   (even CTA): the producers of both CTAs land their halves on it; the
//             even producer posts the expected bytes of both;
//   empty[s]  (both CTAs): the MMA commit arrives on both, multicast;
//   tfull[a]  (both CTAs): the tile's last commit, multicast;
//   tempty[a] (even CTA): the 16 epilogue warps of both CTAs arrive on it.
// ---------------------------------------------------------------------------
constexpr int P_A_BYTES = BM * BK * 2;            // this CTA's 128 rows of A
constexpr int P_B_BYTES = (BN / 2) * BK * 2;      // this CTA's 128 columns of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;


// Pair tiles: G.mtiles counts 256-row blocks.  ti.tm is this CTA's 128-row block.
__device__ __forceinline__ Tile decode_pair(const NsParams& p, int t, int rank) {
  Tile ti;
  int g = 0;
  while (g + 1 < p.ngroups && p.g[g + 1].tile_begin <= t) ++g;
  const NsGroup& G = p.g[g];
  const int lt = t - G.tile_begin;
  ti.g = g;
  ti.mat = lt / G.tiles_per_mat;
  int r = lt - ti.mat * G.tiles_per_mat;
  int tp;
  if (p.kind == GEMM_UPDATE) {
    ti.tn = r / G.mtiles;
    tp = r - ti.tn * G.mtiles;
  } else {
    // upper-triangle 256 x 256 tiles: column block tn holds row blocks 0 .. tn
    int tn = 0;
    while (true) {
      const int cnt = min(tn + 1, G.mtiles);
      if (r < cnt) break;
      r -= cnt;
      ++tn;
    }
    ti.tn = tn;
    tp = r;
  }
  ti.tm = 2 * tp + rank;
  return ti;
}

// Epilogue warps of either kernel form: drain each tile's accumulator, combine it with
// the chunk inputs, store.  kPairMode: tiles are 256 x 256 pair tiles walked by
// cluster, tile rows are this CTA's half, and the accumulator-empty barrier lives in
// the even CTA.
template <bool kOsq, bool kPairMode>
__device__ __forceinline__ void epilogue_loop(const NsParams& p, int t0, int tstride, int rank, int warp, int lane,
                                              uint32_t tmem_base, uint64_t* tfull, uint64_t* tempty,
                                              volatile int* abort_flag) {
  const int quarter = warp & 3;            // TMEM lanes this warp may access
  const int half = (warp - 2) >> 2;        // which half of the 256 columns it drains
  const int row_in_tile = quarter * 32 + lane;
  const int ew = warp - 2;
  int it = 0;
  for (int t = t0; t < p.total_tiles; t += tstride, ++it) {
    const Tile ti = kPairMode ? decode_pair(p, t, rank) : decode(p, t);
    const NsGroup& G = p.g[ti.g];
    const int acc = it & 1;
    const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
    const int r = ti.tm * BM + row_in_tile;
    const int cbase = ti.tn * BN + half * (EPI_CHUNKS * 32);
    ChunkIn in_a, in_b;
    float osq = 0.f;
    epi_prefetch(p, G, ti, r, cbase, in_a);   // does not depend on this tile's accumulator
    int ok = 1;
    if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, p, true) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    ptx::tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + half * EPI_CHUNKS * 32);
#pragma unroll
    for (int k = 0; k < EPI_CHUNKS; ++k) {
      const int c0 = cbase + k * 32;
      ChunkIn& cur = (k & 1) ? in_b : in_a;
      ChunkIn& nxt = (k & 1) ? in_a : in_b;
      float v[32];
      ptx::tmem_ld_32x32b_x32(tbase + k * 32, v);
      if (k + 1 < EPI_CHUNKS) epi_prefetch(p, G, ti, r, c0 + 32, nxt);
      epi_finish<kOsq>(p, G, ti, r, c0, v, cur, osq);
    }
    if (kOsq && p.last_iter) {   // one fixed slot per (tile, CTA, epilogue warp)
      osq = warp_sum(osq);
      if (lane == 0) {
        const size_t slot_i = kPairMode ? ((size_t)t * 2 + rank) * NUM_EPI_WARPS + ew : (size_t)t * NUM_EPI_WARPS + ew;
        p.osq_part[slot_i] = osq;
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (!kPairMode || rank == 0) ptx::mbar_arrive(&tempty[acc]);
      else ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_addr(&tempty[acc]), 0));
    }
  }
}

// kOsq: the last UPDATE also writes per-warp partial sums of O^2 (only launches
// that need them pay for them).  kStages: depth of the TMA/MMA ring.
template <bool kOsq, int kStages>
__global__ void __launch_bounds__(NUM_THREADS, 1) ns_tc_kernel(const __grid_constant__ NsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * STAGE_BYTES);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mdone = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], NUM_EPI_WARPS);
    }
    ptx::mbar_init(mdone, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  const int kind = p.kind;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !(p.debug_flags & MUON_DEBUG_STALL_PRODUCER)) {
      for (int g = 0; g < p.ngroups; ++g) {
        ptx::prefetch_tmap(&p.g[g].mapA);
        ptx::prefetch_tmap(&p.g[g].mapB);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0, pend_phase = 0;  // bit s: stage s has an issued load
      bool stop = false;
      for (int t = blockIdx.x; t < p.total_tiles && !stop; t += gridDim.x) {
        const Tile ti = decode(p, t);
        const NsGroup& G = p.g[ti.g];
        const int K = (kind == GEMM_GRAM) ? G.m : G.n;
        const int nkb = (K + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p, true)) { stop = true; break; }
          ptx::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          const uint32_t sa = ptx::smem_addr(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          ptx::tma_load_3d(sa, &G.mapA, &full[stage], k0, ti.tm * BM, ti.mat);
          if (kind == GEMM_UPDATE) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              ptx::tma_load_3d(sb + j * (64 * BK * 2), &G.mapB, &full[stage], ti.tn * BN + 64 * j, k0, ti.mat);
          } else {
            ptx::tma_load_3d(sb, &G.mapB, &full[stage], k0, ti.tn * BN, ti.mat);
          }
          pending |= 1u << stage;
          pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // drain: every issued copy must land before the CTA may exit
      for (int s = 0; s < kStages; ++s)
        if (pending & (1u << s)) wait_bounded(&full[s], (pend_phase >> s) & 1u, abort_flag, p, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, false, kind == GEMM_UPDATE);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < p.total_tiles && !stop; t += gridDim.x, ++it) {
        const Tile ti = decode(p, t);
        const NsGroup& G = p.g[ti.g];
        const int K = (kind == GEMM_GRAM) ? G.m : G.n;
        const int nkb = (K + BK - 1) / BK;
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p, true)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, abort_flag, p, true)) { stop = true; break; }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; K step = 32 B.
            const uint64_t adesc = ptx::smem_desc_sw128(sa + k * 32, 16, 1024);
            // B: K-major like A (GRAM/POLY), or MN-major (UPDATE): 64-column
            // atoms 8 KB apart (LBO), 8-row K groups 1024 B apart (SBO), K step = 16 rows.
            const uint64_t bdesc = (kind == GEMM_UPDATE) ? ptx::smem_desc_sw128(sb + k * 2048, 64 * BK * 2, 1024)
                                                         : ptx::smem_desc_sw128(sb + k * 32, 16, 1024);
            ptx::mma_bf16(d, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (stop) break;
        ptx::mma_commit(&tfull[acc]);
      }
      // drain: all issued MMAs complete before TMEM is released
      ptx::mma_commit(mdone);
      wait_bounded(mdone, 0, abort_flag, p, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    epilogue_loop<kOsq, false>(p, blockIdx.x, gridDim.x, 0, warp, lane, tmem_base, tfull, tempty, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
}

template <bool kOsq, int kStages>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_tc_pair_kernel(const __grid_constant__ NsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * P_STAGE_BYTES);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mdone = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)ptx::cluster_ctarank();
  const bool even = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 2 * NUM_EPI_WARPS);
    }
    ptx::mbar_init(mdone, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();   // both CTAs' barriers initialised and tensor memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  const int kind = p.kind;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0 && !(p.debug_flags & MUON_DEBUG_STALL_PRODUCER)) {
      for (int g = 0; g < p.ngroups; ++g) {
        ptx::prefetch_tmap(&p.g[g].mapA);
        ptx::prefetch_tmap(&p.g[g].mapB);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0, pend_phase = 0;
      bool stop = false;
      for (int t = pair; t < p.total_tiles && !stop; t += npairs) {
        const Tile ti = decode_pair(p, t, rank);
        const NsGroup& G = p.g[ti.g];
        const int K = (kind == GEMM_GRAM) ? G.m : G.n;
        const int nkb = (K + BK - 1) / BK;
        const int n0 = ti.tn * BN + rank * (BN / 2);   // this CTA's half of the N columns
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p, true)) { stop = true; break; }
          const uint32_t fb = ptx::mapa_shared(ptx::smem_addr(&full[stage]), 0);
          if (even) ptx::mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
          const uint32_t sa = ptx::smem_addr(smem + stage * P_STAGE_BYTES);
          const uint32_t sb = sa + P_A_BYTES;
          const int k0 = kb * BK;
          ptx::tma_load_3d_pair(sa, &G.mapA, fb, k0, ti.tm * BM, ti.mat);
          if (kind == GEMM_UPDATE) {
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              ptx::tma_load_3d_pair(sb + j * (64 * BK * 2), &G.mapB, fb, n0 + 64 * j, k0, ti.mat);
          } else {
            ptx::tma_load_3d_pair(sb, &G.mapB, fb, k0, n0, ti.mat);
          }
          pending |= 1u << stage;
          pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // drain: the even CTA's full barriers count both CTAs' copies; the odd CTA's
      // copies have landed once the even CTA has seen them (it waits at the final
      // cluster barrier for that)
      if (even)
        for (int s = 0; s < kStages; ++s)
          if (pending & (1u << s)) wait_bounded(&full[s], (pend_phase >> s) & 1u, abort_flag, p, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (even && lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, BN, false, kind == GEMM_UPDATE);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool stop = false;
      for (int t = pair; t < p.total_tiles && !stop; t += npairs, ++it) {
        const Tile ti = decode_pair(p, t, 0);
        const NsGroup& G = p.g[ti.g];
        const int K = (kind == GEMM_GRAM) ? G.m : G.n;
        const int nkb = (K + BK - 1) / BK;
        const int acc = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p, true)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&full[stage], phase, abort_flag, p, true)) { stop = true; break; }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_addr(smem + stage * P_STAGE_BYTES);
          const uint32_t sb = sa + P_A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc = ptx::smem_desc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bdesc = (kind == GEMM_UPDATE) ? ptx::smem_desc_sw128(sb + k * 2048, 64 * BK * 2, 1024)
                                                         : ptx::smem_desc_sw128(sb + k * 32, 16, 1024);
            ptx::mma_bf16_pair(d, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          ptx::mma_commit_pair_mc(&empty[stage], 3);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (stop) break;
        ptx::mma_commit_pair_mc(&tfull[acc], 3);
      }
      // drain: all issued MMAs complete before either CTA releases its tensor memory
      ptx::mma_commit_pair_mc(mdone, 1);
      wait_bounded(mdone, 0, abort_flag, p, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    epilogue_loop<kOsq, true>(p, pair, npairs, rank, warp, lane, tmem_base, tfull, tempty, abort_flag);
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();   // no CTA leaves while its pair may still read its shared memory
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace tc

// Kernel attributes (dynamic shared memory beyond 48 KB) apply per device for the
// whole process: set once per device, under a lock, with the number of CTA pairs
// that fit on the device at once.
namespace {
std::mutex g_tc_mu;
std::map<int, int> g_tc_pairs;   // device -> co-resident 2-CTA clusters
// Ring depth of the 2-CTA form (32 KB a stage), for launches whose epilogue reads no
// global input (the Gram products, the UPDATE of iteration 3) and for the others.
// Four stages hold as many K steps in flight as the one-CTA form's four, in 128 KB
// instead of 192, and leave L1 room for the row-per-lane epilogue loads.  Measured
// (step ms, 15B / 1.3B; MMA-EPI stages): 4-4 205.6 / 11.35, 6-4 208.1 / 11.25,
// 6-5 215.1 / 11.18, 6-3 222.9 / 11.77; the one-CTA form 205.8 / 11.68.  Deeper
// rings lose at 15B, where the step runs under the power cap.
#ifndef MUON_PAIR_STAGES_MMA
#define MUON_PAIR_STAGES_MMA 4
#endif
#ifndef MUON_PAIR_STAGES_EPI
#define MUON_PAIR_STAGES_EPI 4
#endif
constexpr int kPairMma = MUON_PAIR_STAGES_MMA, kPairEpi = MUON_PAIR_STAGES_EPI;

template <class K>
cudaError_t allow_smem(K kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_LIMIT);
}

// Whether a launch's epilogue reads global inputs: POLY (S), the first UPDATE (fp32
// M), the UPDATEs that carry X's residual, and the last UPDATE when it applies to W.
bool reads_epilogue_inputs(const NsParams& p) {
  if (p.kind == GEMM_POLY) return true;
  if (p.kind != GEMM_UPDATE) return false;
  if (p.first_iter) return true;
  for (int g = 0; g < p.ngroups; ++g)
    if (p.g[g].lo_in) return true;
  return p.last_iter && p.dst_mode == 1;
}
}  // namespace

cudaError_t prepare_ns_tc() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  if (g_tc_pairs.count(dev)) return cudaSuccess;
  if ((e = allow_smem(tc::ns_tc_kernel<false, 4>)) != cudaSuccess) return e;
  if ((e = allow_smem(tc::ns_tc_kernel<false, 3>)) != cudaSuccess) return e;
  if ((e = allow_smem(tc::ns_tc_kernel<true, 4>)) != cudaSuccess) return e;
  if ((e = allow_smem(tc::ns_tc_pair_kernel<false, kPairMma>)) != cudaSuccess) return e;
  if ((e = allow_smem(tc::ns_tc_pair_kernel<false, kPairEpi>)) != cudaSuccess) return e;
  if ((e = allow_smem(tc::ns_tc_pair_kernel<true, kPairMma>)) != cudaSuccess) return e;
  if ((e = allow_smem(tc::ns_tc_pair_kernel<true, kPairEpi>)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(tc::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = tc::smem_bytes(tc::P_STAGE_BYTES, kPairMma > kPairEpi ? kPairMma : kPairEpi);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, tc::ns_tc_pair_kernel<false, kPairMma>, &cfg);
  if (e != cudaSuccess) return e;
  g_tc_pairs[dev] = clusters;
  return cudaSuccess;
}

int ns_tc_pairs() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  auto it = g_tc_pairs.find(dev);
  return it == g_tc_pairs.end() ? 0 : it->second;
}

cudaError_t launch_ns_tc(const NsParams& p, cudaStream_t s, int num_sms) {
  if (p.total_tiles <= 0) return cudaSuccess;
  cudaError_t e = prepare_ns_tc();
  if (e != cudaSuccess) return e;
  const bool osq = p.osq_part && p.last_iter;
  const bool inputs = reads_epilogue_inputs(p);
  if (p.pair) {
    const int pairs = ns_tc_pairs();
    if (pairs < 1) return cudaErrorInvalidConfiguration;
    const int grid = 2 * (p.total_tiles < pairs ? p.total_tiles : pairs);
    const int smem = tc::smem_bytes(tc::P_STAGE_BYTES, inputs ? kPairEpi : kPairMma);
    if (osq && inputs)
      tc::ns_tc_pair_kernel<true, kPairEpi><<<grid, tc::NUM_THREADS, smem, s>>>(p);
    else if (osq)
      tc::ns_tc_pair_kernel<true, kPairMma><<<grid, tc::NUM_THREADS, smem, s>>>(p);
    else if (inputs)
      tc::ns_tc_pair_kernel<false, kPairEpi><<<grid, tc::NUM_THREADS, smem, s>>>(p);
    else
      tc::ns_tc_pair_kernel<false, kPairMma><<<grid, tc::NUM_THREADS, smem, s>>>(p);
    return cudaGetLastError();
  }
  const int grid = p.total_tiles < num_sms ? p.total_tiles : num_sms;
  // One-CTA form, 48 KB a stage.  Three stages for POLY and the first UPDATE: the 48 KB
  // they free go to L1, where those launches' epilogue loads gain more than a shallower
  // ring costs them (per launch on the 1.3B set: POLY 655 -> 584 us, UPDATE 0 4371 ->
  // 4024 us; the long-K Gram product and the later UPDATEs lose 14-15% with three).
  const bool three = !osq && (p.kind == GEMM_POLY || (p.kind == GEMM_UPDATE && p.first_iter));
  const int smem = tc::smem_bytes(tc::STAGE_BYTES, three ? 3 : 4);
  if (osq)
    tc::ns_tc_kernel<true, 4><<<grid, tc::NUM_THREADS, smem, s>>>(p);
  else if (three)
    tc::ns_tc_kernel<false, 3><<<grid, tc::NUM_THREADS, smem, s>>>(p);
  else
    tc::ns_tc_kernel<false, 4><<<grid, tc::NUM_THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// host: tensor maps (driver entry point through the runtime, no -lcuda)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

bool encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace muon
