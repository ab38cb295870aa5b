// Internal declarations: launch-parameter tables, the workspace plan, and the
// launchers each kernel file provides to the C ABI layer (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/muon.h"

namespace muon {

// ---------------------------------------------------------------------------
// element-wise tile kernels (64 x 128 tiles of the A x B matrix)
// ---------------------------------------------------------------------------
constexpr int TILE_R = 64;
constexpr int TILE_C = 128;
constexpr int EW_THREADS = 256;
constexpr int EW_MAX_MATS = 96;  // matrices per launch (kernel-parameter table)

enum EwMode : int {
  EW_MOMENTUM = 1,   // M <- mu*M + G (stored)
  EW_FRO = 2,        // per-tile sum of squares of M -> part[tile]
  EW_XT = 4,         // X~ = M on the short-side orientation -> aux (ld_aux)
  EW_LINEPART = 8,   // per-tile line partial sums of squares -> line_part
  EW_APPLY_LINE = 16,// W <- W - eta*(s*M*inv_line + lambda*W)
  EW_WRITE_R = 32,   // R = M*inv_line -> aux (fp32, ld = B)
};

struct EwMat {
  void* W;
  const void* G;
  float* M;
  void* aux;               // X~ (EW_XT) or R (EW_WRITE_R)
  float* part;             // per-tile partials of this matrix (EW_FRO)
  float* line_part;        // [tiles along the long dim][lines] (EW_LINEPART)
  const float* line_inv;   // [lines] (EW_APPLY_LINE / EW_WRITE_R)
  int rows, cols;
  int ld_aux;
  int tiles_c;             // ceil(cols / TILE_C)
  int tile_begin;          // first tile of this matrix in the launch
  int tall;                // rows > cols
  float scale;             // apply scale s (already includes gamma)
  int vec;                 // 4-wide vector path allowed
};

struct EwParams {
  EwMat mat[EW_MAX_MATS];
  int nmat;
  int total_tiles;
  float mu, eta, lam;
};

// single-pass RowNorm step for wide / square matrices (one CTA per row)
constexpr int ROWS_MAX_MATS = 128;
constexpr int ROWS_MAX_COLS = 16384;

struct RowsMat {
  void* W;
  const void* G;
  float* M;
  int* nz;                 // optional: count of nonzero rows (update-RMS telemetry)
  int rows, cols;
  int row_begin;
  float scale;
  int vec;
};
struct RowsParams {
  RowsMat mat[ROWS_MAX_MATS];
  int nmat;
  int total_rows;
  float mu, eta, lam;
  unsigned int* status;    // finite check: DEV_NONFINITE when a row norm is NaN or Inf (null: off)
};

// single-pass RowNorm step for tall matrices: one thread-block cluster per
// column strip, the strip's new momentum held in shared memory
constexpr int COLS_MAX_MATS = 128;
constexpr int COLS_MAX_SMEM = 200 * 1024;     // opt-in dynamic shared memory per CTA
constexpr int COLS_SMEM_TARGET = 112 * 1024;  // two 512-thread CTAs per SM
struct ColsMat {
  void* W;
  const void* G;
  float* M;
  int* nz;                 // optional: count of nonzero columns (update-RMS telemetry)
  int rows, cols;
  int unit_begin;          // first column strip of this matrix in the launch
  float scale;
};
struct ColsParams {
  ColsMat mat[COLS_MAX_MATS];
  int nmat;
  int total_units;
  int slab_max;            // rows per CTA slab (ceil(max rows / cluster size))
  float mu, eta, lam;
  unsigned int* status;    // finite check: DEV_NONFINITE when a column norm is NaN or Inf (null: off)
};

// RowNorm step for tall matrices as two row-contiguous passes (tall.cu): chunks
// of TALL_CB columns x all rows, tiles of TALL_RB rows of a chunk.  Every matrix
// of one launch has the same shape.
constexpr int TALL_RB = 256;
constexpr int TALL_CB = 128;
constexpr int TALL_MAX_MATS = 128;
// New momentum (bytes) that waits in L2 between a chunk's first and second pass: the
// pass-2 lag in chunks is this over a chunk's A x TALL_CB x 4 bytes, in [2, 32].
// Measured on the 1.3B set (24 / 32 / 48 / 64 MB): a shorter lag makes pass-2 tiles
// wait, a longer one spills the momentum out of L2.
#ifndef MUON_TALL_LAG_BYTES
#define MUON_TALL_LAG_BYTES 48e6
#endif
constexpr double TALL_LAG_BYTES = MUON_TALL_LAG_BYTES;
struct TallMat {
  void* W;
  const void* G;
  float* M;
  float* part;             // [ceil(rows / TALL_RB)][cols] tile column sums of squares
  float* inv;              // [cols] inverse column norms
  int* nz;                 // optional: count of nonzero columns (update-RMS telemetry)
};
struct TallParams {
  TallMat mat[TALL_MAX_MATS];
  int nmat;
  int rows, cols;          // shape shared by every matrix of the launch
  int ncb;                 // column blocks per matrix
  int nrb;                 // row blocks (tiles) per chunk
  int nchunks;             // nmat * ncb
  int lag;                 // chunks between a chunk's pass 1 and pass 2 in ticket order (<= nchunks)
  int total;               // tickets: 2 * nchunks * nrb
  float mu, eta, lam, scale;
  unsigned* ctrl;          // [0] ticket, [1 + c] tiles done, [1 + NC + c] ready, [1 + 2 NC] abort
  unsigned int* status;    // workspace status word
  unsigned long long timeout_ns;
  int stall;               // test hook: publish no column norms, so that pass 2 times out
  int check_finite;        // finite check: DEV_NONFINITE in *status when a column norm is NaN or Inf
};

// Status-word bits: a kernel's bounded wait expired; a momentum norm was NaN or Inf
// (recorded only when the caller asked for the finite check).
constexpr uint32_t DEV_TIMEOUT = 1u;
constexpr uint32_t DEV_NONFINITE = 2u;

#ifdef __CUDACC__
// Finite check of a sum of squares of the momentum (status null: check off).
__device__ __forceinline__ void note_nonfinite(unsigned int* status, float ss) {
  if (status && !isfinite(ss)) atomicOr(status, DEV_NONFINITE);
}
#endif

// apply from a given direction U
constexpr int APPLY_MAX_MATS = 128;
constexpr int APPLY_CHUNK = 4096;  // elements per CTA
struct ApplyMat {
  void* W;
  const void* U;
  int64_t numel;
  int block_begin;
  float scale;
  int vec;
};
struct ApplyParams {
  ApplyMat mat[APPLY_MAX_MATS];
  int nmat;
  int total_blocks;
  float eta, lam;
};

// fixed-order finalisers
constexpr int FIN_MAX_MATS = 512;
struct FroFinalParams {
  const float* part;          // tile partials
  int begin[FIN_MAX_MATS];    // first partial of matrix i
  int count[FIN_MAX_MATS];    // number of partials of matrix i
  int out_index[FIN_MAX_MATS];// output slot of matrix i
  int nmat;
  float* fro_sq;              // optional outputs, indexed by out_index
  float* inv_norm;
  float* fro;
  unsigned int* status;       // finite check: DEV_NONFINITE when a ||M||^2 is NaN or Inf (null: off)
};
constexpr int LINE_MAX_MATS = 256;
struct LineFinalMat {
  const float* part;          // [parts][lines]
  float* inv;                 // [lines]
  int* nz;                    // optional: count of nonzero lines
  int parts, lines, line_begin;
};

// sum of squares of the Newton-Schulz output per matrix -> RMS and Eq. (6) scale
struct OsqFinalParams {
  const float* part;          // per-tile (x slot) partial sums of O^2
  long long begin[FIN_MAX_MATS];
  int count[FIN_MAX_MATS];
  int out_index[FIN_MAX_MATS];
  double numel[FIN_MAX_MATS]; // A*B
  int nmat;
  float* rms_out;             // optional, indexed by out_index
  float* scale_out;           // optional: rms_match / RMS (0 for a zero output)
  float rms_match;
};

// RMS of a RowNorm direction from its count of nonzero lines: sqrt(nz / (A*B))
struct NzRmsParams {
  const int* nz;              // per out_index
  double numel[FIN_MAX_MATS];
  int out_index[FIN_MAX_MATS];
  int nmat;
  float* rms_out;
};

// W <- W - eta*(scale_i*O + lambda*W) with O from the workspace (short-side layout)
constexpr int APPLYWS_MAX_MATS = 256;
constexpr int APPLYWS_TILE = 64;
struct ApplyWsMat {
  void* W;
  const void* O;              // bf16 (with optional bf16 residual) or fp32, n x ld
  const void* O_lo;           // bf16 residual or null
  int n, m, ld;
  int tall;
  int tiles_c;                // ceil(m / 64)
  int tile_begin;
  int scale_index;
  int vec;                    // W 16-byte aligned with rows a multiple of 8 elements: 16-byte accesses
  int ovec;                   // O's rows start 16-byte aligned (ld a multiple of 8): 16-byte loads
};
struct ApplyWsParams {
  ApplyWsMat mat[APPLYWS_MAX_MATS];
  int nmat;
  int total_tiles;
  const float* scale;         // per scale_index
  float eta, lam;
};
struct LineFinalParams {
  LineFinalMat mat[LINE_MAX_MATS];
  int nmat;
  int total_lines;
  unsigned int* status;       // finite check: DEV_NONFINITE when a line norm is NaN or Inf (null: off)
};

// ---------------------------------------------------------------------------
// Newton-Schulz GEMMs
// ---------------------------------------------------------------------------
enum GemmKind : int { GEMM_GRAM = 0, GEMM_POLY = 1, GEMM_UPDATE = 2 };
// NS_MVEC / NS_WVEC: M rows / the destination's rows take 16-byte vectors; the
// ...8 forms: 32-byte vectors (256-bit accesses, 32-byte aligned rows).
// NS_MTALL16 / NS_WTALL16: a tall matrix whose M / W rows start 16-byte aligned (n a
// multiple of 4 / 8 elements and an aligned base), so the epilogue can fetch 32 of
// its short-side elements with one bulk copy.
enum NsFlags : int { NS_TALL = 1, NS_MVEC = 2, NS_WVEC = 4, NS_MVEC8 = 8, NS_WVEC8 = 16, NS_MTALL16 = 32,
                     NS_WTALL16 = 64 };
// Iterations 1..NS_LO_ITERS add a*X_lo, the bf16 residual of X, to (B + aI) X_hi
// (X carried with ~16 significant bits where the small singular directions are
// still far below the element magnitudes).
constexpr int NS_LO_ITERS = 2;

constexpr int NS_MAX_GROUPS = 8;
constexpr int NS_MAX_MATS = 512;

// One shape group (same short side n and long side m) inside one GEMM launch.
struct NsGroup {
  CUtensorMap mapA;        // tensor-core path: K-major A operand
  CUtensorMap mapB;        // tensor-core path: B operand (K-major or MN-major)
  const void* opA;         // SIMT path: A operand base
  const void* opB;         // SIMT path: B operand base
  const void* epi_in;      // POLY: S (b*S term); UPDATE: X_in (a*X term)
  void* out;               // GRAM: S; POLY: B; UPDATE: X_out
  const void* lo_in;       // UPDATE (tensor-core path): bf16 residual of X_in, or null
  void* lo_out;            // UPDATE (tensor-core path): bf16 residual of X_out, or null
  long long stride_nn;     // elements between matrices of an n x n buffer
  long long stride_nm;     // elements between matrices of an n x m buffer
  int ld_n, ld_m;          // leading dims of n x n and n x m buffers
  int n, m;
  int count;
  int mtiles, ntiles;      // output tiles (rows, cols)
  int tiles_per_mat;
  int tile_begin;
  int mat_base;            // index of the group's first matrix in the launch tables
};

struct NsParams {
  NsGroup g[NS_MAX_GROUPS];
  int ngroups;
  int total_tiles;
  int kind;
  float a, b, c;
  int first_iter;          // fold 1/||M|| (UPDATE) or 1/||M||^2 (GRAM)
  int last_iter;           // UPDATE: write O or apply to W instead of X_out
  int fold_a;              // POLY writes B + a*I and UPDATE computes (B + a*I) X on the
                           // tensor cores, without reading X in the epilogue
  const float* inv_norm;   // per matrix (launch table order)
  // last-iteration outputs, per matrix (launch table order)
  void* dst[NS_MAX_MATS];  // W (apply) or O (output)
  const float* msrc[NS_MAX_MATS];  // fp32 momentum, the exact X0 for the first a*X term
  unsigned char flags[NS_MAX_MATS];  // NsFlags
  int dst_mode;            // 0: O in dst_dtype; 1: apply to W of dst_dtype;
                           // 2: O to X_out (+ residual) in the workspace
  float* osq_part;         // last UPDATE: partial sums of O^2, [tile][NUM_EPI_WARPS] (or [tile])
  int dst_dtype;           // MUON_DTYPE_*
  float eta, lam, rms_match;
  unsigned int* status;    // device status word
  unsigned long long timeout_ns;
  int debug_flags;
  int pair;                // tensor-core path: 2-CTA clusters on 256 x 256 tiles (mtiles counts
                           // 256-row blocks), else one CTA per 128 x 256 tile
};

// ---------------------------------------------------------------------------
// workspace plan (identical for every entry point given the same matrix list)
// ---------------------------------------------------------------------------
struct MatPlan {
  int A, B;
  int n, m;                // short / long side
  int tall;
  int group;
  int idx_in_group;
  int tiles;               // 64 x 128 tiles
  size_t fro_part;         // float offset of this matrix's tile partials
  size_t line_part;        // float offset of line partials
  size_t line_inv;         // float offset of inverse line norms
  int line_tiles;          // number of partial rows (tiles along the long dim)
  int lines;               // n
  size_t osq;              // float offset of this matrix's O^2 partials
};

struct GroupPlan {
  int n, m;
  int count;
  std::vector<int> mats;   // indices into the matrix list
  int ld_n, ld_m;
  size_t x0, x1, s, bm;    // byte offsets in the workspace
  size_t lo;               // bf16 residual of X (tensor-core mode only), updated in place
};

struct Plan {
  std::vector<MatPlan> mats;
  std::vector<GroupPlan> groups;
  int ns5_mode;
  size_t status;           // byte offset of the status word (always 0)
  size_t fro_part;         // byte offset of the fp32 tile-partial area
  size_t fro_sq;           // per matrix ||M||^2
  size_t inv_norm;         // per matrix 1/||M||
  size_t line_part;
  size_t line_inv;
  size_t osq_part;         // partial sums of O^2 (telemetry / Eq. (6))
  size_t scale;            // per matrix Eq. (6) scale
  size_t nz;               // per matrix nonzero-line counts (int)
  size_t tall_ctrl;        // control words of the tall-matrix RowNorm kernel (unsigned)
  int tall_chunks;         // column blocks over all tall matrices
  size_t total;
};

// launchers (return a cudaError_t from the launch)
cudaError_t launch_ew(int mode, int w_dt, int g_dt, int x_dt, const EwParams& p, cudaStream_t s);
cudaError_t launch_rows(int w_dt, int g_dt, int max_cols, const RowsParams& p, cudaStream_t s);
cudaError_t launch_apply(int w_dt, int u_dt, const ApplyParams& p, cudaStream_t s);
cudaError_t launch_cols(int w_dt, int g_dt, int cw, const ColsParams& p, cudaStream_t s);
cudaError_t launch_tall(int w_dt, int g_dt, const TallParams& p, int num_sms, cudaStream_t s);
int tall_ctrl_words(int nchunks);
// one-time set-up of the current device (kernel attributes, occupancy), process-wide
cudaError_t prepare_ns_tc();
int ns_tc_pairs();          // co-resident 2-CTA clusters of the pair kernel on the current device
cudaError_t prepare_tall();
int cols_cluster_size();
int cols_strip_width(int max_rows, int stage_elem_bytes);
cudaError_t launch_fro_final(const FroFinalParams& p, cudaStream_t s);
cudaError_t launch_line_final(const LineFinalParams& p, cudaStream_t s);
cudaError_t launch_osq_final(const OsqFinalParams& p, cudaStream_t s);
cudaError_t launch_nz_rms(const NzRmsParams& p, cudaStream_t s);
cudaError_t launch_apply_ws(int w_dt, int o_dt, const ApplyWsParams& p, cudaStream_t s);
cudaError_t launch_ns_simt(const NsParams& p, cudaStream_t s);
cudaError_t launch_ns_tc(const NsParams& p, cudaStream_t s, int num_sms);

// tensor map encoding (driver entry point obtained through the runtime)
bool encode_tmap_bf16(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1);

}  // namespace muon

namespace muon {
// Kernel parameters are limited to 32764 bytes.
static_assert(sizeof(EwParams) < 32000, "EwParams too large");
static_assert(sizeof(RowsParams) < 32000, "RowsParams too large");
static_assert(sizeof(TallParams) < 32000, "TallParams too large");
static_assert(sizeof(ApplyParams) < 32000, "ApplyParams too large");
static_assert(sizeof(FroFinalParams) < 32000, "FroFinalParams too large");
static_assert(sizeof(LineFinalParams) < 32000, "LineFinalParams too large");
static_assert(sizeof(NsParams) < 32000, "NsParams too large");
static_assert(sizeof(ColsParams) < 32000, "ColsParams too large");
static_assert(sizeof(OsqFinalParams) < 32000, "OsqFinalParams too large");
static_assert(sizeof(NzRmsParams) < 32000, "NzRmsParams too large");
static_assert(sizeof(ApplyWsParams) < 32000, "ApplyWsParams too large");
}  // namespace muon
