// C ABI of the Muon / Periodic Row-wise Muon step: argument validation,
// workspace planning, launch tables and the order of kernels per entry point.
// All device work is enqueued on the caller's stream; nothing here allocates
// device memory or synchronises (except muon_check_status).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "internal.h"

using namespace muon;

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeader = 256;  // status word(s)
constexpr float kRmsMatch = 0.2f;
// Newton-Schulz quintic coefficients and iteration count ("Muon is Scalable for
// LLM Training" notes, section 2.1 after Eq. (2); section 2.2 for N = 5).
constexpr float kNsA = 3.4445f, kNsB = -4.7750f, kNsC = 2.0315f;
constexpr int kNsSteps = 5;

std::atomic<int> g_debug_flags{0};
std::atomic<int> g_timeout_ms{4000};
thread_local int t_launches = 0;
std::mutex g_prof_mu;
cudaEvent_t g_prof_ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};

void prof_record(int i, cudaStream_t s) {
  cudaEvent_t e;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    e = g_prof_ev[i];
  }
  if (e) cudaEventRecord(e, s);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t dsize(int dt) { return dt == MUON_DTYPE_BF16 ? 2 : 4; }

struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

int device_info(DevInfo* out) {
  static std::mutex mu;
  static std::map<int, DevInfo> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    DevInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MUON_ERR_NO_DEVICE;
    it = cache.emplace(dev, d).first;
  }
  if (it->second.major != 10 || it->second.minor != 3) return MUON_ERR_NO_DEVICE;
  *out = it->second;
  return MUON_OK;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
struct Check {
  int w_dt = MUON_DTYPE_BF16, g_dt = MUON_DTYPE_BF16;
};

int validate(const muon_matrix* mats, int n, bool need_m, bool need_w, bool need_g, Check* ck) {
  if (n < 0) return MUON_ERR_INVALID;
  if (n == 0) return MUON_OK;
  if (!mats) return MUON_ERR_INVALID;
  ck->w_dt = mats[0].w_dtype;
  ck->g_dt = mats[0].g_dtype;
  for (int i = 0; i < n; ++i) {
    const muon_matrix& a = mats[i];
    if (a.rows < 0 || a.cols < 0 || a.rows >= (1LL << 31) || a.cols >= (1LL << 31)) return MUON_ERR_INVALID;
    if (a.w_dtype != MUON_DTYPE_F32 && a.w_dtype != MUON_DTYPE_BF16) return MUON_ERR_UNSUPPORTED;
    if (a.g_dtype != MUON_DTYPE_F32 && a.g_dtype != MUON_DTYPE_BF16) return MUON_ERR_UNSUPPORTED;
    if (a.w_dtype != ck->w_dt || a.g_dtype != ck->g_dt) return MUON_ERR_UNSUPPORTED;
    if (a.rows == 0 || a.cols == 0) continue;
    if ((long long)cdiv(a.rows, TILE_R) * cdiv(a.cols, TILE_C) >= (1LL << 30)) return MUON_ERR_UNSUPPORTED;
    if (need_m && (!a.M || !aligned(a.M, 4))) return MUON_ERR_INVALID;
    if (need_w && (!a.W || !aligned(a.W, dsize(a.w_dtype)))) return MUON_ERR_INVALID;
    if (need_g && (!a.G || !aligned(a.G, dsize(a.g_dtype)))) return MUON_ERR_INVALID;
  }
  return MUON_OK;
}

bool nonempty(const muon_matrix& a) { return a.rows > 0 && a.cols > 0; }

// ---------------------------------------------------------------------------
// workspace plan
// ---------------------------------------------------------------------------
bool make_plan(const muon_matrix* mats, int n, int ns5_mode, Plan* P) {
  P->mats.assign(n, MatPlan{});
  P->groups.clear();
  P->ns5_mode = ns5_mode;
  const size_t esize = ns5_mode == MUON_NS5_F32 ? 4 : 2;
  size_t fro_floats = 0, line_floats = 0, inv_floats = 0, osq_floats = 0;
  P->tall_chunks = 0;
  std::map<std::pair<int, int>, std::vector<int>> open;  // (n, m) -> current group indices
  for (int i = 0; i < n; ++i) {
    MatPlan& mp = P->mats[i];
    mp.A = (int)mats[i].rows;
    mp.B = (int)mats[i].cols;
    mp.tall = mp.A > mp.B;
    mp.n = std::min(mp.A, mp.B);
    mp.m = std::max(mp.A, mp.B);
    mp.group = -1;
    if (!nonempty(mats[i])) continue;
    mp.tiles = cdiv(mp.A, TILE_R) * cdiv(mp.B, TILE_C);
    mp.fro_part = fro_floats;
    fro_floats += mp.tiles;
    mp.lines = mp.n;
    mp.line_tiles = mp.tall ? cdiv(mp.A, TILE_R) : cdiv(mp.B, TILE_C);
    mp.line_part = line_floats;
    line_floats += (size_t)mp.line_tiles * mp.lines;
    mp.line_inv = inv_floats;
    inv_floats += mp.lines;
    if (mp.tall) P->tall_chunks += cdiv(mp.B, TALL_CB);
    // O^2 partials of the last UPDATE: [256x256 pair tile][16 epilogue warps],
    // [128x256 tile][8 epilogue warps] or [64x64 tile]
    mp.osq = osq_floats;
    osq_floats += std::max({(size_t)cdiv(mp.n, 256) * cdiv(mp.m, 256) * 16, (size_t)cdiv(mp.n, 128) * cdiv(mp.m, 256) * 8,
                            (size_t)cdiv(mp.n, 64) * cdiv(mp.m, 64)});
    // shape groups of at most NS_MAX_MATS matrices, first-appearance order
    const auto key = std::make_pair(mp.n, mp.m);
    int gi = -1;
    auto it = open.find(key);
    if (it != open.end() && P->groups[it->second.back()].count < NS_MAX_MATS) gi = it->second.back();
    if (gi < 0) {
      GroupPlan g;
      g.n = mp.n;
      g.m = mp.m;
      g.count = 0;
      // rows padded to 16 elements (32 bytes): the GEMM epilogues move them with
      // 256-bit accesses
      g.ld_n = (int)align_up(mp.n, 16);
      g.ld_m = (int)align_up(mp.m, 16);
      P->groups.push_back(g);
      gi = (int)P->groups.size() - 1;
      open[key].push_back(gi);
    }
    mp.group = gi;
    mp.idx_in_group = P->groups[gi].count++;
    P->groups[gi].mats.push_back(i);
  }
  size_t off = 0;
  P->status = off;
  off += kHeader;
  P->fro_part = off;
  off = align_up(off + fro_floats * 4, kAlign);
  P->fro_sq = off;
  off = align_up(off + (size_t)std::max(n, 1) * 4, kAlign);
  P->inv_norm = off;
  off = align_up(off + (size_t)std::max(n, 1) * 4, kAlign);
  P->line_part = off;
  off = align_up(off + line_floats * 4, kAlign);
  P->line_inv = off;
  off = align_up(off + inv_floats * 4, kAlign);
  P->osq_part = off;
  off = align_up(off + osq_floats * 4, kAlign);
  P->scale = off;
  off = align_up(off + (size_t)std::max(n, 1) * 4, kAlign);
  P->nz = off;
  off = align_up(off + (size_t)std::max(n, 1) * 4, kAlign);
  P->tall_ctrl = off;
  off = align_up(off + (size_t)tall_ctrl_words(P->tall_chunks) * 4, kAlign);
  for (GroupPlan& g : P->groups) {
    const size_t xb = (size_t)g.count * g.n * g.ld_m * esize;
    const size_t sb = (size_t)g.count * g.n * g.ld_n * esize;
    g.x0 = off;
    off = align_up(off + xb, kAlign);
    g.x1 = off;
    off = align_up(off + xb, kAlign);
    g.s = off;
    off = align_up(off + sb, kAlign);
    g.bm = off;
    off = align_up(off + sb, kAlign);
    const size_t lb = ns5_mode == MUON_NS5_BF16 ? (size_t)g.count * g.n * g.ld_m * 2 : 0;
    g.lo = off;
    off = align_up(off + lb, kAlign);
  }
  P->total = off;
  return true;
}

int check_ws(const Plan& P, void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, kAlign) || ws_bytes < P.total) return MUON_ERR_WORKSPACE;
  return MUON_OK;
}

// A second stream per (host thread, device) for running independent kernels of one
// step side by side, with the events that fork it from and join it back to the
// caller's stream.  Created on first use; they are not device memory.
struct AuxStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

AuxStream* aux_stream() {
  static thread_local std::map<int, AuxStream> per_device;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  AuxStream& a = per_device[dev];
  if (!a.stream) {
    if (cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess) {
      a = AuxStream{};
      return nullptr;
    }
  }
  return &a;
}

int cuda_status(cudaError_t e) {
  if (e != cudaSuccess) return MUON_ERR_CUDA;
  ++t_launches;
  return MUON_OK;
}

// ---------------------------------------------------------------------------
// element-wise launches over a list of matrices, chunked by the table size
// ---------------------------------------------------------------------------
template <class Fill>
int run_ew(const muon_matrix* mats, const std::vector<int>& idx, int mode, int w_dt, int g_dt, int x_dt, float mu,
           float eta, float lam, Fill fill, cudaStream_t s) {
  static thread_local EwParams prm;
  size_t k = 0;
  while (k < idx.size()) {
    std::memset(&prm, 0, sizeof(prm));
    prm.mu = mu;
    prm.eta = eta;
    prm.lam = lam;
    int tiles = 0;
    int j = 0;
    for (; k < idx.size() && j < EW_MAX_MATS; ++k) {
      const int i = idx[k];
      const muon_matrix& a = mats[i];
      if (!nonempty(a)) continue;
      EwMat& e = prm.mat[j++];
      e.W = a.W;
      e.G = a.G;
      e.M = a.M;
      e.rows = (int)a.rows;
      e.cols = (int)a.cols;
      e.tiles_c = cdiv(a.cols, TILE_C);
      e.tile_begin = tiles;
      e.tall = a.rows > a.cols;
      bool vec = (a.cols % 4 == 0) && aligned(a.M, 16);
      if (mode & EW_MOMENTUM) vec = vec && aligned(a.G, 4 * dsize(g_dt));
      if (mode & EW_APPLY_LINE) vec = vec && aligned(a.W, 4 * dsize(w_dt));
      e.vec = vec;
      fill(e, i);
      if ((mode & EW_WRITE_R) && !aligned(e.aux, 16)) e.vec = 0;
      tiles += cdiv(a.rows, TILE_R) * e.tiles_c;
    }
    prm.nmat = j;
    prm.total_tiles = tiles;
    if (j > 0) {
      const int rc = cuda_status(launch_ew(mode, w_dt, g_dt, x_dt, prm, s));
      if (rc != MUON_OK) return rc;
    }
  }
  return MUON_OK;
}

// ||M_i||^2 (and derived values) from the tile partials, fixed order.
int run_fro_final(const Plan& P, uint8_t* ws, const std::vector<int>& idx, const std::vector<int>& out_idx,
                  float* fro_sq, float* inv_norm, float* fro, cudaStream_t s, unsigned int* status = nullptr) {
  static thread_local FroFinalParams prm;
  size_t k = 0;
  while (k < idx.size()) {
    std::memset(&prm, 0, sizeof(prm));
    prm.part = reinterpret_cast<const float*>(ws + P.fro_part);
    prm.fro_sq = fro_sq;
    prm.inv_norm = inv_norm;
    prm.fro = fro;
    prm.status = status;
    int j = 0;
    for (; k < idx.size() && j < FIN_MAX_MATS; ++k, ++j) {
      const MatPlan& mp = P.mats[idx[k]];
      const bool ne = mp.A > 0 && mp.B > 0;
      prm.begin[j] = ne ? (int)mp.fro_part : 0;
      prm.count[j] = ne ? mp.tiles : 0;
      prm.out_index[j] = out_idx[k];
    }
    prm.nmat = j;
    const int rc = cuda_status(launch_fro_final(prm, s));
    if (rc != MUON_OK) return rc;
  }
  return MUON_OK;
}

int run_line_final(const Plan& P, uint8_t* ws, const std::vector<int>& idx, cudaStream_t s, int* nz = nullptr,
                   unsigned int* status = nullptr) {
  static thread_local LineFinalParams prm;
  size_t k = 0;
  while (k < idx.size()) {
    std::memset(&prm, 0, sizeof(prm));
    prm.status = status;
    int j = 0, lines = 0;
    for (; k < idx.size() && j < LINE_MAX_MATS; ++k) {
      const MatPlan& mp = P.mats[idx[k]];
      if (mp.A == 0 || mp.B == 0) continue;
      LineFinalMat& e = prm.mat[j++];
      e.part = reinterpret_cast<const float*>(ws + P.line_part) + mp.line_part;
      e.inv = reinterpret_cast<float*>(ws + P.line_inv) + mp.line_inv;
      e.nz = nz ? nz + idx[k] : nullptr;
      e.parts = mp.line_tiles;
      e.lines = mp.lines;
      e.line_begin = lines;
      lines += mp.lines;
    }
    prm.nmat = j;
    prm.total_lines = lines;
    if (j > 0) {
      const int rc = cuda_status(launch_line_final(prm, s));
      if (rc != MUON_OK) return rc;
    }
  }
  return MUON_OK;
}

// Global matrix order used by the NS5 tables: groups in order, matrices in group order.
std::vector<int> group_order(const Plan& P) {
  std::vector<int> o;
  for (const GroupPlan& g : P.groups) o.insert(o.end(), g.mats.begin(), g.mats.end());
  return o;
}

// ---------------------------------------------------------------------------
// Newton-Schulz driver: 5 iterations x (GRAM, POLY, UPDATE)
// ---------------------------------------------------------------------------
struct GroupMaps {
  CUtensorMap x128[2], x256[2], x64[2], s128, s256, b128;
};

// Partials of sum(O^2) written by the last UPDATE: where each matrix's lie.
struct OsqLayout {
  std::vector<long long> begin;  // list order
  std::vector<int> count;
};

int run_ns5(const Plan& P, const muon_matrix* mats, uint8_t* ws, int dst_mode, int dst_dtype,
            void* const* dst_ptrs /* list order */, float eta, float lam, int sms, cudaStream_t s,
            OsqLayout* osq = nullptr) {
  const bool tcmode = P.ns5_mode == MUON_NS5_BF16;
  const size_t esize = tcmode ? 2 : 4;
  const int ng = (int)P.groups.size();
  if (ng == 0) return MUON_OK;
  std::vector<GroupMaps> maps;
  if (tcmode) {
    maps.resize(ng);
    for (int gi = 0; gi < ng; ++gi) {
      const GroupPlan& g = P.groups[gi];
      const uint64_t sx1 = (uint64_t)g.ld_m * 2, sx2 = (uint64_t)g.n * g.ld_m * 2;
      const uint64_t ss1 = (uint64_t)g.ld_n * 2, ss2 = (uint64_t)g.n * g.ld_n * 2;
      bool ok = true;
      for (int b = 0; b < 2; ++b) {
        const void* xb = ws + (b == 0 ? g.x0 : g.x1);
        ok = ok && encode_tmap_bf16(&maps[gi].x128[b], xb, g.m, g.n, g.count, sx1, sx2, 64, 128);
        ok = ok && encode_tmap_bf16(&maps[gi].x256[b], xb, g.m, g.n, g.count, sx1, sx2, 64, 256);
        ok = ok && encode_tmap_bf16(&maps[gi].x64[b], xb, g.m, g.n, g.count, sx1, sx2, 64, 64);
      }
      ok = ok && encode_tmap_bf16(&maps[gi].s128, ws + g.s, g.n, g.n, g.count, ss1, ss2, 64, 128);
      ok = ok && encode_tmap_bf16(&maps[gi].s256, ws + g.s, g.n, g.n, g.count, ss1, ss2, 64, 256);
      ok = ok && encode_tmap_bf16(&maps[gi].b128, ws + g.bm, g.n, g.n, g.count, ss1, ss2, 64, 128);
      if (!ok) return MUON_ERR_CUDA;
    }
  }
  // launches cover consecutive groups: <= NS_MAX_GROUPS groups and <= NS_MAX_MATS matrices
  std::vector<std::pair<int, int>> chunks;  // [g0, g1)
  {
    int g0 = 0;
    while (g0 < ng) {
      int g1 = g0, mats_in = 0;
      while (g1 < ng && g1 - g0 < NS_MAX_GROUPS && mats_in + P.groups[g1].count <= NS_MAX_MATS) {
        mats_in += P.groups[g1].count;
        ++g1;
      }
      chunks.push_back({g0, g1});
      g0 = g1;
    }
  }
  // first global (group-order) index of each group
  std::vector<int> gbase(ng + 1, 0);
  for (int gi = 0; gi < ng; ++gi) gbase[gi + 1] = gbase[gi] + P.groups[gi].count;
  const float* inv_norm_all = reinterpret_cast<const float*>(ws + P.inv_norm);
  // Tensor-core launches run as 2-CTA clusters on 256 x 256 tiles (tcgen05 cta_group::2),
  // or with one CTA per 128 x 256 tile under the test hook MUON_DEBUG_NO_PAIR.
  const bool pair = tcmode && !(g_debug_flags.load() & MUON_DEBUG_NO_PAIR);
  // O^2 partials per tile: one per epilogue warp (of both CTAs of a pair), or one per CTA
  const int slots = tcmode ? (pair ? 16 : 8) : 1;
  long long osq_off = 0;
  if (osq) {
    osq->begin.assign(P.mats.size(), 0);
    osq->count.assign(P.mats.size(), 0);
  }
  static thread_local NsParams prm;
  for (int iter = 0; iter < kNsSteps; ++iter) {
    const int cur = iter & 1;
    for (int kind = GEMM_GRAM; kind <= GEMM_UPDATE; ++kind) {
      for (const auto& ch : chunks) {
        std::memset(&prm, 0, sizeof(prm));
        prm.kind = kind;
        prm.a = kNsA;
        prm.b = kNsB;
        prm.c = kNsC;
        prm.first_iter = iter == 0;
        prm.last_iter = (iter == kNsSteps - 1) && kind == GEMM_UPDATE;
        // Iterations after the first take a*X_hi inside the tensor-core product
        // ((B + aI) X_hi with B + aI rounded to bf16); the epilogue adds a*X_lo where
        // the residual is carried.  The first iteration takes a*X0 from the fp32 M.
        prm.fold_a = tcmode && iter >= 1 && kind != GEMM_GRAM;
        prm.inv_norm = inv_norm_all + gbase[ch.first];
        prm.dst_mode = dst_mode;
        prm.dst_dtype = dst_dtype;
        prm.eta = eta;
        prm.lam = lam;
        prm.rms_match = kRmsMatch;
        prm.status = reinterpret_cast<unsigned int*>(ws + P.status);
        prm.timeout_ns = (unsigned long long)g_timeout_ms.load() * 1000000ull;
        prm.debug_flags = g_debug_flags.load();
        prm.pair = pair ? 1 : 0;
        int tiles = 0, mbase = 0;
        prm.ngroups = ch.second - ch.first;
        for (int gi = ch.first; gi < ch.second; ++gi) {
          const GroupPlan& g = P.groups[gi];
          NsGroup& G = prm.g[gi - ch.first];
          uint8_t* xin = ws + (cur == 0 ? g.x0 : g.x1);
          uint8_t* xout = ws + (cur == 0 ? g.x1 : g.x0);
          G.n = g.n;
          G.m = g.m;
          G.count = g.count;
          G.ld_n = g.ld_n;
          G.ld_m = g.ld_m;
          G.stride_nn = (long long)g.n * g.ld_n;
          G.stride_nm = (long long)g.n * g.ld_m;
          G.mat_base = mbase;
          G.tile_begin = tiles;
          G.lo_in = nullptr;
          G.lo_out = nullptr;
          if (kind == GEMM_GRAM) {
            G.opA = xin;
            G.opB = xin;
            G.epi_in = nullptr;
            G.out = ws + g.s;
            if (tcmode) { G.mapA = maps[gi].x128[cur]; G.mapB = pair ? maps[gi].x128[cur] : maps[gi].x256[cur]; }
          } else if (kind == GEMM_POLY) {
            G.opA = ws + g.s;
            G.opB = ws + g.s;
            G.epi_in = ws + g.s;
            G.out = ws + g.bm;
            if (tcmode) { G.mapA = maps[gi].s128; G.mapB = pair ? maps[gi].s128 : maps[gi].s256; }
          } else {
            G.opA = ws + g.bm;
            G.opB = xin;
            G.epi_in = xin;
            G.out = xout;
            if (tcmode) {
              // iteration k writes the residual of X_{k+1} when k < NS_LO_ITERS and reads the
              // residual of X_k when 1 <= k <= NS_LO_ITERS, both in the one
              // residual buffer: an epilogue lane reads the element it then overwrites, and
              // no other tile reads it, so iteration 1 updates the buffer in place
              if (iter < NS_LO_ITERS && iter + 1 < kNsSteps) G.lo_out = ws + g.lo;
              if (iter >= 1 && iter <= NS_LO_ITERS) G.lo_in = ws + g.lo;
              // O kept in the workspace (Eq. (6)): its bf16 residual goes to the same buffer
              if (dst_mode == 2 && iter == kNsSteps - 1) G.lo_out = ws + g.lo;
            }
            if (tcmode) { G.mapA = maps[gi].b128; G.mapB = maps[gi].x64[cur]; }
          }
          if (tcmode && pair) {
            // 256 x 256 tiles; the symmetric products take column block tn's row blocks 0..tn
            G.mtiles = cdiv(g.n, 256);
            if (kind == GEMM_UPDATE) {
              G.ntiles = cdiv(g.m, 256);
              G.tiles_per_mat = G.mtiles * G.ntiles;
            } else {
              G.ntiles = cdiv(g.n, 256);
              int t = 0;
              for (int tn = 0; tn < G.ntiles; ++tn) t += std::min(tn + 1, G.mtiles);
              G.tiles_per_mat = t;
            }
          } else if (tcmode) {
            G.mtiles = cdiv(g.n, 128);
            if (kind == GEMM_UPDATE) {
              G.ntiles = cdiv(g.m, 256);
              G.tiles_per_mat = G.mtiles * G.ntiles;
            } else {
              G.ntiles = cdiv(g.n, 256);
              int t = 0;
              for (int tn = 0; tn < G.ntiles; ++tn) t += std::min(2 * tn + 2, G.mtiles);
              G.tiles_per_mat = t;
            }
          } else {
            G.mtiles = cdiv(g.n, 64);
            G.ntiles = cdiv(kind == GEMM_UPDATE ? g.m : g.n, 64);
            G.tiles_per_mat = G.mtiles * G.ntiles;
          }
          if ((long long)tiles + (long long)G.tiles_per_mat * g.count >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
          tiles += G.tiles_per_mat * g.count;
          for (int q = 0; q < g.count; ++q) {
            const int li = g.mats[q];
            prm.dst[mbase + q] = dst_ptrs ? dst_ptrs[li] : nullptr;
            const muon_matrix& a = mats[li];
            prm.msrc[mbase + q] = a.M;
            const void* dptr = dst_ptrs ? dst_ptrs[li] : nullptr;
            prm.flags[mbase + q] = (unsigned char)((a.rows > a.cols ? NS_TALL : 0) |
                                                   ((a.cols % 4 == 0 && aligned(a.M, 16)) ? NS_MVEC : 0) |
                                                   ((a.cols % 8 == 0 && aligned(a.M, 32)) ? NS_MVEC8 : 0) |
                                                   ((a.rows <= a.cols && a.cols % 8 == 0 && aligned(dptr, 16)) ? NS_WVEC : 0) |
                                                   ((a.rows <= a.cols && a.cols % 16 == 0 && aligned(dptr, 32)) ? NS_WVEC8 : 0) |
                                                   ((a.rows > a.cols && a.cols % 4 == 0 && aligned(a.M, 16)) ? NS_MTALL16 : 0) |
                                                   ((a.rows > a.cols && a.cols % 8 == 0 && aligned(dptr, 16)) ? NS_WTALL16 : 0));
          }
          mbase += g.count;
        }
        prm.total_tiles = tiles;
        if (osq && prm.last_iter) {
          prm.osq_part = reinterpret_cast<float*>(ws + P.osq_part) + osq_off;
          for (int gi = ch.first; gi < ch.second; ++gi) {
            const NsGroup& G = prm.g[gi - ch.first];
            for (int q = 0; q < G.count; ++q) {
              const int li = P.groups[gi].mats[q];
              osq->begin[li] = osq_off + (long long)(G.tile_begin + q * G.tiles_per_mat) * slots;
              osq->count[li] = G.tiles_per_mat * slots;
            }
          }
          osq_off += (long long)tiles * slots;
        }
        const cudaError_t e = tcmode ? launch_ns_tc(prm, s, sms) : launch_ns_simt(prm, s);
        if (cuda_status(e) != MUON_OK) return MUON_ERR_CUDA;
      }
    }
  }
  (void)esize;
  return MUON_OK;
}

// X~ (short-side copy of M) and ||M||^2 partials, then 1/||M|| per matrix.
int run_ns5_prep(const Plan& P, const muon_matrix* mats, int n, uint8_t* ws, bool momentum, float mu,
                 int w_dt, int g_dt, cudaStream_t s, unsigned int* status = nullptr) {
  std::vector<int> all;
  for (int i = 0; i < n; ++i)
    if (nonempty(mats[i])) all.push_back(i);
  const int x_dt = P.ns5_mode == MUON_NS5_F32 ? MUON_DTYPE_F32 : MUON_DTYPE_BF16;
  const size_t esize = x_dt == MUON_DTYPE_F32 ? 4 : 2;
  int mode = EW_FRO | EW_XT | (momentum ? EW_MOMENTUM : 0);
  int rc = run_ew(mats, all, mode, w_dt, g_dt, x_dt, mu, 0.f, 0.f,
                  [&](EwMat& e, int i) {
                    const MatPlan& mp = P.mats[i];
                    const GroupPlan& g = P.groups[mp.group];
                    e.aux = ws + g.x0 + (size_t)mp.idx_in_group * g.n * g.ld_m * esize;
                    e.ld_aux = g.ld_m;
                    e.part = reinterpret_cast<float*>(ws + P.fro_part) + mp.fro_part;
                  },
                  s);
  if (rc != MUON_OK) return rc;
  // inverse norms in group order
  const std::vector<int> order = group_order(P);
  std::vector<int> outi(order.size());
  for (size_t k = 0; k < order.size(); ++k) outi[k] = (int)k;
  return run_fro_final(P, ws, order, outi, reinterpret_cast<float*>(ws + P.fro_sq),
                       reinterpret_cast<float*>(ws + P.inv_norm), nullptr, s, status);
}

int common_checks(int n, DevInfo* di) {
  if (n == 0) return MUON_OK;
  return device_info(di);
}

}  // namespace

// ===========================================================================
// exported entry points
// ===========================================================================
extern "C" {

int muon_abi_version(void) { return MUON_ABI_VERSION; }

const char* muon_status_str(int st) {
  switch (st) {
    case MUON_OK: return "ok";
    case MUON_ERR_INVALID: return "invalid argument";
    case MUON_ERR_UNSUPPORTED: return "unsupported dtype or size";
    case MUON_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MUON_ERR_CUDA: return "CUDA call failed";
    case MUON_ERR_TIMEOUT: return "device-side wait timed out";
    case MUON_ERR_NO_DEVICE: return "no sm_103 device is current";
    case MUON_ERR_NONFINITE: return "a momentum norm was NaN or Inf";
    default: return "unknown status";
  }
}

int muon_init(void) {
  DevInfo di;
  int rc = device_info(&di);
  if (rc != MUON_OK) return rc;
  if (!aux_stream()) return MUON_ERR_CUDA;
  if (prepare_ns_tc() != cudaSuccess || prepare_tall() != cudaSuccess) return MUON_ERR_CUDA;
  return MUON_OK;
}

int muon_debug_set(int flags, int timeout_ms) {
  if (timeout_ms < 0) return MUON_ERR_INVALID;
  g_debug_flags.store(flags);
  g_timeout_ms.store(timeout_ms == 0 ? 4000 : timeout_ms);
  return MUON_OK;
}

size_t muon_workspace_size(const muon_matrix* mats, int n, int ns5_mode) {
  if (n == 0) return 0;
  Check ck;
  if (ns5_mode != MUON_NS5_BF16 && ns5_mode != MUON_NS5_F32) return (size_t)-1;
  if (validate(mats, n, false, false, false, &ck) != MUON_OK) return (size_t)-1;
  Plan P;
  make_plan(mats, n, ns5_mode, &P);
  return P.total;
}

int muon_workspace_init(void* ws, size_t ws_bytes, muon_stream_t stream) {
  if (!ws || !aligned(ws, kAlign) || ws_bytes < kHeader) return MUON_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, kHeader, static_cast<cudaStream_t>(stream)));
}

int muon_check_status(void* ws, size_t ws_bytes, muon_stream_t stream) {
  if (!ws || !aligned(ws, kAlign) || ws_bytes < kHeader) return MUON_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MUON_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return MUON_ERR_CUDA;
    return (word & DEV_TIMEOUT) ? MUON_ERR_TIMEOUT : MUON_ERR_NONFINITE;
  }
  return MUON_OK;
}

int muon_momentum(const muon_matrix* mats, int n, float mu, float* fro_sq_out, void* ws, size_t ws_bytes,
                  muon_stream_t stream) {
  Check ck;
  t_launches = 0;
  int rc = validate(mats, n, true, false, true, &ck);
  if (rc != MUON_OK || n == 0) return rc;
  DevInfo di;
  if ((rc = common_checks(n, &di)) != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<int> all;
  for (int i = 0; i < n; ++i) all.push_back(i);
  if (!fro_sq_out) {
    return run_ew(mats, all, EW_MOMENTUM, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, mu, 0.f, 0.f,
                  [](EwMat&, int) {}, s);
  }
  Plan P;
  make_plan(mats, n, MUON_NS5_BF16, &P);
  if ((rc = check_ws(P, ws, ws_bytes)) != MUON_OK) return rc;
  uint8_t* w = static_cast<uint8_t*>(ws);
  rc = run_ew(mats, all, EW_MOMENTUM | EW_FRO, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, mu, 0.f, 0.f,
              [&](EwMat& e, int i) { e.part = reinterpret_cast<float*>(w + P.fro_part) + P.mats[i].fro_part; }, s);
  if (rc != MUON_OK) return rc;
  return run_fro_final(P, w, all, all, fro_sq_out, nullptr, nullptr, s);
}

int muon_fro_norm(const muon_matrix* mats, int n, float* fro_out, void* ws, size_t ws_bytes,
                  muon_stream_t stream) {
  Check ck;
  t_launches = 0;
  int rc = validate(mats, n, true, false, false, &ck);
  if (rc != MUON_OK || n == 0) return rc;
  if (!fro_out) return MUON_ERR_INVALID;
  DevInfo di;
  if ((rc = common_checks(n, &di)) != MUON_OK) return rc;
  Plan P;
  make_plan(mats, n, MUON_NS5_BF16, &P);
  if ((rc = check_ws(P, ws, ws_bytes)) != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  std::vector<int> all;
  for (int i = 0; i < n; ++i) all.push_back(i);
  rc = run_ew(mats, all, EW_FRO, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, 0.f, 0.f, 0.f,
              [&](EwMat& e, int i) { e.part = reinterpret_cast<float*>(w + P.fro_part) + P.mats[i].fro_part; }, s);
  if (rc != MUON_OK) return rc;
  return run_fro_final(P, w, all, all, nullptr, nullptr, fro_out, s);
}

int muon_ns5_batched(const muon_matrix* mats, int n, int ns5_mode, void* const* O_out, int o_dtype, void* ws,
                     size_t ws_bytes, muon_stream_t stream) {
  Check ck;
  t_launches = 0;
  int rc = validate(mats, n, true, false, false, &ck);
  if (rc != MUON_OK || n == 0) return rc;
  if (ns5_mode != MUON_NS5_BF16 && ns5_mode != MUON_NS5_F32) return MUON_ERR_UNSUPPORTED;
  if (o_dtype != MUON_DTYPE_BF16 && o_dtype != MUON_DTYPE_F32) return MUON_ERR_UNSUPPORTED;
  if (!O_out) return MUON_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (nonempty(mats[i]) && (!O_out[i] || !aligned(O_out[i], dsize(o_dtype)))) return MUON_ERR_INVALID;
  DevInfo di;
  if ((rc = common_checks(n, &di)) != MUON_OK) return rc;
  Plan P;
  make_plan(mats, n, ns5_mode, &P);
  if ((rc = check_ws(P, ws, ws_bytes)) != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  rc = run_ns5_prep(P, mats, n, w, false, 0.f, ck.w_dt, ck.g_dt, s);
  if (rc != MUON_OK) return rc;
  return run_ns5(P, mats, w, 0, o_dtype, O_out, 0.f, 0.f, di.sms, s);
}

int muon_rownorm(const muon_matrix* mats, int n, float* const* R_out, void* ws, size_t ws_bytes,
                 muon_stream_t stream) {
  Check ck;
  t_launches = 0;
  int rc = validate(mats, n, true, false, false, &ck);
  if (rc != MUON_OK || n == 0) return rc;
  if (!R_out) return MUON_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (nonempty(mats[i]) && (!R_out[i] || !aligned(R_out[i], 4))) return MUON_ERR_INVALID;
  DevInfo di;
  if ((rc = common_checks(n, &di)) != MUON_OK) return rc;
  Plan P;
  make_plan(mats, n, MUON_NS5_BF16, &P);
  if ((rc = check_ws(P, ws, ws_bytes)) != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  std::vector<int> all;
  for (int i = 0; i < n; ++i) all.push_back(i);
  auto lines = [&](EwMat& e, int i) {
    const MatPlan& mp = P.mats[i];
    e.line_part = reinterpret_cast<float*>(w + P.line_part) + mp.line_part;
    e.line_inv = reinterpret_cast<float*>(w + P.line_inv) + mp.line_inv;
    e.aux = R_out[i];
  };
  rc = run_ew(mats, all, EW_LINEPART, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, 0.f, 0.f, 0.f, lines, s);
  if (rc != MUON_OK) return rc;
  rc = run_line_final(P, w, all, s);
  if (rc != MUON_OK) return rc;
  return run_ew(mats, all, EW_WRITE_R, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, 0.f, 0.f, 0.f, lines, s);
}

int muon_apply(const muon_matrix* mats, int n, const void* const* U, int u_dtype, float scale_mul, float eta,
               float lambda, muon_stream_t stream) {
  Check ck;
  t_launches = 0;
  int rc = validate(mats, n, false, true, false, &ck);
  if (rc != MUON_OK || n == 0) return rc;
  if (u_dtype != MUON_DTYPE_BF16 && u_dtype != MUON_DTYPE_F32) return MUON_ERR_UNSUPPORTED;
  if (!U) return MUON_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (nonempty(mats[i]) && (!U[i] || !aligned(U[i], dsize(u_dtype)))) return MUON_ERR_INVALID;
  DevInfo di;
  if ((rc = common_checks(n, &di)) != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static thread_local ApplyParams prm;
  int k = 0;
  while (k < n) {
    std::memset(&prm, 0, sizeof(prm));
    prm.eta = eta;
    prm.lam = lambda;
    int j = 0, blocks = 0;
    for (; k < n && j < APPLY_MAX_MATS; ++k) {
      const muon_matrix& a = mats[k];
      if (!nonempty(a)) continue;
      ApplyMat& e = prm.mat[j++];
      e.W = a.W;
      e.U = U[k];
      e.numel = a.rows * a.cols;
      e.block_begin = blocks;
      e.scale = scale_mul * std::sqrt((float)std::max(a.rows, a.cols));
      e.vec = aligned(a.W, 4 * dsize(ck.w_dt)) && aligned(U[k], 4 * dsize(u_dtype));
      const long long nb = (e.numel + APPLY_CHUNK - 1) / APPLY_CHUNK;
      if ((long long)blocks + nb >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
      blocks += (int)nb;
    }
    prm.nmat = j;
    prm.total_blocks = blocks;
    if (j > 0 && (rc = cuda_status(launch_apply(ck.w_dt, u_dtype, prm, s))) != MUON_OK) return rc;
  }
  return MUON_OK;
}

int muon_periodic_step(const muon_matrix* mats, int n, int64_t step, int K, float gamma, float mu, float eta,
                       float lambda, int ns5_mode, void* ws, size_t ws_bytes, muon_stream_t stream,
                       int* branch_out) {
  return muon_periodic_step_ex(mats, n, step, K, gamma, mu, eta, lambda, ns5_mode, nullptr, ws, ws_bytes, stream,
                               branch_out);
}

int muon_periodic_step_ex(const muon_matrix* mats, int n, int64_t step, int K, float gamma, float mu, float eta,
                          float lambda, int ns5_mode, const muon_step_options* opts, void* ws, size_t ws_bytes,
                          muon_stream_t stream, int* branch_out) {
  t_launches = 0;
  if (K < 1 || step < 0) return MUON_ERR_INVALID;
  if (ns5_mode != MUON_NS5_BF16 && ns5_mode != MUON_NS5_F32) return MUON_ERR_UNSUPPORTED;
  const int scale_mode = opts ? opts->scale_mode : MUON_SCALE_ADJUSTED_LR;
  float* update_rms = opts ? opts->update_rms : nullptr;
  const bool check_finite = opts && opts->check_finite;
  if (scale_mode != MUON_SCALE_ADJUSTED_LR && scale_mode != MUON_SCALE_UPDATE_NORM) return MUON_ERR_UNSUPPORTED;
  if (update_rms && !aligned(update_rms, 4)) return MUON_ERR_INVALID;
  Check ck;
  t_launches = 0;
  int rc = validate(mats, n, true, true, true, &ck);
  if (rc != MUON_OK) return rc;
  // Periodic schedule: full Newton-Schulz refresh when step % K == 0 (step from 0).
  const bool refresh = (step % K) == 0;
  if (branch_out) *branch_out = refresh ? MUON_BRANCH_NS5 : MUON_BRANCH_ROWNORM;
  if (n == 0) return MUON_OK;
  DevInfo di;
  if ((rc = common_checks(n, &di)) != MUON_OK) return rc;
  Plan P;
  make_plan(mats, n, ns5_mode, &P);
  if ((rc = check_ws(P, ws, ws_bytes)) != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  // finite check: the kernels that reduce the momentum's norms report NaN or Inf here
  unsigned int* fin_status = check_finite ? reinterpret_cast<unsigned int*>(w + P.status) : nullptr;

  if (refresh) {
    prof_record(0, s);
    rc = run_ns5_prep(P, mats, n, w, true, mu, ck.w_dt, ck.g_dt, s, fin_status);
    if (rc != MUON_OK) return rc;
    std::vector<void*> dst(n);
    for (int i = 0; i < n; ++i) dst[i] = mats[i].W;
    prof_record(1, s);
    OsqLayout osq;
    const bool norm = scale_mode == MUON_SCALE_UPDATE_NORM;
    const bool want_osq = norm || update_rms;
    // Eq. (4)/(7): the apply is fused into the last UPDATE.  Eq. (6): O stays in
    // the workspace until its RMS is known, then a separate pass applies it.
    rc = run_ns5(P, mats, w, norm ? 2 : 1, ck.w_dt, dst.data(), eta, lambda, di.sms, s, want_osq ? &osq : nullptr);
    if (rc != MUON_OK) return rc;
    if (want_osq) {
      float* scale = reinterpret_cast<float*>(w + P.scale);
      static thread_local OsqFinalParams fp;
      int i = 0;
      while (i < n) {
        std::memset(&fp, 0, sizeof(fp));
        fp.part = reinterpret_cast<const float*>(w + P.osq_part);
        fp.rms_out = update_rms;
        fp.scale_out = norm ? scale : nullptr;
        fp.rms_match = kRmsMatch;
        int j = 0;
        for (; i < n && j < FIN_MAX_MATS; ++i, ++j) {
          fp.begin[j] = osq.begin[i];
          fp.count[j] = osq.count[i];
          fp.out_index[j] = i;
          fp.numel[j] = (double)mats[i].rows * (double)mats[i].cols;
        }
        fp.nmat = j;
        if ((rc = cuda_status(launch_osq_final(fp, s))) != MUON_OK) return rc;
      }
      if (norm) {
        const bool tc = ns5_mode == MUON_NS5_BF16;
        const size_t esize = tc ? 2 : 4;
        static thread_local ApplyWsParams ap;
        int k = 0;
        while (k < n) {
          std::memset(&ap, 0, sizeof(ap));
          ap.scale = scale;
          ap.eta = eta;
          ap.lam = lambda;
          int j = 0, tiles = 0;
          for (; k < n && j < APPLYWS_MAX_MATS; ++k) {
            if (!nonempty(mats[k])) continue;
            const MatPlan& mp = P.mats[k];
            const GroupPlan& g = P.groups[mp.group];
            ApplyWsMat& e = ap.mat[j++];
            const size_t moff = (size_t)mp.idx_in_group * g.n * g.ld_m;
            e.W = mats[k].W;
            e.O = w + g.x1 + moff * esize;                       // output of the last UPDATE
            e.O_lo = tc ? (const void*)(w + g.lo + moff * 2) : nullptr;
            if (tc && mp.tall) {
              // the tensor-core path wrote a tall matrix's O in W's orientation
              // (m x n, leading dimension n): an elementwise pass over W
              e.n = g.m;
              e.m = g.n;
              e.ld = g.n;
              e.tall = 0;
            } else {
              e.n = g.n;
              e.m = g.m;
              e.ld = g.ld_m;
              e.tall = mp.tall;
            }
            e.tiles_c = cdiv(e.m, APPLYWS_TILE);
            e.tile_begin = tiles;
            e.scale_index = k;
            e.vec = aligned(mats[k].W, 16) && (e.tall ? e.n % 8 == 0 : e.m % 8 == 0);
            e.ovec = e.ld % 8 == 0;
            tiles += cdiv(e.n, APPLYWS_TILE) * e.tiles_c;
          }
          ap.nmat = j;
          ap.total_tiles = tiles;
          if (j > 0 && (rc = cuda_status(launch_apply_ws(ck.w_dt, tc ? MUON_DTYPE_BF16 : MUON_DTYPE_F32, ap, s))) !=
                           MUON_OK)
            return rc;
        }
      }
    }
    prof_record(2, s);
    return MUON_OK;
  }
  prof_record(3, s);
  // Update-RMS telemetry of a RowNorm step: count the nonzero lines.
  int* nz = update_rms ? reinterpret_cast<int*>(w + P.nz) : nullptr;
  if (nz && cudaMemsetAsync(nz, 0, sizeof(int) * (size_t)n, s) != cudaSuccess) return MUON_ERR_CUDA;

  // RowNorm branch: s = gamma * 0.2 * sqrt(max(A, B))
  std::vector<int> two_pass;
  std::map<int, std::vector<int>> rows_by_cols;
  for (int i = 0; i < n; ++i) {
    if (!nonempty(mats[i])) continue;
    if (mats[i].rows <= mats[i].cols && mats[i].cols <= ROWS_MAX_COLS) rows_by_cols[(int)mats[i].cols].push_back(i);
    else two_pass.push_back(i);
  }
  // Wide rows and tall columns are independent: when both are present the rows
  // kernels run on a second stream next to the tall-matrix kernels, so that
  // one kernel's CTAs stream while the other's wait on their line reductions.
  cudaStream_t rs = s;
  AuxStream* aux = nullptr;
  if (!rows_by_cols.empty() && !two_pass.empty() && !(g_debug_flags.load() & MUON_DEBUG_NO_OVERLAP)) {
    aux = aux_stream();
    if (aux) {
      if (cudaEventRecord(aux->fork, s) != cudaSuccess || cudaStreamWaitEvent(aux->stream, aux->fork, 0) != cudaSuccess)
        return MUON_ERR_CUDA;
      rs = aux->stream;
    }
  }
  static thread_local RowsParams rp;
  for (const auto& kv : rows_by_cols) {
    const std::vector<int>& v = kv.second;
    size_t k = 0;
    while (k < v.size()) {
      std::memset(&rp, 0, sizeof(rp));
      rp.mu = mu;
      rp.eta = eta;
      rp.lam = lambda;
      rp.status = fin_status;
      int j = 0, rows = 0;
      for (; k < v.size() && j < ROWS_MAX_MATS; ++k) {
        const muon_matrix& a = mats[v[k]];
        RowsMat& e = rp.mat[j++];
        e.W = a.W;
        e.G = a.G;
        e.M = a.M;
        e.nz = nz ? nz + v[k] : nullptr;
        e.rows = (int)a.rows;
        e.cols = (int)a.cols;
        e.row_begin = rows;
        e.scale = gamma * kRmsMatch * std::sqrt((float)a.cols);
        e.vec = (a.cols % 4 == 0) && aligned(a.M, 16) && aligned(a.G, 4 * dsize(ck.g_dt)) &&
                aligned(a.W, 4 * dsize(ck.w_dt));
        if ((long long)rows + a.rows >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
        rows += (int)a.rows;
      }
      rp.nmat = j;
      rp.total_rows = rows;
      if ((rc = cuda_status(launch_rows(ck.w_dt, ck.g_dt, kv.first, rp, rs))) != MUON_OK) return rc;
    }
  }
  const int dbg = g_debug_flags.load();
  if (!(dbg & MUON_DEBUG_NO_CLUSTER) && !(dbg & MUON_DEBUG_TALL_CLUSTER)) {
    // tall matrices: two row-contiguous passes, the second re-reading M from L2
    std::map<std::pair<int, int>, std::vector<int>> tall_by_shape;
    std::vector<int> rest;
    for (int i : two_pass) {
      const muon_matrix& a = mats[i];
      const bool ok = a.rows > a.cols && a.cols % 4 == 0 && aligned(a.M, 16) && aligned(a.G, 4 * dsize(ck.g_dt)) &&
                      aligned(a.W, 4 * dsize(ck.w_dt));
      if (ok) tall_by_shape[std::make_pair((int)a.rows, (int)a.cols)].push_back(i);
      else rest.push_back(i);
    }
    static thread_local TallParams tp;
    unsigned* ctrl = reinterpret_cast<unsigned*>(w + P.tall_ctrl);
    for (const auto& kv : tall_by_shape) {
      const std::vector<int>& v = kv.second;
      const int A = kv.first.first, Bc = kv.first.second;
      size_t k = 0;
      while (k < v.size()) {
        std::memset(&tp, 0, sizeof(tp));
        tp.rows = A;
        tp.cols = Bc;
        tp.ncb = cdiv(Bc, TALL_CB);
        tp.nrb = cdiv(A, TALL_RB);
        tp.mu = mu;
        tp.eta = eta;
        tp.lam = lambda;
        tp.scale = gamma * kRmsMatch * std::sqrt((float)A);
        int j = 0;
        for (; k < v.size() && j < TALL_MAX_MATS; ++k) {
          const muon_matrix& a = mats[v[k]];
          const MatPlan& mp = P.mats[v[k]];
          TallMat& e = tp.mat[j++];
          e.W = a.W;
          e.G = a.G;
          e.M = a.M;
          e.part = reinterpret_cast<float*>(w + P.line_part) + mp.line_part;
          e.inv = reinterpret_cast<float*>(w + P.line_inv) + mp.line_inv;
          e.nz = nz ? nz + v[k] : nullptr;
        }
        tp.nmat = j;
        tp.nchunks = j * tp.ncb;
        const int lag = (int)std::lround(TALL_LAG_BYTES / ((double)A * TALL_CB * 4.0));
        tp.lag = std::min(std::max(2, std::min(lag, 32)), tp.nchunks);
        if (2LL * tp.nchunks * tp.nrb >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
        tp.total = 2 * tp.nchunks * tp.nrb;
        tp.ctrl = ctrl;
        tp.status = reinterpret_cast<unsigned int*>(w + P.status);
        tp.timeout_ns = (unsigned long long)g_timeout_ms.load() * 1000000ull;
        tp.stall = (dbg & MUON_DEBUG_STALL_PRODUCER) ? 1 : 0;
        tp.check_finite = check_finite ? 1 : 0;
        if (cudaMemsetAsync(ctrl, 0, sizeof(unsigned) * (size_t)tall_ctrl_words(tp.nchunks), s) != cudaSuccess)
          return MUON_ERR_CUDA;
        if ((rc = cuda_status(launch_tall(ck.w_dt, ck.g_dt, tp, di.sms, s))) != MUON_OK) return rc;
      }
    }
    two_pass.swap(rest);
  } else if (!(dbg & MUON_DEBUG_NO_CLUSTER)) {
    // tall matrices: single pass, one thread-block cluster per column strip
    std::map<int, std::vector<int>> tall_by_rows;
    std::vector<int> rest;
    const int stage = (int)std::max(dsize(ck.w_dt), dsize(ck.g_dt));
    for (int i : two_pass) {
      const muon_matrix& a = mats[i];
      const bool ok = a.rows > a.cols && a.cols % 4 == 0 && aligned(a.M, 16) && aligned(a.G, 4 * dsize(ck.g_dt)) &&
                      aligned(a.W, 4 * dsize(ck.w_dt)) && cols_strip_width((int)a.rows, stage) > 0;
      if (ok) tall_by_rows[(int)a.rows].push_back(i);
      else rest.push_back(i);
    }
    static thread_local ColsParams cp;
    for (const auto& kv : tall_by_rows) {
      const std::vector<int>& v = kv.second;
      const int cw = cols_strip_width(kv.first, stage);
      size_t k = 0;
      while (k < v.size()) {
        const size_t k0 = k;
        std::memset(&cp, 0, sizeof(cp));
        cp.mu = mu;
        cp.eta = eta;
        cp.lam = lambda;
        cp.slab_max = (kv.first + cols_cluster_size() - 1) / cols_cluster_size();
        cp.status = fin_status;
        int j = 0, units = 0;
        for (; k < v.size() && j < COLS_MAX_MATS; ++k) {
          const muon_matrix& a = mats[v[k]];
          ColsMat& e = cp.mat[j++];
          e.W = a.W;
          e.G = a.G;
          e.M = a.M;
          e.nz = nz ? nz + v[k] : nullptr;
          e.rows = (int)a.rows;
          e.cols = (int)a.cols;
          e.unit_begin = units;
          e.scale = gamma * kRmsMatch * std::sqrt((float)a.rows);
          units += cdiv(a.cols, cw);
        }
        cp.nmat = j;
        cp.total_units = units;
        const cudaError_t e = launch_cols(ck.w_dt, ck.g_dt, cw, cp, s);
        if (e == cudaErrorInvalidClusterSize) {
          // the cluster shape does not fit this device: these go the two-pass way
          cudaGetLastError();
          rest.insert(rest.end(), v.begin() + (long)k0, v.begin() + (long)k);
          continue;
        }
        if ((rc = cuda_status(e)) != MUON_OK) return rc;
      }
    }
    two_pass.swap(rest);
  }
  if (!two_pass.empty()) {
    auto fill = [&](EwMat& e, int i) {
      const MatPlan& mp = P.mats[i];
      e.line_part = reinterpret_cast<float*>(w + P.line_part) + mp.line_part;
      e.line_inv = reinterpret_cast<float*>(w + P.line_inv) + mp.line_inv;
      e.scale = gamma * kRmsMatch * std::sqrt((float)mp.m);
    };
    rc = run_ew(mats, two_pass, EW_MOMENTUM | EW_LINEPART, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, mu, eta, lambda,
                fill, s);
    if (rc != MUON_OK) return rc;
    rc = run_line_final(P, w, two_pass, s, nz, fin_status);
    if (rc != MUON_OK) return rc;
    rc = run_ew(mats, two_pass, EW_APPLY_LINE, ck.w_dt, ck.g_dt, MUON_DTYPE_F32, mu, eta, lambda, fill, s);
    if (rc != MUON_OK) return rc;
  }
  if (aux) {
    if (cudaEventRecord(aux->join, aux->stream) != cudaSuccess || cudaStreamWaitEvent(s, aux->join, 0) != cudaSuccess)
      return MUON_ERR_CUDA;
  }
  if (nz) {
    static thread_local NzRmsParams zp;
    int i = 0;
    while (i < n) {
      std::memset(&zp, 0, sizeof(zp));
      zp.nz = nz;
      zp.rms_out = update_rms;
      int j = 0;
      for (; i < n && j < FIN_MAX_MATS; ++i, ++j) {
        zp.out_index[j] = i;
        zp.numel[j] = (double)mats[i].rows * (double)mats[i].cols;
      }
      zp.nmat = j;
      if ((rc = cuda_status(launch_nz_rms(zp, s))) != MUON_OK) return rc;
    }
  }
  prof_record(4, s);
  return MUON_OK;
}

int muon_profile_events(void* const* events, int n) {
  if (n < 0 || n > 5 || (n > 0 && !events)) return MUON_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < 5; ++i) g_prof_ev[i] = (i < n) ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  return MUON_OK;
}

int muon_launch_count(void) { return t_launches; }

}  // extern "C"
