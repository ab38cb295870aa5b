// RowNorm step for tall matrices (A > B, so the RowNorm lines are the B columns;
// "Scaling Muon for Diffusion Transformers", distributed-implementation
// paragraph: tall matrices reduce per-column norm scalars) as two row-contiguous
// passes whose second pass finds the new momentum still in L2.
//
// A chunk is one 128-column block of one matrix, all A rows.  A tile is 256 rows
// of a chunk.  Pass 1 of a tile computes M <- mu*M + G, stores M and writes the
// tile's 128 column sums of squares; the CTA that completes a chunk's last
// pass-1 tile adds the chunk's tile sums in row-block order and publishes the
// 128 inverse column norms.  Pass 2 of a tile re-reads M and applies
//   W <- W - eta*(s*M/||column|| + lambda*W).
// Persistent CTAs take tiles from one atomic ticket counter in a fixed order in
// which pass 2 of chunk c comes a few chunks (about 48 MB of momentum) after its
// pass 1: pass-1 tiles never wait, and by the time a pass-2 tile is handed out
// its chunk is normally finished, while the chunk's new momentum is still in L2.  HBM
// traffic is then G 2 + M 4 + M 4 + W 2 + W 2 = 14 bytes per element, with
// every access a 512-byte (M) or 256-byte (G, W) row segment.
//
// Deadlock freedom: a pass-2 tile waits only for pass-1 tiles of its own chunk,
// which all precede it in ticket order and so are held by running CTAs that
// never wait.  The wait is still bounded: on expiry the kernel sets its abort
// word and the workspace status word, and every CTA stops taking tiles.
// Sums are in a fixed order (rows within a thread, warps, then row blocks), so
// results are bit-reproducible.
#include <climits>
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace muon {
namespace {

constexpr int TL_NT = 256;                     // threads per CTA: 8 warps
constexpr int TL_WARPS = TL_NT / 32;
constexpr int TL_RPT = TALL_RB / TL_WARPS;     // rows per thread per tile (32)
constexpr int TL_U = 4;                        // rows in flight per thread (measured best with 3 CTAs/SM)
static_assert(TALL_CB == 128, "one warp covers 128 columns (4 per lane)");
static_assert(TL_RPT % TL_U == 0, "tile rows split into whole batches");

struct TallTicket {
  int pass;   // 1 or 2
  int chunk;
  int rb;     // row block within the chunk
};

// Ticket t -> (pass, chunk, row block).  Order: pass 1 of chunks 0..L-1, then for
// c = L..NC-1 [pass 1 of c, pass 2 of c-L], then pass 2 of the last L chunks.
__device__ __forceinline__ TallTicket tall_decode(int t, int NC, int T, int L) {
  TallTicket k;
  if (t < L * T) {
    k.pass = 1; k.chunk = t / T; k.rb = t - k.chunk * T;
    return k;
  }
  t -= L * T;
  if (t < (NC - L) * 2 * T) {
    const int pair = t / (2 * T), w = t - pair * 2 * T;
    if (w < T) { k.pass = 1; k.chunk = pair + L; k.rb = w; }
    else { k.pass = 2; k.chunk = pair; k.rb = w - T; }
    return k;
  }
  t -= (NC - L) * 2 * T;
  k.pass = 2; k.chunk = NC - L + t / T; k.rb = t - (k.chunk - (NC - L)) * T;
  return k;
}

__device__ __forceinline__ float4 ld_cg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// L2 eviction priority: the new momentum written by pass 1 is kept (evict-last)
// until pass 2 reads it back, and that read marks it evict-first.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ float4 ld_cg4_hint(const float* a, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ void st4_hint(float* a, const float v[4], uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(a), "f"(v[0]), "f"(v[1]), "f"(v[2]),
               "f"(v[3]), "l"(pol)
               : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// bf16 W and G fit three CTAs per SM; fp32 inputs take more registers (two).
template <typename WT, typename GT>
__global__ void __launch_bounds__(TL_NT, sizeof(WT) + sizeof(GT) <= 4 ? 3 : 2) tall_kernel(const __grid_constant__ TallParams p) {
  __shared__ float red[TL_WARPS][TALL_CB];
  __shared__ int s_ticket;
  __shared__ int s_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = p.nchunks, T = p.nrb, A = p.rows, B = p.cols;
  const int L = p.lag;
  unsigned* const ticket = p.ctrl;
  unsigned* const done = p.ctrl + 1;
  unsigned* const ready = p.ctrl + 1 + NC;
  volatile unsigned* const abort_word = p.ctrl + 1 + 2 * NC;

  for (;;) {
    __syncthreads();  // the previous tile is finished with s_ticket, s_flag and red
    if (tid == 0) s_ticket = *abort_word ? INT_MAX : (int)atomicAdd(ticket, 1u);
    __syncthreads();
    const int t = s_ticket;
    if (t >= p.total) break;
    const TallTicket k = tall_decode(t, NC, T, L);
    const int mi = k.chunk / p.ncb, cb = k.chunk - mi * p.ncb;
    const TallMat& mt = p.mat[mi];
    const int c = cb * TALL_CB + lane * 4;       // this lane's first column
    const bool colok = c < B;                    // B % 4 == 0: a 4-column group is wholly in or out
    const int r0 = k.rb * TALL_RB;

    if (k.pass == 1) {
      const GT* __restrict__ G = reinterpret_cast<const GT*>(mt.G);
      float* __restrict__ M = mt.M;
      float cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int b = 0; b < TL_RPT / TL_U; ++b) {
        float4 mr[TL_U];
        typename Raw4<GT>::type gr[TL_U];
#pragma unroll
        for (int u = 0; u < TL_U; ++u) {
          const int r = r0 + warp + TL_WARPS * (b * TL_U + u);
          if (r < A && colok) {
            const size_t off = (size_t)r * B + c;
            mr[u] = ld_cg4(M + off);
            gr[u] = ldraw_stream(G + off);
          }
        }
#pragma unroll
        for (int u = 0; u < TL_U; ++u) {
          const int r = r0 + warp + TL_WARPS * (b * TL_U + u);
          if (r < A && colok) {
            float g[4], v[4];
            cvt4(gr[u], g);
            v[0] = p.mu * mr[u].x + g[0];
            v[1] = p.mu * mr[u].y + g[1];
            v[2] = p.mu * mr[u].z + g[2];
            v[3] = p.mu * mr[u].w + g[3];
            st4_hint(M + (size_t)r * B + c, v, l2_policy_evict_last());
#pragma unroll
            for (int j = 0; j < 4; ++j) cs[j] = fmaf(v[j], v[j], cs[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) red[warp][lane * 4 + j] = cs[j];
      __syncthreads();
      if (tid < TALL_CB) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < TL_WARPS; ++w) s += red[w][tid];
        const int col = cb * TALL_CB + tid;
        if (col < B) mt.part[(size_t)k.rb * B + col] = s;
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        s_flag = atomicAdd(done + k.chunk, 1u) == (unsigned)(T - 1);
      }
      __syncthreads();
      if (s_flag) {
        // last tile of the chunk: column norms from the tile sums, in row-block order
        __threadfence();
        int nonzero = 0;
        if (tid < TALL_CB) {
          const int col = cb * TALL_CB + tid;
          if (col < B) {
            float ss = 0.f;
#pragma unroll 4
            for (int q = 0; q < T; ++q) ss += __ldcg(mt.part + (size_t)q * B + col);
            if (p.check_finite) note_nonfinite(p.status, ss);
            const float iv = inv_norm_from_sumsq(ss);
            __stcg(mt.inv + col, iv);
            nonzero = iv > 0.f;
          }
        }
        const int count = __syncthreads_count(nonzero);
        if (tid == 0) {
          if (mt.nz && count) atomicAdd(mt.nz, count);   // telemetry: nonzero columns
          __threadfence();
          if (!p.stall) st_release(ready + k.chunk, 1u);
        }
      }
    } else {
      if (tid == 0) {
        int ok = 1;
        if (!ld_acquire(ready + k.chunk)) {
          const uint64_t t0 = ptx::globaltimer();
          while (!ld_acquire(ready + k.chunk)) {
            if (*abort_word) { ok = 0; break; }
            if (ptx::globaltimer() - t0 > p.timeout_ns) {
              *abort_word = 1u;
              if (p.status) atomicOr(p.status, DEV_TIMEOUT);
              ok = 0;
              break;
            }
            __nanosleep(256);
          }
        }
        s_flag = ok;
      }
      __syncthreads();
      if (!s_flag) continue;
      WT* __restrict__ W = reinterpret_cast<WT*>(mt.W);
      const float* __restrict__ M = mt.M;
      float iv[4] = {0.f, 0.f, 0.f, 0.f};
      if (colok) {
#pragma unroll
        for (int j = 0; j < 4; ++j) iv[j] = __ldcg(mt.inv + c + j);   // per-matrix inv need not be 16-byte aligned
      }
#pragma unroll 1
      for (int b = 0; b < TL_RPT / TL_U; ++b) {
        float4 mr[TL_U];
        typename Raw4<WT>::type wr[TL_U];
#pragma unroll
        for (int u = 0; u < TL_U; ++u) {
          const int r = r0 + warp + TL_WARPS * (b * TL_U + u);
          if (r < A && colok) {
            const size_t off = (size_t)r * B + c;
            mr[u] = ld_cg4_hint(M + off, l2_policy_evict_first());
            wr[u] = ldraw(W + off);
          }
        }
#pragma unroll
        for (int u = 0; u < TL_U; ++u) {
          const int r = r0 + warp + TL_WARPS * (b * TL_U + u);
          if (r < A && colok) {
            float w[4], m[4], o[4];
            cvt4(wr[u], w);
            cvt4(mr[u], m);
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = w[j] - p.eta * (p.scale * (m[j] * iv[j]) + p.lam * w[j]);
            st4(W + (size_t)r * B + c, o);
          }
        }
      }
    }
  }
}

// Resident CTAs per SM of one instantiation on the current device (queried once per
// device, process-wide).
template <typename WT, typename GT>
cudaError_t tall_resident(int* per_sm) {
  auto kern = tall_kernel<WT, GT>;
  static std::mutex mu;
  static std::map<int, int> resident;   // device -> CTAs per SM
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  auto it = resident.find(dev);
  if (it == resident.end()) {
    int n = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, TL_NT, 0)) != cudaSuccess) return e;
    it = resident.emplace(dev, n).first;
  }
  *per_sm = it->second;
  return cudaSuccess;
}

template <typename WT, typename GT>
cudaError_t launch_tall_t(const TallParams& p, int num_sms, cudaStream_t s) {
  auto kern = tall_kernel<WT, GT>;
  int per_sm = 0;
  cudaError_t e = tall_resident<WT, GT>(&per_sm);
  if (e != cudaSuccess) return e;
  long long grid = (long long)num_sms * (per_sm > 0 ? per_sm : 1);
  if (grid > p.total) grid = p.total;
  kern<<<(unsigned)grid, TL_NT, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int tall_ctrl_words(int nchunks) { return 2 + 2 * nchunks; }

cudaError_t prepare_tall() {
  int n = 0;
  cudaError_t e;
  if ((e = tall_resident<bf16, bf16>(&n)) != cudaSuccess) return e;
  if ((e = tall_resident<bf16, float>(&n)) != cudaSuccess) return e;
  if ((e = tall_resident<float, bf16>(&n)) != cudaSuccess) return e;
  return tall_resident<float, float>(&n);
}

cudaError_t launch_tall(int w_dt, int g_dt, const TallParams& p, int num_sms, cudaStream_t s) {
  if (p.total <= 0) return cudaSuccess;
  const bool wb = w_dt == MUON_DTYPE_BF16, gb = g_dt == MUON_DTYPE_BF16;
  if (wb && gb) return launch_tall_t<bf16, bf16>(p, num_sms, s);
  if (wb && !gb) return launch_tall_t<bf16, float>(p, num_sms, s);
  if (!wb && gb) return launch_tall_t<float, bf16>(p, num_sms, s);
  return launch_tall_t<float, float>(p, num_sms, s);
}

}  // namespace muon
