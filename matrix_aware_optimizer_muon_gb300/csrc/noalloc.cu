// Frobenius norm of the momentum without a caller workspace.
//
// Some callers cannot allocate device memory at all: code running as a plugin
// inside a host framework that owns every device allocation, or code that must
// not call cudaMalloc in the middle of a step because the allocation would
// synchronise the device.  For them, muon_fro_norm_noalloc keeps its scratch (the
// per-tile partial sums of squares) in one fixed array compiled into the library
// instead of in a workspace.  Every GPU that loads the library holds this array
// (4 MiB) until the process exits.
//
// The kernels are the same ones muon_fro_norm launches; only the scratch address
// differs.
#include <cstring>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace muon {
namespace {

constexpr int kNoallocMaxPartials = 1 << 20;  // 64 x 128 tiles, i.e. up to ~8.6e9 elements per call

// One 64 x 128 tile of M writes one partial here.  Every slot a call reads was
// written earlier in the same call, so nothing needs clearing between calls.
static __device__ __align__(256) float g_noalloc_partials[kNoallocMaxPartials];

// Device address of the scratch array on the current device.  The host-side symbol
// itself is not a device address.  The address is looked up on every call rather
// than cached: a device reset or a new primary context reloads the module, and the
// array may then sit elsewhere.  The lookup does not allocate; on the first call on a
// device it may load the library's module there.
int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MUON_ERR_NO_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MUON_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return MUON_ERR_NO_DEVICE;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return MUON_ERR_CUDA;
  *out = static_cast<float*>(p);
  return MUON_OK;
}

int cdiv_i(long long a, long long b) { return (int)((a + b - 1) / b); }

}  // namespace
}  // namespace muon

using namespace muon;

extern "C" int muon_fro_norm_noalloc(const muon_matrix* mats, int n, float* fro_out, muon_stream_t stream) {
  if (n < 0) return MUON_ERR_INVALID;
  if (n == 0) return MUON_OK;
  if (!mats || !fro_out) return MUON_ERR_INVALID;
  long long total_tiles = 0;
  for (int i = 0; i < n; ++i) {
    const muon_matrix& a = mats[i];
    if (a.rows < 0 || a.cols < 0 || a.rows >= (1LL << 31) || a.cols >= (1LL << 31)) return MUON_ERR_INVALID;
    // the same dtype rules as every other entry point (muon_fro_norm returns the same status)
    if (a.w_dtype != MUON_DTYPE_F32 && a.w_dtype != MUON_DTYPE_BF16) return MUON_ERR_UNSUPPORTED;
    if (a.g_dtype != MUON_DTYPE_F32 && a.g_dtype != MUON_DTYPE_BF16) return MUON_ERR_UNSUPPORTED;
    if (a.w_dtype != mats[0].w_dtype || a.g_dtype != mats[0].g_dtype) return MUON_ERR_UNSUPPORTED;
    if (a.rows == 0 || a.cols == 0) continue;
    if (!a.M || reinterpret_cast<uintptr_t>(a.M) % 4 != 0) return MUON_ERR_INVALID;
    total_tiles += (long long)cdiv_i(a.rows, TILE_R) * cdiv_i(a.cols, TILE_C);
  }
  if (total_tiles > kNoallocMaxPartials) return MUON_ERR_UNSUPPORTED;  // beyond the fixed scratch
  float* part = nullptr;
  int rc = scratch_for_current_device(&part);
  if (rc != MUON_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // pass 1: per-tile sums of squares into the fixed scratch
  std::vector<int> first(n, 0), count(n, 0);
  static thread_local EwParams ew;
  int i = 0, offset = 0;
  while (i < n) {
    std::memset(&ew, 0, sizeof(ew));
    int j = 0, tiles = 0;
    for (; i < n && j < EW_MAX_MATS; ++i) {
      const muon_matrix& a = mats[i];
      if (a.rows == 0 || a.cols == 0) continue;
      EwMat& e = ew.mat[j++];
      e.M = a.M;
      e.rows = (int)a.rows;
      e.cols = (int)a.cols;
      e.tiles_c = cdiv_i(a.cols, TILE_C);
      e.tile_begin = tiles;
      e.tall = a.rows > a.cols;
      e.vec = (a.cols % 4 == 0) && reinterpret_cast<uintptr_t>(a.M) % 16 == 0;
      e.part = part + offset;
      first[i] = offset;
      count[i] = cdiv_i(a.rows, TILE_R) * e.tiles_c;
      offset += count[i];
      tiles += count[i];
    }
    ew.nmat = j;
    ew.total_tiles = tiles;
    if (j > 0 && launch_ew(EW_FRO, MUON_DTYPE_F32, MUON_DTYPE_F32, MUON_DTYPE_F32, ew, s) != cudaSuccess)
      return MUON_ERR_CUDA;
  }

  // pass 2: fixed-order sum per matrix, ||M_i||_F = sqrt(sum)
  static thread_local FroFinalParams fin;
  i = 0;
  while (i < n) {
    std::memset(&fin, 0, sizeof(fin));
    fin.part = part;
    fin.fro = fro_out;
    int j = 0;
    for (; i < n && j < FIN_MAX_MATS; ++i, ++j) {
      fin.begin[j] = first[i];
      fin.count[j] = count[i];
      fin.out_index[j] = i;
    }
    fin.nmat = j;
    if (launch_fro_final(fin, s) != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
