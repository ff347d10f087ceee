// scape_static.cu -- scape_topk_mask_static(): the partitioned top-k mask
// without any device allocation.
//
// Who needs this: some callers cannot call cudaMalloc at the point where they
// want a mask.  Examples are code running inside a custom device allocator or
// memory-pool callback (allocating there would re-enter the allocator), plug-ins
// and runtimes that are handed only their input and output buffers and must not
// allocate, and latency-critical loops that cannot afford cudaMalloc's implicit
// device synchronisation.  Those callers cannot provide the workspace that
// scape_bind() needs, so this entry point keeps its scratch in one fixed-size
// array inside the library instead.
//
// The scratch is a file-scope __device__ array of kScratchBytes (under 1 MiB).
// Every GPU that loads the library holds it until the process exits.  All calls
// share it and it keeps the last call's contents, so each call clears or fully
// rewrites every part it reads; calls that overlap on the GPU (different
// streams, or different host threads on one device) race on it and must be
// ordered by the caller.
#include <cmath>
#include <mutex>

#include "scape_internal.cuh"

namespace scapek {
namespace {

constexpr int64_t kStaticMaxP = SCAPE_STATIC_MAX_P;
constexpr int kStaticMaxW = SCAPE_STATIC_MAX_WORKERS;

constexpr size_t kAlignS = 256;
constexpr size_t up(size_t x) { return (x + kAlignS - 1) / kAlignS * kAlignS; }

// Regions of the scratch array (bytes), each 256-byte aligned.
constexpr size_t kHistBytes = up((size_t)kStaticMaxW * kBins * 4);
constexpr size_t kSelBytes = up((size_t)kStaticMaxW * sizeof(ShardSel));
// W * ceil(ceil(P/W) / 4096) <= P/4096 + 2W chunk counters
constexpr size_t kEqBytes = up((size_t)(kStaticMaxP / kTieChunk + 2 * kStaticMaxW) * 4);
constexpr size_t kTileCntBytes = up((size_t)(kStaticMaxP / kTile + 1) * 4);
constexpr size_t kTileBaseBytes = up((size_t)(kStaticMaxP / kTile + 2) * 4);
constexpr size_t kStartBytes = up((size_t)(kStaticMaxW + 1) * 8);
constexpr size_t kKBytes = up((size_t)kStaticMaxW * 8);
constexpr size_t kScanBytes = up((size_t)(2 * (kStaticMaxP / kTile / 2048 + 1)) * 4);

constexpr size_t kOffHist = 0;
constexpr size_t kOffSel = kOffHist + kHistBytes;
constexpr size_t kOffEq = kOffSel + kSelBytes;
constexpr size_t kOffTileCnt = kOffEq + kEqBytes;
constexpr size_t kOffTileBase = kOffTileCnt + kTileCntBytes;
constexpr size_t kOffStart = kOffTileBase + kTileBaseBytes;
constexpr size_t kOffK = kOffStart + kStartBytes;
constexpr size_t kOffScan = kOffK + kKBytes;
constexpr size_t kScratchBytes = kOffScan + kScanBytes;
static_assert(kScratchBytes < (1u << 20), "static scratch must stay under 1 MiB");

__device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

// Shard table on the device: boundaries floor(s*P/W) and
// k_s = ceil(n_s * (1e6 - ppm) / 1e6).  One block, W + 1 <= 65 threads used.
__global__ void static_layout_kernel(int64_t P, int W, int64_t ppm) {
  int64_t* start = reinterpret_cast<int64_t*>(g_static_scratch + kOffStart);
  int64_t* ks = reinterpret_cast<int64_t*>(g_static_scratch + kOffK);
  const int s = threadIdx.x;
  if (s <= W) start[s] = ((int64_t)s * P) / W;
  if (s < W) {
    const int64_t n = ((int64_t)(s + 1) * P) / W - ((int64_t)s * P) / W;
    ks[s] = (n * (1000000 - ppm) + 999999) / 1000000;
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
unsigned char* g_static_addr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once
// per device (host code must not use the symbol's name as an address).  The
// address belongs to the device's primary context; a cudaDeviceReset() would
// invalidate it, which the header tells callers not to do between calls.
cudaError_t static_scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace scapek

using namespace scapek;

extern "C" int scape_topk_mask_static(const float* m, int64_t P, int W, double sparsity,
                                      uint32_t* bits, uint32_t* idx, void* stream) {
  if (!m || !bits || !idx) return SCAPE_EINVAL;
  if (P < 1 || P > kStaticMaxP) return SCAPE_EINVAL;
  if (W < 1 || W > kStaticMaxW) return SCAPE_EINVAL;
  if (!(sparsity >= 0.0 && sparsity < 1.0)) return SCAPE_EINVAL;
  const int64_t ppm = std::llround(sparsity * 1e6);
  if (ppm >= 1000000) return SCAPE_EINVAL;
  if ((reinterpret_cast<uintptr_t>(m) & 15u) != 0) return SCAPE_EINVAL;

  // host copy of the shard sizes: chunk-table stride and the all-kept case
  int64_t nmax = 0, ktot = 0;
  bool all_dense = true;
  for (int s = 0; s < W; ++s) {
    const int64_t n = ((int64_t)(s + 1) * P) / W - ((int64_t)s * P) / W;
    const int64_t k = (n * (1000000 - ppm) + 999999) / 1000000;
    nmax = n > nmax ? n : nmax;
    ktot += k;
    if (k != n) all_dense = false;
  }
  const int64_t nchunk = nmax > 0 ? (nmax + kTieChunk - 1) / kTieChunk : 1;
  const int64_t ntiles = (P + kTile - 1) / kTile;

  unsigned char* base = nullptr;
  cudaError_t e = static_scratch_address(&base);
  if (e != cudaSuccess) return SCAPE_ECUDA;
  uint32_t* hist = reinterpret_cast<uint32_t*>(base + kOffHist);
  ShardSel* sel = reinterpret_cast<ShardSel*>(base + kOffSel);
  uint32_t* eqcnt = reinterpret_cast<uint32_t*>(base + kOffEq);
  uint32_t* tile_cnt = reinterpret_cast<uint32_t*>(base + kOffTileCnt);
  uint32_t* tile_base = reinterpret_cast<uint32_t*>(base + kOffTileBase);
  const int64_t* start = reinterpret_cast<const int64_t*>(base + kOffStart);
  const int64_t* ks = reinterpret_cast<const int64_t*>(base + kOffK);
  uint32_t* scan_scratch = reinterpret_cast<uint32_t*>(base + kOffScan);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // the histogram rows must start at zero; everything else is rewritten
  e = cudaMemsetAsync(hist, 0, (size_t)W * kBins * 4, st);
  if (e != cudaSuccess) return SCAPE_ECUDA;
  static_layout_kernel<<<1, 128, 0, st>>>(P, W, ppm);
  if ((e = cudaGetLastError()) != cudaSuccess) return SCAPE_ECUDA;
  if (!all_dense && (e = launch_hist(0, m, P, whole_map(P, W), start, sel, hist, st)) != cudaSuccess)
    return SCAPE_ECUDA;
  if ((e = launch_select(0, W, start, ks, sel, hist, st)) != cudaSuccess) return SCAPE_ECUDA;
  if (!all_dense) {
    for (int pass = 1; pass <= 2; ++pass) {
      if ((e = launch_hist(pass, m, P, whole_map(P, W), start, sel, hist, st)) != cudaSuccess) return SCAPE_ECUDA;
      if ((e = launch_select(pass, W, start, ks, sel, hist, st)) != cudaSuccess) return SCAPE_ECUDA;
    }
    if ((e = launch_tie_count(m, W, start, sel, eqcnt, nchunk, st)) != cudaSuccess)
      return SCAPE_ECUDA;
    if ((e = launch_tie_select(m, W, start, sel, eqcnt, nchunk, st)) != cudaSuccess)
      return SCAPE_ECUDA;
  }
  if ((e = launch_mark(m, P, whole_map(P, W), start, sel, bits, tile_cnt, st)) != cudaSuccess) return SCAPE_ECUDA;
  if ((e = launch_scan(tile_cnt, ntiles, tile_base, scan_scratch, st)) != cudaSuccess)
    return SCAPE_ECUDA;
  if ((e = launch_index(bits, P, tile_base, idx, ktot, st)) != cudaSuccess) return SCAPE_ECUDA;
  return SCAPE_OK;
}
