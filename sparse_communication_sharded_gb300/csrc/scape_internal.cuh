// scape_internal.cuh -- types, constants and device helpers shared by the
// SCAPE library's translation units (kernels and the C ABI host code).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "scape.h"

namespace scapek {

// Compaction tile: 2048 parameters = 64 bitmap words, 256 threads x 8 elements.
// The per-tile rank table built by the mask refresh is indexed by this tile.
constexpr int kTile = 2048;
constexpr int kTileThreads = 256;
constexpr int kTileWords = kTile / 32;

// Radix select over 31-bit magnitude keys: digits of 11, 11 and 9 bits.
constexpr int kBins = 2048;
constexpr int kShift0 = 20;  // pass 0: key bits 30..20
constexpr int kShift1 = 9;   // pass 1: key bits 19..9
// pass 2: key bits 8..0 (512 bins)

// Segment of m read by one block of a histogram pass.
constexpr int kSeg = 4096;
// Chunk of a shard scanned by one block when resolving equal keys.
constexpr int kTieChunk = 4096;

struct WorkerPtrs {
  const void* g[SCAPE_MAX_WORKERS];
  float* e[SCAPE_MAX_WORKERS];
};

// Per-shard state of the radix select.
enum SelMode : uint32_t {
  kSelEmpty = 0,   // shard holds no parameter
  kSelDone = 1,    // threshold final (kstar, istar valid)
  kSelSearch = 2,  // radix passes still narrowing the threshold
  kSelTie = 3      // kstar final, istar to be found among equal keys
};

struct ShardSel {
  uint32_t mode;
  uint32_t prefix;    // key bits fixed by the passes so far
  uint32_t krem;      // selections still owed among keys matching prefix
  uint32_t kstar;     // threshold key: every key > kstar is selected
  uint32_t need;      // how many keys == kstar are selected (lowest indices)
  uint32_t count_eq;  // how many keys == kstar the shard holds
  int64_t istar;      // keys == kstar with index <= istar are selected
  uint64_t cprefix;   // composite-key bits fixed so far (candidate select)
  uint32_t guess;     // first-digit bucket of the previous refresh (0xFFFFFFFF: none)
  uint32_t flags;     // kSelNeedCollect, kSelRemark, kSelNeedHist
  uint32_t kstar_prev;  // the threshold the speculative bitmap was written with
  uint32_t guess_prev;  // first-digit bucket of the refresh before (0xFFFFFFFF: none)
  int64_t istar_prev;
};
constexpr uint32_t kNoGuess = 0xFFFFFFFFu;
constexpr uint32_t kSelNeedCollect = 1u;  // the threshold bucket moved: collect again
constexpr uint32_t kSelRemark = 2u;       // the speculative bitmap of this shard is unusable
constexpr uint32_t kSelNeedHist = 4u;     // warm refresh missed: count the shard fully

// AdamS constants of one step; all computed on the host in float.
struct AdamsConst {
  float beta1, beta2, one_minus_b1, one_minus_b2, bc1, bc2, lr, eps, wd;
};

// Profiling ids; must stay in sync with kKernelNames in scape_api.cu.
enum KernelId {
  kKDenseStep = 0,
  kKEfCompact,
  kKReduce,
  kKAdamsSparse,
  kKCandHist0,
  kKCandSelect,
  kKCandCollect,
  kKCandHist,
  kKMark,
  kKScan,
  kKIndex,
  kKShardCount,
  kKTileCount,
  kKOffmask,
  kKDenseAdams,
  kKAdamW,
  kKEfAdd,
  kKUnionMove,
  kKSpecMark,
  kKFixup,
  kKRemark,
  kKParamPatch,
  kKDenseUpdate,
  kKXcMove,
  kKProbeRmw,
  kNumKernels
};
static_assert(kNumKernels == SCAPE_NUM_KERNELS, "kernel table size");

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t magnitude_key(float x) {
  return __float_as_uint(x) & 0x7FFFFFFFu;
}

// The shards a handle covers: S consecutive optimizer shards a .. a + S - 1 of
// an even Wg-way split of Pg parameters ("SCAPE" Sec. II-A: the distributed
// optimizer partitions the states evenly), whose first parameter is global
// index `off`; local parameter i is global parameter off + i.  A whole-problem
// handle has Pg = P, off = 0, Wg = S, a = 0.
struct ShardMap {
  int64_t Pg;
  int64_t off;
  int Wg;
  int a;
  int S;
  // local shard holding local parameter i: the largest global s with
  // floor(s * Pg / Wg) <= off + i, minus a
  __device__ __forceinline__ int of(int64_t i) const {
    return (int)(((i + off + 1) * (int64_t)Wg - 1) / Pg) - a;
  }
};

inline ShardMap whole_map(int64_t P, int S) { return ShardMap{P, 0, S, 0, S}; }

// Exclusive prefix sum over a block of NT threads (NT a multiple of 32).
// `warp_tot` holds NT/32 words of shared memory; callers __syncthreads()
// before reusing it.  *total receives the block sum.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  uint32_t off = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    uint32_t t = warp_tot[i];
    off += (i < warp) ? t : 0u;
    tot += t;
  }
  *total = tot;
  return off + x - v;
}

// AdamS update of one coordinate ("SCAPE" Sec. II-C, Eq. 2 with bias
// corrections), one IEEE binary32 operation at a time in a fixed order so
// that results do not depend on compiler contraction.
__device__ __forceinline__ void adams_update(float g, float& w, float& m, const AdamsConst& c) {
  const float m_prev = m, w_prev = w;
  const float m_new = __fadd_rn(__fmul_rn(c.beta1, m_prev), __fmul_rn(c.one_minus_b1, g));
  const float v = __fadd_rn(__fmul_rn(c.beta2, __fmul_rn(m_prev, m_prev)),
                            __fmul_rn(c.one_minus_b2, __fmul_rn(g, g)));
  const float m_hat = __fdiv_rn(m_new, c.bc1);
  const float v_hat = __fdiv_rn(v, c.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), c.eps);
  const float upd = __fadd_rn(__fdiv_rn(m_hat, denom), __fmul_rn(c.wd, w_prev));
  w = __fsub_rn(w_prev, __fmul_rn(c.lr, upd));
  m = m_new;
}

// AdamW update of one coordinate (dense baseline): v is an EMA of g^2.
__device__ __forceinline__ void adamw_update(float g, float& w, float& m, float& v,
                                             const AdamsConst& c) {
  const float w_prev = w;
  const float m_new = __fadd_rn(__fmul_rn(c.beta1, m), __fmul_rn(c.one_minus_b1, g));
  const float v_new = __fadd_rn(__fmul_rn(c.beta2, v), __fmul_rn(c.one_minus_b2, __fmul_rn(g, g)));
  const float m_hat = __fdiv_rn(m_new, c.bc1);
  const float v_hat = __fdiv_rn(v_new, c.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), c.eps);
  const float upd = __fadd_rn(__fdiv_rn(m_hat, denom), __fmul_rn(c.wd, w_prev));
  w = __fsub_rn(w_prev, __fmul_rn(c.lr, upd));
  m = m_new;
  v = v_new;
}

// AdamS update when the synchronised buffer holds the first moment b
// (m_t = b) and the gradient is recovered as g = (b - b1 m_{t-1}) / (1 - b1).
__device__ __forceinline__ void adams_update_from_moment(float b, float& w, float& m,
                                                         const AdamsConst& c) {
  const float m_prev = m, w_prev = w;
  const float g = __fdiv_rn(__fsub_rn(b, __fmul_rn(c.beta1, m_prev)), c.one_minus_b1);
  const float v = __fadd_rn(__fmul_rn(c.beta2, __fmul_rn(m_prev, m_prev)),
                            __fmul_rn(c.one_minus_b2, __fmul_rn(g, g)));
  const float m_hat = __fdiv_rn(b, c.bc1);
  const float v_hat = __fdiv_rn(v, c.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), c.eps);
  const float upd = __fadd_rn(__fdiv_rn(m_hat, denom), __fmul_rn(c.wd, w_prev));
  w = __fsub_rn(w_prev, __fmul_rn(c.lr, upd));
  m = b;
}

// First-moment packing of the compaction (variant reading): m_{t-1} and b1.
struct MomentPack {
  const float* m;
  float beta1, c1;
};

// Reduction and update carried by a compaction launch.  A launch covers a
// group of consecutive workers; with kEfAccum it keeps, per selected slot, the
// worker-ordered sum of the packed values (started from the group's first
// worker, or with kEfResume from the partial sum left in gbar by the previous
// group) and stores it back to gbar; with kEfFinish it stores g_bar = sum / W
// instead (no reduce launch needed), and with kEfUpdate also applies AdamS at
// the selected coordinates (no adams_sparse launch needed).
constexpr int kEfAccum = 1, kEfResume = 2, kEfFinish = 4, kEfUpdate = 8;
struct EfFuse {
  float* gbar;
  float* w;
  float* m;
  AdamsConst c;
  int W_total;
  int flags;
};

// Streaming multiprocessors of the current device (persistent grids are sized
// from it).  Looked up once per device and cached; safe to call from any host
// thread.
int sm_count();

// ---------------------------------------------------------------- launchers
// Each returns cudaGetLastError() after enqueueing on `st`.
// moment: step 1 under the first-moment buffer reading.
cudaError_t launch_dense_step(const WorkerPtrs& p, int W, int64_t P, int dtype, bool vec,
                              float* w, float* m, const AdamsConst& c, bool moment,
                              cudaStream_t st);
// mp == nullptr: the selected a^w are packed; else b = b1 m + (1 - b1) a^w.
cudaError_t launch_ef_compact(const WorkerPtrs& p, int W, int64_t P, int dtype, bool vec,
                              const uint32_t* bits, const uint32_t* tile_base, float* pack,
                              int64_t pack_stride, const MomentPack* mp, const EfFuse& fz,
                              cudaStream_t st);
cudaError_t launch_dense_baseline(bool adamw, const WorkerPtrs& p, int W, int64_t P, int dtype,
                                  bool vec, float* w, float* m, float* v, const AdamsConst& c,
                                  cudaStream_t st);
cudaError_t launch_offmask(const uint32_t* bits, int64_t P, float* w, float* m, const AdamsConst& c,
                           cudaStream_t st);
// dst[idx[j]] = w[idx[j]], j < k (dst: device address of mapped host memory)
cudaError_t launch_param_patch(const uint32_t* idx, int64_t k, const float* w, float* dst,
                               cudaStream_t st);
cudaError_t launch_reduce(const float* pack, int64_t pack_stride, int W, int64_t k, float* gbar,
                          cudaStream_t st);
// Timing probe: adams_sparse's memory accesses without its arithmetic (w and m
// written back unchanged).
cudaError_t launch_probe_rmw(const uint32_t* idx, const float* gbar, int64_t k, float* w,
                             float* m, cudaStream_t st);
// multi-rank exchange helpers (step_kernels.cu)
cudaError_t launch_adams_dense(const float* gbar, int64_t n, float* w, float* m,
                               const AdamsConst& c, cudaStream_t st);
cudaError_t launch_index_move(bool scatter, const uint32_t* idx, int64_t k, const float* src,
                              float* dst, cudaStream_t st);
cudaError_t launch_align_bits(const uint32_t* local, int64_t n, int shift, uint32_t* out,
                              int64_t nw_out, cudaStream_t st);
cudaError_t launch_or_words(const uint32_t* src, int64_t nw, uint32_t* dst, cudaStream_t st);
cudaError_t launch_adams_sparse(const uint32_t* idx, const float* gbar, int64_t k, float* w,
                                float* m, const AdamsConst& c, bool msync, cudaStream_t st);

cudaError_t launch_hist(int pass, const float* m, int64_t P, const ShardMap& sm,
                        const int64_t* shard_start,
                        const ShardSel* sel, uint32_t* hist, cudaStream_t st);
cudaError_t launch_select(int pass, int W, const int64_t* shard_start, const int64_t* shard_k,
                          ShardSel* sel, uint32_t* hist, cudaStream_t st);
cudaError_t launch_tie_count(const float* m, int W, const int64_t* shard_start,
                             const ShardSel* sel, uint32_t* eqcnt, int64_t nchunk,
                             cudaStream_t st);
cudaError_t launch_tie_select(const float* m, int W, const int64_t* shard_start, ShardSel* sel,
                              const uint32_t* eqcnt, int64_t nchunk, cudaStream_t st);
// accumulate: OR the new bits into `bits` instead of overwriting them.
cudaError_t launch_mark(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                        const ShardSel* sel, uint32_t* bits, uint32_t* tile_cnt,
                        cudaStream_t st, bool accumulate = false);
// union-mask baseline (union_kernels.cu)
cudaError_t launch_ef_add(const WorkerPtrs& p, int W, int64_t P, int dtype, bool vec,
                          cudaStream_t st);
cudaError_t launch_union_move(const WorkerPtrs& p, int W, const uint32_t* idx, int64_t k,
                              float* pack, int64_t stride, cudaStream_t st);
cudaError_t launch_tile_count(const uint32_t* bits, int64_t P, uint32_t* tile_cnt,
                              cudaStream_t st);
// Three launches; `scratch` holds scan_scratch_words(ntiles) words.
int64_t scan_scratch_words(int64_t ntiles);
cudaError_t launch_scan(const uint32_t* tile_cnt, int64_t ntiles, uint32_t* tile_base,
                        uint32_t* scratch, cudaStream_t st);
constexpr int kScanLaunches = 3;
// k: number of set bits if known (picks the kernel for the density), else -1.
cudaError_t launch_index(const uint32_t* bits, int64_t P, const uint32_t* tile_base,
                         uint32_t* idx, int64_t k, cudaStream_t st);
// candidate-based exact top-k threshold (topk_kernels.cu)
// First digit of the candidate select: the top kDigit0 bits of the 31-bit
// magnitude key (8 exponent bits + 5 mantissa bits: buckets 1/32 of an octave
// wide), key >> kKeyShift0.
constexpr int kDigit0 = 13;
constexpr int kKeyShift0 = 31 - kDigit0;
constexpr int kCandBins0 = 1 << kDigit0;
// selective: only shards flagged kSelNeedHist, and nothing staged.
cudaError_t launch_chist0(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                          const ShardSel* sel, uint32_t* hist, uint2* cand, uint32_t* cand_cnt,
                          bool selective, int growth, cudaStream_t st);
// Warm refresh: one read of m that writes the bitmap words and popcounts of
// every whole single-shard tile from the shard's previous threshold (tile_cnt
// zeroed first), stages the candidates of the previous bucket window and counts
// the parameters above it (above_cnt zeroed first).
cudaError_t launch_spec(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                        const ShardSel* sel, uint2* cand, uint32_t* cand_cnt, uint32_t* above_cnt,
                        uint32_t* bits, uint32_t* tile_cnt, int growth, cudaStream_t st);
// Window histogram of the staged candidates with the outside counts lumped.
cudaError_t launch_whist(int W, int blocks_per_shard, const int64_t* shard_start,
                         const ShardSel* sel, const uint2* cand, const uint32_t* cand_cnt,
                         const uint32_t* above_cnt, uint32_t* hist, int growth, cudaStream_t st);
// Flip the candidates whose selection differs between the previous and the new
// threshold (shards without kSelRemark).
cudaError_t launch_fixup(const int64_t* shard_start, const ShardSel* sel, const uint2* cand,
                         const uint32_t* cand_cnt, int W, int blocks_per_shard, uint32_t* bits,
                         uint32_t* tile_cnt, cudaStream_t st);
// Mark the tiles the speculative bitmap does not cover: every tile starting in
// a kSelRemark shard, and each shard's last tile when it crosses the shard end
// or the end of the vector.
cudaError_t launch_remark(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                          const ShardSel* sel, uint32_t* bits, uint32_t* tile_cnt,
                          cudaStream_t st);
// form (pass 0): kSelFormCold on a full histogram, kSelFormWarm on the window
// histogram, kSelFormRerun for the kSelNeedHist shards after their full count.
constexpr int kSelFormCold = 0, kSelFormWarm = 1, kSelFormRerun = 2;
// growth: how many first-digit buckets above the previous threshold's the
// window of a warm refresh also covers (the expected growth of the first
// moments since the previous refresh); 0 elsewhere.
cudaError_t launch_cselect(int pass, int W, const int64_t* shard_start, const int64_t* shard_k,
                           ShardSel* sel, uint32_t* hist, uint32_t* cand_cnt, int form,
                           int growth, cudaStream_t st);
cudaError_t launch_collect(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                           const ShardSel* sel, uint2* cand, uint32_t* cand_cnt, cudaStream_t st);
// nar (optional): per-shard rows of nar_cap candidates, counts in nar_cnt
// (zeroed before pass 2): pass 2 narrows the list there for passes 3 to 5.
constexpr uint32_t kNarrowCap = 4096;
cudaError_t launch_chist(int pass, int W, int blocks_per_shard, const int64_t* shard_start,
                         const ShardSel* sel, const uint2* cand, const uint32_t* cand_cnt,
                         uint32_t* hist, uint2* nar, uint32_t* nar_cnt, uint32_t nar_cap,
                         cudaStream_t st);
cudaError_t launch_shard_count(const uint32_t* bits, int64_t P, int64_t nwords, const ShardMap& sm,
                               uint32_t* counts, cudaStream_t st);

}  // namespace scapek
