// scape_handle.cuh -- the handle behind scape_t and the host helpers shared by
// the C ABI's translation units (scape_api.cu, scape_xc.cu).  Not installed:
// callers see only include/scape.h.
#pragma once

#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "scape_internal.cuh"

namespace scapek {
namespace host {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// kernel names, indexed by KernelId (scape_api.cu)
extern const char* const kKernelNames[kNumKernels];

struct ProfRec {
  int kid;
  int nlaunch;
  cudaEvent_t a, b;
};

}  // namespace host
}  // namespace scapek

using scapek::AdamsConst;
using scapek::kNumKernels;
using scapek::ShardMap;
using scapek::ShardSel;

struct scape {
  // configuration
  int64_t P = 0;       // parameters this handle covers
  int W = 0;           // workers (gradient slices per step)
  int S = 0;           // optimizer shards this handle covers
  int64_t ppm = 0;
  // global layout: shards [shard_begin, shard_begin + S) of an even W-way split
  // of P_global parameters, the first at global index offset
  int64_t P_global = 0, offset = 0;
  int shard_begin = 0;
  ShardMap map{};
  float beta1 = 0, beta2 = 0, lr = 0, eps = 0, wd = 0;
  int dtype = SCAPE_BF16;
  std::vector<int64_t> shard_start, shard_k;
  int64_t k = 0;
  int64_t ntiles = 0, nwords = 0, kstride = 0;
  int cand_blocks = 1;  // blocks per shard of the candidate histogram passes
  bool all_dense = false;  // every shard keeps all of its coordinates
  int variant = SCAPE_VARIANT_PAPER;
  int fusion = SCAPE_FUSE_SUM;  // what the compaction pass also does
  // workspace offsets (bytes)
  size_t off_bits = 0, off_idx = 0, off_tbase = 0, off_tcnt = 0, off_pack = 0, off_gbar = 0,
         off_hist = 0, off_sel = 0, off_cand = 0, off_ccnt = 0, off_scan = 0, off_sstart = 0,
         off_sk = 0, off_counts = 0, off_nar = 0,
         ws_need = 0;
  // bound memory
  bool bound = false;
  float* w = nullptr;
  float* m = nullptr;
  std::vector<float*> e;
  char* ws = nullptr;
  // state
  int64_t t = 0;
  bool mask_ready = false;
  bool warm = false;  // the select state holds a finished threshold per shard
  bool buffers_valid = false;
  int64_t launches = 0;
  // union-mask baseline: workspace whose per-worker selection state is live
  const void* union_ws = nullptr;
  // end-to-end pipelining (created on the first scape_step_host call)
  static constexpr int kMaxGroups = 16;
  bool aux_ready = false;
  cudaStream_t copy_stream = nullptr, down_stream = nullptr;
  cudaEvent_t ev_start = nullptr, ev_updated = nullptr, ev_done = nullptr, ev_down = nullptr;
  cudaEvent_t ev_group[kMaxGroups] = {};
  // residuals in host memory moved through a device staging buffer
  bool e_on_host = false;          // every e^w is host memory
  float* stage = nullptr;          // staging buffer (caller-owned device memory)
  int stage_workers = 0;           // residual rows it holds
  int64_t stage_stride = 0;        // floats per row (P rounded up to 64)
  std::vector<cudaEvent_t> ev_in, ev_comp, ev_out;  // per worker group
  // CUDA graph of the steady warm refresh (and the rebuild of its index list):
  // captured once on an internal stream, replayed on the caller's stream
  bool graphs = true;               // scape_set_graphs
  bool graph_failed = false;        // capture or instantiation failed: eager from then on
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t refresh_exec = nullptr;
  int64_t graph_launches = 0;       // kernel launches one replay makes
  // profiling
  bool prof = false;
  uint32_t prof_mask = 0xFFFFFFFFu;  // kernels whose launches are bracketed by events
  std::vector<scapek::host::ProfRec> pending;
  std::vector<cudaEvent_t> pool;
  double prof_ms[kNumKernels] = {};
  int64_t prof_n[kNumKernels] = {};
  std::string err;

  template <class T>
  T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
  uint32_t* bits() const { return at<uint32_t>(off_bits); }
  uint32_t* idx() const { return at<uint32_t>(off_idx); }
  uint32_t* tile_base() const { return at<uint32_t>(off_tbase); }
  uint32_t* tile_cnt() const { return at<uint32_t>(off_tcnt); }
  float* pack() const { return at<float>(off_pack); }
  float* gbar() const { return at<float>(off_gbar); }
  uint32_t* hist() const { return at<uint32_t>(off_hist); }
  ShardSel* sel() const { return at<ShardSel>(off_sel); }
  uint2* cand() const { return at<uint2>(off_cand); }
  uint32_t* cand_cnt() const { return at<uint32_t>(off_ccnt); }
  uint32_t* above_cnt() const { return at<uint32_t>(off_ccnt) + S; }
  uint32_t* nar_cnt() const { return at<uint32_t>(off_ccnt) + 2 * S; }
  uint2* nar() const { return at<uint2>(off_nar); }
  uint32_t* scan_scratch() const { return at<uint32_t>(off_scan); }
  int64_t* d_shard_start() const { return at<int64_t>(off_sstart); }
  int64_t* d_shard_k() const { return at<int64_t>(off_sk); }
  uint32_t* counts() const { return at<uint32_t>(off_counts); }
};

namespace scapek {
namespace host {

inline int fail(scape_t* h, int code, const std::string& msg) {
  if (h) h->err = msg;
  return code;
}

inline int cuda_fail(scape_t* h, cudaError_t e, const char* what) {
  return fail(h, SCAPE_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

inline cudaEvent_t take_event(scape_t* h) {
  if (!h->pool.empty()) {
    cudaEvent_t ev = h->pool.back();
    h->pool.pop_back();
    return ev;
  }
  cudaEvent_t ev = nullptr;
  if (cudaEventCreate(&ev) != cudaSuccess) return nullptr;
  return ev;
}

// Enqueue one kernel through `fn` (which returns the launch status), with
// optional event bracketing for per-kernel timing.
template <class F>
int run_kernel(scape_t* h, int kid, cudaStream_t st, F&& fn, int nlaunch = 1) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool timed = h->prof && ((h->prof_mask >> kid) & 1u);
  if (timed) {
    a = take_event(h);
    b = take_event(h);
    if (a && b) cudaEventRecord(a, st);
  }
  // a named host range per launch for timeline tools (no cost without one)
  nvtxRangePushA(kKernelNames[kid]);
  const cudaError_t e = fn();
  nvtxRangePop();
  h->launches += nlaunch;
  if (timed && a && b) {
    cudaEventRecord(b, st);
    h->pending.push_back({kid, nlaunch, a, b});
  }
  if (e != cudaSuccess) return cuda_fail(h, e, kKernelNames[kid]);
  return SCAPE_OK;
}

inline AdamsConst make_const(const scape_t* h, int64_t t) {
  AdamsConst c;
  c.beta1 = h->beta1;
  c.beta2 = h->beta2;
  c.one_minus_b1 = 1.0f - h->beta1;
  c.one_minus_b2 = 1.0f - h->beta2;
  c.bc1 = (float)(1.0 - std::pow((double)h->beta1, (double)t));
  c.bc2 = (float)(1.0 - std::pow((double)h->beta2, (double)t));
  c.lr = h->lr;
  c.eps = h->eps;
  c.wd = h->wd;
  return c;
}

// Free the captured refresh graph (its launches point into the bound workspace).
inline void drop_graph(scape_t* h) {
  if (h->refresh_exec) cudaGraphExecDestroy(h->refresh_exec);
  h->refresh_exec = nullptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace host
}  // namespace scapek
