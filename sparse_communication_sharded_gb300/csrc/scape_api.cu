// scape_api.cu -- host implementation of the SCAPE C ABI (include/scape.h).
//
// Holds the shard layout, the caller-bound device pointers, the step count and
// the carve-up of the caller's workspace; enqueues the kernels of
// step_kernels.cu, topk_kernels.cu, refresh_kernels.cu and union_kernels.cu on
// the caller's stream (plus internal copy streams for the host-memory paths).
// Never allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "scape_handle.cuh"

using namespace scapek;

namespace scapek {

int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return 152;
  }
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace scapek

namespace scapek {
namespace host {

const char* const kKernelNames[kNumKernels] = {
    "dense_step",  "ef_compact", "reduce", "adams_sparse", "cand_hist0", "cand_select",
    "cand_collect", "cand_hist",  "mark",   "scan",         "index",      "shard_count",
    "tile_count",  "offmask",    "dense_adams", "adamw", "ef_add", "union_move", "spec_mark",
    "fixup", "remark", "param_patch", "dense_update", "xc_move", "probe_rmw"};

}  // namespace host
}  // namespace scapek

using namespace scapek::host;

namespace {

thread_local std::string g_create_error;

// Compaction of workers [w0, w1) into rows w0.. of the packed buffers; with
// the fused update, the ordered sum continues across the groups in g_bar and
// the group that ends at W applies AdamS.
int enqueue_compact(scape_t* h, const WorkerPtrs& all, int w0, int w1, bool vec,
                    const AdamsConst& c, cudaStream_t st) {
  const MomentPack mp{h->m, h->beta1, 1.0f - h->beta1};
  const MomentPack* mpp = (h->variant & SCAPE_VARIANT_MOMENT_SYNC) ? &mp : nullptr;
  WorkerPtrs p;
  std::memset(&p, 0, sizeof p);
  for (int w = w0; w < w1; ++w) {
    p.g[w - w0] = all.g[w];
    p.e[w - w0] = all.e[w];
  }
  EfFuse fz{h->gbar(), h->w, h->m, c, h->W, 0};
  if (h->fusion != SCAPE_FUSE_NONE) {
    fz.flags = kEfAccum;
    if (w0 > 0) fz.flags |= kEfResume;
    if (w1 == h->W) fz.flags |= kEfFinish;
    if (w1 == h->W && h->fusion == SCAPE_FUSE_UPDATE) fz.flags |= kEfUpdate;
  }
  return run_kernel(h, kKEfCompact, st, [&] {
    return launch_ef_compact(p, w1 - w0, h->P, h->dtype, vec, h->bits(), h->tile_base(),
                             h->pack() + (int64_t)w0 * h->kstride, h->kstride, mpp, fz, st);
  });
}

// The ordered sum of the packed buffers and the sparse AdamS update, unless
// the compaction already applied them (plus, under the dense off-mask
// reading, the zero-gradient update elsewhere).
int enqueue_update(scape_t* h, const AdamsConst& c, cudaStream_t st) {
  int rc = SCAPE_OK;
  if (h->fusion == SCAPE_FUSE_NONE) {
    rc = run_kernel(h, kKReduce, st, [&] {
      return launch_reduce(h->pack(), h->kstride, h->W, h->k, h->gbar(), st);
    });
    if (rc) return rc;
  }
  if (h->fusion != SCAPE_FUSE_UPDATE) {
    const bool msync = (h->variant & SCAPE_VARIANT_MOMENT_SYNC) != 0;
    if (h->all_dense && !msync) {
      // every coordinate kept: slot j is coordinate j, no index list to read
      rc = run_kernel(h, kKDenseUpdate, st, [&] {
        return launch_adams_dense(h->gbar(), h->P, h->w, h->m, c, st);
      });
    } else {
      rc = run_kernel(h, kKAdamsSparse, st, [&] {
        return launch_adams_sparse(h->idx(), h->gbar(), h->k, h->w, h->m, c, msync, st);
      });
    }
  }
  if (rc || !(h->variant & SCAPE_VARIANT_DENSE_OFFMASK)) return rc;
  return run_kernel(h, kKOffmask, st,
                    [&] { return launch_offmask(h->bits(), h->P, h->w, h->m, c, st); });
}

// Rank table and index list from the bitmap already in the workspace.
int rebuild_from_bits(scape_t* h, cudaStream_t st, bool counts_ready) {
  int rc;
  if (!counts_ready) {
    rc = run_kernel(h, kKTileCount, st,
                    [&] { return launch_tile_count(h->bits(), h->P, h->tile_cnt(), st); });
    if (rc) return rc;
  }
  rc = run_kernel(
      h, kKScan, st,
      [&] { return launch_scan(h->tile_cnt(), h->ntiles, h->tile_base(), h->scan_scratch(), st); },
      kScanLaunches);
  if (rc) return rc;
  return run_kernel(h, kKIndex, st,
                    [&] { return launch_index(h->bits(), h->P, h->tile_base(), h->idx(), h->k, st); });
}

// Internal streams and events of the pipelined paths (created on first use).
int ensure_aux(scape_t* h) {
  if (h->aux_ready) return SCAPE_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->down_stream, cudaStreamNonBlocking);
  for (auto* ev : {&h->ev_start, &h->ev_updated, &h->ev_done, &h->ev_down})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int g = 0; g < scape_t::kMaxGroups && e == cudaSuccess; ++g)
    e = cudaEventCreateWithFlags(&h->ev_group[g], cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_fail(h, e, "stream/event setup");
  h->aux_ready = true;
  return SCAPE_OK;
}

// A sparse step whose residuals live in host memory, moved through the
// device staging buffer in worker groups: three groups are in flight, one
// copying in (copy stream), one being compacted (`st`), one copying back
// (download stream), so both directions of the host link stay busy.  The
// staging rows of group g are reused by group g + 3 once its copy-back ended.
int step_staged(scape_t* h, const WorkerPtrs& grads, bool vec, const AdamsConst& c,
                cudaStream_t st) {
  int rc = ensure_aux(h);
  if (rc) return rc;
  const int gsz = h->stage_workers / 3;
  const int G = (h->W + gsz - 1) / gsz;
  cudaError_t e = cudaSuccess;
  for (auto* v : {&h->ev_in, &h->ev_comp, &h->ev_out})
    while ((int)v->size() < G && e == cudaSuccess) {
      cudaEvent_t ev = nullptr;
      e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e == cudaSuccess) v->push_back(ev);
    }
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step: staging events");
  cudaStream_t cp = h->copy_stream, dn = h->down_stream;
  const size_t eb = (size_t)h->P * 4;
  e = cudaEventRecord(h->ev_start, st);  // the residuals' earlier users
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cp, h->ev_start, 0);
  for (int g = 0; g < G && e == cudaSuccess; ++g) {
    const int w0 = g * gsz, w1 = w0 + gsz < h->W ? w0 + gsz : h->W;
    float* rows = h->stage + (int64_t)(g % 3) * gsz * h->stage_stride;
    if (g >= 3) e = cudaStreamWaitEvent(cp, h->ev_out[g - 3], 0);
    for (int w = w0; w < w1 && e == cudaSuccess; ++w)
      e = cudaMemcpyAsync(rows + (int64_t)(w - w0) * h->stage_stride, h->e[w], eb,
                          cudaMemcpyHostToDevice, cp);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[g], cp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_in[g], 0);
    if (e != cudaSuccess) break;
    WorkerPtrs p = grads;
    for (int w = w0; w < w1; ++w) p.e[w] = rows + (int64_t)(w - w0) * h->stage_stride;
    rc = enqueue_compact(h, p, w0, w1, vec, c, st);
    if (rc) return rc;
    e = cudaEventRecord(h->ev_comp[g], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(dn, h->ev_comp[g], 0);
    for (int w = w0; w < w1 && e == cudaSuccess; ++w)
      e = cudaMemcpyAsync(h->e[w], rows + (int64_t)(w - w0) * h->stage_stride, eb,
                          cudaMemcpyDeviceToHost, dn);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[g], dn);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step: residual staging");
  rc = enqueue_update(h, c, st);
  if (rc) return rc;
  // the step is complete once the last residuals are home
  e = cudaStreamWaitEvent(st, h->ev_out[G - 1], 0);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step: stream wait");
  return SCAPE_OK;
}

}  // namespace

namespace {

// Handle for shards [a, b) of the even W-way split of the layers' P_global
// parameters (a = 0, b = W: the whole problem).
int create_handle(scape_t** out, int n_layers, const int64_t* host_layer_numel, int W, int a,
                  int b, double sparsity, float beta1, float beta2, float lr, float eps,
                  float weight_decay, int grad_dtype) {
  g_create_error.clear();
  auto bad = [&](const char* msg) {
    g_create_error = msg;
    return SCAPE_EINVAL;
  };
  if (!out) return bad("out is NULL");
  *out = nullptr;
  if (n_layers < 1 || !host_layer_numel) return bad("need at least one layer size");
  int64_t P = 0;
  for (int i = 0; i < n_layers; ++i) {
    if (host_layer_numel[i] < 0) return bad("negative layer size");
    P += host_layer_numel[i];
    if (P > 2147483647LL) return bad("P exceeds 2^31 - 1");
  }
  if (P < 1) return bad("P must be >= 1");
  if (W < 1 || W > SCAPE_MAX_WORKERS) return bad("W out of range [1, SCAPE_MAX_WORKERS]");
  if (a < 0 || b > W || a >= b) return bad("shard range must satisfy 0 <= begin < end <= W");
  const int64_t lo = ((int64_t)a * P) / W, hi = ((int64_t)b * P) / W;
  if (hi <= lo) return bad("the shard range holds no parameter");
  if (!(sparsity >= 0.0 && sparsity < 1.0)) return bad("sparsity must be in [0, 1)");
  const int64_t ppm = std::llround(sparsity * 1e6);
  if (ppm >= 1000000) return bad("sparsity rounds to 1 (nothing would be sent)");
  if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f))
    return bad("betas must be in [0, 1)");
  if (!(eps > 0.f) || !std::isfinite(eps)) return bad("eps must be finite and > 0");
  if (!std::isfinite(lr)) return bad("lr must be finite");
  if (!(weight_decay >= 0.f) || !std::isfinite(weight_decay))
    return bad("weight_decay must be finite and >= 0");
  if (grad_dtype != SCAPE_F32 && grad_dtype != SCAPE_BF16) return bad("unknown grad dtype");

  scape_t* h = new (std::nothrow) scape_t();
  if (!h) return bad("out of host memory");
  h->P = hi - lo;
  h->W = W;
  h->S = b - a;
  h->P_global = P;
  h->offset = lo;
  h->shard_begin = a;
  h->map = ShardMap{P, lo, W, a, b - a};
  h->ppm = ppm;
  h->beta1 = beta1;
  h->beta2 = beta2;
  h->lr = lr;
  h->eps = eps;
  h->wd = weight_decay;
  h->dtype = grad_dtype;
  const int S = b - a;
  h->shard_start.resize(S + 1);
  h->shard_k.resize(S);
  int64_t nmax = 0;
  h->all_dense = true;
  // local boundaries: the global ones of shards a..b, less the range's start
  for (int s = 0; s <= S; ++s) h->shard_start[s] = ((int64_t)(a + s) * P) / W - lo;
  for (int s = 0; s < S; ++s) {
    const int64_t n = h->shard_start[s + 1] - h->shard_start[s];
    h->shard_k[s] = (n * (1000000 - ppm) + 999999) / 1000000;
    h->k += h->shard_k[s];
    nmax = n > nmax ? n : nmax;
    if (h->shard_k[s] != n) h->all_dense = false;
  }
  // Default fusion level by density: from 5% of coordinates selected (0.5%
  // with one or two workers, whose compaction streams little per tile) the
  // update inside the compaction pass beats a separate scattered launch;
  // below that, and when every coordinate is kept (coalesced dense update),
  // the separate launch.
  const bool fuse_update = h->k * 20 >= h->P || (W <= 2 && h->k * 200 >= h->P);
  h->fusion = (!h->all_dense && fuse_update) ? SCAPE_FUSE_UPDATE : SCAPE_FUSE_SUM;
  P = h->P;  // from here on: the parameters this handle covers
  h->ntiles = (P + kTile - 1) / kTile;
  h->nwords = (P + 31) / 32;
  h->kstride = (int64_t)align_up((size_t)(h->k > 0 ? h->k : 1), 64);
  // candidate passes: about 1200 blocks in total, at least one per shard
  h->cand_blocks = S >= 1200 ? 1 : 1200 / S;
  (void)nmax;

  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  h->off_bits = carve(align_up((size_t)h->nwords, 64) * 4);
  h->off_idx = carve((size_t)h->kstride * 4);
  h->off_tbase = carve((size_t)(h->ntiles + 1) * 4);
  h->off_tcnt = carve((size_t)h->ntiles * 4);
  h->off_pack = carve((size_t)W * h->kstride * 4);
  h->off_gbar = carve((size_t)h->kstride * 4);
  h->off_hist = carve((size_t)S * kCandBins0 * 4);
  h->off_sel = carve((size_t)S * sizeof(ShardSel));
  // candidates of shard s live in [shard_start[s], shard_start[s+1]): capacity = shard size
  h->off_cand = carve((size_t)P * sizeof(uint2));
  h->off_ccnt = carve((size_t)S * 3 * 4);  // candidate, above-window and narrow-row counts
  h->off_nar = carve((size_t)S * kNarrowCap * sizeof(uint2));
  h->off_scan = carve((size_t)scan_scratch_words(h->ntiles) * 4);
  h->off_sstart = carve((size_t)(S + 1) * 8);
  h->off_sk = carve((size_t)S * 8);
  h->off_counts = carve((size_t)(S + 1) * 4);
  h->ws_need = off;
  *out = h;
  return SCAPE_OK;
}

}  // namespace

extern "C" {

int scape_create(scape_t** out, int n_layers, const int64_t* host_layer_numel, int W,
                 double sparsity, float beta1, float beta2, float lr, float eps,
                 float weight_decay, int grad_dtype) {
  return create_handle(out, n_layers, host_layer_numel, W, 0, W, sparsity, beta1, beta2, lr, eps,
                       weight_decay, grad_dtype);
}

int scape_create_range(scape_t** out, int n_layers, const int64_t* host_layer_numel, int W,
                       int shard_begin, int shard_end, double sparsity, float beta1, float beta2,
                       float lr, float eps, float weight_decay, int grad_dtype) {
  return create_handle(out, n_layers, host_layer_numel, W, shard_begin, shard_end, sparsity,
                       beta1, beta2, lr, eps, weight_decay, grad_dtype);
}

void scape_destroy(scape_t* h) {
  if (!h) return;
  drop_graph(h);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  for (auto& r : h->pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto ev : h->pool) cudaEventDestroy(ev);
  if (h->aux_ready) {
    for (auto ev : h->ev_group) cudaEventDestroy(ev);
    cudaEventDestroy(h->ev_start);
    cudaEventDestroy(h->ev_updated);
    cudaEventDestroy(h->ev_done);
    cudaEventDestroy(h->ev_down);
    cudaStreamDestroy(h->copy_stream);
    cudaStreamDestroy(h->down_stream);
  }
  for (auto* v : {&h->ev_in, &h->ev_comp, &h->ev_out})
    for (auto ev : *v) cudaEventDestroy(ev);
  delete h;
}

const char* scape_last_error(const scape_t* h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

int scape_get_geometry(const scape_t* h, int64_t* P, int* W, int64_t* k, int64_t* host_shard_start,
                       int64_t* host_shard_k) {
  if (!h) return SCAPE_EINVAL;
  if (P) *P = h->P;
  if (W) *W = h->W;
  if (k) *k = h->k;
  if (host_shard_start)
    std::memcpy(host_shard_start, h->shard_start.data(), sizeof(int64_t) * (h->S + 1));
  if (host_shard_k) std::memcpy(host_shard_k, h->shard_k.data(), sizeof(int64_t) * h->S);
  return SCAPE_OK;
}

int scape_get_range(const scape_t* h, int64_t* P_global, int64_t* offset, int* shard_begin,
                    int* shard_end) {
  if (!h) return SCAPE_EINVAL;
  if (P_global) *P_global = h->P_global;
  if (offset) *offset = h->offset;
  if (shard_begin) *shard_begin = h->shard_begin;
  if (shard_end) *shard_end = h->shard_begin + h->S;
  return SCAPE_OK;
}

int scape_workspace_bytes(const scape_t* h, size_t* bytes) {
  if (!h || !bytes) return SCAPE_EINVAL;
  *bytes = h->ws_need;
  return SCAPE_OK;
}

int scape_bind(scape_t* h, float* params, float* m, float* const* host_e_ptrs, void* workspace,
               size_t ws_bytes) {
  if (!h) return SCAPE_EINVAL;
  if (!params || !m || !host_e_ptrs || !workspace)
    return fail(h, SCAPE_EINVAL, "scape_bind: NULL pointer");
  if (ws_bytes < h->ws_need) return fail(h, SCAPE_EINVAL, "scape_bind: workspace too small");
  if ((reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return fail(h, SCAPE_EINVAL, "scape_bind: workspace must be 256-byte aligned");
  if (!aligned16(params) || !aligned16(m))
    return fail(h, SCAPE_EINVAL, "scape_bind: params and m must be 16-byte aligned");
  h->e.assign(h->W, nullptr);
  for (int w = 0; w < h->W; ++w) {
    if (!host_e_ptrs[w]) return fail(h, SCAPE_EINVAL, "scape_bind: NULL residual pointer");
    if (!aligned16(host_e_ptrs[w]))
      return fail(h, SCAPE_EINVAL, "scape_bind: residuals must be 16-byte aligned");
    h->e[w] = host_e_ptrs[w];
  }
  // residuals in host memory (page-locked, or pageable where the device can
  // address it): candidates for the staged step
  h->e_on_host = true;
  for (int w = 0; w < h->W; ++w) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h->e[w]) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;  // not known to CUDA: host memory
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) h->e_on_host = false;
  }
  h->w = params;
  h->m = m;
  h->ws = static_cast<char*>(workspace);
  // the small shard table lives in the workspace for the kernels
  cudaError_t e = cudaMemcpy(h->d_shard_start(), h->shard_start.data(), 8 * (h->S + 1),
                             cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_shard_k(), h->shard_k.data(), 8 * h->S, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_bind: shard table upload");
  // no previous mask: every shard starts without a bucket guess
  e = cudaMemset(h->sel(), 0xFF, sizeof(ShardSel) * h->S);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_bind: select state reset");
  drop_graph(h);  // its launches point into the previous workspace
  h->bound = true;
  h->t = 0;
  h->mask_ready = false;
  h->warm = false;
  h->buffers_valid = false;
  return SCAPE_OK;
}

int scape_step(scape_t* h, const void* const* host_grad_ptrs, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return fail(h, SCAPE_ESTATE, "scape_step: call scape_bind first");
  if (!host_grad_ptrs) return fail(h, SCAPE_EINVAL, "scape_step: NULL gradient table");
  if (h->t >= 1 && !h->mask_ready)
    return fail(h, SCAPE_ESTATE, "scape_step: no mask yet; call scape_refresh_mask after step 1");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WorkerPtrs p;
  std::memset(&p, 0, sizeof p);
  bool vec = true;
  for (int w = 0; w < h->W; ++w) {
    if (!host_grad_ptrs[w]) return fail(h, SCAPE_EINVAL, "scape_step: NULL gradient pointer");
    p.g[w] = host_grad_ptrs[w];
    p.e[w] = h->e[w];
    vec = vec && aligned16(host_grad_ptrs[w]);
  }
  const int64_t t = h->t + 1;
  const AdamsConst c = make_const(h, t);
  int rc;
  if (t == 1) {
    rc = run_kernel(h, kKDenseStep, st, [&] {
      return launch_dense_step(p, h->W, h->P, h->dtype, vec, h->w, h->m, c,
                               (h->variant & SCAPE_VARIANT_MOMENT_SYNC) != 0, st);
    });
    if (rc) return rc;
    h->buffers_valid = false;
  } else if (h->e_on_host && h->stage) {
    rc = step_staged(h, p, vec, c, st);
    if (rc) return rc;
    h->buffers_valid = true;
  } else {
    rc = enqueue_compact(h, p, 0, h->W, vec, c, st);
    if (rc) return rc;
    rc = enqueue_update(h, c, st);
    if (rc) return rc;
    h->buffers_valid = true;
  }
  h->t = t;
  return SCAPE_OK;
}

namespace {

// Radix passes 1..5 over the staged candidates.
int enqueue_radix(scape_t* h, cudaStream_t st) {
  for (int pass = 1; pass <= 5; ++pass) {
    int rc = run_kernel(h, kKCandHist, st, [&] {
      return launch_chist(pass, h->S, h->cand_blocks, h->d_shard_start(), h->sel(), h->cand(),
                          h->cand_cnt(), h->hist(), h->nar(), h->nar_cnt(), kNarrowCap, st);
    });
    if (rc) return rc;
    rc = run_kernel(h, kKCandSelect, st, [&] {
      return launch_cselect(pass, h->S, h->d_shard_start(), h->d_shard_k(), h->sel(), h->hist(),
                            h->cand_cnt(), kSelFormCold, 0, st);
    });
    if (rc) return rc;
  }
  return SCAPE_OK;
}

// First refresh after bind (and every refresh of a mask of all ones): full
// histogram, bucket, collect on a miss, radix passes, then the mark pass.
int refresh_cold(scape_t* h, cudaStream_t st) {
  int rc;
  if (!h->all_dense) {
    cudaError_t e = cudaMemsetAsync(h->hist(), 0, (size_t)h->S * kCandBins0 * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->cand_cnt(), 0, (size_t)h->S * 3 * 4, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "scape_refresh_mask: histogram clear");
    rc = run_kernel(h, kKCandHist0, st, [&] {
      return launch_chist0(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->hist(), h->cand(),
                           h->cand_cnt(), false, 0, st);
    });
    if (rc) return rc;
  }
  rc = run_kernel(h, kKCandSelect, st, [&] {
    return launch_cselect(0, h->S, h->d_shard_start(), h->d_shard_k(), h->sel(), h->hist(),
                          h->cand_cnt(), kSelFormCold, 0, st);
  });
  if (rc) return rc;
  if (!h->all_dense) {
    rc = run_kernel(h, kKCandCollect, st, [&] {
      return launch_collect(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->cand(),
                            h->cand_cnt(), st);
    });
    if (rc) return rc;
    rc = enqueue_radix(h, st);
    if (rc) return rc;
  }
  return run_kernel(h, kKMark, st, [&] {
    return launch_mark(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->bits(), h->tile_cnt(),
                       st);
  });
}

// Warm-up widening of the bucket windows for the refresh after step t: the
// expected growth of the selected first moments since the previous refresh,
// the ratio of the bias corrections (1 - b1^t) / (1 - b1^(t-1)) in first-digit
// buckets (32 per octave), while it is at least kWidenFrom buckets -- the
// refreshes after steps 2 to 4 with b1 = 0.9, whose thresholds move by up to
// about 10 buckets either way -- and 0 afterwards (the trend then suffices).
constexpr int kWidenFrom = 11;

int warm_growth(const scape_t* h) {
  if (h->t < 2 || !(h->beta1 > 0.f)) return 0;
  const double b1 = h->beta1;
  const double r = (1.0 - std::pow(b1, (double)h->t)) / (1.0 - std::pow(b1, (double)(h->t - 1)));
  const int g = (int)std::lround(32.0 * std::log2(r));
  return g >= kWidenFrom ? g : 0;
}

// Every later refresh: the bitmap is written speculatively from the previous
// thresholds in the same read of m that stages the candidates; the new
// thresholds only correct it.  Every launch is enqueued whatever the data
// holds; the kernels for the rare cases (a shard whose threshold left its
// bucket window) return at once when no shard needs them.
int refresh_warm(scape_t* h, cudaStream_t st, int growth) {
  // the histogram rows need no clearing: every refresh leaves them zero (each
  // select pass clears the rows it read, and rows of shards no pass reads are
  // never written); the cold refresh after a bind clears them once
  cudaError_t e = cudaMemsetAsync(h->cand_cnt(), 0, (size_t)h->S * 3 * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->tile_cnt(), 0, (size_t)h->ntiles * 4, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_refresh_mask: count clear");
  int rc = run_kernel(h, kKSpecMark, st, [&] {
    return launch_spec(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->cand(), h->cand_cnt(),
                       h->above_cnt(), h->bits(), h->tile_cnt(), growth, st);
  });
  if (rc) return rc;
  rc = run_kernel(h, kKCandHist, st, [&] {
    return launch_whist(h->S, h->cand_blocks, h->d_shard_start(), h->sel(), h->cand(),
                        h->cand_cnt(), h->above_cnt(), h->hist(), growth, st);
  });
  if (rc) return rc;
  rc = run_kernel(h, kKCandSelect, st, [&] {
    return launch_cselect(0, h->S, h->d_shard_start(), h->d_shard_k(), h->sel(), h->hist(),
                          h->cand_cnt(), kSelFormWarm, growth, st);
  });
  if (rc) return rc;
  rc = run_kernel(h, kKCandHist0, st, [&] {
    return launch_chist0(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->hist(), h->cand(),
                         h->cand_cnt(), true, 0, st);
  });
  if (rc) return rc;
  rc = run_kernel(h, kKCandSelect, st, [&] {
    return launch_cselect(0, h->S, h->d_shard_start(), h->d_shard_k(), h->sel(), h->hist(),
                          h->cand_cnt(), kSelFormRerun, 0, st);
  });
  if (rc) return rc;
  rc = run_kernel(h, kKCandCollect, st, [&] {
    return launch_collect(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->cand(),
                          h->cand_cnt(), st);
  });
  if (rc) return rc;
  rc = enqueue_radix(h, st);
  if (rc) return rc;
  rc = run_kernel(h, kKFixup, st, [&] {
    return launch_fixup(h->d_shard_start(), h->sel(), h->cand(), h->cand_cnt(), h->S,
                        h->cand_blocks, h->bits(), h->tile_cnt(), st);
  });
  if (rc) return rc;
  return run_kernel(h, kKRemark, st, [&] {
    return launch_remark(h->m, h->P, h->map, h->d_shard_start(), h->sel(), h->bits(),
                         h->tile_cnt(), st);
  });
}

// Capture the steady warm refresh (growth 0) and the rebuild of the rank
// table and index list into a graph, on an internal stream; the captured
// work does not run.  On any failure the handle stays eager.
void capture_refresh(scape_t* h) {
  cudaError_t e = cudaSuccess;
  if (!h->cap_stream) e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    h->graph_failed = true;
    return;
  }
  const int64_t n0 = h->launches;
  cudaGraph_t graph = nullptr;
  e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
  int rc = SCAPE_ECUDA;
  if (e == cudaSuccess) {
    rc = refresh_warm(h, h->cap_stream, 0);
    if (rc == SCAPE_OK) rc = rebuild_from_bits(h, h->cap_stream, true);
    e = cudaStreamEndCapture(h->cap_stream, &graph);
  }
  h->graph_launches = h->launches - n0;
  h->launches = n0;  // nothing ran yet
  if (e == cudaSuccess && rc == SCAPE_OK && graph)
    e = cudaGraphInstantiate(&h->refresh_exec, graph, 0);
  if (graph) cudaGraphDestroy(graph);
  if (e != cudaSuccess || rc != SCAPE_OK || !h->refresh_exec) {
    (void)cudaGetLastError();
    h->err.clear();
    h->refresh_exec = nullptr;
    h->graph_failed = true;
  }
}

}  // namespace

int scape_refresh_mask(scape_t* h, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return fail(h, SCAPE_ESTATE, "scape_refresh_mask: call scape_bind first");
  if (h->t < 1) return fail(h, SCAPE_ESTATE, "scape_refresh_mask: no step taken yet");
  // every shard keeps all of its coordinates: the mask is all ones whatever m
  // holds, and the one built already (bitmap, index list, rank table) stands
  if (h->all_dense && h->mask_ready) return SCAPE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool warm = h->warm && !h->all_dense;
  const int growth = warm ? warm_growth(h) : 0;
  // The steady warm refresh enqueues the same launches with the same
  // arguments every time: replay it as one graph (unless profiling brackets
  // its launches, or the caller is capturing its own stream).
  constexpr uint32_t kRefreshKernels =
      (1u << kKCandHist0) | (1u << kKCandSelect) | (1u << kKCandCollect) | (1u << kKCandHist) |
      (1u << kKScan) | (1u << kKIndex) | (1u << kKSpecMark) | (1u << kKFixup) | (1u << kKRemark);
  const bool bracketed = h->prof && (h->prof_mask & kRefreshKernels);
  if (warm && growth == 0 && h->graphs && !h->graph_failed && !bracketed) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
      if (!h->refresh_exec) capture_refresh(h);
      if (h->refresh_exec) {
        const cudaError_t e = cudaGraphLaunch(h->refresh_exec, st);
        if (e != cudaSuccess) return cuda_fail(h, e, "scape_refresh_mask: graph launch");
        h->launches += h->graph_launches;
        h->mask_ready = true;
        return SCAPE_OK;
      }
    } else {
      (void)cudaGetLastError();
    }
  }
  int rc = warm ? refresh_warm(h, st, growth) : refresh_cold(h, st);
  if (rc) {
    h->warm = false;
    return rc;
  }
  rc = rebuild_from_bits(h, st, true);
  if (rc) return rc;
  h->warm = true;
  h->mask_ready = true;
  return SCAPE_OK;
}

int scape_set_graphs(scape_t* h, int on) {
  if (!h) return SCAPE_EINVAL;
  h->graphs = on != 0;
  return SCAPE_OK;
}

int scape_set_residual_staging(scape_t* h, void* device_buffer, size_t bytes) {
  if (!h) return SCAPE_EINVAL;
  const int64_t stride = (h->P + 63) / 64 * 64;
  if (!device_buffer || bytes == 0) {
    h->stage = nullptr;
    h->stage_workers = 0;
    return SCAPE_OK;
  }
  if (!aligned16(device_buffer))
    return fail(h, SCAPE_EINVAL, "scape_set_residual_staging: buffer must be 16-byte aligned");
  const int64_t rows = (int64_t)(bytes / ((size_t)stride * 4));
  if (rows < 3)
    return fail(h, SCAPE_EINVAL,
                "scape_set_residual_staging: buffer holds fewer than 3 residual rows");
  h->stage = static_cast<float*>(device_buffer);
  h->stage_workers = (int)(rows < h->W ? rows : h->W);
  if (h->stage_workers < 3) h->stage_workers = 3;  // W < 3: groups of one worker
  h->stage_stride = stride;
  return SCAPE_OK;
}

int scape_residual_staging_bytes(const scape_t* h, int rows, size_t* bytes) {
  if (!h || !bytes || rows < 3) return SCAPE_EINVAL;
  *bytes = (size_t)rows * (size_t)((h->P + 63) / 64 * 64) * 4;
  return SCAPE_OK;
}

int scape_get_fusion(const scape_t* h, int* level) {
  if (!h || !level) return SCAPE_EINVAL;
  *level = h->fusion;
  return SCAPE_OK;
}

int scape_set_fusion(scape_t* h, int level) {
  if (!h) return SCAPE_EINVAL;
  if (level != SCAPE_FUSE_NONE && level != SCAPE_FUSE_SUM && level != SCAPE_FUSE_UPDATE)
    return fail(h, SCAPE_EINVAL, "scape_set_fusion: unknown level");
  h->fusion = level;
  return SCAPE_OK;
}

int scape_set_variant(scape_t* h, int flags) {
  if (!h) return SCAPE_EINVAL;
  if (flags & ~(SCAPE_VARIANT_DENSE_OFFMASK | SCAPE_VARIANT_MOMENT_SYNC))
    return fail(h, SCAPE_EINVAL, "scape_set_variant: unknown flag");
  h->variant = flags;
  return SCAPE_OK;
}

// Dense baselines: plain mean of the workers' gradients, AdamS or AdamW on
// every coordinate; no error feedback, no mask.
static int dense_baseline(scape_t* h, const void* const* grads, float* v, bool adamw,
                          void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return fail(h, SCAPE_ESTATE, "dense baseline: call scape_bind first");
  if (!grads || (adamw && !v)) return fail(h, SCAPE_EINVAL, "dense baseline: NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WorkerPtrs p;
  std::memset(&p, 0, sizeof p);
  bool vec = true;
  for (int w = 0; w < h->W; ++w) {
    if (!grads[w]) return fail(h, SCAPE_EINVAL, "dense baseline: NULL gradient pointer");
    p.g[w] = grads[w];
    p.e[w] = h->e[w];
    vec = vec && aligned16(grads[w]);
  }
  const int64_t t = h->t + 1;
  const AdamsConst c = make_const(h, t);
  const int rc = run_kernel(h, adamw ? kKAdamW : kKDenseAdams, st, [&] {
    return launch_dense_baseline(adamw, p, h->W, h->P, h->dtype, vec, h->w, h->m, v, c, st);
  });
  if (rc) return rc;
  h->t = t;
  return SCAPE_OK;
}

int scape_dense_adams_step(scape_t* h, const void* const* host_grad_ptrs, void* stream) {
  return dense_baseline(h, host_grad_ptrs, nullptr, false, stream);
}

int scape_adamw_step(scape_t* h, const void* const* host_grad_ptrs, float* v, void* stream) {
  return dense_baseline(h, host_grad_ptrs, v, true, stream);
}

// ------------------------------------------------------------------ union-mask baseline
namespace {
struct UnionLayout {
  size_t start, kk, sel, hist, cand, ccnt, bits, tcnt, tbase, scan, idx, pack, gbar, total;
  int64_t cstride;
};

UnionLayout union_layout(const scape_t* h, int64_t cap) {
  UnionLayout L;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  L.cstride = (int64_t)align_up((size_t)cap, 64);
  L.start = carve(2 * 8);
  L.kk = carve(8);
  L.sel = carve(sizeof(ShardSel) * h->W);
  L.hist = carve((size_t)kCandBins0 * 4);
  L.cand = carve((size_t)h->P * sizeof(uint2));
  L.ccnt = carve(4);
  L.bits = carve(align_up((size_t)h->nwords, 64) * 4);
  L.tcnt = carve((size_t)h->ntiles * 4);
  L.tbase = carve((size_t)(h->ntiles + 1) * 4);
  L.scan = carve((size_t)scan_scratch_words(h->ntiles) * 4);
  L.idx = carve((size_t)h->P * 4);
  L.pack = carve((size_t)h->W * L.cstride * 4);
  L.gbar = carve((size_t)L.cstride * 4);
  L.total = off;
  return L;
}

int64_t union_k_worker(const scape_t* h) { return (h->P * (1000000 - h->ppm) + 999999) / 1000000; }
}  // namespace

int scape_union_workspace_bytes(const scape_t* h, int64_t capacity, size_t* bytes) {
  if (!h || !bytes || capacity < 1 || capacity > h->P) return SCAPE_EINVAL;
  *bytes = union_layout(h, capacity).total;
  return SCAPE_OK;
}

int scape_union_step(scape_t* h, const void* const* host_grad_ptrs, void* workspace,
                     size_t ws_bytes, int64_t capacity, int64_t* host_k_union, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return fail(h, SCAPE_ESTATE, "scape_union_step: call scape_bind first");
  if (!host_grad_ptrs || !workspace || !host_k_union)
    return fail(h, SCAPE_EINVAL, "scape_union_step: NULL pointer");
  if (capacity < 1 || capacity > h->P)
    return fail(h, SCAPE_EINVAL, "scape_union_step: capacity out of [1, P]");
  const UnionLayout L = union_layout(h, capacity);
  if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return fail(h, SCAPE_EINVAL, "scape_union_step: workspace too small or not 256-byte aligned");
  char* ws = static_cast<char*>(workspace);
  int64_t* ustart = reinterpret_cast<int64_t*>(ws + L.start);
  int64_t* uk = reinterpret_cast<int64_t*>(ws + L.kk);
  ShardSel* usel = reinterpret_cast<ShardSel*>(ws + L.sel);
  uint32_t* uhist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint2* ucand = reinterpret_cast<uint2*>(ws + L.cand);
  uint32_t* ucnt = reinterpret_cast<uint32_t*>(ws + L.ccnt);
  uint32_t* ubits = reinterpret_cast<uint32_t*>(ws + L.bits);
  uint32_t* utcnt = reinterpret_cast<uint32_t*>(ws + L.tcnt);
  uint32_t* utbase = reinterpret_cast<uint32_t*>(ws + L.tbase);
  uint32_t* uscan = reinterpret_cast<uint32_t*>(ws + L.scan);
  uint32_t* uidx = reinterpret_cast<uint32_t*>(ws + L.idx);
  float* upack = reinterpret_cast<float*>(ws + L.pack);
  float* ugbar = reinterpret_cast<float*>(ws + L.gbar);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t kw = union_k_worker(h);
  cudaError_t e = cudaSuccess;
  if (h->union_ws != workspace) {
    // new workspace: one-shard table over the whole vector, no bucket guesses
    const int64_t tab[3] = {0, h->P, kw};
    e = cudaMemcpy(ustart, tab, 16, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(uk, tab + 2, 8, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(usel, 0xFF, sizeof(ShardSel) * h->W);
    if (e != cudaSuccess) return cuda_fail(h, e, "scape_union_step: workspace setup");
    h->union_ws = workspace;
  }
  WorkerPtrs p;
  std::memset(&p, 0, sizeof p);
  bool vec = true;
  for (int w = 0; w < h->W; ++w) {
    if (!host_grad_ptrs[w]) return fail(h, SCAPE_EINVAL, "scape_union_step: NULL gradient pointer");
    p.g[w] = host_grad_ptrs[w];
    p.e[w] = h->e[w];
    vec = vec && aligned16(host_grad_ptrs[w]);
  }
  const int64_t t = h->t + 1;
  const AdamsConst c = make_const(h, t);
  // 1. a^w = g^w + e^w, kept in the residual buffers
  int rc = run_kernel(h, kKEfAdd, st, [&] { return launch_ef_add(p, h->W, h->P, h->dtype, vec, st); });
  if (rc) return rc;
  e = cudaMemsetAsync(ubits, 0, (size_t)h->nwords * 4, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_union_step: bitmap clear");
  // 2. each worker's top-k over the whole vector, OR-ed into the union
  for (int w = 0; w < h->W; ++w) {
    const float* a = h->e[w];
    ShardSel* sw = usel + w;
    if (kw < h->P) {
      e = cudaMemsetAsync(uhist, 0, (size_t)kCandBins0 * 4, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(ucnt, 0, 4, st);
      if (e != cudaSuccess) return cuda_fail(h, e, "scape_union_step: histogram clear");
      rc = run_kernel(h, kKCandHist0, st, [&] {
        return launch_chist0(a, h->P, whole_map(h->P, 1), ustart, sw, uhist, ucand, ucnt, false, 0,
                             st);
      });
      if (rc) return rc;
    }
    rc = run_kernel(h, kKCandSelect, st,
                    [&] { return launch_cselect(0, 1, ustart, uk, sw, uhist, ucnt, kSelFormCold, 0, st); });
    if (rc) return rc;
    if (kw < h->P) {
      rc = run_kernel(h, kKCandCollect, st, [&] {
        return launch_collect(a, h->P, whole_map(h->P, 1), ustart, sw, ucand, ucnt, st);
      });
      if (rc) return rc;
      for (int pass = 1; pass <= 5; ++pass) {
        rc = run_kernel(h, kKCandHist, st, [&] {
          return launch_chist(pass, 1, 1200, ustart, sw, ucand, ucnt, uhist, nullptr, nullptr, 0,
                              st);
        });
        if (rc) return rc;
        rc = run_kernel(h, kKCandSelect, st,
                        [&] { return launch_cselect(pass, 1, ustart, uk, sw, uhist, ucnt, kSelFormCold, 0, st); });
        if (rc) return rc;
      }
    }
    rc = run_kernel(h, kKMark, st, [&] {
      return launch_mark(a, h->P, whole_map(h->P, 1), ustart, sw, ubits, utcnt, st, /*accumulate=*/true);
    });
    if (rc) return rc;
  }
  // 3. rank table and index list of the union; its size to the host
  rc = run_kernel(h, kKTileCount, st, [&] { return launch_tile_count(ubits, h->P, utcnt, st); });
  if (rc) return rc;
  rc = run_kernel(
      h, kKScan, st, [&] { return launch_scan(utcnt, h->ntiles, utbase, uscan, st); },
      kScanLaunches);
  if (rc) return rc;
  rc = run_kernel(h, kKIndex, st, [&] { return launch_index(ubits, h->P, utbase, uidx, -1, st); });
  if (rc) return rc;
  uint32_t ku = 0;
  e = cudaMemcpyAsync(&ku, utbase + h->ntiles, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_union_step: union size readback");
  *host_k_union = ku;
  if ((int64_t)ku > capacity)
    return fail(h, SCAPE_EINVAL,
                "scape_union_step: union larger than capacity (residuals now hold g + e)");
  // 4. every worker sends its values at every union position; mean; AdamS
  rc = run_kernel(h, kKUnionMove, st,
                  [&] { return launch_union_move(p, h->W, uidx, ku, upack, L.cstride, st); });
  if (rc) return rc;
  rc = run_kernel(h, kKReduce, st,
                  [&] { return launch_reduce(upack, L.cstride, h->W, ku, ugbar, st); });
  if (rc) return rc;
  rc = run_kernel(h, kKAdamsSparse, st, [&] {
    return launch_adams_sparse(uidx, ugbar, ku, h->w, h->m, c, false, st);
  });
  if (rc) return rc;
  h->t = t;
  return SCAPE_OK;
}

int scape_set_lr(scape_t* h, float lr) {
  if (!h) return SCAPE_EINVAL;
  if (!std::isfinite(lr)) return fail(h, SCAPE_EINVAL, "scape_set_lr: lr must be finite");
  h->lr = lr;
  return SCAPE_OK;
}

int scape_get_state(const scape_t* h, int64_t* t, int64_t* k, const uint32_t** bits,
                    const uint32_t** idx) {
  if (!h) return SCAPE_EINVAL;
  if (t) *t = h->t;
  if (k) *k = h->k;
  if (bits) *bits = h->bound ? h->bits() : nullptr;
  if (idx) *idx = h->bound ? h->idx() : nullptr;
  return SCAPE_OK;
}

int scape_get_buffers(const scape_t* h, const float** pack, int64_t* pack_stride,
                      const float** gbar) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound || !h->buffers_valid) {
    const_cast<scape_t*>(h)->err = "scape_get_buffers: no sparse step taken since bind";
    return SCAPE_ESTATE;
  }
  if (pack) *pack = h->pack();
  if (pack_stride) *pack_stride = h->kstride;
  if (gbar) *gbar = h->gbar();
  return SCAPE_OK;
}

int scape_set_state(scape_t* h, int64_t t, const uint32_t* bits, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return fail(h, SCAPE_ESTATE, "scape_set_state: call scape_bind first");
  if (t < 1 || !bits) return fail(h, SCAPE_EINVAL, "scape_set_state: need t >= 1 and a bitmap");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h->bits(), bits, (size_t)h->nwords * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->counts(), 0, (size_t)(h->S + 1) * 4, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_set_state: copy");
  int rc = run_kernel(h, kKShardCount, st, [&] {
    return launch_shard_count(h->bits(), h->P, h->nwords, h->map, h->counts(), st);
  });
  if (rc) return rc;
  std::vector<uint32_t> cnt(h->S + 1);
  e = cudaMemcpyAsync(cnt.data(), h->counts(), (size_t)(h->S + 1) * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_set_state: count readback");
  if (cnt[h->S] != 0) {
    h->mask_ready = false;
    return fail(h, SCAPE_EINVAL, "scape_set_state: bitmap has bits set past P");
  }
  for (int s = 0; s < h->S; ++s) {
    if ((int64_t)cnt[s] != h->shard_k[s]) {
      h->mask_ready = false;
      char buf[160];
      std::snprintf(buf, sizeof buf, "scape_set_state: shard %d has %u set bits, expected %lld", s,
                    cnt[s], (long long)h->shard_k[s]);
      return fail(h, SCAPE_EINVAL, buf);
    }
  }
  rc = rebuild_from_bits(h, st, false);
  if (rc) return rc;
  h->t = t;
  h->mask_ready = true;
  h->buffers_valid = false;
  return SCAPE_OK;
}

int scape_step_host(scape_t* h, const void* const* host_grads_src, void* const* host_dev_grad_ptrs,
                    float* host_params_out, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return fail(h, SCAPE_ESTATE, "scape_step_host: call scape_bind first");
  if (!host_grads_src || !host_dev_grad_ptrs || !host_params_out)
    return fail(h, SCAPE_EINVAL, "scape_step_host: NULL pointer");
  for (int w = 0; w < h->W; ++w)
    if (!host_grads_src[w] || !host_dev_grad_ptrs[w])
      return fail(h, SCAPE_EINVAL, "scape_step_host: NULL gradient pointer");
  if (h->t >= 1 && !h->mask_ready)
    return fail(h, SCAPE_ESTATE, "scape_step_host: no mask yet; refresh after step 1");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t gbytes = (size_t)h->P * (h->dtype == SCAPE_BF16 ? 2 : 4);
  cudaError_t e = cudaSuccess;
  if (h->t == 0) {
    // dense first step: every worker is needed at once
    for (int w = 0; w < h->W && e == cudaSuccess; ++w)
      e = cudaMemcpyAsync(host_dev_grad_ptrs[w], host_grads_src[w], gbytes, cudaMemcpyHostToDevice,
                          st);
    if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: gradient upload");
    int rc = scape_step(h, reinterpret_cast<const void* const*>(host_dev_grad_ptrs), stream);
    if (rc) return rc;
    rc = scape_refresh_mask(h, stream);
    if (rc) return rc;
    e = cudaMemcpyAsync(host_params_out, h->w, (size_t)h->P * 4, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: parameter download");
    return SCAPE_OK;
  }
  {
    const int rc = ensure_aux(h);
    if (rc) return rc;
  }
  // Parameters: under the paper's reading a step changes w only at its k
  // selected coordinates, so the dense download of w runs first (the previous
  // parameters, on the second copy direction, while the gradients upload) and
  // the k new values are written into the host copy afterwards by a kernel,
  // through the page-locked buffer's device address.  Otherwise (pageable
  // output, or every coordinate updated) w is downloaded after the update.
  float* host_out_dev = nullptr;
  const bool patch = !(h->variant & SCAPE_VARIANT_DENSE_OFFMASK) &&
                     cudaHostGetDevicePointer(reinterpret_cast<void**>(&host_out_dev),
                                              host_params_out, 0) == cudaSuccess;
  if (!patch) (void)cudaGetLastError();  // not page-locked: clear the lookup's error
  // Worker groups: group g's uploads run on the copy stream while the
  // compaction of the groups before it runs on `stream`.
  const int G = h->W < scape_t::kMaxGroups ? h->W : scape_t::kMaxGroups;
  cudaStream_t cp = h->copy_stream, dn = h->down_stream;
  e = cudaEventRecord(h->ev_start, st);  // earlier users of the gradient and output buffers
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cp, h->ev_start, 0);
  if (e == cudaSuccess && patch) {
    e = cudaStreamWaitEvent(dn, h->ev_start, 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(host_params_out, h->w, (size_t)h->P * 4, cudaMemcpyDeviceToHost, dn);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_down, dn);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: parameter download");
  for (int g = 0; g < G && e == cudaSuccess; ++g) {
    for (int w = g * h->W / G; w < (g + 1) * h->W / G && e == cudaSuccess; ++w)
      e = cudaMemcpyAsync(host_dev_grad_ptrs[w], host_grads_src[w], gbytes, cudaMemcpyHostToDevice,
                          cp);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_group[g], cp);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: gradient upload");
  WorkerPtrs p;
  std::memset(&p, 0, sizeof p);
  bool vec = true;
  for (int w = 0; w < h->W; ++w) {
    p.g[w] = host_dev_grad_ptrs[w];
    p.e[w] = h->e[w];
    vec = vec && aligned16(host_dev_grad_ptrs[w]);
  }
  const int64_t t = h->t + 1;
  const AdamsConst c = make_const(h, t);
  for (int g = 0; g < G; ++g) {
    e = cudaStreamWaitEvent(st, h->ev_group[g], 0);
    // w changes from the last group on: the dense download must have read it
    if (e == cudaSuccess && patch && g == G - 1) e = cudaStreamWaitEvent(st, h->ev_down, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: stream wait");
    const int rc = enqueue_compact(h, p, g * h->W / G, (g + 1) * h->W / G, vec, c, st);
    if (rc) return rc;
  }
  int rc = enqueue_update(h, c, st);
  if (rc) return rc;
  h->t = t;
  h->buffers_valid = true;
  if (patch) {
    rc = run_kernel(h, kKParamPatch, st, [&] {
      return launch_param_patch(h->idx(), h->k, h->w, host_out_dev, st);
    });
    if (rc) return rc;
    return scape_refresh_mask(h, stream);
  }
  // the parameter download overlaps the mask refresh
  e = cudaEventRecord(h->ev_updated, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(dn, h->ev_updated, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(host_params_out, h->w, (size_t)h->P * 4, cudaMemcpyDeviceToHost, dn);
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_done, dn);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: parameter download");
  rc = scape_refresh_mask(h, stream);
  if (rc) return rc;
  e = cudaStreamWaitEvent(st, h->ev_done, 0);
  if (e != cudaSuccess) return cuda_fail(h, e, "scape_step_host: stream wait");
  return SCAPE_OK;
}

int scape_probe_random_access(scape_t* h, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound || !h->mask_ready)
    return fail(h, SCAPE_ESTATE, "scape_probe_random_access: needs a bound handle with a mask");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run_kernel(h, kKProbeRmw, st, [&] {
    return launch_probe_rmw(h->idx(), h->gbar(), h->k, h->w, h->m, st);
  });
}

int scape_profile_enable(scape_t* h, int on) {
  if (!h) return SCAPE_EINVAL;
  h->prof = on != 0;
  return SCAPE_OK;
}

int scape_profile_select(scape_t* h, uint32_t kernel_mask) {
  if (!h) return SCAPE_EINVAL;
  h->prof_mask = kernel_mask;
  return SCAPE_OK;
}

int scape_profile_collect(scape_t* h) {
  if (!h) return SCAPE_EINVAL;
  int rc = SCAPE_OK;
  for (auto& r : h->pending) {
    cudaError_t e = cudaEventSynchronize(r.b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) {
      rc = cuda_fail(h, e, "scape_profile_collect");
    } else {
      h->prof_ms[r.kid] += ms;
      h->prof_n[r.kid] += r.nlaunch;
    }
    h->pool.push_back(r.a);
    h->pool.push_back(r.b);
  }
  h->pending.clear();
  return rc;
}

int scape_profile_read(const scape_t* h, double* host_ms, int64_t* host_launches) {
  if (!h) return SCAPE_EINVAL;
  for (int i = 0; i < kNumKernels; ++i) {
    if (host_ms) host_ms[i] = h->prof_ms[i];
    if (host_launches) host_launches[i] = h->prof_n[i];
  }
  return SCAPE_OK;
}

int scape_profile_reset(scape_t* h) {
  if (!h) return SCAPE_EINVAL;
  for (int i = 0; i < kNumKernels; ++i) {
    h->prof_ms[i] = 0;
    h->prof_n[i] = 0;
  }
  return SCAPE_OK;
}

const char* scape_kernel_name(int i) {
  return (i >= 0 && i < kNumKernels) ? kKernelNames[i] : "";
}

int64_t scape_launch_count(const scape_t* h) { return h ? h->launches : -1; }

}  // extern "C"
