// scape_xc.cu -- SCAPE over several data-parallel ranks with a real exchange
// (the scape_xc_* entry points of include/scape.h).
//
// Rank r of G owns the workers and the optimizer shards [a_r, b_r) of W (one
// shard per worker, "SCAPE" Sec. II-A: the distributed optimizer partitions
// states and parameters evenly over the workers).  It holds the full
// parameters w[P] (a replica), its own shards' first moment m[lo_r, hi_r), and
// the full-length residual and gradient of each of its workers.  A step is
// split around the three collectives the caller issues between the calls:
//   pack     error feedback + compaction of the local workers with the global
//            (lagged) mask into the packed rows, re-laid out as one block per
//            owner rank                                   ("SCAPE" Sec. II-B)
//   -- all-to-all: each owner receives the W workers' values of its shards
//      (the sparse reduce-scatter of "SCAPE" Sec. I, with the sum done by the
//      owner in worker order, so that results do not depend on the number of
//      ranks)
//   update   ordered mean of the W received rows, AdamS at the owned selected
//            coordinates ("SCAPE" Sec. II-C, Eq. 2; "Sintesi Tecnica: SCAPE"
//            Sec. 2, single synchronised buffer), the updated values gathered
//            for the parameter all-gather
//   -- all-gather of the updated parameters (sparse model reconstruction,
//      "SCAPE" Sec. I)
//   refresh  top-k of the owned shards' first moment (the next step's mask
//            for them, "Sintesi Tecnica: SCAPE" Sec. 2 partitioned mask),
//            aligned to the global word grid for the mask all-gather
//   -- all-gather of the mask words (overlaps the parameter all-gather: the
//      one-step lag means nothing of this step waits for it)
//   finish   the other ranks' updated parameters written into w; the mask
//            words merged into the global bitmap, whose rank table and index
//            list the next step's compaction uses.
// Step 1 is dense (every coordinate sent), as on one device.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "scape_handle.cuh"

using namespace scapek;
using namespace scapek::host;

struct scape_xc {
  // global layout
  int64_t P = 0;
  int W = 0, G = 0, rank = 0;
  int dtype = SCAPE_BF16;
  std::vector<int64_t> start, ks;  // W + 1 shard boundaries, W k_s
  int64_t k = 0, ntiles = 0, nwords = 0, kstride = 0;
  // per rank q: worker/shard range [sa[q], sa[q+1]), parameter range, k_q,
  // first selected column, mask words spanned
  std::vector<int> sa;
  std::vector<int64_t> lo, hi, kq, kofs, wlo, nwq;
  int Wl = 0;                   // local workers
  int64_t pmax = 0, wmax = 0;   // per-rank strides of the gathered params / mask words
  scape_t* own = nullptr;       // range handle of the owned shards (refresh, state)
  // workspace offsets
  size_t off_bits = 0, off_tcnt = 0, off_tbase = 0, off_scan = 0, off_idx = 0, off_pack = 0,
         off_send = 0, off_recv = 0, off_gbar = 0, off_psend = 0, off_precv = 0, off_msend = 0,
         off_mrecv = 0, off_own = 0, ws_need = 0;
  // bound memory
  bool bound = false;
  float* w = nullptr;
  float* m_own = nullptr;
  std::vector<float*> e;
  char* ws = nullptr;
  // state
  int64_t t = 0;           // steps completed
  int phase = 0;           // 0 idle, 1 packed, 2 updated, 3 refreshed
  bool mask_ready = false;
  std::string err;

  template <class T>
  T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
  bool dense() const { return t == 0; }  // the step being taken is step 1
  int64_t cols(int q) const { return dense() ? hi[q] - lo[q] : kq[q]; }
  // row length of rank q's columns in the exchange buffers: a multiple of 4
  // floats, so that every row starts 16-byte aligned for the vector loads
  int64_t cpad(int q) const { return (cols(q) + 3) / 4 * 4; }
  int64_t col0(int q) const { return dense() ? lo[q] : kofs[q]; }
};

namespace {

thread_local std::string g_xc_create_error;

int xfail(scape_xc_t* h, int code, const std::string& msg) {
  if (h) h->err = msg;
  return code;
}

int xcuda(scape_xc_t* h, cudaError_t e, const char* what) {
  return xfail(h, SCAPE_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Bits [lo, lo + n) of a global bitmap moved to bit 0 of `local` (the inverse
// of the realignment of the owned shards' words in scape_xc_refresh); bits past
// lo + n are cleared.
__global__ void __launch_bounds__(256)
extract_bits_kernel(const uint32_t* __restrict__ global, int64_t nw_global, int64_t lo, int64_t n,
                    uint32_t* __restrict__ local) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= (n + 31) / 32) return;
  const int64_t w0 = lo / 32 + j;
  const int s = (int)(lo % 32);
  uint32_t v = __ldg(global + w0) >> s;
  if (s && w0 + 1 < nw_global) v |= __ldg(global + w0 + 1) << (32 - s);
  const int64_t rem = n - 32 * j;  // bits of this word inside [lo, lo + n)
  if (rem < 32) v &= (1u << rem) - 1u;
  local[j] = v;
}

// Rebuild the global rank table and index list from the global bitmap.
int rebuild_global(scape_xc_t* h, cudaStream_t st) {
  scape_t* o = h->own;
  uint32_t* bits = h->at<uint32_t>(h->off_bits);
  uint32_t* tcnt = h->at<uint32_t>(h->off_tcnt);
  uint32_t* tbase = h->at<uint32_t>(h->off_tbase);
  int rc = run_kernel(o, kKTileCount, st, [&] { return launch_tile_count(bits, h->P, tcnt, st); });
  if (rc) return xfail(h, rc, o->err);
  rc = run_kernel(
      o, kKScan, st,
      [&] { return launch_scan(tcnt, h->ntiles, tbase, h->at<uint32_t>(h->off_scan), st); },
      kScanLaunches);
  if (rc) return xfail(h, rc, o->err);
  rc = run_kernel(o, kKIndex, st, [&] {
    return launch_index(bits, h->P, tbase, h->at<uint32_t>(h->off_idx), h->k, st);
  });
  return rc ? xfail(h, rc, o->err) : SCAPE_OK;
}

}  // namespace

extern "C" {

int scape_xc_create(scape_xc_t** out, int n_layers, const int64_t* host_layer_numel, int W, int G,
                    int rank, double sparsity, float beta1, float beta2, float lr, float eps,
                    float weight_decay, int grad_dtype) {
  g_xc_create_error.clear();
  if (!out) return SCAPE_EINVAL;
  *out = nullptr;
  if (G < 1 || G > W || rank < 0 || rank >= G) {
    g_xc_create_error = "need 1 <= G <= W and 0 <= rank < G";
    return SCAPE_EINVAL;
  }
  const int a = (int)((int64_t)W * rank / G), b = (int)((int64_t)W * (rank + 1) / G);
  scape_t* own = nullptr;
  int rc = scape_create_range(&own, n_layers, host_layer_numel, W, a, b, sparsity, beta1, beta2,
                              lr, eps, weight_decay, grad_dtype);
  if (rc) {
    g_xc_create_error = scape_last_error(nullptr);
    return rc;
  }
  scape_xc_t* h = new (std::nothrow) scape_xc_t();
  if (!h) {
    scape_destroy(own);
    g_xc_create_error = "out of host memory";
    return SCAPE_EINVAL;
  }
  h->own = own;
  h->P = own->P_global;
  h->W = W;
  h->G = G;
  h->rank = rank;
  h->dtype = grad_dtype;
  const int64_t P = h->P;
  h->start.resize(W + 1);
  h->ks.resize(W);
  for (int s = 0; s <= W; ++s) h->start[s] = (int64_t)s * P / W;
  for (int s = 0; s < W; ++s) {
    const int64_t n = h->start[s + 1] - h->start[s];
    h->ks[s] = (n * (1000000 - own->ppm) + 999999) / 1000000;
    h->k += h->ks[s];
  }
  h->sa.resize(G + 1);
  h->lo.resize(G);
  h->hi.resize(G);
  h->kq.resize(G);
  h->kofs.resize(G + 1);
  h->wlo.resize(G);
  h->nwq.resize(G);
  for (int q = 0; q <= G; ++q) h->sa[q] = (int)((int64_t)W * q / G);
  h->kofs[0] = 0;
  for (int q = 0; q < G; ++q) {
    h->lo[q] = h->start[h->sa[q]];
    h->hi[q] = h->start[h->sa[q + 1]];
    int64_t kk = 0;
    for (int s = h->sa[q]; s < h->sa[q + 1]; ++s) kk += h->ks[s];
    h->kq[q] = kk;
    h->kofs[q + 1] = h->kofs[q] + kk;
    h->wlo[q] = h->lo[q] / 32;
    h->nwq[q] = h->hi[q] > h->lo[q] ? (h->hi[q] + 31) / 32 - h->wlo[q] : 0;
    h->pmax = std::max(h->pmax, h->hi[q] - h->lo[q]);
    h->wmax = std::max(h->wmax, h->nwq[q]);
  }
  h->Wl = b - a;
  h->ntiles = (P + kTile - 1) / kTile;
  h->nwords = (P + 31) / 32;
  h->kstride = (int64_t)align_up((size_t)std::max<int64_t>(h->k, 1), 64);
  const int64_t n_own = h->hi[rank] - h->lo[rank];
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  h->off_bits = carve(align_up((size_t)h->nwords, 64) * 4);
  h->off_tcnt = carve((size_t)h->ntiles * 4);
  h->off_tbase = carve((size_t)(h->ntiles + 1) * 4);
  h->off_scan = carve((size_t)scan_scratch_words(h->ntiles) * 4);
  h->off_idx = carve((size_t)h->kstride * 4);
  h->off_pack = carve((size_t)h->Wl * h->kstride * 4);
  h->off_send = carve((size_t)h->Wl * (std::max<int64_t>(P, h->k) + 4 * G) * 4);
  h->off_recv = carve((size_t)W * ((n_own + 3) / 4 * 4) * 4);
  h->off_gbar = carve((size_t)std::max<int64_t>(n_own, 1) * 4);
  h->off_psend = carve((size_t)std::max<int64_t>(h->pmax, 1) * 4);
  h->off_precv = carve((size_t)G * std::max<int64_t>(h->pmax, 1) * 4);
  h->off_msend = carve((size_t)std::max<int64_t>(h->wmax, 1) * 4);
  h->off_mrecv = carve((size_t)G * std::max<int64_t>(h->wmax, 1) * 4);
  h->off_own = carve(own->ws_need);
  h->ws_need = off;
  *out = h;
  return SCAPE_OK;
}

void scape_xc_destroy(scape_xc_t* h) {
  if (!h) return;
  scape_destroy(h->own);
  delete h;
}

const char* scape_xc_last_error(const scape_xc_t* h) {
  return h ? h->err.c_str() : g_xc_create_error.c_str();
}

int scape_xc_layout(const scape_xc_t* h, int64_t* P, int64_t* k, int* local_workers,
                    int64_t* own_begin, int64_t* own_end, int64_t* own_k, size_t* ws_bytes) {
  if (!h) return SCAPE_EINVAL;
  if (P) *P = h->P;
  if (k) *k = h->k;
  if (local_workers) *local_workers = h->Wl;
  if (own_begin) *own_begin = h->lo[h->rank];
  if (own_end) *own_end = h->hi[h->rank];
  if (own_k) *own_k = h->kq[h->rank];
  if (ws_bytes) *ws_bytes = h->ws_need;
  return SCAPE_OK;
}

int scape_xc_bind(scape_xc_t* h, float* params, float* m_own, float* const* host_e_ptrs,
                  void* workspace, size_t ws_bytes) {
  if (!h) return SCAPE_EINVAL;
  if (!params || !m_own || !host_e_ptrs || !workspace)
    return xfail(h, SCAPE_EINVAL, "scape_xc_bind: NULL pointer");
  if (ws_bytes < h->ws_need || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return xfail(h, SCAPE_EINVAL, "scape_xc_bind: workspace too small or not 256-byte aligned");
  if (!aligned16(params) || !aligned16(m_own))
    return xfail(h, SCAPE_EINVAL, "scape_xc_bind: params and m must be 16-byte aligned");
  h->e.assign(h->Wl, nullptr);
  for (int w = 0; w < h->Wl; ++w) {
    if (!host_e_ptrs[w] || !aligned16(host_e_ptrs[w]))
      return xfail(h, SCAPE_EINVAL, "scape_xc_bind: residuals must be non-NULL, 16-byte aligned");
    h->e[w] = host_e_ptrs[w];
  }
  h->w = params;
  h->m_own = m_own;
  h->ws = static_cast<char*>(workspace);
  // the owned shards' handle works on w[lo, hi) of the replica and m_own; it
  // never runs a compaction, so its residual table is a placeholder
  scape_t* o = h->own;
  std::vector<float*> none(h->W, m_own);
  const int rc = scape_bind(o, m_own, m_own, none.data(), h->ws + h->off_own, o->ws_need);
  if (rc) return xfail(h, rc, o->err);
  o->w = params + h->lo[h->rank];
  h->bound = true;
  h->t = 0;
  h->phase = 0;
  h->mask_ready = false;
  return SCAPE_OK;
}

int scape_xc_counts(const scape_xc_t* h, int64_t* host_send_counts, int64_t* host_recv_counts,
                    int64_t* params_per_rank, int64_t* param_stride, int64_t* mask_words_per_rank,
                    int64_t* mask_stride) {
  if (!h) return SCAPE_EINVAL;
  const int r = h->rank;
  for (int q = 0; q < h->G; ++q) {
    if (host_send_counts) host_send_counts[q] = (int64_t)h->Wl * h->cpad(q);
    if (host_recv_counts) host_recv_counts[q] = (int64_t)(h->sa[q + 1] - h->sa[q]) * h->cpad(r);
    if (params_per_rank) params_per_rank[q] = h->cols(q);
    if (mask_words_per_rank) mask_words_per_rank[q] = h->nwq[q];
  }
  if (param_stride) *param_stride = std::max<int64_t>(h->pmax, 1);
  if (mask_stride) *mask_stride = std::max<int64_t>(h->wmax, 1);
  return SCAPE_OK;
}

int scape_xc_buffers(const scape_xc_t* h, float** send, float** recv, float** param_send,
                     float** param_recv, uint32_t** mask_send, uint32_t** mask_recv,
                     const uint32_t** global_bits) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return SCAPE_ESTATE;
  if (send) *send = h->at<float>(h->off_send);
  if (recv) *recv = h->at<float>(h->off_recv);
  if (param_send) *param_send = h->at<float>(h->off_psend);
  if (param_recv) *param_recv = h->at<float>(h->off_precv);
  if (mask_send) *mask_send = h->at<uint32_t>(h->off_msend);
  if (mask_recv) *mask_recv = h->at<uint32_t>(h->off_mrecv);
  if (global_bits) *global_bits = h->at<uint32_t>(h->off_bits);
  return SCAPE_OK;
}

int scape_xc_pack(scape_xc_t* h, const void* const* host_grad_ptrs, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return xfail(h, SCAPE_ESTATE, "scape_xc_pack: call scape_xc_bind first");
  if (h->phase != 0) return xfail(h, SCAPE_ESTATE, "scape_xc_pack: previous step not finished");
  if (h->t >= 1 && !h->mask_ready) return xfail(h, SCAPE_ESTATE, "scape_xc_pack: no mask");
  if (!host_grad_ptrs) return xfail(h, SCAPE_EINVAL, "scape_xc_pack: NULL gradient table");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  scape_t* o = h->own;
  WorkerPtrs p;
  std::memset(&p, 0, sizeof p);
  bool vec = true;
  for (int w = 0; w < h->Wl; ++w) {
    if (!host_grad_ptrs[w]) return xfail(h, SCAPE_EINVAL, "scape_xc_pack: NULL gradient pointer");
    p.g[w] = host_grad_ptrs[w];
    p.e[w] = h->e[w];
    vec = vec && aligned16(host_grad_ptrs[w]) && aligned16(h->e[w]);
  }
  uint32_t* bits = h->at<uint32_t>(h->off_bits);
  uint32_t* tbase = h->at<uint32_t>(h->off_tbase);
  float* send = h->at<float>(h->off_send);
  const EfFuse fz{nullptr, nullptr, nullptr, AdamsConst{}, h->W, 0};
  cudaError_t e = cudaSuccess;
  int rc = SCAPE_OK;
  if (h->dense()) {
    // Step 1 selects every coordinate.  Each destination's parameter range
    // is compacted on its own, straight into its block of the send buffer,
    // with an all-ones mask of the range's length (its rank table is the
    // identity: tile t starts at slot 2048 t).
    e = cudaMemsetAsync(bits, 0xFF, (size_t)h->nwords * 4, st);
    if (e != cudaSuccess) return xcuda(h, e, "scape_xc_pack: dense mask");
    rc = run_kernel(o, kKTileCount, st, [&] {
      return launch_tile_count(bits, (int64_t)h->nwords * 32, h->at<uint32_t>(h->off_tcnt), st);
    });
    if (rc == SCAPE_OK)
      rc = run_kernel(
          o, kKScan, st,
          [&] {
            return launch_scan(h->at<uint32_t>(h->off_tcnt), h->ntiles, tbase,
                               h->at<uint32_t>(h->off_scan), st);
          },
          kScanLaunches);
    if (rc) return xfail(h, rc, o->err);
    int64_t soff = 0;
    for (int q = 0; q < h->G; ++q) {
      const int64_t n = h->cols(q), lo = h->lo[q];
      if (n > 0 && h->Wl > 0) {
        // ones for bits [0, n), zeros after (bytes of the little-endian words)
        const size_t full = (size_t)(n / 8), tail_bits = (size_t)(n % 8);
        const size_t nbytes = (size_t)h->nwords * 4;
        e = cudaMemsetAsync(bits, 0xFF, full, st);
        if (e == cudaSuccess && full < nbytes)
          e = cudaMemsetAsync(reinterpret_cast<char*>(bits) + full,
                              (int)((1u << tail_bits) - 1u), 1, st);
        if (e == cudaSuccess && full + 1 < nbytes)
          e = cudaMemsetAsync(reinterpret_cast<char*>(bits) + full + 1, 0, nbytes - full - 1, st);
        if (e != cudaSuccess) return xcuda(h, e, "scape_xc_pack: dense range mask");
        WorkerPtrs pq;
        std::memset(&pq, 0, sizeof pq);
        bool vq = true;
        for (int w = 0; w < h->Wl; ++w) {
          const size_t gsz = h->dtype == SCAPE_BF16 ? 2 : 4;
          pq.g[w] = static_cast<const char*>(p.g[w]) + (size_t)lo * gsz;
          pq.e[w] = p.e[w] + lo;
          vq = vq && aligned16(pq.g[w]) && aligned16(pq.e[w]);
        }
        rc = run_kernel(o, kKEfCompact, st, [&] {
          return launch_ef_compact(pq, h->Wl, n, h->dtype, vq, bits, tbase, send + soff,
                                   h->cpad(q), nullptr, fz, st);
        });
        if (rc) return xfail(h, rc, o->err);
      }
      soff += (int64_t)h->Wl * h->cpad(q);
    }
    h->phase = 1;
    return SCAPE_OK;
  }
  // error feedback + compaction of the local workers: row w_l of `pack` holds
  // the selected a^w in global column order
  float* pack = h->at<float>(h->off_pack);
  rc = run_kernel(o, kKEfCompact, st, [&] {
    return launch_ef_compact(p, h->Wl, h->P, h->dtype, vec, bits, tbase, pack, h->kstride,
                             nullptr, fz, st);
  });
  if (rc) return xfail(h, rc, o->err);
  // one contiguous block per destination rank q: [local worker][its columns,
  // padded to cpad(q)]
  int64_t soff = 0;
  for (int q = 0; q < h->G && e == cudaSuccess; ++q) {
    const int64_t c = h->cols(q);
    if (c > 0 && h->Wl > 0)
      e = cudaMemcpy2DAsync(send + soff, (size_t)h->cpad(q) * 4, pack + h->col0(q),
                            (size_t)h->kstride * 4, (size_t)c * 4, (size_t)h->Wl,
                            cudaMemcpyDeviceToDevice, st);
    soff += (int64_t)h->Wl * h->cpad(q);
  }
  if (e != cudaSuccess) return xcuda(h, e, "scape_xc_pack: send layout");
  h->phase = 1;
  return SCAPE_OK;
}

int scape_xc_update(scape_xc_t* h, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (h->phase != 1) return xfail(h, SCAPE_ESTATE, "scape_xc_update: call scape_xc_pack first");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  scape_t* o = h->own;
  const int r = h->rank;
  const int64_t c = h->cols(r);
  const int64_t t = h->t + 1;
  const AdamsConst ac = make_const(o, t);
  float* gbar = h->at<float>(h->off_gbar);
  float* recv = h->at<float>(h->off_recv);
  float* psend = h->at<float>(h->off_psend);
  float* w_own = h->w + h->lo[r];
  // recv holds [worker 0 .. W-1][cpad]: the ordered sum over workers / W
  const int64_t cp = h->cpad(r);
  int rc = run_kernel(o, kKReduce, st, [&] { return launch_reduce(recv, cp, h->W, c, gbar, st); });
  if (rc) return xfail(h, rc, o->err);
  if (h->dense()) {
    rc = run_kernel(o, kKDenseUpdate, st,
                    [&] { return launch_adams_dense(gbar, c, w_own, h->m_own, ac, st); });
    if (rc) return xfail(h, rc, o->err);
    const cudaError_t e = c > 0 ? cudaMemcpyAsync(psend, w_own, (size_t)c * 4,
                                                  cudaMemcpyDeviceToDevice, st)
                                : cudaSuccess;
    if (e != cudaSuccess) return xcuda(h, e, "scape_xc_update: parameter copy");
  } else {
    // the owned shards' mask (local indices) is the one the compaction used
    rc = run_kernel(o, kKAdamsSparse, st, [&] {
      return launch_adams_sparse(o->idx(), gbar, c, w_own, h->m_own, ac, false, st);
    });
    if (rc) return xfail(h, rc, o->err);
    rc = run_kernel(o, kKXcMove, st,
                    [&] { return launch_index_move(false, o->idx(), c, w_own, psend, st); });
    if (rc) return xfail(h, rc, o->err);
  }
  h->phase = 2;
  return SCAPE_OK;
}

int scape_xc_refresh(scape_xc_t* h, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (h->phase != 2) return xfail(h, SCAPE_ESTATE, "scape_xc_refresh: call scape_xc_update first");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  scape_t* o = h->own;
  const int r = h->rank;
  o->t = h->t + 1;  // the owned shards' first moment is now m_t
  int rc = scape_refresh_mask(o, stream);
  if (rc) return xfail(h, rc, o->err);
  rc = run_kernel(o, kKXcMove, st, [&] {
    return launch_align_bits(o->bits(), h->hi[r] - h->lo[r], (int)(h->lo[r] % 32),
                             h->at<uint32_t>(h->off_msend), h->nwq[r], st);
  });
  if (rc) return xfail(h, rc, o->err);
  h->phase = 3;
  return SCAPE_OK;
}

int scape_xc_finish(scape_xc_t* h, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (h->phase != 3) return xfail(h, SCAPE_ESTATE, "scape_xc_finish: call scape_xc_refresh first");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  scape_t* o = h->own;
  const int64_t ps = std::max<int64_t>(h->pmax, 1), ms = std::max<int64_t>(h->wmax, 1);
  float* precv = h->at<float>(h->off_precv);
  uint32_t* mrecv = h->at<uint32_t>(h->off_mrecv);
  uint32_t* bits = h->at<uint32_t>(h->off_bits);
  // 1. the other owners' updated parameters, at the positions of the mask
  //    this step used (before the global mask is replaced)
  cudaError_t e = cudaSuccess;
  for (int q = 0; q < h->G; ++q) {
    if (q == h->rank) continue;
    const int64_t c = h->cols(q);
    if (c <= 0) continue;
    if (h->dense()) {
      e = cudaMemcpyAsync(h->w + h->lo[q], precv + q * ps, (size_t)c * 4,
                          cudaMemcpyDeviceToDevice, st);
      if (e != cudaSuccess) return xcuda(h, e, "scape_xc_finish: parameter copy");
    } else {
      const int rc = run_kernel(o, kKXcMove, st, [&] {
        return launch_index_move(true, h->at<uint32_t>(h->off_idx) + h->kofs[q], c,
                                 precv + q * ps, h->w, st);
      });
      if (rc) return xfail(h, rc, o->err);
    }
  }
  // 2. the next step's global mask from every owner's words
  e = cudaMemsetAsync(bits, 0, (size_t)h->nwords * 4, st);
  if (e != cudaSuccess) return xcuda(h, e, "scape_xc_finish: mask clear");
  for (int q = 0; q < h->G; ++q) {
    const int rc = run_kernel(o, kKXcMove, st, [&] {
      return launch_or_words(mrecv + q * ms, h->nwq[q], bits + h->wlo[q], st);
    });
    if (rc) return xfail(h, rc, o->err);
  }
  const int rc = rebuild_global(h, st);
  if (rc) return rc;
  h->t += 1;
  h->phase = 0;
  h->mask_ready = true;
  return SCAPE_OK;
}

int scape_xc_get_state(const scape_xc_t* h, int64_t* t, const uint32_t** own_bits,
                       const uint32_t** own_idx) {
  if (!h) return SCAPE_EINVAL;
  if (t) *t = h->t;
  if (own_bits) *own_bits = h->bound ? h->own->bits() : nullptr;
  if (own_idx) *own_idx = h->bound ? h->own->idx() : nullptr;
  return SCAPE_OK;
}

int scape_xc_set_state(scape_xc_t* h, int64_t t, const uint32_t* global_bits, void* stream) {
  if (!h) return SCAPE_EINVAL;
  if (!h->bound) return xfail(h, SCAPE_ESTATE, "scape_xc_set_state: call scape_xc_bind first");
  if (h->phase != 0) return xfail(h, SCAPE_ESTATE, "scape_xc_set_state: a step is in progress");
  if (t < 1 || !global_bits)
    return xfail(h, SCAPE_EINVAL, "scape_xc_set_state: need t >= 1 and a bitmap");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  scape_t* o = h->own;
  const int r = h->rank;
  const int64_t n = h->hi[r] - h->lo[r];
  // the owned shards' words, moved to bit 0, in the (idle) mask-gather buffer
  uint32_t* local = h->at<uint32_t>(h->off_mrecv);
  int rc = run_kernel(o, kKXcMove, st, [&] {
    extract_bits_kernel<<<(unsigned)(((n + 31) / 32 + 255) / 256), 256, 0, st>>>(
        global_bits, h->nwords, h->lo[r], n, local);
    return cudaGetLastError();
  });
  if (rc) return xfail(h, rc, o->err);
  // validates the owned shards' counts and rebuilds their rank table
  rc = scape_set_state(o, t, local, stream);
  if (rc) {
    h->mask_ready = false;
    return xfail(h, rc, o->err);
  }
  const cudaError_t e = cudaMemcpyAsync(h->at<uint32_t>(h->off_bits), global_bits,
                                        (size_t)h->nwords * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return xcuda(h, e, "scape_xc_set_state: copy");
  rc = rebuild_global(h, st);
  if (rc) return rc;
  h->t = t;
  h->mask_ready = true;
  return SCAPE_OK;
}

int64_t scape_xc_launch_count(const scape_xc_t* h) { return h ? h->own->launches : -1; }

}  // extern "C"
