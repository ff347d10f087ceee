// step_kernels.cu -- the per-step kernels of the SCAPE optimizer step.
//
//   dense_step   step 1 (mask of all ones): error-feedback add, ordered mean
//                over workers, AdamS on every coordinate, residual <- 0.
//   ef_compact   error-feedback add + lagged-mask compaction + residual
//                ("SCAPE" Sec. II-B: sent = TopK(g + e) through the mask,
//                e <- g + e - sent), one pass over every worker's g and e.
//                It can also form the ordered sum of the packed values
//                (g_bar; done by default) and apply AdamS at the selected
//                coordinates (EfFuse flags; by default from 5% density).
//   reduce       ordered sum of the W packed buffers / W: the single
//                synchronised sparse buffer ("Sintesi Tecnica: SCAPE" Sec. 2)
//                (separate-launch form, and the union-mask baseline).
//   adams_sparse unpack + AdamS ("SCAPE" Sec. II-C, Eq. 2) at the k selected
//                coordinates, m and v both from that one buffer.
#include "scape_internal.cuh"

namespace scapek {
namespace {

template <typename GT>
struct GradIO;

template <>
struct GradIO<float> {
  // 8 consecutive gradients as loaded (kept packed until used)
  struct Raw {
    float4 a, b;
  };
  static __device__ __forceinline__ Raw load_raw(const void* base, int64_t i0) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i0);
    return Raw{__ldcs(p), __ldcs(p + 1)};
  }
  static __device__ __forceinline__ float at(const Raw& r, int j) {
    const float4& v = j < 4 ? r.a : r.b;
    const int q = j & 3;
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
  }
  // 8 consecutive gradients starting at a 32-byte multiple of the base.
  static __device__ __forceinline__ void load8(const void* base, int64_t i0, float (&g)[8]) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i0);
    float4 a = __ldcs(p), b = __ldcs(p + 1);
    g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
    g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
  }
  static __device__ __forceinline__ float load1(const void* base, int64_t i) {
    return __ldcs(static_cast<const float*>(base) + i);
  }
};

template <>
struct GradIO<__nv_bfloat16> {
  // 8 bfloat16 gradients in four 32-bit words, widened only when used
  using Raw = uint4;
  static __device__ __forceinline__ Raw load_raw(const void* base, int64_t i0) {
    return __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + i0));
  }
  static __device__ __forceinline__ float at(const Raw& r, int j) {
    const uint32_t u = (j >> 1) == 0 ? r.x : (j >> 1) == 1 ? r.y : (j >> 1) == 2 ? r.z : r.w;
    // bfloat16 is the high half of a binary32: widening is exact.
    return __uint_as_float((j & 1) ? (u & 0xFFFF0000u) : (u << 16));
  }
  static __device__ __forceinline__ void load8(const void* base, int64_t i0, float (&g)[8]) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + i0);
    uint4 v = __ldcs(p);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // bfloat16 is the high half of a binary32: widening is exact.
      g[2 * q] = __uint_as_float(u[q] << 16);
      g[2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ float load1(const void* base, int64_t i) {
    const unsigned short h =
        __ldcs(reinterpret_cast<const unsigned short*>(static_cast<const __nv_bfloat16*>(base) + i));
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
};

__device__ __forceinline__ void load8_f32(const float* p, float (&x)[8]) {
  const float4* q = reinterpret_cast<const float4*>(p);
  float4 a = __ldcs(q), b = __ldcs(q + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void store8_f32(float* p, const float (&x)[8]) {
  float4* q = reinterpret_cast<float4*>(p);
  __stcs(q, make_float4(x[0], x[1], x[2], x[3]));
  __stcs(q + 1, make_float4(x[4], x[5], x[6], x[7]));
}

// ------------------------------------------------------------------ ef_compact
// One block per 2048-parameter tile; each thread owns 8 consecutive parameters
// (one byte of the mask bitmap).  The rank of every selected parameter in the
// packed buffers is the tile's base (from the refresh's rank table) plus the
// block-exclusive popcount prefix, computed once and reused for all W workers.
// Workers whose loads are issued together, and resident blocks per SM (64
// registers): measured best of {1,2,4} x {2,3,4} on GB300 (6.70 TB/s).
//
// Because one block sees every worker of its tile, the synchronised buffer's
// sum can be formed here, in worker order, while the workers stream through:
// each selected slot's running sum sits in shared memory (owned by the thread
// of that slot), and after the last worker the same thread divides by W and
// writes g_bar, and can apply AdamS to its selected coordinates (EfFuse
// flags; w and m at those coordinates are fetched into shared memory by
// cp.async at the block's start).  The packed buffers are still written: they
// are what each worker sends.
constexpr int kWorkerUnroll = 2;
// bfloat16, up to kEfPrefetchMaxW workers: each worker group first asks L2 for
// the next group's rows of the tile (prefetch, no registers held), so that
// their loads wait on L2 rather than on DRAM.  Measured on one box, A/B:
// Llama-1.8B (W = 8) 15.55 against 15.77 ms per launch, GPT-345M (W = 8,
// update inside) 4.95 against 4.98 ms; Llama-500M (W = 32) 26.53 against
// 26.50 ms, so not with many workers.
constexpr int kEfPrefetchMaxW = 16;
constexpr int kEfMinBlocks = 4;

// With MSYNC (first-moment buffer reading) a selected parameter is sent as
// b = b1 m_{t-1} + (1 - b1) a instead of a; the residual is the same.
// Every selected value is also added to its slot's running sum (started at
// -0.0, the identity of IEEE addition, so the sum equals the worker-ordered
// sum that begins with worker 0's value).
// `full`: all eight parameters selected and their slots 16-byte aligned (in
// the packed row and in the running sums): the same values are then moved by
// vector loads and stores (the case of masks that keep most coordinates).
template <bool MSYNC, class G>
__device__ __forceinline__ void ef_select8(G&& g, const float (&e)[8], uint32_t byte, bool full,
                                           float* __restrict__ prow, float (&out)[8],
                                           const MomentPack& mp, int64_t i0, float* ssum) {
  if (full) {
    float4* p4 = reinterpret_cast<float4*>(prow);
    float4* s4 = reinterpret_cast<float4*>(ssum);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // four values at a time: fewer live registers
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = __fadd_rn(g(4 * h + j), e[4 * h + j]);  // error-feedback add
        v[j] = a;
        if (MSYNC)
          v[j] = __fadd_rn(__fmul_rn(mp.beta1, mp.m[i0 + 4 * h + j]), __fmul_rn(mp.c1, a));
        out[4 * h + j] = __fsub_rn(a, a);  // residual: everything was sent
      }
      p4[h] = make_float4(v[0], v[1], v[2], v[3]);
      float4 sv = s4[h];
      sv.x = __fadd_rn(sv.x, v[0]);
      sv.y = __fadd_rn(sv.y, v[1]);
      sv.z = __fadd_rn(sv.z, v[2]);
      sv.w = __fadd_rn(sv.w, v[3]);
      s4[h] = sv;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float a = __fadd_rn(g(j), e[j]);  // error-feedback add
    float sent = 0.f;
    if ((byte >> j) & 1u) {
      sent = a;
      float val = a;
      if (MSYNC) val = __fadd_rn(__fmul_rn(mp.beta1, mp.m[i0 + j]), __fmul_rn(mp.c1, a));
      const int r = __popc(byte & ((1u << j) - 1u));
      prow[r] = val;
      ssum[r] = __fadd_rn(ssum[r], val);
    }
    out[j] = __fsub_rn(a, sent);  // residual: g + e - sent
  }
}

// 4-byte global -> shared copy that completes in the background (cp.async);
// the issuing thread waits for its own copies with cp_async_wait<n>.
__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename GT, bool VEC, bool MSYNC, bool HOIST>
__global__ void __launch_bounds__(kTileThreads, kEfMinBlocks)
ef_compact_kernel(const __grid_constant__ WorkerPtrs ptrs, int W, int64_t P,
                  const uint32_t* __restrict__ bits, const uint32_t* __restrict__ tile_base,
                  float* __restrict__ pack, int64_t pack_stride, MomentPack mp, EfFuse fz) {
  __shared__ uint32_t warp_tot[kTileThreads / 32];
  __shared__ __align__(16) float tile_sum[kTile];
  __shared__ float tile_w[kTile], tile_m[kTile];  // w, m at the selected slots (finishing launch)
  const int64_t tile = blockIdx.x;
  const int64_t i0 = tile * kTile + (int64_t)threadIdx.x * 8;
  // full tile with aligned buffers: 16-byte loads and stores, the loads of a
  // worker group issued before any of it is stored (float32 gradients: one
  // worker in flight, two would spill at 64 registers)
  constexpr int U = sizeof(GT) == 2 ? kWorkerUnroll : 1;
  const bool vec_tile = VEC && (tile + 1) * kTile <= P;
  typename GradIO<GT>::Raw g[U];
  float e[U][8];
  // HOIST (one or two workers: a block has little else to wait for): the
  // first group's values, which do not depend on the mask, are loaded before
  // the block's prologue (bitmap word, block scan, rank-table base), which
  // then runs under them.  With more workers the host picks the kernel
  // without it: its longer live ranges cost registers there.
  const bool hoist = HOIST && vec_tile;
  if (hoist) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u < W) {
        g[u] = GradIO<GT>::load_raw(ptrs.g[u], i0);
        load8_f32(ptrs.e[u] + i0, e[u]);
      }
    }
  }
  uint32_t byte = 0;
  if (i0 < P) byte = (__ldg(bits + (i0 >> 5)) >> (uint32_t)(i0 & 31)) & 0xFFu;
  uint32_t total;
  const uint32_t excl = block_exclusive_scan<kTileThreads>(__popc(byte), warp_tot, &total);
  const int64_t slot0 = (int64_t)__ldg(tile_base + tile) + excl;
  // every parameter of this thread selected, slots 16-byte aligned: vector
  // path (float32 gradients only: with bfloat16 ones two workers are in
  // flight and the extra registers would spill)
  const bool full =
      sizeof(GT) == 4 && byte == 0xFFu && ((slot0 | (int64_t)excl) & 3) == 0;
  float* const pbase = pack + slot0;
  // this thread's selected slots: tile_sum[excl .. excl + popc(byte))
  float* const ssum = tile_sum + excl;
  // Background copies, so that no load of the update waits at the block's end:
  // group 0 the partial sums of the previous worker group, group 1 w and m at
  // this thread's selected coordinates.
  if ((fz.flags & (kEfAccum | kEfResume)) == (kEfAccum | kEfResume)) {
    for (int r = 0; r < __popc(byte); ++r) cp_async4(ssum + r, fz.gbar + slot0 + r);
  } else {
    for (int r = 0; r < __popc(byte); ++r) ssum[r] = -0.0f;
  }
  cp_async_commit();
  if ((fz.flags & (kEfAccum | kEfFinish | kEfUpdate)) == (kEfAccum | kEfFinish | kEfUpdate)) {
    uint32_t rest = byte;
    for (int r = 0; rest != 0u; ++r, rest &= rest - 1u) {
      const int64_t i = i0 + (__ffs(rest) - 1);
      cp_async4(tile_w + excl + r, fz.w + i);
      cp_async4(tile_m + excl + r, fz.m + i);
    }
  }
  cp_async_commit();
  cp_async_wait<1>();  // the partial sums have landed

  if (vec_tile) {
    for (int w0 = 0; w0 < W; w0 += U) {
      if (!HOIST && sizeof(GT) == 2 && W <= kEfPrefetchMaxW && w0 + U < W) {
        // the next group's gradient and residual rows of this tile into L2,
        // one 128-byte line per thread
        constexpr int kLinesG = kTile * (int)sizeof(GT) / 128, kLinesE = kTile * 4 / 128;
        const int ln = (int)threadIdx.x;
        if (ln < U * (kLinesG + kLinesE)) {
          const int u = ln / (kLinesG + kLinesE), l = ln % (kLinesG + kLinesE);
          if (w0 + U + u < W) {
            const char* a =
                l < kLinesG
                    ? reinterpret_cast<const char*>(static_cast<const GT*>(ptrs.g[w0 + U + u]) +
                                                    tile * kTile) + 128 * l
                    : reinterpret_cast<const char*>(ptrs.e[w0 + U + u] + tile * kTile) +
                          128 * (l - kLinesG);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
          }
        }
      }
      if (w0 > 0 || !hoist) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (w0 + u < W) {
            g[u] = GradIO<GT>::load_raw(ptrs.g[w0 + u], i0);
            load8_f32(ptrs.e[w0 + u] + i0, e[u]);
          }
        }
      }

#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (w0 + u < W) {
          float out[8];
          const auto& gu = g[u];
          ef_select8<MSYNC>([&](int j) { return GradIO<GT>::at(gu, j); }, e[u], byte, full,
                            pbase + (int64_t)(w0 + u) * pack_stride, out, mp, i0, ssum);
          store8_f32(ptrs.e[w0 + u] + i0, out);
        }
      }
    }
  } else {
    // ragged last tile, or unaligned buffers: element by element
    for (int wk = 0; wk < W; ++wk) {
      float g[8], e[8], out[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool in = i0 + j < P;
        g[j] = in ? GradIO<GT>::load1(ptrs.g[wk], i0 + j) : 0.f;
        e[j] = in ? __ldcs(ptrs.e[wk] + i0 + j) : 0.f;
      }
      ef_select8<MSYNC>([&](int j) { return g[j]; }, e, byte, false,
                        pbase + (int64_t)wk * pack_stride,
                        out, mp, i0, ssum);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (i0 + j < P) __stcs(ptrs.e[wk] + i0 + j, out[j]);
    }
  }
  if (!(fz.flags & kEfAccum)) return;
  // g_bar = (((p_0 + p_1) + ...) + p_{W-1}) / W and AdamS at each selected
  // coordinate ("SCAPE" Sec. II-C, Eq. 2); or the partial sum for the next group
  const float fw = (float)fz.W_total;
  if (!(fz.flags & kEfUpdate)) {
    const bool fin = (fz.flags & kEfFinish) != 0;
    if (full) {
      // eight consecutive aligned slots: two 16-byte stores (else a warp's
      // stores would be 4 bytes at a 32-byte stride)
      const float4* s4 = reinterpret_cast<const float4*>(ssum);
      float4* g4 = reinterpret_cast<float4*>(fz.gbar + slot0);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 v = s4[h];
        if (fin) {
          v.x = __fdiv_rn(v.x, fw);
          v.y = __fdiv_rn(v.y, fw);
          v.z = __fdiv_rn(v.z, fw);
          v.w = __fdiv_rn(v.w, fw);
        }
        g4[h] = v;
      }
    } else {
      for (int r = 0; r < __popc(byte); ++r)
        fz.gbar[slot0 + r] = fin ? __fdiv_rn(ssum[r], fw) : ssum[r];
    }
    return;
  }
  cp_async_wait<0>();
  uint32_t rest = byte;
  for (int r = 0; rest != 0u; ++r, rest &= rest - 1u) {
    const float gm = __fdiv_rn(ssum[r], fw);
    fz.gbar[slot0 + r] = gm;
    float wv = tile_w[(ssum - tile_sum) + r], mv = tile_m[(ssum - tile_sum) + r];
    if (MSYNC) adams_update_from_moment(gm, wv, mv, fz.c);
    else adams_update(gm, wv, mv, fz.c);
    const int64_t i = i0 + (__ffs(rest) - 1);
    fz.w[i] = wv;
    fz.m[i] = mv;
  }
}

// ------------------------------------------------------------------ dense_step
// KIND == kDenseScape: SCAPE step 1.  Every coordinate is selected, so the
// synchronised buffer is the ordered mean of all a^w = g^w + e^w and the
// residuals become a - a.
// KIND == kDenseAdams / kDenseAdamW: the dense baselines the pages compare
// against, on the ordered mean of the g^w alone (no error feedback): AdamS
// ("SCAPE" Sec. II-C, Eq. 2) and AdamW (v an EMA of g^2, kept in `var`).
// KIND == kDenseScapeMoment: step 1 under the first-moment buffer reading (the
// workers send b = b1 m + (1 - b1) a; m_t is their mean).
constexpr int kDenseScape = 0, kDenseAdams = 1, kDenseAdamW = 2, kDenseScapeMoment = 3;

template <typename GT, bool VEC, int KIND>
__global__ void __launch_bounds__(256)
dense_step_kernel(const __grid_constant__ WorkerPtrs ptrs, int W, int64_t P,
                  float* __restrict__ wts, float* __restrict__ mom, float* __restrict__ var,
                  AdamsConst c) {
  constexpr bool EF = KIND == kDenseScape || KIND == kDenseScapeMoment;
  constexpr bool MOM = KIND == kDenseScapeMoment;
  const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i0 >= P) return;
  const bool full = VEC && (i0 + 8 <= P);
  const int n = full ? 8 : (int)(P - i0 < 8 ? P - i0 : 8);
  float sum[8], m0[8];
  if (MOM)
    for (int j = 0; j < 8; ++j) m0[j] = j < n ? mom[i0 + j] : 0.f;
  for (int wk = 0; wk < W; ++wk) {
    float g[8], e[8], z[8];
    if (full) {
      GradIO<GT>::load8(ptrs.g[wk], i0, g);
      if (EF) load8_f32(ptrs.e[wk] + i0, e);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g[j] = j < n ? GradIO<GT>::load1(ptrs.g[wk], i0 + j) : 0.f;
        e[j] = (EF && j < n) ? ptrs.e[wk][i0 + j] : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float a = EF ? __fadd_rn(g[j], e[j]) : g[j];
      const float b = MOM ? __fadd_rn(__fmul_rn(c.beta1, m0[j]), __fmul_rn(c.one_minus_b1, a)) : a;
      sum[j] = (wk == 0) ? b : __fadd_rn(sum[j], b);
      z[j] = __fsub_rn(a, a);
    }
    if (EF) {
      if (full) {
        store8_f32(ptrs.e[wk] + i0, z);
      } else {
        for (int j = 0; j < n; ++j) ptrs.e[wk][i0 + j] = z[j];
      }
    }
  }
  const float fw = (float)W;
  for (int j = 0; j < n; ++j) {
    const float gm = __fdiv_rn(sum[j], fw);
    float wv = wts[i0 + j], mv = mom[i0 + j];
    if (KIND == kDenseAdamW) {
      float vv = var[i0 + j];
      adamw_update(gm, wv, mv, vv, c);
      var[i0 + j] = vv;
    } else if (MOM) {
      adams_update_from_moment(gm, wv, mv, c);
    } else {
      adams_update(gm, wv, mv, c);
    }
    wts[i0 + j] = wv;
    mom[i0 + j] = mv;
  }
}

// ------------------------------------------------------------------ offmask
// Dense off-mask reading: every unselected coordinate takes the AdamS update
// with a zero synchronised gradient.  4 parameters per thread.
__global__ void __launch_bounds__(256)
offmask_kernel(const uint32_t* __restrict__ bits, int64_t P, float* __restrict__ wts,
               float* __restrict__ mom, AdamsConst c) {
  const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i0 >= P) return;
  const uint32_t nib = (__ldg(bits + (i0 >> 5)) >> (uint32_t)(i0 & 31)) & 0xFu;
  if (nib == 0xFu) return;  // all four selected: already updated
  for (int j = 0; j < 4 && i0 + j < P; ++j) {
    if ((nib >> j) & 1u) continue;
    float wv = wts[i0 + j], mv = mom[i0 + j];
    adams_update(0.0f, wv, mv, c);
    wts[i0 + j] = wv;
    mom[i0 + j] = mv;
  }
}

// ------------------------------------------------------------------ reduce
// g_bar[j] = (((p_0 + p_1) + p_2) + ... + p_{W-1}) / W, 4 slots per thread.
__global__ void __launch_bounds__(256)
reduce_kernel(const float* __restrict__ pack, int64_t stride, int W, int64_t k,
              float* __restrict__ gbar) {
  const int64_t j0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (j0 >= k) return;
  const float fw = (float)W;
  if (j0 + 4 <= k) {
    float4 s = __ldg(reinterpret_cast<const float4*>(pack + j0));
#pragma unroll 8
    for (int wk = 1; wk < W; ++wk) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(pack + (int64_t)wk * stride + j0));
      s.x = __fadd_rn(s.x, v.x);
      s.y = __fadd_rn(s.y, v.y);
      s.z = __fadd_rn(s.z, v.z);
      s.w = __fadd_rn(s.w, v.w);
    }
    *reinterpret_cast<float4*>(gbar + j0) =
        make_float4(__fdiv_rn(s.x, fw), __fdiv_rn(s.y, fw), __fdiv_rn(s.z, fw), __fdiv_rn(s.w, fw));
  } else {
    for (int64_t j = j0; j < k; ++j) {
      float s = pack[j];
      for (int wk = 1; wk < W; ++wk) s = __fadd_rn(s, pack[(int64_t)wk * stride + j]);
      gbar[j] = __fdiv_rn(s, fw);
    }
  }
}

// ------------------------------------------------------------------ adams_sparse
// For the k selected coordinates i = idx[j]: AdamS with g = g_bar[j]; with
// MSYNC the buffer holds the synchronised first moment instead (m_t = b_bar,
// g recovered from it for the second moment).
template <bool MSYNC>
__device__ __forceinline__ void sparse_update(float b, float& w, float& m, const AdamsConst& c) {
  if (MSYNC) adams_update_from_moment(b, w, m, c);
  else adams_update(b, w, m, c);
}

// Slots of a 256-thread block: 256 kUpdSlots consecutive ones; thread t takes
// slots t, t + 256, ... of them, so that each load instruction of a warp
// covers 32 consecutive slots (neighbouring coordinates).  Measured on the
// Llama-500M shape: 4 consecutive slots per thread by 16-byte loads of idx
// and g_bar 0.55 ms, 4 slots 256 apart 0.49 ms on the same box; on another,
// 1, 2, 4 and 8 slots 256 apart 0.409, 0.402, 0.421 and 0.432 ms (Llama-1.8B:
// 0.973, 0.951, 0.996, 1.012 ms).
constexpr int kUpdSlots = 2;  // slots per thread

template <bool MSYNC>
__global__ void __launch_bounds__(256)
adams_sparse_kernel(const uint32_t* __restrict__ idx, const float* __restrict__ gbar, int64_t k,
                    float* __restrict__ wts, float* __restrict__ mom, AdamsConst c) {
  const int64_t j0 = (int64_t)blockIdx.x * (256 * kUpdSlots) + threadIdx.x;
  uint32_t ii[kUpdSlots];
  float gg[kUpdSlots], wv[kUpdSlots], mv[kUpdSlots];
#pragma unroll
  for (int q = 0; q < kUpdSlots; ++q) {
    const int64_t j = j0 + 256 * q;
    ii[q] = j < k ? __ldg(idx + j) : 0u;
    gg[q] = j < k ? __ldg(gbar + j) : 0.f;
  }
#pragma unroll
  for (int q = 0; q < kUpdSlots; ++q) {
    if (j0 + 256 * q < k) {
      wv[q] = wts[ii[q]];
      mv[q] = mom[ii[q]];
    }
  }
#pragma unroll
  for (int q = 0; q < kUpdSlots; ++q) {
    if (j0 + 256 * q < k) {
      sparse_update<MSYNC>(gg[q], wv[q], mv[q], c);
      wts[ii[q]] = wv[q];
      mom[ii[q]] = mv[q];
    }
  }
}

// ------------------------------------------------------------------ probe_rmw
// A timing probe of the machine, not part of the method: the memory accesses
// of adams_sparse with none of its arithmetic -- idx and g_bar read in
// order, w[i] and m[i] read and written back unchanged at the k selected
// coordinates -- so that its time is the floor the scattered update can
// reach on this GPU.  The stores are inline PTX so that the compiler keeps
// them; the values written are the values read (bit for bit).
__device__ __forceinline__ void st_keep(float* p, float v) {
  asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__global__ void __launch_bounds__(256)
probe_rmw_kernel(const uint32_t* __restrict__ idx, const float* __restrict__ gbar, int64_t k,
                 float* __restrict__ wts, float* __restrict__ mom) {
  // the same slots per thread and the same loads as adams_sparse
  const int64_t j0 = (int64_t)blockIdx.x * (256 * kUpdSlots) + threadIdx.x;
  uint32_t ii[kUpdSlots];
  float wv[kUpdSlots], mv[kUpdSlots], gsum = 0.f;
#pragma unroll
  for (int q = 0; q < kUpdSlots; ++q) {
    const int64_t j = j0 + 256 * q;
    ii[q] = j < k ? __ldg(idx + j) : 0u;
    gsum += j < k ? __ldg(gbar + j) : 0.f;
  }
  if (gsum == 1.0e30f) asm volatile("" ::: "memory");  // keep g_bar's loads
#pragma unroll
  for (int q = 0; q < kUpdSlots; ++q) {
    if (j0 + 256 * q < k) {
      wv[q] = wts[ii[q]];
      mv[q] = mom[ii[q]];
    }
  }
#pragma unroll
  for (int q = 0; q < kUpdSlots; ++q) {
    if (j0 + 256 * q < k) {
      st_keep(wts + ii[q], wv[q]);
      st_keep(mom + ii[q], mv[q]);
    }
  }
}

// ------------------------------------------------------------------ param_patch
// dst[idx[j]] = w[idx[j]] for the k coordinates a step changed; dst is the
// device address of the caller's page-locked host copy of the parameters,
// whose other coordinates already hold the (unchanged) previous values.
__global__ void __launch_bounds__(256)
param_patch_kernel(const uint32_t* __restrict__ idx, int64_t k, const float* __restrict__ w,
                   float* __restrict__ dst) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const uint32_t i = __ldg(idx + j);
  dst[i] = __ldg(w + i);
}

// ------------------------------------------------------------------ exchange helpers
// Used by the multi-rank exchange (scape_xc.cu).
// AdamS on every coordinate of a range from the synchronised buffer of the
// dense first step: g_bar[i] is coordinate i's averaged gradient.
__global__ void __launch_bounds__(256)
adams_dense_kernel(const float* __restrict__ gbar, int64_t n, float* __restrict__ wts,
                   float* __restrict__ mom, AdamsConst c) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float wv = wts[i], mv = mom[i];
  adams_update(gbar[i], wv, mv, c);
  wts[i] = wv;
  mom[i] = mv;
}

// dst[j] = src[idx[j]] (gather) or dst[idx[j]] = src[j] (scatter), j < k.
template <bool SCATTER>
__global__ void __launch_bounds__(256)
index_move_kernel(const uint32_t* __restrict__ idx, int64_t k, const float* __restrict__ src,
                  float* __restrict__ dst) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const uint32_t i = __ldg(idx + j);
  if (SCATTER) dst[i] = __ldg(src + j);
  else dst[j] = __ldg(src + i);
}

// A bitmap whose bit 0 is global parameter lo, re-aligned to the global word
// grid: out[j] holds global bits 32 (lo / 32 + j) .. + 31 of it (bits of the
// global word outside [lo, lo + n) are zero).  The source's bits past n are zero.
__global__ void __launch_bounds__(256)
align_bits_kernel(const uint32_t* __restrict__ local, int64_t n, int shift,
                  uint32_t* __restrict__ out, int64_t nw_out) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= nw_out) return;
  const int64_t nl = (n + 31) / 32;
  uint32_t v = j < nl ? (__ldg(local + j) << shift) : 0u;
  if (shift && j >= 1 && j - 1 < nl) v |= __ldg(local + j - 1) >> (32 - shift);
  out[j] = v;
}

// dst[j] |= src[j]: a rank's aligned mask words merged into the global bitmap
// (atomic: the first and last words are shared with the neighbouring ranks).
__global__ void __launch_bounds__(256)
or_words_kernel(const uint32_t* __restrict__ src, int64_t nw, uint32_t* __restrict__ dst) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= nw) return;
  const uint32_t v = __ldg(src + j);
  if (v) atomicOr(dst + j, v);
}

template <typename GT, int KIND>
void dense_kind(const WorkerPtrs& p, int W, int64_t P, bool vec, float* w, float* m, float* v,
                const AdamsConst& c, cudaStream_t st) {
  const int64_t threads = (P + 7) / 8;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  if (vec) dense_step_kernel<GT, true, KIND><<<grid, 256, 0, st>>>(p, W, P, w, m, v, c);
  else dense_step_kernel<GT, false, KIND><<<grid, 256, 0, st>>>(p, W, P, w, m, v, c);
}

template <typename GT, bool MSYNC>
void compact_kind(const WorkerPtrs& p, int W, int64_t P, bool vec, const uint32_t* bits,
                  const uint32_t* tile_base, float* pack, int64_t pack_stride,
                  const MomentPack& mp, const EfFuse& fz, cudaStream_t st) {
  const unsigned grid = (unsigned)((P + kTile - 1) / kTile);
  if (vec && W <= 2)
    ef_compact_kernel<GT, true, MSYNC, true>
        <<<grid, kTileThreads, 0, st>>>(p, W, P, bits, tile_base, pack, pack_stride, mp, fz);
  else if (vec)
    ef_compact_kernel<GT, true, MSYNC, false>
        <<<grid, kTileThreads, 0, st>>>(p, W, P, bits, tile_base, pack, pack_stride, mp, fz);
  else
    ef_compact_kernel<GT, false, MSYNC, false>
        <<<grid, kTileThreads, 0, st>>>(p, W, P, bits, tile_base, pack, pack_stride, mp, fz);
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_dense_step(const WorkerPtrs& p, int W, int64_t P, int dtype, bool vec,
                              float* w, float* m, const AdamsConst& c, bool moment,
                              cudaStream_t st) {
  if (dtype == SCAPE_BF16) {
    if (moment) dense_kind<__nv_bfloat16, kDenseScapeMoment>(p, W, P, vec, w, m, nullptr, c, st);
    else dense_kind<__nv_bfloat16, kDenseScape>(p, W, P, vec, w, m, nullptr, c, st);
  } else {
    if (moment) dense_kind<float, kDenseScapeMoment>(p, W, P, vec, w, m, nullptr, c, st);
    else dense_kind<float, kDenseScape>(p, W, P, vec, w, m, nullptr, c, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_dense_baseline(bool adamw, const WorkerPtrs& p, int W, int64_t P, int dtype,
                                  bool vec, float* w, float* m, float* v, const AdamsConst& c,
                                  cudaStream_t st) {
  if (dtype == SCAPE_BF16) {
    if (adamw) dense_kind<__nv_bfloat16, kDenseAdamW>(p, W, P, vec, w, m, v, c, st);
    else dense_kind<__nv_bfloat16, kDenseAdams>(p, W, P, vec, w, m, v, c, st);
  } else {
    if (adamw) dense_kind<float, kDenseAdamW>(p, W, P, vec, w, m, v, c, st);
    else dense_kind<float, kDenseAdams>(p, W, P, vec, w, m, v, c, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_ef_compact(const WorkerPtrs& p, int W, int64_t P, int dtype, bool vec,
                              const uint32_t* bits, const uint32_t* tile_base, float* pack,
                              int64_t pack_stride, const MomentPack* mp, const EfFuse& fz,
                              cudaStream_t st) {
  const MomentPack none{nullptr, 0.f, 0.f};
  if (dtype == SCAPE_BF16) {
    if (mp) compact_kind<__nv_bfloat16, true>(p, W, P, vec, bits, tile_base, pack, pack_stride, *mp, fz, st);
    else compact_kind<__nv_bfloat16, false>(p, W, P, vec, bits, tile_base, pack, pack_stride, none, fz, st);
  } else {
    if (mp) compact_kind<float, true>(p, W, P, vec, bits, tile_base, pack, pack_stride, *mp, fz, st);
    else compact_kind<float, false>(p, W, P, vec, bits, tile_base, pack, pack_stride, none, fz, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce(const float* pack, int64_t pack_stride, int W, int64_t k, float* gbar,
                          cudaStream_t st) {
  if (k <= 0) return cudaSuccess;
  const int64_t threads = (k + 3) / 4;
  reduce_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(pack, pack_stride, W, k, gbar);
  return cudaGetLastError();
}

cudaError_t launch_adams_sparse(const uint32_t* idx, const float* gbar, int64_t k, float* w,
                                float* m, const AdamsConst& c, bool msync, cudaStream_t st) {
  if (k <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((k + 256 * kUpdSlots - 1) / (256 * kUpdSlots));
  if (msync) adams_sparse_kernel<true><<<grid, 256, 0, st>>>(idx, gbar, k, w, m, c);
  else adams_sparse_kernel<false><<<grid, 256, 0, st>>>(idx, gbar, k, w, m, c);
  return cudaGetLastError();
}

cudaError_t launch_probe_rmw(const uint32_t* idx, const float* gbar, int64_t k, float* w,
                             float* m, cudaStream_t st) {
  if (k <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((k + 256 * kUpdSlots - 1) / (256 * kUpdSlots));
  probe_rmw_kernel<<<grid, 256, 0, st>>>(idx, gbar, k, w, m);
  return cudaGetLastError();
}

cudaError_t launch_param_patch(const uint32_t* idx, int64_t k, const float* w, float* dst,
                               cudaStream_t st) {
  if (k <= 0) return cudaSuccess;
  param_patch_kernel<<<(unsigned)((k + 255) / 256), 256, 0, st>>>(idx, k, w, dst);
  return cudaGetLastError();
}

cudaError_t launch_adams_dense(const float* gbar, int64_t n, float* w, float* m,
                               const AdamsConst& c, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  adams_dense_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(gbar, n, w, m, c);
  return cudaGetLastError();
}

cudaError_t launch_index_move(bool scatter, const uint32_t* idx, int64_t k, const float* src,
                              float* dst, cudaStream_t st) {
  if (k <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((k + 255) / 256);
  if (scatter) index_move_kernel<true><<<grid, 256, 0, st>>>(idx, k, src, dst);
  else index_move_kernel<false><<<grid, 256, 0, st>>>(idx, k, src, dst);
  return cudaGetLastError();
}

cudaError_t launch_align_bits(const uint32_t* local, int64_t n, int shift, uint32_t* out,
                              int64_t nw_out, cudaStream_t st) {
  if (nw_out <= 0) return cudaSuccess;
  align_bits_kernel<<<(unsigned)((nw_out + 255) / 256), 256, 0, st>>>(local, n, shift, out,
                                                                      nw_out);
  return cudaGetLastError();
}

cudaError_t launch_or_words(const uint32_t* src, int64_t nw, uint32_t* dst, cudaStream_t st) {
  if (nw <= 0) return cudaSuccess;
  or_words_kernel<<<(unsigned)((nw + 255) / 256), 256, 0, st>>>(src, nw, dst);
  return cudaGetLastError();
}

cudaError_t launch_offmask(const uint32_t* bits, int64_t P, float* w, float* m, const AdamsConst& c,
                           cudaStream_t st) {
  const int64_t threads = (P + 3) / 4;
  offmask_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(bits, P, w, m, c);
  return cudaGetLastError();
}

}  // namespace scapek
