// topk_kernels.cu -- exact per-shard top-k threshold of the mask refresh,
// resolved on a candidate list instead of repeated passes over m.
//
// Order: "larger |m| first, then lower index" ("Sintesi Tecnica: SCAPE" Sec. 2
// partitioned top-k on first-moment statistics; ties to the lower index).  It
// is the order of the 63-bit composite key
//     comp(i) = (bits(m_i) & 0x7FFFFFFF) << 32  |  (0xFFFFFFFF - i)
// which is distinct for every parameter, so the k_s-th largest composite of a
// shard fixes the selection exactly: i is selected iff comp(i) >= kstar64.
//
//   chist0    one read of m: per-shard histogram of composite bits 62..51
//             (the top 12 bits of |m|); stages candidates near last step's
//             bucket
//   cselect0  per shard: the bucket holding the k_s-th largest key
//   collect   second read of m, only for shards whose bucket moved: (key,
//             index) of every parameter in that bucket
//   chist/cselect 1..5   radix passes over the candidates only, digits
//             50..40, 39..29, 28..18, 17..7, 6..0 of the composite key
// The result is written as (kstar, istar) into the shard's ShardSel for the
// mark kernel: bit_i = key_i > kstar || (key_i == kstar && i <= istar).
#include "scape_internal.cuh"

namespace scapek {
namespace {

constexpr int kCBins0 = kCandBins0;  // 12-bit first digit

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t i) {
  return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - i);
}

// ------------------------------------------------------------------ passes over m
// One kernel for both reads of m.  Blocks are persistent: block b walks a
// contiguous run of 2048-parameter segments, following the shard boundaries
// incrementally, so it meets at most a few of them.  Per shard piece it
//   HIST:    adds the 12-bit first digit of every key to a shared-memory
//            histogram (flushed to the shard's row when the shard changes), and
//            stages candidates whose digit lies within one bucket of the
//            previous refresh's bucket (`guess`): the mask is stable from step
//            to step, so that bucket usually still holds the threshold;
//   COLLECT: (second pass, only for shards whose guess missed) stages every
//            parameter whose digit equals the bucket just selected.
// Each warp stages its candidates in a private shared-memory buffer (ballot
// append) and flushes it to the shard's range of `cand` with one global
// atomic, so segments need no block-wide barrier.
constexpr int kMSeg = 2048;       // parameters per segment (256 threads x 2 x float4)
constexpr int kWarpStage = 384;   // staged candidates per warp

template <bool HIST>
__global__ void __launch_bounds__(256)
mpass_kernel(const float* __restrict__ m, int64_t P, int W, const int64_t* __restrict__ shard_start,
             const ShardSel* __restrict__ sel, uint32_t* __restrict__ hist,
             uint2* __restrict__ cand, uint32_t* __restrict__ cand_cnt, int64_t segs_per_block) {
  __shared__ uint32_t sh[HIST ? kCBins0 : 1];
  __shared__ uint2 wbuf[8][kWarpStage];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nseg = (P + kMSeg - 1) / kMSeg;
  const int64_t g0 = (int64_t)blockIdx.x * segs_per_block;
  const int64_t g1 = min(g0 + segs_per_block, nseg);
  if (g0 >= g1) return;
  const int64_t r0 = g0 * kMSeg, r1 = min(g1 * kMSeg, P);
  int s = shard_of(r0, P, W);
  if (!HIST) {
    // nothing to do unless a shard of this block's range must be collected
    bool any = false;
    for (int q = s; q < W && __ldg(shard_start + q) < r1; ++q)
      any |= sel[q].mode == kSelSearch && (sel[q].flags & kSelNeedCollect);
    if (!any) return;
  }
  if (HIST) {
    for (int b = threadIdx.x; b < kCBins0; b += blockDim.x) sh[b] = 0;
    __syncthreads();
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint2* const mybuf = wbuf[warp];
  uint32_t wn = 0;  // entries in this warp's buffer (same value in every lane)

  auto flush_warp = [&](int shard) {
    if (wn == 0) return;
    __syncwarp();
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(cand_cnt + shard, wn);
    base = __shfl_sync(0xffffffffu, base, 0);
    uint2* out = cand + __ldg(shard_start + shard) + base;
    for (uint32_t j = lane; j < wn; j += 32) out[j] = mybuf[j];
    __syncwarp();
    wn = 0;
  };

  int64_t s_hi = __ldg(shard_start + s + 1);
  uint32_t wlo = 0xFFFFFFFFu, wwid = 0;  // window of digits: d - wlo <= wwid (unsigned)
  bool active = false;
  int cur = -1;
  for (int64_t g = g0; g < g1; ++g) {
    const int64_t seg0 = g * kMSeg;
    const int64_t seg1 = min(seg0 + (int64_t)kMSeg, P);
    for (;;) {
      while (seg0 >= s_hi && s < W - 1) s_hi = __ldg(shard_start + (++s) + 1);
      if (s != cur) {
        if (cur >= 0) {
          flush_warp(cur);
          if (HIST) {
            __syncthreads();
            uint32_t* row = hist + (int64_t)cur * kCBins0;
            for (int b = threadIdx.x; b < kCBins0; b += blockDim.x) {
              const uint32_t c = sh[b];
              if (c) {
                atomicAdd(row + b, c);
                sh[b] = 0;
              }
            }
            __syncthreads();
          }
        }
        cur = s;
        const ShardSel ss = sel[s];
        if (HIST) {
          active = true;
          wlo = 0xFFFFFFFFu;
          wwid = 0;
          if (ss.guess != kNoGuess) {
            wlo = ss.guess > 0 ? ss.guess - 1 : 0;
            wwid = ss.guess + 1 - wlo;
          }
        } else {
          active = ss.mode == kSelSearch && (ss.flags & kSelNeedCollect);
          wlo = (uint32_t)ss.cprefix;
          wwid = 0;
        }
      }
      const int64_t lo = max(seg0, __ldg(shard_start + s)), hi = min(seg1, s_hi);
      if (active && lo < hi) {
        if (lo == seg0 && hi - lo == kMSeg) {
          const float4* p4 = reinterpret_cast<const float4*>(m + seg0);
          float4 v[kMSeg / 4 / 256];
#pragma unroll
          for (int r = 0; r < kMSeg / 4 / 256; ++r) v[r] = __ldcs(p4 + threadIdx.x + 256 * r);
#pragma unroll
          for (int r = 0; r < kMSeg / 4 / 256; ++r) {
            const uint32_t i0 = (uint32_t)(seg0 + 4 * (threadIdx.x + 256 * r));
            const float x[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t key = magnitude_key(x[q]);
              const uint32_t d = key >> 19;
              if (HIST) atomicAdd(&sh[d], 1u);
              const bool hit = d - wlo <= wwid;
              const uint32_t ball = __ballot_sync(0xffffffffu, hit);
              if (ball) {
                if (hit) mybuf[wn + __popc(ball & lt_mask)] = make_uint2(key, i0 + q);
                wn += __popc(ball);
                if (wn > kWarpStage - 32) flush_warp(s);
              }
            }
          }
        } else {
          // shard piece: warp-uniform trip count so ballots see every lane
          for (int64_t b0 = lo; b0 < hi; b0 += 256) {
            const int64_t i = b0 + threadIdx.x;
            const bool in = i < hi;
            const uint32_t key = in ? magnitude_key(__ldcs(m + i)) : 0u;
            const uint32_t d = key >> 19;
            if (HIST && in) atomicAdd(&sh[d], 1u);
            const bool hit = in && d - wlo <= wwid;
            const uint32_t ball = __ballot_sync(0xffffffffu, hit);
            if (ball) {
              if (hit) mybuf[wn + __popc(ball & lt_mask)] = make_uint2(key, (uint32_t)i);
              wn += __popc(ball);
              if (wn > kWarpStage - 32) flush_warp(s);
            }
          }
        }
      }
      if (s_hi >= seg1 || s == W - 1) break;
      s_hi = __ldg(shard_start + (++s) + 1);
    }
  }
  if (cur >= 0) {
    flush_warp(cur);
    if (HIST) {
      __syncthreads();
      uint32_t* row = hist + (int64_t)cur * kCBins0;
      for (int b = threadIdx.x; b < kCBins0; b += blockDim.x) {
        const uint32_t c = sh[b];
        if (c) atomicAdd(row + b, c);
      }
    }
  }
}

// ------------------------------------------------------------------ cselect
// One block per shard: find the digit of the pass holding the krem-th largest
// composite among those matching the prefix, narrow the prefix, clear the row.
template <int PASS>
__global__ void __launch_bounds__(256)
cselect_kernel(const int64_t* __restrict__ shard_start, const int64_t* __restrict__ shard_k,
               ShardSel* __restrict__ sel, uint32_t* __restrict__ hist,
               uint32_t* __restrict__ cand_cnt) {
  constexpr int WID = PASS == 0 ? 12 : (PASS == 5 ? 7 : 11);
  constexpr int NB = 1 << WID;
  constexpr int PER = NB >= 256 ? NB / 256 : 1;
  __shared__ uint32_t warp_tot[8];
  __shared__ uint32_t sh_digit, sh_above;
  const int s = blockIdx.x;
  uint32_t* row = hist + (int64_t)s * kCBins0;
  const int64_t s_lo = shard_start[s], s_hi = shard_start[s + 1];
  ShardSel st;
  if (PASS == 0) {
    const int64_t n = s_hi - s_lo, k = shard_k[s];
    st.prefix = 0;
    st.krem = (uint32_t)k;
    st.kstar = 0;
    st.need = 0;
    st.count_eq = 0;
    st.istar = s_hi - 1;
    st.cprefix = 0;
    st.guess = sel[s].guess;
    st.flags = 0;
    if (n <= 0 || k <= 0) st.mode = kSelEmpty;
    else if (k >= n) st.mode = kSelDone;  // every key selected: kstar = 0, istar = last
    else st.mode = kSelSearch;
  } else {
    st = sel[s];
  }
  if (st.mode != kSelSearch) {
    __syncthreads();  // every thread has read sel[s] before thread 0 rewrites it
    if (threadIdx.x == 0 && PASS == 0) sel[s] = st;
    for (int b = threadIdx.x; b < kCBins0; b += blockDim.x) row[b] = 0;
    return;
  }
  if (threadIdx.x == 0) {
    sh_digit = 0;
    sh_above = 0;
  }
  // thread t owns bins [NB - PER*(t+1), NB - PER*t) when they exist: descending order
  uint32_t h[PER];
  uint32_t local = 0;
  const int top = NB - PER * (int)threadIdx.x - 1;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    h[q] = (top - q >= 0) ? row[top - q] : 0u;
    local += h[q];
  }
  uint32_t total;
  const uint32_t excl = block_exclusive_scan<256>(local, warp_tot, &total);
  if (excl < st.krem && st.krem <= excl + local) {
    uint32_t cum = excl;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      if (cum + h[q] >= st.krem) {
        sh_digit = (uint32_t)(top - q);
        sh_above = cum;
        break;
      }
      cum += h[q];
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kCBins0; b += blockDim.x) row[b] = 0;
  if (threadIdx.x == 0) {
    st.cprefix = (st.cprefix << WID) | sh_digit;
    st.krem -= sh_above;
    if (PASS == 0) {
      // candidates were staged during the histogram pass for buckets within
      // one of the previous refresh's; otherwise a collect pass gathers them
      const bool hit = st.guess != kNoGuess && sh_digit + 1 >= st.guess && sh_digit <= st.guess + 1;
      if (!hit) {
        cand_cnt[s] = 0;
        st.flags = kSelNeedCollect;
      }
    }
    if (PASS == 5) {
      // the composite of the k_s-th largest parameter of the shard
      st.guess = (uint32_t)(st.cprefix >> 51);
      st.kstar = (uint32_t)(st.cprefix >> 32);
      st.istar = (int64_t)(0xFFFFFFFFu - (uint32_t)(st.cprefix & 0xFFFFFFFFu));
      st.mode = kSelDone;
    }
    sel[s] = st;
  }
}

// ------------------------------------------------------------------ chist 1..5
// grid (G, W): blocks of shard s stride over its candidates, histogramming the
// pass's digit of the composite key among those matching the prefix.
template <int PASS>
__global__ void __launch_bounds__(256)
chist_kernel(const int64_t* __restrict__ shard_start, const ShardSel* __restrict__ sel,
             const uint2* __restrict__ cand, const uint32_t* __restrict__ cand_cnt,
             uint32_t* __restrict__ hist) {
  constexpr int WID = PASS == 5 ? 7 : 11;
  constexpr int NB = 1 << WID;
  constexpr int SHIFT = PASS == 1 ? 40 : PASS == 2 ? 29 : PASS == 3 ? 18 : PASS == 4 ? 7 : 0;
  __shared__ uint32_t sh[NB];
  const int s = blockIdx.y;
  if (sel[s].mode != kSelSearch) return;
  const uint64_t prefix = sel[s].cprefix;
  const uint32_t cnt = cand_cnt[s];
  const uint2* c = cand + shard_start[s];
  for (int b = threadIdx.x; b < NB; b += blockDim.x) sh[b] = 0;
  __syncthreads();
  for (uint32_t j = blockIdx.x * blockDim.x + threadIdx.x; j < cnt; j += gridDim.x * blockDim.x) {
    const uint2 v = __ldg(c + j);
    const uint64_t comp = composite(v.x, v.y);
    if ((comp >> (SHIFT + WID)) == prefix) atomicAdd(&sh[(uint32_t)(comp >> SHIFT) & (NB - 1)], 1u);
  }
  __syncthreads();
  uint32_t* row = hist + (int64_t)s * kCBins0;
  for (int b = threadIdx.x; b < NB; b += blockDim.x) {
    const uint32_t v = sh[b];
    if (v) atomicAdd(row + b, v);
  }
}

int mpass_grid(int64_t P, int64_t* segs_per_block) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      sms = n;
    else
      sms = 148;
  }
  const int64_t nseg = (P + kMSeg - 1) / kMSeg;
  const int64_t want = (int64_t)sms * 5;  // ~40 KB of shared memory per block: 5 per SM
  const int64_t grid = nseg < want ? nseg : want;
  *segs_per_block = (nseg + grid - 1) / grid;
  return (int)((nseg + *segs_per_block - 1) / *segs_per_block);
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_chist0(const float* m, int64_t P, int W, const int64_t* shard_start,
                          const ShardSel* sel, uint32_t* hist, uint2* cand, uint32_t* cand_cnt,
                          cudaStream_t st) {
  int64_t spb = 1;
  const int grid = mpass_grid(P, &spb);
  mpass_kernel<true><<<grid, 256, 0, st>>>(m, P, W, shard_start, sel, hist, cand, cand_cnt, spb);
  return cudaGetLastError();
}

cudaError_t launch_collect(const float* m, int64_t P, int W, const int64_t* shard_start,
                           const ShardSel* sel, uint2* cand, uint32_t* cand_cnt, cudaStream_t st) {
  int64_t spb = 1;
  const int grid = mpass_grid(P, &spb);
  mpass_kernel<false><<<grid, 256, 0, st>>>(m, P, W, shard_start, sel, nullptr, cand, cand_cnt,
                                            spb);
  return cudaGetLastError();
}

cudaError_t launch_cselect(int pass, int W, const int64_t* shard_start, const int64_t* shard_k,
                           ShardSel* sel, uint32_t* hist, uint32_t* cand_cnt, cudaStream_t st) {
  switch (pass) {
    case 0: cselect_kernel<0><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist, cand_cnt); break;
    case 1: cselect_kernel<1><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist, cand_cnt); break;
    case 2: cselect_kernel<2><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist, cand_cnt); break;
    case 3: cselect_kernel<3><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist, cand_cnt); break;
    case 4: cselect_kernel<4><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist, cand_cnt); break;
    default: cselect_kernel<5><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist, cand_cnt); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_chist(int pass, int W, int blocks_per_shard, const int64_t* shard_start,
                         const ShardSel* sel, const uint2* cand, const uint32_t* cand_cnt,
                         uint32_t* hist, cudaStream_t st) {
  dim3 grid((unsigned)blocks_per_shard, (unsigned)W);
  switch (pass) {
    case 1: chist_kernel<1><<<grid, 256, 0, st>>>(shard_start, sel, cand, cand_cnt, hist); break;
    case 2: chist_kernel<2><<<grid, 256, 0, st>>>(shard_start, sel, cand, cand_cnt, hist); break;
    case 3: chist_kernel<3><<<grid, 256, 0, st>>>(shard_start, sel, cand, cand_cnt, hist); break;
    case 4: chist_kernel<4><<<grid, 256, 0, st>>>(shard_start, sel, cand, cand_cnt, hist); break;
    default: chist_kernel<5><<<grid, 256, 0, st>>>(shard_start, sel, cand, cand_cnt, hist); break;
  }
  return cudaGetLastError();
}

}  // namespace scapek
