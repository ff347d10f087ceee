// refresh_kernels.cu -- partitioned top-k mask refresh of the SCAPE step:
// bitmap, rank table and index list.
//
// For every optimizer shard s independently ("Sintesi Tecnica: SCAPE" Sec. 2,
// partitioned mask synchronisation), the k_s parameters with the largest
// first-moment magnitude (key = bits(m) & 0x7FFFFFFF, so the order of the keys
// as unsigned integers is the order of |m|) are selected, equal keys going to
// the lower index.  The threshold (kstar, istar) comes from the candidate
// select of topk_kernels.cu; this file holds
//   mark      the bitmap elementwise, bit_i = key_i > kstar || (key_i == kstar
//             && i <= istar), with per-tile popcounts (or, in accumulate mode,
//             OR-ed into an existing bitmap) -- the first refresh, and the
//             union baseline;
//   remark    the same for the tiles a warm refresh's speculative bitmap does
//             not cover;
//   scan      per-tile counts -> rank table; index the ascending index list;
//   shard_count / tile_count   counts of a restored bitmap.
// It also keeps an exact select that works on m alone, for the allocation-free
// entry point (scape_static.cu), whose scratch cannot hold a candidate list:
//   hist<0>/select<0>   11-bit digit 30..20 of every key of the shard
//   hist<1>/select<1>   11-bit digit 19..9 of the keys matching the prefix
//   hist<2>/select<2>    9-bit digit  8..0 of the keys matching the prefix
// fix kstar and how many keys equal to it are selected (need); when fewer than
// all equal keys are selected, tie_count and tie_select find the index istar of
// the need-th equal key in index order.
#include "scape_internal.cuh"

namespace scapek {
namespace {


// ------------------------------------------------------------------ histograms
// One block per 4096-parameter segment of the flat vector.  A segment that
// straddles shard boundaries is processed one shard piece at a time.
template <int PASS>
__global__ void __launch_bounds__(256)
radix_hist_kernel(const float* __restrict__ m, int64_t P, ShardMap sm,
                  const int64_t* __restrict__ shard_start, const ShardSel* __restrict__ sel,
                  uint32_t* __restrict__ hist) {
  constexpr int NB = (PASS == 2) ? 512 : kBins;
  __shared__ uint32_t sh[NB];
  const int64_t seg0 = (int64_t)blockIdx.x * kSeg;
  const int64_t seg1 = min(seg0 + (int64_t)kSeg, P);
  const int W = sm.S;
  int s = sm.of(seg0);
  for (;;) {
    const int64_t s_lo = __ldg(shard_start + s), s_hi = __ldg(shard_start + s + 1);
    const int64_t lo = max(seg0, s_lo), hi = min(seg1, s_hi);
    const uint32_t mode = (PASS == 0) ? (uint32_t)kSelSearch : sel[s].mode;
    if (lo < hi && mode == kSelSearch) {
      const uint32_t prefix = (PASS == 0) ? 0u : sel[s].prefix;
      for (int b = threadIdx.x; b < NB; b += blockDim.x) sh[b] = 0;
      __syncthreads();
      if (lo == seg0 && hi - lo == kSeg) {
        // whole segment in one shard: 16-byte loads, four per thread
        const float4* p4 = reinterpret_cast<const float4*>(m + seg0);
        float4 v[kSeg / 4 / 256];
#pragma unroll
        for (int r = 0; r < kSeg / 4 / 256; ++r) v[r] = __ldcs(p4 + threadIdx.x + 256 * r);
#pragma unroll
        for (int r = 0; r < kSeg / 4 / 256; ++r) {
          const float x[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t key = magnitude_key(x[q]);
            if (PASS == 0) atomicAdd(&sh[key >> kShift0], 1u);
            if (PASS == 1 && (key >> kShift0) == prefix) atomicAdd(&sh[(key >> kShift1) & 0x7FFu], 1u);
            if (PASS == 2 && (key >> kShift1) == prefix) atomicAdd(&sh[key & 0x1FFu], 1u);
          }
        }
      } else {
        for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
          const uint32_t key = magnitude_key(__ldcs(m + i));
          if (PASS == 0) atomicAdd(&sh[key >> kShift0], 1u);
          if (PASS == 1 && (key >> kShift0) == prefix) atomicAdd(&sh[(key >> kShift1) & 0x7FFu], 1u);
          if (PASS == 2 && (key >> kShift1) == prefix) atomicAdd(&sh[key & 0x1FFu], 1u);
        }
      }
      __syncthreads();
      for (int b = threadIdx.x; b < NB; b += blockDim.x) {
        const uint32_t c = sh[b];
        if (c) atomicAdd(hist + (int64_t)s * kBins + b, c);
      }
      __syncthreads();
    }
    if (s_hi >= seg1 || s == W - 1) break;
    ++s;
  }
}

// ------------------------------------------------------------------ select
// One block (256 threads) per shard: find the digit holding the krem-th
// largest key among those matching the prefix, narrow the prefix, and clear
// the histogram row for the next pass.
template <int PASS>
__global__ void __launch_bounds__(256)
radix_select_kernel(const int64_t* __restrict__ shard_start, const int64_t* __restrict__ shard_k,
                    ShardSel* __restrict__ sel, uint32_t* __restrict__ hist) {
  constexpr int NB = (PASS == 2) ? 512 : kBins;
  constexpr int PER = NB / 256;
  __shared__ uint32_t warp_tot[8];
  __shared__ uint32_t sh_digit, sh_above, sh_count;
  const int s = blockIdx.x;
  uint32_t* row = hist + (int64_t)s * kBins;
  const int64_t s_lo = shard_start[s], s_hi = shard_start[s + 1];
  const int64_t n = s_hi - s_lo, k = shard_k[s];

  ShardSel st;
  if (PASS == 0) {
    st.prefix = 0;
    st.krem = (uint32_t)k;
    st.kstar = 0;
    st.need = 0;
    st.count_eq = 0;
    st.istar = s_hi - 1;
    st.cprefix = 0;
    st.guess = kNoGuess;
    st.flags = 0;
    if (n <= 0 || k <= 0) st.mode = kSelEmpty;
    else if (k >= n) st.mode = kSelDone;  // every key selected: kstar = 0, istar = last
    else st.mode = kSelSearch;
  } else {
    st = sel[s];
  }
  if (st.mode != kSelSearch) {
    if (threadIdx.x == 0 && PASS == 0) sel[s] = st;
    for (int b = threadIdx.x; b < kBins; b += blockDim.x) row[b] = 0;
    return;
  }

  // thread t owns bins [NB - PER*(t+1), NB - PER*t): descending order
  if (threadIdx.x == 0) {
    sh_digit = 0;
    sh_above = 0;
    sh_count = 0;
  }
  uint32_t h[PER];
  uint32_t local = 0;
  const int top = NB - PER * (int)threadIdx.x - 1;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    h[q] = row[top - q];
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
        sh_count = h[q];
        break;
      }
      cum += h[q];
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += blockDim.x) row[b] = 0;
  if (threadIdx.x == 0) {
    const int bitsw = (PASS == 2) ? 9 : 11;
    st.prefix = (st.prefix << bitsw) | sh_digit;
    st.krem -= sh_above;
    if (PASS == 2) {
      st.kstar = st.prefix;
      st.need = st.krem;
      st.count_eq = sh_count;
      if (st.need == st.count_eq) {
        st.istar = s_hi - 1;  // every key equal to kstar is selected
        st.mode = kSelDone;
      } else {
        st.istar = -1;
        st.mode = kSelTie;
      }
    }
    sel[s] = st;
  }
}

// ------------------------------------------------------------------ ties
// Count keys equal to kstar per 4096-parameter chunk of each tied shard.
__global__ void __launch_bounds__(256)
tie_count_kernel(const float* __restrict__ m, const int64_t* __restrict__ shard_start,
                 const ShardSel* __restrict__ sel, uint32_t* __restrict__ eqcnt, int64_t nchunk) {
  __shared__ uint32_t warp_tot[8];
  const int s = blockIdx.y;
  const int64_t c = blockIdx.x;
  if (sel[s].mode != kSelTie) return;
  const int64_t lo = shard_start[s] + c * kTieChunk;
  const int64_t hi = min(lo + (int64_t)kTieChunk, shard_start[s + 1]);
  if (lo >= hi) return;
  const uint32_t kstar = sel[s].kstar;
  uint32_t cnt = 0;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x)
    cnt += magnitude_key(__ldcs(m + i)) == kstar;
  uint32_t total;
  block_exclusive_scan<256>(cnt, warp_tot, &total);
  if (threadIdx.x == 0) eqcnt[(int64_t)s * nchunk + c] = total;
}

// One block per tied shard: locate the chunk holding the need-th equal key,
// then the key itself, scanning in index order.
__global__ void __launch_bounds__(256)
tie_select_kernel(const float* __restrict__ m, const int64_t* __restrict__ shard_start,
                  ShardSel* __restrict__ sel, const uint32_t* __restrict__ eqcnt, int64_t nchunk) {
  __shared__ uint32_t warp_tot[8];
  __shared__ int64_t sh_chunk;
  __shared__ uint32_t sh_before;
  __shared__ int64_t sh_istar;
  const int s = blockIdx.x;
  ShardSel st = sel[s];
  if (st.mode != kSelTie) return;
  const int64_t s_lo = shard_start[s], s_hi = shard_start[s + 1];
  const int64_t nch = (s_hi - s_lo + kTieChunk - 1) / kTieChunk;
  const uint32_t* row = eqcnt + (int64_t)s * nchunk;

  if (threadIdx.x == 0) {
    sh_chunk = 0;
    sh_before = 0;
    sh_istar = s_hi - 1;
  }
  // 1) chunk: each thread sums a contiguous run of chunk counts
  const int64_t per = (nch + 255) / 256;
  const int64_t c0 = min(nch, per * threadIdx.x), c1 = min(nch, c0 + per);
  uint32_t local = 0;
  for (int64_t c = c0; c < c1; ++c) local += row[c];
  uint32_t total;
  const uint32_t excl = block_exclusive_scan<256>(local, warp_tot, &total);
  if (excl < st.need && st.need <= excl + local) {
    uint32_t cum = excl;
    for (int64_t c = c0; c < c1; ++c) {
      if (cum + row[c] >= st.need) {
        sh_chunk = c;
        sh_before = cum;
        break;
      }
      cum += row[c];
    }
  }
  __syncthreads();
  const int64_t lo = s_lo + sh_chunk * kTieChunk;
  const int64_t hi = min(lo + (int64_t)kTieChunk, s_hi);
  uint32_t want = st.need - sh_before;  // 1-based rank among equal keys of this chunk
  // 2) rounds of 256 parameters in index order
  for (int64_t r0 = lo; r0 < hi; r0 += 256) {
    const int64_t i = r0 + threadIdx.x;
    const uint32_t eq = (i < hi) && magnitude_key(m[i]) == st.kstar;
    __syncthreads();
    uint32_t round_total;
    const uint32_t before = block_exclusive_scan<256>(eq, warp_tot, &round_total);
    if (eq && before + 1 == want) sh_istar = i;
    __syncthreads();
    if (round_total >= want) break;
    want -= round_total;
  }
  if (threadIdx.x == 0) {
    st.istar = sh_istar;
    st.mode = kSelDone;
    sel[s] = st;
  }
}

// ------------------------------------------------------------------ mark
// One 128-thread block per 2048-parameter tile.  Warp q covers parameters
// [512q, 512q + 512) of the tile in four rounds of 128: lane l decides the four
// parameters of one 16-byte load, the 4-bit pieces of 8 neighbouring lanes are
// OR-ed into one 32-bit word by shuffles, and lane 8g writes word g of the round.
__device__ __forceinline__ void mark_tile(int64_t tile, const float* __restrict__ m, int64_t P,
                                          const ShardMap& sm,
                                          const int64_t* __restrict__ shard_start,
                                          const ShardSel* __restrict__ sel,
                                          uint32_t* __restrict__ bits,
                                          uint32_t* __restrict__ tile_cnt, bool accumulate) {
  __shared__ uint32_t warp_cnt[4];
  __shared__ int sh_s, sh_uniform, sh_lim;
  __shared__ uint32_t sh_kstar;
  const int64_t t0 = tile * kTile;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t wb = t0 + warp * 512;
  const bool full = t0 + kTile <= P;
  // the tile's shard and threshold, found once per block (a 64-bit division)
  // and broadcast; the m loads below do not wait for it
  float4 v[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t i0 = wb + 128 * r + 4 * lane;
    if (full) {
      v[r] = __ldcs(reinterpret_cast<const float4*>(m + i0));
    } else {
      v[r].x = i0 < P ? __ldcs(m + i0) : 0.f;
      v[r].y = i0 + 1 < P ? __ldcs(m + i0 + 1) : 0.f;
      v[r].z = i0 + 2 < P ? __ldcs(m + i0 + 2) : 0.f;
      v[r].w = i0 + 3 < P ? __ldcs(m + i0 + 3) : 0.f;
    }
  }
  if (threadIdx.x == 0) {
    const int s0 = sm.of(t0);
    const int64_t t1 = min(t0 + (int64_t)kTile, P);
    const int64_t ist = sel[s0].istar;
    const int64_t rel64 = ist - t0;
    sh_s = s0;
    sh_uniform = __ldg(shard_start + s0 + 1) >= t1;
    sh_kstar = sel[s0].kstar;
    sh_lim = rel64 < 0 ? -1 : (rel64 >= kTile ? kTile : (int)rel64);
  }
  __syncthreads();
  const int s = sh_s;
  const bool uniform = sh_uniform != 0;
  const uint32_t kstar_s = sh_kstar;

  const int64_t nwords = (P + 31) / 32;
  // Whole-tile fast path: "key > kstar, or key == kstar and i <= istar" is
  // "key >= kstar + (i > istar)", with i taken relative to the tile in 32 bits.
  const int lim = sh_lim;
  uint32_t cnt = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t i0 = wb + 128 * r + 4 * lane;
    const float x[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
    uint32_t nib = 0;
    if (uniform && full) {
      const int li = warp * 512 + 128 * r + 4 * lane;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        nib |= (uint32_t)(magnitude_key(x[q]) >= kstar_s + (uint32_t)(li + q > lim)) << q;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t i = i0 + q;
        if (i < P) {
          int si = s;
          while (si < sm.S - 1 && i >= __ldg(shard_start + si + 1)) ++si;
          const uint32_t kstar = sel[si].kstar;
          const int64_t istar = sel[si].istar;
          const uint32_t key = magnitude_key(x[q]);
          nib |= (uint32_t)(key > kstar || (key == kstar && i <= istar)) << q;
        }
      }
    }
    uint32_t word = nib << (4 * (lane & 7));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    const int64_t widx = (wb + 128 * r) / 32 + (lane >> 3);
    if ((lane & 7) == 0) {
      if (widx < nwords) bits[widx] = accumulate ? (bits[widx] | word) : word;
      cnt += __popc(word);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) warp_cnt[warp] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) tile_cnt[tile] = warp_cnt[0] + warp_cnt[1] + warp_cnt[2] + warp_cnt[3];
}

__global__ void __launch_bounds__(128)
mark_kernel(const float* __restrict__ m, int64_t P, ShardMap sm,
            const int64_t* __restrict__ shard_start,
            const ShardSel* __restrict__ sel, uint32_t* __restrict__ bits,
            uint32_t* __restrict__ tile_cnt, bool accumulate) {
  mark_tile(blockIdx.x, m, P, sm, shard_start, sel, bits, tile_cnt, accumulate);
}

// Warm refresh, grid (G, W): the tiles starting in shard s that the
// speculative bitmap does not cover -- all of them when the shard is flagged
// kSelRemark, else only its last one when it crosses the shard's end (or the
// end of the vector).  Each tile is owned by the shard it starts in.
__global__ void __launch_bounds__(128)
remark_kernel(const float* __restrict__ m, int64_t P, ShardMap sm,
              const int64_t* __restrict__ shard_start, const ShardSel* __restrict__ sel,
              uint32_t* __restrict__ bits, uint32_t* __restrict__ tile_cnt) {
  const int s = blockIdx.y;
  const int64_t s_lo = shard_start[s], s_hi = shard_start[s + 1];
  if (s_lo >= s_hi) return;
  int64_t t_begin = (s_lo + kTile - 1) / kTile;
  const int64_t t_end = (s_hi + kTile - 1) / kTile;
  if (!(sel[s].flags & kSelRemark)) {
    if (t_end <= t_begin || t_end * kTile == s_hi) return;
    t_begin = t_end - 1;
  }
  for (int64_t t = t_begin + blockIdx.x; t < t_end; t += gridDim.x)
    mark_tile(t, m, P, sm, shard_start, sel, bits, tile_cnt, false);
}

// Per-tile popcount of an existing bitmap (checkpoint resume).
__global__ void __launch_bounds__(64)
tile_count_kernel(const uint32_t* __restrict__ bits, int64_t nwords, uint32_t* __restrict__ tile_cnt) {
  const int64_t wi = (int64_t)blockIdx.x * kTileWords + threadIdx.x;
  uint32_t c = wi < nwords ? __popc(bits[wi]) : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  __shared__ uint32_t part[2];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) tile_cnt[blockIdx.x] = part[0] + part[1];
}

// ------------------------------------------------------------------ scan
// Exclusive scan of the per-tile counts into the rank table, in three
// launches: local scans of 2048-tile chunks, a scan of the chunk totals
// (at most 512 chunks for P < 2^31), and the chunk offsets added back.
constexpr int kScanChunk = 2048;

__global__ void __launch_bounds__(256)
scan_local_kernel(const uint32_t* __restrict__ cnt, int64_t n, uint32_t* __restrict__ base,
                  uint32_t* __restrict__ chunk_tot) {
  __shared__ uint32_t warp_tot[8];
  const int64_t c0 = (int64_t)blockIdx.x * kScanChunk + threadIdx.x * 8;
  uint32_t v[8], local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = c0 + j < n ? cnt[c0 + j] : 0u;
    local += v[j];
  }
  uint32_t total;
  uint32_t run = block_exclusive_scan<256>(local, warp_tot, &total);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (c0 + j < n) base[c0 + j] = run;
    run += v[j];
  }
  if (threadIdx.x == 0) chunk_tot[blockIdx.x] = total;
}

__global__ void __launch_bounds__(1024)
scan_top_kernel(const uint32_t* __restrict__ chunk_tot, int64_t nchunks,
                uint32_t* __restrict__ chunk_base, uint32_t* __restrict__ base_total) {
  __shared__ uint32_t warp_tot[32];
  const uint32_t v = threadIdx.x < nchunks ? chunk_tot[threadIdx.x] : 0u;
  uint32_t total;
  const uint32_t ex = block_exclusive_scan<1024>(v, warp_tot, &total);
  if (threadIdx.x < nchunks) chunk_base[threadIdx.x] = ex;
  if (threadIdx.x == 0) *base_total = total;
}

__global__ void __launch_bounds__(256)
scan_add_kernel(uint32_t* __restrict__ base, int64_t n, const uint32_t* __restrict__ chunk_base) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n) base[t] += chunk_base[t / kScanChunk];
}

// ------------------------------------------------------------------ index
// idx[rank] = i for every set bit, ranks ascending.  Persistent warps, one
// 2048-parameter tile at a time (lane l owns bitmap words 2l and 2l + 1); the
// next tile's words and rank base are loaded before the current tile's
// indices are written, so a warp is not idle for a load round trip per tile.
// STAGED (denser masks): lanes write their set positions into the warp's
// shared-memory buffer at their exclusive offsets and the warp copies the
// tile's contiguous run out with coalesced stores; otherwise (sparse masks)
// each lane writes its few positions straight to their ranks.
template <bool STAGED>
__global__ void __launch_bounds__(STAGED ? 128 : 256)
index_kernel(const uint32_t* __restrict__ bits, int64_t P, int64_t ntiles,
             const uint32_t* __restrict__ tile_base, uint32_t* __restrict__ idx) {
  constexpr int kWarps = STAGED ? 4 : 8;  // staged: 8 KB of shared memory per warp
  __shared__ uint32_t buf[STAGED ? kWarps : 1][STAGED ? kTile : 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nwords = (P + 31) / 32;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  int64_t tile = (int64_t)blockIdx.x * kWarps + warp;
  if (tile >= ntiles) return;
  auto load = [&](int64_t t, uint32_t& a, uint32_t& b, uint32_t& base) {
    const int64_t w0 = t * kTileWords + 2 * lane;
    a = w0 < nwords ? __ldg(bits + w0) : 0u;
    b = w0 + 1 < nwords ? __ldg(bits + w0 + 1) : 0u;
    base = __ldg(tile_base + t);
  };
  uint32_t a, b, base;
  load(tile, a, b, base);
  for (; tile < ntiles; tile += stride) {
    uint32_t na = 0, nb = 0, nbase = 0;
    if (tile + stride < ntiles) load(tile + stride, na, nb, nbase);
    const uint32_t c = __popc(a) + __popc(b);
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const uint32_t ia = (uint32_t)((tile * kTileWords + 2 * lane) * 32), ib = ia + 32;
    if (STAGED) {
      const uint32_t total = __shfl_sync(0xffffffffu, x, 31);
      uint32_t* sb = buf[warp];
      uint32_t o = x - c;
      while (a) {
        sb[o++] = ia + (uint32_t)(__ffs(a) - 1);
        a &= a - 1;
      }
      while (b) {
        sb[o++] = ib + (uint32_t)(__ffs(b) - 1);
        b &= b - 1;
      }
      __syncwarp();
      uint32_t* out = idx + base;
      for (uint32_t j = lane; j < total; j += 32) out[j] = sb[j];
      __syncwarp();  // the buffer is rewritten for the next tile
    } else {
      uint32_t* out = idx + base + (x - c);
      while (a) {
        *out++ = ia + (uint32_t)(__ffs(a) - 1);
        a &= a - 1;
      }
      while (b) {
        *out++ = ib + (uint32_t)(__ffs(b) - 1);
        b &= b - 1;
      }
    }
    a = na;
    b = nb;
    base = nbase;
  }
}

// Per-shard popcount of a bitmap plus the count of bits set past P (in
// counts[W]); used to validate a restored mask.
__global__ void __launch_bounds__(256)
shard_count_kernel(const uint32_t* __restrict__ bits, int64_t P, int64_t nwords, ShardMap sm,
                   uint32_t* __restrict__ counts) {
  const int64_t wi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (wi >= nwords) return;
  uint32_t word = bits[wi];
  while (word) {
    const int b = __ffs(word) - 1;
    word &= word - 1;
    const int64_t i = wi * 32 + b;
    if (i >= P) atomicAdd(counts + sm.S, 1u);
    else atomicAdd(counts + sm.of(i), 1u);
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_hist(int pass, const float* m, int64_t P, const ShardMap& sm,
                        const int64_t* shard_start, const ShardSel* sel, uint32_t* hist,
                        cudaStream_t st) {
  const unsigned grid = (unsigned)((P + kSeg - 1) / kSeg);
  if (pass == 0) radix_hist_kernel<0><<<grid, 256, 0, st>>>(m, P, sm, shard_start, sel, hist);
  else if (pass == 1) radix_hist_kernel<1><<<grid, 256, 0, st>>>(m, P, sm, shard_start, sel, hist);
  else radix_hist_kernel<2><<<grid, 256, 0, st>>>(m, P, sm, shard_start, sel, hist);
  return cudaGetLastError();
}

cudaError_t launch_select(int pass, int W, const int64_t* shard_start, const int64_t* shard_k,
                          ShardSel* sel, uint32_t* hist, cudaStream_t st) {
  if (pass == 0) radix_select_kernel<0><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist);
  else if (pass == 1) radix_select_kernel<1><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist);
  else radix_select_kernel<2><<<W, 256, 0, st>>>(shard_start, shard_k, sel, hist);
  return cudaGetLastError();
}

cudaError_t launch_tie_count(const float* m, int W, const int64_t* shard_start,
                             const ShardSel* sel, uint32_t* eqcnt, int64_t nchunk,
                             cudaStream_t st) {
  dim3 grid((unsigned)nchunk, (unsigned)W);
  tie_count_kernel<<<grid, 256, 0, st>>>(m, shard_start, sel, eqcnt, nchunk);
  return cudaGetLastError();
}

cudaError_t launch_tie_select(const float* m, int W, const int64_t* shard_start, ShardSel* sel,
                              const uint32_t* eqcnt, int64_t nchunk, cudaStream_t st) {
  tie_select_kernel<<<W, 256, 0, st>>>(m, shard_start, sel, eqcnt, nchunk);
  return cudaGetLastError();
}

cudaError_t launch_mark(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                        const ShardSel* sel, uint32_t* bits, uint32_t* tile_cnt,
                        cudaStream_t st, bool accumulate) {
  const unsigned grid = (unsigned)((P + kTile - 1) / kTile);
  mark_kernel<<<grid, 128, 0, st>>>(m, P, sm, shard_start, sel, bits, tile_cnt, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_remark(const float* m, int64_t P, const ShardMap& sm, const int64_t* shard_start,
                          const ShardSel* sel, uint32_t* bits, uint32_t* tile_cnt,
                          cudaStream_t st) {
  // enough 128-thread blocks to fill the GPU when every shard is re-marked;
  // in the common case all but one block per shard return at once
  const int sms = sm_count();
  const int W = sm.S;
  const int64_t ntiles = (P + kTile - 1) / kTile;
  const int64_t per_shard = (ntiles + W - 1) / W + 1;
  int64_t gx = ((int64_t)sms * 16 + W - 1) / W;
  if (gx > per_shard) gx = per_shard;
  if (gx < 1) gx = 1;
  remark_kernel<<<dim3((unsigned)gx, (unsigned)W), 128, 0, st>>>(m, P, sm, shard_start, sel, bits,
                                                                 tile_cnt);
  return cudaGetLastError();
}

cudaError_t launch_tile_count(const uint32_t* bits, int64_t P, uint32_t* tile_cnt,
                              cudaStream_t st) {
  const unsigned grid = (unsigned)((P + kTile - 1) / kTile);
  tile_count_kernel<<<grid, kTileWords, 0, st>>>(bits, (P + 31) / 32, tile_cnt);
  return cudaGetLastError();
}

int64_t scan_scratch_words(int64_t ntiles) { return 2 * ((ntiles + kScanChunk - 1) / kScanChunk); }

cudaError_t launch_scan(const uint32_t* tile_cnt, int64_t ntiles, uint32_t* tile_base,
                        uint32_t* scratch, cudaStream_t st) {
  const int64_t nchunks = (ntiles + kScanChunk - 1) / kScanChunk;
  if (nchunks > 1024) return cudaErrorInvalidValue;
  uint32_t* chunk_tot = scratch;
  uint32_t* chunk_base = scratch + nchunks;
  scan_local_kernel<<<(unsigned)nchunks, 256, 0, st>>>(tile_cnt, ntiles, tile_base, chunk_tot);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scan_top_kernel<<<1, 1024, 0, st>>>(chunk_tot, nchunks, chunk_base, tile_base + ntiles);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scan_add_kernel<<<(unsigned)((ntiles + 255) / 256), 256, 0, st>>>(tile_base, ntiles, chunk_base);
  return cudaGetLastError();
}

cudaError_t launch_index(const uint32_t* bits, int64_t P, const uint32_t* tile_base,
                         uint32_t* idx, int64_t k, cudaStream_t st) {
  const int64_t ntiles = (P + kTile - 1) / kTile;
  const int sms = sm_count();
  // measured on GB300: direct stores win at 1% density, staged stores at 10%
  const bool staged = !(k >= 0 && k * 20 < P);
  // persistent: staged blocks (4 warps, 32 KB) 6 per SM, direct ones (8 warps) 8 per SM
  const int warps = staged ? 4 : 8;
  const int64_t want = (int64_t)sms * (staged ? 6 : 8);
  const int64_t need = (ntiles + warps - 1) / warps;
  const unsigned grid = (unsigned)(need < want ? need : want);
  if (staged)
    index_kernel<true><<<grid, 128, 0, st>>>(bits, P, ntiles, tile_base, idx);
  else
    index_kernel<false><<<grid, 256, 0, st>>>(bits, P, ntiles, tile_base, idx);
  return cudaGetLastError();
}

cudaError_t launch_shard_count(const uint32_t* bits, int64_t P, int64_t nwords, const ShardMap& sm,
                               uint32_t* counts, cudaStream_t st) {
  shard_count_kernel<<<(unsigned)((nwords + 255) / 256), 256, 0, st>>>(bits, P, nwords, sm, counts);
  return cudaGetLastError();
}

}  // namespace scapek
