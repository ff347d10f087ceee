// union_kernels.cu -- kernels of the union-mask gradient top-k baseline (the
// second synchronisation scheme of "SCAPE" Sec. II-B): every worker selects
// the top-k of its own error-fed gradient over the whole vector, the masks
// are OR-ed into their union, and every worker sends its values at every
// union position.
//
//   ef_add      e^w <- g^w + e^w for every worker (the error-fed gradient a^w,
//               kept in the residual buffer until the union is known)
//   union_move  for each union position i (ascending, rank j) and worker w:
//               pack[w][j] = a^w_i and e^w_i <- a - a (sent)
// The per-worker selection reuses the refresh kernels on a^w with a one-shard
// table; the union bitmap is built by mark in accumulate mode.
#include "scape_internal.cuh"

namespace scapek {
namespace {

template <typename GT>
__device__ __forceinline__ float grad_at(const void* g, int64_t i) {
  if (sizeof(GT) == 2)
    return __uint_as_float(
        (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(g) + i) << 16);
  return __ldcs(static_cast<const float*>(g) + i);
}

// 4 parameters per thread, all workers; 16-byte accesses of e when aligned.
template <typename GT, bool VEC>
__global__ void __launch_bounds__(256)
ef_add_kernel(const __grid_constant__ WorkerPtrs ptrs, int W, int64_t P) {
  const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i0 >= P) return;
  const bool full = VEC && i0 + 4 <= P;
  for (int wk = 0; wk < W; ++wk) {
    float* e = ptrs.e[wk];
    if (full) {
      float4 ev = __ldcs(reinterpret_cast<const float4*>(e + i0));
      float g[4];
      if (sizeof(GT) == 2) {
        const uint2 u = __ldcs(reinterpret_cast<const uint2*>(
            static_cast<const unsigned short*>(ptrs.g[wk]) + i0));
        g[0] = __uint_as_float(u.x << 16);
        g[1] = __uint_as_float(u.x & 0xFFFF0000u);
        g[2] = __uint_as_float(u.y << 16);
        g[3] = __uint_as_float(u.y & 0xFFFF0000u);
      } else {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(
            static_cast<const float*>(ptrs.g[wk]) + i0));
        g[0] = v.x; g[1] = v.y; g[2] = v.z; g[3] = v.w;
      }
      ev.x = __fadd_rn(g[0], ev.x);
      ev.y = __fadd_rn(g[1], ev.y);
      ev.z = __fadd_rn(g[2], ev.z);
      ev.w = __fadd_rn(g[3], ev.w);
      __stcs(reinterpret_cast<float4*>(e + i0), ev);
    } else {
      for (int j = 0; j < 4 && i0 + j < P; ++j)
        e[i0 + j] = __fadd_rn(grad_at<GT>(ptrs.g[wk], i0 + j), e[i0 + j]);
    }
  }
}

// One thread per union position: gather the W error-fed gradients into the
// packed buffers and clear the sent residuals.
__global__ void __launch_bounds__(256)
union_move_kernel(const __grid_constant__ WorkerPtrs ptrs, int W, const uint32_t* __restrict__ idx,
                  int64_t k, float* __restrict__ pack, int64_t stride) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const uint32_t i = __ldg(idx + j);
  for (int wk = 0; wk < W; ++wk) {
    const float a = ptrs.e[wk][i];
    pack[(int64_t)wk * stride + j] = a;
    ptrs.e[wk][i] = __fsub_rn(a, a);
  }
}

}  // namespace

cudaError_t launch_ef_add(const WorkerPtrs& p, int W, int64_t P, int dtype, bool vec,
                          cudaStream_t st) {
  const unsigned grid = (unsigned)(((P + 3) / 4 + 255) / 256);
  if (dtype == SCAPE_BF16) {
    if (vec) ef_add_kernel<__nv_bfloat16, true><<<grid, 256, 0, st>>>(p, W, P);
    else ef_add_kernel<__nv_bfloat16, false><<<grid, 256, 0, st>>>(p, W, P);
  } else {
    if (vec) ef_add_kernel<float, true><<<grid, 256, 0, st>>>(p, W, P);
    else ef_add_kernel<float, false><<<grid, 256, 0, st>>>(p, W, P);
  }
  return cudaGetLastError();
}

cudaError_t launch_union_move(const WorkerPtrs& p, int W, const uint32_t* idx, int64_t k,
                              float* pack, int64_t stride, cudaStream_t st) {
  if (k <= 0) return cudaSuccess;
  union_move_kernel<<<(unsigned)((k + 255) / 256), 256, 0, st>>>(p, W, idx, k, pack, stride);
  return cudaGetLastError();
}

}  // namespace scapek
