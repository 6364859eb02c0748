// Memory-bound kernels of the Muon optimizer step around NS.  Master weights
// W and momentum M are fp32, the NS runs in bf16 (the `ns_dtype` setting of
// param-decomp PR #978, What: "masters/momentum stay fp32"); the step is the
// one prime-rl PR #3873 (Summary) speeds up, with the update rule of
// muon_step_ws() in include/muon_ns.h:
//
//   muon_momentum_norm   M' = mu M + G;  U = bf16(G + mu M') (Nesterov) or
//                        bf16(M');  and ||U||_F per matrix.  The norm uses the
//                        chunks, per-thread order and reduction tree of
//                        ns_norm_partial over the stored U, so it is the same
//                        fp32 value bit for bit and the NS that follows is
//                        exactly the NS of U.
//   muon_apply           W' = decay W - lrs O for the bf16 NS output O
//                        (decay = 1 - lr wd, lrs = lr scale): the per-step form
//                        of what the last update product does in a whole step.
//
// Both read and write 16-byte vectors (4 fp32, or 8 bf16); rows and columns
// are multiples of 8, so every matrix starts on a 32-byte boundary of the
// fp32 stacks.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

#include "norm.cuh"
#include "ptx.cuh"

namespace mns {

namespace detail {

// One 8-element vector of the step: m' = fma(mu, m, g); u = fma(mu, m', g)
// (Nesterov) or m'; u rounded to bf16, packed low element first.
__device__ __forceinline__ uint4 momentum8(const float4 g0, const float4 g1, float4& m0, float4& m1, float mu,
                                          int nesterov) {
  float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float u[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    m[j] = fmaf(mu, m[j], g[j]);
    u[j] = nesterov ? fmaf(mu, m[j], g[j]) : m[j];
  }
  m0 = make_float4(m[0], m[1], m[2], m[3]);
  m1 = make_float4(m[4], m[5], m[6], m[7]);
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(u[2 * h], u[2 * h + 1]);
    w[h] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace detail

// grid (chunks, min(batch, 65535)), kNormThreads threads.  G, M: fp32
// [batch][R][C]; U: bf16 [batch][R][C]; vec_per_matrix = R * C / 8.  A CTA
// takes matrices blockIdx.y, blockIdx.y + gridDim.y, ... (the grid's y extent
// stops at the hardware limit).  The CTA that takes the last ticket of its
// matrix writes norms[b] (tickets zeroed beforehand).
__global__ void __launch_bounds__(kNormThreads)
    muon_momentum_norm(const float4* __restrict__ G, float4* __restrict__ M, uint4* __restrict__ U,
                       long long vec_per_matrix, int chunks, int batch, float mu, int nesterov,
                       float* __restrict__ partials, unsigned int* __restrict__ tickets,
                       float* __restrict__ norms) {
  __shared__ float red[kNormThreads / 32];
  __shared__ int is_last;
  ptx::griddep_wait();
  const int chunk = blockIdx.x;
  const long long base = static_cast<long long>(chunk) * kNormChunkVec;
  for (int b = blockIdx.y; b < batch; b += gridDim.y) {
    const long long mat = static_cast<long long>(b) * vec_per_matrix;
    // The thread's vectors in two halves: the loads of a half (8 fp32 vectors
    // in flight), then its arithmetic and stores.  Halves keep the registers
    // low enough for several CTAs per SM; the norm still adds the vectors'
    // sums of squares in the order ns_norm_partial does.
    constexpr int kHalf = kNormVecPerThread / 2;
    float acc = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 g[2 * kHalf], m[2 * kHalf];
#pragma unroll
      for (int q = 0; q < kHalf; ++q) {
        const long long i = base + (h * kHalf + q) * kNormThreads + threadIdx.x;
        if (i < vec_per_matrix) {
          const long long v = 2 * (mat + i);
          g[2 * q] = __ldcs(G + v);
          g[2 * q + 1] = __ldcs(G + v + 1);
          m[2 * q] = M[v];
          m[2 * q + 1] = M[v + 1];
        }
      }
#pragma unroll
      for (int q = 0; q < kHalf; ++q) {
        const long long i = base + (h * kHalf + q) * kNormThreads + threadIdx.x;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (i < vec_per_matrix) {
          u = detail::momentum8(g[2 * q], g[2 * q + 1], m[2 * q], m[2 * q + 1], mu, nesterov);
          const long long v = 2 * (mat + i);
          __stcs(M + v, m[2 * q]);
          __stcs(M + v + 1, m[2 * q + 1]);
          U[mat + i] = u;
        }
        acc += detail::sumsq_bf16x8(u);
      }
    }
    // The first product of the NS reads U: it may start as this grid drains
    // (signalled once, after the CTA's first matrix).
    if (b == static_cast<int>(blockIdx.y)) ptx::griddep_launch_dependents();

    const float part = detail::block_sum_fixed(acc, red);
    if (threadIdx.x == 0) {
      partials[static_cast<long long>(b) * chunks + chunk] = part;
      __threadfence();
      const unsigned int ticket = atomicAdd(&tickets[b], 1u);
      is_last = (ticket == static_cast<unsigned int>(chunks - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (is_last) {  // CTA-uniform
      __threadfence();
      float s = 0.0f;
      for (int i = threadIdx.x; i < chunks; i += kNormThreads)
        s += __ldcg(&partials[static_cast<long long>(b) * chunks + i]);
      const float total = detail::block_sum_fixed(s, red);
      if (threadIdx.x == 0) norms[b] = sqrtf(total);
    }
    __syncthreads();  // is_last and red are rewritten for the next matrix
  }
}

// W' = decay W - lrs O over n8 vectors of 8 elements (grid-stride).  W fp32,
// O bf16, the same element order.
__global__ void __launch_bounds__(256)
    muon_apply(float4* __restrict__ W, const uint4* __restrict__ O, long long n8, float decay, float lrs) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < n8; v += stride) {
    const uint4 o = __ldcs(O + v);
    float4 w0 = __ldcs(W + 2 * v), w1 = __ldcs(W + 2 * v + 1);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
    float of[8];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      of[2 * h] = __uint_as_float(ow[h] << 16);
      of[2 * h + 1] = __uint_as_float(ow[h] & 0xFFFF0000u);
    }
    w0 = make_float4(fmaf(-lrs, of[0], decay * w0.x), fmaf(-lrs, of[1], decay * w0.y),
                     fmaf(-lrs, of[2], decay * w0.z), fmaf(-lrs, of[3], decay * w0.w));
    w1 = make_float4(fmaf(-lrs, of[4], decay * w1.x), fmaf(-lrs, of[5], decay * w1.y),
                     fmaf(-lrs, of[6], decay * w1.z), fmaf(-lrs, of[7], decay * w1.w));
    __stcs(W + 2 * v, w0);
    __stcs(W + 2 * v + 1, w1);
  }
}

}  // namespace mns
