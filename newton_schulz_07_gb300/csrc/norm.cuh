// Frobenius norm and scale: the first step of NS, X = G / (||G||_F + eps).
//
// Two memory-bound kernels over a stack of matrices stored as 16-byte vectors
// of 8 bf16 values (rows and columns are multiples of 8, so every matrix
// starts on a 16-byte boundary):
//
//   ns_norm_partial  grid (chunks, min(batch, 65535)): each CTA sums the squares of one
//                    chunk of kNormChunkVec vectors in fp32 (per thread, then a
//                    fixed xor-shuffle tree per warp, then the warps in order)
//                    and stores the partial.  The CTA that takes the last
//                    ticket of its matrix adds the partials in a fixed order
//                    and writes ||G||_F.  The chunking depends only on the
//                    matrix size, so a matrix gets bit-identical norms alone or
//                    in any stack.
//   ns_scale         grid (chunks, min(batch, 65535)): X = bf16_rn(G * (1 / (nu + eps))),
//                    elementwise in the input orientation (G may equal X).
// Both are templated on F32: stacks of fp32 (the fp32 NS mode) instead of bf16.
// The grid's y extent stops at the hardware limit of 65535: a CTA takes
// matrices blockIdx.y, blockIdx.y + gridDim.y, ... of a larger stack, each
// exactly as a CTA of its own would.
//
// The norm is the per-matrix Frobenius normalisation of Dion's dense NS named
// by prime-rl PR #3873, Summary item 1.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mns {

constexpr int kNormThreads = 256;
constexpr int kNormVecPerThread = 8;
constexpr long long kNormChunkVec = static_cast<long long>(kNormThreads) * kNormVecPerThread;

namespace detail {

__device__ __forceinline__ float sumsq_bf16x8(const uint4 w) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float lo = __uint_as_float(ws[h] << 16);
    const float hi = __uint_as_float(ws[h] & 0xFFFF0000u);
    s = fmaf(lo, lo, s);
    s = fmaf(hi, hi, s);
  }
  return s;
}

__device__ __forceinline__ float sumsq_f32x4(const uint4 w) {
  const float a = __uint_as_float(w.x), b = __uint_as_float(w.y);
  const float c = __uint_as_float(w.z), d = __uint_as_float(w.w);
  return fmaf(d, d, fmaf(c, c, fmaf(b, b, a * a)));
}

__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float total = 0.0f;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) total += red[w];
  }
  __syncthreads();
  return total;  // valid in thread 0
}

}  // namespace detail

// F32: the stack holds fp32 (4 per 16-byte vector) instead of bf16 (8).
template <bool F32>
__global__ void __launch_bounds__(kNormThreads)
    ns_norm_partial(const uint4* __restrict__ G, long long vec_per_matrix, int chunks, int batch,
                    float* __restrict__ partials, unsigned int* __restrict__ tickets,
                    float* __restrict__ norms) {
  __shared__ float red[kNormThreads / 32];
  __shared__ int is_last;
  ptx::griddep_wait();
  const int chunk = blockIdx.x;
  const long long base = static_cast<long long>(chunk) * kNormChunkVec;
  for (int b = blockIdx.y; b < batch; b += gridDim.y) {
    const uint4* g = G + static_cast<long long>(b) * vec_per_matrix;
    uint4 w[kNormVecPerThread];
#pragma unroll
    for (int it = 0; it < kNormVecPerThread; ++it) {
      const long long i = base + it * kNormThreads + threadIdx.x;
      w[it] = i < vec_per_matrix ? __ldcs(g + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    float acc = 0.0f;
#pragma unroll
    for (int it = 0; it < kNormVecPerThread; ++it)
      acc += F32 ? detail::sumsq_f32x4(w[it]) : detail::sumsq_bf16x8(w[it]);

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

template <bool F32>
__global__ void __launch_bounds__(kNormThreads)
    ns_scale(const uint4* G, uint4* X, long long vec_per_matrix, int batch, const float* __restrict__ norms,
             float eps) {
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const long long base = static_cast<long long>(blockIdx.x) * kNormChunkVec;
  for (int b = blockIdx.y; b < batch; b += gridDim.y) {
    const float s = 1.0f / (norms[b] + eps);
    const uint4* g = G + static_cast<long long>(b) * vec_per_matrix;
    uint4* x = X + static_cast<long long>(b) * vec_per_matrix;
    uint4 w[kNormVecPerThread];
#pragma unroll
    for (int it = 0; it < kNormVecPerThread; ++it) {
      const long long i = base + it * kNormThreads + threadIdx.x;
      w[it] = i < vec_per_matrix ? g[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < kNormVecPerThread; ++it) {
      const long long i = base + it * kNormThreads + threadIdx.x;
      if (i >= vec_per_matrix) continue;
      uint32_t ws[4] = {w[it].x, w[it].y, w[it].z, w[it].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (F32) {
          ws[h] = __float_as_uint(__uint_as_float(ws[h]) * s);
        } else {
          const float lo = __uint_as_float(ws[h] << 16) * s;
          const float hi = __uint_as_float(ws[h] & 0xFFFF0000u) * s;
          ws[h] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
                  (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
        }
      }
      x[i] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
    }
  }
}

// out[b][c][r] = in[b][r][c] for fp32 stacks [batch][R][C], through a padded
// 32 x 33 shared tile (coalesced reads and writes).  grid (ceil(C/32),
// ceil(R/32), min(batch, 65535)), block (32, 8); a CTA takes matrices
// blockIdx.z, blockIdx.z + gridDim.z, ...  The fp32 NS path uses it once per
// call to give the first step both orientations of G.
__global__ void __launch_bounds__(256)
    ns_transpose_f32(const float* __restrict__ in, float* __restrict__ out, int R, int C, int batch) {
  __shared__ float tile[32][33];
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const long long mat = static_cast<long long>(R) * C;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int b = blockIdx.z; b < batch; b += gridDim.z) {
    const float* src = in + b * mat;
    float* dst = out + b * mat;
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
      const int r = r0 + threadIdx.y + k, c = c0 + threadIdx.x;
      if (r < R && c < C) tile[threadIdx.y + k][threadIdx.x] = src[static_cast<long long>(r) * C + c];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
      const int c = c0 + threadIdx.y + k, r = r0 + threadIdx.x;
      if (r < R && c < C) dst[static_cast<long long>(c) * R + r] = tile[threadIdx.x][threadIdx.y + k];
    }
    __syncthreads();  // the tile is rewritten for the next matrix
  }
}

}  // namespace mns
