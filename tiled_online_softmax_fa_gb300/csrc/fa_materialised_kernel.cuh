// fa_materialised_kernel.cuh -- the row softmax of the materialised attention baseline.
//
// The baseline is the pages' `standard_attention` (aiml.sh "Speed up long contexts with
// FlashAttention", lab.py) run on the GPU with the N x N matrices in HBM:
//   S = scale * Q K^T        (fp32, [BH, N, N], written by a cuBLAS batched GEMM)
//   P = exp(S - rowmax) + mask, row sums (row_softmax_kernel: bf16 P, natural-log lse)
//   acc = P V                (a second cuBLAS batched GEMM, fp32 result)
//   O = acc / row sum        (normalise_kernel, bf16)
// Dividing after the product keeps each row's weights summing to one exactly as the
// GEMM applies them (the bf16 P are summed as rounded), as the tiled kernels do.
// It exists to measure what the tiled kernels avoid: the HBM traffic of the N x N
// scores and probabilities that the pages model as 4 H N^2 elements per batch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fa_sm103 {
namespace mat {

constexpr int kRowThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Block-wide (max, sum) reduction of per-thread online-softmax states.
__device__ __forceinline__ void combine(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  l = l * exp2f((m - mn) * kLog2e) + l2 * exp2f((m2 - mn) * kLog2e);
  m = mn;
}

// Block-wide sum of one float per thread (result valid in every thread).
__device__ __forceinline__ float block_sum(float x, float* scratch) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // scratch may still be read from an earlier reduction
  if (lane == 0) scratch[warp] = x;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += scratch[w];
  return t;
}

// One CTA per row r = bh * N + i of S.  Columns j <= last (causal: last = i) get
// p = exp(s - m) rounded to bf16 (so the row maximum is exactly 1), the others 0.
// l_round[r] = sum of the rounded p (the weights the second GEMM applies, used to
// normalise O), lse[r] = m + ln(sum of the exact p).  Two passes over the row: an
// online (max, sum) pass, then the write pass (the row is re-read from L2).
__global__ void __launch_bounds__(kRowThreads)
    row_softmax_kernel(const float* __restrict__ S, __nv_bfloat16* __restrict__ P,
                       float* __restrict__ l_round, float* __restrict__ lse, int N, int causal) {
  const int64_t r = blockIdx.x;
  const int i = static_cast<int>(r % N);
  const int last = causal ? i : N - 1;
  const float* srow = S + r * static_cast<int64_t>(N);
  __nv_bfloat16* prow = P + r * static_cast<int64_t>(N);
  float m = -INFINITY, l = 0.f;
  for (int j = threadIdx.x; j <= last; j += kRowThreads) {
    const float s = srow[j];
    if (s > m) {
      l = (m == -INFINITY) ? 0.f : l * exp2f((m - s) * kLog2e);
      m = s;
    }
    l += exp2f((s - m) * kLog2e);
  }
  // reduce across the warp, then across the warps through shared memory
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, off);
    combine(m, l, m2, l2);
  }
  __shared__ float sm[kRowThreads / 32], sl[kRowThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[warp] = m;
    sl[warp] = l;
  }
  __syncthreads();
  m = -INFINITY;
  l = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) combine(m, l, sm[w], sl[w]);
  float rsum = 0.f;
  for (int j = threadIdx.x; j < N; j += kRowThreads) {
    const __nv_bfloat16 pb =
        __float2bfloat16_rn(j <= last ? exp2f((srow[j] - m) * kLog2e) : 0.f);
    prow[j] = pb;
    rsum += __bfloat162float(pb);
  }
  __shared__ float scratch[kRowThreads / 32];
  rsum = block_sum(rsum, scratch);
  if (threadIdx.x == 0) {
    l_round[r] = rsum;
    if (lse != nullptr) lse[r] = m + logf(l);
  }
}

// O[r][c] = acc[r][c] / l_round[r], rounded to bf16; four elements per thread (d % 4 == 0).
__global__ void normalise_kernel(const float4* __restrict__ acc, const float* __restrict__ l_round,
                                 uint2* __restrict__ o, int64_t quads, int d) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= quads) return;
  const float inv = 1.f / l_round[(t * 4) / d];
  const float4 a = acc[t];
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * inv, a.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * inv, a.w * inv);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&lo);
  w.y = *reinterpret_cast<const uint32_t*>(&hi);
  o[t] = w;
}

}  // namespace mat
}  // namespace fa_sm103
