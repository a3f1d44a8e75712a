// fa_merge_kernel.cuh -- combines the per-KV-range partial results of a split launch.
//
// For one query row, KV range s produced a normalised partial output O_s and the
// logsumexp lse_s of its scores.  The full softmax over the union of the ranges is
//     lse = ln sum_s exp(lse_s),    O = sum_s exp(lse_s - lse) O_s
// (each range's weights sum to one, so exp(lse_s - lse) is that range's share of the
// row's total probability mass).  Memory bound: one warp per row, coalesced loads.
#pragma once

#include <cuda_bf16.h>

#include "fa_fwd_kernel.cuh"

namespace fa_sm103 {

constexpr int kMergeThreads = 256;  // 8 rows per block

template <int HD>
__global__ void __launch_bounds__(kMergeThreads)
    fa_merge_kernel(const Params p) {
  constexpr int E = HD >= 32 ? HD / 32 : 1;       // output elements per lane
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
  if (gw >= static_cast<int64_t>(p.BH) * p.N) return;
  const int bh = static_cast<int>(gw / p.N), row = static_cast<int>(gw - static_cast<int64_t>(bh) * p.N);
  const int qb = row / kUnitRows, rin = row - qb * kUnitRows, t = rin / kBlockM;
  // unit of (bh, qb): the inverse of unit_coords
  const int g = bh / p.group_heads, first = g * p.group_heads;
  const int heads = (p.BH - first) < p.group_heads ? (p.BH - first) : p.group_heads;
  const int u = g * p.group_heads * p.nqb + (p.nqb - 1 - qb) * heads + (bh - first);
  const bool active = lane * E < HD;

  float m = -INFINITY;
  for (int sp = 0; sp < p.splits; ++sp) {
    Item it;
    item_coords<true>(u * p.splits + sp, p, it);
    if (it.end(t) <= it.k0) continue;  // no key of this range is admissible for the row
    m = fmaxf(m, p.ws_lse[static_cast<size_t>(u * p.splits + sp) * kUnitRows + rin]);
  }
  float acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;
  float denom = 0.f;
  for (int sp = 0; sp < p.splits; ++sp) {
    Item it;
    item_coords<true>(u * p.splits + sp, p, it);
    if (it.end(t) <= it.k0) continue;
    const size_t slot = static_cast<size_t>(u * p.splits + sp) * kUnitRows + rin;
    const float wgt = expf(p.ws_lse[slot] - m);
    denom += wgt;
    if (active) {
      const float* src = p.ws_o + slot * HD + lane * E;
      if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y; acc[2] += wgt * x.z; acc[3] += wgt * x.w;
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) acc[i] += wgt * src[i];
      }
    }
  }
  const float inv = 1.f / denom;
  __nv_bfloat16* dst = p.o + (static_cast<size_t>(bh) * p.N + row) * HD + lane * E;
  if (active) {
#pragma unroll
    for (int i = 0; i < E; ++i) dst[i] = __float2bfloat16_rn(acc[i] * inv);
  }
  if (lane == 0 && p.lse != nullptr) p.lse[static_cast<size_t>(bh) * p.N + row] = m + logf(denom);
}

}  // namespace fa_sm103
