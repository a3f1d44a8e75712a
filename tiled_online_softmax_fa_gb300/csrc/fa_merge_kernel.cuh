// fa_merge_kernel.cuh -- combines the per-KV-range partial results of a split launch.
//
// For one query row, KV range s produced a normalised partial output O_s and the
// logsumexp lse_s of its scores.  The full softmax over the union of the ranges is
//     lse = ln sum_s exp(lse_s),    O = sum_s exp(lse_s - lse) O_s
// (each range's weights sum to one, so exp(lse_s - lse) is that range's share of the
// row's total probability mass).  One warp per row, coalesced loads.  The kernel is as
// much instruction- as memory-bound: the row's unit and each piece's key range come from
// 32-bit arithmetic on the row's query block, and the weights and lse from ex2 / lg2.
#pragma once

#include <cuda_bf16.h>

#include "fa_fwd_1tile_kernel.cuh"
#include "fa_fwd_kernel.cuh"

namespace fa_sm103 {

constexpr int kMergeThreads = 256;  // 8 rows per block
constexpr float kLog2e = 1.4426950408889634f;

// E consecutive fp32 values of a partial output (E = 1, 2, 4 or 8 per lane).
template <int E>
__device__ __forceinline__ void load_partial(const float* src, float (&x)[E]) {
  if constexpr (E == 8) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(src));
    const float4 c = __ldcs(reinterpret_cast<const float4*>(src + 4));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  } else if constexpr (E == 4) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(src));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else if constexpr (E == 2) {
    const float2 v = __ldcs(reinterpret_cast<const float2*>(src));
    x[0] = v.x; x[1] = v.y;
  } else {
    x[0] = __ldcs(src);
  }
}

// The merge of one query row, in two halves so that a warp can put the loads of several
// rows in flight before it needs any of them (merge_load, then merge_finish).
struct MergeRow {
  int bh, row, rin, t, qb;
  size_t base;  // the row's first piece (item index)
  bool valid;   // row < BH * N
};

template <int UNIT_ROWS>
__device__ __forceinline__ MergeRow merge_row(const Params& p, int64_t gw) {
  MergeRow r;
  const int64_t rows = static_cast<int64_t>(p.BH) * p.N;
  r.valid = gw < rows;
  if (!r.valid) gw = 0;
  if (rows <= 0x7FFFFFFF) {  // 32-bit division where the row count allows (a 64-bit one is a call)
    r.bh = static_cast<int>(static_cast<uint32_t>(gw) / static_cast<uint32_t>(p.N));
    r.row = static_cast<int>(gw) - r.bh * p.N;
  } else {
    r.bh = static_cast<int>(gw / p.N);
    r.row = static_cast<int>(gw - static_cast<int64_t>(r.bh) * p.N);
  }
  const int qb = r.row / UNIT_ROWS;
  r.qb = qb;
  r.rin = r.row - qb * UNIT_ROWS;
  r.t = r.rin / kBlockM;
  // unit of (bh, qb): the inverse of unit_coords
  const int g = r.bh / p.group_heads, first = g * p.group_heads;
  const int heads = (p.BH - first) < p.group_heads ? (p.BH - first) : p.group_heads;
  const int u = g * p.group_heads * p.nqb + (p.nqb - 1 - qb) * heads + (r.bh - first);
  r.base = static_cast<size_t>(u) * p.splits;
  return r;
}

// One warp per query row.  The row's pieces are found in the lanes (lane s holds piece s
// and s + 32): their lse values give the row maximum and the weights exp(lse_s - m)
// through two warp reductions.  Each lane reads its E columns of every piece and writes
// its E bf16 outputs with one vector store.  With at most NP pieces (NP = 2 or 8; the
// host picks the smallest that holds the launch's split count) the partial outputs are
// loaded before the lse values are known, so a row costs one memory round trip instead
// of two, and the registers for them are sized to NP; NP = 0 loads each piece once its
// weight is known.  With R = 2 a warp merges two consecutive rows, all of their loads
// issued before either row is finished (measured slower than R = 1; the host launches
// R = 1).  At head dims up to 128 the host takes fa_merge2_kernel (below) for up to four
// pieces and this kernel for more, or for head dim 256.  A piece without an
// admissible key for the row (its key range starts past the row's diagonal tile, its
// partial never written) has weight 0 and its loaded values are not used.
// UNIT_ROWS: the query rows of the split kernel's work unit -- kUnitRows (two-tile
// kernel: a piece may hold no admissible key for tile 0's rows) or kUnitRows1 (one-tile
// kernel: every non-empty piece holds some).  BN: the key-tile width of the split kernel
// (its pieces are ranges of key tiles).
template <int HD, int UNIT_ROWS, int NP, int BN = kBlockN, int R = 1>
__global__ void __launch_bounds__(kMergeThreads)
    fa_merge_kernel(const Params p) {
  static_assert(HD <= 256, "head dims 16 to 256");
  constexpr int E = HD >= 256 ? 8 : (HD >= 128 ? 4 : (HD >= 64 ? 2 : 1));  // per lane
  constexpr int kLanes = HD / E;                          // lanes that hold columns
  constexpr bool eager = NP > 0;
  const int lane = threadIdx.x & 31;
  const int64_t gw0 = (static_cast<int64_t>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5)) * R;
  const bool active = lane < kLanes;
  MergeRow mr[R];
  float xe[R][eager ? NP : 1][E];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    mr[r] = merge_row<UNIT_ROWS>(p, gw0 + r);
    if (eager && active && mr[r].valid) {
#pragma unroll
      for (int sp = 0; sp < (eager ? NP : 1); ++sp)
        if (sp < p.splits)
          load_partial<E>(p.ws_o + ((mr[r].base + sp) * UNIT_ROWS + mr[r].rin) * HD + lane * E,
                          xe[r][sp]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!mr[r].valid) continue;  // warp-uniform
    const MergeRow& m0 = mr[r];
    // pieces s = lane and lane + 32: their lse, or -inf without an admissible key
    float ls[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int sp = lane + 32 * h;
      if (sp < p.splits) {
        // piece sp of the row's unit holds an admissible key for the row's Q tile (the
        // kernels' item_coords, from the row's query block)
        bool holds;
        if constexpr (UNIT_ROWS == kUnitRows) {
          const int row0 = m0.qb * kUnitRows;
          const int n0 = tiles_for<BN>(row0, p), n1 = tiles_for<BN>(row0 + kBlockM, p);
          const int n = n0 > n1 ? n0 : n1;
          const int k0 = sp * n / p.splits, k1 = (sp + 1) * n / p.splits;
          const int nt = m0.t == 0 ? n0 : n1;
          holds = (nt < k1 ? nt : k1) > k0;
        } else {
          const int n = tiles_for(m0.qb * one::kUnitRows1, p);
          holds = (sp + 1) * n / p.splits > sp * n / p.splits;
        }
        if (holds) ls[h] = p.ws_lse[(m0.base + sp) * UNIT_ROWS + m0.rin];
      }
    }
    float m = fmaxf(ls[0], ls[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    float w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) w[h] = ls[h] == -INFINITY ? 0.f : ex2_approx((ls[h] - m) * kLog2e);
    float denom = w[0] + w[1];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xFFFFFFFFu, denom, off);

    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    if constexpr (eager) {
#pragma unroll
      for (int sp = 0; sp < NP; ++sp) {
        if (sp >= p.splits) break;
        const float wgt = __shfl_sync(0xFFFFFFFFu, w[0], sp);
        if (wgt != 0.f && active) {
#pragma unroll
          for (int i = 0; i < E; ++i) acc[i] += wgt * xe[r][sp][i];
        }
      }
    } else {
#pragma unroll 4
      for (int sp = 0; sp < p.splits; ++sp) {
        const float wgt = __shfl_sync(0xFFFFFFFFu, sp < 32 ? w[0] : w[1], sp & 31);
        if (wgt != 0.f && active) {
          float x[E];
          load_partial<E>(p.ws_o + ((m0.base + sp) * UNIT_ROWS + m0.rin) * HD + lane * E, x);
#pragma unroll
          for (int i = 0; i < E; ++i) acc[i] += wgt * x[i];
        }
      }
    }
    const float inv = 1.f / denom;
    if (active) {
      __nv_bfloat16* dst = p.o + (static_cast<size_t>(m0.bh) * p.N + m0.row) * HD + lane * E;
      if constexpr (E == 8) {
        uint4 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(dst) = v;
      } else if constexpr (E == 4) {
        uint2 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = v;
      } else if constexpr (E == 2) {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      } else {
        dst[0] = __float2bfloat16_rn(acc[0] * inv);
      }
    }
    if (lane == 0 && p.lse != nullptr)
      p.lse[static_cast<size_t>(m0.bh) * p.N + m0.row] = m + lg2_approx(denom) * kLn2;
  }
}


// Merge of up to NP pieces with two rows per warp (head dims up to 128): each half-warp
// takes one row, 16 lanes x HD/16 columns, so one instruction stream serves two rows.
// Otherwise the same arithmetic as fa_merge_kernel with NP up-front pieces.
template <int HD, int UNIT_ROWS, int BN, int NP = 2>
__global__ void __launch_bounds__(kMergeThreads)
    fa_merge2_kernel(const Params p) {
  static_assert(HD <= 128, "head dims 16 to 128");
  constexpr int E = HD / 16;  // columns per lane
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5)) * 2 + half;
  const MergeRow m0 = merge_row<UNIT_ROWS>(p, gw);
  float x[NP][E];
#pragma unroll
  for (int sp = 0; sp < NP; ++sp)
    if (sp < p.splits && m0.valid)
      load_partial<E>(p.ws_o + ((m0.base + sp) * UNIT_ROWS + m0.rin) * HD + hl * E, x[sp]);
  // piece hl (lanes 0 and 1 of the half): its lse, or -inf without an admissible key
  float ls = -INFINITY;
  if (hl < p.splits && m0.valid) {
    bool holds;
    if constexpr (UNIT_ROWS == kUnitRows) {
      const int row0 = m0.qb * kUnitRows;
      const int n0 = tiles_for<BN>(row0, p), n1 = tiles_for<BN>(row0 + kBlockM, p);
      const int n = n0 > n1 ? n0 : n1;
      const int k0 = hl * n / p.splits, k1 = (hl + 1) * n / p.splits;
      const int nt = m0.t == 0 ? n0 : n1;
      holds = (nt < k1 ? nt : k1) > k0;
    } else {
      const int n = tiles_for(m0.qb * one::kUnitRows1, p);
      holds = (hl + 1) * n / p.splits > hl * n / p.splits;
    }
    if (holds) ls = p.ws_lse[(m0.base + hl) * UNIT_ROWS + m0.rin];
  }
  float mx = ls;
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  float w = ls == -INFINITY ? 0.f : ex2_approx((ls - mx) * kLog2e);
  float denom = w;
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) denom += __shfl_xor_sync(0xFFFFFFFFu, denom, off);
  float wp[NP];
#pragma unroll
  for (int sp = 0; sp < NP; ++sp) wp[sp] = __shfl_sync(0xFFFFFFFFu, w, half * 16 + sp);
  if (!m0.valid) return;
  float acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;
#pragma unroll
  for (int sp = 0; sp < NP; ++sp)
    if (sp < p.splits && wp[sp] != 0.f) {
#pragma unroll
      for (int i = 0; i < E; ++i) acc[i] += wp[sp] * x[sp][i];
    }
  const float inv = 1.f / denom;
  __nv_bfloat16* dst = p.o + (static_cast<size_t>(m0.bh) * p.N + m0.row) * HD + hl * E;
  if constexpr (E == 8) {
    uint4 v;
    v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(dst) = v;
  } else if constexpr (E == 4) {
    uint2 v;
    v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = v;
  } else if constexpr (E == 2) {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    dst[0] = __float2bfloat16_rn(acc[0] * inv);
  }
  if (hl == 0 && p.lse != nullptr)
    p.lse[static_cast<size_t>(m0.bh) * p.N + m0.row] = mx + lg2_approx(denom) * kLn2;
}

}  // namespace fa_sm103
