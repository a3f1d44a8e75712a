// fa_fwd_1tile_kernel.cuh -- the one-Q-tile attention forward kernel (head dims 32 to 256).
//
// Same method and numerics as fa_fwd_kernel (blocked online softmax of the aiml.sh
// "Speed up long contexts with FlashAttention" lab.py `tiled_flash_attention`, lazy
// rescale, exact and bf16-rounded row sums), laid out for a 256-wide head:
//   * Tensor memory (512 columns): S buffer 0 | S buffer 1 | O (HD fp32 columns).
//     At head dim 256 two 128-row Q tiles (the other kernel's unit) would need 768
//     columns, so a work unit here is one (batch*head, 128-query-row tile).  At head
//     dims 32 to 128 the same half-size unit serves launches with too few 256-row
//     units to fill the SMs evenly (the host picks the kernel from a schedule model).
//   * The two S buffers let S(j+1) be computed while the softmax works on S(j): MMA
//     order S(0), S(1), then for each KV tile j: PV(j), S(j+2).  P(j) is written over
//     S buffer j % 2; S(j+2) reuses it only after PV(j) (MMAs of one thread run in
//     order).  An O rescale first waits for PV(j-1) through a per-PV barrier.
//   * Shared memory, filled by TMA with the 128-byte swizzle: at head dim 256 one
//     64 KB Q tile and a 2-slot ring of 64 KB K/V tiles (192 KB + 1 KB alignment); at
//     head dim 128 two 32 KB Q buffers (the next unit's Q loads during this one) and a
//     3-slot ring of 32 KB K/V tiles, each followed by a 16 KB block of bf16 ones
//     (208 KB); at 64 and 32 two Q buffers, an 8-slot ring and one ones block (176 KB
//     and 88 KB).
//   * Warps (384 threads): 0-7 softmax (each row shared by two threads, one per half
//     of the key columns, exchanging maxima and sums through shared memory), 8 MMA
//     issuer, 9 TMA producer.  Every wait is bounded and sleeps.  Warps signal the
//     barriers with one arrival each (lane 0 after __syncwarp); the sum of the rounded
//     P is taken by the PV MMA itself at head dims up to 128: 16 more output columns
//     read a block of bf16 ones (O's column HD; TMEM has room beside O there); at 256 it
//     is summed from P after P has been handed to the MMA.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa_sm103 {
namespace one {

constexpr int kUnitRows1 = kBlockM;       // one Q tile per work unit
constexpr int kSoftmaxWarps1 = 8;
constexpr int kThreads1 = 384;
constexpr int kMmaWarp1 = 8;
constexpr int kLoadWarp1 = 9;
constexpr uint32_t kColS0_1 = 0, kColS1_1 = 128, kColO_1 = 256;

template <int HD>
struct Cfg1 {
  // each output row is written by two threads in 32-column chunks: head dim >= 32
  static_assert(HD == 256 || HD == 128 || HD == 64 || HD == 32,
                "the one-tile layout serves head dims 32 to 256");
  using C = Cfg<HD>;
  static constexpr int QBUF = HD == 256 ? 1 : 2;
  static constexpr int NSLOT = HD == 256 ? 2 : HD == 128 ? 3 : 8;
  // head dims up to 64: the PV MMA's 16 extra output columns read a block of bf16 ones
  // placed after the ring (as in the two-tile kernel), so O's column HD holds the row sum
  // of the rounded P
  // (at head dim 128 every ring slot carries its own 16 KB ones block right after the tile,
  // where the descriptor's regular chunk stride puts B's third column chunk)
  static constexpr bool ONES = HD <= 128;
  static constexpr int NO = ONES ? HD + 16 : HD;  // PV MMA output columns
  static constexpr int SLOT_BYTES = C::TILE_BYTES + (HD == 128 ? C::KV_CHUNK_BYTES : 0);
  static constexpr int ONES_BYTES = (ONES && HD < 128) ? C::KV_CHUNK_BYTES : 0;  // after the ring
  static constexpr int SMEM_BYTES = QBUF * C::TILE_BYTES + NSLOT * SLOT_BYTES + ONES_BYTES + 1024;
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(kBlockM, NO, true);
};

struct Barriers1 {
  uint64_t q_full[2], q_empty[2];  // per Q buffer
  uint64_t s_full[2], p_full[2];   // per S buffer
  uint64_t pv_done;                // one completion per PV MMA group
  uint64_t o_full, o_empty, drain;
  uint64_t slot_full[8], slot_empty[8];
  uint64_t pair[4];                // [row quadrant]: the two halves of a row meet here
  uint32_t tmem_base;
  int abort;
};

struct Xchg1 {
  float mx[2][2][kBlockM];     // [parity][half][row]: partial row maxima
  float sum[2][2][kBlockM];    // [half][exact|rounded][row]: partial row sums
};

// Unit u -> (head, first query row), the grouped longest-first order of unit_coords
// with 128-row units (p.nqb = ceil(N / 128)).
__device__ __forceinline__ void unit_coords1(int u, const Params& p, int& bh, int& row0) {
  const int per_group = p.group_heads * p.nqb;
  const int g = u / per_group;
  const int first = g * p.group_heads;
  const int heads = (p.BH - first) < p.group_heads ? (p.BH - first) : p.group_heads;
  const int r = u - g * per_group;
  const int qb = p.nqb - 1 - r / heads;
  bh = first + r % heads;
  row0 = qb * kUnitRows1;
}

// Item w -> (head, first query row, key tiles [k0, k1)).  Without SPLIT an item is a
// whole unit; with SPLIT item w is piece w % splits of unit w / splits, the unit's key
// tiles cut as evenly as integers allow.  An item with k1 <= k0 (more pieces than key
// tiles) is empty and every role skips it.  Under the causal mask every key tile of a
// unit holds admissible keys for all its rows, so a non-empty piece does too.
template <bool SPLIT>
__device__ __forceinline__ void item_coords1(int w, const Params& p, int& bh, int& row0, int& k0,
                                             int& k1) {
  const int u = SPLIT ? w / p.splits : w;
  const int sp = SPLIT ? w - u * p.splits : 0;
  unit_coords1(u, p, bh, row0);
  const int n = tiles_for(row0, p);
  k0 = SPLIT ? sp * n / p.splits : 0;
  k1 = SPLIT ? (sp + 1) * n / p.splits : n;
}

// The next item after round k that this CTA takes and that has work (k advances).
template <bool SPLIT>
__device__ __forceinline__ bool next_item1(int& k, const Params& p, int& bh, int& row0, int& k0,
                                           int& k1) {
  while (++k < p.num_rounds) {
    const int u = item_of(k, p);
    if (u < 0) continue;
    item_coords1<SPLIT>(u, p, bh, row0, k0, k1);
    if (k1 > k0) return true;
  }
  return false;
}

// ------------------------------------------------------------------------------------
// half-row softmax helpers: each query row is shared by two threads, one per 64-column
// half of a 128-key score tile
// ------------------------------------------------------------------------------------
// P = 2^(s*c - m) on columns [32*part, 32*part + 32) of this thread's 64 (packed f32x2
// FMA), rounded to bf16x2 into pk[16*part .. 16*part + 15].  `lim` = last admissible
// column of the 64 (MASK).  Returns the sum of the fp32 P; the sum of the rounded P is
// taken after P has been handed to the MMA (rounded_sum32).
template <bool MASK>
__device__ __forceinline__ float exp_pack32(const uint32_t (&s)[64], uint32_t (&pk)[32], int part,
                                           uint64_t c2, uint64_t negm2, int lim) {
  uint64_t esum[2] = {0, 0};  // two fp32 zeros each
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int col = 32 * part + 2 * i;
    const uint64_t x = fma_f32x2(f32x2(__uint_as_float(s[col]), __uint_as_float(s[col + 1])), c2,
                                 negm2);
    float a0, a1;
    f32x2_split(x, a0, a1);
    float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
    if (MASK) {
      if (col > lim) p0 = 0.f;
      if (col + 1 > lim) p1 = 0.f;
    }
    pk[16 * part + i] = pack_bf16x2(p0, p1);
    esum[i & 1] = add_f32x2(esum[i & 1], f32x2(p0, p1));
  }
  float e0, e1, e2, e3;
  f32x2_split(esum[0], e0, e1);
  f32x2_split(esum[1], e2, e3);
  return (e0 + e1) + (e2 + e3);
}

// Sum of the 64 bf16 values packed in pk (exact widening, fp32 additions).
__device__ __forceinline__ float rounded_sum32(const uint32_t (&pk)[32]) {
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; ++i) a[i & 3] = add_bf16x2_to_f32(a[i & 3], pk[i]);
  return (a[0] + a[1]) + (a[2] + a[3]);
}

template <bool MASK>
__device__ __forceinline__ float row_max64(const uint32_t (&s)[64], int lim) {
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 64; i += 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float x0 = __uint_as_float(s[i + 2 * k]), x1 = __uint_as_float(s[i + 2 * k + 1]);
      if (MASK) {
        if (i + 2 * k > lim) x0 = -INFINITY;
        if (i + 2 * k + 1 > lim) x1 = -INFINITY;
      }
      m[k] = max3(m[k], x0, x1);
    }
  }
  return max3(m[0], m[1], fmaxf(m[2], m[3]));
}

__device__ __forceinline__ void raise_abort1(Barriers1& b) {
  *reinterpret_cast<volatile int*>(&b.abort) = 1;
  atomicOr(&g_device_status, 1u);
}
__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, const Params& p, Barriers1& b) {
  return mbar_wait_bounded(bar, parity, p.budget, &b.abort);
}
__device__ __forceinline__ bool warp_wait1(uint64_t* bar, uint32_t parity, const Params& p,
                                           Barriers1& b) {
  const bool ok = wait1(bar, parity, p, b);
  return __all_sync(0xFFFFFFFFu, ok);
}
// The issuer's wait: warp-wide when the whole warp runs the issuer.
template <bool WARP>
__device__ __forceinline__ bool wait1w(uint64_t* bar, uint32_t parity, const Params& p, Barriers1& b) {
  if constexpr (WARP) return warp_wait1(bar, parity, p, b);
  return wait1(bar, parity, p, b);
}

// ------------------------------------------------------------------------------------
// TMA producer (one lane).  Ring order per item of key tiles [k0, k1): K_k0, K_k0+1,
// then for j = k0 .. k1-1: V_j, K_{j+2} (the order the MMA issuer consumes).
// ------------------------------------------------------------------------------------
struct RingState1 {
  uint32_t ring = 0;
  uint32_t skipped = 0xFFFFFFFFu;
};

template <int HD>
__device__ __forceinline__ bool emit_kv1(const CUtensorMap* tm, int tile, int bh, int u,
                                         uint8_t* sRing, Barriers1& b, const Params& p,
                                         RingState1& rs) {
  using C = Cfg<HD>;
  constexpr int NS = Cfg1<HD>::NSLOT;
  const uint32_t slot = rs.ring % NS, round = rs.ring / NS;
  if (round > 0 && !wait1(&b.slot_empty[slot], (round - 1) & 1, p, b)) return false;
  const bool skip = p.inject > 0 && u == 0 && rs.ring + 1 == static_cast<uint32_t>(p.inject);
  if (skip) {
    rs.skipped = rs.ring;
  } else {
    mbar_arrive_expect_tx(&b.slot_full[slot], C::TILE_BYTES);
    for (int c = 0; c < C::NCH; ++c)
      tma_load_3d(sRing + slot * Cfg1<HD>::SLOT_BYTES + c * C::CHUNK_BYTES, tm, &b.slot_full[slot],
                  c * C::W, tile * kBlockN, bh);
  }
  ++rs.ring;
  return true;
}

template <int HD, bool SPLIT>
__device__ void load_role1(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                           uint8_t* sQ, uint8_t* sRing, Barriers1& b, const Params& p) {
  using C = Cfg<HD>;
  constexpr int QB = Cfg1<HD>::QBUF, NS = Cfg1<HD>::NSLOT;
  prefetch_tmap(tmQ);
  prefetch_tmap(tmK);
  prefetch_tmap(tmV);
  RingState1 rs;
  uint32_t units = 0;
  for (int k = 0; k < p.num_rounds; ++k) {
    const int u = item_of(k, p);
    if (u < 0) continue;
    int bh, row0, k0, k1;
    item_coords1<SPLIT>(u, p, bh, row0, k0, k1);
    if (k1 <= k0) continue;
    const uint32_t qb = units % QB;
    // this Q buffer is free once the S MMAs of the item that used it last are done
    if (units >= QB && !wait1(&b.q_empty[qb], ((units / QB) - 1) & 1, p, b)) goto fail;
    mbar_arrive_expect_tx(&b.q_full[qb], C::TILE_BYTES);
    for (int c = 0; c < C::NCH; ++c)
      tma_load_3d(sQ + qb * C::TILE_BYTES + c * C::CHUNK_BYTES, tmQ, &b.q_full[qb], c * C::W,
                  row0, bh);
    ++units;
    if (!emit_kv1<HD>(tmK, k0, bh, u, sRing, b, p, rs)) goto fail;
    if (k0 + 1 < k1 && !emit_kv1<HD>(tmK, k0 + 1, bh, u, sRing, b, p, rs)) goto fail;
    for (int j = k0; j < k1; ++j) {
      if (!emit_kv1<HD>(tmV, j, bh, u, sRing, b, p, rs)) goto fail;
      if (j + 2 < k1 && !emit_kv1<HD>(tmK, j + 2, bh, u, sRing, b, p, rs)) goto fail;
    }
  }
  goto drain;
fail:
  raise_abort1(b);
drain:
  for (uint32_t i = rs.ring > NS ? rs.ring - NS : 0; i < rs.ring; ++i)
    if (i != rs.skipped) drain_bar(&b.slot_full[i % NS], (i / NS) & 1, p);
  for (uint32_t i = units > QB ? units - QB : 0; i < units; ++i)
    drain_bar(&b.q_full[i % QB], (i / QB) & 1, p);
}

// O (+ the 16 ones columns) += P V for the one-tile kernel.  Up to head dim 64 V's one
// column chunk is followed, at the descriptor's chunk stride (ones_addr - v_addr), by the
// ones block after the ring; at 128 each slot carries its ones block right after the
// tile, where the regular chunk stride puts B's third chunk.  At 256: plain O += P V.
template <int HD, bool WARP>
__device__ __forceinline__ void issue_pv1(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_addr,
                                          bool accumulate, uint32_t ones_addr) {
  using C = Cfg<HD>;
  const uint32_t lbo = (Cfg1<HD>::ONES && C::NCH == 1) ? ones_addr - v_addr : C::KV_CHUNK_BYTES;
#pragma unroll
  for (int kk = 0; kk < kBlockN / 16; ++kk) {
    const uint64_t bd = smem_desc(v_addr + kk * 16 * C::SWB, lbo, 8 * C::SWB, C::SWZ);
    mma_bf16_ts<WARP>(tmem_o, tmem_p + kk * 8, bd, Cfg1<HD>::IDESC_O, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer (one lane)
// ------------------------------------------------------------------------------------
// WARP: run by the whole warp (one elected lane issues) or by one thread (head dim 256).
template <int HD, bool SPLIT, bool WARP>
__device__ void mma_role1(uint8_t* sQ, uint8_t* sRing, uint32_t tmem, Barriers1& b,
                          const Params& p) {
  using C = Cfg<HD>;
  constexpr int QB = Cfg1<HD>::QBUF, NS = Cfg1<HD>::NSLOT;
  uint32_t ring = 0, units = 0, oe_cnt = 0;
  uint32_t p_cnt0 = 0, p_cnt1 = 0;  // p_full completions seen, per S buffer
  const uint32_t ring_addr = smem_u32(sRing);
  // the next item is decoded after this item's first S MMAs are issued, off the boundary
  int k_nxt = -1, nbh, nrow0, nk0, nk1;
  bool has_nxt = next_item1<SPLIT>(k_nxt, p, nbh, nrow0, nk0, nk1);
  while (has_nxt) {
    const int k0 = nk0, k1 = nk1;
    const int n = k1 - k0;  // key tiles of this item; tile j of the loops is k0 + j
    const uint32_t qb = units % QB;
    const uint32_t q_addr = smem_u32(sQ + qb * C::TILE_BYTES);
    if (!wait1w<WARP>(&b.q_full[qb], (units / QB) & 1, p, b)) goto fail;
    ++units;
    // S(0) and S(1) into the two S buffers
    for (int j = 0; j < 2 && j < n; ++j) {
      const uint32_t ks = ring % NS;
      if (!wait1w<WARP>(&b.slot_full[ks], (ring / NS) & 1, p, b)) goto fail;
      ++ring;
      tc_fence_after_sync();
      issue_s<HD, kBlockN, WARP>(tmem + (j == 0 ? kColS0_1 : kColS1_1), q_addr, ring_addr + ks * Cfg1<HD>::SLOT_BYTES);
      mma_commit<WARP>(&b.s_full[j]);
      mma_commit<WARP>(&b.slot_empty[ks]);
    }
    if (n <= 2) mma_commit<WARP>(&b.q_empty[qb]);  // every S MMA of the unit is issued
    has_nxt = next_item1<SPLIT>(k_nxt, p, nbh, nrow0, nk0, nk1);
    for (int j = 0; j < n; ++j) {
      const int sb = j & 1;
      const uint32_t colS = sb == 0 ? kColS0_1 : kColS1_1;
      const uint32_t vs = ring % NS;
      if (!wait1w<WARP>(&b.slot_full[vs], (ring / NS) & 1, p, b)) goto fail;
      ++ring;
      if (j == 0) {  // O must have been read out by the previous item's epilogue
        if (!wait1w<WARP>(&b.o_empty, (oe_cnt & 1) ^ 1, p, b)) goto fail;
        ++oe_cnt;
      }
      uint32_t& p_cnt = sb == 0 ? p_cnt0 : p_cnt1;
      if (!wait1w<WARP>(&b.p_full[sb], p_cnt & 1, p, b)) goto fail;
      ++p_cnt;
      tc_fence_after_sync();
      issue_pv1<HD, WARP>(tmem + kColO_1, tmem + colS, ring_addr + vs * Cfg1<HD>::SLOT_BYTES, j > 0,
                          ring_addr + NS * Cfg1<HD>::SLOT_BYTES);
      mma_commit<WARP>(&b.pv_done);
      if (j == n - 1) mma_commit<WARP>(&b.o_full);
      mma_commit<WARP>(&b.slot_empty[vs]);
      if (j + 2 < n) {
        const uint32_t ks = ring % NS;
        if (!wait1w<WARP>(&b.slot_full[ks], (ring / NS) & 1, p, b)) goto fail;
        ++ring;
        tc_fence_after_sync();
        issue_s<HD, kBlockN, WARP>(tmem + colS, q_addr, ring_addr + ks * Cfg1<HD>::SLOT_BYTES);
        mma_commit<WARP>(&b.s_full[sb]);
        mma_commit<WARP>(&b.slot_empty[ks]);
        if (j + 2 == n - 1) mma_commit<WARP>(&b.q_empty[qb]);
      }
    }
  }
  goto drain;
fail:
  raise_abort1(b);
drain:
  mma_commit<WARP>(&b.drain);
  drain_bar(&b.drain, 0, p);
}

// ------------------------------------------------------------------------------------
// softmax / epilogue (warps 0-7)
// ------------------------------------------------------------------------------------
template <int HD, bool SPLIT>
__device__ void softmax_role1(uint32_t tmem, Barriers1& b, Xchg1& x, const Params& p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = (warp >> 2) & 1, wq = warp & 3;
  const int lrow = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tO = tmem + lane_base + kColO_1;
  uint64_t* pair = &b.pair[wq];
  const float c = p.scale_log2;
  const uint64_t c2 = f32x2(c, c);
  uint32_t s_cnt0 = 0, s_cnt1 = 0;  // s_full completions seen, per S buffer
  uint32_t o_cnt = 0, x_cnt = 0, pv_cnt = 0;
  for (int k = 0; k < p.num_rounds; ++k) {
    const int u = item_of(k, p);
    if (u < 0) continue;
    int bh, row0, k0, k1;
    item_coords1<SPLIT>(u, p, bh, row0, k0, k1);
    if (k1 <= k0) continue;
    const int n = k1 - k0;  // key tiles of this item; tile j of the loop is k0 + j
    const int row = row0 + lrow;
    const int last_key = p.causal ? (row < p.N - 1 ? row : p.N - 1) : p.N - 1;
    float m_ref = -INFINITY;
    float l_exact = 0.f, l_round = 0.f;
    for (int j = 0; j < n; ++j, ++pv_cnt) {
      const int sb = j & 1;
      const uint32_t colS = sb == 0 ? kColS0_1 : kColS1_1;
      uint32_t& s_cnt = sb == 0 ? s_cnt0 : s_cnt1;
      if (!warp_wait1(&b.s_full[sb], s_cnt & 1, p, b)) goto fail;
      ++s_cnt;
      tc_fence_after_sync();
      uint32_t s[64];
      tmem_ld_x64(tmem + lane_base + colS + 64 * h, s);
      tmem_wait_ld(s);
      const int kv0 = (k0 + j) * kBlockN + 64 * h;
      const int lim = last_key - kv0;
      const bool warp_mask = __any_sync(0xFFFFFFFFu, kv0 + 63 > last_key);
      const float pm = warp_mask ? row_max64<true>(s, lim) : row_max64<false>(s, lim);
      x.mx[x_cnt & 1][h][lrow] = pm;
      __syncwarp();
      if (lane == 0) mbar_arrive(pair);
      if (!warp_wait1(pair, x_cnt & 1, p, b)) goto fail;
      const float mx = fmaxf(pm, x.mx[x_cnt & 1][h ^ 1][lrow]);
      ++x_cnt;
      const float mt = mx * c;
      const bool need = mt > m_ref + kRescaleLog2;
      const bool warp_rescale = __any_sync(0xFFFFFFFFu, need);
      float alpha = 1.f;
      if (need) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
        m_ref = mt;
        l_exact *= alpha;
        l_round *= alpha;
      }
      const uint64_t negm2 = f32x2(-m_ref, -m_ref);
      const uint32_t tP = tmem + lane_base + colS + 32 * h;
      uint32_t pk[32];  // P as bf16 pairs, kept for the rounded row sum below
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        l_exact += warp_mask ? exp_pack32<true>(s, pk, part, c2, negm2, lim)
                             : exp_pack32<false>(s, pk, part, c2, negm2, lim);
        tmem_st_x16(tP + 16 * part, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * part]));
      }
      if (warp_rescale && j > 0) {
        // O holds the sum up to tile j-1 once PV(j-1) has completed
        if (!warp_wait1(&b.pv_done, (pv_cnt - 1) & 1, p, b)) goto fail;
        tc_fence_after_sync();
#pragma unroll
        for (int c0 = 32 * h; c0 < Cfg1<HD>::NO; c0 += 64) {  // with the ones columns
          uint32_t o[32];
          tmem_ld_x32(tO + c0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_x32(tO + c0, o);
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.p_full[sb]);
      // off the critical path: the MMA already has P
      if constexpr (!Cfg1<HD>::ONES) l_round += rounded_sum32(pk);
    }
    // epilogue: O = acc / l_round in bf16, lse = (m_ref + log2 l_exact) ln 2
    x.sum[h][0][lrow] = l_exact;
    x.sum[h][1][lrow] = l_round;
    __syncwarp();
    if (lane == 0) mbar_arrive(pair);
    if (!warp_wait1(pair, x_cnt & 1, p, b)) goto fail;
    ++x_cnt;
    l_exact += x.sum[h ^ 1][0][lrow];
    l_round += x.sum[h ^ 1][1][lrow];
    if (!warp_wait1(&b.o_full, o_cnt & 1, p, b)) goto fail;
    ++o_cnt;
    tc_fence_after_sync();
    if constexpr (Cfg1<HD>::ONES) {  // the PV MMA's ones columns: the row sum of the rounded P
      uint32_t ls[16];
      tmem_ld_x16(tO + HD, ls);
      tmem_wait_ld(ls);
      l_round = __uint_as_float(ls[0]);
    }
    if constexpr (SPLIT) {
      // this piece's normalised partial output (fp32) and the lse of its scores
      const float inv_l = 1.f / l_round;
      const bool store = row < p.N;
      const size_t slot = static_cast<size_t>(u) * kUnitRows1 + lrow;
      float* orow = p.ws_o + slot * HD;
#pragma unroll
      for (int c0 = 32 * h; c0 < HD; c0 += 64) {
        uint32_t o[32];
        tmem_ld_x32(tO + c0, o);
        tmem_wait_ld(o);
        if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 32; v4 += 4)
            *reinterpret_cast<float4*>(orow + c0 + v4) =
                make_float4(__uint_as_float(o[v4]) * inv_l, __uint_as_float(o[v4 + 1]) * inv_l,
                            __uint_as_float(o[v4 + 2]) * inv_l, __uint_as_float(o[v4 + 3]) * inv_l);
        }
      }
      if (h == 0 && store) p.ws_lse[slot] = (m_ref + lg2_approx(l_exact)) * kLn2;
    } else {
      const float inv_l = 1.f / l_round;
      const bool store = row < p.N;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N + row) * HD;
#pragma unroll
      for (int c0 = 32 * h; c0 < HD; c0 += 64) {
        uint32_t o[32];
        tmem_ld_x32(tO + c0, o);
        tmem_wait_ld(o);
        if (store) {
#pragma unroll
          for (int v8 = 0; v8 < 32; v8 += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[v8 + 0]) * inv_l, __uint_as_float(o[v8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[v8 + 2]) * inv_l, __uint_as_float(o[v8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[v8 + 4]) * inv_l, __uint_as_float(o[v8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[v8 + 6]) * inv_l, __uint_as_float(o[v8 + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c0 + v8) = w;
          }
        }
      }
      if (h == 0 && store && p.lse != nullptr)
        p.lse[static_cast<size_t>(bh) * p.N + row] = (m_ref + lg2_approx(l_exact)) * kLn2;
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&b.o_empty);
  }
  return;
fail:
  raise_abort1(b);
}

// ------------------------------------------------------------------------------------
template <int HD, bool SPLIT>
__global__ void __launch_bounds__(kThreads1, 1)
    fa_fwd_1tile_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<HD>;
  constexpr int QB = Cfg1<HD>::QBUF, NS = Cfg1<HD>::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + QB * C::TILE_BYTES;
  __shared__ Barriers1 b;
  __shared__ Xchg1 xchg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    b.abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.q_full[i], 1);
      mbar_init(&b.q_empty[i], 1);
      mbar_init(&b.s_full[i], 1);
      mbar_init(&b.p_full[i], kSoftmaxWarps1);
    }
    mbar_init(&b.pv_done, 1);
    mbar_init(&b.o_full, 1);
    mbar_init(&b.o_empty, kSoftmaxWarps1);
    mbar_init(&b.drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&b.pair[q], 2);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&b.slot_full[s], 1);
      mbar_init(&b.slot_empty[s], 1);
    }
    fence_barrier_init();
  }
  if constexpr (Cfg1<HD>::ONES) {  // bf16 1.0 everywhere in the ones blocks, seen by the tensor core
    constexpr int OB = HD == 128 ? C::KV_CHUNK_BYTES : Cfg1<HD>::ONES_BYTES;  // bytes per block
    constexpr int NB = HD == 128 ? NS : 1;                                     // blocks
    for (int i = threadIdx.x; i < NB * OB / 16; i += kThreads1) {
      const int blk = i / (OB / 16), off = i % (OB / 16);
      uint8_t* base = HD == 128 ? sRing + blk * Cfg1<HD>::SLOT_BYTES + C::TILE_BYTES
                                : sRing + NS * Cfg1<HD>::SLOT_BYTES;
      reinterpret_cast<uint4*>(base)[off] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    }
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp1) {
    tmem_alloc(&b.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = b.tmem_base;

  if (warp < kSoftmaxWarps1) {
    softmax_role1<HD, SPLIT>(tmem, b, xchg, p);
  } else if (warp == kMmaWarp1) {
    if constexpr (HD != 256)
      mma_role1<HD, SPLIT, true>(sQ, sRing, tmem, b, p);  // the whole warp; one elected lane issues
    else if (lane == 0)
      mma_role1<HD, SPLIT, false>(sQ, sRing, tmem, b, p);
    __syncwarp();
  } else if (warp == kLoadWarp1) {
    if (lane == 0) load_role1<HD, SPLIT>(&tmQ, &tmK, &tmV, sQ, sRing, b, p);
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace one
}  // namespace fa_sm103
