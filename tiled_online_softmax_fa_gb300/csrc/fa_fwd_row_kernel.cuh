// fa_fwd_row_kernel.cuh -- the attention forward kernel for head dims 16..128 with one
// softmax thread per query row.
//
// Same method, work units, TMA producer and MMA issuer as fa_fwd_kernel (the blocked
// online softmax of aiml.sh "Speed up long contexts with FlashAttention", lab.py
// `tiled_flash_attention`: running maximum, running sum, accumulator rescaled when the
// maximum grows, causal blocks above the diagonal skipped, the diagonal block masked).
// What differs is how the softmax is laid out on the SM:
//   * Warps (512 threads = 4 warpgroups): warpgroup 0 = softmax for Q tile 0,
//     warpgroup 1 = softmax for Q tile 1, warpgroup 2 = epilogue (O / l, logsumexp,
//     stores), warp 12 = tcgen05 MMA issuer (the whole warp; one elected lane issues),
//     warp 13 = TMA producer (one lane), warps 14-15 idle.  Warp w reads TMEM lane quadrant w % 4, so every SM
//     sub-partition holds one warp of each role.
//   * Each softmax thread owns one query row and all 128 key columns of a score tile:
//     the row maximum needs no exchange between threads.  Registers are moved to the
//     softmax warpgroups with setmaxnreg (176 each; epilogue 72; control 88 -- the
//     sum is exactly the 512 x 128 registers the block is launched with).
//   * The epilogue warpgroup takes the finished accumulator O_t out of TMEM while the
//     softmax warps already work on the next unit's first score tile.  Row statistics
//     (reference maximum, exact and rounded row sums) pass through shared memory,
//     double-buffered by unit parity.
// Numerics are those of fa_fwd_kernel: exp2 with the scale folded into one FMA, lazy
// rescale (threshold 8 in log2 units), P rounded to bf16 for the PV MMA, l_round (sum
// of the rounded P) normalises O, l_exact gives the logsumexp.  Up to head dim 128,
// l_round is summed from the packed P after P has been handed to the MMA, so it stays
// off the chain S ready -> P ready that the tensor core waits on.  Up to head dim 64 the
// tensor core sums it: the PV MMA runs HD + 16 output columns, the extra 16 reading a
// shared-memory block of bf16 ones, so O's column HD accumulates sum_k P_k in fp32 like
// the rest of O (TMEM has the room there), rescaled with O and read by the epilogue.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa_sm103 {
namespace rowk {

constexpr int kThreadsR = 512;
constexpr int kEpilogueWarp0 = 8;
constexpr int kMmaWarpR = 12;
constexpr int kLoadWarpR = 13;
// Barriers the softmax and epilogue warps signal take one arrival per warp (lane 0,
// after __syncwarp): 128 per-thread arrivals on one shared-memory word are serialised
// and were measured to cost ~500 cycles on the path S ready -> P ready.
constexpr uint32_t kRowWarpsPerTile = 4;
// Dynamic shared memory of a launch: split launches add the epilogue's store blocks.
template <int HD, int BN, bool SPLIT>
constexpr int row_kernel_smem() { return Cfg<HD, BN>::SMEM_BYTES + (SPLIT ? 4 * 4096 : 0); }
constexpr uint32_t kEpilogueWarps = 4;
// Registers per thread the kernel must be compiled to (512 threads x 128 = the SM's 64K),
// and the per-warpgroup shares setmaxnreg moves them to.  The shares add up to exactly
// the launch's pool: a setmaxnreg.inc that asks for more than the pool can give waits
// without a bound, so the host refuses to launch a build whose allocation differs from
// kLaunchRegs (see the register check in the host code).
constexpr int kLaunchRegs = 128;
constexpr uint32_t kRegsSoftmax = 176, kRegsEpilogue = 72, kRegsControl = 88;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsEpilogue + 128 * kRegsControl ==
                  kThreadsR * kLaunchRegs,
              "the register split must hand out exactly the launch's registers");

// Row statistics handed from a softmax thread to the epilogue thread of the same row.
struct RowStats {
  float m_ref[2][2][kBlockM];    // [tile][unit parity][row], log2 units
  float l_exact[2][2][kBlockM];
  float l_round[2][2][kBlockM];
};

// Row maximum of the BN raw scores (columns > lim masked when MASK).
template <int BN, bool MASK>
__device__ __forceinline__ float row_max(const uint32_t (&s)[BN], int lim) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = -INFINITY;
#pragma unroll
  for (int i = 0; i < BN; i += 16) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float x0 = __uint_as_float(s[i + 2 * k]), x1 = __uint_as_float(s[i + 2 * k + 1]);
      if (MASK) {
        if (i + 2 * k > lim) x0 = -INFINITY;
        if (i + 2 * k + 1 > lim) x1 = -INFINITY;
      }
      m[k] = max3(m[k], x0, x1);
    }
  }
  return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// P = 2^(s*c - m) for columns [32*part, 32*part + 32), packed to bf16x2 into
// pk[16*part .. 16*part + 15].  Returns the sum of the fp32 P; two accumulators keep
// the addition chain short.  The sum of the rounded P is taken later (rounded_sum),
// after P has been handed to the MMA.
template <int BN, bool MASK>
__device__ __forceinline__ float exp_pack32_row(const uint32_t (&s)[BN], uint32_t (&pk)[BN / 2],
                                                int part, uint64_t c2, uint64_t negm2, int lim) {
  uint64_t esum[2] = {0, 0};
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

// Sum of the BN bf16 values packed in pk (exact widening, fp32 additions).
template <int NW>
__device__ __forceinline__ float rounded_sum(const uint32_t (&pk)[NW]) {
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < NW; ++i) a[i & 3] = add_bf16x2_to_f32(a[i & 3], pk[i]);
  return (a[0] + a[1]) + (a[2] + a[3]);
}

// ------------------------------------------------------------------------------------
// softmax (warpgroups 0 and 1): thread = one query row of Q tile t = warp / 4
// ------------------------------------------------------------------------------------
template <int HD, int BN, bool SPLIT>
__device__ void softmax_row_role(uint32_t tmem, Barriers& b, RowStats& rs, const Params& p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = warp >> 2, wq = warp & 3;
  const int lrow = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lane_base + (t == 0 ? kColS0 : kColS1);
  const uint32_t tO = tmem + lane_base + (t == 0 ? kColO0 : kColO1);
  const float c = p.scale_log2;
  const uint64_t c2 = f32x2(c, c);
  uint32_t s_cnt = 0, u_cnt = 0;
  // At head dim 128 (unsplit) the next item is decoded after this item's first P is
  // handed over, when the next S is far off, so the boundary does not wait for it (+1.2 %
  // at the headline); at smaller head dims, where a step is short, and in split launches,
  // whose items are short, decoding there cost 2-4 %, so they decode at the boundary.
  // k_pre / pre: the round and item found ahead.
  constexpr bool kEarlyDecode = HD >= 128 && !SPLIT;
  int k_pre = -1;
  Item pre;
  for (int k = 0; k < p.num_rounds; ++k) {
    Item it;
    if (kEarlyDecode && k == k_pre) {
      it = pre;
    } else {
      const int u = item_of(k, p);
      if (u < 0) continue;
      item_coords<SPLIT, BN>(u, p, it);
    }
    const int e_t = it.end(t);
    if (e_t <= it.k0) continue;  // this Q tile has no key tile in the item
    const int row = it.row0 + t * kBlockM + lrow;
    // admissible keys for this row: j <= last_key
    const int last_key = p.causal ? (row < p.N - 1 ? row : p.N - 1) : p.N - 1;
    float m_ref = -INFINITY;  // reference maximum, log2 units
    float l_exact = 0.f, l_round = 0.f;
    for (int j = it.k0; j < e_t; ++j) {
      if (!warp_wait(&b.s_full[t], s_cnt & 1, p, b)) goto fail;
      ++s_cnt;
      tc_fence_after_sync();
      uint32_t s[BN];
#pragma unroll
      for (int h = 0; h < BN; h += 64) tmem_ld_x64(tS + h, *reinterpret_cast<uint32_t(*)[64]>(&s[h]));
      tmem_wait_ld(s);
      const int kv0 = j * BN;
      const int lim = last_key - kv0;  // last admissible column of the tile
      const bool warp_mask = __any_sync(0xFFFFFFFFu, kv0 + BN - 1 > last_key);
      const float mx = warp_mask ? row_max<BN, true>(s, lim) : row_max<BN, false>(s, lim);
      const float mt = mx * c;
      const bool need = mt > m_ref + kRescaleLog2;  // also true while m_ref is -inf
      const bool warp_rescale = __any_sync(0xFFFFFFFFu, need);
      float alpha = 1.f;
      if (need) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
        m_ref = mt;
        l_exact *= alpha;
        l_round *= alpha;
      }
      const uint64_t negm2 = f32x2(-m_ref, -m_ref);
      uint32_t pk[BN / 2];  // P as bf16 pairs, kept for the rounded row sum below
#pragma unroll
      for (int part = 0; part < BN / 32; ++part) {
        l_exact += warp_mask ? exp_pack32_row<BN, true>(s, pk, part, c2, negm2, lim)
                             : exp_pack32_row<BN, false>(s, pk, part, c2, negm2, lim);
        // P (bf16 pairs) over the first BN/2 columns of S
        tmem_st_x16(tS + 16 * part, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * part]));
      }
      if (warp_rescale && j > it.k0) {
        // PV_t(j-1) has completed (S_t(j) was issued after it) and PV_t(j) waits for
        // this thread's arrival below: rescale this row of O in place (with the ones
        // columns, which hold the row sum, at head dims up to 64).
#pragma unroll
        for (int c0 = 0; c0 < Cfg<HD, BN>::NO; c0 += 32) {
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
      if (lane == 0) mbar_arrive(&b.p_full[t]);
      // off the critical path: the MMA already has P, the next S is not ready yet
      if (kEarlyDecode && j == it.k0) {
        int kk = k, u_pre;
        if (!next_item<SPLIT, BN>(kk, p, pre, u_pre)) kk = p.num_rounds;
        k_pre = kk;
      }
      if constexpr (!Cfg<HD, BN>::ONES) l_round += rounded_sum(pk);
    }
    {
      // hand the row statistics to the epilogue (buffer = parity of this tile's units)
      const int par = u_cnt & 1;
      rs.m_ref[t][par][lrow] = m_ref;
      rs.l_exact[t][par][lrow] = l_exact;
      rs.l_round[t][par][lrow] = l_round;
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.stats_full[t][par]);
      ++u_cnt;
    }
    if (kEarlyDecode) k = k_pre - 1;  // the rounds before k_pre hold no work
  }
  return;
fail:
  raise_abort(b);
}

// ------------------------------------------------------------------------------------
// Coalesced stores of a split item's fp32 partial output.  Each lane holds one row, so
// a direct store would touch 32 rows with 16 bytes each; instead a warp passes the rows
// through a 4 KB shared-memory block of its own and writes whole 128-byte row pieces.
// ------------------------------------------------------------------------------------
constexpr int kEpiScratchBytes = 4096;  // per epilogue warp: 32 rows x 128 bytes

// A warp's 32-row block (one row per lane) of RB bytes per row in its scratch: lane l
// puts 16-byte piece c of row l with stage_piece (pieces rotated by row, piece_rot, so
// the 8 lanes of a shared-memory phase hit the 8 16-byte bank groups of a 128-byte line
// once each), then flush_rows reads the block back
// with consecutive lanes on consecutive pieces of one row and writes whole rows: one
// warp store covers 32*16/RB rows of RB contiguous bytes.  Rows >= rows_valid are not
// written; gbase = first row's first byte, stride = bytes between rows in global memory.
template <int RB>
__device__ __forceinline__ int piece_rot(int r) {  // rows sharing a 128-byte line rotate alike
  return (r / (128 / RB)) % (RB / 16);
}

template <int RB>
__device__ __forceinline__ void stage_piece(uint32_t scratch, int lane, int c, uint32_t a,
                                            uint32_t b, uint32_t cc, uint32_t d) {
  st_shared_v4(scratch + lane * RB + ((c ^ piece_rot<RB>(lane)) * 16), a, b, cc, d);
}

template <int RB>
__device__ __forceinline__ void flush_rows(uint32_t scratch, int lane, uint8_t* gbase, size_t stride,
                                           int rows_valid) {
  constexpr int P = RB / 16;   // 16-byte pieces per row
  constexpr int RPI = 32 / P;  // rows one warp store covers
  __syncwarp();
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int rr = i * RPI + lane / P, c = lane % P;
    uint4 x;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                 : "r"(scratch + rr * RB + ((c ^ piece_rot<RB>(rr)) * 16)));
    if (rr < rows_valid) *reinterpret_cast<uint4*>(gbase + rr * stride + c * 16) = x;
  }
  __syncwarp();  // the block is reused by the warp's next chunk
}

// ------------------------------------------------------------------------------------
// epilogue (warpgroup 2): thread = one row of the Q tile being finished.  O = acc /
// l_round rounded to bf16 (or, for a split item, the normalised fp32 partial O), and
// lse = (m_ref + log2 l_exact) ln 2.
// ------------------------------------------------------------------------------------
template <int HD, int BN, bool SPLIT>
__device__ void epilogue_role(uint32_t tmem, Barriers& b, RowStats& rs, const Params& p,
                              uint8_t* sScratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int lrow = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t scratch = smem_u32(sScratch) + wq * kEpiScratchBytes;  // split items only
  uint32_t cnt[2] = {0, 0};  // units finished per Q tile
  for (int k = 0; k < p.num_rounds; ++k) {
    const int u = item_of(k, p);
    if (u < 0) continue;
    Item it;
    item_coords<SPLIT, BN>(u, p, it);
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {
      if (it.end(t) <= it.k0) continue;
      const uint32_t c = t == 0 ? cnt[0] : cnt[1];
      if (t == 0) ++cnt[0]; else ++cnt[1];
      const int par = c & 1;
      if (!warp_wait(&b.stats_full[t][par], (c >> 1) & 1, p, b)) goto fail;
      const float m_ref = rs.m_ref[t][par][lrow];
      const float l_exact = rs.l_exact[t][par][lrow];
      float l_round = rs.l_round[t][par][lrow];
      if (!warp_wait(&b.o_full[t], c & 1, p, b)) goto fail;
      tc_fence_after_sync();
      const uint32_t tO = tmem + lane_base + (t == 0 ? kColO0 : kColO1);
      if constexpr (Cfg<HD, BN>::ONES) {  // the PV MMA's ones columns: sum of the bf16 P
        uint32_t ls[16];
        tmem_ld_x16(tO + HD, ls);
        tmem_wait_ld(ls);
        l_round = __uint_as_float(ls[0]);
      }
      const int row = it.row0 + t * kBlockM + lrow;
      const bool store = row < p.N;
      const float inv_l = 1.f / l_round;
      constexpr int NV = HD < 32 ? HD : 32;  // columns of O per 32-column TMEM load
      if constexpr (SPLIT) {
        // normalised fp32 partial O: chunks of 32 columns (128 bytes per row), read from
        // TMEM 16 columns at a time
        constexpr int CW = HD < 32 ? HD : 32;
        const int row0w = it.row0 + t * kBlockM + wq * 32;  // the warp's first row
        const size_t slot0 = static_cast<size_t>(u) * kUnitRows + t * kBlockM + wq * 32;
        uint8_t* gbase = reinterpret_cast<uint8_t*>(p.ws_o + slot0 * HD);
#pragma unroll 1
        for (int c0 = 0; c0 < HD; c0 += CW) {
#pragma unroll
          for (int h = 0; h < CW; h += 16) {
            uint32_t o[16];
            tmem_ld_x16(tO + c0 + h, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              stage_piece<CW * 4>(scratch, lane, h / 4 + q,
                                  __float_as_uint(__uint_as_float(o[4 * q + 0]) * inv_l),
                                  __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv_l),
                                  __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv_l),
                                  __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv_l));
          }
          flush_rows<CW * 4>(scratch, lane, gbase + c0 * 4, static_cast<size_t>(HD) * 4, p.N - row0w);
        }
        if (store) p.ws_lse[slot0 + lane] = (m_ref + lg2_approx(l_exact)) * kLn2;
      } else {
        __nv_bfloat16* orow = p.o + (static_cast<size_t>(it.bh) * p.N + row) * HD;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(tO + c0, o);
          tmem_wait_ld(o);
          if (store) {
#pragma unroll
            for (int v8 = 0; v8 < NV; v8 += 8) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[v8 + 0]) * inv_l, __uint_as_float(o[v8 + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(o[v8 + 2]) * inv_l, __uint_as_float(o[v8 + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(o[v8 + 4]) * inv_l, __uint_as_float(o[v8 + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(o[v8 + 6]) * inv_l, __uint_as_float(o[v8 + 7]) * inv_l);
              *reinterpret_cast<uint4*>(orow + c0 + v8) = w;
            }
          }
        }
        if (store && p.lse != nullptr)
          p.lse[static_cast<size_t>(it.bh) * p.N + row] = (m_ref + lg2_approx(l_exact)) * kLn2;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.o_empty[t]);
    }
  }
  return;
fail:
  raise_abort(b);
}

// ------------------------------------------------------------------------------------
template <int HD, int BN, bool SPLIT>
__global__ void __launch_bounds__(kThreadsR, 1)
    fa_fwd_row_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Params p) {
  static_assert(HD <= 128, "the row kernel serves head dims 16..128");
  using C = Cfg<HD, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::SMEM_Q;
  uint8_t* sScratch = sRing + C::NSLOT * C::KV_TILE_BYTES + C::ONES_BYTES;  // split launches: epilogue store blocks
  __shared__ Barriers b;
  __shared__ RowStats rs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    b.abort = 0;
    mbar_init(&b.q_full, 1);
    mbar_init(&b.q_empty, 1);
    mbar_init(&b.drain, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&b.s_full[t], 1);
      mbar_init(&b.p_full[t], kRowWarpsPerTile);
      mbar_init(&b.o_full[t], 1);
      mbar_init(&b.o_empty[t], kEpilogueWarps);
      mbar_init(&b.stats_full[t][0], kRowWarpsPerTile);
      mbar_init(&b.stats_full[t][1], kRowWarpsPerTile);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&b.slot_full[s], 1);
      mbar_init(&b.slot_empty[s], 1);
    }
    fence_barrier_init();
  }
  if constexpr (C::ONES) {  // bf16 1.0 everywhere in the ones block, seen by the tensor core
    uint4* ones = reinterpret_cast<uint4*>(sRing + C::NSLOT * C::KV_TILE_BYTES);
    for (int i = threadIdx.x; i < C::ONES_BYTES / 16; i += kThreadsR)
      ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarpR) {
    tmem_alloc(&b.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = b.tmem_base;

  if (warp < kEpilogueWarp0) {
    setmaxnreg_inc<kRegsSoftmax>();
    softmax_row_role<HD, BN, SPLIT>(tmem, b, rs, p);
    setmaxnreg_dec<128>();
  } else if (warp < kMmaWarpR) {
    setmaxnreg_dec<kRegsEpilogue>();
    epilogue_role<HD, BN, SPLIT>(tmem, b, rs, p, sScratch);
    setmaxnreg_inc<128>();
  } else {
    setmaxnreg_dec<kRegsControl>();
    if (warp == kMmaWarpR) {
      mma_role<HD, BN, SPLIT>(sQ, sRing, tmem, b, p);
      __syncwarp();
    } else if (warp == kLoadWarpR) {
      if (lane == 0) load_role<HD, BN, SPLIT>(&tmQ, &tmK, &tmV, sQ, sRing, b, p);
      __syncwarp();
    }
    setmaxnreg_inc<128>();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarpR) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace rowk
}  // namespace fa_sm103
