// fa_fwd_kernel.cuh -- the sm_103a attention forward kernel.
//
// Method: the blocked online softmax of aiml.sh "Speed up long contexts with
// FlashAttention" (lab.py, `tiled_flash_attention`): per query row a running maximum
// m, a running sum l and an accumulator rescaled by exp(m_old - m_new) when m grows,
// finished by O = acc / l.  Causal key blocks entirely above the diagonal are never
// visited and the diagonal block is masked (j <= i).
//
// GB300 mapping (not from the pages; designed for sm_103a):
//   * Work unit = one (batch*head, 256-query-row block) = two 128-row Q tiles that
//     share every K/V tile.  Persistent CTAs (one per SM) take units in a snake
//     (boustrophedon) round-robin over this order: heads in groups whose K and V fit
//     comfortably in L2, and inside a group the longest causal blocks first, so the
//     units running at one time share a few heads' K/V through L2 and the per-CTA
//     work evens out.
//   * Warp roles (640 threads = 5 warpgroups): warps 0-7 = softmax for Q tile 0,
//     warps 8-15 = softmax for Q tile 1 (two threads per query row, one per half of
//     the key columns, in the same TMEM lane quadrant and SM sub-partition), warp 16 =
//     tcgen05 MMA issuer (one lane), warp 17 = TMA producer (one lane), warps 18-19
//     idle.  5 warps per SM sub-partition leave 96 registers a thread, enough for a
//     half row of scores (64) and its packed P without spilling.
//   * Shared memory: Q0, Q1 pinned for the unit; K and V tiles stream through an
//     NSLOT-deep ring of 128-row slots filled by TMA (128/64/32-byte swizzle).
//   * Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  The
//     softmax writes P (bf16, two per column) over the first 64 columns of its S.
//   * MMA order per KV tile j: PV0(j), S0(j+1), PV1(j), S1(j+1).  tcgen05 MMAs from
//     one thread run in issue order, so when S_t(j+1) is complete PV_t(j) is too: the
//     softmax may then rescale O_t in place before publishing P_t(j+1).
//   * Lazy rescale: the reference maximum m_ref (log2 units) only moves when a tile's
//     maximum exceeds it by more than kRescaleLog2, so P <= 2^kRescaleLog2 and O is
//     rarely touched.  Two running sums: l_exact (fp32 P, for the logsumexp) and
//     l_round (the bf16-rounded P the MMA multiplies by V, used to normalise O so
//     the weights of every output row sum to one exactly as applied).
//   * Every mbarrier wait is bounded; a wait that runs out sets the CTA's abort flag
//     and the device status word, and every role then winds down without hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx_sm103.cuh"

namespace fa_sm103 {

// bit 0: a bounded wait inside the kernel ran out
__device__ unsigned int g_device_status;

constexpr int kBlockM = 128;                // query rows per Q tile (TMEM lanes)
constexpr int kBlockN = 128;                // keys per K/V tile
constexpr int kUnitRows = 2 * kBlockM;      // query rows per work unit
constexpr int kSoftmaxWarps = 16;
constexpr int kThreads = 640;               // 16 softmax warps + 1 control warpgroup
constexpr int kMmaWarp = 16;
constexpr int kLoadWarp = 17;
constexpr uint32_t kSoftmaxThreadsPerTile = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
constexpr float kRescaleLog2 = 8.0f;        // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.693147180559945309f;

template <int HD>
struct Cfg {
  static_assert(HD == 16 || HD == 32 || HD == 64 || HD == 128 || HD == 256, "head dim");
  static constexpr int W = HD < 64 ? HD : 64;          // elements per swizzled smem row
  static constexpr int SWB = 2 * W;                     // bytes per swizzled smem row
  static constexpr int NCH = HD / W;                    // row chunks across the head dim
  static constexpr int TILE_BYTES = kBlockM * HD * 2;   // one 128-row bf16 tile
  static constexpr int CHUNK_BYTES = kBlockM * SWB;     // one chunk of a tile
  static constexpr int NSLOT = HD == 128 ? 4 : 8;       // K/V ring depth
  static constexpr int SMEM_Q = 2 * TILE_BYTES;
  static constexpr int SMEM_BYTES = SMEM_Q + NSLOT * TILE_BYTES + 1024;  // + alignment pad
  static constexpr uint32_t SWZ = swizzle_code(SWB);
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(kBlockM, kBlockN, false);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(kBlockM, HD, true);
};

struct Params {
  __nv_bfloat16* o;   // [BH, N, HD]
  float* lse;         // [BH, N] or null
  int BH;             // batch * heads
  int N;              // sequence length
  int nkv;            // ceil(N / 128)
  int nqb;            // ceil(N / 256)
  int num_units;      // nqb * BH
  int splits;         // KV ranges per unit (1 = no split)
  int num_items;      // num_units * splits
  int group_heads;    // heads whose units are interleaved (K/V of a group fit in L2)
  float* ws_o;        // splits > 1: per item, normalised partial O [256 rows][HD] (fp32)
  float* ws_lse;      // splits > 1: per item, partial logsumexp [256 rows]
  int causal;
  float scale_log2;   // scale * log2(e), >= 0
  long long budget;   // cycles a single wait may take
  int inject;         // > 0: unit 0 never issues its inject-th K/V ring load
};

struct Barriers {
  uint64_t q_full, q_empty, drain;
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t slot_full[8], slot_empty[8];
  uint64_t pair[2][4];          // [tile][row quadrant]: the two halves of a row meet here
  uint32_t tmem_base;
  int abort;
};

// Unit u -> (head, first query row).  Heads are taken in groups of group_heads (the
// last group may be smaller); inside a group the highest query block of every head
// comes first, then the next block of every head, and so on.
__device__ __forceinline__ void unit_coords(int u, const Params& p, int& bh, int& row0) {
  const int per_group = p.group_heads * p.nqb;
  const int g = u / per_group;
  const int first = g * p.group_heads;
  const int heads = (p.BH - first) < p.group_heads ? (p.BH - first) : p.group_heads;
  const int r = u - g * per_group;
  const int qb = p.nqb - 1 - r / heads;
  bh = first + r % heads;
  row0 = qb * kUnitRows;
}

// The k-th unit of this CTA (snake order over the grid); may be >= num_units.
__device__ __forceinline__ int unit_of(int k) {
  const int pos = (k & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                          : static_cast<int>(blockIdx.x);
  return k * static_cast<int>(gridDim.x) + pos;
}

// Number of K/V tiles a Q tile starting at `row_start` visits (0 if it holds no row < N).
__device__ __forceinline__ int tiles_for(int row_start, const Params& p) {
  if (row_start >= p.N) return 0;
  if (!p.causal) return p.nkv;
  const int t = row_start / kBlockN + 1;  // tiles up to and including the diagonal one
  return t < p.nkv ? t : p.nkv;
}

// A work item: one unit's KV tiles [k0, k1).  Q tile t visits [k0, e[t]), which is
// empty when e[t] <= k0.  With splits = 1 an item is the whole unit.
struct Item {
  int bh, row0, k0, k1;
  int e[2];
  // e[t] without a run-time array index (which would put the struct in local memory)
  __device__ __forceinline__ int end(int t) const { return t == 0 ? e[0] : e[1]; }
};

// SPLIT = false compiles the unsplit kernel: an item is a whole unit, k0 = 0.
template <bool SPLIT = true>
__device__ __forceinline__ void item_coords(int w, const Params& p, Item& it) {
  const int u = SPLIT ? w / p.splits : w;
  const int sp = SPLIT ? w - u * p.splits : 0;
  unit_coords(u, p, it.bh, it.row0);
  const int n0 = tiles_for(it.row0, p), n1 = tiles_for(it.row0 + kBlockM, p);
  const int n = n0 > n1 ? n0 : n1;
  it.k0 = SPLIT ? sp * n / p.splits : 0;
  it.k1 = SPLIT ? (sp + 1) * n / p.splits : n;
  it.e[0] = n0 < it.k1 ? n0 : it.k1;
  it.e[1] = n1 < it.k1 ? n1 : it.k1;
}

__device__ __forceinline__ void raise_abort(Barriers& b) {
  *reinterpret_cast<volatile int*>(&b.abort) = 1;
  atomicOr(&g_device_status, 1u);
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Params& p,
                                         Barriers& b) {
  return mbar_wait_bounded(bar, parity, p.budget, &b.abort);
}

// Time-bounded wait that ignores the abort flag (used to drain in-flight async work).
__device__ __forceinline__ bool drain_bar(uint64_t* bar, uint32_t parity, const Params& p) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > p.budget) return false;
  return true;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* ptr) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
  return reinterpret_cast<uint8_t*>((a + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------------------------
// TMA producer (one lane)
// ------------------------------------------------------------------------------------
template <int HD, bool SPLIT>
__device__ void load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                          uint8_t* sQ, uint8_t* sRing, Barriers& b, const Params& p) {
  using C = Cfg<HD>;
  prefetch_tmap(tmQ);
  prefetch_tmap(tmK);
  prefetch_tmap(tmV);
  uint32_t ring = 0;          // K/V ring entries issued so far
  uint32_t units = 0;         // units whose Q was issued
  uint32_t skipped = 0xFFFFFFFFu;
  for (int k = 0; k * static_cast<int>(gridDim.x) < p.num_items; ++k) {
    const int u = unit_of(k);
    if (u >= p.num_items) continue;
    Item it;
    item_coords<SPLIT>(u, p, it);
    if (it.k1 <= it.k0) continue;  // an empty KV range (more splits than tiles)
    const int bh = it.bh, row0 = it.row0;
    // Q smem is free once the previous item's last S MMA has completed
    if (units > 0 && !wait_bar(&b.q_empty, (units - 1) & 1, p, b)) goto fail;
    mbar_arrive_expect_tx(&b.q_full, 2 * C::TILE_BYTES);
    for (int t = 0; t < 2; ++t)
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, tmQ, &b.q_full, c * C::W,
                    row0 + t * kBlockM, bh);
    ++units;
    for (int j = it.k0; j < it.k1; ++j) {
      for (int kv = 0; kv < 2; ++kv) {
        const uint32_t slot = ring % C::NSLOT, round = ring / C::NSLOT;
        if (round > 0 && !wait_bar(&b.slot_empty[slot], (round - 1) & 1, p, b)) goto fail;
        const bool skip = p.inject > 0 && u == 0 && ring + 1 == static_cast<uint32_t>(p.inject);
        if (skip) {
          skipped = ring;
        } else {
          mbar_arrive_expect_tx(&b.slot_full[slot], C::TILE_BYTES);
          const CUtensorMap* m = kv == 0 ? tmK : tmV;
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sRing + slot * C::TILE_BYTES + c * C::CHUNK_BYTES, m, &b.slot_full[slot],
                        c * C::W, j * kBlockN, bh);
        }
        ++ring;
      }
    }
  }
  goto drain;
fail:
  raise_abort(b);
drain:
  // let every load this CTA issued land before shared memory is released
  for (uint32_t i = ring > C::NSLOT ? ring - C::NSLOT : 0; i < ring; ++i)
    if (i != skipped) drain_bar(&b.slot_full[i % C::NSLOT], (i / C::NSLOT) & 1, p);
  if (units > 0) drain_bar(&b.q_full, (units - 1) & 1, p);
}

// ------------------------------------------------------------------------------------
// MMA issuer (one lane)
// ------------------------------------------------------------------------------------
template <int HD>
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_addr, uint32_t k_addr) {
  using C = Cfg<HD>;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const int ch = (kk * 16) / C::W, off = ((kk * 16) % C::W) * 2;
    const uint64_t a = smem_desc(q_addr + ch * C::CHUNK_BYTES + off, 16, 8 * C::SWB, C::SWZ);
    const uint64_t bd = smem_desc(k_addr + ch * C::CHUNK_BYTES + off, 16, 8 * C::SWB, C::SWZ);
    mma_bf16_ss(tmem_d, a, bd, C::IDESC_S, kk > 0);
  }
}

template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_addr,
                                         bool accumulate) {
  using C = Cfg<HD>;
#pragma unroll
  for (int kk = 0; kk < kBlockN / 16; ++kk) {
    // V tile is [key][d]: the B operand (K = keys, N = d) is MN-major
    const uint64_t bd = smem_desc(v_addr + kk * 16 * C::SWB, C::CHUNK_BYTES, 8 * C::SWB, C::SWZ);
    mma_bf16_ts(tmem_o, tmem_p + kk * 8, bd, C::IDESC_O, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int HD, bool SPLIT>
__device__ void mma_role(uint8_t* sQ, uint8_t* sRing, uint32_t tmem, Barriers& b, const Params& p) {
  using C = Cfg<HD>;
  uint32_t ring = 0, units = 0;
  uint32_t p_cnt[2] = {0, 0}, oe_cnt[2] = {0, 0};
  const uint32_t q_addr[2] = {smem_u32(sQ), smem_u32(sQ + C::TILE_BYTES)};
  const uint32_t col_s[2] = {kColS0, kColS1}, col_o[2] = {kColO0, kColO1};
  const uint32_t ring_addr = smem_u32(sRing);
  for (int k = 0; k * static_cast<int>(gridDim.x) < p.num_items; ++k) {
    const int u = unit_of(k);
    if (u >= p.num_items) continue;
    Item it;
    item_coords<SPLIT>(u, p, it);
    if (it.k1 <= it.k0) continue;
    const int k0 = it.k0, k1 = it.k1;
    if (!wait_bar(&b.q_full, units & 1, p, b)) goto fail;
    ++units;
    uint32_t ks = ring % C::NSLOT;
    if (!wait_bar(&b.slot_full[ks], (ring / C::NSLOT) & 1, p, b)) goto fail;
    ++ring;
    tc_fence_after_sync();
    for (int t = 0; t < 2; ++t)
      if (it.e[t] > k0) {
        issue_s<HD>(tmem + col_s[t], q_addr[t], ring_addr + ks * C::TILE_BYTES);
        mma_commit(&b.s_full[t]);
      }
    mma_commit(&b.slot_empty[ks]);
    if (k1 - k0 == 1) mma_commit(&b.q_empty);
    for (int j = k0; j < k1; ++j) {
      const uint32_t vs = ring % C::NSLOT;
      if (!wait_bar(&b.slot_full[vs], (ring / C::NSLOT) & 1, p, b)) goto fail;
      ++ring;
      const bool next = j + 1 < k1;
      if (next) {
        ks = ring % C::NSLOT;
        if (!wait_bar(&b.slot_full[ks], (ring / C::NSLOT) & 1, p, b)) goto fail;
        ++ring;
      }
      tc_fence_after_sync();
      for (int t = 0; t < 2; ++t) {
        if (j < it.e[t]) {
          if (j == k0) {  // O_t must have been read out by the previous item's epilogue
            if (!wait_bar(&b.o_empty[t], (oe_cnt[t] & 1) ^ 1, p, b)) goto fail;
            ++oe_cnt[t];
          }
          if (!wait_bar(&b.p_full[t], p_cnt[t] & 1, p, b)) goto fail;
          ++p_cnt[t];
          tc_fence_after_sync();
          issue_pv<HD>(tmem + col_o[t], tmem + col_s[t], ring_addr + vs * C::TILE_BYTES, j > k0);
          if (j == it.e[t] - 1) mma_commit(&b.o_full[t]);
        }
        if (next && j + 1 < it.e[t]) {
          issue_s<HD>(tmem + col_s[t], q_addr[t], ring_addr + ks * C::TILE_BYTES);
          mma_commit(&b.s_full[t]);
        }
      }
      mma_commit(&b.slot_empty[vs]);
      if (next) {
        mma_commit(&b.slot_empty[ks]);
        if (j + 1 == k1 - 1) mma_commit(&b.q_empty);
      }
    }
  }
  goto drain;
fail:
  raise_abort(b);
drain:
  // every MMA this thread issued has completed once this commit arrives
  mma_commit(&b.drain);
  drain_bar(&b.drain, 0, p);
}

// ------------------------------------------------------------------------------------
// softmax / epilogue (warps 0-15).  Q tile t = warp / 8.  Each query row is shared by
// two threads of the same TMEM lane quadrant (warp % 4) and SM sub-partition: the
// thread in warp w takes key columns [64h, 64h + 64) with h = (warp / 4) % 2.  The two
// halves exchange their row maxima (and, once per unit, their row sums) through
// shared memory, synchronised by a 64-arrival mbarrier per row quadrant.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Params& p,
                                          Barriers& b) {
  const bool ok = wait_bar(bar, parity, p, b);
  return __all_sync(0xFFFFFFFFu, ok);
}

// P = 2^(s*c - m) on columns [32*part, 32*part + 32) of this thread's 64 (packed f32x2
// FMA), rounded to bf16x2 into pk.  `lim` = last admissible column of the 64 (MASK).
// Returns {sum of the exact fp32 P, sum of the bf16-rounded P}.
template <bool MASK>
__device__ __forceinline__ float2 exp_pack32(const uint32_t (&s)[64], uint32_t (&pk)[16], int part,
                                             uint64_t c2, uint64_t negm2, int lim) {
  uint64_t esum = 0, rsum = 0;  // two fp32 zeros each
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
    const uint32_t w = pack_bf16x2(p0, p1);
    pk[i] = w;
    esum = add_f32x2(esum, f32x2(p0, p1));
    rsum = add_f32x2(rsum, f32x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)));
  }
  float e0, e1, r0, r1;
  f32x2_split(esum, e0, e1);
  f32x2_split(rsum, r0, r1);
  return make_float2(e0 + e1, r0 + r1);
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

// Exchange slots in shared memory (floats).
struct Xchg {
  float mx[2][2][2][kBlockM];     // [tile][parity][half][row]: partial row maxima
  float sum[2][2][2][kBlockM];    // [tile][half][exact|rounded][row]: partial row sums
};

template <int HD, bool SPLIT>
__device__ void softmax_role(uint32_t tmem, Barriers& b, Xchg& x, const Params& p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = warp >> 3, h = (warp >> 2) & 1, wq = warp & 3;
  const int lrow = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t colS = t == 0 ? kColS0 : kColS1;
  const uint32_t tS = tmem + lane_base + colS + 64 * h;  // this thread's 64 score columns
  const uint32_t tP = tmem + lane_base + colS + 32 * h;  // its 32 packed P columns
  const uint32_t tO = tmem + lane_base + (t == 0 ? kColO0 : kColO1);
  uint64_t* pair = &b.pair[t][wq];
  const float c = p.scale_log2;
  const uint64_t c2 = f32x2(c, c);
  uint32_t s_cnt = 0, o_cnt = 0, x_cnt = 0;
  for (int k = 0; k * static_cast<int>(gridDim.x) < p.num_items; ++k) {
    const int u = unit_of(k);
    if (u >= p.num_items) continue;
    Item it;
    item_coords<SPLIT>(u, p, it);
    const int e_t = it.end(t);
    if (e_t <= it.k0) continue;  // this Q tile has no key tile in the item
    const int bh = it.bh, row0 = it.row0;
    const int row_start = row0 + t * kBlockM;
    const int row = row_start + lrow;
    // admissible keys for this row: j <= last_key
    const int last_key = p.causal ? (row < p.N - 1 ? row : p.N - 1) : p.N - 1;
    float m_ref = -INFINITY;  // reference maximum, log2 units (identical in both halves)
    float l_exact = 0.f, l_round = 0.f;  // this half's partial sums
    for (int j = it.k0; j < e_t; ++j) {
      if (!warp_wait(&b.s_full[t], s_cnt & 1, p, b)) goto fail;
      tc_fence_after_sync();
      uint32_t s[64];
      tmem_ld_x64(tS, s);
      tmem_wait_ld(s);
      const int kv0 = j * kBlockN + 64 * h;
      const int lim = last_key - kv0;               // last admissible column of the 64
      const bool warp_mask = __any_sync(0xFFFFFFFFu, kv0 + 63 > last_key);
      const float pm = warp_mask ? row_max64<true>(s, lim) : row_max64<false>(s, lim);
      // combine with the other half of the row
      x.mx[t][s_cnt & 1][h][lrow] = pm;
      mbar_arrive(pair);
      if (!warp_wait(pair, x_cnt & 1, p, b)) goto fail;
      ++x_cnt;
      const float mx = fmaxf(pm, x.mx[t][s_cnt & 1][h ^ 1][lrow]);
      ++s_cnt;
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
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t pk[16];
        const float2 sums = warp_mask ? exp_pack32<true>(s, pk, part, c2, negm2, lim)
                                      : exp_pack32<false>(s, pk, part, c2, negm2, lim);
        l_exact += sums.x;
        l_round += sums.y;
        tmem_st_x16(tP + 16 * part, pk);
      }
      if (warp_rescale && j > it.k0) {
        // PV_t(j-1) has completed (S_t(j) was issued after it) and PV_t(j) waits for
        // this thread's arrival below: rescale this half's O chunks in place.
#pragma unroll
        for (int c0 = 32 * h; c0 < HD; c0 += 64) {
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
      mbar_arrive(&b.p_full[t]);
    }
    // epilogue: O = acc / l_round in bf16, lse = (m_ref + log2 l_exact) ln 2
    x.sum[t][h][0][lrow] = l_exact;
    x.sum[t][h][1][lrow] = l_round;
    mbar_arrive(pair);
    if (!warp_wait(pair, x_cnt & 1, p, b)) goto fail;
    ++x_cnt;
    l_exact += x.sum[t][h ^ 1][0][lrow];
    l_round += x.sum[t][h ^ 1][1][lrow];
    if (!warp_wait(&b.o_full[t], o_cnt & 1, p, b)) goto fail;
    ++o_cnt;
    tc_fence_after_sync();
    if constexpr (SPLIT) {
      // partial result of this KV range: normalised O (fp32) and its logsumexp
      const float inv_l = 1.f / l_round;
      const bool store = row < p.N;
      const size_t slot = static_cast<size_t>(u) * kUnitRows + t * kBlockM + lrow;
      float* orow = p.ws_o + slot * HD;
#pragma unroll
      for (int c0 = 32 * h; c0 < HD; c0 += 64) {
        uint32_t o[32];
        tmem_ld_x32(tO + c0, o);
        tmem_wait_ld(o);
        if (store) {
          constexpr int NV = HD < 32 ? HD : 32;
#pragma unroll
          for (int v4 = 0; v4 < NV; v4 += 4)
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
          constexpr int NV = HD < 32 ? HD : 32;
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
      if (h == 0 && store && p.lse != nullptr)
        p.lse[static_cast<size_t>(bh) * p.N + row] = (m_ref + lg2_approx(l_exact)) * kLn2;
    }
    tc_fence_before_sync();
    mbar_arrive(&b.o_empty[t]);
  }
  return;
fail:
  raise_abort(b);
}

// ------------------------------------------------------------------------------------
template <int HD, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::SMEM_Q;
  __shared__ Barriers b;
  __shared__ Xchg xchg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    b.abort = 0;
    mbar_init(&b.q_full, 1);
    mbar_init(&b.q_empty, 1);
    mbar_init(&b.drain, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&b.s_full[t], 1);
      mbar_init(&b.p_full[t], kSoftmaxThreadsPerTile);
      mbar_init(&b.o_full[t], 1);
      mbar_init(&b.o_empty[t], kSoftmaxThreadsPerTile);
      for (int q = 0; q < 4; ++q) mbar_init(&b.pair[t][q], 64);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&b.slot_full[s], 1);
      mbar_init(&b.slot_empty[s], 1);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&b.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = b.tmem_base;

  if (warp < kSoftmaxWarps) {
    softmax_role<HD, SPLIT>(tmem, b, xchg, p);
  } else {
    if (warp == kMmaWarp) {
      if (lane == 0) mma_role<HD, SPLIT>(sQ, sRing, tmem, b, p);
      __syncwarp();
    } else if (warp == kLoadWarp) {
      if (lane == 0) load_role<HD, SPLIT>(&tmQ, &tmK, &tmV, sQ, sRing, b, p);
      __syncwarp();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa_sm103
