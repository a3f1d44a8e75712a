// fa_fwd_kernel.cuh -- pieces shared by the sm_103a attention forward kernels: launch
// parameters, work units and their order, the mbarrier set, the TMA producer and the
// tcgen05 MMA issuer of the two-Q-tile kernel (fa_fwd_row_kernel.cuh).
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
constexpr int kBlockN = 128;                // keys per K/V tile (the two-tile kernel also runs 64)
constexpr int kUnitRows = 2 * kBlockM;      // query rows per work unit
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
constexpr float kRescaleLog2 = 8.0f;        // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.693147180559945309f;

// Tile shapes for head dim HD and key tiles of BN keys (BN = 128, or 64 on the two-tile
// kernel).  Q tiles are always 128 rows; K and V tiles are BN rows.
template <int HD, int BN = kBlockN>
struct Cfg {
  static_assert(HD == 16 || HD == 32 || HD == 64 || HD == 128 || HD == 256, "head dim");
  static_assert(BN == 64 || BN == 128, "key tile width");
  static constexpr int W = HD < 64 ? HD : 64;          // elements per swizzled smem row
  static constexpr int SWB = 2 * W;                     // bytes per swizzled smem row
  static constexpr int NCH = HD / W;                    // row chunks across the head dim
  static constexpr int TILE_BYTES = kBlockM * HD * 2;   // one 128-row bf16 tile (Q)
  static constexpr int CHUNK_BYTES = kBlockM * SWB;     // one chunk of a Q tile
  static constexpr int KV_TILE_BYTES = BN * HD * 2;     // one K or V tile
  static constexpr int KV_CHUNK_BYTES = BN * SWB;       // one chunk of a K or V tile
  // K/V ring: 4 x 32 KB at HD = 128 and BN = 128, otherwise as many tiles as fit 128 KB
  // (at most 8)
  static constexpr int NSLOT = (HD == 128 && BN == 128) ? 4
                               : ((128 * 1024) / KV_TILE_BYTES < 8 ? (128 * 1024) / KV_TILE_BYTES : 8);
  static constexpr int SMEM_Q = 2 * TILE_BYTES;
  // Two-tile kernel, head dims up to 64: the PV MMA runs NO = HD + 16 output columns, the
  // last 16 reading a block of bf16 ones placed after the ring (ONES_BYTES, one V column
  // chunk), so O's column HD accumulates the row sum of the rounded P.  The one-tile
  // kernel sizes its own shared memory and does not use these.
  static constexpr bool ONES = HD <= 64;
  static constexpr int NO = ONES ? HD + 16 : HD;
  static constexpr int ONES_BYTES = ONES ? KV_CHUNK_BYTES : 0;
  static constexpr int SMEM_BYTES = SMEM_Q + NSLOT * KV_TILE_BYTES + ONES_BYTES + 1024;  // + alignment pad
  static constexpr uint32_t SWZ = swizzle_code(SWB);
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(kBlockM, BN, false);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(kBlockM, HD, true);
  static constexpr uint32_t IDESC_O_ONES = idesc_bf16_f32(kBlockM, NO, true);
  // the ones block's offset from any V tile must fit the descriptor's 14-bit stride field
  static_assert(!ONES || NSLOT * KV_TILE_BYTES < (1 << 18), "ones block out of descriptor reach");
};

struct Params {
  __nv_bfloat16* o;   // [BH, N, HD]
  float* lse;         // [BH, N] or null
  int BH;             // batch * heads
  int N;              // sequence length
  int nkv;            // ceil(N / key tile width)
  int nqb;            // ceil(N / 256)
  int num_units;      // nqb * BH
  int splits;         // KV ranges per unit (1 = no split)
  int num_items;      // num_units * splits
  int group_heads;    // heads whose units are interleaved (K/V of a group fit in L2)
  int order;          // item order over the grid: 0 one snake, 1 / 2 a snake per head group
  int group_shift;    // order 2: CTA offset added per group (mod gridDim.x)
  int group_items;    // items of a full head group (group_heads * nqb * splits)
  int rounds_per_group;  // order 1: ceil(group_items / gridDim.x)
  int num_rounds;     // rounds every role iterates over
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
  uint64_t stats_full[2][2];    // [tile][unit parity]: row statistics handed to the epilogue
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

// The item this CTA takes in round k (0 <= k < num_rounds), or -1.  Items are numbered
// in the grouped longest-first order of unit_coords (the pieces of a split unit next to
// each other); G = gridDim.x.
//   order 0: one snake over all items -- round k gives CTA c item k G + c (k even) or
//            k G + G - 1 - c (k odd);
//   order 1: that snake restarted in every head group, with the CTA order mirrored in
//            odd groups, so the CTAs that took the light end of one group's last round
//            take the heaviest items of the next.  Each group then balances by itself.
//   order 2: the snake restarted in every head group, group g's positions shifted by
//            g * group_shift CTAs: each group starts right after the CTAs that took its
//            predecessor's part-filled last round (all full groups fill that round alike).
__device__ __forceinline__ int item_of(int k, const Params& p) {
  const int G = static_cast<int>(gridDim.x), c0 = static_cast<int>(blockIdx.x);
  if (p.order == 0) {
    const int i = k * G + ((k & 1) ? G - 1 - c0 : c0);
    return i < p.num_items ? i : -1;
  }
  const int g = k / p.rounds_per_group, kg = k - g * p.rounds_per_group;
  int c;
  if (p.order == 1) {
    c = (g & 1) ? G - 1 - c0 : c0;
  } else {
    // 32-bit arithmetic only: (g mod G) * group_shift < G^2 (G <= 1024 CTAs); a 64-bit
    // remainder here compiles to a subroutine call in every role's loop
    c = c0 - ((g % G) * p.group_shift) % G;
    if (c < 0) c += G;
  }
  const int i = kg * G + ((kg & 1) ? G - 1 - c : c);
  const int base = g * p.group_items;
  const int n = p.num_items - base < p.group_items ? p.num_items - base : p.group_items;
  return i < n ? base + i : -1;
}

// Number of K/V tiles (BN keys each) a 128-row Q tile starting at `row_start` visits (0 if
// it holds no row < N).
template <int BN = kBlockN>
__device__ __forceinline__ int tiles_for(int row_start, const Params& p) {
  if (row_start >= p.N) return 0;
  if (!p.causal) return p.nkv;
  const int t = (row_start + kBlockM - 1) / BN + 1;  // tiles up to and including the diagonal one
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
template <bool SPLIT = true, int BN = kBlockN>
__device__ __forceinline__ void item_coords(int w, const Params& p, Item& it) {
  const int u = SPLIT ? w / p.splits : w;
  const int sp = SPLIT ? w - u * p.splits : 0;
  unit_coords(u, p, it.bh, it.row0);
  const int n0 = tiles_for<BN>(it.row0, p), n1 = tiles_for<BN>(it.row0 + kBlockM, p);
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

// A bounded wait taken by a whole warp: true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Params& p,
                                          Barriers& b) {
  const bool ok = wait_bar(bar, parity, p, b);
  return __all_sync(0xFFFFFFFFu, ok);
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

// The next item after round k that this CTA takes and that has work (k advances).
template <bool SPLIT, int BN>
__device__ __forceinline__ bool next_item(int& k, const Params& p, Item& it, int& u) {
  while (++k < p.num_rounds) {
    u = item_of(k, p);
    if (u < 0) continue;
    item_coords<SPLIT, BN>(u, p, it);
    if (it.k1 > it.k0) return true;  // not an empty KV range (more splits than tiles)
  }
  return false;
}

// ------------------------------------------------------------------------------------
// TMA producer (one lane)
// ------------------------------------------------------------------------------------
template <int HD, int BN, bool SPLIT>
__device__ void load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                          uint8_t* sQ, uint8_t* sRing, Barriers& b, const Params& p) {
  using C = Cfg<HD, BN>;
  prefetch_tmap(tmQ);
  prefetch_tmap(tmK);
  prefetch_tmap(tmV);
  uint32_t ring = 0;          // K/V ring entries issued so far
  uint32_t units = 0;         // units whose Q was issued
  uint32_t skipped = 0xFFFFFFFFu;
  for (int k = 0; k < p.num_rounds; ++k) {
    const int u = item_of(k, p);
    if (u < 0) continue;
    Item it;
    item_coords<SPLIT, BN>(u, p, it);
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
          mbar_arrive_expect_tx(&b.slot_full[slot], C::KV_TILE_BYTES);
          const CUtensorMap* m = kv == 0 ? tmK : tmV;
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sRing + slot * C::KV_TILE_BYTES + c * C::KV_CHUNK_BYTES, m,
                        &b.slot_full[slot], c * C::W, j * BN, bh);
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
// MMA issuer (one whole warp; one elected lane issues each MMA and commit)
// ------------------------------------------------------------------------------------
template <int HD, int BN = kBlockN, bool WARP = true>
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_addr, uint32_t k_addr) {
  using C = Cfg<HD, BN>;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const int ch = (kk * 16) / C::W, off = ((kk * 16) % C::W) * 2;
    const uint64_t a = smem_desc(q_addr + ch * C::CHUNK_BYTES + off, 16, 8 * C::SWB, C::SWZ);
    const uint64_t bd = smem_desc(k_addr + ch * C::KV_CHUNK_BYTES + off, 16, 8 * C::SWB, C::SWZ);
    mma_bf16_ss<WARP>(tmem_d, a, bd, C::IDESC_S, kk > 0);
  }
}

// ones_addr != 0 (two-tile kernel, Cfg::ONES): N = HD + 16, and B's second column chunk
// comes from the ones block: its offset from the V tile is passed as the descriptor's
// stride between column chunks, so the MMA reads HD columns of V, then 16 columns of ones.
template <int HD, int BN = kBlockN, bool WARP = true>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_addr,
                                         bool accumulate, uint32_t ones_addr = 0) {
  using C = Cfg<HD, BN>;
  const uint32_t lbo = ones_addr ? ones_addr - v_addr : C::KV_CHUNK_BYTES;
  const uint32_t idesc = ones_addr ? C::IDESC_O_ONES : C::IDESC_O;
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    // V tile is [key][d]: the B operand (K = keys, N = d) is MN-major
    const uint64_t bd = smem_desc(v_addr + kk * 16 * C::SWB, lbo, 8 * C::SWB, C::SWZ);
    mma_bf16_ts<WARP>(tmem_o, tmem_p + kk * 8, bd, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int HD, int BN, bool SPLIT>
__device__ void mma_role(uint8_t* sQ, uint8_t* sRing, uint32_t tmem, Barriers& b, const Params& p) {
  using C = Cfg<HD, BN>;
  uint32_t ring = 0, units = 0;
  uint32_t p_cnt[2] = {0, 0}, oe_cnt[2] = {0, 0};
  const uint32_t q_addr[2] = {smem_u32(sQ), smem_u32(sQ + C::TILE_BYTES)};
  const uint32_t col_s[2] = {kColS0, kColS1}, col_o[2] = {kColO0, kColO1};
  const uint32_t ring_addr = smem_u32(sRing);
  // The next item is decoded (item_of, item_coords: a handful of integer divisions) right
  // after this item's first S MMAs are issued, while the issuer would otherwise wait for
  // the first P; decoded at the boundary it delayed the next item's first MMAs.
  int k_nxt = -1, u_nxt = -1;
  Item nxt;
  bool has_nxt = next_item<SPLIT, BN>(k_nxt, p, nxt, u_nxt);
  while (has_nxt) {
    const Item it = nxt;
    const int k0 = it.k0, k1 = it.k1;
    if (!warp_wait(&b.q_full, units & 1, p, b)) goto fail;
    ++units;
    uint32_t ks = ring % C::NSLOT;
    if (!warp_wait(&b.slot_full[ks], (ring / C::NSLOT) & 1, p, b)) goto fail;
    ++ring;
    tc_fence_after_sync();
    for (int t = 0; t < 2; ++t)
      if (it.e[t] > k0) {
        issue_s<HD, BN>(tmem + col_s[t], q_addr[t], ring_addr + ks * C::KV_TILE_BYTES);
        mma_commit(&b.s_full[t]);
      }
    mma_commit(&b.slot_empty[ks]);
    if (k1 - k0 == 1) mma_commit(&b.q_empty);
    has_nxt = next_item<SPLIT, BN>(k_nxt, p, nxt, u_nxt);
    for (int j = k0; j < k1; ++j) {
      const uint32_t vs = ring % C::NSLOT;
      if (!warp_wait(&b.slot_full[vs], (ring / C::NSLOT) & 1, p, b)) goto fail;
      ++ring;
      const bool next = j + 1 < k1;
      if (next) {
        ks = ring % C::NSLOT;
        if (!warp_wait(&b.slot_full[ks], (ring / C::NSLOT) & 1, p, b)) goto fail;
        ++ring;
      }
      tc_fence_after_sync();
      for (int t = 0; t < 2; ++t) {
        if (j < it.e[t]) {
          if (j == k0) {  // O_t must have been read out by the previous item's epilogue
            if (!warp_wait(&b.o_empty[t], (oe_cnt[t] & 1) ^ 1, p, b)) goto fail;
            ++oe_cnt[t];
          }
          if (!warp_wait(&b.p_full[t], p_cnt[t] & 1, p, b)) goto fail;
          ++p_cnt[t];
          tc_fence_after_sync();
          issue_pv<HD, BN>(tmem + col_o[t], tmem + col_s[t], ring_addr + vs * C::KV_TILE_BYTES, j > k0,
                           C::ONES ? ring_addr + C::NSLOT * C::KV_TILE_BYTES : 0u);
          if (j == it.e[t] - 1) mma_commit(&b.o_full[t]);
        }
        if (next && j + 1 < it.e[t]) {
          issue_s<HD, BN>(tmem + col_s[t], q_addr[t], ring_addr + ks * C::KV_TILE_BYTES);
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


}  // namespace fa_sm103
