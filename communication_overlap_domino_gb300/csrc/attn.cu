// Causal multi-head attention core of the sliced tensor-parallel attention
// block, flash-style on the tensor cores (tcgen05).
//
// One work item = one head of one sequence of one shard and one 128-query
// tile: O = softmax(Q K^T / sqrt(dh) + causal mask) V for those 128 queries,
// dh = 128.  The keys are visited in blocks of 128 (only the blocks at or below
// the diagonal); the softmax is kept online (running row maximum m and sum l,
// the output rescaled by exp2(m_old - m_new) when the maximum grows), so no
// score matrix ever reaches global memory.
//
// Persistent kernel, one CTA per SM, running two independent streams of items
// ("lanes" 0 and 1) that share only the tensor cores: while the softmax warps
// of one lane turn a block of scores into probabilities, the tensor cores
// multiply the other lane's probabilities by V and compute its next scores.
// Each lane has its own producer, MMA issuer and softmax warps, so one lane
// waiting on a load never holds up the other.  12 warps:
//   warps 0, 10 TMA producer of lane 0, lane 1: the lane's Q tile (one slot)
//               and its key and value blocks through a 2-slot ring of 32 KB
//               slots, in the order its MMAs consume them.
//   warps 1, 11 lane 0 of each issues its lane's MMAs (warp 1 also allocates
//               the 512 tensor-memory columns): per step, O += P_b V_b for the
//               block b whose probabilities are ready (A operand from tensor
//               memory), then S_{b+1} = Q K_{b+1}^T (M 128, N 128, K 128) into
//               the same tensor-memory columns, which P_b occupied.  The tensor
//               cores execute one thread's MMAs in issue order, so the P V
//               product has read P_b before S_{b+1} overwrites it.
//   warps 2-5   softmax of lane 0, warps 6-9 of lane 1: one thread per query
//               row (warp w reads tensor-memory lanes 32 (w % 4) ..).  Per key
//               block: the row maximum over the 128 scores, lazy rescaling (the
//               running maximum m only moves when a block's maximum exceeds it
//               by more than 2^8 in the exp2 domain; then the warp rescales its
//               output rows in tensor memory, which the previous P V product
//               has finished updating), and the 128 probabilities
//               p = exp2(s c - m) written as bf16 pairs over score columns
//               64-127.  After an item's last block: O / l as bf16 to global
//               memory.
// Tensor memory per lane L: scores / probabilities at columns 128 L, the
// output accumulator at 256 + 128 L.
//
// Barriers (all waits bounded), per lane: q_full / q_empty, ring full / empty
// per slot, s_full, p_full, o_full / o_empty, final.  The softmax warps arrive
// once per warp, after __syncwarp.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <type_traits>

#include "attn.h"
#include "ptx.cuh"

namespace domino {

namespace {

constexpr int kAttnThreads = 384;
constexpr int kLaneWarps = 4;                     // softmax warps per lane; consumer barriers count one per warp
constexpr int kTile = 128;                        // queries per item, keys per block, head width
constexpr int kSub = kTile * 64 * 2;              // 16 KB: 128 rows x 64 bf16 (one 128-byte-swizzled box)
constexpr int kQBytes = 2 * kSub;                 // Q tile: dh halves 0-63 and 64-127
constexpr int kSlotBytes = 2 * kSub;              // one K block (dh halves) or one V block (MN-major boxes)
constexpr int kRing = 2;                          // K / V ring slots per lane
constexpr int kAttnSmemBytes = 2 * (kQBytes + kRing * kSlotBytes) + 1024 + 512;
static_assert(kAttnSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kAttnTmemCols = 512;
constexpr uint32_t kOCol = 256;                   // output accumulator of lane L at kOCol + 128 L
constexpr uint32_t kPCol = 64;                    // probabilities at score columns 64-127 (keys 2q, 2q + 1 in 64 + q)
constexpr float kRescaleLog2 = 8.0f;              // lazy rescaling threshold: the maximum may lag by 2^8

struct AttnItem {
  int p, b, h, i;  // shard, sequence of the chunk, head of the shard, query tile
};

// Items in order of decreasing query tile: the diagonal makes tile i cost i + 1
// key blocks, so the longest items start first.
__device__ __forceinline__ AttnItem attn_item(const AttnParams& a, int t) {
  const int per_tile = a.P * a.seqs * a.Hp;
  AttnItem it;
  it.i = a.nq - 1 - t / per_tile;
  int r = t - (a.nq - 1 - it.i) * per_tile;
  it.p = r / (a.seqs * a.Hp);
  r -= it.p * a.seqs * a.Hp;
  it.b = r / a.Hp;
  it.h = r - it.b * a.Hp;
  return it;
}

// The item lane `lane` of this CTA runs in its k-th round.  Each round deals 2 x gridDim items (longest
// first) to the lanes in a fixed order in which a CTA's two lanes stand at opposite ends (lane 0 of CTA c at
// position c, lane 1 at 2 gridDim - 1 - c), and the rounds alternate direction: in every round one lane of a
// CTA takes one of the longer items and the other one of the shorter, and each lane alternates between the
// two from round to round (with causal items of 1 .. nq key blocks this evens the lanes' and the CTAs' loads).
// Every item is dealt exactly once; a lane's first index past num_items ends its rounds (only the last round
// can be partial).
__device__ __forceinline__ int attn_round_item(int k, int lane) {
  const int g = 2 * static_cast<int>(gridDim.x);
  const int v = lane == 0 ? static_cast<int>(blockIdx.x) : g - 1 - static_cast<int>(blockIdx.x);
  return k * g + ((k & 1) ? g - 1 - v : v);
}

// One lane's sequence of key blocks, flattened over its items: block (item t, j) for j = 0 .. i.  `cur` is
// the next block whose scores are to be computed, `prev` the block whose probabilities feed the next P V.
// The producer and the MMA issuer step identical copies of it, so they agree on every load and MMA.
struct LaneWalk {
  int round = 0;
  int t = 0;      // current item (>= num_items: none left)
  AttnItem it{};
  int j = 0;      // next block of the current item whose scores are computed
  bool has_prev = false;
  AttnItem prev_it{};
  int prev_j = 0;
  int items = 0;  // items started (their first block's scores issued)

  __device__ __forceinline__ void start(const AttnParams& a, int lane) {
    t = attn_round_item(0, lane);
    if (t < a.num_items) it = attn_item(a, t);
  }
  __device__ __forceinline__ bool has_cur(const AttnParams& a) const { return t < a.num_items; }
  __device__ __forceinline__ bool done(const AttnParams& a) const { return !has_prev && !has_cur(a); }
  // after one step: the current block becomes `prev`, the walk moves to the next block or item
  __device__ __forceinline__ void advance(const AttnParams& a, int lane) {
    if (!has_cur(a)) {
      has_prev = false;
      return;
    }
    has_prev = true;
    prev_it = it;
    prev_j = j;
    if (j == 0) ++items;
    if (++j > it.i) {
      j = 0;
      t = attn_round_item(++round, lane);
      if (t < a.num_items) it = attn_item(a, t);
    }
  }
};

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulation: the A operand (M rows in lanes, K along
// the columns, two bf16 per 32-bit column) is read from tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // per lane: Q tile | kRing K / V slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * (kQBytes + kRing * kSlotBytes));
  // per lane L, at bars + 16 L: ring full [kRing], ring empty [kRing], q_full, q_empty, s_full, p_full, o_full,
  // o_empty, final
  constexpr int kBarsPerLane = 16;
  static_assert(2 * kRing + 7 <= kBarsPerLane, "barrier block");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kBarsPerLane);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int l = 0; l < 2; ++l) {
      uint64_t* b = bars + kBarsPerLane * l;
      for (int s = 0; s < kRing; ++s) {
        mbar_init(&b[s], 1);
        mbar_init(&b[kRing + s], 1);
      }
      mbar_init(&b[2 * kRing + 0], 1);           // q_full
      mbar_init(&b[2 * kRing + 1], 1);           // q_empty
      mbar_init(&b[2 * kRing + 2], 1);           // s_full
      mbar_init(&b[2 * kRing + 3], kLaneWarps);  // p_full
      mbar_init(&b[2 * kRing + 4], 1);           // o_full
      mbar_init(&b[2 * kRing + 5], kLaneWarps);  // o_empty
      mbar_init(&b[2 * kRing + 6], 1);           // final
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kAttnTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t tmo = a.timeout_ns;

  // the lane a control warp serves: warps 0 and 1 lane 0, warps 10 and 11 lane 1
  const int ctl_lane = warp >= 10 ? 1 : 0;
  uint8_t* sq = smem + ctl_lane * (kQBytes + kRing * kSlotBytes);
  uint8_t* ring = sq + kQBytes;
  uint64_t* lb = bars + kBarsPerLane * ctl_lane;
  uint64_t* ring_full = lb;
  uint64_t* ring_empty = lb + kRing;
  uint64_t* q_full = lb + 2 * kRing;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_full + 2;
  uint64_t* p_full = q_full + 3;
  uint64_t* o_full = q_full + 4;
  uint64_t* o_empty = q_full + 5;
  uint64_t* final_bar = q_full + 6;

  if ((warp == 0 || warp == 10) && lane == 0) {
    // ------------------------------------------------------------ producer
    const int L = ctl_lane;
    uint32_t g = 0, q_count = 0;  // ring loads and Q loads issued
    uint32_t ring_issued = 0, ring_parity = 0;
    bool ok = true;
    // one K block (two boxes of 64 dh x 128 keys) or one V block (the MN-major B operand: per 64-key block,
    // two boxes of 64 dh x 64 keys) into the next ring slot
    auto load_block = [&](bool is_k, const AttnItem& it, int j, int t) -> bool {
      const uint32_t st = g % kRing, ph = (g / kRing) & 1;
      if (!mbar_wait(&ring_empty[st], ph ^ 1, abort_flag, tmo, a.status, kSiteProducerEmpty, t)) return false;
      uint8_t* dst = ring + st * kSlotBytes;
      const int y = a.row0 + it.b * a.S + j * kTile;
      mbar_arrive_expect_tx(&ring_full[st], kSlotBytes);
      if (is_k) {
        const int kx = (a.Hp + it.h) * kTile;
        tma_load_2d(dst, &a.map_qk[it.p], &ring_full[st], kx, y);
        tma_load_2d(dst + kSub, &a.map_qk[it.p], &ring_full[st], kx + 64, y);
      } else {
        const int vx = (2 * a.Hp + it.h) * kTile;
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_2d(dst + kb * kSub, &a.map_v[it.p], &ring_full[st], vx, y + kb * 64);
          tma_load_2d(dst + kb * kSub + 8192, &a.map_v[it.p], &ring_full[st], vx + 64, y + kb * 64);
        }
      }
      ring_issued |= 1u << st;
      ring_parity = (ring_parity & ~(1u << st)) | (ph << st);
      ++g;
      return true;
    };
    LaneWalk lw;
    lw.start(a, L);
    while (ok && !*abort_flag && !lw.done(a)) {
      // one step: the previous block's V, then the current block's Q (first block) and K
      if (lw.has_prev) ok = load_block(false, lw.prev_it, lw.prev_j, lw.t);
      if (ok && lw.has_cur(a)) {
        if (lw.j == 0) {  // the item's Q tile, once the lane's previous item has issued its last scores
          if (!mbar_wait(q_empty, (q_count & 1) ^ 1, abort_flag, tmo, a.status, kSiteProducerEmpty, lw.t)) break;
          ++q_count;
          const int qx = lw.it.h * kTile;
          const int qy = a.row0 + lw.it.b * a.S + lw.it.i * kTile;
          mbar_arrive_expect_tx(q_full, kQBytes);
          tma_load_2d(sq, &a.map_qk[lw.it.p], q_full, qx, qy);
          tma_load_2d(sq + kSub, &a.map_qk[lw.it.p], q_full, qx + 64, qy);
        }
        ok = load_block(true, lw.it, lw.j, lw.t);
      }
      lw.advance(a, L);
    }
    // drain: every load issued has landed before the CTA can exit
    volatile int no_abort = 0;
    if (q_count > 0) mbar_wait(q_full, (q_count - 1) & 1, &no_abort, tmo, a.status, kSiteDrain, 0);
    for (int s = 0; s < kRing; ++s)
      if (ring_issued & (1u << s))
        mbar_wait(&ring_full[s], (ring_parity >> s) & 1, &no_abort, tmo, a.status, kSiteDrain, 1 + s);
  } else if ((warp == 1 || warp == 11) && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const int L = ctl_lane;
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
    const uint32_t t_s = tmem_base + L * kTile;          // scores, then probabilities
    const uint32_t t_o = tmem_base + kOCol + L * kTile;  // output accumulator
    const uint32_t qa = smem_u32(sq);
    uint32_t g = 0, q_count = 0, p_count = 0, o_items = 0;
    LaneWalk lw;
    lw.start(a, L);
    while (!*abort_flag && !lw.done(a)) {
      if (lw.has_prev) {
        // ---- O += P V for the previous block, once its probabilities are written
        const uint32_t st = g % kRing, ph = (g / kRing) & 1;
        if (lw.prev_j == 0) {  // the accumulator is free once the lane's previous item's output was read
          if (!mbar_wait(o_empty, (o_items & 1) ^ 1, abort_flag, tmo, a.status, kSiteMmaTmemEmpty, lw.t)) break;
          ++o_items;
        }
        if (!mbar_wait(p_full, p_count & 1, abort_flag, tmo, a.status, kSiteAttnP, lw.t) ||
            !mbar_wait(&ring_full[st], ph, abort_flag, tmo, a.status, kSiteMmaFull, lw.t))
          break;
        ++p_count;
        tc_fence_after_sync();
        const uint32_t va = smem_u32(ring + st * kSlotBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 16 keys per step: 8 columns of P in tensor memory
          const uint64_t bd = smem_desc_mn128(va + (k >> 2) * kSub) + (2048 >> 4) * (k & 3);
          mma_bf16_ts(t_o, t_s + kPCol + 8 * k, bd, idesc_pv, (lw.prev_j | k) != 0 ? 1u : 0u);
        }
        mma_commit(&ring_empty[st]);
        if (lw.prev_j == lw.prev_it.i) mma_commit(o_full);
        ++g;
      }
      if (lw.has_cur(a)) {
        // ---- S = Q K^T for the current block, into the columns P just left
        const uint32_t st = g % kRing, ph = (g / kRing) & 1;
        if (lw.j == 0) {
          if (!mbar_wait(q_full, q_count & 1, abort_flag, tmo, a.status, kSiteMmaFull, lw.t)) break;
          ++q_count;
        }
        if (!mbar_wait(&ring_full[st], ph, abort_flag, tmo, a.status, kSiteMmaFull, lw.t)) break;
        tc_fence_after_sync();
        const uint32_t ka = smem_u32(ring + st * kSlotBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = smem_desc_k128(qa + (k >> 2) * kSub) + 2 * (k & 3);
          const uint64_t bd = smem_desc_k128(ka + (k >> 2) * kSub) + 2 * (k & 3);
          mma_bf16_ss(t_s, ad, bd, idesc_s, k != 0 ? 1u : 0u);
        }
        mma_commit(&ring_empty[st]);
        mma_commit(s_full);
        if (lw.j == lw.it.i) mma_commit(q_empty);  // the item's last scores: its Q tile is free
        ++g;
      }
      lw.advance(a, L);
    }
    mma_commit(final_bar);
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, a.status, kSiteDrain, 99);
  } else if (warp >= 2 && warp < 10) {
    // --------------------------------------------------- softmax / output
    const int L = (warp - 2) / kLaneWarps;
    uint64_t* sb = bars + kBarsPerLane * L + 2 * kRing;  // this lane's q_full .. final
    uint64_t* s_full = sb + 2;
    uint64_t* p_full = sb + 3;
    uint64_t* o_full = sb + 4;
    uint64_t* o_empty = sb + 5;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t ts = tmem_base + lane_off + L * kTile;          // this row's scores / probabilities
    const uint32_t to = tmem_base + lane_off + kOCol + L * kTile;  // this row's output accumulator
    const float c = a.scale_log2;
    uint32_t s_count = 0, item_count = 0;
    for (int k = 0, t = attn_round_item(0, L); t < a.num_items && !*abort_flag;
         t = attn_round_item(++k, L), ++item_count) {
      const AttnItem it = attn_item(a, t);
      float m_run = -INFINITY, l_run = 0.0f;
      bool ok = true;
      for (int j = 0; j <= it.i; ++j, ++s_count) {
        if (!mbar_wait(s_full, s_count & 1, abort_flag, tmo, a.status, kSiteEpilogueTmemFull, t)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const bool diag = j == it.i;  // keys 0 .. r of this block are visible to row r
        // pass 1: the row maximum of the visible scores, in two batches of 64 columns; the second batch stays
        // in registers for pass 2
        float mx = -INFINITY;
        uint32_t w0[32], w1[32];
        {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(ts, v0);
          tmem_ld_32x32b_x32(ts + 32, v1);
          tmem_ld_wait();
          tmem_ld_32x32b_x32(ts + 64, w0);
          tmem_ld_32x32b_x32(ts + 96, w1);
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (e <= r) mx = fmaxf(mx, __uint_as_float(v0[e]));
              if (32 + e <= r) mx = fmaxf(mx, __uint_as_float(v1[e]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = max3(mx, __uint_as_float(v0[e]), __uint_as_float(v1[e]));
          }
          tmem_ld_wait();
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (64 + e <= r) mx = fmaxf(mx, __uint_as_float(w0[e]));
              if (96 + e <= r) mx = fmaxf(mx, __uint_as_float(w1[e]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = max3(mx, __uint_as_float(w0[e]), __uint_as_float(w1[e]));
          }
        }
        const float m_blk = mx * c;
        const bool grow_m = m_blk > m_run + kRescaleLog2;
        float alpha = 1.0f;
        if (grow_m) {
          alpha = ex2_approx(m_run - m_blk);  // 0 for the first block
          m_run = m_blk;
        }
        // tensor-memory loads and stores are warp-wide: the whole warp rescales its rows (alpha = 1 where the
        // maximum stayed) once the previous P V has finished (its completion preceded these scores')
        if (j > 0 && __any_sync(0xffffffffu, grow_m)) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(to + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float y0, y1;
              mul2(y0, y1, __uint_as_float(v[e]), __uint_as_float(v[e + 1]), alpha, alpha);
              v[e] = __float_as_uint(y0);
              v[e + 1] = __float_as_uint(y1);
            }
            tmem_st_32x32b_x32(to + cc * 32, v);
          }
        }
        // pass 2: the 128 probabilities as bf16 pairs over score columns 64-127 (keys 2q, 2q + 1 -> column
        // 64 + q).  Keys 64-127 first, from the registers of pass 1 (their probabilities overwrite the scores
        // of those keys), then keys 0-63, reloaded (their probabilities overwrite scores 64-95, already read).
        float sum_even = 0.0f, sum_odd = 0.0f;
        const float nm = -m_run;
        // diag_c: std::true_type for the diagonal block (keys past the row masked), std::false_type for the
        // others, so that the blocks below the diagonal carry no masking instructions
        auto probs = [&](auto diag_c, const uint32_t (&x0)[32], const uint32_t (&x1)[32], int kbase,
                         uint32_t (&pk)[32]) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int k0 = kbase + 2 * e, k1 = k0 + 32;
            float y0, y1, y2, y3;
            fma2(y0, y1, __uint_as_float(x0[2 * e]), __uint_as_float(x0[2 * e + 1]), c, c, nm, nm);
            fma2(y2, y3, __uint_as_float(x1[2 * e]), __uint_as_float(x1[2 * e + 1]), c, c, nm, nm);
            float p0 = ex2_approx(y0), p1 = ex2_approx(y1), p2 = ex2_approx(y2), p3 = ex2_approx(y3);
            if constexpr (decltype(diag_c)::value) {
              p0 = k0 <= r ? p0 : 0.0f;
              p1 = k0 + 1 <= r ? p1 : 0.0f;
              p2 = k1 <= r ? p2 : 0.0f;
              p3 = k1 + 1 <= r ? p3 : 0.0f;
            }
            add2(sum_even, sum_odd, sum_even, sum_odd, p0, p1);
            add2(sum_even, sum_odd, sum_even, sum_odd, p2, p3);
            pk[e] = pack_bf16(p0, p1);
            pk[16 + e] = pack_bf16(p2, p3);
          }
        };
        {
          uint32_t pk[32];
          if (diag) probs(std::true_type{}, w0, w1, 64, pk);
          else probs(std::false_type{}, w0, w1, 64, pk);
          tmem_st_32x32b_x32(ts + kPCol + 32, pk);
        }
        {
          uint32_t v0[32], v1[32], pk[32];
          tmem_ld_32x32b_x32(ts, v0);
          tmem_ld_32x32b_x32(ts + 32, v1);
          tmem_ld_wait();
          if (diag) probs(std::true_type{}, v0, v1, 0, pk);
          else probs(std::false_type{}, v0, v1, 0, pk);
          tmem_st_32x32b_x32(ts + kPCol, pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();  // the warp's probabilities (and any rescaled output) are written: one arrival per warp
        if (lane == 0) mbar_arrive(p_full);
        l_run = l_run * alpha + (sum_even + sum_odd);
      }
      if (!ok) break;
      // the item's last P V has landed: read the output row, free the accumulator, store O / l as bf16
      if (!mbar_wait(o_full, item_count & 1, abort_flag, tmo, a.status, kSiteAttnPV, t)) break;
      tc_fence_after_sync();
      const int64_t grow = a.row0 + static_cast<int64_t>(it.b) * a.S + it.i * kTile + r;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o[it.p]) + grow * a.ldo + it.h * kTile);
      const float inv = 1.0f / l_run;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t o0[32], o1[32];
        tmem_ld_32x32b_x32(to + hb * 64, o0);
        tmem_ld_32x32b_x32(to + hb * 64 + 32, o1);
        tmem_ld_wait();
        if (hb == 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty);
        }
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const uint32_t* oh = q8 < 4 ? o0 + 8 * q8 : o1 + 8 * (q8 - 4);
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            mul2(y[e], y[e + 1], __uint_as_float(oh[e]), __uint_as_float(oh[e + 1]), inv, inv);
          dst[hb * 8 + q8] = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                                        pack_bf16(y[6], y[7]));
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kAttnTmemCols);
  }
}

}  // namespace

cudaError_t prepare_attn_kernel() {
  return cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmemBytes);
}

domino_status_t launch_attn_fwd(const AttnLaunch& L, int num_sms, cudaStream_t stream, std::string* err) {
  AttnParams a;
  memset(&a, 0, sizeof a);
  if (L.P < 1 || L.P > kMaxShards || L.dh != kTile || L.S % kTile != 0) {
    if (err) *err = "launch_attn_fwd: unsupported shape";
    return DOMINO_ERR_UNSUPPORTED;
  }
  const int64_t qkv_cols = 3 * static_cast<int64_t>(L.Hp) * L.dh;
  for (int p = 0; p < L.P; ++p) {
    const Operand2D op{L.qkv[p], L.M, qkv_cols, qkv_cols};
    if (!encode_bf16_sw128(&a.map_qk[p], op, kTile, err)) return DOMINO_ERR_CUDA;
    if (!encode_bf16_sw128(&a.map_v[p], op, 64, err)) return DOMINO_ERR_CUDA;
    a.o[p] = L.o[p];
  }
  a.ldo = static_cast<int64_t>(L.Hp) * L.dh;
  a.row0 = L.row0;
  a.S = static_cast<int32_t>(L.S);
  a.Hp = L.Hp;
  a.seqs = L.seqs;
  a.P = L.P;
  a.nq = static_cast<int32_t>(L.S / kTile);
  a.num_items = a.P * a.seqs * a.Hp * a.nq;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(L.dh)));
  a.status = L.status;
  a.timeout_ns = L.timeout_ns;
  if (a.num_items == 0) return DOMINO_OK;
  const int lanes_needed = (a.num_items + 1) / 2;  // two lanes of items per CTA
  const int grid = lanes_needed < num_sms ? lanes_needed : num_sms;
  void* args[] = {&a};
  const cudaError_t st = cudaLaunchKernel(reinterpret_cast<const void*>(&attn_fwd_kernel), dim3(grid),
                                          dim3(kAttnThreads), args, kAttnSmemBytes, stream);
  if (st != cudaSuccess) {
    if (err) *err = std::string("attention launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace domino
