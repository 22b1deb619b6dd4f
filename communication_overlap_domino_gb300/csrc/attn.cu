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
// Persistent kernel, one CTA per SM, 10 warps:
//   warp 0      TMA producer: the Q tile once per item, then the key blocks K_j
//               and value blocks V_j into two 2-slot rings, K one block ahead
//               of V (K_{j+1} is needed for the next scores before V_j is
//               needed for P_j V_j).
//   warp 1      tensor-memory allocation; lane 0 issues the MMAs:
//               S_j = Q K_j^T (M 128, N 128, K 128) into one of two TMEM score
//               buffers, and O += P_j V_j into the TMEM output accumulator,
//               with P_j (the A operand) read from tensor memory too.
//               S_{j+1} is issued before P_j V_j, so the next scores are
//               computed while the softmax of block j runs.
//   warps 2-9   two threads per query row (warps w and w + 4 read the same
//               tensor-memory lanes), each owning 64 of the row's 128 key and
//               output columns.  Both take the row maximum over all 128 scores,
//               so they agree on it.  Lazy rescaling: the running maximum m only
//               moves when a block's maximum exceeds it by more than 2^8 (in the
//               exp2 domain); then the thread rescales its half of the output
//               row in tensor memory (after P_{j-1} V_{j-1} has landed) and its
//               part of the row sum.  Each writes its 64 probabilities
//               p = exp2(s * c - m) as bf16 pairs into the P columns of tensor
//               memory, its query row's lane (once P_{j-1} V_{j-1} has finished
//               reading them).  After the last block the two parts of the row
//               sum are added through shared memory and O / l is stored as bf16.
//
// Barriers (all waits bounded, as in the GEMMs): q_full / q_empty, k_full[s] /
// k_empty[s], v_full[s] / v_empty[s], s_full[b] / s_empty[b], p_full, pv_full,
// o_empty, l_ready[2], final; the softmax warps arrive once per warp, after
// __syncwarp, on s_empty, p_full, o_empty and l_ready.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "attn.h"
#include "ptx.cuh"

namespace domino {

namespace {

constexpr int kAttnThreads = 320;
constexpr int kSoftmaxWarps = 8;  // consumer barriers count one arrival per softmax warp
constexpr int kTile = 128;                        // queries per item, keys per block, head width
constexpr int kSub = kTile * 64 * 2;              // 16 KB: 128 rows x 64 bf16 (one 128-byte-swizzled box)
constexpr int kQBytes = 2 * kSub;                 // Q tile: dh halves 0-63 and 64-127
constexpr int kKBytes = 2 * kSub;                 // K tile: dh halves
constexpr int kVBytes = 2 * kSub;                 // V tile: 2 blocks of 64 keys x (2 boxes of 64 dh x 64 keys)
constexpr int kSlots = 2;                         // slots of the K ring and of the V ring
constexpr int kLsumBytes = 2 * 2 * kTile * 4;     // row-sum halves, double-buffered by item
constexpr int kAttnSmemBytes = kQBytes + kSlots * (kKBytes + kVBytes) + kLsumBytes + 1024 + 256;
static_assert(kAttnSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kAttnTmemCols = 512;           // S buffers at 0 and 128, the output O at 256, P at 384
constexpr uint32_t kOCol = 256;
constexpr uint32_t kPCol = 384;                   // P as bf16 pairs: 64 columns, key 2c and 2c + 1 in column c
constexpr float kRescaleLog2 = 8.0f;              // lazy rescaling threshold: the maximum may lag by 2^8

struct AttnItem {
  int p, b, h, i;  // shard, sequence of the chunk, head of the shard, query tile
};

// Items in order of decreasing query tile: the diagonal makes tile i cost i + 1
// key blocks, so the longest items start first on the persistent CTAs.
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

// The item a CTA runs in its k-th round: the rounds deal the items (longest first) across the persistent
// CTAs in alternating directions, so a CTA that took one of a round's longest items takes one of the next
// round's shortest.  With causal items of 1 .. nq key blocks this evens the CTAs' loads (GPT-style chunk:
// at most 10 key blocks per CTA against 14 when every round deals in the same direction; the mean is 9.5).
// Every item is dealt exactly once; a CTA's first index past num_items ends its rounds (only the last round
// can be partial).
__device__ __forceinline__ int attn_round_item(int k) {
  const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  return k * g + ((k & 1) ? g - 1 - b : b);
}

// Issues S = Q K^T for the key block in K-ring slot k_idx % 2 into score
// buffer s_idx % 2, once the block has landed and the buffer is free; the slot
// is released when the MMAs have read it.
__device__ __forceinline__ bool attn_issue_s(const AttnParams& a, uint32_t tmem_base, uint32_t qa, uint8_t* sk,
                                             uint64_t* k_full, uint64_t* k_empty, uint64_t* s_empty,
                                             uint64_t* s_full, uint32_t k_idx, uint32_t s_idx,
                                             volatile int* abort_flag, int t) {
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
  const uint32_t st = k_idx & 1, sb = s_idx & 1;
  if (!mbar_wait(&k_full[st], (k_idx >> 1) & 1, abort_flag, a.timeout_ns, a.status, kSiteMmaFull, t)) return false;
  if (!mbar_wait(&s_empty[sb], ((s_idx >> 1) & 1) ^ 1, abort_flag, a.timeout_ns, a.status, kSiteMmaTmemEmpty, t))
    return false;
  tc_fence_after_sync();
  const uint32_t ka = smem_u32(sk + st * kKBytes);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint64_t ad = smem_desc_k128(qa + (k >> 2) * kSub) + 2 * (k & 3);
    const uint64_t bd = smem_desc_k128(ka + (k >> 2) * kSub) + 2 * (k & 3);
    mma_bf16_ss(tmem_base + sb * kTile, ad, bd, idesc_s, k != 0 ? 1u : 0u);
  }
  mma_commit(&s_full[sb]);
  mma_commit(&k_empty[st]);
  return true;
}

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
  uint8_t* sq = smem;
  uint8_t* sk = sq + kQBytes;             // K ring: kSlots x 32 KB
  uint8_t* sv = sk + kSlots * kKBytes;    // V ring: kSlots x 32 KB
  float* lsum = reinterpret_cast<float*>(sv + kSlots * kVBytes);  // [2 buffers][2 halves][128 rows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(lsum + 2 * 2 * kTile);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;    // [2]
  uint64_t* k_empty = bars + 4;   // [2]
  uint64_t* v_full = bars + 6;    // [2]
  uint64_t* v_empty = bars + 8;   // [2]
  uint64_t* s_full = bars + 10;   // [2]
  uint64_t* s_empty = bars + 12;  // [2]
  uint64_t* p_full = bars + 14;
  uint64_t* pv_full = bars + 15;
  uint64_t* o_empty = bars + 16;
  uint64_t* final_bar = bars + 17;
  uint64_t* l_ready = bars + 18;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kSoftmaxWarps);
      mbar_init(&l_ready[s], kSoftmaxWarps);
    }
    mbar_init(p_full, kSoftmaxWarps);
    mbar_init(pv_full, 1);
    mbar_init(o_empty, kSoftmaxWarps);
    mbar_init(final_bar, 1);
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t q_phase = 0, k_count = 0, v_count = 0;
    uint32_t issued_q = 0, issued_k = 0, issued_v = 0, k_parity = 0, v_parity = 0;
    bool ok = true;
    // one K or V block into its ring slot (waits until the slot's previous block has been read)
    auto load_block = [&](bool is_k, uint32_t idx, const CUtensorMap* mqk, const CUtensorMap* mv, int col, int y,
                          int t) -> bool {
      const uint32_t st = idx & 1, ph = (idx >> 1) & 1;
      uint64_t* full = is_k ? &k_full[st] : &v_full[st];
      if (!mbar_wait(is_k ? &k_empty[st] : &v_empty[st], ph ^ 1, abort_flag, tmo, a.status, kSiteProducerEmpty, t))
        return false;
      if (is_k) {
        uint8_t* dst = sk + st * kKBytes;
        mbar_arrive_expect_tx(full, kKBytes);
        tma_load_2d(dst, mqk, full, col, y);
        tma_load_2d(dst + kSub, mqk, full, col + 64, y);
        issued_k |= 1u << st;
        k_parity = (k_parity & ~(1u << st)) | (ph << st);
      } else {
        // V as the MN-major B operand: per 64-key block, two boxes of 64 dh x 64 keys
        uint8_t* dst = sv + st * kVBytes;
        mbar_arrive_expect_tx(full, kVBytes);
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_2d(dst + kb * kSub, mv, full, col, y + kb * 64);
          tma_load_2d(dst + kb * kSub + 8192, mv, full, col + 64, y + kb * 64);
        }
        issued_v |= 1u << st;
        v_parity = (v_parity & ~(1u << st)) | (ph << st);
      }
      return true;
    };
    for (int k = 0, t = attn_round_item(0); t < a.num_items && ok && !*abort_flag; t = attn_round_item(++k)) {
      const AttnItem it = attn_item(a, t);
      const CUtensorMap* mqk = &a.map_qk[it.p];
      const CUtensorMap* mv = &a.map_v[it.p];
      const int seq_row0 = a.row0 + it.b * a.S;
      if (!mbar_wait(q_empty, q_phase ^ 1, abort_flag, tmo, a.status, kSiteProducerEmpty, t)) break;
      q_phase ^= 1;
      mbar_arrive_expect_tx(q_full, kQBytes);
      const int qx = it.h * kTile;
      const int qy = seq_row0 + it.i * kTile;
      tma_load_2d(sq, mqk, q_full, qx, qy);
      tma_load_2d(sq + kSub, mqk, q_full, qx + 64, qy);
      issued_q = 1;
      const int kx = (a.Hp + it.h) * kTile;
      const int vx = (2 * a.Hp + it.h) * kTile;
      // K runs one block ahead of V: K_0, K_1, V_0, K_2, V_1, ..., V_i
      for (int j = 0; j <= it.i + 1 && ok; ++j) {
        if (j <= it.i) ok = load_block(true, k_count++, mqk, mv, kx, seq_row0 + j * kTile, t);
        if (ok && j >= 1) ok = load_block(false, v_count++, mqk, mv, vx, seq_row0 + (j - 1) * kTile, t);
      }
    }
    // drain: every load issued has landed before the CTA can exit
    volatile int no_abort = 0;
    if (issued_q) mbar_wait(q_full, (q_phase ^ 1) & 1, &no_abort, tmo, a.status, kSiteDrain, 0);
    for (int s = 0; s < 2; ++s) {
      if (issued_k & (1u << s)) mbar_wait(&k_full[s], (k_parity >> s) & 1, &no_abort, tmo, a.status, kSiteDrain, 1 + s);
      if (issued_v & (1u << s)) mbar_wait(&v_full[s], (v_parity >> s) & 1, &no_abort, tmo, a.status, kSiteDrain, 3 + s);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
    uint32_t q_phase = 0, kv_count = 0, s_count = 0, p_phase = 0, o_phase = 0;
    const uint32_t qa = smem_u32(sq);
    bool ok = true;
    for (int k = 0, t = attn_round_item(0); t < a.num_items && ok && !*abort_flag; t = attn_round_item(++k)) {
      const AttnItem it = attn_item(a, t);
      if (!mbar_wait(q_full, q_phase, abort_flag, tmo, a.status, kSiteMmaFull, t)) break;
      q_phase ^= 1;
      const uint32_t kv0 = kv_count;  // K and V blocks are counted alike
      if (!attn_issue_s(a, tmem_base, qa, sk, k_full, k_empty, s_empty, s_full, kv_count, s_count, abort_flag, t))
        break;
      if (it.i == 0) mma_commit(q_empty);  // Q is read by the score MMAs only: free after the item's last one
      // the output accumulator is free once the previous item's output has been read
      if (!mbar_wait(o_empty, o_phase ^ 1, abort_flag, tmo, a.status, kSiteMmaTmemEmpty, t)) break;
      o_phase ^= 1;
      for (int j = 0; j <= it.i; ++j) {
        if (j + 1 <= it.i) {
          if (!attn_issue_s(a, tmem_base, qa, sk, k_full, k_empty, s_empty, s_full, kv0 + j + 1, s_count + j + 1,
                            abort_flag, t)) {
            ok = false;
            break;
          }
          if (j + 1 == it.i) mma_commit(q_empty);
        }
        const uint32_t vi = kv0 + j, st = vi & 1;
        if (!mbar_wait(p_full, p_phase, abort_flag, tmo, a.status, kSiteAttnP, t) ||
            !mbar_wait(&v_full[st], (vi >> 1) & 1, abort_flag, tmo, a.status, kSiteMmaFull, t)) {
          ok = false;
          break;
        }
        p_phase ^= 1;
        tc_fence_after_sync();
        const uint32_t va = smem_u32(sv + st * kVBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 16 keys per step: 8 columns of P in tensor memory
          const uint64_t bd = smem_desc_mn128(va + (k >> 2) * kSub) + (2048 >> 4) * (k & 3);
          mma_bf16_ts(tmem_base + kOCol, tmem_base + kPCol + 8 * k, bd, idesc_pv, (j | k) != 0 ? 1u : 0u);
        }
        mma_commit(pv_full);
        mma_commit(&v_empty[st]);
      }
      kv_count = kv0 + it.i + 1;
      s_count += it.i + 1;
      if (!ok) break;
    }
    mma_commit(final_bar);
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, a.status, kSiteDrain, 99);
  } else if (warp >= 2) {
    // --------------------------------------------------- softmax / output
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;   // key / output columns half * 64 .. + 64
    const int r = quarter * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t to = tmem_base + lane_off + kOCol + half * 64;  // this thread's half of the output row
    uint32_t s_count = 0, pv_phase = 0, item_count = 0;
    for (int k = 0, t = attn_round_item(0); t < a.num_items && !*abort_flag; t = attn_round_item(++k), ++item_count) {
      const AttnItem it = attn_item(a, t);
      float m_run = -INFINITY, l_run = 0.0f;
      bool ok = true;
      for (int j = 0; j <= it.i; ++j, ++s_count) {
        const uint32_t sb = s_count & 1;
        if (!mbar_wait(&s_full[sb], (s_count >> 1) & 1, abort_flag, tmo, a.status, kSiteEpilogueTmemFull, t)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t ts = tmem_base + lane_off + sb * kTile;
        const bool diag = j == it.i;
        // the row's 128 scores in two batches of tensor-memory loads: this thread's own 64 keys (half * 64 ..)
        // stay in registers for the probabilities, the other 64 serve only the maximum (two batches, as all
        // 128 at once would not fit the 168 registers a thread of this 10-warp block can have)
        uint32_t vo0[32], vo1[32];
        float mx = -INFINITY;
        {
          const int ko = half * 64, kx = (half ^ 1) * 64;
          uint32_t vx[32];
          tmem_ld_32x32b_x32(ts + ko, vo0);
          tmem_ld_32x32b_x32(ts + ko + 32, vo1);
          tmem_ld_32x32b_x32(ts + kx, vx);
          tmem_ld_wait();
          // pass 1: row maximum of the visible scores
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (ko + e <= r) mx = fmaxf(mx, __uint_as_float(vo0[e]));
              if (ko + 32 + e <= r) mx = fmaxf(mx, __uint_as_float(vo1[e]));
              if (kx + e <= r) mx = fmaxf(mx, __uint_as_float(vx[e]));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = max3(mx, __uint_as_float(vo0[e]), __uint_as_float(vo1[e]));
#pragma unroll
            for (int e = 0; e < 32; e += 2) mx = max3(mx, __uint_as_float(vx[e]), __uint_as_float(vx[e + 1]));
          }
          tmem_ld_32x32b_x32(ts + kx + 32, vx);
          tmem_ld_wait();
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (kx + 32 + e <= r) mx = fmaxf(mx, __uint_as_float(vx[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) mx = max3(mx, __uint_as_float(vx[e]), __uint_as_float(vx[e + 1]));
          }
        }
        const float m_blk = mx * a.scale_log2;
        const bool rescale = m_blk > m_run + kRescaleLog2;
        float alpha = 1.0f;
        if (rescale) {
          alpha = ex2_approx(m_run - m_blk);
          m_run = m_blk;
        }
        // pass 2: this thread's 64 probabilities, packed as bf16 pairs
        uint32_t pk[32];
        float sum_even = 0.0f, sum_odd = 0.0f;  // the row sum of this thread's even and odd keys
        {
          const float c = a.scale_log2, nm = -m_run;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int k0 = half * 64 + 2 * e, k1 = k0 + 32;
            float x0, x1, x2, x3;
            fma2(x0, x1, __uint_as_float(vo0[2 * e]), __uint_as_float(vo0[2 * e + 1]), c, c, nm, nm);
            fma2(x2, x3, __uint_as_float(vo1[2 * e]), __uint_as_float(vo1[2 * e + 1]), c, c, nm, nm);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            if (diag) {
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
        }
        const float sum = sum_even + sum_odd;
        // P_{j-1} V_{j-1} has landed: the P buffer is free and the output up to date
        if (j > 0) {
          if (!mbar_wait(pv_full, pv_phase, abort_flag, tmo, a.status, kSiteAttnPV, t)) {
            ok = false;
            break;
          }
          pv_phase ^= 1;
          tc_fence_after_sync();
          if (rescale) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
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
            tmem_st_wait();
          }
        }
        // this thread's 64 keys as 32 bf16 pairs: pk[c] holds keys half * 64 + 2c, + 1 -> P column half * 32 + c
        tmem_st_32x32b_x32(tmem_base + lane_off + kPCol + half * 32, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();  // the warp's scores are read and its P stored: one arrival per warp
        if (lane == 0) {
          mbar_arrive(&s_empty[sb]);
          mbar_arrive(p_full);
        }
        l_run = l_run * alpha + sum;
      }
      if (!ok) break;
      // the last P V has landed: read this thread's half of the output row
      if (!mbar_wait(pv_full, pv_phase, abort_flag, tmo, a.status, kSiteAttnPV, t)) break;
      pv_phase ^= 1;
      tc_fence_after_sync();
      uint32_t o0[32], o1[32];
      tmem_ld_32x32b_x32(to, o0);
      tmem_ld_32x32b_x32(to + 32, o1);
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      // the row sum: this thread's part plus its partner's, through shared memory
      const uint32_t lb = item_count & 1;
      float* lbuf = lsum + lb * 2 * kTile;
      lbuf[half * kTile + r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&l_ready[lb]);
      if (!mbar_wait(&l_ready[lb], (item_count >> 1) & 1, abort_flag, tmo, a.status, kSiteAttnPV, t)) break;
      const float inv = 1.0f / (lbuf[r] + lbuf[kTile + r]);
      // O / l as bf16: this thread's 128 contiguous bytes of the row
      const int64_t grow = a.row0 + static_cast<int64_t>(it.b) * a.S + it.i * kTile + r;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o[it.p]) + grow * a.ldo + it.h * kTile +
                                            half * 64);
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const uint32_t* oh = q8 < 4 ? o0 + 8 * q8 : o1 + 8 * (q8 - 4);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; e += 2)
          mul2(y[e], y[e + 1], __uint_as_float(oh[e]), __uint_as_float(oh[e + 1]), inv, inv);
        dst[q8] = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                             pack_bf16(y[6], y[7]));
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
  const int grid = a.num_items < num_sms ? a.num_items : num_sms;
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
