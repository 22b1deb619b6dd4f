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
// Persistent kernel, one CTA per SM, one item at a time, with three score
// buffers in tensor memory: the tensor cores compute the scores of the next key
// blocks (and the P V products of the previous ones) while the softmax warps
// turn the scores of block j into probabilities, so a key block costs the longer
// of the two, not their sum.  14 warps:
//   warp 0      TMA producer: the item's Q tile (two slots, so the next item's
//               tile loads during the current item) and its key and value
//               blocks through a 4-slot ring of 32 KB slots, in the order the
//               MMAs consume them.
//   warp 1      lane 0 issues the MMAs (the warp also allocates the 512
//               tensor-memory columns), over the CTA's blocks in sequence s:
//               S_0 .. S_2, then per s: O += P_s V_s, S_{s+3}.  S_s goes to
//               score buffer s % 3; P_s overwrites it, and S_{s+3} is issued
//               after the P V product that reads P_s: the tensor cores execute
//               one thread's MMAs in issue order, so the product has read P_s
//               before S_{s+3} overwrites it.  An item's products accumulate in
//               the output accumulator, whose first product of the next item
//               waits until the output warps have read it.
//   warps 2-5   output: one thread per query row reads the item's finished
//               output row from tensor memory, frees the buffer and stores
//               O / l as bf16, while the softmax warps go on with the next item.
//   warps 6-13  softmax: two threads per query row, one per half of the key
//               block (warp w reads tensor-memory lanes 32 (w % 4) ..; warps
//               6-9 take keys 0-63, warps 10-13 keys 64-127).  Per key block and
//               thread: the maximum over its 64 scores, exchanged with the
//               partner thread of the same row through shared memory (one
//               mbarrier per row quarter, two arrivals: one per warp); lazy
//               rescaling (the running maximum m only moves when the block's
//               row maximum exceeds it by more than 2^8 in the exp2 domain;
//               both partners take the same decision from the same maximum and
//               each rescales its half of the output row in tensor memory once
//               the previous block's P V product has landed, the only wait on
//               the products); its 64
//               probabilities p = exp2(s c - m) as bf16 pairs over the first 32
//               of its own score columns, which it has already read.  After an
//               item's last block the partners add their row sums and hand the
//               sum to the output warps through shared memory.
// Tensor memory: score buffers at columns 0, 128 and 256 (keys 2q, 2q + 1 of
// half h in column 64 h + q once they are probabilities), the output
// accumulator at 384.
//
// Barriers (all waits bounded): ring full / empty per slot, q_full / q_empty
// per Q slot, s_full / p_full per score buffer, o_full / o_empty for the output
// accumulator, l_full / l_empty per row-sum slot, pv for the P V products of
// even and of odd index (one phase per product), the four row-quarter exchange
// barriers, final.  Warps arrive once per warp, after __syncwarp.
#include <cuda_bf16.h>

#include <cmath>
#include <cstring>
#include <string>
#include <type_traits>

#include "attn.h"
#include "ptx.cuh"

namespace domino {

namespace {

constexpr int kAttnWarps = 14;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kOutWarp0 = 2;                      // warps 2-5: output
constexpr int kSoftWarp0 = 6;                     // warps 6-13: softmax
constexpr int kSoftWarps = 8;
constexpr int kTile = 128;                        // queries per item, keys per block, head width
constexpr int kSub = kTile * 64 * 2;              // 16 KB: 128 rows x 64 bf16 (one 128-byte-swizzled box)
constexpr int kQBytes = 2 * kSub;                 // Q tile: dh halves 0-63 and 64-127
constexpr int kSlotBytes = 2 * kSub;              // one K block (dh halves) or one V block (MN-major boxes)
constexpr int kQSlots = 2;
constexpr int kRing = 4;                          // K / V ring slots
constexpr int kDataBytes = kQSlots * kQBytes + kRing * kSlotBytes;

// barrier indices
constexpr int kBarRingFull = 0;
constexpr int kBarRingEmpty = kBarRingFull + kRing;
constexpr int kBarQFull = kBarRingEmpty + kRing;
constexpr int kBarQEmpty = kBarQFull + kQSlots;
constexpr int kSBufs = 3;                         // score buffers in tensor memory
constexpr int kBarSFull = kBarQEmpty + kQSlots;
constexpr int kBarPFull = kBarSFull + kSBufs;
constexpr int kBarOFull = kBarPFull + kSBufs;
constexpr int kBarOEmpty = kBarOFull + 1;
constexpr int kBarLFull = kBarOEmpty + 1;
constexpr int kBarLEmpty = kBarLFull + 2;
constexpr int kBarPV = kBarLEmpty + 2;            // 2: P V products of even and odd index
constexpr int kBarX = kBarPV + 2;                 // 4: one per row quarter
constexpr int kBarFinal = kBarX + 4;
constexpr int kNumBars = kBarFinal + 1;

constexpr int kBarOff = kDataBytes;
constexpr int kMiscOff = kBarOff + 8 * 32;        // TMEM base, abort flag
static_assert(kNumBars <= 32, "barrier block");
constexpr int kXOff = kMiscOff + 16;              // exchange slots: parity x row quarter x half x 32 rows (fp32)
constexpr int kXFloats = 2 * 4 * 2 * 32;
constexpr int kLOff = kXOff + 4 * kXFloats;       // row sums: item parity x 128 rows (fp32)
constexpr int kAttnSmemBytes = kLOff + 4 * 2 * kTile + 1024;  // + alignment slack for the 1024-byte-aligned base
static_assert(kAttnSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kAttnTmemCols = 512;
constexpr uint32_t kOCol = kSBufs * 128;          // output accumulator, after the score buffers
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

// The item this CTA runs in its k-th round.  Each round deals gridDim items (longest first), and the rounds
// alternate direction, so a CTA that took one of the longest items of a round takes one of the shortest of
// the next (with causal items of 1 .. nq key blocks this evens the CTAs' loads).  Every item is dealt exactly
// once; the first index past num_items ends a CTA's rounds (only the last round can be partial).
__device__ __forceinline__ int attn_round_item(int k) {
  const int g = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  return k * g + ((k & 1) ? g - 1 - c : c);
}

// The CTA's key blocks in sequence: block j of its e-th item, j = 0 .. i.  The producer and the MMA issuer
// step copies of it (one for the scores, one for the P V products), so they agree on every load and MMA.
struct BlockWalk {
  int e = 0;  // position of the current item in the CTA's sequence
  int t = 0;  // the item (>= num_items: none left)
  AttnItem it{};
  int j = 0;
  __device__ __forceinline__ void start(const AttnParams& a) {
    t = attn_round_item(0);
    if (t < a.num_items) it = attn_item(a, t);
  }
  __device__ __forceinline__ bool valid(const AttnParams& a) const { return t < a.num_items; }
  __device__ __forceinline__ void next(const AttnParams& a) {
    if (++j > it.i) {
      j = 0;
      t = attn_round_item(++e);
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

// 32 lanes x 16 consecutive 32-bit columns from registers into tensor memory
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// true if the phase of `bar` with the given parity has completed (never blocks)
__device__ __forceinline__ bool mbar_test(const uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams a) {
  grid_dependency_wait();  // launched as a dependent of the stream's previous kernel
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;                              // Q slots
  uint8_t* ring = smem + kQSlots * kQBytes;        // K / V ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  float* xslots = reinterpret_cast<float*>(smem + kXOff);
  float* lsum = reinterpret_cast<float*>(smem + kLOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&bars[kBarRingFull + s], 1);
      mbar_init(&bars[kBarRingEmpty + s], 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&bars[kBarSFull + b], 1);
      mbar_init(&bars[kBarPFull + b], kSoftWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kBarQFull + b], 1);
      mbar_init(&bars[kBarQEmpty + b], 1);
      mbar_init(&bars[kBarLFull + b], 4);       // the softmax warps of key half 0
      mbar_init(&bars[kBarLEmpty + b], 4);      // the output warps
      mbar_init(&bars[kBarPV + b], 1);
    }
    mbar_init(&bars[kBarOFull], 1);
    mbar_init(&bars[kBarOEmpty], 4);            // the output warps
    for (int q = 0; q < 4; ++q) mbar_init(&bars[kBarX + q], 2);  // the row quarter's two softmax warps
    mbar_init(&bars[kBarFinal], 1);
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
  uint64_t* ring_full = bars + kBarRingFull;
  uint64_t* ring_empty = bars + kBarRingEmpty;
  uint64_t* q_full = bars + kBarQFull;
  uint64_t* q_empty = bars + kBarQEmpty;
  uint64_t* s_full = bars + kBarSFull;
  uint64_t* p_full = bars + kBarPFull;
  uint64_t* o_full = bars + kBarOFull;
  uint64_t* o_empty = bars + kBarOEmpty;
  uint64_t* l_full = bars + kBarLFull;
  uint64_t* l_empty = bars + kBarLEmpty;
  uint64_t* pv_bar = bars + kBarPV;
  uint64_t* final_bar = bars + kBarFinal;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t g = 0;                       // ring loads issued
    uint32_t ring_issued = 0, ring_parity = 0, q_issued = 0, q_parity = 0;
    // the next S block's K (and, for an item's first block, its Q tile) or the next P V block's V into the
    // next ring slot: one K block is two boxes of 64 dh x 128 keys; one V block (the MN-major B operand) is,
    // per 64-key half, two boxes of 64 dh x 64 keys
    auto load_block = [&](bool is_k, const BlockWalk& w) -> bool {
      if (is_k && w.j == 0) {  // the item's Q tile, once the item two back has issued its last scores
        const int qs = w.e & 1;
        const uint32_t ph = (w.e >> 1) & 1;
        if (!mbar_wait(&q_empty[qs], ph ^ 1, abort_flag, tmo, a.status, kSiteProducerEmpty, w.t)) return false;
        const int qx = w.it.h * kTile;
        const int qy = a.row0 + w.it.b * a.S + w.it.i * kTile;
        uint8_t* dst = sq + qs * kQBytes;
        mbar_arrive_expect_tx(&q_full[qs], kQBytes);
        tma_load_2d(dst, &a.map_qk[w.it.p], &q_full[qs], qx, qy);
        tma_load_2d(dst + kSub, &a.map_qk[w.it.p], &q_full[qs], qx + 64, qy);
        q_issued |= 1u << qs;
        q_parity = (q_parity & ~(1u << qs)) | (ph << qs);
      }
      const uint32_t st = g % kRing, ph = (g / kRing) & 1;
      if (!mbar_wait(&ring_empty[st], ph ^ 1, abort_flag, tmo, a.status, kSiteProducerEmpty, w.t)) return false;
      uint8_t* dst = ring + st * kSlotBytes;
      const int y = a.row0 + w.it.b * a.S + w.j * kTile;
      mbar_arrive_expect_tx(&ring_full[st], kSlotBytes);
      if (is_k) {
        const int kx = (a.Hp + w.it.h) * kTile;
        tma_load_2d(dst, &a.map_qk[w.it.p], &ring_full[st], kx, y);
        tma_load_2d(dst + kSub, &a.map_qk[w.it.p], &ring_full[st], kx + 64, y);
      } else {
        const int vx = (2 * a.Hp + w.it.h) * kTile;
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_2d(dst + kb * kSub, &a.map_v[w.it.p], &ring_full[st], vx, y + kb * 64);
          tma_load_2d(dst + kb * kSub + 8192, &a.map_v[w.it.p], &ring_full[st], vx + 64, y + kb * 64);
        }
      }
      ring_issued |= 1u << st;
      ring_parity = (ring_parity & ~(1u << st)) | (ph << st);
      ++g;
      return true;
    };
    // the MMAs' order: S_0 .. S_2, then per s: P V_s, S_{s+3}
    BlockWalk ws, wv;
    ws.start(a);
    wv.start(a);
    bool ok = true;
    for (int n = 0; n < kSBufs && ok && ws.valid(a); ++n) {
      ok = load_block(true, ws);
      ws.next(a);
    }
    while (ok && wv.valid(a)) {
      ok = load_block(false, wv);
      wv.next(a);
      if (ok && ws.valid(a)) {
        ok = load_block(true, ws);
        ws.next(a);
      }
    }
    // drain: every load issued has landed before the CTA can exit
    volatile int no_abort = 0;
    for (int s = 0; s < kQSlots; ++s)
      if (q_issued & (1u << s)) mbar_wait(&q_full[s], (q_parity >> s) & 1, &no_abort, tmo, a.status, kSiteDrain, 0);
    for (int s = 0; s < kRing; ++s)
      if (ring_issued & (1u << s))
        mbar_wait(&ring_full[s], (ring_parity >> s) & 1, &no_abort, tmo, a.status, kSiteDrain, 1 + s);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, false, true);
    uint32_t g = 0, n_pv = 0;              // ring slots consumed, P V steps issued
    uint32_t s_buf = 0, s_ph = 0;          // score buffer and its phase for the next S step
    uint32_t p_buf = 0, p_ph = 0;          // the same for the next P V step
    BlockWalk ws, wp;
    ws.start(a);
    wp.start(a);
    // S = Q K^T for the next S block into score buffer s_buf
    auto issue_s = [&](bool ready) -> bool {
      const int qs = ws.e & 1;
      const uint32_t st = g % kRing, ph = (g / kRing) & 1;
      if (!ready) {
        if (ws.j == 0 && !mbar_wait(&q_full[qs], (ws.e >> 1) & 1, abort_flag, tmo, a.status, kSiteMmaFull, ws.t))
          return false;
        if (!mbar_wait(&ring_full[st], ph, abort_flag, tmo, a.status, kSiteMmaFull, ws.t)) return false;
      }
      tc_fence_after_sync();
      const uint32_t qa = smem_u32(sq + qs * kQBytes);
      const uint32_t ka = smem_u32(ring + st * kSlotBytes);
      const uint32_t t_s = tmem_base + s_buf * kTile;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t ad = smem_desc_k128(qa + (k >> 2) * kSub) + 2 * (k & 3);
        const uint64_t bd = smem_desc_k128(ka + (k >> 2) * kSub) + 2 * (k & 3);
        mma_bf16_ss(t_s, ad, bd, idesc_s, k != 0 ? 1u : 0u);
      }
      mma_commit(&ring_empty[st]);
      mma_commit(&s_full[s_buf]);
      if (ws.j == ws.it.i) mma_commit(&q_empty[qs]);  // the item's last scores: its Q slot is free
      ++g;
      if (++s_buf == kSBufs) {
        s_buf = 0;
        s_ph ^= 1;
      }
      ws.next(a);
      return true;
    };
    // O += P V for the next P V block, once its probabilities are written (and, for an item's first block,
    // once the output warps have read the previous item's output)
    auto issue_pv = [&](bool ready) -> bool {
      const uint32_t st = g % kRing, ph = (g / kRing) & 1;
      if (!ready) {
        if (wp.j == 0 && !mbar_wait(o_empty, (wp.e & 1) ^ 1, abort_flag, tmo, a.status, kSiteMmaTmemEmpty, wp.t))
          return false;
        if (!mbar_wait(&p_full[p_buf], p_ph, abort_flag, tmo, a.status, kSiteAttnP, wp.t)) return false;
        if (!mbar_wait(&ring_full[st], ph, abort_flag, tmo, a.status, kSiteMmaFull, wp.t)) return false;
      }
      tc_fence_after_sync();
      const uint32_t va = smem_u32(ring + st * kSlotBytes);
      const uint32_t t_p = tmem_base + p_buf * kTile;
      const uint32_t t_o = tmem_base + kOCol;
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // 16 keys per step: 8 columns of P (keys 0-63 at 0-31, 64-127 at 64-95)
        const uint64_t bd = smem_desc_mn128(va + (k >> 2) * kSub) + (2048 >> 4) * (k & 3);
        mma_bf16_ts(t_o, t_p + 64 * (k >> 2) + 8 * (k & 3), bd, idesc_pv, (wp.j | k) != 0 ? 1u : 0u);
      }
      mma_commit(&ring_empty[st]);
      mma_commit(&pv_bar[n_pv & 1]);
      if (wp.j == wp.it.i) mma_commit(o_full);
      ++g;
      ++n_pv;
      if (++p_buf == kSBufs) {
        p_buf = 0;
        p_ph ^= 1;
      }
      wp.next(a);
      return true;
    };
    bool ok = true;
    for (int n = 0; n < kSBufs && ok && ws.valid(a); ++n) ok = issue_s(false);
    while (ok && wp.valid(a)) {
      // a step's barriers tested back to back, without blocking; if any is not complete, the step's bounded
      // waits run one by one
      const bool has_s = ws.valid(a);
      const uint32_t g1 = g + 1;
      const bool ready =
          mbar_test(&p_full[p_buf], p_ph) & mbar_test(&ring_full[g % kRing], (g / kRing) & 1) &
          (wp.j != 0 || mbar_test(o_empty, (wp.e & 1) ^ 1)) &
          (!has_s || (mbar_test(&ring_full[g1 % kRing], (g1 / kRing) & 1) &
                      (ws.j != 0 || mbar_test(&q_full[ws.e & 1], (ws.e >> 1) & 1))));
      ok = issue_pv(ready);
      if (ok && has_s) ok = issue_s(ready);
    }
    mma_commit(final_bar);
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, a.status, kSiteDrain, 99);
  } else if (warp >= kOutWarp0 && warp < kOutWarp0 + 4) {
    // --------------------------------------------------- output
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t to = tmem_base + lane_off + kOCol;
    for (int e = 0, t = attn_round_item(0); t < a.num_items && !*abort_flag; t = attn_round_item(++e)) {
      const AttnItem it = attn_item(a, t);
      const int lb = e & 1;
      if (!mbar_wait(&l_full[lb], (e >> 1) & 1, abort_flag, tmo, a.status, kSiteAttnPV, t) ||
          !mbar_wait(o_full, e & 1, abort_flag, tmo, a.status, kSiteAttnPV, t))
        break;
      tc_fence_after_sync();
      const float inv = 1.0f / lsum[lb * kTile + r];
      const int64_t grow = a.row0 + static_cast<int64_t>(it.b) * a.S + it.i * kTile + r;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o[it.p]) + grow * a.ldo + it.h * kTile);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t o0[32], o1[32];
        tmem_ld_32x32b_x32(to + hb * 64, o0);
        tmem_ld_32x32b_x32(to + hb * 64 + 32, o1);
        tmem_ld_wait();
        if (hb == 1) {  // the output row and its sum are read: the accumulator and the sum's slot are free
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(o_empty);
            mbar_arrive(&l_empty[lb]);
          }
        }
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const uint32_t* oh = q8 < 4 ? o0 + 8 * q8 : o1 + 8 * (q8 - 4);
          float y[8];
#pragma unroll
          for (int e2 = 0; e2 < 8; e2 += 2)
            mul2(y[e2], y[e2 + 1], __uint_as_float(oh[e2]), __uint_as_float(oh[e2 + 1]), inv, inv);
          dst[hb * 8 + q8] = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                                        pack_bf16(y[6], y[7]));
        }
      }
    }
  } else if (warp >= kSoftWarp0) {
    // --------------------------------------------------- softmax
    const int h = (warp - kSoftWarp0) >> 2;  // half of the key block: keys 64 h .. 64 h + 63
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // query row within the tile
    const int rr = r - 64 * h;               // on the diagonal block, keys 64 h + e with e <= rr are visible
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t to = tmem_base + lane_off + kOCol + 64 * h;  // this half of the output row
    uint64_t* xbar = bars + kBarX + quarter;
    float* xq = xslots + quarter * 64;       // + parity * 256 + half * 32 + row
    const float c = a.scale_log2;
    uint32_t s = 0, x_count = 0;             // the CTA's key blocks processed, exchanges made
    uint32_t s_buf = 0, s_ph = 0;            // score buffer of block s and its phase
    // one value with the partner thread of the same row (the other half): both write their own slot, arrive
    // once per warp and read the other's slot.  Slots alternate by parity, so a slot is written again only
    // after the partner has arrived at the next exchange, i.e. after it has read this one.
    auto exchange = [&](float v, float& other, int t) -> bool {
      float* slot = xq + (x_count & 1) * 256;
      slot[h * 32 + lane] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      if (!mbar_wait(xbar, x_count & 1, abort_flag, tmo, a.status, kSiteAttnX, t)) return false;
      other = slot[(1 - h) * 32 + lane];
      ++x_count;
      return true;
    };
    for (int e = 0, t = attn_round_item(0); t < a.num_items && !*abort_flag; t = attn_round_item(++e)) {
      const AttnItem it = attn_item(a, t);
      float m_run = -INFINITY, l_run = 0.0f;
      bool ok = true;
      for (int j = 0; j <= it.i; ++j, ++s) {
        const uint32_t sb = s_buf;
        if (!mbar_wait(&s_full[sb], s_ph, abort_flag, tmo, a.status, kSiteEpilogueTmemFull, t)) {
          ok = false;
          break;
        }
        if (++s_buf == kSBufs) {
          s_buf = 0;
          s_ph ^= 1;
        }
        tc_fence_after_sync();
        const uint32_t ts = tmem_base + lane_off + sb * kTile + 64 * h;  // this half's scores / probabilities
        const bool diag = j == it.i;
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(ts, v0);
        tmem_ld_32x32b_x32(ts + 32, v1);
        tmem_ld_wait();
        float mx = -INFINITY;
        if (diag) {
#pragma unroll
          for (int e2 = 0; e2 < 32; ++e2) {
            if (e2 <= rr) mx = fmaxf(mx, __uint_as_float(v0[e2]));
            if (32 + e2 <= rr) mx = fmaxf(mx, __uint_as_float(v1[e2]));
          }
        } else {
#pragma unroll
          for (int e2 = 0; e2 < 32; ++e2) mx = max3(mx, __uint_as_float(v0[e2]), __uint_as_float(v1[e2]));
        }
        float mx_other;
        if (!exchange(mx, mx_other, t)) {
          ok = false;
          break;
        }
        const float m_blk = fmaxf(mx, mx_other) * c;  // the row's maximum, the same in both partners
        const bool grow_m = m_blk > m_run + kRescaleLog2;
        float alpha = 1.0f;
        if (grow_m) {
          alpha = ex2_approx(m_run - m_blk);  // 0 for the first block
          m_run = m_blk;
        }
        // the 64 probabilities as bf16 pairs (keys 64 h + 2q, 64 h + 2q + 1 -> column q of this half), over
        // score columns this thread has read (the P V product that read this buffer's previous probabilities
        // preceded these scores).  diag_c: std::true_type for the diagonal block (keys past the row masked),
        // std::false_type for the others, so that the blocks below it carry no masking
        float sum_even = 0.0f, sum_odd = 0.0f;
        const float nm = -m_run;
        // x: 32 scores (keys 64 h + kb + e), packed into 16 columns
        auto probs = [&](auto diag_c, const uint32_t (&x)[32], int kb, uint32_t (&pk)[16]) {
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            float y0, y1;
            fma2(y0, y1, __uint_as_float(x[2 * e2]), __uint_as_float(x[2 * e2 + 1]), c, c, nm, nm);
            float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
            if constexpr (decltype(diag_c)::value) {
              p0 = kb + 2 * e2 <= rr ? p0 : 0.0f;
              p1 = kb + 2 * e2 + 1 <= rr ? p1 : 0.0f;
            }
            add2(sum_even, sum_odd, sum_even, sum_odd, p0, p1);
            pk[e2] = pack_bf16(p0, p1);
          }
        };
        {
          uint32_t pk[16];
          if (diag) probs(std::true_type{}, v0, 0, pk);
          else probs(std::false_type{}, v0, 0, pk);
          tmem_st_32x32b_x16(ts, pk);
        }
        {
          uint32_t pk[16];
          if (diag) probs(std::true_type{}, v1, 32, pk);
          else probs(std::false_type{}, v1, 32, pk);
          tmem_st_32x32b_x16(ts + 16, pk);
        }
        // rescaling the output (rare) waits for the previous block's P V product.  Products of even and odd
        // index complete on two barriers; the one of block s - 1 is the next phase of its barrier: the product
        // of block s - 3 preceded these scores, and that of block s + 1 cannot start before this block's
        // probabilities.  Tensor-memory loads and stores are warp-wide: the whole warp rescales its half rows
        // (alpha = 1 where the maximum stayed).
        if (j > 0 && __any_sync(0xffffffffu, grow_m)) {
          if (!mbar_wait(&pv_bar[(s - 1) & 1], ((s - 1) >> 1) & 1, abort_flag, tmo, a.status, kSiteAttnPV, t)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(to + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e2 = 0; e2 < 32; e2 += 2) {
              float y0, y1;
              mul2(y0, y1, __uint_as_float(v[e2]), __uint_as_float(v[e2 + 1]), alpha, alpha);
              v[e2] = __float_as_uint(y0);
              v[e2 + 1] = __float_as_uint(y1);
            }
            tmem_st_32x32b_x32(to + cc * 32, v);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();  // the warp's probabilities (and any rescaled output) are written: one arrival per warp
        if (lane == 0) mbar_arrive(&p_full[sb]);
        l_run = l_run * alpha + (sum_even + sum_odd);
      }
      if (!ok) break;
      // the row sum for the output warps, in the slot of this item's parity once they have read the item two back
      float l_other;
      if (!exchange(l_run, l_other, t)) break;
      if (h == 0) {
        if (!mbar_wait(&l_empty[e & 1], ((e >> 1) & 1) ^ 1, abort_flag, tmo, a.status, kSiteMmaTmemEmpty, t)) break;
        lsum[(e & 1) * kTile + r] = l_run + l_other;
        __syncwarp();
        if (lane == 0) mbar_arrive(&l_full[e & 1]);
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
  const cudaError_t st = launch_after_previous(reinterpret_cast<const void*>(&attn_fwd_kernel), dim3(grid),
                                               dim3(kAttnThreads), kAttnSmemBytes, stream, args);
  if (st != cudaSuccess) {
    if (err) *err = std::string("attention launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace domino
