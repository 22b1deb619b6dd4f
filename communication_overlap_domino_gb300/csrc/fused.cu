// Fused forward pass: both projections and the shard-sum of every chunk in ONE
// persistent, cooperative launch.
//
// The Domino page ("Domino: Eliminating Communication in LLM Training via
// Generic Tensor Slicing and Overlapping", Abstract) hides each piece's
// communication behind the computation of the next piece.  Here the pieces are
// made as small as one output tile: the shard-sum of output tile (k, m, n) of
// chunk k starts as soon as the P row-parallel partials of that tile exist, on
// reducer warps of the same SMs that keep running GEMM tiles, so the
// memory-bound exchange overlaps tensor-core work at tile granularity and only
// the reduction of the last tiles is left exposed.
//
// Work, in one global order shared by all CTAs (static round-robin, tile t is
// processed by CTA t mod gridDim.x, in increasing t):
//   for each chunk k:  GEMM1 tiles, then GEMM2 tiles (shard, column block, row
//                      block; the last chunk's GEMM2 in groups of 8 row blocks,
//                      its last group column by column, and cut to 4 when that
//                      leaves it two waves of tiles)
// Dependencies, through counters in the workspace (release/acquire at GPU scope):
//   GEMM2 tile (k, m, n, p) needs H_{k,p}[row block m] complete: hcnt[k][p][m]
//     counts finished 32-row quarters of GEMM1 tiles (target tiles_n1 * 4); the
//     TMA producer polls it before loading H (then a proxy fence orders the
//     generic-proxy stores before its async-proxy reads).
//   shard-sum of (k, m, n), quarter q: zcnt[k][m][n][q] counts the GEMM2 tiles
//     whose quarter q is stored (target P).  The shard-sum runs in 8-row pieces
//     taken from a kernel-wide queue (an atomic ticket) by the reducer warps,
//     and by every other warp once its own role is done.
// GEMM tiles never wait on the reducers and a GEMM2 tile only waits on GEMM1
// tiles earlier in the global order, so with all CTAs resident (the cooperative
// launch guarantees it) every wait ends; each is still bounded by timeout_ns.
//
// Warp roles (256 threads, one CTA per SM):
//   warp 0 lane 0: TMA producer      warp 1: TMEM allocator, lane 0 issues MMAs
//   warps 2..5   : epilogue          warps 6..7: reducers (shard-sum)
#include <cuda_bf16.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "epilogue.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace domino {

namespace {

constexpr int kFusedThreads = 256;  // 8 warps: 2 per SM sub-partition, so up to 255 registers
constexpr int kFirstReducerWarp = 6;

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* ptr, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_u4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr)
               : "memory");
  return v;
}

struct FusedTile {
  int phase;  // 0: GEMM1 (column-parallel + activation), 1: GEMM2 (row-parallel partial)
  int k, p, m, n;
};

// Tiles of one phase of one chunk, in groups of G row blocks: for each group:
// for each shard p: for each column block n: for each row block of the group.
// With G = all row blocks this is the order of the separate launches (a column
// block of the weights is loaded once and reused by every row block while it is
// in L2).  The last chunk's GEMM2 uses smaller groups, so the P partials of its
// first output tiles are complete -- and their shard-sum runs -- while the rest
// of the chunk is still being multiplied; its last group is taken column
// block by column block, and (when it keeps two waves of tiles) cut to G / 2
// row blocks (the group before it takes the rest, so the weights are read as
// often as with equal groups), because the shard-sum of that last group is
// the one reduction nothing overlaps.
constexpr int kLastChunkGroupM = 8;

__device__ __forceinline__ void grouped_coords(int r, int G, int P, int tiles_m, int tiles_n, int& p, int& m,
                                               int& n) {
  const int full = P * tiles_n * G;
  const int g = r / full;
  const int r2 = r - g * full;
  const int rows_left = tiles_m - g * G;
  const int gm = rows_left < G ? rows_left : G;
  const int per_p = tiles_n * gm;
  p = r2 / per_p;
  const int r3 = r2 - p * per_p;
  n = r3 / gm;
  m = g * G + (r3 - n * gm);
}

// The same order for the last chunk's GEMM2: with n = ceil(tiles_m / G) >= 2
// groups, groups 0 .. n-3 hold G row blocks, group n-2 the rest but the last
// L = G / 2, group n-1 those L.  The last group goes column block by column
// block (for each n: for each shard: for each row block), so that its output
// tiles get their P partials -- and their shard-sum starts -- one column block
// after another instead of all during the last shard's pass; its rows of H
// (L row blocks of every shard) stay in L2 across the column blocks.
__device__ __forceinline__ void grouped_coords_tail(int r, int G, int P, int tiles_m, int tiles_n, int& p, int& m,
                                                    int& n) {
  const int ngroups = (tiles_m + G - 1) / G;
  const int L = G / 2;
  const int full = P * tiles_n * G;
  const int uniform = (ngroups - 2) * full;
  if (ngroups < 2 || L < 1 || r < uniform) {
    grouped_coords(r, G, P, tiles_m, tiles_n, p, m, n);
    return;
  }
  int r2 = r - uniform;
  const int m0a = (ngroups - 2) * G;
  const int size_a = tiles_m - m0a - L;
  if (r2 < P * tiles_n * size_a) {
    const int per_p = tiles_n * size_a;
    p = r2 / per_p;
    const int r3 = r2 - p * per_p;
    n = r3 / size_a;
    m = m0a + (r3 - n * size_a);
    return;
  }
  r2 -= P * tiles_n * size_a;
  const int per_n = P * L;
  n = r2 / per_n;
  const int r3 = r2 - n * per_n;
  p = r3 / L;
  m = tiles_m - L + (r3 - p * L);
}

// The graded order pays only when the cut-down last group still has tiles
// enough (two waves over the CTAs or clusters) for the shard-sum of the group
// before it to hide behind: on the GPT-style layer, whose last group would be
// about one wave, it made the layer 1.9% slower.
__device__ __forceinline__ bool graded_tail(int last_group_tiles, int units) {
  return last_group_tiles >= 2 * units;
}

// Without the grading: equal groups of G, the last one (whatever its size)
// taken column block by column block.
__device__ __forceinline__ void grouped_coords_last_cols(int r, int G, int P, int tiles_m, int tiles_n, int& p,
                                                         int& m, int& n) {
  const int ngroups = (tiles_m + G - 1) / G;
  const int uniform = (ngroups - 1) * P * tiles_n * G;
  if (r < uniform) {
    grouped_coords(r, G, P, tiles_m, tiles_n, p, m, n);
    return;
  }
  const int L = tiles_m - (ngroups - 1) * G;
  const int r2 = r - uniform;
  const int per_n = P * L;
  n = r2 / per_n;
  const int r3 = r2 - n * per_n;
  p = r3 / L;
  m = tiles_m - L + (r3 - p * L);
}

__device__ __forceinline__ FusedTile fused_tile(const FusedParams& f, int t) {
  FusedTile T;
  const int per_chunk = f.tiles_a + f.tiles_b;
  T.k = t / per_chunk;
  int r = t - T.k * per_chunk;
  if (r < f.tiles_a) {
    T.phase = 0;
    grouped_coords(r, f.tiles_m, f.P, f.tiles_m, f.tiles_n1, T.p, T.m, T.n);
  } else {
    T.phase = 1;
    if (T.k == f.mu - 1) {
      const int G = f.tiles_m < kLastChunkGroupM ? f.tiles_m : kLastChunkGroupM;
      if (graded_tail(f.P * f.tiles_n2 * (G / 2), static_cast<int>(gridDim.x)))
        grouped_coords_tail(r - f.tiles_a, G, f.P, f.tiles_m, f.tiles_n2, T.p, T.m, T.n);
      else
        grouped_coords_last_cols(r - f.tiles_a, G, f.P, f.tiles_m, f.tiles_n2, T.p, T.m, T.n);
    } else {
      grouped_coords(r - f.tiles_a, f.tiles_m, f.P, f.tiles_m, f.tiles_n2, T.p, T.m, T.n);
    }
  }
  return T;
}

// Paired kernel: tiles of 256 rows (T.m counts 256-row blocks; the even CTA
// owns 128-row block 2*T.m, the odd one 2*T.m + 1), same order as above.
__device__ __forceinline__ FusedTile fused_pair_tile(const FusedParams& f, int t) {
  FusedTile T;
  const int per_chunk = f.tiles_a2 + f.tiles_b2;
  T.k = t / per_chunk;
  int r = t - T.k * per_chunk;
  if (r < f.tiles_a2) {
    T.phase = 0;
    grouped_coords(r, f.tiles_m2, f.P, f.tiles_m2, f.tiles_n1, T.p, T.m, T.n);
  } else {
    T.phase = 1;
    const int g2 = kLastChunkGroupM / 2;
    if (T.k == f.mu - 1) {
      const int G = f.tiles_m2 < g2 ? f.tiles_m2 : g2;
      if (graded_tail(f.P * f.tiles_n2 * (G / 2), static_cast<int>(gridDim.x >> 1)))
        grouped_coords_tail(r - f.tiles_a2, G, f.P, f.tiles_m2, f.tiles_n2, T.p, T.m, T.n);
      else
        grouped_coords_last_cols(r - f.tiles_a2, G, f.P, f.tiles_m2, f.tiles_n2, T.p, T.m, T.n);
    } else {
      grouped_coords(r - f.tiles_a2, f.tiles_m2, f.P, f.tiles_m2, f.tiles_n2, T.p, T.m, T.n);
    }
  }
  return T;
}

// Waits until *ctr >= target (acquire).  Bounded: gives up on *abort or after
// timeout_ns, recording the error.  Executed by every lane of a warp, or by a
// single thread.
__device__ __forceinline__ bool wait_counter(const uint32_t* ctr, uint32_t target, volatile int* abort,
                                             uint64_t timeout_ns, DeviceStatus* st, uint32_t where, uint32_t aux) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(ctr) >= target) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort = 1;
      record_error(st, kStatusTimeout, where, aux);
      return false;
    }
  }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] += __uint_as_float(w[q] << 16);
    acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Shard-sum of up to 32 rows x 8 columns per lane (the lane's 16-byte slice of
// the 256-column tile): y = bf16(sum_{p=0}^{P-1} z_p), fp32 accumulation in
// shard order.  Several rows' loads are in flight per step.
template <int NP, bool F32>
__device__ __forceinline__ void reduce_rows(const FusedParams& f, int64_t row0, int nrows, int64_t col, int P) {
  if constexpr (NP == 0) {
    // any shard count: one row at a time, loads consumed as they arrive
    for (int rr = 0; rr < nrows; ++rr) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      for (int s = 0; s < P; ++s) {
        if constexpr (F32) {
          const float* src = static_cast<const float*>(f.z[s]) + (row0 + rr) * f.d + col;
          const uint4 lo = ld_u4(src), hi = ld_u4(src + 4);
          acc[0] += __uint_as_float(lo.x);
          acc[1] += __uint_as_float(lo.y);
          acc[2] += __uint_as_float(lo.z);
          acc[3] += __uint_as_float(lo.w);
          acc[4] += __uint_as_float(hi.x);
          acc[5] += __uint_as_float(hi.y);
          acc[6] += __uint_as_float(hi.z);
          acc[7] += __uint_as_float(hi.w);
        } else {
          add_bf16x8(acc, ld_u4(static_cast<const __nv_bfloat16*>(f.z[s]) + (row0 + rr) * f.d + col));
        }
      }
      uint4 o;
      o.x = pack2(acc[0], acc[1]);
      o.y = pack2(acc[2], acc[3]);
      o.z = pack2(acc[4], acc[5]);
      o.w = pack2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(f.y) + (row0 + rr) * f.d + col) = o;
    }
    return;
  }
  // rows in flight per step: about 16 sixteen-byte loads per lane
  constexpr int kNP = NP > 0 ? NP : 1;
  constexpr int kVec = F32 ? 2 : 1;
  constexpr int kRowsRaw = 16 / (kNP * kVec);
  constexpr int kRows = kRowsRaw < 1 ? 1 : (kRowsRaw > 4 ? 4 : kRowsRaw);
  for (int rr = 0; rr < nrows; rr += kRows) {
    const int nr = nrows - rr >= kRows ? kRows : nrows - rr;
    uint4 x[kRows][kNP][kVec];
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int s = 0; s < kNP; ++s)
#pragma unroll
        for (int v = 0; v < kVec; ++v)
          if (i < nr) {
            const uint8_t* base = static_cast<const uint8_t*>(f.z[s]);
            x[i][s][v] = ld_u4(base + ((row0 + rr + i) * f.d + col) * (F32 ? 4 : 2) + 16 * v);
          }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      if (i < nr) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int s = 0; s < kNP; ++s) {
          if constexpr (F32) {
            acc[0] += __uint_as_float(x[i][s][0].x);
            acc[1] += __uint_as_float(x[i][s][0].y);
            acc[2] += __uint_as_float(x[i][s][0].z);
            acc[3] += __uint_as_float(x[i][s][0].w);
            acc[4] += __uint_as_float(x[i][s][kVec - 1].x);
            acc[5] += __uint_as_float(x[i][s][kVec - 1].y);
            acc[6] += __uint_as_float(x[i][s][kVec - 1].z);
            acc[7] += __uint_as_float(x[i][s][kVec - 1].w);
          } else {
            add_bf16x8(acc, x[i][s][0]);
          }
        }
        uint4 o;
        o.x = pack2(acc[0], acc[1]);
        o.y = pack2(acc[2], acc[3]);
        o.z = pack2(acc[4], acc[5]);
        o.w = pack2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(f.y) + (row0 + rr + i) * f.d + col) = o;
      }
    }
  }
}

template <bool F32>
__device__ __forceinline__ void reduce_dispatch(const FusedParams& f, int64_t row0, int nrows, int64_t col) {
  switch (f.P) {
    case 1: reduce_rows<1, F32>(f, row0, nrows, col, 1); break;
    case 2: reduce_rows<2, F32>(f, row0, nrows, col, 2); break;
    case 4: reduce_rows<4, F32>(f, row0, nrows, col, 4); break;
    case 8: reduce_rows<8, F32>(f, row0, nrows, col, 8); break;
    default: reduce_rows<0, F32>(f, row0, nrows, col, f.P); break;
  }
}

// Takes reduction pieces (8 rows x 256 columns of one output tile) from the
// kernel-wide queue in order and sums each one once the P partials of its
// 32-row quarter (counter zcnt[j / 4]) are stored.  Pieces are small so that
// the last ones, which nothing else overlaps, finish quickly: one warp keeps
// about 8 KB of loads in flight.  Run by the reducer warps from the start and by
// every other warp once its own role is done (so a piece never waits on work of
// the warp that holds it).  Returns false if a wait gave up.
constexpr int kPieceRows = 8;

template <bool F32>
__device__ __forceinline__ bool run_reduction_pieces(const FusedParams& f, volatile int* abort, int lane) {
  constexpr int kPiecesPerQuarter = 32 / kPieceRows;
  const int num_pieces = f.num_red_items * 4 * kPiecesPerQuarter;
  const int per_k = f.tiles_m * f.tiles_n2;
  while (!*abort) {
    int j = 0;
    if (lane == 0) j = static_cast<int>(atomicAdd(f.red_next, 1u));
    j = __shfl_sync(0xffffffffu, j, 0);
    if (j >= num_pieces) break;
    const int quarter_id = j / kPiecesPerQuarter;  // index into zcnt
    const int sub = j - quarter_id * kPiecesPerQuarter;
    const int item = quarter_id >> 2, q = quarter_id & 3;
    const int k = item / per_k;
    const int r = item - k * per_k;
    const int m = r / f.tiles_n2;
    const int n = r - m * f.tiles_n2;
    if (!wait_counter(f.zcnt + quarter_id, static_cast<uint32_t>(f.P), abort, f.timeout_ns, f.status, kSiteFusedZ,
                      quarter_id))
      return false;
    const int row_lo = m * kBM + q * 32 + sub * kPieceRows;
    int nrows = f.Mc - row_lo;
    nrows = nrows > kPieceRows ? kPieceRows : nrows;
    const int64_t col = static_cast<int64_t>(n) * kBN + lane * 8;
    if (nrows > 0 && col < f.d) reduce_dispatch<F32>(f, static_cast<int64_t>(k) * f.Mc + row_lo, nrows, col);
    __syncwarp();
    if (lane == 0)
      atomicMax(reinterpret_cast<unsigned long long*>(&f.timeline[2]),
                static_cast<unsigned long long>(globaltimer_ns()));
  }
  return true;
}

template <int EPI_A, int EPI_B>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_fwd_kernel(const __grid_constant__ FusedParams f) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + kStages * kAStageBytes;
  uint8_t* smem_out = smem_b + kStages * kBStageBytes;  // epilogue staging, 4 warps x 8 KB
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem_out + kStageOutBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* tfull_bar = empty_bar + kStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* final_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 4 * 32);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    atomicMax(reinterpret_cast<unsigned long long*>(&f.timeline[0]),  // ~start: zero is the initial value
              ~static_cast<unsigned long long>(globaltimer_ns()));
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = f.num_gemm_tiles;
  const uint64_t tmo = f.timeout_ns;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    prefetch_tmap(&f.map_x);
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    const uint64_t keep_a = l2_policy_evict_last();  // X and H: re-read by every column block
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
      const FusedTile T = fused_tile(f, t);
      const CUtensorMap *ma, *mb0, *mb1;
      int ya, yb0, yb1, nkb;
      if (T.phase == 0) {
        ma = &f.map_x;
        mb0 = &f.map_w1a[T.p];
        mb1 = &f.map_w1b[T.p];
        ya = T.k * f.Mc + T.m * kBM;
        yb0 = T.n * f.n_tile1;
        yb1 = yb0 + f.b1_off1;
        nkb = f.kb1;
      } else {
        const uint32_t* ctr = f.hcnt + (T.k * f.P + T.p) * f.tiles_m + T.m;
        if (!wait_counter(ctr, static_cast<uint32_t>(f.tiles_n1) * 4, abort_flag, tmo, f.status, kSiteFusedH, t))
          break;
        fence_proxy_async_global();  // H was written through the generic proxy; TMA reads it
        ma = &f.map_h[T.p];
        mb0 = &f.map_w2[T.p];
        mb1 = mb0;
        ya = T.k * f.Mc + T.m * kBM;
        yb0 = T.n * kBN;
        yb1 = yb0 + kBN / 2;
        nkb = f.kb2;
      }
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, tmo, f.status, kSiteProducerEmpty, t)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem_a + stage * kAStageBytes;
        uint8_t* sb = smem_b + stage * kBStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kAStageBytes + kBStageBytes);
        const int k0 = kb * kBK;
        tma_load_2d(sa, ma, &full_bar[stage], k0, ya, keep_a);
        tma_load_2d(sb, mb0, &full_bar[stage], k0, yb0);
        tma_load_2d(sb + kBStageBytes / 2, mb1, &full_bar[stage], k0, yb1);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    for (int s = 0; s < kStages; ++s) {
      if (issued_mask & (1u << s)) {
        volatile int no_abort = 0;
        mbar_wait(&full_bar[s], (issued_parity >> s) & 1u, &no_abort, tmo, f.status, kSiteDrain, s);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
    uint32_t stage = 0, phase = 0;
    int i = 0;
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x, ++i) {
      const FusedTile T = fused_tile(f, t);
      const int nkb = T.phase == 0 ? f.kb1 : f.kb2;
      const uint32_t acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag, tmo, f.status, kSiteMmaTmemEmpty, t)) break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + acc * kBN;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, abort_flag, tmo, f.status, kSiteMmaFull, t)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t adesc = smem_desc_k128(smem_u32(smem_a + stage * kAStageBytes));
        const uint64_t bdesc = smem_desc_k128(smem_u32(smem_b + stage * kBStageBytes));
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
        mma_commit(&empty_bar[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      mma_commit(&tfull_bar[acc]);
    }
    mma_commit(final_bar);
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, f.status, kSiteDrain, 99);
  } else if (warp >= 2 && warp < kFirstReducerWarp) {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint8_t* stage = smem_out + (warp - 2) * kStageOutBytesPerWarp;
    int sbuf = 0;
    int i = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++i) {
      const uint32_t acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, tmo, f.status, kSiteEpilogueTmemFull, t)) break;
      tc_fence_after_sync();
      const FusedTile T = fused_tile(f, t);
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
      if (T.phase == 0) {
        const EpiArgs e{f.h[T.p], f.aux[T.p], f.Fp, f.ld_aux, f.aux_u_off, 0,
                        f.Mc, static_cast<int32_t>(T.k * f.Mc), static_cast<int32_t>(f.Fp),
                        &f.map_hout[T.p], stage};
        epilogue_tile<EPI_A>(e, tacc, T.m, T.n * f.n_tile1, row_in_tile, sbuf);
        tc_fence_before_sync();
        mbar_arrive(&tempty_bar[acc]);
        // publish: the TMA stores of this quarter are complete, then release the counter
        if (lane == 0) bulk_wait_group<0>();
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_gpu_add(f.hcnt + (T.k * f.P + T.p) * f.tiles_m + T.m, 1);
      } else {
        const EpiArgs e{f.z[T.p], nullptr, f.d, 0, 0, 0, f.Mc, static_cast<int32_t>(T.k * f.Mc),
                        static_cast<int32_t>(f.d), &f.map_zout[T.p], stage};
        epilogue_tile<EPI_B>(e, tacc, T.m, T.n * kBN, row_in_tile, sbuf);
        tc_fence_before_sync();
        mbar_arrive(&tempty_bar[acc]);
        if (lane == 0) bulk_wait_group<0>();
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0)
          red_release_gpu_add(f.zcnt + ((static_cast<int64_t>(T.k) * f.tiles_m + T.m) * f.tiles_n2 + T.n) * 4 +
                                  quarter, 1);
      }
    }
    if (lane == 0)
      atomicMax(reinterpret_cast<unsigned long long*>(&f.timeline[1]),
                static_cast<unsigned long long>(globaltimer_ns()));
    __syncwarp();
    run_reduction_pieces<EPI_B == EPI_Z_F32>(f, abort_flag, lane);
  } else if (warp >= kFirstReducerWarp) {
    // -------------------------------------------------------------- reducers
    run_reduction_pieces<EPI_B == EPI_Z_F32>(f, abort_flag, lane);
  }

  __syncwarp();
  if (warp < 2) {
    // the producer and MMA warps join the shard-sum once their roles are done
    run_reduction_pieces<EPI_B == EPI_Z_F32>(f, abort_flag, lane);
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}


// The fused forward pass with paired-CTA tiles: each 2-CTA cluster computes
// 256-row tiles with tcgen05 cta_group::2 MMAs issued by its even CTA (see
// gemm_pair.cu for the operand split and the barrier protocol).  Each CTA's
// epilogue drains, stores and publishes its own 128-row block, so the counters
// and the shard-sum pieces are the same as in the one-CTA kernel.  The odd
// CTA's warp 1, which issues no MMAs, works on the shard-sum from the start.
template <int EPI_A, int EPI_B, bool B2_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFusedThreads, 1)
    fused_fwd_pair_kernel(const __grid_constant__ FusedParams f) {
  constexpr int kPStages = 6;
  constexpr int kPA = 128 * kBK * 2, kPB = 128 * kBK * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + kPStages * kPA;
  uint8_t* smem_out = smem_b + kPStages * kPB;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem_out + kStageOutBytes);
  uint64_t* empty_bar = full_bar + kPStages;
  uint64_t* tfull_bar = empty_bar + kPStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* final_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 2 * 4 * 32);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    atomicMax(reinterpret_cast<unsigned long long*>(&f.timeline[0]),  // ~start: zero is the initial value
              ~static_cast<unsigned long long>(globaltimer_ns()));
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_alloc_permit_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = f.num_pair_tiles;
  const uint64_t tmo = f.timeout_ns;
  const int num_clusters = gridDim.x >> 1;
  const int cluster_id = blockIdx.x >> 1;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    if (!f.a2_input) prefetch_tmap(&f.map_x);
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), 0);
    // X (GEMM1) and H (GEMM2) are the operands every column block re-reads while the weights stream past:
    // their lines are the last the L2 gives up
    const uint64_t keep_a = l2_policy_evict_last();
    for (int t = cluster_id; t < num_tiles && !*abort_flag; t += num_clusters) {
      const FusedTile T = fused_pair_tile(f, t);
      const int m = 2 * T.m + static_cast<int>(rank);  // this CTA's 128-row block
      const CUtensorMap *ma, *mb;
      int ya, yb, nkb;
      if (T.phase == 0) {
        ma = &f.map_x;
        mb = leader ? &f.map_w1a[T.p] : &f.map_w1b[T.p];
        ya = T.k * f.Mc + m * kBM;
        yb = T.n * f.n_tile1 + (leader ? 0 : f.b1_off1);
        nkb = f.kb1;
      } else {
        if (m < f.tiles_m && !f.a2_input) {
          const uint32_t* ctr = f.hcnt + (T.k * f.P + T.p) * f.tiles_m + m;
          if (!wait_counter(ctr, static_cast<uint32_t>(f.tiles_n1) * 4, abort_flag, tmo, f.status, kSiteFusedH, t))
            break;
          fence_proxy_async_global();
        }
        ma = &f.map_h[T.p];
        mb = &f.map_w2[T.p];
        ya = T.k * f.Mc + m * kBM;
        yb = T.n * kBN + (leader ? 0 : kBN / 2);
        nkb = f.kb2;
      }
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, tmo, f.status, kSiteProducerEmpty, t)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem_a + stage * kPA;
        uint8_t* sb = smem_b + stage * kPB;
        if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * (kPA + kPB));
        const uint32_t bar = full0 + stage * 8;
        const int k0 = kb * kBK;
        tma_load_2d_pair(sa, ma, bar, k0, ya, keep_a);
        if (B2_MN && T.phase == 1) {
          // the CTA's 128 output columns of B, stored [K][N]: two boxes of 64 columns x 64 K rows
          tma_load_2d_pair(sb, mb, bar, yb, k0);
          tma_load_2d_pair(sb + 8192, mb, bar, yb + 64, k0);
        } else {
          tma_load_2d_pair(sb, mb, bar, k0, yb);
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    if (leader) {
      for (int s = 0; s < kPStages; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait_cluster(&full_bar[s], (issued_parity >> s) & 1u, &no_abort, tmo, f.status, kSiteDrain, s);
        }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------- MMA issuer (even CTA)
    constexpr uint32_t idesc_a = idesc_bf16_f32(256, kBN);
    constexpr uint32_t idesc_b = idesc_bf16_f32(256, kBN, false, B2_MN);
    uint32_t stage = 0, phase = 0;
    int i = 0;
    for (int t = cluster_id; t < num_tiles && !*abort_flag; t += num_clusters, ++i) {
      const FusedTile T = fused_pair_tile(f, t);
      const int nkb = T.phase == 0 ? f.kb1 : f.kb2;
      const bool b_mn = B2_MN && T.phase == 1;
      const uint32_t acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1, abort_flag, tmo, f.status, kSiteMmaTmemEmpty, t)) break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + acc * kBN;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_cluster(&full_bar[stage], phase, abort_flag, tmo, f.status, kSiteMmaFull, t)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t adesc = smem_desc_k128(smem_u32(smem_a + stage * kPA));
        if (b_mn) {  // MN-major B: a K step of 16 rows advances 2 KB
          const uint64_t bdesc = smem_desc_mn128(smem_u32(smem_b + stage * kPB));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ss_pair(d_tmem, adesc + 2 * k, bdesc + (2048 >> 4) * k, idesc_b, (kb | k) != 0 ? 1u : 0u);
        } else {
          const uint64_t bdesc = smem_desc_k128(smem_u32(smem_b + stage * kPB));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ss_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_a, (kb | k) != 0 ? 1u : 0u);
        }
        mma_commit_pair_multicast(&empty_bar[stage], 0x3);
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      mma_commit_pair_multicast(&tfull_bar[acc], 0x3);
    }
    mma_commit_pair_multicast(final_bar, 0x1);
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, f.status, kSiteDrain, 99);
  } else if (warp >= 2 && warp < kFirstReducerWarp) {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint8_t* stage = smem_out + (warp - 2) * kStageOutBytesPerWarp;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty_bar[0]), 0);
    int sbuf = 0;
    int i = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++i) {
      const uint32_t acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, tmo, f.status, kSiteEpilogueTmemFull, t)) break;
      tc_fence_after_sync();
      const FusedTile T = fused_pair_tile(f, t);
      const int m = 2 * T.m + static_cast<int>(rank);
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
      if (T.phase == 0) {
        const EpiArgs e{f.h[T.p], f.aux[T.p], f.Fp, f.ld_aux, f.aux_u_off, 0,
                        f.Mc, static_cast<int32_t>(T.k * f.Mc), static_cast<int32_t>(f.Fp),
                        &f.map_hout[T.p], stage};
        epilogue_tile<EPI_A>(e, tacc, m, T.n * f.n_tile1, row_in_tile, sbuf);
      } else {
        const EpiArgs e{f.z[T.p], nullptr, f.d, 0, 0, 0, f.Mc, static_cast<int32_t>(T.k * f.Mc),
                        static_cast<int32_t>(f.d), &f.map_zout[T.p], stage};
        epilogue_tile<EPI_B>(e, tacc, m, T.n * kBN, row_in_tile, sbuf);
      }
      tc_fence_before_sync();
      if (leader)
        mbar_arrive(&tempty_bar[acc]);
      else
        mbar_arrive_cluster(tempty_leader + acc * 8);
      if (m < f.tiles_m) {
        // publish: this quarter's stores are complete, then release its counter
        if (lane == 0) bulk_wait_group<0>();
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          if (T.phase == 0)
            red_release_gpu_add(f.hcnt + (T.k * f.P + T.p) * f.tiles_m + m, 1);
          else
            red_release_gpu_add(
                f.zcnt + ((static_cast<int64_t>(T.k) * f.tiles_m + m) * f.tiles_n2 + T.n) * 4 + quarter, 1);
        }
      }
    }
    if (lane == 0) {
      bulk_wait_group<0>();
      atomicMax(reinterpret_cast<unsigned long long*>(&f.timeline[1]),
                static_cast<unsigned long long>(globaltimer_ns()));
    }
    __syncwarp();
    run_reduction_pieces<EPI_B == EPI_Z_F32>(f, abort_flag, lane);
  } else if (warp >= kFirstReducerWarp || (warp == 1 && !leader)) {
    // -------------------------------------------------------------- reducers
    run_reduction_pieces<EPI_B == EPI_Z_F32>(f, abort_flag, lane);
  }

  __syncwarp();
  if (warp == 0 || (warp == 1 && leader)) run_reduction_pieces<EPI_B == EPI_Z_F32>(f, abort_flag, lane);
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int A, int B>
void* fused_ptr() {
  return reinterpret_cast<void*>(&fused_fwd_kernel<A, B>);
}

template <int A, int B>
void* fused_pair_ptr() {
  return reinterpret_cast<void*>(&fused_fwd_pair_kernel<A, B, false>);
}

// The GEMM2-only launches (no GEMM1 phase): with the MN-major weight shard as B (the backward's partial input
// gradients) or K-major (the forward identity kernel's GEMM2 phase: a row-parallel projection).
void* fused_gemm2_kernel_for(bool f32, bool b_mn) {
  if (b_mn)
    return f32 ? reinterpret_cast<void*>(&fused_fwd_pair_kernel<EPI_H_IDENTITY, EPI_Z_F32, true>)
               : reinterpret_cast<void*>(&fused_fwd_pair_kernel<EPI_H_IDENTITY, EPI_Z_BF16, true>);
  return f32 ? reinterpret_cast<void*>(&fused_fwd_pair_kernel<EPI_H_IDENTITY, EPI_Z_F32, false>)
             : reinterpret_cast<void*>(&fused_fwd_pair_kernel<EPI_H_IDENTITY, EPI_Z_BF16, false>);
}

void* fused_pair_kernel_for(int epi_a, bool f32) {
  switch (epi_a) {
    case EPI_H_GELU: return f32 ? fused_pair_ptr<EPI_H_GELU, EPI_Z_F32>() : fused_pair_ptr<EPI_H_GELU, EPI_Z_BF16>();
    case EPI_H_GELU_TANH:
      return f32 ? fused_pair_ptr<EPI_H_GELU_TANH, EPI_Z_F32>() : fused_pair_ptr<EPI_H_GELU_TANH, EPI_Z_BF16>();
    case EPI_H_IDENTITY:
      return f32 ? fused_pair_ptr<EPI_H_IDENTITY, EPI_Z_F32>() : fused_pair_ptr<EPI_H_IDENTITY, EPI_Z_BF16>();
    case EPI_H_SWIGLU:
      return f32 ? fused_pair_ptr<EPI_H_SWIGLU, EPI_Z_F32>() : fused_pair_ptr<EPI_H_SWIGLU, EPI_Z_BF16>();
    default: return nullptr;
  }
}

void* fused_kernel_for(int epi_a, bool f32) {
  switch (epi_a) {
    case EPI_H_GELU: return f32 ? fused_ptr<EPI_H_GELU, EPI_Z_F32>() : fused_ptr<EPI_H_GELU, EPI_Z_BF16>();
    case EPI_H_GELU_TANH:
      return f32 ? fused_ptr<EPI_H_GELU_TANH, EPI_Z_F32>() : fused_ptr<EPI_H_GELU_TANH, EPI_Z_BF16>();
    case EPI_H_IDENTITY:
      return f32 ? fused_ptr<EPI_H_IDENTITY, EPI_Z_F32>() : fused_ptr<EPI_H_IDENTITY, EPI_Z_BF16>();
    case EPI_H_SWIGLU: return f32 ? fused_ptr<EPI_H_SWIGLU, EPI_Z_F32>() : fused_ptr<EPI_H_SWIGLU, EPI_Z_BF16>();
    default: return nullptr;
  }
}

}  // namespace

size_t fused_sync_bytes(int64_t Mc, int64_t d, int P, int mu) {
  const int64_t tiles_m = (Mc + kBM - 1) / kBM;
  const int64_t tiles_n2 = (d + kBN - 1) / kBN;
  return static_cast<size_t>(4 * (mu * P * tiles_m + mu * tiles_m * tiles_n2 * 4 + 1));
}

cudaError_t prepare_fused_kernels(int* max_ctas_per_sm, int* max_pair_clusters) {
  const int epis[4] = {EPI_H_GELU, EPI_H_GELU_TANH, EPI_H_IDENTITY, EPI_H_SWIGLU};
  int clusters = 1 << 30;
  for (int a = 0; a < 4; ++a) {
    for (int f32 = 0; f32 < 2; ++f32) {
      void* fn = fused_pair_kernel_for(epis[a], f32 != 0);
      cudaError_t st = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
      if (st != cudaSuccess) return st;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 512);
      cfg.blockDim = dim3(kFusedThreads);
      cfg.dynamicSmemBytes = kGemmSmemBytes;
      int n = 0;
      st = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
      if (st != cudaSuccess) return st;
      clusters = n < clusters ? n : clusters;
    }
  }
  for (int f32 = 0; f32 < 2; ++f32) {
    void* fn = fused_gemm2_kernel_for(f32 != 0, true);
    cudaError_t st = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
    if (st != cudaSuccess) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 512);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
    int n = 0;
    st = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (st != cudaSuccess) return st;
    clusters = n < clusters ? n : clusters;
  }
  *max_pair_clusters = clusters;
  int occ = 1 << 30;
  for (int a = 0; a < 4; ++a) {
    for (int f32 = 0; f32 < 2; ++f32) {
      void* fn = fused_kernel_for(epis[a], f32 != 0);
      cudaError_t st = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
      if (st != cudaSuccess) return st;
      int n = 0;
      st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kFusedThreads, kGemmSmemBytes);
      if (st != cudaSuccess) return st;
      occ = n < occ ? n : occ;
    }
  }
  *max_ctas_per_sm = occ;
  return cudaSuccess;
}

domino_status_t launch_fused_fwd(const FusedLaunch& L, int max_ctas, int max_pair_clusters, cudaStream_t stream,
                                 std::string* err) {
  FusedParams f;
  memset(&f, 0, sizeof f);
  const int64_t Fp = L.Fp;
  const bool swiglu = L.epi_a == EPI_H_SWIGLU;
  if (!encode_bf16_sw128(&f.map_x, Operand2D{L.X, L.M, L.d, L.d}, kBM, err)) return DOMINO_ERR_CUDA;
  for (int p = 0; p < L.P; ++p) {
    const uint8_t* W1 = static_cast<const uint8_t*>(L.A_shards[p]);
    const Operand2D w1a{W1, Fp, L.d, L.d};
    const Operand2D w1b = swiglu ? Operand2D{W1 + static_cast<size_t>(Fp) * L.d * 2, Fp, L.d, L.d} : w1a;
    if (!encode_bf16_sw128(&f.map_w1a[p], w1a, kBN / 2, err)) return DOMINO_ERR_CUDA;
    if (!encode_bf16_sw128(&f.map_w1b[p], w1b, kBN / 2, err)) return DOMINO_ERR_CUDA;
    if (!encode_bf16_sw128(&f.map_h[p], Operand2D{L.H[p], L.M, Fp, Fp}, kBM, err)) return DOMINO_ERR_CUDA;
    if (!encode_bf16_sw128(&f.map_w2[p], Operand2D{L.B_shards[p], L.d, Fp, Fp}, kBN / 2, err))
      return DOMINO_ERR_CUDA;
    if (!encode_store_map(&f.map_hout[p], L.H[p], L.M, Fp, Fp, false, 64, err)) return DOMINO_ERR_CUDA;
    if (!encode_store_map(&f.map_zout[p], L.Z[p], L.M, L.d, L.d, L.partial_f32, L.partial_f32 ? 32 : 64, err))
      return DOMINO_ERR_CUDA;
    f.h[p] = L.H[p];
    f.aux[p] = L.aux[p];
    f.z[p] = L.Z[p];
  }
  f.y = L.Y;
  f.hcnt = L.sync;
  f.Mc = static_cast<int32_t>(L.M / L.mu);
  f.tiles_m = (f.Mc + kBM - 1) / kBM;
  f.tiles_n1 = static_cast<int32_t>((Fp + (swiglu ? kBN / 2 : kBN) - 1) / (swiglu ? kBN / 2 : kBN));
  f.tiles_n2 = static_cast<int32_t>((L.d + kBN - 1) / kBN);
  f.zcnt = L.sync + static_cast<int64_t>(L.mu) * L.P * f.tiles_m;
  f.red_next = f.zcnt + static_cast<int64_t>(L.mu) * f.tiles_m * f.tiles_n2 * 4;
  f.timeline = L.timeline;
  f.d = L.d;
  f.Fp = Fp;
  f.mu = L.mu;
  f.P = L.P;
  f.n_tile1 = swiglu ? kBN / 2 : kBN;
  f.b1_off1 = swiglu ? 0 : kBN / 2;
  f.ld_aux = Fp * (swiglu ? 2 : 1);
  f.aux_u_off = Fp;
  f.tiles_a = L.P * f.tiles_m * f.tiles_n1;
  f.tiles_b = L.P * f.tiles_m * f.tiles_n2;
  f.num_gemm_tiles = L.mu * (f.tiles_a + f.tiles_b);
  f.num_red_items = L.reduce ? L.mu * f.tiles_m * f.tiles_n2 : 0;
  f.kb1 = static_cast<int32_t>((L.d + kBK - 1) / kBK);
  f.kb2 = static_cast<int32_t>((Fp + kBK - 1) / kBK);
  f.tiles_m2 = (f.tiles_m + 1) / 2;
  f.tiles_a2 = L.P * f.tiles_m2 * f.tiles_n1;
  f.tiles_b2 = L.P * f.tiles_m2 * f.tiles_n2;
  f.num_pair_tiles = L.mu * (f.tiles_a2 + f.tiles_b2);
  f.status = L.status;
  f.timeout_ns = L.timeout_ns;
  if (f.num_gemm_tiles == 0) return DOMINO_OK;
  if (L.pair && max_pair_clusters > 0) {
    // paired tiles: 2-CTA clusters, launched cooperatively (all CTAs resident)
    void* fn = fused_pair_kernel_for(L.epi_a, L.partial_f32);
    const int clusters = f.num_pair_tiles < max_pair_clusters ? f.num_pair_tiles : max_pair_clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&f};
    cudaError_t st = cudaLaunchKernelExC(&cfg, fn, args);
    if (st == cudaSuccess) return DOMINO_OK;
    if (err) *err = std::string("paired fused launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_UNSUPPORTED;
  }
  void* fn = fused_kernel_for(L.epi_a, L.partial_f32);
  if (!fn) {
    if (err) *err = "launch_fused_fwd: bad activation";
    return DOMINO_ERR_INVALID_ARG;
  }
  const int grid = f.num_gemm_tiles < max_ctas ? f.num_gemm_tiles : max_ctas;
  void* args[] = {&f};
  cudaError_t st = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kFusedThreads), args, kGemmSmemBytes, stream);
  if (st != cudaSuccess) {
    if (err) *err = std::string("fused launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace domino

namespace domino {

domino_status_t launch_fused_gemm2(const FusedGemm2Launch& L, int max_pair_clusters, cudaStream_t stream,
                                   std::string* err) {
  if (max_pair_clusters < 1) {
    if (err) *err = "fused GEMM2 + shard-sum kernel: no paired cooperative launch on this device";
    return DOMINO_ERR_UNSUPPORTED;
  }
  FusedParams f;
  memset(&f, 0, sizeof f);
  for (int p = 0; p < L.P; ++p) {
    // A: [M, K2] K-major, 128-row boxes; B: [K2, d] MN-major in 64 x 64 boxes, or [d, K2] K-major in 128-row boxes
    if (!encode_bf16_sw128(&f.map_h[p], Operand2D{L.A[p], L.M, L.K2, L.K2}, kBM, err)) return DOMINO_ERR_CUDA;
    const bool ok = L.b_mn ? encode_bf16_sw128(&f.map_w2[p], Operand2D{L.B[p], L.K2, L.d, L.d}, kBK, err)
                           : encode_bf16_sw128(&f.map_w2[p], Operand2D{L.B[p], L.d, L.K2, L.K2}, kBN / 2, err);
    if (!ok) return DOMINO_ERR_CUDA;
    if (!encode_store_map(&f.map_zout[p], L.Z[p], L.M, L.d, L.d, L.partial_f32, L.partial_f32 ? 32 : 64, err))
      return DOMINO_ERR_CUDA;
    f.z[p] = L.Z[p];
  }
  f.y = L.Y;
  f.Mc = static_cast<int32_t>(L.M / L.mu);
  f.tiles_m = (f.Mc + kBM - 1) / kBM;
  f.tiles_n2 = static_cast<int32_t>((L.d + kBN - 1) / kBN);
  f.hcnt = L.sync;
  f.zcnt = L.sync + static_cast<int64_t>(L.mu) * L.P * f.tiles_m;
  f.red_next = f.zcnt + static_cast<int64_t>(L.mu) * f.tiles_m * f.tiles_n2 * 4;
  f.timeline = L.timeline;
  f.d = L.d;
  f.mu = L.mu;
  f.P = L.P;
  f.tiles_b = L.P * f.tiles_m * f.tiles_n2;
  f.num_red_items = L.mu * f.tiles_m * f.tiles_n2;
  f.kb2 = static_cast<int32_t>((L.K2 + kBK - 1) / kBK);
  f.tiles_m2 = (f.tiles_m + 1) / 2;
  f.tiles_a2 = 0;  // no GEMM1 phase
  f.tiles_b2 = L.P * f.tiles_m2 * f.tiles_n2;
  f.num_pair_tiles = L.mu * f.tiles_b2;
  f.a2_input = 1;
  f.status = L.status;
  f.timeout_ns = L.timeout_ns;
  if (f.num_pair_tiles == 0) return DOMINO_OK;
  void* fn = fused_gemm2_kernel_for(L.partial_f32, L.b_mn);
  const int clusters = f.num_pair_tiles < max_pair_clusters ? f.num_pair_tiles : max_pair_clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&f};
  const cudaError_t st = cudaLaunchKernelExC(&cfg, fn, args);
  if (st == cudaSuccess) return DOMINO_OK;
  if (err) *err = std::string("fused GEMM2 + shard-sum launch: ") + cudaGetErrorString(st);
  return DOMINO_ERR_UNSUPPORTED;
}

}  // namespace domino
