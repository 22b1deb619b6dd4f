// Paired-CTA variant of the grouped GEMM (tcgen05 cta_group::2).
//
// A 2-CTA cluster computes one 256 x 256 output tile: each CTA TMA-loads its
// own 128 rows of A and its own 128 rows of B per K block into its shared
// memory, and one MMA issued by the even CTA multiplies the whole 256 x 256 x 16
// step, reading A and B halves from both CTAs' shared memory; each CTA's tensor
// memory holds its 128 accumulator rows.  Per SM this halves the B operand that
// has to be staged in and read from shared memory, which is what limits the
// one-CTA 128 x 256 tile.
//
// Synchronisation (all waits bounded, as in the one-CTA kernel):
//   full[s]  only the even CTA's barrier is used: its producer arms it with the
//            bytes of both CTAs (64 KB), and both CTAs' tensor loads count their
//            bytes on it (the odd CTA addresses it in the cluster's shared
//            window).  The even CTA's MMA thread waits on it.
//   empty[s] the MMA completion is multicast to both CTAs' empty[s].
//   tfull[a] the tile's MMA completion is multicast to both CTAs' tfull[a].
//   tempty[a] in the even CTA, count 256: its own 128 epilogue threads plus the
//            odd CTA's 128, which arrive remotely once they have read their rows.
// Tensor memory is allocated collectively by warp 1 of both CTAs.

#include <cuda_bf16.h>

#include <cstdio>
#include <cstring>
#include <string>

#include "epilogue.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace domino {

namespace {

constexpr int kPairStages = 6;
constexpr int kPairAStage = 128 * kBK * 2;  // 16 KB: this CTA's 128 rows of A
constexpr int kPairBStage = 128 * kBK * 2;  // 16 KB: this CTA's 128 rows of B
constexpr int kPairSmemBytes = kPairStages * (kPairAStage + kPairBStage) + kStageOutBytes + 1024 + 256;
static_assert(kPairSmemBytes <= 232448, "shared memory budget");

// Accumulator buffers in tensor memory (256 columns each): double-buffered, so
// the epilogue of one tile overlaps the main loop of the next.
constexpr int kPairAccBufs = 2;
constexpr uint32_t kPairTmemCols = 256 * kPairAccBufs;

// Tile t -> (shard, pair row block (256 rows), column block).  Rows go in groups of
// group_m blocks; within a group: for each shard, for each column block, the
// group's row blocks.  Consecutive tiles (run at the same time by the clusters)
// share a column block of B; a group's rows of A stay in L2 while every shard
// and column block passes over them, so A is read about once and B once per
// group.
__device__ __forceinline__ void pair_tile_coords(const GemmParams& p, int t, int& shard, int& mb2, int& nb) {
  const int G = p.group_m;
  const int per_group = G * p.tiles_n * p.num_shards;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int rows_left = p.tiles_m - g * G;
  const int gm = rows_left < G ? rows_left : G;
  const int per_shard = gm * p.tiles_n;
  shard = r / per_shard;
  const int r2 = r - shard * per_shard;
  nb = r2 / gm;
  mb2 = g * G + (r2 - nb * gm);
}

template <int EPI, bool A_MN, bool B_MN>
__device__ __forceinline__ void gemm_pair_body(const GemmParams& p) {
  constexpr int kCluster = 2;
  constexpr int kTileRows = 128 * kCluster;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + kPairStages * kPairAStage;
  uint8_t* smem_out = smem_b + kPairStages * kPairBStage;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem_out + kStageOutBytes);
  uint64_t* empty_bar = full_bar + kPairStages;
  uint64_t* tfull_bar = empty_bar + kPairStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* final_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank & 1u) == 0;  // the pair's even CTA issues its MMAs
  const uint32_t leader_rank = rank & ~1u;
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << leader_rank);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
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
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPairTmemCols);
    tmem_relinquish_alloc_permit_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = p.num_tiles;
  const uint64_t tmo = p.timeout_ns;
  const int num_clusters = gridDim.x / kCluster;
  const int cluster_id = blockIdx.x / kCluster;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), leader_rank);  // the pair leader's full[0]
    for (int t = cluster_id; t < num_tiles && !*abort_flag; t += num_clusters) {
      int shard, mbx, nb;
      pair_tile_coords(p, t, shard, mbx, nb);
      const int ya = p.a_row0 + mbx * kTileRows + 128 * static_cast<int>(rank);
      const int yb = p.n_base + nb * p.n_tile + (leader ? 0 : p.b1_off);
      const CUtensorMap* mapb = leader ? &p.map_b0[shard] : &p.map_b1[shard];
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, tmo, p.status, kSiteProducerEmpty, t)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem_a + stage * kPairAStage;
        uint8_t* sb = smem_b + stage * kPairBStage;
        if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * (kPairAStage + kPairBStage));
        const uint32_t bar = full0 + stage * 8;
        const int k0 = kb * kBK;
        if constexpr (A_MN) {
          tma_load_2d_pair(sa, &p.map_a[shard], bar, ya, k0);
          tma_load_2d_pair(sa + 8192, &p.map_a[shard], bar, ya + 64, k0);
        } else {
          tma_load_2d_pair(sa, &p.map_a[shard], bar, k0, ya);
        }
        if constexpr (B_MN) {
          tma_load_2d_pair(sb, mapb, bar, yb, k0);
          tma_load_2d_pair(sb + 8192, mapb, bar, yb + 64, k0);
        } else {
          tma_load_2d_pair(sb, mapb, bar, k0, yb);
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    // Drain: the even CTA waits until every load counted on its barriers (its
    // own and the odd CTA's) has landed; loads into the odd CTA complete no
    // later than the cluster barrier below, which the even CTA reaches only
    // after this.
    if (leader) {
      for (int s = 0; s < kPairStages; ++s) {
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          mbar_wait_cluster(&full_bar[s], (issued_parity >> s) & 1u, &no_abort, tmo, p.status, kSiteDrain, s);
        }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------- MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(256, kBN, A_MN, B_MN);
    constexpr uint64_t kAdvA = A_MN ? (2048 >> 4) : (32 >> 4);
    constexpr uint64_t kAdvB = B_MN ? (2048 >> 4) : (32 >> 4);
    uint32_t stage = 0, phase = 0;
    int i = 0;
    for (int t = cluster_id; t < num_tiles && !*abort_flag; t += num_clusters, ++i) {
      const uint32_t acc = kPairAccBufs == 2 ? (i & 1) : 0;
      const uint32_t acc_phase = kPairAccBufs == 2 ? ((i >> 1) & 1) : (i & 1);
      if (!mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1, abort_flag, tmo, p.status, kSiteMmaTmemEmpty, t)) break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + acc * kBN;
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_wait_cluster(&full_bar[stage], phase, abort_flag, tmo, p.status, kSiteMmaFull, t)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sa = smem_u32(smem_a + stage * kPairAStage);
        const uint32_t sb = smem_u32(smem_b + stage * kPairBStage);
        const uint64_t adesc = A_MN ? smem_desc_mn128(sa) : smem_desc_k128(sa);
        const uint64_t bdesc = B_MN ? smem_desc_mn128(sb) : smem_desc_k128(sb);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss_pair(d_tmem, adesc + kAdvA * k, bdesc + kAdvB * k, idesc, (kb | k) != 0 ? 1u : 0u);
        // frees the stage in both CTAs of the pair
        mma_commit_pair_multicast(&empty_bar[stage], pair_mask);
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      mma_commit_pair_multicast(&tfull_bar[acc], pair_mask);
    }
    mma_commit_pair_multicast(final_bar, static_cast<uint16_t>(1u << leader_rank));
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, p.status, kSiteDrain, 99);
  } else if (warp >= 2) {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint8_t* stage = smem_out + (warp - 2) * kStageOutBytesPerWarp;
    int sbuf = 0;
    int i = 0;
    for (int t = cluster_id; t < num_tiles; t += num_clusters, ++i) {
      const uint32_t acc = kPairAccBufs == 2 ? (i & 1) : 0;
      const uint32_t acc_phase = kPairAccBufs == 2 ? ((i >> 1) & 1) : (i & 1);
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, tmo, p.status, kSiteEpilogueTmemFull, t)) break;
      tc_fence_after_sync();
      int shard, mbx, nb;
      pair_tile_coords(p, t, shard, mbx, nb);
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
      const EpiArgs e{p.out[shard], p.aux[shard], p.ldo, p.ld_aux, p.aux_u_off, p.out_u_off,
                      p.rows, p.out_row0, p.n_end, p.use_tma_store ? &p.map_out[shard] : nullptr, stage};
      const int col0 = p.n_base + nb * p.n_tile;
      const int mb = kCluster * mbx + static_cast<int>(rank);  // this CTA's 128-row block
      if constexpr (is_dg(EPI))
        epilogue_tile_dg<EPI>(e, tacc, mb, col0, row_in_tile, sbuf);
      else
        epilogue_tile<EPI>(e, tacc, mb, col0, row_in_tile, sbuf);
      tc_fence_before_sync();
      if (leader)
        mbar_arrive(&tempty_bar[acc]);
      else
        mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), leader_rank));
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the leader's MMAs no longer read this CTA's shared memory
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

template <int EPI, bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  grid_dependency_wait();  // launched as a dependent of the stream's previous kernel
  gemm_pair_body<EPI, A_MN, B_MN>(p);
}

template <int EPI, bool A_MN, bool B_MN>
void* pair_ptr() {
  return reinterpret_cast<void*>(&gemm_pair_kernel<EPI, A_MN, B_MN>);
}

struct PairEntry {
  int epi;
  bool a_mn, b_mn;
  void* fn;  // 2-CTA clusters
};

const PairEntry* pair_table(int* n) {
  static const PairEntry table[] = {
      {EPI_H_GELU, false, false, pair_ptr<EPI_H_GELU, false, false>()},
      {EPI_H_GELU_TANH, false, false, pair_ptr<EPI_H_GELU_TANH, false, false>()},
      {EPI_H_IDENTITY, false, false, pair_ptr<EPI_H_IDENTITY, false, false>()},
      {EPI_H_SWIGLU, false, false, pair_ptr<EPI_H_SWIGLU, false, false>()},
      {EPI_Z_F32, false, false, pair_ptr<EPI_Z_F32, false, false>()},
      {EPI_Z_BF16, false, false, pair_ptr<EPI_Z_BF16, false, false>()},
      {EPI_DG_GELU, false, true, pair_ptr<EPI_DG_GELU, false, true>()},
      {EPI_DG_GELU_TANH, false, true, pair_ptr<EPI_DG_GELU_TANH, false, true>()},
      {EPI_DG_IDENTITY, false, true, pair_ptr<EPI_DG_IDENTITY, false, true>()},
      {EPI_DG_SWIGLU, false, true, pair_ptr<EPI_DG_SWIGLU, false, true>()},
      {EPI_Z_F32, false, true, pair_ptr<EPI_Z_F32, false, true>()},
      {EPI_Z_BF16, false, true, pair_ptr<EPI_Z_BF16, false, true>()},
      {EPI_Z_BF16, true, true, pair_ptr<EPI_Z_BF16, true, true>()},
  };
  *n = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}

}  // namespace

// Sets the shared-memory attribute of every paired kernel and returns how many
// 2-CTA clusters can be resident at once (the persistent grid size): the GPU's
// SMs need not group evenly.
cudaError_t prepare_pair_kernels(int* max_clusters) {
  int n = 0;
  const PairEntry* t = pair_table(&n);
  int best = 1 << 30;
  for (int i = 0; i < n; ++i) {
    cudaError_t st = cudaFuncSetAttribute(t[i].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes);
    if (st != cudaSuccess) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 512);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    int clusters = 0;
    st = cudaOccupancyMaxActiveClusters(&clusters, t[i].fn, &cfg);
    if (st != cudaSuccess) return st;
    best = clusters < best ? clusters : best;
  }
  *max_clusters = best;
  return cudaSuccess;
}

domino_status_t launch_gemm_pair(const GemmLaunch& L, int max_clusters, cudaStream_t stream,
                                 std::string* err) {
  GemmParams p;
  memset(&p, 0, sizeof p);
  if (L.num_shards < 1 || L.num_shards > kMaxShards) {
    if (err) *err = "launch_gemm_pair: bad shard count";
    return DOMINO_ERR_INVALID_ARG;
  }
  const int tile_rows = 256;
  const int a_box = L.a_mn ? kBK : 128;
  const int b_box = L.b_mn ? kBK : 128;
  for (int s = 0; s < L.num_shards; ++s) {
    if (!encode_bf16_sw128(&p.map_a[s], L.a[s], a_box, err)) return DOMINO_ERR_CUDA;
    if (!encode_bf16_sw128(&p.map_b0[s], L.b0[s], b_box, err)) return DOMINO_ERR_CUDA;
    if (!encode_bf16_sw128(&p.map_b1[s], L.b1[s], b_box, err)) return DOMINO_ERR_CUDA;
    p.out[s] = L.out[s];
    p.aux[s] = L.aux[s];
  }
  const bool store_epi = L.epi == EPI_H_GELU || L.epi == EPI_H_GELU_TANH || L.epi == EPI_H_IDENTITY ||
                         L.epi == EPI_H_SWIGLU || L.epi == EPI_Z_F32 || L.epi == EPI_Z_BF16 ||
                         L.epi == EPI_DG_GELU || L.epi == EPI_DG_GELU_TANH || L.epi == EPI_DG_IDENTITY ||
                         L.epi == EPI_DG_SWIGLU;
  if (store_epi && L.out_rows > 0 && L.out_cols > 0) {
    for (int s = 0; s < L.num_shards; ++s)
      if (!encode_store_map(&p.map_out[s], L.out[s], L.out_rows, L.out_cols, L.ldo, L.epi == EPI_Z_F32,
                            store_box_cols(L.epi, L.epi == EPI_Z_F32), err))
        return DOMINO_ERR_CUDA;
    p.use_tma_store = 1;
  }
  p.ldo = L.ldo;
  p.ld_aux = L.ld_aux;
  p.aux_u_off = L.aux_u_off;
  p.out_u_off = L.out_u_off;
  p.a_row0 = L.a_row0;
  p.out_row0 = L.out_row0;
  p.rows = L.rows;
  p.n_base = L.n_base;
  p.n_end = L.n_end;
  p.n_tile = L.n_tile;
  p.b1_off = L.b1_off;
  p.num_kb = static_cast<int32_t>((L.K + kBK - 1) / kBK);
  p.tiles_m = (L.rows + tile_rows - 1) / tile_rows;
  p.tiles_n = (L.n_end - L.n_base + L.n_tile - 1) / L.n_tile;
  p.num_shards = L.num_shards;
  p.num_tiles = p.tiles_m * p.tiles_n * p.num_shards;
  p.group_m = L.group_rows > 0 ? (L.group_rows + tile_rows - 1) / tile_rows : p.tiles_m;
  if (p.group_m > p.tiles_m) p.group_m = p.tiles_m;
  if (p.group_m < 1) p.group_m = 1;
  p.status = L.status;
  p.timeout_ns = L.timeout_ns;
  if (p.num_tiles == 0) return DOMINO_OK;
  void* fn = nullptr;
  int n = 0;
  const PairEntry* t = pair_table(&n);
  for (int i = 0; i < n; ++i)
    if (t[i].epi == L.epi && t[i].a_mn == L.a_mn && t[i].b_mn == L.b_mn) fn = t[i].fn;
  if (!fn) {
    if (err) *err = "launch_gemm_pair: no kernel for this epilogue and operand layout";
    return DOMINO_ERR_INVALID_ARG;
  }
  const int clusters = p.num_tiles < max_clusters ? p.num_tiles : max_clusters;
  void* args[] = {&p};
  cudaError_t st = launch_after_previous(fn, dim3(2 * clusters), dim3(kGemmThreads), kPairSmemBytes, stream, args);
  if (st != cudaSuccess) {
    if (err) *err = std::string("pair gemm launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace domino
