// Grouped persistent tcgen05 GEMM for the two projections of the sliced MLP.
//
// One launch covers every tensor-parallel shard of one row chunk (and one
// output column slice): C_s = A_s B_s^T for s = 0..P-1, with A_s and B_s bf16,
// K-major, read by TMA into a 4-stage shared-memory ring, multiplied by
// tcgen05.mma (M=128, N=256, K=16 per instruction) into an fp32 accumulator in
// tensor memory, and drained by a fused epilogue:
//   GEMM1 (column-parallel, Megatron-LM MLP): H = act(X_k A_p), act = GeLU,
//         tanh-GeLU, identity, or SwiGLU (gate and up accumulated side by side
//         in one N=256 tile, H = silu(gate) * up);
//   GEMM2 (row-parallel): the partial Z_{k,p} = H_{k,p} B_p of shard p, in
//         fp32 or bf16, into that shard's own partial buffer -- the operand of
//         the shard-sum that stands in for the tensor-parallel all-reduce
//         (Domino page, Abstract: each piece's communication is issued as soon
//         as the piece is computed);
//   backward: dH = dY B^T with the activation derivative fused (reads the
//         saved pre-activations), the partial input gradients dG A^T, and the
//         weight gradients X^T dG, dY^T H.  These read operands MN-major
//         (stored [K, rows]); the tensor core takes either major-ness.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0 lane 0: TMA producer     warp 1: TMEM allocator; lane 0 issues MMAs
//   warps 2..5   : epilogue (warp w reads TMEM lanes 32*(w%4) .. +31)
// The accumulator is double-buffered in TMEM (2 x 256 columns), so the
// epilogue of tile i overlaps the main loop of tile i+1.
// Every wait is bounded (see mbar_wait); a wait that runs out records
// DOMINO_ERR_TIMEOUT in the status words and the CTA unwinds cleanly.
#include <cuda_bf16.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "epilogue.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace domino {

__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& shard, int& mb, int& nb) {
  const int per = p.tiles_m * p.tiles_n;
  shard = t / per;
  const int r = t - shard * per;
  nb = r / p.tiles_m;
  mb = r - nb * p.tiles_m;
}

// ------------------------------------------------------------------- kernel

template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_tcgen05_kernel(const __grid_constant__ GemmParams p) {
  grid_dependency_wait();  // launched as a dependent of the stream's previous kernel
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
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.num_shards; ++s) {
      prefetch_tmap(&p.map_a[s]);
      prefetch_tmap(&p.map_b0[s]);
      prefetch_tmap(&p.map_b1[s]);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int num_tiles = p.num_tiles;
  const uint64_t tmo = p.timeout_ns;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;  // per stage: a load was issued / its phase parity
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x) {
      int shard, mb, nb;
      tile_coords(p, t, shard, mb, nb);
      const int ya = p.a_row0 + mb * kBM;
      const int yb0 = p.n_base + nb * p.n_tile;
      const int yb1 = yb0 + p.b1_off;
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, tmo, p.status, kSiteProducerEmpty, t)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem_a + stage * kAStageBytes;
        uint8_t* sb = smem_b + stage * kBStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kAStageBytes + kBStageBytes);
        const int k0 = kb * kBK;
        if constexpr (A_MN) {
          // two boxes of 64 rows x 64 K (MN innermost), 8 KB apart
          tma_load_2d(sa, &p.map_a[shard], &full_bar[stage], ya, k0);
          tma_load_2d(sa + 8192, &p.map_a[shard], &full_bar[stage], ya + 64, k0);
        } else {
          tma_load_2d(sa, &p.map_a[shard], &full_bar[stage], k0, ya);
        }
        if constexpr (B_MN) {
          tma_load_2d(sb, &p.map_b0[shard], &full_bar[stage], yb0, k0);
          tma_load_2d(sb + 8192, &p.map_b0[shard], &full_bar[stage], yb0 + 64, k0);
          tma_load_2d(sb + 16384, &p.map_b1[shard], &full_bar[stage], yb1, k0);
          tma_load_2d(sb + 24576, &p.map_b1[shard], &full_bar[stage], yb1 + 64, k0);
        } else {
          tma_load_2d(sb, &p.map_b0[shard], &full_bar[stage], k0, yb0);
          tma_load_2d(sb + kBStageBytes / 2, &p.map_b1[shard], &full_bar[stage], k0, yb1);
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    // Drain: every issued copy must have landed before shared memory is released.
    for (int s = 0; s < kStages; ++s) {
      if (issued_mask & (1u << s)) {
        volatile int no_abort = 0;
        mbar_wait(&full_bar[s], (issued_parity >> s) & 1u, &no_abort, tmo, p.status, kSiteDrain, s);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, A_MN, B_MN);
    // K advance per MMA (16 bf16), in the descriptor's (address >> 4) units:
    // K-major: 32 bytes along a 128-byte row; MN-major: 16 K-rows of 128 bytes.
    constexpr uint64_t kAdvA = A_MN ? (2048 >> 4) : (32 >> 4);
    constexpr uint64_t kAdvB = B_MN ? (2048 >> 4) : (32 >> 4);
    uint32_t stage = 0, phase = 0;
    int i = 0;
    for (int t = blockIdx.x; t < num_tiles && !*abort_flag; t += gridDim.x, ++i) {
      const uint32_t acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag, tmo, p.status, kSiteMmaTmemEmpty, t)) break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + acc * kBN;
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, abort_flag, tmo, p.status, kSiteMmaFull, t)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sa = smem_u32(smem_a + stage * kAStageBytes);
        const uint32_t sb = smem_u32(smem_b + stage * kBStageBytes);
        const uint64_t adesc = A_MN ? smem_desc_mn128(sa) : smem_desc_k128(sa);
        const uint64_t bdesc = B_MN ? smem_desc_mn128(sb) : smem_desc_k128(sb);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss(d_tmem, adesc + kAdvA * k, bdesc + kAdvB * k, idesc, (kb | k) != 0 ? 1u : 0u);
        mma_commit(&empty_bar[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      mma_commit(&tfull_bar[acc]);
    }
    // All MMAs issued by this thread complete before TMEM is released.
    mma_commit(final_bar);
    volatile int no_abort = 0;
    mbar_wait(final_bar, 0, &no_abort, tmo, p.status, kSiteDrain, 99);
  } else if (warp >= 2) {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    uint8_t* stage = smem_out + (warp - 2) * kStageOutBytesPerWarp;
    int sbuf = 0;
    int i = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++i) {
      const uint32_t acc = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, tmo, p.status, kSiteEpilogueTmemFull, t)) break;
      tc_fence_after_sync();
      int shard, mb, nb;
      tile_coords(p, t, shard, mb, nb);
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
      const EpiArgs e{p.out[shard], p.aux[shard], p.ldo, p.ld_aux, p.aux_u_off, p.out_u_off,
                      p.rows, p.out_row0, p.n_end, p.use_tma_store ? &p.map_out[shard] : nullptr, stage};
      const int col0 = p.n_base + nb * p.n_tile;
      if constexpr (is_dg(EPI))
        epilogue_tile_dg<EPI>(e, tacc, mb, col0, row_in_tile, sbuf);
      else
        epilogue_tile<EPI>(e, tacc, mb, col0, row_in_tile, sbuf);
      tc_fence_before_sync();
      mbar_arrive(&tempty_bar[acc]);
    }
    if (lane == 0) bulk_wait_group<0>();  // stores complete before the CTA releases its shared memory
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

// --------------------------------------------------------------------- host

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn(std::string* err) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (status == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  if (fn == nullptr && err) *err = "cuTensorMapEncodeTiled entry point unavailable";
  return fn;
}

template <int EPI, bool A_MN, bool B_MN>
void* kernel_ptr() {
  return reinterpret_cast<void*>(&gemm_bf16_tcgen05_kernel<EPI, A_MN, B_MN>);
}

// The instantiations the library uses: forward (K-major x K-major), backward
// dH and dX (K-major A, MN-major B), weight gradients (MN-major x MN-major).
struct KernelEntry {
  int epi;
  bool a_mn, b_mn;
  void* fn;
};

const KernelEntry* kernel_table(int* n) {
  static const KernelEntry table[] = {
      {EPI_H_GELU, false, false, kernel_ptr<EPI_H_GELU, false, false>()},
      {EPI_H_GELU_TANH, false, false, kernel_ptr<EPI_H_GELU_TANH, false, false>()},
      {EPI_H_IDENTITY, false, false, kernel_ptr<EPI_H_IDENTITY, false, false>()},
      {EPI_H_SWIGLU, false, false, kernel_ptr<EPI_H_SWIGLU, false, false>()},
      {EPI_Z_F32, false, false, kernel_ptr<EPI_Z_F32, false, false>()},
      {EPI_Z_BF16, false, false, kernel_ptr<EPI_Z_BF16, false, false>()},
      {EPI_DG_GELU, false, true, kernel_ptr<EPI_DG_GELU, false, true>()},
      {EPI_DG_GELU_TANH, false, true, kernel_ptr<EPI_DG_GELU_TANH, false, true>()},
      {EPI_DG_IDENTITY, false, true, kernel_ptr<EPI_DG_IDENTITY, false, true>()},
      {EPI_DG_SWIGLU, false, true, kernel_ptr<EPI_DG_SWIGLU, false, true>()},
      {EPI_Z_F32, false, true, kernel_ptr<EPI_Z_F32, false, true>()},
      {EPI_Z_BF16, false, true, kernel_ptr<EPI_Z_BF16, false, true>()},
      {EPI_Z_BF16, true, true, kernel_ptr<EPI_Z_BF16, true, true>()},
  };
  *n = static_cast<int>(sizeof(table) / sizeof(table[0]));
  return table;
}

void* kernel_for(int epi, bool a_mn, bool b_mn) {
  int n = 0;
  const KernelEntry* t = kernel_table(&n);
  for (int i = 0; i < n; ++i)
    if (t[i].epi == epi && t[i].a_mn == a_mn && t[i].b_mn == b_mn) return t[i].fn;
  return nullptr;
}

}  // namespace

// TMA map of a bf16 row-major matrix with the 128-byte swizzle: box of 64
// innermost elements (one 128-byte row) x box_rows rows; zero fill outside.
bool encode_bf16_sw128(CUtensorMap* map, const Operand2D& op, int box_rows, std::string* err) {
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(op.cols), static_cast<cuuint64_t>(op.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(op.ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(64), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(op.base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) {
      char buf[256];
      snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) rows=%lld cols=%lld ld=%lld", (int)r,
               (long long)op.rows, (long long)op.cols, (long long)op.ld);
      *err = buf;
    }
    return false;
  }
  return true;
}

// TMA store map of a row-major output [rows, cols] (leading dimension ld
// elements): box 32 x 32, 128-byte swizzle for fp32 (128-byte rows), 64-byte
// swizzle for bf16 (64-byte rows), matching stage_and_store's staging layout.
bool encode_store_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld, bool f32,
                      int box_cols, std::string* err) {
  EncodeTiledFn enc = get_encode_fn(err);
  if (!enc) return false;
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32};
  const bool row128 = box_cols * esz == 128;
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   row128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) {
      char buf[256];
      snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (store) failed (%d) rows=%lld cols=%lld ld=%lld", (int)r,
               (long long)rows, (long long)cols, (long long)ld);
      *err = buf;
    }
    return false;
  }
  return true;
}

cudaError_t prepare_gemm_kernels() {
  int n = 0;
  const KernelEntry* t = kernel_table(&n);
  for (int i = 0; i < n; ++i) {
    cudaError_t st = cudaFuncSetAttribute(t[i].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
    if (st != cudaSuccess) return st;
  }
  return cudaSuccess;
}

domino_status_t launch_gemm(const GemmLaunch& L, int max_ctas, cudaStream_t stream, std::string* err) {
  GemmParams p;
  memset(&p, 0, sizeof p);
  if (L.num_shards < 1 || L.num_shards > kMaxShards) {
    if (err) *err = "launch_gemm: bad shard count";
    return DOMINO_ERR_INVALID_ARG;
  }
  const int a_box = L.a_mn ? kBK : kBM;     // MN-major: 64 x 64 boxes; K-major: 64 x 128
  const int b_box = L.b_mn ? kBK : kBN / 2;
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
  p.tiles_m = (L.rows + kBM - 1) / kBM;
  p.tiles_n = (L.n_end - L.n_base + L.n_tile - 1) / L.n_tile;
  p.num_shards = L.num_shards;
  p.num_tiles = p.tiles_m * p.tiles_n * p.num_shards;
  p.status = L.status;
  p.timeout_ns = L.timeout_ns;
  if (p.num_tiles == 0) return DOMINO_OK;
  const int grid = p.num_tiles < max_ctas ? p.num_tiles : max_ctas;
  void* fn = kernel_for(L.epi, L.a_mn, L.b_mn);
  if (!fn) {
    if (err) *err = "launch_gemm: no kernel for this epilogue and operand layout";
    return DOMINO_ERR_INVALID_ARG;
  }
  void* args[] = {&p};
  cudaError_t st = launch_after_previous(fn, dim3(grid), dim3(kGemmThreads), kGemmSmemBytes, stream, args);
  if (st != cudaSuccess) {
    if (err) *err = std::string("gemm launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace domino
