// Structures shared by the host launch code and the device kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "domino.h"

namespace domino {

constexpr int kMaxShards = DOMINO_MAX_SHARDS;

// Device status words, first 16 bytes of the caller's workspace.
struct DeviceStatus {
  uint32_t code;   // first error code recorded (0 = none)
  uint32_t where;  // which wait gave up (site id, see kSite*)
  uint32_t block;  // blockIdx.x of the CTA that recorded it
  uint32_t aux;    // site-defined detail (tile index)
};

// Wait sites reported in DeviceStatus::where.
enum : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaTmemEmpty = 3,
  kSiteEpilogueTmemFull = 4,
  kSiteDrain = 5,
  kSiteFusedH = 6,  // fused kernel: GEMM2 producer waiting for H row block
  kSiteFusedZ = 7,  // fused kernel: reducer waiting for the P partials of a tile
  kSiteSelfTest = 8,  // domino_selftest_wait_timeout
  kSiteAttnP = 9,     // attention: MMA waiting for the softmax's P tile
  kSiteAttnPV = 10,   // attention: softmax waiting for P V
  kSiteAttnX = 11,    // attention: softmax waiting for the partner half of its row
};

// Epilogue of the tcgen05 GEMM: what is done with each fp32 accumulator tile.
enum Epi : int {
  EPI_H_GELU = 0,        // H = gelu(acc) -> bf16            (forward GEMM1, GeLU)
  EPI_H_GELU_TANH = 1,   // H = gelu_tanh(acc) -> bf16
  EPI_H_IDENTITY = 2,    // H = acc -> bf16
  EPI_H_SWIGLU = 3,      // H = silu(acc[:, :128]) * acc[:, 128:] -> bf16 (gate | up in one N=256 tile)
  EPI_Z_F32 = 4,         // C = acc, fp32                    (forward GEMM2 partials, backward dX partials)
  EPI_Z_BF16 = 5,        // C = acc -> bf16                  (bf16 partials, weight gradients)
  EPI_DG_GELU = 6,       // dG = acc * gelu'(g), g read from the saved pre-activations (backward dH GEMM)
  EPI_DG_GELU_TANH = 7,  // dG = acc * gelu_tanh'(g)
  EPI_DG_IDENTITY = 8,   // dG = acc
  EPI_DG_SWIGLU = 9,     // dg = acc * u * silu'(g), du = acc * silu(g), written side by side
  EPI_COUNT = 10
};

// GEMM tile shape: one CTA computes a 128 x 256 fp32 accumulator (tcgen05
// M=128, N=256) over K in blocks of 64 bf16 (one 128-byte swizzle row).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kAStageBytes = kBM * kBK * 2;
constexpr int kBStageBytes = kBN * kBK * 2;
// Epilogue staging for TMA stores: per epilogue warp two 4 KB buffers (a 32 x 32
// chunk of fp32 or bf16 output), swizzled to match the store's tensor map.
constexpr int kStageOutBytesPerWarp = 2 * 4096;
constexpr int kStageOutBytes = 4 * kStageOutBytesPerWarp;
constexpr int kGemmSmemBytes =
    kStages * (kAStageBytes + kBStageBytes) + kStageOutBytes + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kTmemCols = 2 * kBN;  // double-buffered accumulator

// One grouped, persistent GEMM launch: C_s = A_s * B_s^T for every shard s,
// through TMA tensor maps.  A_s is [rows, K] and B_s [N, K]; each is read
// K-major (K contiguous in memory, box 64 K x 128 rows) or MN-major (the
// matrix is stored [K, rows] with rows contiguous, box 64 rows x 64 K).
struct GemmParams {  // CUtensorMap members carry 64-byte alignment
  CUtensorMap map_a[kMaxShards];   // A operand
  CUtensorMap map_b0[kMaxShards];  // B operand rows [n0, n0+128)
  CUtensorMap map_b1[kMaxShards];  // B operand rows for accumulator columns 128..255
  CUtensorMap map_out[kMaxShards]; // output store map (box 32 rows x 32 or 64 columns), when use_tma_store
  void* out[kMaxShards];           // output matrix per shard
  void* aux[kMaxShards];           // optional copy of the pre-activation(s) (bf16), or null
  int64_t ldo;                     // leading dimension of out (elements)
  int64_t ld_aux;                  // leading dimension of aux (elements)
  int64_t aux_u_off;               // SwiGLU: column offset of u inside aux
  int64_t out_u_off;               // SwiGLU backward: column offset of du inside out
  int32_t a_row0;                  // first row of A read by tile row 0
  int32_t out_row0;                // first output row written by tile row 0
  int32_t rows;                    // valid rows (tile rows >= rows are not stored)
  int32_t n_base;                  // output column of tile column 0 (and B row of map_b0)
  int32_t n_end;                   // output columns >= n_end are not stored
  int32_t n_tile;                  // output columns per tile (256, or 128 for SwiGLU)
  int32_t b1_off;                  // B row of the second 128-row box relative to the first
  int32_t num_kb;                  // K blocks of 64
  int32_t tiles_m, tiles_n, num_shards, num_tiles;
  int32_t group_m;                 // paired kernel: row blocks per group of the tile order
  int32_t use_tma_store;           // epilogue writes full chunks through map_out
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// The fused forward kernel (fused.cu): both projections and the shard-sum of
// every chunk in one persistent launch, ordered by counters in the workspace.
struct FusedParams {
  CUtensorMap map_x;                 // X [M, d], box 64 x 128
  CUtensorMap map_w1a[kMaxShards];   // GEMM1 B operand, accumulator columns 0..127 (SwiGLU: gate)
  CUtensorMap map_w1b[kMaxShards];   // GEMM1 B operand, accumulator columns 128..255 (SwiGLU: up)
  CUtensorMap map_h[kMaxShards];     // H_p [M, Fp], box 64 x 128
  CUtensorMap map_w2[kMaxShards];    // B_p^T [d, Fp], box 64 x 128
  CUtensorMap map_hout[kMaxShards];  // H_p store map, box 32 x 32
  CUtensorMap map_zout[kMaxShards];  // Z_p store map, box 32 x 32
  void* h[kMaxShards];
  void* aux[kMaxShards];             // saved pre-activations or null
  void* z[kMaxShards];               // partial outputs [M, d]
  void* y;                           // output [M, d] bf16
  uint32_t* hcnt;                    // [mu][P][tiles_m]: finished GEMM1 tile quarters
  uint32_t* zcnt;                    // [mu][tiles_m][tiles_n2][4]: finished GEMM2 tile quarters
  uint32_t* red_next;                // ticket of the next reduction piece
  uint64_t* timeline;                // [0] ~(first CTA start), [1] last GEMM tile end, [2] last reduction end (ns)
  int64_t d, Fp;
  int64_t ld_aux, aux_u_off;
  int32_t Mc, mu, P;
  int32_t n_tile1, b1_off1;          // GEMM1 output columns per tile and second-box row offset
  int32_t tiles_m, tiles_n1, tiles_n2;
  int32_t tiles_a, tiles_b;          // GEMM1 / GEMM2 tiles per chunk (all shards)
  int32_t num_gemm_tiles, num_red_items;
  int32_t tiles_m2, tiles_a2, tiles_b2;  // paired kernel: 256-row blocks, tiles per chunk and phase
  int32_t num_pair_tiles;
  int32_t kb1, kb2;                  // K blocks of GEMM1 (d) and GEMM2 (Fp, or the backward's nact Fp)
  int32_t a2_input;                  // 1: GEMM2's A operand is an input complete before the launch (no GEMM1
                                     // tiles, no H counters): the backward's partial input gradients
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// The shard-sum: y[r, c] = bf16(sum_p part[p][r, c]).
struct ShardSumParams {
  const void* part[kMaxShards];
  int64_t rows, cols;  // cols multiple of 8
  int64_t ld_part;     // elements
  int64_t ld_y;        // elements
  void* y;
  int32_t P;
  int32_t f32;  // 1: fp32 partials, 0: bf16 partials
};

// Launches `fn` as a programmatic dependent of the stream's previous kernel, so that its launch overlaps that
// kernel's end instead of following it; the kernel calls grid_dependency_wait() before its first
// global-memory access.  Without a previous kernel (or after another stream operation) it is a plain launch.
inline cudaError_t launch_after_previous(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                         void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace domino
