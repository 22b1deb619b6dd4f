// Host-side interface of the grouped tcgen05 GEMM (gemm.cu) and the shard-sum
// (shard_sum.cu), used by the C-ABI layer (api.cu).
#pragma once

#include <string>

#include "common.h"

namespace domino {

// A bf16 row-major matrix [rows, cols] with leading dimension ld (elements), as
// stored in memory.  For a K-major operand rows = the operand's M (or N) extent
// and cols = K; for an MN-major operand rows = K and cols = the M (or N) extent.
struct Operand2D {
  const void* base = nullptr;
  int64_t rows = 0;
  int64_t cols = 0;
  int64_t ld = 0;
};

// One grouped GEMM launch: for every shard s, out_s = epi(A_s B_s^T), where
// A_s = operand rows [a_row0, a_row0 + rows) of a[s], B_s = operand rows
// [n_base + nb*n_tile, ...) of b0[s] (accumulator columns 0..127) and b1[s]
// (columns 128..255, at operand-row offset b1_off from the b0 box), contraction
// length K.  a_mn / b_mn select MN-major storage of A / B.
struct GemmLaunch {
  int epi = 0;
  bool a_mn = false;
  bool b_mn = false;
  int num_shards = 0;
  Operand2D a[kMaxShards];
  Operand2D b0[kMaxShards];
  Operand2D b1[kMaxShards];
  void* out[kMaxShards] = {};
  void* aux[kMaxShards] = {};
  int64_t ldo = 0, ld_aux = 0, aux_u_off = 0, out_u_off = 0;
  int64_t out_rows = 0, out_cols = 0;  // extent of each out[s]; 0: no TMA stores (direct stores only)
  int32_t a_row0 = 0, out_row0 = 0, rows = 0;
  int32_t n_base = 0, n_end = 0, n_tile = kBN, b1_off = kBN / 2;
  // Paired kernel tile order: rows in groups of group_rows (0: all rows in one
  // group), and within a group every shard and column block, rows innermost.
  int32_t group_rows = 0;
  int64_t K = 0;
  DeviceStatus* status = nullptr;
  uint64_t timeout_ns = 0;
};

cudaError_t prepare_gemm_kernels();
cudaError_t prepare_pair_kernels(int* max_clusters);
// Paired-CTA GEMM (gemm_pair.cu): same launch description, 2-CTA clusters.
domino_status_t launch_gemm_pair(const GemmLaunch& L, int max_clusters, cudaStream_t stream,
                                 std::string* err);
bool encode_bf16_sw128(CUtensorMap* map, const Operand2D& op, int box_rows, std::string* err);
// TMA store map of a row-major output: box 32 rows x box_cols, 128-byte rows
// (fp32 x 32 or bf16 x 64, 128-byte swizzle) or 64-byte rows (bf16 x 32, the
// backward dG outputs, 64-byte swizzle).
bool encode_store_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld, bool f32,
                      int box_cols, std::string* err);
// Store-box width the epilogue of `epi` writes.
inline int store_box_cols(int epi, bool f32) {
  if (f32) return 32;
  return (epi == EPI_DG_GELU || epi == EPI_DG_GELU_TANH || epi == EPI_DG_IDENTITY || epi == EPI_DG_SWIGLU) ? 32 : 64;
}
domino_status_t launch_gemm(const GemmLaunch& L, int max_ctas, cudaStream_t stream, std::string* err);

// The fused forward pass (fused.cu).
struct FusedLaunch {
  const void* X = nullptr;
  const void* A_shards[kMaxShards] = {};
  const void* B_shards[kMaxShards] = {};
  void* H[kMaxShards] = {};
  void* aux[kMaxShards] = {};
  void* Z[kMaxShards] = {};
  void* Y = nullptr;
  uint32_t* sync = nullptr;      // fused_sync_bytes() of zeroed counters
  uint64_t* timeline = nullptr;  // 3 words, zero before the launch ([0] receives ~start)
  int64_t M = 0, d = 0, Fp = 0;
  int mu = 1, P = 1;
  int epi_a = EPI_H_GELU;
  bool partial_f32 = true;
  bool pair = false;    // paired-CTA tiles (2-CTA clusters)
  bool reduce = true;   // false: the partials are the result (no shard-sum pieces; Y unused)
  DeviceStatus* status = nullptr;
  uint64_t timeout_ns = 0;
};
// A row-parallel GEMM and its shard-sum in one cooperative launch of the paired fused kernel (no GEMM1
// phase): Z_p = A_p B_p for every chunk and shard, each 128x256 output tile summed over the shards as soon as
// its P partials exist, Y = bf16(sum_p Z_p).  A_p [M, K2] is K-major; B_p is [d, K2] (K-major, the forward
// layout of a row-parallel weight) or, with b_mn, [K2, d] (MN-major: the backward's partial input gradients
// dG_p A_shards[p]).
struct FusedGemm2Launch {
  const void* A[kMaxShards] = {};
  const void* B[kMaxShards] = {};
  void* Z[kMaxShards] = {};
  void* Y = nullptr;
  uint32_t* sync = nullptr;      // fused_sync_bytes(M / mu, d, P, mu) of zeroed counters
  uint64_t* timeline = nullptr;  // 3 words, zero before the launch
  int64_t M = 0, d = 0, K2 = 0;
  int mu = 1, P = 1;
  bool b_mn = false;
  bool partial_f32 = true;
  DeviceStatus* status = nullptr;
  uint64_t timeout_ns = 0;
};
// Returns DOMINO_ERR_UNSUPPORTED (with nothing launched) if no paired cooperative launch is possible.
domino_status_t launch_fused_gemm2(const FusedGemm2Launch& L, int max_pair_clusters, cudaStream_t stream,
                                   std::string* err);
size_t fused_sync_bytes(int64_t Mc, int64_t d, int P, int mu);
cudaError_t prepare_fused_kernels(int* max_ctas_per_sm, int* max_pair_clusters);
// Returns DOMINO_ERR_UNSUPPORTED (with nothing launched) if a paired launch is refused.
domino_status_t launch_fused_fwd(const FusedLaunch& L, int max_ctas, int max_pair_clusters, cudaStream_t stream,
                                 std::string* err);

// Records a detailed message for domino_last_error() (api.cu).
void set_last_error(const std::string& msg);
// Validates a descriptor the way domino_mlp_fwd does (sets the last error on failure).
domino_status_t validate_desc(const domino_mlp_desc_t* desc);

// Bounded-wait self-test (shard_sum.cu).
domino_status_t launch_selftest_wait(void* workspace, uint64_t timeout_ns, cudaStream_t stream, std::string* err);

// Shard-sum launch (shard_sum.cu).
domino_status_t launch_shard_sum(const ShardSumParams& p, int num_sms, cudaStream_t stream, std::string* err);

}  // namespace domino
