// Schedule selection: the number of row chunks mu and the schedule for one
// problem, from its sizes and three hardware figures (host code only).
//
// Why the rule looks at the L2: every forward schedule multiplies a chunk's
// GEMM1 output H back in GEMM2 right after writing it.  While one chunk's H
// (all shards) fits in the L2, GEMM2 reads it from there; once it does not, H
// makes a round trip through HBM and, under the GPU's power cap, the extra
// traffic costs clock.  Smaller chunks keep H in L2 but give each GEMM fewer
// tiles and the schedule more per-chunk steps, so the rule takes the fewest
// chunks whose H fits, as long as each chunk still fills the GPU with tiles.
// Measured on the GPT-, Llama- and large SwiGLU-style layers (mu in 1..8, both
// overlapping schedules) this picks the fastest mu or one within 0.5% of it;
// the attention form of the rule is below.
#include <cuda_runtime.h>

#include <string>

#include "domino.h"
#include "gemm.h"

namespace domino {
// Validates an attention descriptor the way domino_attn_fwd does (api.cu; sets
// the last error on failure).
domino_status_t validate_attn_desc(const domino_attn_desc_t* desc);
}  // namespace domino

namespace {

constexpr int kPairTileRows = 256;   // rows of a paired GEMM tile
constexpr int kPairTileCols = 256;   // output columns of a paired GEMM1 tile (GeLU / identity)
constexpr int kPairTileColsGlu = 128;  // H columns of a paired SwiGLU GEMM1 tile (gate and up side by side)

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Paired tiles of one chunk's Q|K|V projection (mc rows; per shard 3 Hp dh
// output columns, identity epilogue).
int64_t attn_proj_tiles(const domino_attn_desc_t& a, int64_t mc) {
  const int64_t cols = 3 * static_cast<int64_t>(a.H / a.P) * a.dh;
  return ceil_div(mc, kPairTileRows) * ceil_div(cols, kPairTileCols) * a.P;
}

// Paired GEMM1 tiles of one chunk of mc rows.
int64_t gemm1_tiles(const domino_mlp_desc_t& p, int64_t mc) {
  const int64_t fp = p.F / p.P;
  const int64_t cols = p.act == DOMINO_ACT_SWIGLU ? kPairTileColsGlu : kPairTileCols;
  return ceil_div(mc, kPairTileRows) * ceil_div(fp, cols) * p.P;
}

domino_status_t query_hw(domino_plan_hw_t* hw, const char* who) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  int v = 0;
  if (e == cudaSuccess && hw->num_sms <= 0) {
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    hw->num_sms = v;
  }
  if (e == cudaSuccess && hw->l2_bytes <= 0) {
    e = cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev);
    hw->l2_bytes = v;
  }
  if (e == cudaSuccess && hw->fused_available < 0) {
    e = cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev);
    hw->fused_available = v != 0;
  }
  if (e != cudaSuccess) {
    domino::set_last_error(std::string(who) + ": device query failed: " + cudaGetErrorString(e));
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace

extern "C" {

domino_status_t domino_mlp_plan(const domino_mlp_desc_t* problem, const domino_plan_hw_t* hw,
                                domino_plan_t* out) {
  if (problem == nullptr || out == nullptr) {
    domino::set_last_error("domino_mlp_plan: problem and out must be non-NULL");
    return DOMINO_ERR_INVALID_ARG;
  }
  domino_mlp_desc_t p = *problem;
  p.mu = 1;
  p.schedule = DOMINO_SCHEDULE_STREAMS;
  p.flags = 0;
  p.reserve_sms = 0;
  const domino_status_t st = domino::validate_desc(&p);
  if (st != DOMINO_OK) return st;

  domino_plan_hw_t h = hw ? *hw : domino_plan_hw_t{0, -1, 0};
  if (h.num_sms <= 0 || h.l2_bytes <= 0 || h.fused_available < 0) {
    const domino_status_t q = query_hw(&h, "domino_mlp_plan");
    if (q != DOMINO_OK) return q;
  }
  const int64_t clusters = h.num_sms / 2 > 0 ? h.num_sms / 2 : 1;
  const int64_t budget = h.l2_bytes / 10 * 9;

  int best_fit = 0, largest_filling = 0;
  for (int64_t mu = 1; mu * p.out_slices <= DOMINO_MAX_PIECES && mu <= p.M; mu *= 2) {
    if (p.M % mu) continue;
    const int64_t mc = p.M / mu;
    if (gemm1_tiles(p, mc) < clusters) break;  // smaller chunks fill the GPU even less
    largest_filling = static_cast<int>(mu);
    if (best_fit == 0 && mc * p.F * 2 <= budget) best_fit = static_cast<int>(mu);
  }
  int32_t reason;
  int mu;
  if (best_fit) {
    mu = best_fit;
    reason = DOMINO_PLAN_FITS_L2;
  } else if (largest_filling) {
    mu = largest_filling;
    reason = DOMINO_PLAN_LARGEST_FILLING;
  } else {
    mu = 1;
    reason = DOMINO_PLAN_SMALL;
  }
  const int64_t mc = p.M > 0 ? p.M / mu : 0;
  out->mu = mu;
  out->schedule = h.fused_available ? DOMINO_SCHEDULE_FUSED : DOMINO_SCHEDULE_STREAMS;
  out->reason = reason;
  out->gemm1_tiles_per_chunk = static_cast<int32_t>(gemm1_tiles(p, mc));
  out->chunk_h_bytes = mc * p.F * 2;
  out->l2_budget_bytes = budget;
  return DOMINO_OK;
}

// The same rule for the attention block, with a chunk's Q|K|V (what the
// projection writes and the attention core reads next) in the place of H.
// There the choice is decided by the balance between the per-chunk kernels'
// efficiency (fewer, larger launches fill the GPU better and pay the launch
// ramp and tail less often) and the shard-sum that chunking hides; measured on
// the GPT- and Llama-style blocks (mu in 1, 2, 4), the Q|K|V size is a proxy
// for it that picks the fastest mu.  The schedule is STREAMS: in the attention
// block the output projection writes its partials at close to the memory's
// rate, and a shard-sum folded into the same launch (FUSED) contends with
// those stores instead of hiding behind tensor-core work.
domino_status_t domino_attn_plan(const domino_attn_desc_t* problem, const domino_plan_hw_t* hw,
                                 domino_plan_t* out) {
  if (problem == nullptr || out == nullptr) {
    domino::set_last_error("domino_attn_plan: problem and out must be non-NULL");
    return DOMINO_ERR_INVALID_ARG;
  }
  domino_attn_desc_t a = *problem;
  a.mu = 1;
  a.schedule = DOMINO_SCHEDULE_STREAMS;
  a.flags = 0;
  const domino_status_t st = domino::validate_attn_desc(&a);
  if (st != DOMINO_OK) return st;

  domino_plan_hw_t h = hw ? *hw : domino_plan_hw_t{0, -1, 0};
  if (h.fused_available < 0) h.fused_available = 0;  // not consulted: the plan is STREAMS
  if (h.num_sms <= 0 || h.l2_bytes <= 0) {
    const domino_status_t q = query_hw(&h, "domino_attn_plan");
    if (q != DOMINO_OK) return q;
  }
  const int64_t clusters = h.num_sms / 2 > 0 ? h.num_sms / 2 : 1;
  const int64_t budget = h.l2_bytes / 10 * 9;
  const int64_t qkv_row_bytes = 3 * static_cast<int64_t>(a.H) * a.dh * 2;

  int best_fit = 0, largest_filling = 0;
  for (int64_t mu = 1; mu <= DOMINO_MAX_PIECES && mu <= a.B; mu *= 2) {
    if (a.B % mu) continue;
    const int64_t mc = a.B / mu * a.S;
    if (attn_proj_tiles(a, mc) < clusters) break;  // smaller chunks fill the GPU even less
    largest_filling = static_cast<int>(mu);
    if (best_fit == 0 && mc * qkv_row_bytes <= budget) best_fit = static_cast<int>(mu);
  }
  int32_t reason;
  int mu;
  if (best_fit) {
    mu = best_fit;
    reason = DOMINO_PLAN_FITS_L2;
  } else if (largest_filling) {
    mu = largest_filling;
    reason = DOMINO_PLAN_LARGEST_FILLING;
  } else {
    mu = 1;
    reason = DOMINO_PLAN_SMALL;
  }
  const int64_t mc = a.B > 0 ? a.B / mu * a.S : 0;
  out->mu = mu;
  out->schedule = DOMINO_SCHEDULE_STREAMS;
  out->reason = reason;
  out->gemm1_tiles_per_chunk = static_cast<int32_t>(attn_proj_tiles(a, mc));
  out->chunk_h_bytes = mc * qkv_row_bytes;
  out->l2_budget_bytes = budget;
  return DOMINO_OK;
}

}  // extern "C"
