// C-ABI layer: argument validation, workspace layout, and the schedule that
// orders the per-piece GEMMs and shard-sums (declared in include/domino.h).
//
// Schedule (Domino page, "Domino: Eliminating Communication in LLM Training via
// Generic Tensor Slicing and Overlapping", Abstract: independent pieces are
// pipelined so that one piece's communication overlaps another's computation):
// for every row chunk k, one grouped GEMM1 launch computes H_{k,p} for all P
// shards; for every output slice s one grouped GEMM2 launch writes the shard
// partials Z_{k,p,s}; the shard-sum of (k, s) then runs
//   SERIAL : next on the caller's stream (fully exposed), or
//   STREAMS: on the library's reduction stream, released by an event recorded
//            after GEMM2(k, s), so that it runs while GEMM1/GEMM2 of the next
//            piece occupy the tensor cores.  The reduction stream is joined back
//            into the caller's stream at the end of the call.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "attn.h"
#include "gemm.h"

using namespace domino;

namespace {

thread_local std::string g_last_error;

domino_status_t fail(domino_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr size_t kHeaderBytes = 256;
// The FUSED attention block: chunk k's output-projection launch keeps its timeline (3 words) at header byte
// 64 + 24 k, so up to 8 chunks fit in the header.
constexpr int kAttnFusedMaxChunks = 8;
constexpr size_t kAttnTimelineOff = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// --------------------------------------------------------------- per device

struct TimedLaunch {
  int32_t call, kind, chunk, slice, stream;
  cudaEvent_t origin, begin, end;
};

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int fused_max_ctas = 0;     // co-resident CTAs of the fused kernel (cooperative launch limit)
  int pair_max_clusters = 0;  // co-resident 2-CTA clusters of the paired GEMM
  int fused_pair_clusters = 0;  // co-resident 2-CTA clusters of the paired fused kernel (0: not usable)
  cudaStream_t reduce_stream = nullptr;
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_join = nullptr;
  cudaEvent_t ev_piece[DOMINO_MAX_PIECES] = {};
  cudaEvent_t ev_piece_b[DOMINO_MAX_PIECES] = {};  // the second strand of an interleaved call
  std::vector<cudaEvent_t> timing_pool;  // events with timing, reused after a log reset
  size_t timing_next = 0;
};

std::mutex g_mutex;
DeviceState g_devices[64];

// Log of launches made by calls with DOMINO_FLAG_KERNEL_TIMES (guarded by g_mutex).
struct TimingLog {
  int32_t calls = 0;
  std::vector<TimedLaunch> launches;
};
TimingLog g_timing;

domino_status_t device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(DOMINO_ERR_DEVICE, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& ds = g_devices[dev];
  if (!ds.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      char buf[128];
      snprintf(buf, sizeof buf, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev, major, minor);
      return fail(DOMINO_ERR_DEVICE, buf);
    }
    e = cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = prepare_gemm_kernels();
    if (e == cudaSuccess) e = prepare_pair_kernels(&ds.pair_max_clusters);
    if (e == cudaSuccess) e = prepare_attn_kernel();
    int per_sm = 0;
    if (e == cudaSuccess) e = prepare_fused_kernels(&per_sm, &ds.fused_pair_clusters);
    ds.fused_max_ctas = per_sm * ds.num_sms;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ds.reduce_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds.ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds.ev_join, cudaEventDisableTiming);
    for (int i = 0; i < DOMINO_MAX_PIECES && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&ds.ev_piece[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ds.ev_piece_b[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("device setup: ") + cudaGetErrorString(e));
    ds.ready = true;
  }
  *out = &ds;
  return DOMINO_OK;
}

// ---------------------------------------------------------------- validation

struct Shape {
  int64_t M, d, F, Fp, Mc, ds;
  int P, mu, S;
  int act, partial, schedule;
  size_t psize;  // bytes per partial element
  int nact;      // pre-activation matrices per shard (2 for SwiGLU)
};

domino_status_t check_desc(const domino_mlp_desc_t* desc, Shape* s) {
  if (desc == nullptr) return fail(DOMINO_ERR_INVALID_ARG, "desc is NULL");
  const domino_mlp_desc_t& d = *desc;
  if (d.M < 0 || d.d <= 0 || d.F <= 0) return fail(DOMINO_ERR_INVALID_ARG, "M must be >= 0 and d, F > 0");
  if (d.P < 1 || d.P > DOMINO_MAX_SHARDS) return fail(DOMINO_ERR_INVALID_ARG, "P must be in 1..DOMINO_MAX_SHARDS");
  if (d.mu < 1 || d.out_slices < 1) return fail(DOMINO_ERR_INVALID_ARG, "mu and out_slices must be >= 1");
  if (d.act < DOMINO_ACT_GELU || d.act > DOMINO_ACT_IDENTITY) return fail(DOMINO_ERR_INVALID_ARG, "unknown act");
  if (d.partial_dtype != DOMINO_PARTIAL_F32 && d.partial_dtype != DOMINO_PARTIAL_BF16)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown partial_dtype");
  if (d.schedule != DOMINO_SCHEDULE_SERIAL && d.schedule != DOMINO_SCHEDULE_STREAMS &&
      d.schedule != DOMINO_SCHEDULE_FUSED)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown schedule");
  if (d.reserve_sms < 0) return fail(DOMINO_ERR_INVALID_ARG, "reserve_sms must be >= 0");
  if ((d.flags & ~(DOMINO_FLAG_KERNEL_TIMES | DOMINO_FLAG_ONE_CTA)) != 0)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown flag bits");
  if (static_cast<int64_t>(d.mu) * d.out_slices > DOMINO_MAX_PIECES)
    return fail(DOMINO_ERR_UNSUPPORTED, "mu * out_slices exceeds DOMINO_MAX_PIECES");
  if (d.F % d.P) return fail(DOMINO_ERR_UNSUPPORTED, "P must divide F");
  if (d.M % d.mu) return fail(DOMINO_ERR_UNSUPPORTED, "mu must divide M");
  if (d.d % d.out_slices) return fail(DOMINO_ERR_UNSUPPORTED, "out_slices must divide d");
  const int64_t Fp = d.F / d.P;
  if (d.d % 8 || Fp % 8 || (d.d / d.out_slices) % 8)
    return fail(DOMINO_ERR_ALIGNMENT, "d, F/P and d/out_slices must be multiples of 8 (16-byte rows)");
  const int64_t lim = int64_t(1) << 30;
  if (d.M >= lim || d.d >= lim || Fp >= lim) return fail(DOMINO_ERR_UNSUPPORTED, "dimension too large");
  // the shard-sum counts 16-byte vectors of Y (8 elements) with 32-bit indices
  if (d.M * (d.d / 8) >= (int64_t(1) << 32)) return fail(DOMINO_ERR_UNSUPPORTED, "M * d / 8 must be below 2^32");
  s->M = d.M;
  s->d = d.d;
  s->F = d.F;
  s->P = d.P;
  s->mu = d.mu;
  s->S = d.out_slices;
  s->Fp = Fp;
  s->Mc = d.M / d.mu;
  s->ds = d.d / d.out_slices;
  s->act = d.act;
  s->partial = d.partial_dtype;
  s->schedule = d.schedule;
  s->psize = d.partial_dtype == DOMINO_PARTIAL_F32 ? 4 : 2;
  s->nact = d.act == DOMINO_ACT_SWIGLU ? 2 : 1;
  return DOMINO_OK;
}

struct WsLayout {
  size_t h_off, h_shard;    // hidden activations [P][M][Fp] bf16
  size_t z_off, z_shard;    // partials [P][M][d]
  size_t dg_off, dg_shard;  // backward: gradient of the pre-activations [P][M][nact*Fp] bf16
  size_t sync_off, sync_bytes;  // fused schedule: tile counters
  size_t total;
};

constexpr size_t kTimelineOff = 64;  // header offset of the fused kernel's 3 timeline words

// The fused schedule's tile counters follow the timeline words directly, so one
// memset clears both before a fused call.
constexpr size_t kSyncOff = 128;

WsLayout ws_layout(const Shape& s, bool with_bwd) {
  WsLayout L;
  L.sync_bytes = fused_sync_bytes(s.Mc, s.d, s.P, s.mu);
  L.sync_off = kSyncOff;
  size_t off = align_up(kSyncOff + L.sync_bytes, 256);
  L.h_shard = static_cast<size_t>(s.M) * s.Fp * 2;
  L.h_off = off;
  off = align_up(off + L.h_shard * s.P, 256);
  L.z_shard = static_cast<size_t>(s.M) * s.d * s.psize;
  L.z_off = off;
  off = align_up(off + L.z_shard * s.P, 256);
  L.dg_shard = static_cast<size_t>(s.M) * s.Fp * s.nact * 2;
  L.dg_off = off;
  if (with_bwd) off = align_up(off + L.dg_shard * s.P, 256);
  L.total = off;
  return L;
}

size_t saved_shard_bytes(const Shape& s) { return static_cast<size_t>(s.M) * s.Fp * (s.nact + 1) * 2; }

// ------------------------------------------------------------------- timing

struct Timer {
  bool on = false;
  DeviceState* ds = nullptr;
  int32_t call = 0;
  cudaEvent_t origin = nullptr;
  cudaEvent_t take() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (ds->timing_next == ds->timing_pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      ds->timing_pool.push_back(e);
    }
    return ds->timing_pool[ds->timing_next++];
  }
  bool start(cudaStream_t s0) {
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      call = g_timing.calls++;
    }
    origin = take();
    if (!origin) return false;
    cudaEventRecord(origin, s0);
    return true;
  }
};

template <typename F>
domino_status_t timed(Timer& T, cudaStream_t st, int32_t stream_id, int32_t kind, int32_t chunk, int32_t slice,
                      F&& launch) {
  if (!T.on) return launch();
  bool room;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    room = g_timing.launches.size() < DOMINO_MAX_TIMED_LAUNCHES;
  }
  if (!room) return launch();
  cudaEvent_t b = T.take(), e = T.take();
  if (!b || !e) return fail(DOMINO_ERR_CUDA, "cudaEventCreate failed");
  cudaEventRecord(b, st);
  domino_status_t r = launch();
  cudaEventRecord(e, st);
  std::lock_guard<std::mutex> lock(g_mutex);
  g_timing.launches.push_back({T.call, kind, chunk, slice, stream_id, T.origin, b, e});
  return r;
}

// The persistent grids of one call: the device's co-residency limits, less the SMs the caller reserves
// (desc->reserve_sms) for work of its own that runs beside the library (a collective, another stream).
struct Grid {
  int num_sms = 0;              // SMs the one-CTA kernels and the shard-sum spread over
  int pair_clusters = 0;        // 2-CTA clusters of the paired GEMM
  int fused_ctas = 0;           // CTAs of the one-CTA fused kernel
  int fused_pair_clusters = 0;  // 2-CTA clusters of the paired fused kernels (0: not usable)
};

Grid grid_for(const DeviceState* ds, int reserve_sms) {
  Grid g;
  const int avail = ds->num_sms - reserve_sms;
  const int per_sm = ds->num_sms > 0 ? ds->fused_max_ctas / ds->num_sms : 0;
  g.num_sms = avail;
  g.pair_clusters = ds->pair_max_clusters < avail / 2 ? ds->pair_max_clusters : avail / 2;
  g.fused_ctas = per_sm * avail;
  g.fused_pair_clusters = ds->fused_pair_clusters < avail / 2 ? ds->fused_pair_clusters : avail / 2;
  return g;
}

domino_status_t check_reserve(const DeviceState* ds, int reserve_sms) {
  if (reserve_sms > ds->num_sms - 2)
    return fail(DOMINO_ERR_INVALID_ARG, "reserve_sms must leave at least 2 SMs to the library");
  return DOMINO_OK;
}

// One grouped GEMM launch, as one-CTA tiles or as paired-CTA clusters.
domino_status_t run_gemm(const GemmLaunch& L, const Grid& g, bool pair, cudaStream_t st, std::string* err) {
  return pair ? launch_gemm_pair(L, g.pair_clusters, st, err) : launch_gemm(L, g.num_sms, st, err);
}

// ------------------------------------------------------- launch sequences

// The forward of one batch as separate launches (SERIAL / STREAMS schedules):
// per chunk k, GEMM1 of all shards, then per slice s GEMM2 and -- on the
// reduction stream, after an event recorded behind that GEMM2 -- the shard-sum
// of piece (k, s).  chunk(k) issues one chunk, so another sequence's launches
// can be placed between chunks.
struct FwdSeq {
  Shape s{};
  DeviceState* ds = nullptr;
  Grid grid{};
  Timer* T = nullptr;
  cudaStream_t s0 = nullptr, sr = nullptr;
  bool pair = true;
  DeviceStatus* status = nullptr;
  uint64_t tmo = 0;
  const void* X = nullptr;
  const void* const* A_shards = nullptr;
  const void* const* B_shards = nullptr;
  void* Y = nullptr;
  void* H[kMaxShards] = {};
  void* pre[kMaxShards] = {};
  void* Z[kMaxShards] = {};
  cudaEvent_t* ev_piece = nullptr;  // mu * S events, one per piece
  bool reduce = true;               // false: the partials are the result (no shard-sum)
  void* const* user_events = nullptr;  // partials only: the caller's piece events (nullable)

  // H and the pre-activations go to `saved` when it is given, else H to the workspace.
  void bind(uint8_t* ws, const WsLayout& W, void* saved) {
    for (int p = 0; p < s.P; ++p) {
      if (saved) {
        uint8_t* blk = static_cast<uint8_t*>(saved) + saved_shard_bytes(s) * p;
        pre[p] = blk;
        H[p] = blk + static_cast<size_t>(s.M) * s.Fp * s.nact * 2;
      } else {
        pre[p] = nullptr;
        H[p] = ws + W.h_off + W.h_shard * p;
      }
      Z[p] = ws + W.z_off + W.z_shard * p;
    }
  }

  domino_status_t chunk(int k, std::string* err) const {
    static const int kEpiOfAct[4] = {EPI_H_GELU, EPI_H_GELU_TANH, EPI_H_SWIGLU, EPI_H_IDENTITY};
    const bool swiglu = s.act == DOMINO_ACT_SWIGLU;
    const int32_t row0 = static_cast<int32_t>(k * s.Mc);
    domino_status_t st;
    // ---- GEMM1: H_{k,p} = act(X_k A_p), all shards in one launch
    {
      GemmLaunch L;
      L.epi = kEpiOfAct[s.act];
      L.num_shards = s.P;
      for (int p = 0; p < s.P; ++p) {
        L.a[p] = {X, s.M, s.d, s.d};
        const uint8_t* Ap = static_cast<const uint8_t*>(A_shards[p]);
        L.b0[p] = {Ap, s.Fp, s.d, s.d};
        L.b1[p] = swiglu ? Operand2D{Ap + static_cast<size_t>(s.Fp) * s.d * 2, s.Fp, s.d, s.d} : L.b0[p];
        L.out[p] = H[p];
        L.aux[p] = pre[p];
      }
      L.n_tile = swiglu ? kBN / 2 : kBN;
      L.b1_off = swiglu ? 0 : kBN / 2;
      L.ldo = s.Fp;
      L.out_rows = s.M;
      L.out_cols = s.Fp;
      L.ld_aux = s.Fp * s.nact;
      L.aux_u_off = s.Fp;
      L.a_row0 = row0;
      L.out_row0 = row0;
      L.rows = static_cast<int32_t>(s.Mc);
      L.n_base = 0;
      L.n_end = static_cast<int32_t>(s.Fp);
      L.K = s.d;
      L.status = status;
      L.timeout_ns = tmo;
      st = timed(*T, s0, 0, DOMINO_KERNEL_GEMM1, k, 0, [&] { return run_gemm(L, grid, pair, s0, err); });
      if (st != DOMINO_OK) return st;
    }
    for (int sl = 0; sl < s.S; ++sl) {
      const int32_t col0 = static_cast<int32_t>(sl * s.ds);
      // ---- GEMM2: Z_{k,p,s} = H_{k,p} B_p[:, slice s]
      GemmLaunch L;
      L.epi = s.partial == DOMINO_PARTIAL_F32 ? EPI_Z_F32 : EPI_Z_BF16;
      L.num_shards = s.P;
      for (int p = 0; p < s.P; ++p) {
        L.a[p] = {H[p], s.M, s.Fp, s.Fp};
        L.b0[p] = {B_shards[p], s.d, s.Fp, s.Fp};
        L.b1[p] = L.b0[p];
        L.out[p] = Z[p];
      }
      L.n_tile = kBN;
      L.b1_off = kBN / 2;
      L.ldo = s.d;
      L.out_rows = s.M;
      L.out_cols = s.d;
      L.a_row0 = row0;
      L.out_row0 = row0;
      L.rows = static_cast<int32_t>(s.Mc);
      L.n_base = col0;
      L.n_end = static_cast<int32_t>(col0 + s.ds);
      L.K = s.Fp;
      L.status = status;
      L.timeout_ns = tmo;
      st = timed(*T, s0, 0, DOMINO_KERNEL_GEMM2, k, sl, [&] { return run_gemm(L, grid, pair, s0, err); });
      if (st != DOMINO_OK) return st;
      if (!reduce) {
        if (user_events) {
          cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(user_events[k * s.S + sl]), s0);
          if (e != cudaSuccess) {
            if (err) *err = std::string("piece event record: ") + cudaGetErrorString(e);
            return DOMINO_ERR_CUDA;
          }
        }
        continue;
      }
      st = shard_sum_piece(k, sl, err);
      if (st != DOMINO_OK) return st;
    }
    return DOMINO_OK;
  }

  // Y_k[:, s] = sum over p of Z_{k,p}[:, s], after the GEMM2 just issued on s0.
  domino_status_t shard_sum_piece(int k, int sl, std::string* err) const {
    const int32_t row0 = static_cast<int32_t>(k * s.Mc);
    const int32_t col0 = static_cast<int32_t>(sl * s.ds);
    if (sr != s0) {
      cudaEvent_t ev = ev_piece[k * s.S + sl];
      cudaEventRecord(ev, s0);
      cudaStreamWaitEvent(sr, ev, 0);
    }
    ShardSumParams q;
    memset(&q, 0, sizeof q);
    const size_t zoff = (static_cast<size_t>(row0) * s.d + col0) * s.psize;
    for (int p = 0; p < s.P; ++p) q.part[p] = static_cast<uint8_t*>(Z[p]) + zoff;
    q.rows = s.Mc;
    q.cols = s.ds;
    q.ld_part = s.d;
    q.ld_y = s.d;
    q.y = static_cast<uint8_t*>(Y) + (static_cast<size_t>(row0) * s.d + col0) * 2;
    q.P = s.P;
    q.f32 = s.partial == DOMINO_PARTIAL_F32;
    return timed(*T, sr, sr != s0, DOMINO_KERNEL_SHARD_SUM, k, sl,
                 [&] { return launch_shard_sum(q, grid.num_sms, sr, err); });
  }
};

// The backward of one batch: dh() over all M, then per chunk dx_chunk(k) (the
// partial input gradients of every slice and their shard-sums on the reduction
// stream), then dw() over all M.
struct BwdSeq {
  Shape s{};
  DeviceState* ds = nullptr;
  Grid grid{};
  Timer* T = nullptr;
  cudaStream_t s0 = nullptr, sr = nullptr;
  bool pair = true;
  DeviceStatus* status = nullptr;
  uint64_t tmo = 0;
  const void* X = nullptr;
  const void* const* A_shards = nullptr;
  const void* const* B_shards = nullptr;
  const void* dY = nullptr;
  void* dX = nullptr;
  void* const* dA_shards = nullptr;
  void* const* dB_shards = nullptr;
  const void* pre[kMaxShards] = {};
  const void* H[kMaxShards] = {};
  void* dG[kMaxShards] = {};
  void* Z[kMaxShards] = {};
  cudaEvent_t* ev_piece = nullptr;  // mu * S events, one per piece

  int64_t nF() const { return s.nact * s.Fp; }  // columns of the pre-activation block / rows of A_shards[p]

  void bind(uint8_t* ws, const WsLayout& W, const void* saved) {
    for (int p = 0; p < s.P; ++p) {
      const uint8_t* blk = static_cast<const uint8_t*>(saved) + saved_shard_bytes(s) * p;
      pre[p] = blk;
      H[p] = blk + static_cast<size_t>(s.M) * nF() * 2;
      dG[p] = ws + W.dg_off + W.dg_shard * p;
      Z[p] = ws + W.z_off + W.z_shard * p;
    }
  }

  // dH_p = dY B_p^T with the activation derivative fused -> dG_p, over all M
  // tokens in one launch: it exchanges nothing, so it needs no chunking, and one
  // launch over M fills the GPU's clusters better than mu launches over M/mu.
  domino_status_t dh(std::string* err) const {
    static const int kDgEpi[4] = {EPI_DG_GELU, EPI_DG_GELU_TANH, EPI_DG_SWIGLU, EPI_DG_IDENTITY};
    GemmLaunch L;
    L.epi = kDgEpi[s.act];
    L.b_mn = true;
    L.num_shards = s.P;
    for (int p = 0; p < s.P; ++p) {
      L.a[p] = {dY, s.M, s.d, s.d};
      L.b0[p] = {B_shards[p], s.d, s.Fp, s.Fp};  // stored [d][Fp]: K = d rows, N = Fp contiguous
      L.b1[p] = L.b0[p];
      L.out[p] = dG[p];
      L.aux[p] = const_cast<void*>(pre[p]);
    }
    L.ldo = nF();
    L.out_rows = s.M;
    L.out_cols = nF();
    L.ld_aux = nF();
    L.aux_u_off = s.Fp;
    L.out_u_off = s.Fp;
    L.a_row0 = 0;
    L.out_row0 = 0;
    L.rows = static_cast<int32_t>(s.M);
    L.group_rows = static_cast<int32_t>(s.Mc);  // dY rows of a group stay in L2 across all column tiles
    L.n_base = 0;
    L.n_end = static_cast<int32_t>(s.Fp);
    L.K = s.d;
    L.status = status;
    L.timeout_ns = tmo;
    return timed(*T, s0, 0, DOMINO_KERNEL_BWD_DH, 0, 0, [&] { return run_gemm(L, grid, pair, s0, err); });
  }

  domino_status_t dx_chunk(int k, std::string* err) const {
    const int32_t row0 = static_cast<int32_t>(k * s.Mc);
    for (int sl = 0; sl < s.S; ++sl) {
      const int32_t col0 = static_cast<int32_t>(sl * s.ds);
      // ---- partial input gradient of shard p: dG_{k,p} A_p^T -> Z_p
      GemmLaunch L;
      L.epi = s.partial == DOMINO_PARTIAL_F32 ? EPI_Z_F32 : EPI_Z_BF16;
      L.b_mn = true;
      L.num_shards = s.P;
      for (int p = 0; p < s.P; ++p) {
        L.a[p] = {dG[p], s.M, nF(), nF()};
        L.b0[p] = {A_shards[p], nF(), s.d, s.d};  // stored [nF][d]: K = nF rows, N = d contiguous
        L.b1[p] = L.b0[p];
        L.out[p] = Z[p];
      }
      L.ldo = s.d;
      L.out_rows = s.M;
      L.out_cols = s.d;
      L.a_row0 = row0;
      L.out_row0 = row0;
      L.rows = static_cast<int32_t>(s.Mc);
      L.n_base = col0;
      L.n_end = static_cast<int32_t>(col0 + s.ds);
      L.K = nF();
      L.status = status;
      L.timeout_ns = tmo;
      domino_status_t st =
          timed(*T, s0, 0, DOMINO_KERNEL_BWD_DX, k, sl, [&] { return run_gemm(L, grid, pair, s0, err); });
      if (st != DOMINO_OK) return st;
      // ---- dX_k[:, s] = sum_p of the partials (the all-reduce of the input gradient)
      if (sr != s0) {
        cudaEvent_t ev = ev_piece[k * s.S + sl];
        cudaEventRecord(ev, s0);
        cudaStreamWaitEvent(sr, ev, 0);
      }
      ShardSumParams q;
      memset(&q, 0, sizeof q);
      const size_t zoff = (static_cast<size_t>(row0) * s.d + col0) * s.psize;
      for (int p = 0; p < s.P; ++p) q.part[p] = static_cast<uint8_t*>(Z[p]) + zoff;
      q.rows = s.Mc;
      q.cols = s.ds;
      q.ld_part = s.d;
      q.ld_y = s.d;
      q.y = static_cast<uint8_t*>(dX) + (static_cast<size_t>(row0) * s.d + col0) * 2;
      q.P = s.P;
      q.f32 = s.partial == DOMINO_PARTIAL_F32;
      st = timed(*T, sr, sr != s0, DOMINO_KERNEL_SHARD_SUM, k, sl,
                 [&] { return launch_shard_sum(q, grid.num_sms, sr, err); });
      if (st != DOMINO_OK) return st;
    }
    return DOMINO_OK;
  }

  // FUSED schedule: the partial input gradients of every chunk and their shard-sum in one cooperative launch
  // (tile-granular overlap, as in the fused forward).  Returns DOMINO_ERR_UNSUPPORTED with nothing launched
  // when the device cannot run it; the caller then issues dx_chunk() per chunk.
  domino_status_t dx_fused(uint8_t* ws, const WsLayout& W, std::string* err) const {
    FusedGemm2Launch F;
    for (int p = 0; p < s.P; ++p) {
      F.A[p] = dG[p];
      F.B[p] = A_shards[p];
      F.Z[p] = Z[p];
    }
    F.Y = dX;
    F.b_mn = true;
    F.sync = reinterpret_cast<uint32_t*>(ws + W.sync_off);
    F.timeline = reinterpret_cast<uint64_t*>(ws + kTimelineOff);
    F.M = s.M;
    F.d = s.d;
    F.K2 = nF();
    F.mu = s.mu;
    F.P = s.P;
    F.partial_f32 = s.partial == DOMINO_PARTIAL_F32;
    F.status = status;
    F.timeout_ns = tmo;
    if (grid.fused_pair_clusters < 1) return DOMINO_ERR_UNSUPPORTED;
    cudaError_t e = cudaMemsetAsync(ws + kTimelineOff, 0, kSyncOff - kTimelineOff + W.sync_bytes, s0);
    if (e != cudaSuccess) {
      if (err) *err = std::string("counter reset: ") + cudaGetErrorString(e);
      return DOMINO_ERR_CUDA;
    }
    return timed(*T, s0, 0, DOMINO_KERNEL_BWD_DX_FUSED, 0, 0,
                 [&] { return launch_fused_gemm2(F, grid.fused_pair_clusters, s0, err); });
  }

  // Weight gradients over all M (they run while the last shard-sum drains).
  domino_status_t dw(std::string* err) const {
    {
      GemmLaunch L;  // dA_p = dG_p^T X : [nF, d], contraction over tokens
      L.epi = EPI_Z_BF16;
      L.a_mn = true;
      L.b_mn = true;
      L.num_shards = s.P;
      for (int p = 0; p < s.P; ++p) {
        L.a[p] = {dG[p], s.M, nF(), nF()};
        L.b0[p] = {X, s.M, s.d, s.d};
        L.b1[p] = L.b0[p];
        L.out[p] = dA_shards[p];
      }
      L.ldo = s.d;
      L.out_rows = nF();
      L.out_cols = s.d;
      L.rows = static_cast<int32_t>(nF());
      L.n_base = 0;
      L.n_end = static_cast<int32_t>(s.d);
      L.K = s.M;
      L.status = status;
      L.timeout_ns = tmo;
      domino_status_t st =
          timed(*T, s0, 0, DOMINO_KERNEL_BWD_DW, 0, 0, [&] { return run_gemm(L, grid, pair, s0, err); });
      if (st != DOMINO_OK) return st;
    }
    GemmLaunch L;  // dB_p = dY^T H_p : [d, Fp]
    L.epi = EPI_Z_BF16;
    L.a_mn = true;
    L.b_mn = true;
    L.num_shards = s.P;
    for (int p = 0; p < s.P; ++p) {
      L.a[p] = {dY, s.M, s.d, s.d};
      L.b0[p] = {H[p], s.M, s.Fp, s.Fp};
      L.b1[p] = L.b0[p];
      L.out[p] = dB_shards[p];
    }
    L.ldo = s.Fp;
    L.out_rows = s.d;
    L.out_cols = s.Fp;
    L.rows = static_cast<int32_t>(s.d);
    L.n_base = 0;
    L.n_end = static_cast<int32_t>(s.Fp);
    L.K = s.M;
    L.status = status;
    L.timeout_ns = tmo;
    return timed(*T, s0, 0, DOMINO_KERNEL_BWD_DW, 0, 1, [&] { return run_gemm(L, grid, pair, s0, err); });
  }
};

// Makes `sr` wait for everything issued on `s0` so far (before a sequence's first
// reduction), and `s0` wait for everything on `sr` (before the call returns).
void fork_streams(const DeviceState* ds, cudaStream_t s0, cudaStream_t sr) {
  if (sr == s0) return;
  cudaEventRecord(ds->ev_fork, s0);
  cudaStreamWaitEvent(sr, ds->ev_fork, 0);
}
void join_streams(const DeviceState* ds, cudaStream_t s0, cudaStream_t sr) {
  if (sr == s0) return;
  cudaEventRecord(ds->ev_join, sr);
  cudaStreamWaitEvent(s0, ds->ev_join, 0);
}

// ------------------------------------------------------- attention block

struct AttnShape {
  int64_t B, S, d, M, Mc;
  int H, dh, P, Hp, mu, partial, schedule;
  size_t psize;
  int64_t qkv_cols() const { return 3 * static_cast<int64_t>(Hp) * dh; }
  int64_t o_cols() const { return static_cast<int64_t>(Hp) * dh; }
};

domino_status_t check_attn_desc(const domino_attn_desc_t* desc, AttnShape* s) {
  if (desc == nullptr) return fail(DOMINO_ERR_INVALID_ARG, "desc is NULL");
  const domino_attn_desc_t& a = *desc;
  if (a.B < 0 || a.S <= 0 || a.d <= 0 || a.H < 1 || a.dh < 1)
    return fail(DOMINO_ERR_INVALID_ARG, "B must be >= 0 and S, d, H, dh > 0");
  if (a.P < 1 || a.P > DOMINO_MAX_SHARDS) return fail(DOMINO_ERR_INVALID_ARG, "P must be in 1..DOMINO_MAX_SHARDS");
  if (a.mu < 1) return fail(DOMINO_ERR_INVALID_ARG, "mu must be >= 1");
  if (a.partial_dtype != DOMINO_PARTIAL_F32 && a.partial_dtype != DOMINO_PARTIAL_BF16)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown partial_dtype");
  if (a.schedule != DOMINO_SCHEDULE_SERIAL && a.schedule != DOMINO_SCHEDULE_STREAMS &&
      a.schedule != DOMINO_SCHEDULE_FUSED)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown schedule");
  if (a.reserved != 0) return fail(DOMINO_ERR_INVALID_ARG, "reserved must be 0");
  if ((a.flags & ~(DOMINO_FLAG_KERNEL_TIMES | DOMINO_FLAG_ONE_CTA)) != 0)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown flag bits");
  if (a.schedule == DOMINO_SCHEDULE_FUSED && a.mu > kAttnFusedMaxChunks)
    return fail(DOMINO_ERR_UNSUPPORTED, "the FUSED attention block takes at most 8 chunks (one timeline slot each)");
  if (a.dh != 128) return fail(DOMINO_ERR_UNSUPPORTED, "head width dh must be 128");
  if (a.S % 128) return fail(DOMINO_ERR_UNSUPPORTED, "S must be a multiple of 128");
  if (a.H % a.P) return fail(DOMINO_ERR_UNSUPPORTED, "P must divide H");
  if (a.B % a.mu) return fail(DOMINO_ERR_UNSUPPORTED, "mu must divide B");
  if (a.mu > DOMINO_MAX_PIECES) return fail(DOMINO_ERR_UNSUPPORTED, "mu exceeds DOMINO_MAX_PIECES");
  if (a.d % 8) return fail(DOMINO_ERR_ALIGNMENT, "d must be a multiple of 8 (16-byte rows)");
  const int64_t lim = int64_t(1) << 30;
  if (a.B * a.S >= lim || a.d >= lim || static_cast<int64_t>(a.H) * a.dh * 3 >= lim)
    return fail(DOMINO_ERR_UNSUPPORTED, "dimension too large");
  s->B = a.B;
  s->S = a.S;
  s->d = a.d;
  s->M = a.B * a.S;
  s->Mc = a.B / a.mu * a.S;
  s->H = a.H;
  s->dh = a.dh;
  s->P = a.P;
  s->Hp = a.H / a.P;
  s->mu = a.mu;
  s->partial = a.partial_dtype;
  s->schedule = a.schedule;
  s->psize = a.partial_dtype == DOMINO_PARTIAL_F32 ? 4 : 2;
  return DOMINO_OK;
}

struct AttnWs {
  size_t sync_off, sync_bytes;  // FUSED: the counters of one chunk's output-projection + shard-sum launch
  size_t qkv_off, qkv_shard, o_off, o_shard, z_off, z_shard, total;
};

AttnWs attn_ws_layout(const AttnShape& s) {
  AttnWs W;
  size_t off = kHeaderBytes;
  W.sync_off = off;
  W.sync_bytes = fused_sync_bytes(s.Mc, s.d, s.P, 1);
  off = align_up(off + W.sync_bytes, 256);
  W.qkv_shard = static_cast<size_t>(s.M) * s.qkv_cols() * 2;
  W.qkv_off = off;
  off = align_up(off + W.qkv_shard * s.P, 256);
  W.o_shard = static_cast<size_t>(s.M) * s.o_cols() * 2;
  W.o_off = off;
  off = align_up(off + W.o_shard * s.P, 256);
  W.z_shard = static_cast<size_t>(s.M) * s.d * s.psize;
  W.z_off = off;
  off = align_up(off + W.z_shard * s.P, 256);
  W.total = off;
  return W;
}

// One chunk of the attention block: projection, attention core, output
// projection into the partials (caller's stream), shard-sum (reduction stream).
struct AttnSeq {
  AttnShape s{};
  DeviceState* ds = nullptr;
  Grid grid{};
  Timer* T = nullptr;
  cudaStream_t s0 = nullptr, sr = nullptr;
  bool pair = true;
  DeviceStatus* status = nullptr;
  uint64_t tmo = 0;
  const void* X = nullptr;
  const void* const* Wqkv = nullptr;
  const void* const* Wo = nullptr;
  void* Y = nullptr;
  void* qkv[kMaxShards] = {};
  void* o[kMaxShards] = {};
  void* Z[kMaxShards] = {};
  uint8_t* ws = nullptr;
  AttnWs W{};

  // FUSED, last chunk: its output projection and its shard-sum in one cooperative launch (each 128x256 tile
  // of Y_k summed as soon as its P partials exist).  DOMINO_ERR_UNSUPPORTED with nothing launched if the device
  // cannot run it.
  domino_status_t out_proj_fused(int k, std::string* err) const {
    if (grid.fused_pair_clusters < 1) return DOMINO_ERR_UNSUPPORTED;
    const size_t row0 = static_cast<size_t>(k) * s.Mc;
    FusedGemm2Launch F;
    for (int p = 0; p < s.P; ++p) {
      F.A[p] = static_cast<const uint8_t*>(o[p]) + row0 * s.o_cols() * 2;
      F.B[p] = Wo[p];
      F.Z[p] = static_cast<uint8_t*>(Z[p]) + row0 * s.d * s.psize;
    }
    F.Y = static_cast<uint8_t*>(Y) + row0 * s.d * 2;
    F.sync = reinterpret_cast<uint32_t*>(ws + W.sync_off);
    F.timeline = reinterpret_cast<uint64_t*>(ws + kAttnTimelineOff + 24 * static_cast<size_t>(k));
    F.M = s.Mc;
    F.d = s.d;
    F.K2 = s.o_cols();
    F.mu = 1;
    F.P = s.P;
    F.b_mn = false;
    F.partial_f32 = s.partial == DOMINO_PARTIAL_F32;
    F.status = status;
    F.timeout_ns = tmo;
    cudaError_t e = cudaMemsetAsync(F.timeline, 0, 24, s0);
    if (e == cudaSuccess) e = cudaMemsetAsync(F.sync, 0, W.sync_bytes, s0);
    if (e != cudaSuccess) {
      if (err) *err = std::string("counter reset: ") + cudaGetErrorString(e);
      return DOMINO_ERR_CUDA;
    }
    return timed(*T, s0, 0, DOMINO_KERNEL_ATTN_OUT_FUSED, k, 0,
                 [&] { return launch_fused_gemm2(F, grid.fused_pair_clusters, s0, err); });
  }

  domino_status_t chunk(int k, std::string* err) const {
    const int32_t row0 = static_cast<int32_t>(k * s.Mc);
    domino_status_t st;
    {  // ---- Q | K | V of every shard's heads: X_k Wqkv_p
      GemmLaunch L;
      L.epi = EPI_H_IDENTITY;
      L.num_shards = s.P;
      for (int p = 0; p < s.P; ++p) {
        L.a[p] = {X, s.M, s.d, s.d};
        L.b0[p] = {Wqkv[p], s.qkv_cols(), s.d, s.d};
        L.b1[p] = L.b0[p];
        L.out[p] = qkv[p];
      }
      L.ldo = s.qkv_cols();
      L.out_rows = s.M;
      L.out_cols = s.qkv_cols();
      L.a_row0 = row0;
      L.out_row0 = row0;
      L.rows = static_cast<int32_t>(s.Mc);
      L.n_base = 0;
      L.n_end = static_cast<int32_t>(s.qkv_cols());
      L.K = s.d;
      L.status = status;
      L.timeout_ns = tmo;
      st = timed(*T, s0, 0, DOMINO_KERNEL_GEMM1, k, 0, [&] { return run_gemm(L, grid, pair, s0, err); });
      if (st != DOMINO_OK) return st;
    }
    {  // ---- attention core of every (shard, sequence, head, query tile) of the chunk
      AttnLaunch L;
      for (int p = 0; p < s.P; ++p) {
        L.qkv[p] = qkv[p];
        L.o[p] = o[p];
      }
      L.M = s.M;
      L.S = s.S;
      L.row0 = row0;
      L.seqs = static_cast<int32_t>(s.B / s.mu);
      L.Hp = s.Hp;
      L.dh = s.dh;
      L.P = s.P;
      L.status = status;
      L.timeout_ns = tmo;
      st = timed(*T, s0, 0, DOMINO_KERNEL_ATTN, k, 0, [&] { return launch_attn_fwd(L, grid.num_sms, s0, err); });
      if (st != DOMINO_OK) return st;
    }
    if (s.schedule == DOMINO_SCHEDULE_FUSED && k == s.mu - 1) {
      // the last chunk's shard-sum has no next chunk to hide under: tile-granular inside its projection
      st = out_proj_fused(k, err);
      if (st != DOMINO_ERR_UNSUPPORTED) return st;  // else: the separate launches below
    }
    {  // ---- output projection of every shard into its partial buffer: O_p Wo_p
      GemmLaunch L;
      L.epi = s.partial == DOMINO_PARTIAL_F32 ? EPI_Z_F32 : EPI_Z_BF16;
      L.num_shards = s.P;
      for (int p = 0; p < s.P; ++p) {
        L.a[p] = {o[p], s.M, s.o_cols(), s.o_cols()};
        L.b0[p] = {Wo[p], s.d, s.o_cols(), s.o_cols()};
        L.b1[p] = L.b0[p];
        L.out[p] = Z[p];
      }
      L.ldo = s.d;
      L.out_rows = s.M;
      L.out_cols = s.d;
      L.a_row0 = row0;
      L.out_row0 = row0;
      L.rows = static_cast<int32_t>(s.Mc);
      L.n_base = 0;
      L.n_end = static_cast<int32_t>(s.d);
      L.K = s.o_cols();
      L.status = status;
      L.timeout_ns = tmo;
      st = timed(*T, s0, 0, DOMINO_KERNEL_GEMM2, k, 0, [&] { return run_gemm(L, grid, pair, s0, err); });
      if (st != DOMINO_OK) return st;
    }
    // ---- Y_k = sum over p of the partials (the all-reduce of the row-parallel projection)
    if (sr != s0) {
      cudaEvent_t ev = ds->ev_piece[k];
      cudaEventRecord(ev, s0);
      cudaStreamWaitEvent(sr, ev, 0);
    }
    ShardSumParams q;
    memset(&q, 0, sizeof q);
    const size_t zoff = static_cast<size_t>(row0) * s.d * s.psize;
    for (int p = 0; p < s.P; ++p) q.part[p] = static_cast<uint8_t*>(Z[p]) + zoff;
    q.rows = s.Mc;
    q.cols = s.d;
    q.ld_part = s.d;
    q.ld_y = s.d;
    q.y = static_cast<uint8_t*>(Y) + static_cast<size_t>(row0) * s.d * 2;
    q.P = s.P;
    q.f32 = s.partial == DOMINO_PARTIAL_F32;
    return timed(*T, sr, sr != s0, DOMINO_KERNEL_SHARD_SUM, k, 0,
                 [&] { return launch_shard_sum(q, grid.num_sms, sr, err); });
  }
};


}  // namespace

namespace domino {
// Lets other translation units of the library report a detailed error through
// domino_last_error().
void set_last_error(const std::string& msg) { g_last_error = msg; }
domino_status_t validate_desc(const domino_mlp_desc_t* desc) {
  Shape s;
  return check_desc(desc, &s);
}
domino_status_t validate_attn_desc(const domino_attn_desc_t* desc) {
  AttnShape s;
  return check_attn_desc(desc, &s);
}
}  // namespace domino

// ====================================================================== ABI

extern "C" {

const char* domino_status_string(domino_status_t status) {
  switch (status) {
    case DOMINO_OK: return "DOMINO_OK";
    case DOMINO_ERR_INVALID_ARG: return "DOMINO_ERR_INVALID_ARG";
    case DOMINO_ERR_UNSUPPORTED: return "DOMINO_ERR_UNSUPPORTED";
    case DOMINO_ERR_ALIGNMENT: return "DOMINO_ERR_ALIGNMENT";
    case DOMINO_ERR_WORKSPACE: return "DOMINO_ERR_WORKSPACE";
    case DOMINO_ERR_CUDA: return "DOMINO_ERR_CUDA";
    case DOMINO_ERR_TIMEOUT: return "DOMINO_ERR_TIMEOUT";
    case DOMINO_ERR_DEVICE: return "DOMINO_ERR_DEVICE";
    default: return "DOMINO_ERR_UNKNOWN";
  }
}

const char* domino_last_error(void) { return g_last_error.c_str(); }

size_t domino_mlp_workspace_size(const domino_mlp_desc_t* desc, int32_t with_bwd) {
  Shape s;
  if (check_desc(desc, &s) != DOMINO_OK) return 0;
  return ws_layout(s, with_bwd != 0).total;
}

size_t domino_mlp_saved_size(const domino_mlp_desc_t* desc) {
  Shape s;
  if (check_desc(desc, &s) != DOMINO_OK) return 0;
  return saved_shard_bytes(s) * s.P;
}

}  // extern "C"

namespace {
// The forward pass of domino_mlp_fwd (Z_out == NULL: partials in the workspace, summed into Y) and of
// domino_mlp_fwd_partials (Z_out != NULL: the partials, written to the caller's buffers, are the result).
domino_status_t mlp_fwd_impl(const domino_mlp_desc_t* desc, const void* X, const void* const* A_shards,
                             const void* const* B_shards, void* Y, void* const* Z_out, void* const* piece_events,
                             void* saved, void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  domino_status_t st = check_desc(desc, &s);
  if (st != DOMINO_OK) return st;
  const bool reduce = Z_out == nullptr;
  if (s.M == 0) return DOMINO_OK;  // an empty batch reads and writes nothing; X and Y may be NULL
  if (!X || !A_shards || !B_shards || (reduce && !Y) || !workspace)
    return fail(DOMINO_ERR_INVALID_ARG, reduce ? "X, A_shards, B_shards, Y and workspace must be non-NULL"
                                               : "X, A_shards, B_shards, Z_shards and workspace must be non-NULL");
  for (int p = 0; p < s.P; ++p) {
    if (!A_shards[p] || !B_shards[p] || (!reduce && !Z_out[p]))
      return fail(DOMINO_ERR_INVALID_ARG, "NULL shard pointer");
    if (!aligned16(A_shards[p]) || !aligned16(B_shards[p]) || (!reduce && !aligned16(Z_out[p])))
      return fail(DOMINO_ERR_ALIGNMENT, "shard pointers must be 16-byte aligned");
  }
  if (!reduce && piece_events)
    for (int i = 0; i < s.mu * s.S; ++i)
      if (!piece_events[i]) return fail(DOMINO_ERR_INVALID_ARG, "NULL piece event");
  if (!aligned16(X) || (reduce && !aligned16(Y)) || (saved && !aligned16(saved)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(DOMINO_ERR_ALIGNMENT, "X, Y, saved must be 16-byte and workspace 256-byte aligned");
  const WsLayout W = ws_layout(s, false);
  if (workspace_bytes < W.total) return fail(DOMINO_ERR_WORKSPACE, "workspace smaller than domino_mlp_workspace_size()");

  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != DOMINO_OK) return st;
  st = check_reserve(ds, desc->reserve_sms);
  if (st != DOMINO_OK) return st;

  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  cudaStream_t sr = s.schedule == DOMINO_SCHEDULE_STREAMS ? ds->reduce_stream : s0;
  const uint64_t tmo = desc->timeout_ns ? desc->timeout_ns : kDefaultTimeoutNs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DeviceStatus* dstat = reinterpret_cast<DeviceStatus*>(ws);

  Timer T;
  T.on = (desc->flags & DOMINO_FLAG_KERNEL_TIMES) != 0;
  T.ds = ds;
  const bool pair = (desc->flags & DOMINO_FLAG_ONE_CTA) == 0 && ds->pair_max_clusters > 0;
  if (T.on && !T.start(s0)) return fail(DOMINO_ERR_CUDA, "cudaEventCreate failed");

  FwdSeq f;
  f.s = s;
  f.ds = ds;
  f.grid = grid_for(ds, desc->reserve_sms);
  f.T = &T;
  f.s0 = s0;
  f.sr = sr;
  f.pair = pair;
  f.status = dstat;
  f.tmo = tmo;
  f.X = X;
  f.A_shards = A_shards;
  f.B_shards = B_shards;
  f.Y = Y;
  f.ev_piece = ds->ev_piece;
  f.bind(ws, W, saved);
  f.reduce = reduce;
  f.user_events = piece_events;
  if (!reduce)
    for (int p = 0; p < s.P; ++p) f.Z[p] = Z_out[p];
  static const int kEpiOfAct[4] = {EPI_H_GELU, EPI_H_GELU_TANH, EPI_H_SWIGLU, EPI_H_IDENTITY};
  std::string err;

  if (s.schedule == DOMINO_SCHEDULE_FUSED) {
    if (f.grid.fused_ctas < 1) return fail(DOMINO_ERR_DEVICE, "fused kernel cannot be resident on this device");
    FusedLaunch F;
    F.X = X;
    for (int p = 0; p < s.P; ++p) {
      F.A_shards[p] = A_shards[p];
      F.B_shards[p] = B_shards[p];
      F.H[p] = f.H[p];
      F.aux[p] = f.pre[p];
      F.Z[p] = f.Z[p];
    }
    F.Y = reduce ? Y : nullptr;
    F.reduce = reduce;
    F.sync = reinterpret_cast<uint32_t*>(ws + W.sync_off);
    F.timeline = reinterpret_cast<uint64_t*>(ws + kTimelineOff);
    F.M = s.M;
    F.d = s.d;
    F.Fp = s.Fp;
    F.mu = s.mu;
    F.P = s.P;
    F.epi_a = kEpiOfAct[s.act];
    F.partial_f32 = s.partial == DOMINO_PARTIAL_F32;
    F.status = dstat;
    F.timeout_ns = tmo;
    static_assert(kTimelineOff + 24 <= kSyncOff, "timeline words precede the counters");
    cudaError_t e = cudaMemsetAsync(ws + kTimelineOff, 0, kSyncOff - kTimelineOff + W.sync_bytes, s0);
    if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("counter reset: ") + cudaGetErrorString(e));
    F.pair = pair;
    st = timed(T, s0, 0, DOMINO_KERNEL_FUSED, 0, 0, [&] {
      domino_status_t r = launch_fused_fwd(F, f.grid.fused_ctas, f.grid.fused_pair_clusters, s0, &err);
      if (r == DOMINO_ERR_UNSUPPORTED && F.pair) {
        // paired cooperative launches refused on this device: use one-CTA tiles from now on
        ds->fused_pair_clusters = 0;
        F.pair = false;
        r = launch_fused_fwd(F, f.grid.fused_ctas, 0, s0, &err);
      }
      return r;
    });
    if (st != DOMINO_OK) return fail(st, err);
    if (!reduce && piece_events)  // one launch: every piece is complete when it ends
      for (int i = 0; i < s.mu * s.S; ++i) {
        cudaError_t e2 = cudaEventRecord(static_cast<cudaEvent_t>(piece_events[i]), s0);
        if (e2 != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("piece event record: ") + cudaGetErrorString(e2));
      }
    return DOMINO_OK;
  }

  fork_streams(ds, s0, sr);
  for (int k = 0; k < s.mu; ++k) {
    st = f.chunk(k, &err);
    if (st != DOMINO_OK) return fail(st, err);
  }
  join_streams(ds, s0, sr);
  return DOMINO_OK;
}
}  // namespace

extern "C" {

domino_status_t domino_mlp_fwd(const domino_mlp_desc_t* desc, const void* X, const void* const* A_shards,
                               const void* const* B_shards, void* Y, void* saved, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return mlp_fwd_impl(desc, X, A_shards, B_shards, Y, nullptr, nullptr, saved, workspace, workspace_bytes, stream);
}

domino_status_t domino_mlp_fwd_partials(const domino_mlp_desc_t* desc, const void* X, const void* const* A_shards,
                                        const void* const* B_shards, void* const* Z_shards, void* const* piece_events,
                                        void* saved, void* workspace, size_t workspace_bytes, void* stream) {
  if (!Z_shards) return fail(DOMINO_ERR_INVALID_ARG, "Z_shards must be non-NULL");
  return mlp_fwd_impl(desc, X, A_shards, B_shards, nullptr, Z_shards, piece_events, saved, workspace,
                      workspace_bytes, stream);
}

domino_status_t domino_mlp_bwd(const domino_mlp_desc_t* desc, const void* X, const void* const* A_shards,
                               const void* const* B_shards, const void* dY, const void* saved, void* dX,
                               void* const* dA_shards, void* const* dB_shards, void* workspace,
                               size_t workspace_bytes, void* stream) {
  Shape s;
  domino_status_t st = check_desc(desc, &s);
  if (st != DOMINO_OK) return st;
  if (!A_shards || !B_shards || !dA_shards || !dB_shards)
    return fail(DOMINO_ERR_INVALID_ARG, "A_shards, B_shards, dA_shards and dB_shards must be non-NULL");
  for (int p = 0; p < s.P; ++p) {
    if (!A_shards[p] || !B_shards[p] || !dA_shards[p] || !dB_shards[p])
      return fail(DOMINO_ERR_INVALID_ARG, "NULL shard pointer");
    if (!aligned16(A_shards[p]) || !aligned16(B_shards[p]) || !aligned16(dA_shards[p]) || !aligned16(dB_shards[p]))
      return fail(DOMINO_ERR_ALIGNMENT, "shard pointers must be 16-byte aligned");
  }
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  if (s.M == 0) {
    // gradients of a sum over no tokens: zero weight gradients, nothing else touched
    for (int p = 0; p < s.P; ++p) {
      cudaError_t e = cudaMemsetAsync(dA_shards[p], 0, static_cast<size_t>(s.nact) * s.Fp * s.d * 2, s0);
      if (e == cudaSuccess) e = cudaMemsetAsync(dB_shards[p], 0, static_cast<size_t>(s.d) * s.Fp * 2, s0);
      if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("memset: ") + cudaGetErrorString(e));
    }
    return DOMINO_OK;
  }
  if (!X || !dY || !saved || !dX || !workspace)
    return fail(DOMINO_ERR_INVALID_ARG, "X, dY, saved, dX and workspace must be non-NULL");
  if (!aligned16(X) || !aligned16(dY) || !aligned16(saved) || !aligned16(dX) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(DOMINO_ERR_ALIGNMENT, "X, dY, saved, dX must be 16-byte and workspace 256-byte aligned");
  const WsLayout W = ws_layout(s, true);
  if (workspace_bytes < W.total)
    return fail(DOMINO_ERR_WORKSPACE, "workspace smaller than domino_mlp_workspace_size(desc, 1)");

  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != DOMINO_OK) return st;
  st = check_reserve(ds, desc->reserve_sms);
  if (st != DOMINO_OK) return st;
  // FUSED: dH, one cooperative launch for the partial input gradients of every chunk and their shard-sum, then
  // the weight gradients (STREAMS if the device cannot run the cooperative launch)
  cudaStream_t sr = s.schedule != DOMINO_SCHEDULE_SERIAL ? ds->reduce_stream : s0;
  const uint64_t tmo = desc->timeout_ns ? desc->timeout_ns : kDefaultTimeoutNs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DeviceStatus* dstat = reinterpret_cast<DeviceStatus*>(ws);
  Timer T;
  T.on = (desc->flags & DOMINO_FLAG_KERNEL_TIMES) != 0;
  T.ds = ds;
  const bool pair = (desc->flags & DOMINO_FLAG_ONE_CTA) == 0 && ds->pair_max_clusters > 0;
  if (T.on && !T.start(s0)) return fail(DOMINO_ERR_CUDA, "cudaEventCreate failed");

  BwdSeq g;
  g.s = s;
  g.ds = ds;
  g.grid = grid_for(ds, desc->reserve_sms);
  g.T = &T;
  g.s0 = s0;
  g.sr = sr;
  g.pair = pair;
  g.status = dstat;
  g.tmo = tmo;
  g.X = X;
  g.A_shards = A_shards;
  g.B_shards = B_shards;
  g.dY = dY;
  g.dX = dX;
  g.dA_shards = dA_shards;
  g.dB_shards = dB_shards;
  g.ev_piece = ds->ev_piece;
  g.bind(ws, W, saved);
  std::string err;
  fork_streams(ds, s0, sr);
  st = g.dh(&err);
  bool fused_dx = false;
  if (st == DOMINO_OK && s.schedule == DOMINO_SCHEDULE_FUSED && pair) {
    const domino_status_t fs = g.dx_fused(ws, W, &err);
    if (fs == DOMINO_OK) fused_dx = true;
    else if (fs != DOMINO_ERR_UNSUPPORTED) st = fs;
  }
  for (int k = 0; k < s.mu && st == DOMINO_OK && !fused_dx; ++k) st = g.dx_chunk(k, &err);
  if (st == DOMINO_OK) st = g.dw(&err);
  if (st != DOMINO_OK) return fail(st, err);
  join_streams(ds, s0, sr);
  return DOMINO_OK;
}

size_t domino_mlp_interleaved_workspace_size(const domino_mlp_desc_t* desc) {
  Shape s;
  if (check_desc(desc, &s) != DOMINO_OK) return 0;
  return align_up(ws_layout(s, false).total, 256) + ws_layout(s, true).total;
}

domino_status_t domino_mlp_fwd_bwd_interleaved(const domino_mlp_desc_t* desc, const void* const* A_shards,
                                               const void* const* B_shards, const void* Xa, void* Ya,
                                               void* saved_a, const void* Xb, const void* dYb, const void* saved_b,
                                               void* dXb, void* const* dA_shards, void* const* dB_shards,
                                               void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  domino_status_t st = check_desc(desc, &s);
  if (st != DOMINO_OK) return st;
  if (s.schedule == DOMINO_SCHEDULE_FUSED)
    return fail(DOMINO_ERR_UNSUPPORTED, "interleaving places launches between pieces: use SERIAL or STREAMS");
  if (!A_shards || !B_shards || !dA_shards || !dB_shards)
    return fail(DOMINO_ERR_INVALID_ARG, "A_shards, B_shards, dA_shards and dB_shards must be non-NULL");
  for (int p = 0; p < s.P; ++p) {
    if (!A_shards[p] || !B_shards[p] || !dA_shards[p] || !dB_shards[p])
      return fail(DOMINO_ERR_INVALID_ARG, "NULL shard pointer");
    if (!aligned16(A_shards[p]) || !aligned16(B_shards[p]) || !aligned16(dA_shards[p]) || !aligned16(dB_shards[p]))
      return fail(DOMINO_ERR_ALIGNMENT, "shard pointers must be 16-byte aligned");
  }
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  if (s.M == 0) {
    // both strands are empty: strand b's weight gradients are zero, nothing else is touched
    for (int p = 0; p < s.P; ++p) {
      cudaError_t e = cudaMemsetAsync(dA_shards[p], 0, static_cast<size_t>(s.nact) * s.Fp * s.d * 2, s0);
      if (e == cudaSuccess) e = cudaMemsetAsync(dB_shards[p], 0, static_cast<size_t>(s.d) * s.Fp * 2, s0);
      if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("memset: ") + cudaGetErrorString(e));
    }
    return DOMINO_OK;
  }
  if (!Xa || !Ya || !Xb || !dYb || !saved_b || !dXb || !workspace)
    return fail(DOMINO_ERR_INVALID_ARG, "Xa, Ya, Xb, dYb, saved_b, dXb and workspace must be non-NULL");
  if (!aligned16(Xa) || !aligned16(Ya) || (saved_a && !aligned16(saved_a)) || !aligned16(Xb) || !aligned16(dYb) ||
      !aligned16(saved_b) || !aligned16(dXb) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(DOMINO_ERR_ALIGNMENT, "tensors must be 16-byte and workspace 256-byte aligned");
  const WsLayout Wa = ws_layout(s, false);
  const WsLayout Wb = ws_layout(s, true);
  const size_t off_b = align_up(Wa.total, 256);
  if (workspace_bytes < off_b + Wb.total)
    return fail(DOMINO_ERR_WORKSPACE, "workspace smaller than domino_mlp_interleaved_workspace_size()");

  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != DOMINO_OK) return st;
  st = check_reserve(ds, desc->reserve_sms);
  if (st != DOMINO_OK) return st;
  cudaStream_t sr = s.schedule == DOMINO_SCHEDULE_STREAMS ? ds->reduce_stream : s0;
  const uint64_t tmo = desc->timeout_ns ? desc->timeout_ns : kDefaultTimeoutNs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DeviceStatus* dstat = reinterpret_cast<DeviceStatus*>(ws);  // both strands report here
  Timer T;
  T.on = (desc->flags & DOMINO_FLAG_KERNEL_TIMES) != 0;
  T.ds = ds;
  const bool pair = (desc->flags & DOMINO_FLAG_ONE_CTA) == 0 && ds->pair_max_clusters > 0;
  if (T.on && !T.start(s0)) return fail(DOMINO_ERR_CUDA, "cudaEventCreate failed");

  FwdSeq f;
  f.s = s;
  f.ds = ds;
  f.grid = grid_for(ds, desc->reserve_sms);
  f.T = &T;
  f.s0 = s0;
  f.sr = sr;
  f.pair = pair;
  f.status = dstat;
  f.tmo = tmo;
  f.X = Xa;
  f.A_shards = A_shards;
  f.B_shards = B_shards;
  f.Y = Ya;
  f.ev_piece = ds->ev_piece;
  f.bind(ws, Wa, saved_a);
  BwdSeq g;
  g.s = s;
  g.ds = ds;
  g.grid = grid_for(ds, desc->reserve_sms);
  g.T = &T;
  g.s0 = s0;
  g.sr = sr;
  g.pair = pair;
  g.status = dstat;
  g.tmo = tmo;
  g.X = Xb;
  g.A_shards = A_shards;
  g.B_shards = B_shards;
  g.dY = dYb;
  g.dX = dXb;
  g.dA_shards = dA_shards;
  g.dB_shards = dB_shards;
  g.ev_piece = ds->ev_piece_b;
  g.bind(ws + off_b, Wb, saved_b);

  // strand b's dH first (no exchange), then the two strands' chunks alternate:
  // the shard-sums of one strand's chunk k run on the reduction stream beside
  // the other strand's GEMMs; strand b's weight gradients cover the last ones.
  std::string err;
  fork_streams(ds, s0, sr);
  st = g.dh(&err);
  for (int k = 0; k < s.mu && st == DOMINO_OK; ++k) {
    st = f.chunk(k, &err);
    if (st == DOMINO_OK) st = g.dx_chunk(k, &err);
  }
  if (st == DOMINO_OK) st = g.dw(&err);
  if (st != DOMINO_OK) return fail(st, err);
  join_streams(ds, s0, sr);
  return DOMINO_OK;
}

size_t domino_attn_workspace_size(const domino_attn_desc_t* desc) {
  AttnShape s;
  if (check_attn_desc(desc, &s) != DOMINO_OK) return 0;
  return attn_ws_layout(s).total;
}

domino_status_t domino_attn_fwd(const domino_attn_desc_t* desc, const void* X, const void* const* Wqkv_shards,
                                const void* const* Wo_shards, void* Y, void* workspace, size_t workspace_bytes,
                                void* stream) {
  AttnShape s;
  domino_status_t st = check_attn_desc(desc, &s);
  if (st != DOMINO_OK) return st;
  if (s.M == 0) return DOMINO_OK;
  if (!X || !Wqkv_shards || !Wo_shards || !Y || !workspace)
    return fail(DOMINO_ERR_INVALID_ARG, "X, Wqkv_shards, Wo_shards, Y and workspace must be non-NULL");
  for (int p = 0; p < s.P; ++p) {
    if (!Wqkv_shards[p] || !Wo_shards[p]) return fail(DOMINO_ERR_INVALID_ARG, "NULL shard pointer");
    if (!aligned16(Wqkv_shards[p]) || !aligned16(Wo_shards[p]))
      return fail(DOMINO_ERR_ALIGNMENT, "shard pointers must be 16-byte aligned");
  }
  if (!aligned16(X) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(DOMINO_ERR_ALIGNMENT, "X, Y must be 16-byte and workspace 256-byte aligned");
  const AttnWs W = attn_ws_layout(s);
  if (workspace_bytes < W.total)
    return fail(DOMINO_ERR_WORKSPACE, "workspace smaller than domino_attn_workspace_size()");

  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != DOMINO_OK) return st;
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  // STREAMS, and FUSED for every chunk but the last: the shard-sum on the reduction stream under the next chunk
  cudaStream_t sr = s.schedule != DOMINO_SCHEDULE_SERIAL ? ds->reduce_stream : s0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Timer T;
  T.on = (desc->flags & DOMINO_FLAG_KERNEL_TIMES) != 0;
  T.ds = ds;
  if (T.on && !T.start(s0)) return fail(DOMINO_ERR_CUDA, "cudaEventCreate failed");

  AttnSeq a;
  a.s = s;
  a.ds = ds;
  a.grid = grid_for(ds, 0);
  a.T = &T;
  a.s0 = s0;
  a.sr = sr;
  a.pair = (desc->flags & DOMINO_FLAG_ONE_CTA) == 0 && ds->pair_max_clusters > 0;
  a.status = reinterpret_cast<DeviceStatus*>(ws);
  a.tmo = desc->timeout_ns ? desc->timeout_ns : kDefaultTimeoutNs;
  a.X = X;
  a.Wqkv = Wqkv_shards;
  a.Wo = Wo_shards;
  a.Y = Y;
  a.ws = ws;
  a.W = W;
  for (int p = 0; p < s.P; ++p) {
    a.qkv[p] = ws + W.qkv_off + W.qkv_shard * p;
    a.o[p] = ws + W.o_off + W.o_shard * p;
    a.Z[p] = ws + W.z_off + W.z_shard * p;
  }
  std::string err;
  fork_streams(ds, s0, sr);
  for (int k = 0; k < s.mu; ++k) {
    st = a.chunk(k, &err);
    if (st != DOMINO_OK) return fail(st, err);
  }
  join_streams(ds, s0, sr);
  return DOMINO_OK;
}

domino_status_t domino_shard_sum(const void* const* partials, int32_t P, int32_t partial_dtype, int64_t rows,
                                 int64_t cols, int64_t ld_partial, void* Y, int64_t ld_y, void* stream) {
  if (!partials || !Y) return fail(DOMINO_ERR_INVALID_ARG, "partials and Y must be non-NULL");
  if (P < 1 || P > DOMINO_MAX_SHARDS) return fail(DOMINO_ERR_INVALID_ARG, "P must be in 1..DOMINO_MAX_SHARDS");
  if (partial_dtype != DOMINO_PARTIAL_F32 && partial_dtype != DOMINO_PARTIAL_BF16)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown partial_dtype");
  if (rows < 0 || cols < 0 || ld_partial < cols || ld_y < cols)
    return fail(DOMINO_ERR_INVALID_ARG, "bad rows/cols/leading dimensions");
  if (cols % 8 || ld_partial % 8 || ld_y % 8)
    return fail(DOMINO_ERR_ALIGNMENT, "cols and leading dimensions must be multiples of 8");
  if (rows > 0 && cols > 0 && rows * (cols / 8) >= (int64_t(1) << 32))
    return fail(DOMINO_ERR_UNSUPPORTED, "rows * cols / 8 must be below 2^32");
  for (int p = 0; p < P; ++p) {
    if (!partials[p]) return fail(DOMINO_ERR_INVALID_ARG, "NULL partial pointer");
    if (!aligned16(partials[p])) return fail(DOMINO_ERR_ALIGNMENT, "partials must be 16-byte aligned");
  }
  if (!aligned16(Y)) return fail(DOMINO_ERR_ALIGNMENT, "Y must be 16-byte aligned");
  if (rows == 0 || cols == 0) return DOMINO_OK;
  DeviceState* ds = nullptr;
  domino_status_t st = device_state(&ds);
  if (st != DOMINO_OK) return st;
  ShardSumParams q;
  memset(&q, 0, sizeof q);
  for (int p = 0; p < P; ++p) q.part[p] = partials[p];
  q.rows = rows;
  q.cols = cols;
  q.ld_part = ld_partial;
  q.ld_y = ld_y;
  q.y = Y;
  q.P = P;
  q.f32 = partial_dtype == DOMINO_PARTIAL_F32;
  std::string err;
  st = launch_shard_sum(q, ds->num_sms, static_cast<cudaStream_t>(stream), &err);
  if (st != DOMINO_OK) return fail(st, err);
  return DOMINO_OK;
}

domino_status_t domino_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, void* stream) {
  if (!workspace) return fail(DOMINO_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(DOMINO_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DeviceState* ds = nullptr;
  domino_status_t st = device_state(&ds);
  if (st != DOMINO_OK) return st;
  std::string err;
  st = launch_selftest_wait(workspace, timeout_ns, static_cast<cudaStream_t>(stream), &err);
  if (st != DOMINO_OK) return fail(st, err);
  return DOMINO_OK;
}

domino_status_t domino_read_timeline(const void* workspace, void* stream, domino_timeline_t* out) {
  if (!workspace || !out) return fail(DOMINO_ERR_INVALID_ARG, "workspace and out must be non-NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess)
    e = cudaMemcpy(out, static_cast<const uint8_t*>(workspace) + kTimelineOff, sizeof(domino_timeline_t),
                   cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("timeline read: ") + cudaGetErrorString(e));
  if (out->start_ns != 0) out->start_ns = ~out->start_ns;  // the kernel keeps the complement of the start
  return DOMINO_OK;
}

domino_status_t domino_query_device_status(void* workspace, void* stream) {
  if (!workspace) return fail(DOMINO_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("stream sync: ") + cudaGetErrorString(e));
  DeviceStatus h;
  e = cudaMemcpy(&h, workspace, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
  if (h.code == 0) return DOMINO_OK;
  e = cudaMemset(workspace, 0, sizeof h);
  if (e != cudaSuccess) return fail(DOMINO_ERR_CUDA, std::string("status clear: ") + cudaGetErrorString(e));
  char buf[160];
  snprintf(buf, sizeof buf, "device wait gave up: site %u, block %u, detail %u", h.where, h.block, h.aux);
  return fail(static_cast<domino_status_t>(h.code), buf);
}

int32_t domino_kernel_times(domino_kernel_time_t* out, int32_t max_records) {
  std::lock_guard<std::mutex> lock(g_mutex);
  const int32_t n = static_cast<int32_t>(g_timing.launches.size());
  for (int32_t i = 0; i < n && out && i < max_records; ++i) {
    const TimedLaunch& t = g_timing.launches[i];
    float b = 0.f, e = 0.f;
    if (cudaEventSynchronize(t.end) != cudaSuccess) return -1;
    cudaEventElapsedTime(&b, t.origin, t.begin);
    cudaEventElapsedTime(&e, t.origin, t.end);
    out[i] = {t.call, t.kind, t.chunk, t.slice, t.stream, b, e};
  }
  return n;
}

void domino_kernel_times_reset(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_timing.calls = 0;
  g_timing.launches.clear();
  for (DeviceState& ds : g_devices) ds.timing_next = 0;
}

}  // extern "C"
