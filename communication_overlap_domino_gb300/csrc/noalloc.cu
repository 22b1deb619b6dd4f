// domino_mlp_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they
// run the layer: code inside a real-time or latency-critical loop that must not
// hit the driver's allocator, embedded or plugin hosts whose memory is handed out
// by someone else, or runtimes that forbid allocation after start-up.  This entry
// point needs no workspace from them: its scratch memory (the hidden activations
// and the shard partials) lives in one file-scope __device__ array of fixed size,
// which every GPU that loads the library holds until the process exits.
//
// The array's name is only a host-side stand-in in host code, so its device
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, during the first call on the device; that first call should
// therefore come before any stream capture.  The computation is the forward
// pass's serial schedule with one-CTA GEMM tiles (the kernels domino_mlp_fwd
// runs with DOMINO_SCHEDULE_SERIAL and DOMINO_FLAG_ONE_CTA, in the same order,
// on `stream`).
//
// The first 256 bytes of the array are a header that every call clears: its
// first 16 bytes are the device status words the GEMMs' bounded waits record a
// timeout into, read back by domino_mlp_fwd_noalloc_status.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "gemm.h"

namespace {

using namespace domino;

__device__ __align__(256) uint8_t g_noalloc_scratch[DOMINO_NOALLOC_SCRATCH_BYTES];

struct NoallocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};

std::mutex g_noalloc_mutex;
NoallocDevice g_noalloc_devices[64];

domino_status_t noalloc_fail(domino_status_t st, const std::string& msg) {
  set_last_error(msg);
  return st;
}

// Once per device, with the device current: the scratch array's device address,
// the SM count and the GEMM kernels' shared-memory attribute.
domino_status_t noalloc_setup(NoallocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(DOMINO_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return noalloc_fail(DOMINO_ERR_DEVICE, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocDevice& nd = g_noalloc_devices[dev];
  if (!nd.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return noalloc_fail(DOMINO_ERR_DEVICE, "this library is built for sm_103a (GB300)");
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return noalloc_fail(DOMINO_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    e = cudaDeviceGetAttribute(&nd.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = prepare_gemm_kernels();
    if (e != cudaSuccess) return noalloc_fail(DOMINO_ERR_CUDA, std::string("setup: ") + cudaGetErrorString(e));
    nd.scratch = static_cast<uint8_t*>(ptr);
    nd.ready = true;
  }
  *out = &nd;
  return DOMINO_OK;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" DOMINO_API domino_status_t domino_mlp_fwd_noalloc(const domino_mlp_desc_t* desc, const void* X,
                                                             const void* const* A_shards,
                                                             const void* const* B_shards, void* Y, void* stream) {
  // Descriptor errors: the same checks and codes as domino_mlp_fwd (which returns
  // before touching anything when the descriptor is invalid).
  const size_t need = domino_mlp_workspace_size(desc, 0);
  if (need == 0) return domino_mlp_fwd(desc, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr);
  if ((desc->flags & DOMINO_FLAG_KERNEL_TIMES) != 0)
    return noalloc_fail(DOMINO_ERR_INVALID_ARG, "domino_mlp_fwd_noalloc does not record kernel times (flags must be 0)");
  if (need > DOMINO_NOALLOC_SCRATCH_BYTES) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "problem needs %zu bytes of scratch; domino_mlp_fwd_noalloc holds %zu (use domino_mlp_fwd with a workspace)",
             need, static_cast<size_t>(DOMINO_NOALLOC_SCRATCH_BYTES));
    return noalloc_fail(DOMINO_ERR_WORKSPACE, buf);
  }
  const int64_t M = desc->M, d = desc->d, F = desc->F;
  const int P = desc->P, mu = desc->mu, S = desc->out_slices;
  if (M == 0) return DOMINO_OK;
  if (!X || !A_shards || !B_shards || !Y)
    return noalloc_fail(DOMINO_ERR_INVALID_ARG, "X, A_shards, B_shards and Y must be non-NULL");
  for (int p = 0; p < P; ++p) {
    if (!A_shards[p] || !B_shards[p]) return noalloc_fail(DOMINO_ERR_INVALID_ARG, "NULL shard pointer");
    if (!is_aligned16(A_shards[p]) || !is_aligned16(B_shards[p]))
      return noalloc_fail(DOMINO_ERR_ALIGNMENT, "shard pointers must be 16-byte aligned");
  }
  if (!is_aligned16(X) || !is_aligned16(Y)) return noalloc_fail(DOMINO_ERR_ALIGNMENT, "X and Y must be 16-byte aligned");

  NoallocDevice* nd = nullptr;
  domino_status_t st = noalloc_setup(&nd);
  if (st != DOMINO_OK) return st;
  const int sms = nd->num_sms - desc->reserve_sms;  // the SMs the persistent grids spread over
  if (sms < 2) return noalloc_fail(DOMINO_ERR_INVALID_ARG, "reserve_sms must leave at least 2 SMs to the library");

  const int64_t Fp = F / P, Mc = M / mu, ds = d / S;
  const bool swiglu = desc->act == DOMINO_ACT_SWIGLU;
  const bool f32 = desc->partial_dtype == DOMINO_PARTIAL_F32;
  const size_t psize = f32 ? 4 : 2;
  const uint64_t tmo = desc->timeout_ns ? desc->timeout_ns : 2000000000ull;
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);

  // Scratch layout: 256-byte header (device status words at bytes 0-15) |
  // H [P][M][Fp] bf16 | Z [P][M][d].  H and Z are fully written before they are
  // read, so only the header is cleared.
  uint8_t* base = nd->scratch;
  const size_t h_shard = static_cast<size_t>(M) * Fp * 2;
  const size_t z_off = (256 + h_shard * P + 255) / 256 * 256;
  const size_t z_shard = static_cast<size_t>(M) * d * psize;
  cudaError_t e = cudaMemsetAsync(base, 0, 256, s0);
  if (e != cudaSuccess) return noalloc_fail(DOMINO_ERR_CUDA, std::string("header clear: ") + cudaGetErrorString(e));

  static const int kEpiOfAct[4] = {EPI_H_GELU, EPI_H_GELU_TANH, EPI_H_SWIGLU, EPI_H_IDENTITY};
  DeviceStatus* status = reinterpret_cast<DeviceStatus*>(base);
  std::string err;
  for (int k = 0; k < mu; ++k) {
    const int32_t row0 = static_cast<int32_t>(k * Mc);
    GemmLaunch L1;
    L1.epi = kEpiOfAct[desc->act];
    L1.num_shards = P;
    for (int p = 0; p < P; ++p) {
      const uint8_t* Ap = static_cast<const uint8_t*>(A_shards[p]);
      L1.a[p] = {X, M, d, d};
      L1.b0[p] = {Ap, Fp, d, d};
      L1.b1[p] = swiglu ? Operand2D{Ap + static_cast<size_t>(Fp) * d * 2, Fp, d, d} : L1.b0[p];
      L1.out[p] = base + 256 + h_shard * p;
    }
    L1.n_tile = swiglu ? kBN / 2 : kBN;
    L1.b1_off = swiglu ? 0 : kBN / 2;
    L1.ldo = Fp;
    L1.a_row0 = row0;
    L1.out_row0 = row0;
    L1.rows = static_cast<int32_t>(Mc);
    L1.n_base = 0;
    L1.n_end = static_cast<int32_t>(Fp);
    L1.K = d;
    L1.status = status;
    L1.timeout_ns = tmo;
    st = launch_gemm(L1, sms, s0, &err);
    if (st != DOMINO_OK) return noalloc_fail(st, err);
    for (int sl = 0; sl < S; ++sl) {
      const int32_t col0 = static_cast<int32_t>(sl * ds);
      GemmLaunch L2;
      L2.epi = f32 ? EPI_Z_F32 : EPI_Z_BF16;
      L2.num_shards = P;
      for (int p = 0; p < P; ++p) {
        L2.a[p] = {base + 256 + h_shard * p, M, Fp, Fp};
        L2.b0[p] = {B_shards[p], d, Fp, Fp};
        L2.b1[p] = L2.b0[p];
        L2.out[p] = base + z_off + z_shard * p;
      }
      L2.ldo = d;
      L2.a_row0 = row0;
      L2.out_row0 = row0;
      L2.rows = static_cast<int32_t>(Mc);
      L2.n_base = col0;
      L2.n_end = static_cast<int32_t>(col0 + ds);
      L2.K = Fp;
      L2.status = status;
      L2.timeout_ns = tmo;
      st = launch_gemm(L2, sms, s0, &err);
      if (st != DOMINO_OK) return noalloc_fail(st, err);
      ShardSumParams q;
      memset(&q, 0, sizeof q);
      const size_t zoff = (static_cast<size_t>(row0) * d + col0) * psize;
      for (int p = 0; p < P; ++p) q.part[p] = base + z_off + z_shard * p + zoff;
      q.rows = Mc;
      q.cols = ds;
      q.ld_part = d;
      q.ld_y = d;
      q.y = static_cast<uint8_t*>(Y) + (static_cast<size_t>(row0) * d + col0) * 2;
      q.P = P;
      q.f32 = f32 ? 1 : 0;
      st = launch_shard_sum(q, sms, s0, &err);
      if (st != DOMINO_OK) return noalloc_fail(st, err);
    }
  }
  return DOMINO_OK;
}

extern "C" DOMINO_API domino_status_t domino_mlp_fwd_noalloc_status(void* stream, void** header) {
  NoallocDevice* nd = nullptr;
  domino_status_t st = noalloc_setup(&nd);
  if (st != DOMINO_OK) return st;
  if (header) *header = nd->scratch;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return noalloc_fail(DOMINO_ERR_CUDA, std::string("stream sync: ") + cudaGetErrorString(e));
  DeviceStatus h;
  e = cudaMemcpy(&h, nd->scratch, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return noalloc_fail(DOMINO_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
  if (h.code == 0) return DOMINO_OK;
  e = cudaMemset(nd->scratch, 0, sizeof h);
  if (e != cudaSuccess) return noalloc_fail(DOMINO_ERR_CUDA, std::string("status clear: ") + cudaGetErrorString(e));
  char buf[160];
  snprintf(buf, sizeof buf, "no-alloc forward: device wait gave up: site %u, block %u, detail %u", h.where, h.block,
           h.aux);
  return noalloc_fail(static_cast<domino_status_t>(h.code), buf);
}
