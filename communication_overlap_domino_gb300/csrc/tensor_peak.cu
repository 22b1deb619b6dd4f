// Tensor-core rate probe: back-to-back paired tcgen05 MMAs (cta_group::2,
// 256 x 256 x 16, bf16 in, fp32 accumulate) on operands already in shared
// memory, with no loads, stores or epilogue.  It measures the ceiling that the
// GEMM kernels' main loops approach on this GPU at its current clock.
//
// Each CTA of a 2-CTA cluster fills its 32 KB operand region (its 128 rows of
// A and of B over 64 K-columns, 128-byte-swizzled K-major; the swizzle does not
// matter for pseudo-random contents) with bf16 values of magnitude in [0.5, 1)
// and random sign, so the tensor cores toggle as they do on real data.  The
// two CTAs allocate 256 TMEM columns together; the even CTA's thread 0 issues
// the MMAs, commits them to a barrier and waits, bounded, until they are done.
// Cluster 0's thread 0 records the SM cycles and nanoseconds around that.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "domino.h"
#include "gemm.h"
#include "ptx.cuh"

namespace domino {

constexpr int kPeakThreads = 128;
constexpr int kPeakOperandBytes = 2 * 128 * kBK * 2;  // this CTA's 128 rows of A and of B, K = 64
// Far more shared memory than the operands need, so that no two CTAs share an
// SM (each SM's tensor core serves one pair member, as in the paired GEMMs).
constexpr int kPeakSmemBytes = 160 * 1024;
constexpr int kPeakClockOff = 16;  // workspace bytes 16-31: cycles and ns of cluster 0

__device__ __forceinline__ uint64_t clock64_now() {
  uint64_t c;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
  return c;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPeakThreads, 1)
    tensor_peak_kernel(int64_t mmas, uint8_t* workspace, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + kPeakOperandBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  DeviceStatus* status = reinterpret_cast<DeviceStatus*>(workspace);
  const int warp = threadIdx.x >> 5;
  const bool leader = cluster_ctarank() == 0;

  uint32_t* words = reinterpret_cast<uint32_t*>(smem);
  for (uint32_t i = threadIdx.x; i < kPeakOperandBytes / 4; i += blockDim.x) {
    uint32_t h = (i + 1u + 7919u * blockIdx.x) * 2654435761u;  // Knuth's multiplicative hash
    h ^= h >> 15;
    // two bf16: exponent of 0.5, 7 random mantissa bits and a random sign each
    const uint32_t lo = 0x3F00u | (h & 0x7Fu) | ((h >> 7) & 1u) << 15;
    const uint32_t hi = 0x3F00u | ((h >> 8) & 0x7Fu) | ((h >> 15) & 1u) << 15;
    words[i] = lo | hi << 16;
  }
  fence_proxy_async_shared();  // the operands are read by the tensor cores
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, 256);
    tmem_relinquish_alloc_permit_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (leader && threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(256, kBN);
    const uint64_t adesc = smem_desc_k128(smem_u32(smem));
    const uint64_t bdesc = smem_desc_k128(smem_u32(smem + kPeakOperandBytes / 2));
    const uint64_t c0 = clock64_now();
    const uint64_t t0 = globaltimer_ns();
    for (int64_t i = 0; i < mmas; ++i)  // K-steps of 16 (32 bytes) through the 64-column rows
      mma_bf16_ss_pair(tmem_base, adesc + 2 * (i & 3), bdesc + 2 * (i & 3), idesc, i > 0 ? 1u : 0u);
    mma_commit_pair_multicast(done, 0x1);
    volatile int abort = 0;
    if (!mbar_wait(done, 0, &abort, timeout_ns, status, kSiteDrain, 0)) {
      abort = 0;  // the MMAs still read shared memory and write TMEM: wait once more, bounded, before freeing
      mbar_wait(done, 0, &abort, timeout_ns, nullptr, kSiteDrain, 0);
    }
    const uint64_t c1 = clock64_now();
    const uint64_t t1 = globaltimer_ns();
    if (blockIdx.x == 0) {
      uint64_t* clk = reinterpret_cast<uint64_t*>(workspace + kPeakClockOff);
      clk[0] = c1 - c0;
      clk[1] = t1 - t0;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs no longer read the odd CTA's shared memory
  tc_fence_after_sync();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, 256);
  }
}

}  // namespace domino

namespace {

using domino::kPeakClockOff;
using domino::kPeakSmemBytes;
using domino::kPeakThreads;

domino_status_t peak_fail(domino_status_t st, const std::string& msg) {
  domino::set_last_error("domino_tensor_peak: " + msg);
  return st;
}

std::mutex g_peak_mutex;
int g_peak_clusters[64] = {};  // co-resident 2-CTA clusters per device (0: not yet asked)

}  // namespace

extern "C" {

domino_status_t domino_tensor_peak(int64_t mmas_per_cluster, int32_t clusters, void* workspace,
                                   size_t workspace_bytes, uint64_t timeout_ns, void* stream,
                                   domino_tensor_peak_t* out) {
  if (!workspace || !out) return peak_fail(DOMINO_ERR_INVALID_ARG, "workspace and out must be non-NULL");
  if (mmas_per_cluster < 1 || mmas_per_cluster > DOMINO_TENSOR_PEAK_MAX_MMAS)
    return peak_fail(DOMINO_ERR_INVALID_ARG, "mmas_per_cluster must be in 1..DOMINO_TENSOR_PEAK_MAX_MMAS");
  if (workspace_bytes < DOMINO_TENSOR_PEAK_WS_BYTES)
    return peak_fail(DOMINO_ERR_WORKSPACE, "workspace smaller than DOMINO_TENSOR_PEAK_WS_BYTES");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return peak_fail(DOMINO_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (timeout_ns == 0) timeout_ns = 5000000000ull;

  int dev = 0, major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return peak_fail(DOMINO_ERR_CUDA, std::string("device query: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return peak_fail(DOMINO_ERR_DEVICE, "device ordinal out of range");
  if (major != 10 || minor != 3) {
    char buf[96];
    snprintf(buf, sizeof buf, "device %d is sm_%d%d, not sm_103 (GB300)", dev, major, minor);
    return peak_fail(DOMINO_ERR_DEVICE, buf);
  }
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(g_peak_mutex);
    if (g_peak_clusters[dev] == 0) {
      e = cudaFuncSetAttribute(domino::tensor_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kPeakSmemBytes);
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(kPeakThreads, 1, 1);
      cfg.dynamicSmemBytes = kPeakSmemBytes;
      int n = 0;
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, domino::tensor_peak_kernel, &cfg);
      if (e != cudaSuccess) return peak_fail(DOMINO_ERR_CUDA, std::string("setup: ") + cudaGetErrorString(e));
      if (n < 1) return peak_fail(DOMINO_ERR_UNSUPPORTED, "no 2-CTA cluster of the probe fits on this device");
      g_peak_clusters[dev] = n;
    }
    max_clusters = g_peak_clusters[dev];
  }
  if (clusters <= 0) clusters = max_clusters;
  if (clusters > max_clusters)
    return peak_fail(DOMINO_ERR_UNSUPPORTED, "more clusters than can be co-resident");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + kPeakClockOff, 0, 16, s);
  if (e == cudaSuccess) e = cudaEventRecord(e0, s);
  if (e == cudaSuccess) {
    void* args[] = {&mmas_per_cluster, &ws, &timeout_ns};
    e = cudaLaunchKernel(reinterpret_cast<const void*>(&domino::tensor_peak_kernel), dim3(2 * clusters),
                         dim3(kPeakThreads), args, kPeakSmemBytes, s);
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  domino::DeviceStatus status = {};
  uint64_t clk[2] = {0, 0};
  if (e == cudaSuccess) e = cudaMemcpy(&status, ws, sizeof status, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(clk, ws + kPeakClockOff, sizeof clk, cudaMemcpyDeviceToHost);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return peak_fail(DOMINO_ERR_CUDA, cudaGetErrorString(e));
  if (status.code != 0) return peak_fail(DOMINO_ERR_TIMEOUT, "the wait for the MMAs gave up");

  const double per_cluster = 2.0 * 256 * domino::kBN * 16 * static_cast<double>(mmas_per_cluster);
  out->ms = ms;
  out->flops = per_cluster * clusters;
  out->tflops = ms > 0.0f ? out->flops / (ms * 1e-3) / 1e12 : 0.0;
  out->sm_mhz = clk[1] ? static_cast<double>(clk[0]) / static_cast<double>(clk[1]) * 1e3 : 0.0;
  out->flops_per_clk_sm = clk[0] ? per_cluster / static_cast<double>(clk[0]) / 2.0 : 0.0;
  out->clusters = clusters;
  out->num_sms = sms;
  return DOMINO_OK;
}

}  // extern "C"
