// The shard-sum: Y = sum over the P tensor-parallel shards of their partial
// outputs.  On P GPUs this is the all-reduce of the row-parallel projection
// (Megatron-LM MLP); Domino (page "Domino: Eliminating Communication in LLM
// Training via Generic Tensor Slicing and Overlapping", Abstract) hides it
// behind the next piece's computation.  Here the shards are buffers on one GPU
// and the exchange becomes this memory-bound kernel: it reads P partials and
// writes one bf16 output, nothing else.
//
// Each thread handles 8 consecutive elements per step: one 16-byte load per
// bf16 partial (two per fp32 partial), all P loads issued before the adds,
// fp32 accumulation in shard order p = 0..P-1, one round-to-nearest-even to
// bf16 and one 16-byte store.  Partials are read once, so loads stream past L1
// without L1 allocation.  Grid: a multiple of the SM count, grid-stride.
#include <cuda_bf16.h>

#include <string>

#include "gemm.h"
#include "ptx.cuh"

namespace domino {

namespace {

__device__ __forceinline__ uint4 ld_stream_u4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] += __uint_as_float(w[q] << 16);
    acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void add_f32x4(float* acc, uint4 v) {
  acc[0] += __uint_as_float(v.x);
  acc[1] += __uint_as_float(v.y);
  acc[2] += __uint_as_float(v.z);
  acc[3] += __uint_as_float(v.w);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// NP > 0: P fixed at compile time; NP == 0: runtime P (<= kMaxShards).
template <int NP, bool F32>
__global__ void __launch_bounds__(256) shard_sum_kernel(const __grid_constant__ ShardSumParams p) {
  grid_dependency_wait();  // launched as a dependent of the stream's previous kernel
  const int P = NP > 0 ? NP : p.P;
  const uint32_t vec_per_row = static_cast<uint32_t>(p.cols / 8);
  const uint32_t nvec = static_cast<uint32_t>(p.rows) * vec_per_row;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const uint32_t r = v / vec_per_row;
    const uint32_t c8 = v - r * vec_per_row;
    const int64_t off = static_cast<int64_t>(r) * p.ld_part + static_cast<int64_t>(c8) * 8;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    if constexpr (F32) {
      constexpr int kMax = NP > 0 ? NP : kMaxShards;
      uint4 lo[kMax], hi[kMax];
#pragma unroll
      for (int s = 0; s < kMax; ++s) {
        if (s < P) {
          const float* src = static_cast<const float*>(p.part[s]) + off;
          lo[s] = ld_stream_u4(src);
          hi[s] = ld_stream_u4(src + 4);
        }
      }
#pragma unroll
      for (int s = 0; s < kMax; ++s) {
        if (s < P) {
          add_f32x4(acc, lo[s]);
          add_f32x4(acc + 4, hi[s]);
        }
      }
    } else {
      constexpr int kMax = NP > 0 ? NP : kMaxShards;
      uint4 x[kMax];
#pragma unroll
      for (int s = 0; s < kMax; ++s)
        if (s < P) x[s] = ld_stream_u4(static_cast<const __nv_bfloat16*>(p.part[s]) + off);
#pragma unroll
      for (int s = 0; s < kMax; ++s)
        if (s < P) add_bf16x8(acc, x[s]);
    }
    uint4 out;
    out.x = pack2(acc[0], acc[1]);
    out.y = pack2(acc[2], acc[3]);
    out.z = pack2(acc[4], acc[5]);
    out.w = pack2(acc[6], acc[7]);
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.y) + static_cast<int64_t>(r) * p.ld_y + c8 * 8;
    *reinterpret_cast<uint4*>(dst) = out;
  }
}

template <bool F32>
void* pick(int P) {
  switch (P) {
    case 1: return reinterpret_cast<void*>(&shard_sum_kernel<1, F32>);
    case 2: return reinterpret_cast<void*>(&shard_sum_kernel<2, F32>);
    case 4: return reinterpret_cast<void*>(&shard_sum_kernel<4, F32>);
    case 8: return reinterpret_cast<void*>(&shard_sum_kernel<8, F32>);
    default: return reinterpret_cast<void*>(&shard_sum_kernel<0, F32>);
  }
}

// One warp waits for a flag word (header offset 32) that nothing sets, through
// the same bounded-wait pattern as the kernels' inter-CTA waits.
__global__ void selftest_wait_kernel(DeviceStatus* st, const uint32_t* flag, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v != 0) return;
    if (globaltimer_ns() - t0 > timeout_ns) {
      if (threadIdx.x == 0) record_error(st, kStatusTimeout, kSiteSelfTest, 0);
      return;
    }
    __nanosleep(1000);
  }
}

}  // namespace

domino_status_t launch_selftest_wait(void* workspace, uint64_t timeout_ns, cudaStream_t stream, std::string* err) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t st = cudaMemsetAsync(ws + 32, 0, 4, stream);
  if (st == cudaSuccess) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<DeviceStatus*>(ws),
                                               reinterpret_cast<const uint32_t*>(ws + 32), timeout_ns);
    st = cudaGetLastError();
  }
  if (st != cudaSuccess) {
    if (err) *err = std::string("self-test launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

domino_status_t launch_shard_sum(const ShardSumParams& p, int num_sms, cudaStream_t stream, std::string* err) {
  const int64_t nvec = p.rows * (p.cols / 8);
  if (nvec == 0) return DOMINO_OK;
  if (nvec >= (int64_t(1) << 32)) {
    if (err) *err = "shard_sum: more than 2^32 vectors";
    return DOMINO_ERR_UNSUPPORTED;
  }
  constexpr int kThreads = 256;
  const int64_t want = (nvec + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 x 256 threads = a full SM
  const int grid = static_cast<int>(want < cap ? want : cap);
  void* fn = p.f32 ? pick<true>(p.P) : pick<false>(p.P);
  ShardSumParams q = p;
  void* args[] = {&q};
  cudaError_t st = launch_after_previous(fn, dim3(grid), dim3(kThreads), 0, stream, args);
  if (st != cudaSuccess) {
    if (err) *err = std::string("shard_sum launch: ") + cudaGetErrorString(st);
    return DOMINO_ERR_CUDA;
  }
  return DOMINO_OK;
}

}  // namespace domino
