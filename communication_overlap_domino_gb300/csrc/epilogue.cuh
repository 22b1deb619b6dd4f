// Epilogue device code shared by the grouped GEMM (gemm.cu) and the fused
// forward kernel (fused.cu): activations and their derivatives, bf16/fp32 row
// stores and loads, and the drain of one 128 x 256 fp32 accumulator tile from
// tensor memory (each epilogue thread owns one accumulator row).
#pragma once

#include <cuda_bf16.h>

#include "common.h"
#include "ptx.cuh"

namespace domino {

// Where one tile's epilogue writes (and, for the backward, reads).
struct EpiArgs {
  void* out;          // output matrix of this shard
  void* aux;          // saved pre-activations (written by GEMM1, read by the backward dH epilogue) or null
  int64_t ldo;        // leading dimension of out (elements)
  int64_t ld_aux;     // leading dimension of aux (elements)
  int64_t aux_u_off;  // SwiGLU: column offset of u inside aux
  int64_t out_u_off;  // SwiGLU backward: column offset of du inside out
  int32_t rows;       // valid accumulator rows (tile rows >= rows are not stored)
  int32_t out_row0;   // output row of accumulator row 0 of tile row-block 0
  int32_t n_end;      // output columns >= n_end are not stored
  const CUtensorMap* out_map;  // TMA store map of `out` (box 32 x 32), or null: direct stores
  uint8_t* stage;              // this warp's two 4 KB staging buffers (1024-byte aligned)
};

// ------------------------------------------------------------------ epilogue

// erf from Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: for z >= 0, erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5)
// exp(-z^2) with t = 1 / (1 + p z), absolute error <= 1.5e-7; odd in z.  One
// fast reciprocal and one fast exponential per value: cheaper in the epilogue
// than the library erff, and far inside the bf16 rounding of H.
__device__ __forceinline__ float erf_as(float z) {
  const float az = fabsf(z);
  const float t = __fdividef(1.0f, fmaf(0.3275911f, az, 1.0f));
  float poly = fmaf(t, 1.061405429f, -1.453152027f);
  poly = fmaf(t, poly, 1.421413741f);
  poly = fmaf(t, poly, -0.284496736f);
  poly = fmaf(t, poly, 0.254829592f);
  poly *= t;
  return copysignf(fmaf(-poly, __expf(-az * az), 1.0f), z);
}

__device__ __forceinline__ float gelu_erf(float x) { return 0.5f * x * (1.0f + erf_as(x * 0.70710678118654752f)); }
// gelu_erf of two values with the fp32 pair instructions: the same operations in the same order, so the
// results equal gelu_erf's; the reciprocal and the exponential stay per value.
__device__ __forceinline__ void gelu_erf2(float& h0, float& h1, float x0, float x1) {
  float z0, z1, d0, d1, p0, p1, q0, q1, s0, s1, r0, r1;
  mul2(z0, z1, x0, x1, 0.70710678118654752f, 0.70710678118654752f);
  const float a0 = fabsf(z0), a1 = fabsf(z1);
  fma2(d0, d1, 0.3275911f, 0.3275911f, a0, a1, 1.0f, 1.0f);
  const float t0 = __fdividef(1.0f, d0), t1 = __fdividef(1.0f, d1);
  fma2(p0, p1, t0, t1, 1.061405429f, 1.061405429f, -1.453152027f, -1.453152027f);
  fma2(p0, p1, t0, t1, p0, p1, 1.421413741f, 1.421413741f);
  fma2(p0, p1, t0, t1, p0, p1, -0.284496736f, -0.284496736f);
  fma2(p0, p1, t0, t1, p0, p1, 0.254829592f, 0.254829592f);
  mul2(p0, p1, p0, p1, t0, t1);
  mul2(s0, s1, -a0, -a1, a0, a1);
  fma2(r0, r1, -p0, -p1, __expf(s0), __expf(s1), 1.0f, 1.0f);
  add2(q0, q1, 1.0f, 1.0f, copysignf(r0, z0), copysignf(r1, z1));
  mul2(h0, h1, 0.5f, 0.5f, x0, x1);
  mul2(h0, h1, h0, h1, q0, q1);
}
__device__ __forceinline__ float gelu_tanh(float x) {
  return 0.5f * x * (1.0f + tanhf(0.79788456080286536f * (x + 0.044715f * x * x * x)));
}
// The logistic function of two values with the fp32 pair instructions, from exp(-x) = 2^(-x log2 e): the
// scaling and the 1 + e go two at a time, the exponential (ex2.approx) and the fast reciprocal stay per
// value (far inside the bf16 rounding of the results).  As x -> -inf, 2^(-x log2 e) overflows to inf and the
// quotient goes to 0.
__device__ __forceinline__ void sigmoid2(float& s0, float& s1, float x0, float x1) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  float a0, a1, d0, d1;
  mul2(a0, a1, x0, x1, kNegLog2e, kNegLog2e);
  add2(d0, d1, ex2_approx(a0), ex2_approx(a1), 1.0f, 1.0f);
  s0 = __fdividef(1.0f, d0);
  s1 = __fdividef(1.0f, d1);
}

// SwiGLU of two (gate, up) pairs: h = silu(g) u = (g sigmoid(g)) u.
__device__ __forceinline__ void swiglu2(float& h0, float& h1, float g0, float g1, float u0, float u1) {
  float s0, s1;
  sigmoid2(s0, s1, g0, g1);
  mul2(s0, s1, s0, s1, g0, g1);
  mul2(h0, h1, s0, s1, u0, u1);
}

// The SwiGLU backward of two (gate, up) pairs, with s = sigmoid(g):
// du = dH silu(g) = (dH g) s and dg = dH u silu'(g) = ((dH u) s)(1 + g (1 - s)).
__device__ __forceinline__ void swiglu_grad2(float& dg0, float& dg1, float& du0, float& du1, float dh0, float dh1,
                                             float g0, float g1, float u0, float u1) {
  float s0, s1, t0, t1, v0, v1, w0, w1;
  sigmoid2(s0, s1, g0, g1);
  mul2(t0, t1, dh0, dh1, g0, g1);
  mul2(du0, du1, t0, t1, s0, s1);
  mul2(v0, v1, dh0, dh1, u0, u1);
  mul2(v0, v1, v0, v1, s0, s1);
  add2(w0, w1, 1.0f, 1.0f, -s0, -s1);
  fma2(w0, w1, g0, g1, w0, w1, 1.0f, 1.0f);
  mul2(dg0, dg1, v0, v1, w0, w1);
}

// Derivatives for the backward epilogue (product and chain rules).
__device__ __forceinline__ float gelu_erf_grad(float x) {
  // d/dx [x Phi(x)] = Phi(x) + x phi(x)
  return 0.5f * (1.0f + erf_as(x * 0.70710678118654752f)) + x * 0.39894228040143268f * __expf(-0.5f * x * x);
}
__device__ __forceinline__ float gelu_tanh_grad(float x) {
  const float k = 0.79788456080286536f;
  const float t = tanhf(k * (x + 0.044715f * x * x * x));
  return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * k * (1.0f + 3.0f * 0.044715f * x * x);
}

template <int EPI>
__device__ __forceinline__ float activate_grad(float x) {
  if constexpr (EPI == EPI_DG_GELU) return gelu_erf_grad(x);
  else if constexpr (EPI == EPI_DG_GELU_TANH) return gelu_tanh_grad(x);
  else return 1.0f;
}

__host__ __device__ constexpr bool is_dg(int epi) { return epi >= EPI_DG_GELU && epi <= EPI_DG_SWIGLU; }

template <int EPI>
__device__ __forceinline__ float activate(float x) {
  if constexpr (EPI == EPI_H_GELU) return gelu_erf(x);
  else if constexpr (EPI == EPI_H_GELU_TANH) return gelu_tanh(x);
  else return x;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Stores v[0..n) (n <= 32) as bf16 at dst (16-byte aligned when n == 32).
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float (&v)[32], int n) {
  if (n >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
      d4[q] = w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) dst[j] = __float2bfloat16_rn(v[j]);
  }
}

// Loads n <= 32 bf16 values from src (16-byte aligned when n == 32) as floats.
__device__ __forceinline__ void load_row_bf16(const __nv_bfloat16* src, float (&v)[32], int n) {
  if (n >= 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = s4[q];
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[8 * q + 2 * e] = __uint_as_float(ww[e] << 16);
        v[8 * q + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = j < n ? __bfloat162float(src[j]) : 0.0f;
  }
}

__device__ __forceinline__ void store_row_f32(float* dst, const float (&v)[32], int n) {
  if (n >= 32) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) dst[j] = v[j];
  }
}

// Writes one 32-row x 32-column chunk (this lane: row `lane`, values v) through
// shared memory and a TMA store at output coordinates (x, y).  The staging
// layout is the store map's swizzle: 128-byte rows (fp32) with the 128-byte
// swizzle, or 64-byte rows (bf16, the backward dG outputs) with the 64-byte
// swizzle, so the 16-byte writes of a warp spread over all banks.  Two buffers alternate; before one is
// rewritten, lane 0 waits until the store that last read it is done reading.  kEvictFirst marks the written
// lines first for eviction from L2 (the backward dG outputs, which no later step of the same launch reads), so
// they do not push out the operands that the launch's other tiles read again.
template <bool F32, bool kEvictFirst = false>
__device__ __forceinline__ void stage_and_store(const EpiArgs& e, const float (&v)[32], int lane, int& sbuf,
                                                int32_t x, int32_t y) {
  uint8_t* buf = e.stage + (sbuf & 1) * 4096;
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  if constexpr (F32) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 w = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                 __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
      *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
      w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
      w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
      w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
      *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = w;
    }
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    if constexpr (kEvictFirst) tma_store_2d_hint(e.out_map, buf, x, y, l2_policy_evict_first());
    else tma_store_2d(e.out_map, buf, x, y);
    bulk_commit_group();
  }
  ++sbuf;
}

// Writes one 32-row x 64-column bf16 chunk (this lane: row `lane`, columns
// v0 then v1) through shared memory and a TMA store at (x, y): 128-byte rows
// with the 128-byte swizzle, two alternating 4 KB buffers per warp.
__device__ __forceinline__ void stage_and_store_bf16x64(const EpiArgs& e, const float (&v0)[32],
                                                        const float (&v1)[32], int lane, int& sbuf, int32_t x,
                                                        int32_t y) {
  uint8_t* buf = e.stage + (sbuf & 1) * 4096;
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float* v = j < 4 ? v0 : v1;
    const int q = j & 3;
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(e.out_map, buf, x, y);
    bulk_commit_group();
  }
  ++sbuf;
}

// One 32-column chunk of the accumulator row: tensor-memory load, the saved
// pre-activations (when e.aux is set) and the activation.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const EpiArgs& e, uint32_t tacc, int c, int col, int n, bool row_ok,
                                               int64_t orow, float (&h)[32]) {
  uint32_t r0[32];
  tmem_ld_32x32b_x32(tacc + c * 32, r0);
  if constexpr (EPI == EPI_H_SWIGLU) {
    uint32_t r1[32];
    tmem_ld_32x32b_x32(tacc + kBN / 2 + c * 32, r1);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; j += 2)
      swiglu2(h[j], h[j + 1], __uint_as_float(r0[j]), __uint_as_float(r0[j + 1]), __uint_as_float(r1[j]),
              __uint_as_float(r1[j + 1]));
    if (row_ok && e.aux != nullptr) {
      float g[32], u[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        g[j] = __uint_as_float(r0[j]);
        u[j] = __uint_as_float(r1[j]);
      }
      __nv_bfloat16* a = static_cast<__nv_bfloat16*>(e.aux) + orow * e.ld_aux + col;
      store_row_bf16(a, g, n);
      store_row_bf16(a + e.aux_u_off, u, n);
    }
  } else {
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) h[j] = __uint_as_float(r0[j]);
    if constexpr (EPI != EPI_Z_F32 && EPI != EPI_Z_BF16) {
      if (row_ok && e.aux != nullptr)
        store_row_bf16(static_cast<__nv_bfloat16*>(e.aux) + orow * e.ld_aux + col, h, n);
      if constexpr (EPI == EPI_H_GELU) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) gelu_erf2(h[j], h[j + 1], h[j], h[j + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] = activate<EPI>(h[j]);
      }
    }
  }
}

// Drains one 128 x 256 accumulator tile (this thread: one row) through the
// epilogue.  fp32 outputs go out in 32 x 32 chunks, bf16 outputs in 32 x 64
// chunks (128-byte rows either way); full chunks inside the valid rows and
// columns go through shared memory and TMA stores when e.out_map is set, edge
// chunks (and the saved pre-activations) use direct stores.  sbuf: the warp's
// staging buffer counter.
template <int EPI>
__device__ __forceinline__ void epilogue_tile(const EpiArgs& e, uint32_t tacc, int mb, int col0, int row_in_tile,
                                              int& sbuf) {
  const int lane = row_in_tile & 31;
  const int64_t grow = static_cast<int64_t>(mb) * kBM + row_in_tile;
  const bool row_ok = grow < e.rows;
  const int64_t orow = e.out_row0 + grow;
  const int64_t warp_row0 = static_cast<int64_t>(mb) * kBM + (row_in_tile & ~31);
  const bool warp_rows_full = warp_row0 + 32 <= e.rows;  // uniform across the warp
  const int32_t y = static_cast<int32_t>(e.out_row0 + warp_row0);
  constexpr int kChunks = (EPI == EPI_H_SWIGLU) ? (kBN / 2) / 32 : kBN / 32;
  if constexpr (EPI == EPI_Z_F32) {
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c) {
      const int col = col0 + c * 32;
      if (col >= e.n_end) break;  // uniform across the warp
      const int n = e.n_end - col;
      float h[32];
      epilogue_chunk<EPI>(e, tacc, c, col, n, row_ok, orow, h);
      if (e.out_map != nullptr && warp_rows_full && n >= 32)
        stage_and_store<true>(e, h, lane, sbuf, col, y);
      else if (row_ok)
        store_row_f32(static_cast<float*>(e.out) + orow * e.ldo + col, h, n);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < kChunks; c += 2) {
      const int col = col0 + c * 32;
      if (col >= e.n_end) break;  // uniform across the warp
      const int n = e.n_end - col;
      float h0[32], h1[32];
      epilogue_chunk<EPI>(e, tacc, c, col, n, row_ok, orow, h0);
      if (n > 32) epilogue_chunk<EPI>(e, tacc, c + 1, col + 32, n - 32, row_ok, orow, h1);
      if (e.out_map != nullptr && warp_rows_full && n >= 64) {
        stage_and_store_bf16x64(e, h0, h1, lane, sbuf, col, y);
      } else if (row_ok) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(e.out) + orow * e.ldo + col;
        store_row_bf16(o, h0, n);
        if (n > 32) store_row_bf16(o + 32, h1, n - 32);
      }
    }
  }
}

__device__ __forceinline__ void unpack_bf16x32(const uint4 (&q)[4], float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * i + 2 * e] = __uint_as_float(w[e] << 16);
      v[8 * i + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
}

// Backward dH epilogue: dG = dH * act'(g) (SwiGLU: dg and du), with the saved
// pre-activations of the next 32-column chunk loaded while the current chunk
// is computed, so their load latency overlaps the tensor-memory reads and math.
template <int EPI>
__device__ __forceinline__ void epilogue_tile_dg(const EpiArgs& e, uint32_t tacc, int mb, int col0,
                                                 int row_in_tile, int& sbuf) {
  const int lane = row_in_tile & 31;
  const int64_t warp_row0 = static_cast<int64_t>(mb) * kBM + (row_in_tile & ~31);
  const bool warp_rows_full = warp_row0 + 32 <= e.rows;  // uniform across the warp
  constexpr bool kSwiglu = EPI == EPI_DG_SWIGLU;
  constexpr int kChunks = kBN / 32;
  const int64_t grow = static_cast<int64_t>(mb) * kBM + row_in_tile;
  const bool row_ok = grow < e.rows;
  const int64_t orow = e.out_row0 + grow;
  const __nv_bfloat16* pre_row = static_cast<const __nv_bfloat16*>(e.aux) + orow * e.ld_aux;
  __nv_bfloat16* dst_row = static_cast<__nv_bfloat16*>(e.out) + orow * e.ldo;
  uint4 gq[4], uq[4];
  auto prefetch = [&](int c) {
    const int col = col0 + c * 32;
    if (row_ok && col + 32 <= e.n_end) {
      const uint4* g4 = reinterpret_cast<const uint4*>(pre_row + col);
#pragma unroll
      for (int i = 0; i < 4; ++i) gq[i] = g4[i];
      if constexpr (kSwiglu) {
        const uint4* u4 = reinterpret_cast<const uint4*>(pre_row + e.aux_u_off + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) uq[i] = u4[i];
      }
    }
  };
  prefetch(0);
#pragma unroll 1
  for (int c = 0; c < kChunks; ++c) {
    const int col = col0 + c * 32;
    if (col >= e.n_end) break;  // uniform across the warp
    const int n = e.n_end - col;
    uint4 gc[4], uc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      gc[i] = gq[i];
      uc[i] = uq[i];
    }
    if (c + 1 < kChunks) prefetch(c + 1);
    uint32_t r0[32];
    tmem_ld_32x32b_x32(tacc + c * 32, r0);
    tmem_ld_wait();
    float g[32], u[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) g[j] = u[j] = 0.0f;
    if (row_ok) {
      if (n >= 32) {
        unpack_bf16x32(gc, g);
        if constexpr (kSwiglu) unpack_bf16x32(uc, u);
      } else {
        load_row_bf16(pre_row + col, g, n);
        if constexpr (kSwiglu) load_row_bf16(pre_row + e.aux_u_off + col, u, n);
      }
    }
    const bool tma = e.out_map != nullptr && warp_rows_full && n >= 32;  // uniform
    const int32_t y = static_cast<int32_t>(e.out_row0 + warp_row0);
    if constexpr (kSwiglu) {
      float dg[32], du[32];
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        swiglu_grad2(dg[j], dg[j + 1], du[j], du[j + 1], __uint_as_float(r0[j]), __uint_as_float(r0[j + 1]), g[j],
                     g[j + 1], u[j], u[j + 1]);
      if (tma) {
        stage_and_store<false, true>(e, dg, lane, sbuf, col, y);
        stage_and_store<false, true>(e, du, lane, sbuf, static_cast<int32_t>(e.out_u_off + col), y);
      } else if (row_ok) {
        store_row_bf16(dst_row + col, dg, n);
        store_row_bf16(dst_row + e.out_u_off + col, du, n);
      }
    } else {
      float dgv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) dgv[j] = __uint_as_float(r0[j]) * activate_grad<EPI>(g[j]);
      if (tma)
        stage_and_store<false, true>(e, dgv, lane, sbuf, col, y);
      else if (row_ok)
        store_row_bf16(dst_row + col, dgv, n);
    }
  }
}

}  // namespace domino
