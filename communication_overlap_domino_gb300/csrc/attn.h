// Host-side interface of the attention core (attn.cu), used by the C-ABI layer.
#pragma once

#include <string>

#include "common.h"
#include "gemm.h"

namespace domino {

// Kernel parameters: per shard p, the projected Q | K | V of its heads, QKV_p
// [M, 3 Hp dh] bf16 (query heads, then key heads, then value heads), read
// through two TMA maps, and the attention output O_p [M, Hp dh] bf16.
struct AttnParams {
  CUtensorMap map_qk[kMaxShards];  // QKV_p, box 64 columns x 128 rows, 128-byte swizzle (Q and K tiles)
  CUtensorMap map_v[kMaxShards];   // QKV_p, box 64 columns x 64 rows, 128-byte swizzle (V tiles, MN-major)
  void* o[kMaxShards];             // O_p
  int64_t ldo;                     // Hp * dh
  int32_t row0;                    // first row of the chunk
  int32_t S;                       // tokens per sequence (multiple of 128)
  int32_t Hp;                      // heads per shard
  int32_t seqs;                    // sequences in the chunk
  int32_t P;                       // shards
  int32_t nq;                      // 128-query tiles per sequence
  int32_t num_items;               // P * seqs * Hp * nq
  float scale_log2;                // log2(e) / sqrt(dh)
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// One launch: every (shard, sequence, head, query tile) of one chunk.
struct AttnLaunch {
  void* qkv[kMaxShards] = {};  // QKV_p [M, 3 Hp dh] bf16
  void* o[kMaxShards] = {};    // O_p [M, Hp dh] bf16
  int64_t M = 0;               // rows of QKV_p / O_p (all chunks)
  int64_t S = 0;               // tokens per sequence
  int32_t row0 = 0;            // first row of the chunk
  int32_t seqs = 0;            // sequences in the chunk
  int32_t Hp = 0, dh = 0, P = 0;
  DeviceStatus* status = nullptr;
  uint64_t timeout_ns = 0;
};

cudaError_t prepare_attn_kernel();
domino_status_t launch_attn_fwd(const AttnLaunch& L, int num_sms, cudaStream_t stream, std::string* err);

}  // namespace domino
