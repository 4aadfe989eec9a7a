// nk_rk8v4.cuh -- the rk8v4 KV format ("NInfer-3090" README, "RotorQuant KV
// (rk8v4)"): keys rotated by the 64-point Hadamard transform and stored as
// INT8 group-64 codes, values unrotated as signed 4-bit codes (15 levels, two
// per byte) with one scale per 32 channels, every scale fp16.
#pragma once

#include "nk_decode.cuh"

namespace nk {

constexpr int kRkVGroup = 32;  // value channels per scale

// Byte offsets inside one rk8v4 (page, kv-head) chunk, in ChunkLayout's fields:
//   Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D/2] (channel 2j in the low
//   nibble of byte j, 2j + 1 in the high one) | Vs[P][D/32] fp16
__host__ __device__ inline ChunkLayout rk8v4_layout(int P, int D) {
  ChunkLayout c;
  c.ks = (int64_t)P * D;
  c.vc = c.ks + (int64_t)P * (D / kGroup) * 2;
  c.vs = c.vc + (int64_t)P * (D / 2);
  c.chunk = c.vs + (int64_t)P * (D / kRkVGroup) * 2;
  return c;
}

cudaError_t launch_rk8v4_append(int sms, const nk_kv_pool& pool, const int32_t* bt, int max_pages,
                                const int32_t* start_pos, const int32_t* cu_new, int B, int total_new, const void* k,
                                const void* v, int32_t* status, cudaStream_t stream);
cudaError_t launch_decode_rk8v4(const DecodeParams& p, cudaStream_t stream);
int decode_rk8v4_ctas_per_sm(int D, int G);

}  // namespace nk
