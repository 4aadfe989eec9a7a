// nk_rk8v4.cuh -- the rk8v4 KV format ("NInfer-3090" README, "RotorQuant KV
// (rk8v4)"): keys rotated by the 64-point Hadamard transform and stored as
// INT8 group-64 codes, values unrotated as signed 4-bit codes (15 levels, two
// per byte) with one scale per 32 channels, every scale fp16.
#pragma once

#include "nk_decode.cuh"

namespace nk {

// The chunk layout (rk8v4_layout) and the value group width (kRkVGroup) are
// in nk_common.cuh with the other formats'.

cudaError_t launch_rk8v4_append(int sms, const nk_kv_pool& pool, const int32_t* bt, int max_pages,
                                const int32_t* start_pos, const int32_t* cu_new, int B, int total_new, const void* k,
                                const void* v, int32_t* status, cudaStream_t stream);
cudaError_t launch_decode_rk8v4(const DecodeParams& p, cudaStream_t stream);
int decode_rk8v4_ctas_per_sm(int D, int G);

}  // namespace nk
