// nk_combine.cu -- log-sum-exp merge of split-KV partial attention results.
//
// Partial s of a row holds O_s normalized by its own softmax sum and
// LSE_s = ln(sum_n exp(score_n)) over its keys. The merged row is
//   O = sum_s exp(LSE_s - M) O_s / sum_s exp(LSE_s - M),  M = max_s LSE_s,
// with empty partials (LSE = -inf) weighted 0. One warp per row; each lane
// owns D/32 channels (vectorized fp32 loads), the weights are recomputed by
// every lane from the S LSE values.
#include "nk_decode.cuh"

namespace nk {

// Merge S partials of one row. Partial s lives in slot slot0 + s; when
// `skip_empty` is set, slots of CTAs whose item range is empty (possible when
// there are more CTAs than page items) are left out: they were never written.
template <int CPL>
__device__ __forceinline__ void merge_row(const float* part_o, const float* part_lse, int64_t slot0,
                                          int64_t slot_stride_rows, int S, int64_t row, int D, int lane,
                                          uint16_t* out_row, int64_t W = 0, int n_ctas = 0, int c0 = 0) {
  auto skip = [&](int s) {
    return W > 0 && cta_begin(W, n_ctas, c0 + s) == cta_begin(W, n_ctas, c0 + s + 1);
  };
  float mx = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (!skip(s)) mx = fmaxf(mx, part_lse[(slot0 + s) * slot_stride_rows + row]);
  float acc[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) acc[j] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      if (skip(s)) continue;
      const float ls = part_lse[(slot0 + s) * slot_stride_rows + row];
      if (ls == -INFINITY) continue;
      const float wgt = expf(ls - mx);
      wsum += wgt;
      const float* src = part_o + ((slot0 + s) * slot_stride_rows + row) * D + lane * CPL;
      if constexpr (CPL % 4 == 0) {
#pragma unroll
        for (int j = 0; j < CPL; j += 4) {
          const float4 v = *reinterpret_cast<const float4*>(src + j);
          acc[j] = fmaf(wgt, v.x, acc[j]);
          acc[j + 1] = fmaf(wgt, v.y, acc[j + 1]);
          acc[j + 2] = fmaf(wgt, v.z, acc[j + 2]);
          acc[j + 3] = fmaf(wgt, v.w, acc[j + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < CPL; ++j) acc[j] = fmaf(wgt, src[j], acc[j]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int j = 0; j < CPL; j += 2) {
    const uint32_t lo = f32_to_bf16(acc[j] * inv), hi = f32_to_bf16(acc[j + 1] * inv);
    *reinterpret_cast<uint32_t*>(out_row + lane * CPL + j) = lo | (hi << 16);
  }
}

// Combine for the decode kernels: one warp per (unit, row); units whose
// pages sit in one CTA were already written by that CTA.
template <int CPL>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p) {
  __shared__ int pre[kMaxBatch + 1];
  __shared__ int warp_tot[8];
  const SplitShape sh = p.shape();
  block_page_prefix(sh, p.ctx, pre, warp_tot);
  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  const int M = p.G * p.T, D = CPL * 32;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= (int64_t)p.B * p.Hkv * M || W == 0) return;
  const int u = (int)(gw / M), r = (int)(gw % M);
  const int b = u / p.Hkv, h = u % p.Hkv;
  const int pages = pre[b + 1] - pre[b];
  if (pages == 0) return;
  const int64_t x0 = (int64_t)pre[b] * p.Hkv + (int64_t)h * pages;
  const int c0 = cta_of_item(W, p.n_ctas, x0);
  const int c1 = cta_of_item(W, p.n_ctas, x0 + pages - 1);
  if (c0 == c1) return;
  const int t = r / p.G, hg = r % p.G;
  uint16_t* orow = p.out + (((int64_t)b * p.T + t) * p.Hq + h * p.G + hg) * D;
  merge_row<CPL>(p.part_o, p.part_lse, (int64_t)c0 + u, M, c1 - c0 + 1, r, D, lane, orow, W, p.n_ctas, c0);
}

// Standalone combine: part_o [S][R][D], part_lse [S][R] -> out [R][D].
template <int CPL>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* part_o, const float* part_lse, int S, int R,
                                                         uint16_t* out) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= R) return;
  const int D = CPL * 32;
  merge_row<CPL>(part_o, part_lse, 0, R, S, row, D, lane, out + row * D);
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t warps = (int64_t)p.B * p.Hkv * p.G * p.T;
  const int64_t grid = (warps + 7) / 8;
  if (grid == 0) return cudaSuccess;
  if (p.D == 256) decode_combine_kernel<8><<<(unsigned)grid, 256, 0, stream>>>(p);
  else if (p.D == 128) decode_combine_kernel<4><<<(unsigned)grid, 256, 0, stream>>>(p);
  else decode_combine_kernel<2><<<(unsigned)grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_combine(const float* part_o, const float* part_lse, int S, int R, int D, uint16_t* out,
                                cudaStream_t stream) {
  const int64_t grid = ((int64_t)R + 7) / 8;
  if (grid == 0) return cudaSuccess;
  if (D == 256) attn_combine_kernel<8><<<(unsigned)grid, 256, 0, stream>>>(part_o, part_lse, S, R, out);
  else if (D == 128) attn_combine_kernel<4><<<(unsigned)grid, 256, 0, stream>>>(part_o, part_lse, S, R, out);
  else attn_combine_kernel<2><<<(unsigned)grid, 256, 0, stream>>>(part_o, part_lse, S, R, out);
  return cudaGetLastError();
}

}  // namespace nk
