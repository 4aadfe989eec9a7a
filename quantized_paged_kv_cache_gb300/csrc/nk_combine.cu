// nk_combine.cu -- log-sum-exp merge of split-KV partial attention results.
//
// Partial s of a row holds O_s normalized by its own softmax sum and
// LSE_s = ln(sum_n exp(score_n)) over its keys. The merged row is
//   O = sum_s exp(LSE_s - M) O_s / sum_s exp(LSE_s - M),  M = max_s LSE_s,
// with empty partials (LSE = -inf) weighted 0.
//
// One warp per (row, 128-channel slice). The lanes first read the S LSE values
// in parallel (max and weights by warp shuffles, weights kept in shared
// memory), then walk the partials with four independent vector loads in
// flight per lane, so the merge is bound by L2/HBM bandwidth rather than by
// one dependent load per partial.
#include "nk_decode.cuh"

namespace nk {

constexpr int kCombWarps = 8;
constexpr int kWtsPerWarp = 512;  // weights kept in shared memory; more partials recompute theirs

// lse_of(s): LSE of partial s (-inf to skip it); row_of(s): its fp32 row slice.
template <int CPL, class LseFn, class RowFn>
__device__ __forceinline__ void merge_slice(int S, LseFn lse_of, RowFn row_of, int lane, float* wts,
                                            uint16_t* out_slice) {
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lse_of(s));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = lane; s < S; s += 32) {
      const float ls = lse_of(s);
      const float w = (ls == -INFINITY) ? 0.f : expf(ls - mx);
      if (s < kWtsPerWarp) wts[s] = w;
      wsum += w;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  __syncwarp();
  float acc[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) acc[j] = 0.f;
  if (mx != -INFINITY) {
    auto weight = [&](int s) {
      if (s < kWtsPerWarp) return wts[s];
      const float ls = lse_of(s);
      return ls == -INFINITY ? 0.f : expf(ls - mx);
    };
    int s = 0;
    for (; s + 4 <= S; s += 4) {
      float w[4];
      float v[4][CPL];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        w[u] = weight(s + u);
        const float* src = row_of(s + u) + lane * CPL;
        if constexpr (CPL == 4) {
          const float4 f = (w[u] != 0.f) ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[u][0] = f.x;
          v[u][1] = f.y;
          v[u][2] = f.z;
          v[u][3] = f.w;
        } else {
          const float2 f = (w[u] != 0.f) ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
          v[u][0] = f.x;
          v[u][1] = f.y;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < CPL; ++j) acc[j] = fmaf(w[u], v[u][j], acc[j]);
    }
    for (; s < S; ++s) {
      const float w = weight(s);
      if (w == 0.f) continue;
      const float* src = row_of(s) + lane * CPL;
#pragma unroll
      for (int j = 0; j < CPL; ++j) acc[j] = fmaf(w, src[j], acc[j]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int j = 0; j < CPL; j += 2) {
    const uint32_t lo = f32_to_bf16(acc[j] * inv), hi = f32_to_bf16(acc[j + 1] * inv);
    *reinterpret_cast<uint32_t*>(out_slice + lane * CPL + j) = lo | (hi << 16);
  }
}

// Combine for the decode kernels: units whose pages sit in one CTA were
// written directly by that CTA; the others merge the partial slots c + u of
// the CTAs c their pages span (CTAs with an empty range wrote nothing).
template <int CPL>
__global__ void __launch_bounds__(kCombWarps * 32) decode_combine_kernel(const DecodeParams p) {
  __shared__ int pre[kMaxBatch + 1];
  __shared__ int warp_tot[8];
  __shared__ float wts_all[kCombWarps][kWtsPerWarp];
  const SplitShape sh = p.shape();
  block_page_prefix(sh, p.ctx, pre, warp_tot);
  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  const int M = p.G * p.T, D = p.D;
  const int slices = D / (CPL * 32);
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t gw = (int64_t)blockIdx.x * kCombWarps + wib;
  if (gw >= (int64_t)p.B * p.Hkv * M * slices || W == 0) return;
  const int slice = (int)(gw % slices);
  const int64_t ur = gw / slices;
  const int u = (int)(ur / M), r = (int)(ur % M);
  const int b = u / p.Hkv, h = u % p.Hkv;
  const int pages = pre[b + 1] - pre[b];
  if (pages == 0) return;
  const int64_t x0 = (int64_t)pre[b] * p.Hkv + (int64_t)h * pages;
  const int c0 = cta_of_item(W, p.n_ctas, x0);
  const int c1 = cta_of_item(W, p.n_ctas, x0 + pages - 1);
  if (c0 == c1) return;
  const int n = p.n_ctas;
  auto lse_of = [&](int s) {
    const int c = c0 + s;
    if (cta_begin(W, n, c) == cta_begin(W, n, c + 1)) return -INFINITY;
    return p.part_lse[((int64_t)c + u) * M + r];
  };
  auto row_of = [&](int s) { return p.part_o + (((int64_t)c0 + s + u) * M + r) * D + slice * CPL * 32; };
  const int t = r / p.G, hg = r % p.G;
  uint16_t* orow = p.out + (((int64_t)b * p.T + t) * p.Hq + h * p.G + hg) * D + slice * CPL * 32;
  merge_slice<CPL>(c1 - c0 + 1, lse_of, row_of, lane, wts_all[wib], orow);
}

// Standalone combine: part_o [S][R][D], part_lse [S][R] -> out [R][D].
template <int CPL>
__global__ void __launch_bounds__(kCombWarps * 32) attn_combine_kernel(const float* part_o, const float* part_lse,
                                                                     int S, int R, int D, uint16_t* out) {
  __shared__ float wts_all[kCombWarps][kWtsPerWarp];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int slices = D / (CPL * 32);
  const int64_t gw = (int64_t)blockIdx.x * kCombWarps + wib;
  if (gw >= (int64_t)R * slices) return;
  const int slice = (int)(gw % slices);
  const int64_t row = gw / slices;
  auto lse_of = [&](int s) { return part_lse[(int64_t)s * R + row]; };
  auto row_of = [&](int s) { return part_o + ((int64_t)s * R + row) * D + slice * CPL * 32; };
  merge_slice<CPL>(S, lse_of, row_of, lane, wts_all[wib], out + row * D + slice * CPL * 32);
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const int cpl = p.D >= 128 ? 4 : 2;
  const int64_t warps = (int64_t)p.B * p.Hkv * p.G * p.T * (p.D / (cpl * 32));
  const int64_t grid = (warps + kCombWarps - 1) / kCombWarps;
  if (grid == 0) return cudaSuccess;
  if (cpl == 4) decode_combine_kernel<4><<<(unsigned)grid, kCombWarps * 32, 0, stream>>>(p);
  else decode_combine_kernel<2><<<(unsigned)grid, kCombWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_combine(const float* part_o, const float* part_lse, int S, int R, int D, uint16_t* out,
                                cudaStream_t stream) {
  const int cpl = D >= 128 ? 4 : 2;
  const int64_t warps = (int64_t)R * (D / (cpl * 32));
  const int64_t grid = (warps + kCombWarps - 1) / kCombWarps;
  if (grid == 0) return cudaSuccess;
  if (cpl == 4)
    attn_combine_kernel<4><<<(unsigned)grid, kCombWarps * 32, 0, stream>>>(part_o, part_lse, S, R, D, out);
  else
    attn_combine_kernel<2><<<(unsigned)grid, kCombWarps * 32, 0, stream>>>(part_o, part_lse, S, R, D, out);
  return cudaGetLastError();
}

}  // namespace nk
