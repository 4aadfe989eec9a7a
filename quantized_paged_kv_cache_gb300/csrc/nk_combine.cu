// nk_combine.cu -- log-sum-exp merge of split-KV partial attention results.
//
// Partial s of a row holds O_s normalized by its own softmax sum and
// LSE_s = ln(sum_n exp(score_n)) over its keys. The merged row is
//   O = sum_s exp(LSE_s - M) O_s / sum_s exp(LSE_s - M),  M = max_s LSE_s,
// with empty partials (LSE = -inf) weighted 0.
//
// One 256-thread block per output row, or per 64-channel slice of a row when
// there are few rows. Thread t owns 4 channels (a float4) and every
// PL = 256 / (C / 4)-th partial (C = channels per block): it issues the loads
// of up to 8 of its partials (LSE and row slice) before using any, merges
// them online (running max, rescaled sum), and the PL partial-lanes of a
// channel group are merged by shuffles within a warp, then through shared
// memory. A row of S partials thus costs about S / (8 PL) dependent memory
// round trips instead of S / 4.
#include "nk_decode.cuh"

namespace nk {

constexpr int kCombThreads = 256;
constexpr int kCombUnroll = 8;

// lse_of(s): LSE of partial s (-inf: skip it); row_of(s): its fp32 row slice
// of D channels (the block's channels).
template <int D, class LseFn, class RowFn>
__device__ __forceinline__ void merge_row(int S, LseFn lse_of, RowFn row_of, uint16_t* out_row) {
  constexpr int CH = D / 4;               // float4 channel groups
  constexpr int PL = kCombThreads / CH;   // partial-lanes
  constexpr int LPW = CH < 32 ? 32 / CH : 1;  // partial-lanes of one channel group within a warp
  constexpr int PW = PL / LPW;            // partial-lanes left after the in-warp merge
  __shared__ float sm_m[PW][CH], sm_l[PW][CH];
  __shared__ float4 sm_o[PW][CH];
  const int t = threadIdx.x, pl = t / CH, ch = t % CH;
  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = pl; s0 < S; s0 += PL * kCombUnroll) {
    float ls[kCombUnroll];
    float4 v[kCombUnroll];
#pragma unroll
    for (int u = 0; u < kCombUnroll; ++u) {
      const int s = s0 + u * PL;
      ls[u] = -INFINITY;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s < S) {
        ls[u] = lse_of(s);
        v[u] = *reinterpret_cast<const float4*>(row_of(s) + ch * 4);  // read even if skipped: never used then
      }
    }
#pragma unroll
    for (int u = 0; u < kCombUnroll; ++u) {
      if (ls[u] == -INFINITY) continue;
      if (ls[u] > m) {
        const float a = expf(m - ls[u]);  // 0 while nothing was merged
        l *= a;
        acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
        m = ls[u];
      }
      const float w = expf(ls[u] - m);
      l += w;
      acc.x = fmaf(w, v[u].x, acc.x);
      acc.y = fmaf(w, v[u].y, acc.y);
      acc.z = fmaf(w, v[u].z, acc.z);
      acc.w = fmaf(w, v[u].w, acc.w);
    }
  }
  // the partial-lanes of a channel group that share a warp merge by shuffles
#pragma unroll
  for (int off = CH; off < 32; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off), lo = __shfl_xor_sync(0xffffffffu, l, off);
    float4 ao;
    ao.x = __shfl_xor_sync(0xffffffffu, acc.x, off);
    ao.y = __shfl_xor_sync(0xffffffffu, acc.y, off);
    ao.z = __shfl_xor_sync(0xffffffffu, acc.z, off);
    ao.w = __shfl_xor_sync(0xffffffffu, acc.w, off);
    const float mx = fmaxf(m, mo);
    const float a = m == -INFINITY ? 0.f : expf(m - mx), b = mo == -INFINITY ? 0.f : expf(mo - mx);
    l = l * a + lo * b;
    acc.x = fmaf(acc.x, a, ao.x * b);
    acc.y = fmaf(acc.y, a, ao.y * b);
    acc.z = fmaf(acc.z, a, ao.z * b);
    acc.w = fmaf(acc.w, a, ao.w * b);
    m = mx;
  }
  if (pl % LPW == 0) {
    sm_m[pl / LPW][ch] = m;
    sm_l[pl / LPW][ch] = l;
    sm_o[pl / LPW][ch] = acc;
  }
  __syncthreads();
  if (pl == 0) {
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < PW; ++q) mx = fmaxf(mx, sm_m[q][ch]);
    float lsum = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mx != -INFINITY) {
#pragma unroll
      for (int q = 0; q < PW; ++q) {
        const float mq = sm_m[q][ch];
        if (mq == -INFINITY) continue;
        const float a = expf(mq - mx);
        const float4 oq = sm_o[q][ch];
        lsum = fmaf(a, sm_l[q][ch], lsum);
        o.x = fmaf(a, oq.x, o.x);
        o.y = fmaf(a, oq.y, o.y);
        o.z = fmaf(a, oq.z, o.z);
        o.w = fmaf(a, oq.w, o.w);
      }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const uint32_t w0 = f32_to_bf16(o.x * inv) | ((uint32_t)f32_to_bf16(o.y * inv) << 16);
    const uint32_t w1 = f32_to_bf16(o.z * inv) | ((uint32_t)f32_to_bf16(o.w * inv) << 16);
    *reinterpret_cast<uint2*>(out_row + ch * 4) = make_uint2(w0, w1);
  }
}

// Combine for the decode kernels: units whose pages sit in one CTA were
// written directly by that CTA; the others merge the partial slots c + u of
// the CTAs c their pages span (CTAs with an empty range wrote nothing).
// Block = one (unit, row) and a slice of C channels.
template <int D, int C>
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(const DecodeParams p) {
  static_assert(D % C == 0, "whole slices");
  __shared__ int pre[kMaxBatch + 1];
  __shared__ int warp_tot[8];
  const SplitShape sh = p.shape();
  // The page prefix runs before the wait for the split kernel: this kernel
  // only ever follows the split kernel of the same call, which could start
  // only once its own predecessor had passed its wait (that predecessor is
  // the caller's previous kernel, or this call's append, which writes only
  // pool pages), so every kernel that could have written the context
  // lengths has completed; the split kernel only reads them. They are read
  // at L2 (the point of coherence), not through L1.
  block_page_prefix<true>(sh, p.ctx, p.trim, pre, warp_tot);
  chain_wait();
  chain_release();
  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  const int M = p.G * p.T;
  const int64_t ur = blockIdx.x / (D / C);
  const int c_off = (int)(blockIdx.x % (D / C)) * C;
  if (ur >= (int64_t)p.B * p.Hkv * M || W == 0) return;
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
    // a CTA can own no item only when there are fewer items than CTAs
    if (W < n && cta_begin(W, n, c) == cta_begin(W, n, c + 1)) return -INFINITY;
    return p.part_lse[((int64_t)c + u) * M + r];
  };
  auto row_of = [&](int s) { return p.part_o + (((int64_t)c0 + s + u) * M + r) * D + c_off; };
  const int t = r / p.G, hg = r % p.G;
  merge_row<C>(c1 - c0 + 1, lse_of, row_of, p.out + (((int64_t)b * p.qT + t) * p.Hq + h * p.G + hg) * D + c_off);
}

// Standalone combine: part_o [S][R][D], part_lse [S][R] -> out [R][D]; block = row.
template <int D>
__global__ void __launch_bounds__(kCombThreads) attn_combine_kernel(const float* part_o, const float* part_lse, int S,
                                                                  int R, uint16_t* out) {
  chain_wait();
  chain_release();
  const int64_t row = blockIdx.x;
  if (row >= R) return;
  auto lse_of = [&](int s) { return part_lse[(int64_t)s * R + row]; };
  auto row_of = [&](int s) { return part_o + ((int64_t)s * R + row) * D; };
  merge_row<D>(S, lse_of, row_of, out + row * D);
}

// Rows are split into 64-channel slices when there are fewer rows than
// kSliceRows: more blocks in flight, fewer partials per thread.
constexpr int kSliceRows = 256;

template <int D>
static cudaError_t launch_combine_d(const DecodeParams& p, int64_t rows, cudaStream_t stream) {
  const dim3 b(kCombThreads);
  if (D > 64 && rows < kSliceRows)
    return launch_chained(decode_combine_kernel<D, 64>, dim3((unsigned)(rows * (D / 64))), b, 0, stream, p);
  return launch_chained(decode_combine_kernel<D, D>, dim3((unsigned)rows), b, 0, stream, p);
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.Hkv * p.G * p.T;
  if (rows == 0) return cudaSuccess;
  if (p.D == 256) return launch_combine_d<256>(p, rows, stream);
  if (p.D == 128) return launch_combine_d<128>(p, rows, stream);
  return launch_combine_d<64>(p, rows, stream);
}

cudaError_t launch_attn_combine(const float* part_o, const float* part_lse, int S, int R, int D, uint16_t* out,
                                cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const dim3 g((unsigned)R), b(kCombThreads);
  if (D == 256) return launch_chained(attn_combine_kernel<256>, g, b, 0, stream, part_o, part_lse, S, R, out);
  if (D == 128) return launch_chained(attn_combine_kernel<128>, g, b, 0, stream, part_o, part_lse, S, R, out);
  return launch_chained(attn_combine_kernel<64>, g, b, 0, stream, part_o, part_lse, S, R, out);
}

}  // namespace nk
