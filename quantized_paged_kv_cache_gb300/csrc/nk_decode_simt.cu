// nk_decode_simt.cu -- split-KV paged attention on fp32 CUDA cores.
//
// The CUDA-core kernel the tensor-core path is measured against. Each CTA
// walks its segments of (sequence, kv-head, page) items; within a segment its
// warps split the pages and the T query columns: warp w serves column
// t = w % T for pages sub, sub + nsub, ... with lane l owning channels
// [l*CPL, (l+1)*CPL). Per key it forms the G partial dot products of its
// channels, all-reduces them over the warp, applies the group scale and the
// online softmax (base-2 exponentials), and accumulates p * Vs * Vc. At the
// end of a segment the warps of one column merge through shared memory and
// the CTA writes either the final bf16 rows (segment = whole unit) or an fp32
// partial with its LSE for the combine.
//
// Attention re-reads the whole cache every step ("NInfer-3090" README,
// "Choosing a KV format"); verify rounds attend draft+1 columns per sequence
// ("Decode after the small-T kernels").
#include "nk_decode.cuh"

namespace nk {

constexpr int kSimtWarps = 8;
constexpr int kSimtMaxG = 8;

// Raw code bytes of one lane for one key (CPL int8 values), loaded ahead of use.
template <int CPL>
struct Raw {
  uint32_t w[CPL >= 4 ? CPL / 4 : 1];
};

template <int CPL>
__device__ __forceinline__ Raw<CPL> load_raw(const uint8_t* src) {
  Raw<CPL> r;
  if constexpr (CPL == 8) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
    r.w[0] = v.x;
    r.w[1] = v.y;
  } else if constexpr (CPL == 4) {
    r.w[0] = __ldg(reinterpret_cast<const unsigned int*>(src));
  } else {
    r.w[0] = __ldg(reinterpret_cast<const unsigned short*>(src));
  }
  return r;
}

template <int CPL>
__device__ __forceinline__ void widen(const Raw<CPL>& r, float (&c)[CPL]) {
#pragma unroll
  for (int i = 0; i < CPL; ++i) c[i] = (float)(int8_t)(r.w[i / 4] >> (8 * (i % 4)));
}

template <int CPL>
__global__ void __launch_bounds__(256) decode_simt_kernel(const DecodeParams p) {
  chain_wait();
  chain_release();
  extern __shared__ float smem[];
  __shared__ int pre[kMaxBatch + 1];
  __shared__ int warp_tot[8];
  const int D = CPL * 32;
  const int G = p.G, T = p.T, M = G * T;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const SplitShape sh = p.shape();
  flag_bad_ctx(p);
  block_page_prefix(sh, p.ctx, p.trim, pre, warp_tot);
  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  if (W == 0) return;
  int64_t x = cta_begin(W, p.n_ctas, blockIdx.x);
  const int64_t x_end = cta_begin(W, p.n_ctas, blockIdx.x + 1);

  float* red_o = smem;                                 // [8 warps][G][D]
  float* red_m = smem + kSimtWarps * G * D;            // [8][G]
  float* red_l = red_m + kSimtWarps * G;               // [8][G]
  const int nsub = kSimtWarps / T;
  const bool active = w < nsub * T;
  const int t = w % T, sub = w / T;
  const int g = D / kGroup;

  Segment seg;
  while (next_segment(sh, pre, x, x_end, seg)) {
    const int L = p.ctx[seg.b] - p.trim;
    const int last = L - T + t;  // last key visible to column t
    float qf[kSimtMaxG][CPL], o[kSimtMaxG][CPL], m[kSimtMaxG], l[kSimtMaxG];
#pragma unroll
    for (int hg = 0; hg < kSimtMaxG; ++hg) {
      m[hg] = -INFINITY;
      l[hg] = 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) { o[hg][j] = 0.f; qf[hg][j] = 0.f; }
      if (hg < G) {
        const uint16_t* qr = p.q + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * D + lane * CPL;
#pragma unroll
        for (int j = 0; j < CPL; ++j) qf[hg][j] = __uint_as_float((uint32_t)__ldg(qr + j) << 16);
      }
    }
    if (active) {
      for (int pi = seg.page_begin + sub; pi < seg.page_end; pi += nsub) {
        if (pi * p.P > last) break;
        const int page = __ldg(p.bt + (int64_t)seg.b * p.max_pages + pi);
        if (page < 0 || page >= p.num_pages) {
          if (lane == 0) flag(p.status, NK_DEVFLAG_BAD_PAGE);
          continue;
        }
        const uint8_t* chunk = p.pool + ((int64_t)page * p.Hkv + seg.h) * p.lay.chunk;
        const int kend = min(p.P, last - pi * p.P + 1);
        // keys in groups of four, the next group's loads issued before the current group's math
        constexpr int KB = 4;
        const int grp = (lane * CPL) / kGroup;
        const float* ksp = reinterpret_cast<const float*>(chunk + p.lay.ks);
        const float* vsp = reinterpret_cast<const float*>(chunk + p.lay.vs);
        Raw<CPL> nkr[KB], nvr[KB];
        float nks[KB], nvs[KB];
        auto load_group = [&](int k0) {
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            const int k = min(k0 + j, kend - 1);  // clamped: a repeated key is never used
            nkr[j] = load_raw<CPL>(chunk + (int64_t)k * D + lane * CPL);
            nvr[j] = load_raw<CPL>(chunk + p.lay.vc + (int64_t)k * D + lane * CPL);
            nks[j] = __ldg(ksp + k * g + grp);
            nvs[j] = __ldg(vsp + k * g + grp);
          }
        };
        load_group(0);
        for (int k0 = 0; k0 < kend; k0 += KB) {
          Raw<CPL> ckr[KB], cvr[KB];
          float cks[KB], cvs[KB];
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            ckr[j] = nkr[j];
            cvr[j] = nvr[j];
            cks[j] = nks[j];
            cvs[j] = nvs[j];
          }
          if (k0 + KB < kend) load_group(k0 + KB);
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            if (k0 + j >= kend) break;
            float kc[CPL], vc[CPL];
            widen<CPL>(ckr[j], kc);
            widen<CPL>(cvr[j], vc);
            const float ks = cks[j], vs = cvs[j];
            float s[kSimtMaxG];
#pragma unroll
            for (int hg = 0; hg < kSimtMaxG; ++hg) {
              float acc = 0.f;
#pragma unroll
              for (int jj = 0; jj < CPL; ++jj) acc = fmaf(qf[hg][jj], kc[jj], acc);
              s[hg] = acc * ks;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
              for (int hg = 0; hg < kSimtMaxG; ++hg) s[hg] += __shfl_xor_sync(0xffffffffu, s[hg], off);
#pragma unroll
            for (int hg = 0; hg < kSimtMaxG; ++hg) {
              if (hg >= G) break;
              const float sc = s[hg] * p.scale2;
              if (sc > m[hg]) {
                const float alpha = exp2f(m[hg] - sc);
                l[hg] *= alpha;
#pragma unroll
                for (int jj = 0; jj < CPL; ++jj) o[hg][jj] *= alpha;
                m[hg] = sc;
              }
              const float pw = exp2f(sc - m[hg]);
              l[hg] += pw;
              const float pv = pw * vs;
#pragma unroll
              for (int jj = 0; jj < CPL; ++jj) o[hg][jj] = fmaf(pv, vc[jj], o[hg][jj]);
            }
          }
        }
      }
    }
    // merge the nsub warps of each column
#pragma unroll
    for (int hg = 0; hg < kSimtMaxG; ++hg) {
      if (hg >= G) break;
#pragma unroll
      for (int j = 0; j < CPL; ++j) red_o[(w * G + hg) * D + lane * CPL + j] = o[hg][j];
      if (lane == 0) {
        red_m[w * G + hg] = active ? m[hg] : -INFINITY;
        red_l[w * G + hg] = active ? l[hg] : 0.f;
      }
    }
    __syncthreads();
    const int seg_slot = blockIdx.x + seg.u;
    for (int i = tid; i < M * D; i += blockDim.x) {
      const int r = i / D, c = i % D;
      const int tt = r / G, hg = r % G;
      float mx = -INFINITY;
      for (int sb = 0; sb < nsub; ++sb) mx = fmaxf(mx, red_m[(sb * T + tt) * G + hg]);
      float lsum = 0.f, acc = 0.f;
      if (mx != -INFINITY) {
        for (int sb = 0; sb < nsub; ++sb) {
          const int ww = sb * T + tt;
          const float mw = red_m[ww * G + hg];
          if (mw == -INFINITY) continue;
          const float sc = exp2f(mw - mx);
          lsum += red_l[ww * G + hg] * sc;
          acc += red_o[(ww * G + hg) * D + c] * sc;
        }
      }
      const float val = lsum > 0.f ? acc / lsum : 0.f;
      if (seg.whole) {
        p.out[(((int64_t)seg.b * p.qT + tt) * p.Hq + seg.h * G + hg) * D + c] = f32_to_bf16(val);
      } else {
        p.part_o[((int64_t)seg_slot * M + r) * D + c] = val;
        if (c == 0) p.part_lse[(int64_t)seg_slot * M + r] = lsum > 0.f ? (mx + log2f(lsum)) * kLn2 : -INFINITY;
      }
    }
    __syncthreads();
  }
}

int decode_simt_ctas_per_sm(int D, int G) {
  int n = 0;
  const size_t smem = (size_t)kSimtWarps * G * (D + 2) * sizeof(float);
  cudaError_t e;
  if (D == 256) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<8>, 256, smem);
  else if (D == 128) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<4>, 256, smem);
  else e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<2>, 256, smem);
  if (e != cudaSuccess) { (void)cudaGetLastError(); return 1; }
  return n < 1 ? 1 : n;
}

template <int CPL>
static cudaError_t launch_simt_t(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(decode_simt_kernel<CPL>), (int)smem);
  if (e != cudaSuccess) return e;
  return launch_chained(decode_simt_kernel<CPL>, dim3(p.n_ctas), dim3(256), smem, stream, p);
}

cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = (size_t)kSimtWarps * p.G * (p.D + 2) * sizeof(float);
  if (p.D == 256) return launch_simt_t<8>(p, smem, stream);
  if (p.D == 128) return launch_simt_t<4>(p, smem, stream);
  return launch_simt_t<2>(p, smem, stream);
}

}  // namespace nk
