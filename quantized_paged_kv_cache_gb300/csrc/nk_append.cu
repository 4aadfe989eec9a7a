// nk_append.cu -- kv_cache_append: quantize new bf16 K/V rows into int8
// 64-channel groups and scatter them into their pages.
//
// The Op that owns KV quantization and stores values from the bf16 source
// directly ("NInfer-3090" README, introduction and "RotorQuant KV (rk8v4)");
// INT8 group-64 storage ("NInfer" README, capability list). Rule per group:
//   a = max|x|, s = fp32(a / 127) (1 if a = 0), q = clamp(rne(fp32(x / s)), +-127).
//
// Bandwidth-bound streaming scatter: each thread owns 16 consecutive channels
// of one (row, kv-head) for both K and V (two 32-byte loads in flight per
// tensor), four threads form a 64-channel group and reduce its absmax with two
// shuffles. The per-element quotient is x * RN(1/s) with an exactness guard:
// the product differs from x/s by less than 2^-16 (|x/s| <= 127.00001) and the
// correctly rounded fp32 quotient differs from x/s by at most 2^-18, so unless
// the product lies within 2^-14 of a half-integer both round to the same
// integer; the rare elements inside that window (and exact ties) take the
// IEEE division out of line.
#include "nk_common.cuh"

namespace nk {

struct AppendParams {
  uint8_t* pool;
  int num_pages, P, Hkv, D;
  ChunkLayout lay;
  const int32_t* bt;
  int max_pages;
  const int32_t* start_pos;
  const int32_t* cu_new;
  int B, total_new;
  const uint4* k;
  const uint4* v;
  int32_t* status;
};

// Exact IEEE path for one element: fp32 quotient, clamp, round half to even.
// Kept out of line: it runs only for elements within 2^-14 of a rounding
// boundary (or for groups with a tiny scale), so the common path stays short.
__device__ __noinline__ uint32_t quantize_exact(float x, float s) {
  float e = __fdiv_rn(x, s);
  e = fminf(fmaxf(e, -127.f), 127.f);
  return (uint32_t)__float2int_rn(e) & 0xffu;
}

// Quantize 16 values (already fp32) of one group slice; returns the scale and
// writes 16 int8 codes packed into 4 words.
__device__ __forceinline__ float quantize16(const float (&x)[16], uint32_t (&packed)[4]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
  // four consecutive lanes hold one 64-channel group
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  const float s = (a == 0.f) ? 1.f : __fdiv_rn(a, 127.f);
  const float y = __frcp_rn(s);
  const bool tiny = s < 7.888609052210118e-31f;  // 2^-100: keep RN(1/s) far from overflow
  // |x * y - x / s| < 2^-16 here, so no clamp is needed on the fast path
  // (|x / s| <= 127 * (1 + 2^-23)); t = r + 1.5 * 2^23 rounds r to an integer
  // (ties to even) whose two's-complement low byte is the low byte of t's bits.
  uint32_t tb[16];
  uint32_t slow = tiny ? 0xffffu : 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float r = __fmul_rn(x[i], y);
    const float t = __fadd_rn(r, 12582912.f);
    const float d = __fsub_rn(r, __fsub_rn(t, 12582912.f));
    if (fabsf(d) > 0.49993896484375f /* 0.5 - 2^-14 */) slow |= 1u << i;
    tb[i] = __float_as_uint(t);
  }
  if (slow) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((slow >> i) & 1u) tb[i] = quantize_exact(x[i], s);
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t lo = __byte_perm(tb[4 * w], tb[4 * w + 1], 0x0040);
    const uint32_t hi = __byte_perm(tb[4 * w + 2], tb[4 * w + 3], 0x0040);
    packed[w] = __byte_perm(lo, hi, 0x5410);
  }
  return s;
}

__device__ __forceinline__ void unpack16(const uint4& lo, const uint4& hi, float (&x)[16]) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }
}

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  const int tpr = p.D / 16;  // threads per (row, head)
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t idx = tid / tpr;  // (row, head) index
  const int part = (int)(tid % tpr);
  const bool live = idx < (int64_t)p.total_new * p.Hkv;
  const int j = live ? (int)(idx / p.Hkv) : 0;
  const int h = live ? (int)(idx % p.Hkv) : 0;

  uint4 klo = make_uint4(0, 0, 0, 0), khi = klo, vlo = klo, vhi = klo;
  if (live) {
    const int64_t base = (idx * p.D + part * 16) / 8;  // in uint4 units
    klo = __ldg(p.k + base);
    khi = __ldg(p.k + base + 1);
    vlo = __ldg(p.v + base);
    vhi = __ldg(p.v + base + 1);
  }

  // destination: sequence b owns rows cu_new[b] .. cu_new[b+1]-1
  bool ok = live;
  int64_t dst = 0;
  int slot = 0;
  if (live) {
    int lo = 0, hi = p.B;  // find b with cu_new[b] <= j < cu_new[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.cu_new + mid) <= j) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int64_t pos = (int64_t)__ldg(p.start_pos + b) + (j - __ldg(p.cu_new + b));
    if (pos < 0 || pos >= (int64_t)p.max_pages * p.P) {
      ok = false;
      if (part == 0) flag(p.status, NK_DEVFLAG_BAD_POS);
    } else {
      const int page = __ldg(p.bt + (int64_t)b * p.max_pages + pos / p.P);
      if (page < 0 || page >= p.num_pages) {
        ok = false;
        if (part == 0) flag(p.status, NK_DEVFLAG_BAD_PAGE);
      } else {
        slot = (int)(pos % p.P);
        dst = ((int64_t)page * p.Hkv + h) * p.lay.chunk;
      }
    }
  }

  const int g = p.D / kGroup;
  float x[16];
  uint32_t packed[4];
  unpack16(klo, khi, x);
  float s = quantize16(x, packed);
  if (ok) {
    *reinterpret_cast<uint4*>(p.pool + dst + (int64_t)slot * p.D + part * 16) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if ((part & 3) == 0) *reinterpret_cast<float*>(p.pool + dst + p.lay.ks + ((int64_t)slot * g + part / 4) * 4) = s;
  }
  unpack16(vlo, vhi, x);
  s = quantize16(x, packed);
  if (ok) {
    *reinterpret_cast<uint4*>(p.pool + dst + p.lay.vc + (int64_t)slot * p.D + part * 16) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if ((part & 3) == 0) *reinterpret_cast<float*>(p.pool + dst + p.lay.vs + ((int64_t)slot * g + part / 4) * 4) = s;
  }
}

cudaError_t launch_kv_append(const nk_kv_pool& pool, const int32_t* bt, int max_pages, const int32_t* start_pos,
                             const int32_t* cu_new, int B, int total_new, const void* k, const void* v,
                             int32_t* status, cudaStream_t stream) {
  AppendParams p;
  p.pool = reinterpret_cast<uint8_t*>(pool.base_dev);
  p.num_pages = pool.num_pages;
  p.P = pool.page_size;
  p.Hkv = pool.num_kv_heads;
  p.D = pool.head_dim;
  p.lay = ChunkLayout::make(p.P, p.D);
  p.bt = bt;
  p.max_pages = max_pages;
  p.start_pos = start_pos;
  p.cu_new = cu_new;
  p.B = B;
  p.total_new = total_new;
  p.k = reinterpret_cast<const uint4*>(k);
  p.v = reinterpret_cast<const uint4*>(v);
  p.status = status;
  const int64_t threads = (int64_t)total_new * p.Hkv * (p.D / 16);
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (grid == 0) return cudaSuccess;
  kv_append_kernel<<<(unsigned)grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nk
