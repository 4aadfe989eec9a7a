// nk_rk8v4.cu -- append and split-KV decode attention for the rk8v4 KV format
// ("NInfer-3090" README, "RotorQuant KV (rk8v4)"): the keys of every
// 64-channel group are rotated by R = H64 / 8 (Sylvester Hadamard, its own
// inverse) and stored as INT8 codes, the values are stored unrotated as 4-bit
// codes over 32-channel groups; all scales are fp16. Attention rotates each
// query row by the same R, so q . k = (R q) . (R k) is scored against the
// stored keys directly and no inverse rotation is needed.
//
// Quantization (both sides of the parity tests take these decisions in the
// same precision):
//   keys   y = R k = RN_fp32(H64 k / 8), one rounding of the exact sum;
//          s = RN_fp16(fp32(max|y| / 127)), q = clamp(rne(fp32(y / s)), +-127);
//   values s = RN_fp16(fp32(max|v| / 7)),   q = clamp(rne(fp32(v / s)), +-7);
//   a scale that rounds to 0 becomes 1 (its codes are then 0), one past the
//   fp16 maximum saturates at 65504 (NK_DEVFLAG_RANGE).
// fp32(a / c) rounded again to fp16 is the correctly rounded fp16 quotient
// here: a / c (c = 127 or 7) is never an fp16 rounding midpoint and lies
// more than half an fp32 ulp away from every one.
//
// The attention kernel runs on fp32 CUDA cores with the split and partial
// layout of the INT8 decode kernels, so their log-sum-exp combine merges its
// partials unchanged.
#include <cuda_fp16.h>

#include "nk_ptx.cuh"
#include "nk_rk8v4.cuh"

namespace nk {

// fp16 scale bits of a group whose absmax is a, for codes up to qmax.
__device__ __forceinline__ uint16_t rk_scale_bits(float a, float qmax, bool& range) {
  uint16_t b = __half_as_ushort(__float2half_rn(__fdiv_rn(a, qmax)));
  if ((b & 0x7fffu) == 0) {
    b = 0x3c00u;
  } else if ((b & 0x7fffu) >= 0x7c00u) {  // past the fp16 range (or not a number)
    b = 0x7bffu;
    range = true;
  }
  return b;
}

__device__ __forceinline__ uint32_t rk_code(float x, float s, int qmax) {
  int q = __float2int_rn(__fdiv_rn(x, s));
  q = q > qmax ? qmax : (q < -qmax ? -qmax : q);
  return (uint32_t)q;
}

// ---------------------------------------------------------------------------
// The key rotation y = RN_fp32(H64 x / 8): every output is the exact signed
// sum of the group's 64 bf16 values, divided by 8 and rounded once.
//
// A finite bf16 value is an integer multiple of the quantum of its exponent
// (2^(e-134) for exponent field e >= 1, 2^-133 for e = 0). When the group's
// non-zero values have exponent fields within 39 of each other, each is an
// integer below 2^47 in units of the smallest one, every partial sum of up
// to 64 of them is an integer below 2^53, so int64 butterflies (a + b,
// a - b) are exact; one int64 -> fp32 conversion rounds to nearest even and
// the unit 2^(emin-137) (the 1/8 included) is applied to the exponent
// field, exact while the result is a normal fp32 number (and an infinity
// where it overflows). Wider groups and results in the fp32 subnormal range
// (rare, degenerate inputs) take rk_rotate_wide: an exact integer sum in
// 32-bit limbs and an explicit round to nearest even. (GB300 runs fp64 at a
// small fraction of its integer rate, so the butterflies stay integer.)
// ---------------------------------------------------------------------------
constexpr int kWideLimbs = 10;  // 320 bits: |x| < 2^128 in 2^-133 units, times 64

// a += units * 2^shift (units < 2^8): the magnitude sum of one sign.
__device__ __forceinline__ void wide_add(uint32_t (&a)[kWideLimbs], uint32_t units, int shift) {
  int k = shift >> 5;
  const uint64_t v = (uint64_t)units << (shift & 31);
  uint64_t cur = (uint64_t)a[k] + (uint32_t)v;
  a[k] = (uint32_t)cur;
  uint64_t carry = (cur >> 32) + (v >> 32);
  for (++k; k < kWideLimbs && carry; ++k) {
    cur = (uint64_t)a[k] + carry;
    a[k] = (uint32_t)cur;
    carry = cur >> 32;
  }
}

// Bit `pos` of a (0 below bit 0).
__device__ __forceinline__ uint32_t wide_bit(const uint32_t (&a)[kWideLimbs], int pos) {
  return pos < 0 ? 0u : (a[pos >> 5] >> (pos & 31)) & 1u;
}

// fp32 bits of RN(m * 2^-136) for the magnitude m in `a`, sign `neg`.
__device__ uint32_t wide_round(const uint32_t (&a)[kWideLimbs], bool neg) {
  int top = -1;
  for (int k = kWideLimbs - 1; k >= 0 && top < 0; --k)
    if (a[k]) top = 32 * k + 31 - __clz(a[k]);
  const uint32_t sign = neg ? 0x80000000u : 0u;
  if (top < 0) return 0u;
  if (top < 24) {  // exact: fewer than 25 significant bits
    const uint32_t m = a[0];
    if (top < 10) return sign | (m << 13);  // fp32 subnormal: m * 2^-136 = (m << 13) * 2^-149
    return sign | ((uint32_t)(top - 9) << 23) | ((m << (23 - top)) & 0x7fffffu);
  }
  const int low = top - 23;
  uint32_t m = 0;
  for (int b = 23; b >= 0; --b) m = (m << 1) | wide_bit(a, low + b);
  const uint32_t guard = wide_bit(a, low - 1);
  bool sticky = false;
  for (int b = 0; b < low - 1; ++b) sticky |= wide_bit(a, b) != 0u;
  if (guard && (sticky || (m & 1u))) ++m;
  int e = top - 9;  // biased exponent of the leading bit 2^(top - 136)
  if (m == (1u << 24)) {
    m >>= 1;
    ++e;
  }
  if (e >= 255) return sign | 0x7f800000u;
  return sign | ((uint32_t)e << 23) | (m & 0x7fffffu);
}

// R x of one group whose exponents span more than 39 binades, exactly.
__device__ void rk_rotate_wide(const uint16_t (&xb)[kGroup], float (&y)[kGroup]) {
  for (int r = 0; r < kGroup; ++r) {
    uint32_t pos[kWideLimbs], ng[kWideLimbs];
    for (int k = 0; k < kWideLimbs; ++k) pos[k] = ng[k] = 0u;
    for (int j = 0; j < kGroup; ++j) {
      const uint32_t b = xb[j], e = (b >> 7) & 0xffu, f = b & 0x7fu;
      if (e == 0u && f == 0u) continue;
      const uint32_t units = e == 0u ? f : 128u + f;
      const int shift = e == 0u ? 0 : (int)e - 1;
      const bool minus = ((b >> 15) ^ (__popc((uint32_t)(r & j)) & 1u)) != 0u;
      wide_add(minus ? ng : pos, units, shift);
    }
    // |pos - ng| and its sign
    bool neg = false;
    for (int k = kWideLimbs - 1; k >= 0; --k)
      if (pos[k] != ng[k]) {
        neg = ng[k] > pos[k];
        break;
      }
    uint32_t d[kWideLimbs];
    uint32_t borrow = 0u;
    for (int k = 0; k < kWideLimbs; ++k) {
      const uint64_t hi = neg ? ng[k] : pos[k], lo = (uint64_t)(neg ? pos[k] : ng[k]) + borrow;
      d[k] = (uint32_t)(hi - lo);
      borrow = hi < lo ? 1u : 0u;
    }
    y[r] = __uint_as_float(wide_round(d, neg));
  }
}

// One key group: 64 bf16 channels -> 64 int8 codes of R k and the fp16 scale.
__device__ __forceinline__ void rk_key_group(const uint4* src, uint4* dst, uint16_t* scale, bool& range) {
  uint16_t xb[kGroup];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = __ldg(src + c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xb[8 * c + 2 * i] = (uint16_t)(ws[i] & 0xffffu);
      xb[8 * c + 2 * i + 1] = (uint16_t)(ws[i] >> 16);
    }
  }
  int emax = 0, emin = 255;  // exponent fields of the non-zero values (subnormals count as 1)
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    if ((xb[i] & 0x7fffu) == 0u) continue;
    const int e = max(1, (xb[i] >> 7) & 0xff);
    emax = max(emax, e);
    emin = min(emin, e);
  }
  float t[kGroup];
  bool wide = emax - emin > 39;
  if (!wide) {
    long long d[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const uint32_t mag = xb[i] & 0x7fffu, e = mag >> 7;
      const long long m = mag == 0u ? 0ll
                                    : (long long)((mag & 0x7fu) | (e != 0u ? 0x80u : 0u))
                                          << ((e != 0u ? (int)e : 1) - emin);
      d[i] = (xb[i] & 0x8000u) ? -m : m;
    }
#pragma unroll
    for (int h = 1; h < kGroup; h <<= 1)
#pragma unroll
      for (int i = 0; i < kGroup; ++i)
        if ((i & h) == 0) {
          const long long a = d[i], b = d[i + h];
          d[i] = a + b;
          d[i + h] = a - b;
        }
    const int k = emin - 137;  // y = d 2^k
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      if (d[i] == 0) {
        t[i] = 0.f;
        continue;
      }
      const uint32_t fb = __float_as_uint(__ll2float_rn(d[i]));  // |d| >= 1: a normal number
      const int ne = (int)((fb >> 23) & 0xffu) + k;
      if (ne >= 255)
        t[i] = __uint_as_float((fb & 0x80000000u) | 0x7f800000u);
      else if (ne >= 1)
        t[i] = __uint_as_float((uint32_t)((int)fb + k * (1 << 23)));
      else
        wide = true;  // an fp32 subnormal result: rounded in the wide path
    }
  }
  if (wide) rk_rotate_wide(xb, t);
  float amax = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < kGroup; ++i) {
    finite &= isfinite(t[i]);
    amax = fmaxf(amax, fabsf(t[i]));
  }
  if (!finite) range = true;
  const uint16_t sb = rk_scale_bits(amax, 127.f, range);
  const float s = __half2float(__ushort_as_half(sb));
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 16 * c + 4 * j;
      w[j] = (rk_code(t[e], s, 127) & 0xffu) | ((rk_code(t[e + 1], s, 127) & 0xffu) << 8) |
             ((rk_code(t[e + 2], s, 127) & 0xffu) << 16) | ((rk_code(t[e + 3], s, 127) & 0xffu) << 24);
    }
    dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  *scale = sb;
}

// One value group: 32 bf16 channels -> 16 bytes of 4-bit codes and the fp16 scale.
__device__ __forceinline__ void rk_value_group(const uint4* src, uint4* dst, uint16_t* scale, bool& range) {
  uint32_t raw[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = __ldg(src + c);
    raw[4 * c] = w.x;
    raw[4 * c + 1] = w.y;
    raw[4 * c + 2] = w.z;
    raw[4 * c + 3] = w.w;
  }
  float amax = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float a = bf16_lo(raw[i]), b = bf16_hi(raw[i]);
    finite &= isfinite(a) && isfinite(b);
    amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
  }
  if (!finite) range = true;
  const uint16_t sb = rk_scale_bits(amax, 7.f, range);
  const float s = __half2float(__ushort_as_half(sb));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // byte i: channel 2i (low nibble), 2i + 1 (high nibble)
    const uint32_t byte = (rk_code(bf16_lo(raw[i]), s, 7) & 0xfu) | ((rk_code(bf16_hi(raw[i]), s, 7) & 0xfu) << 4);
    w[i / 4] |= byte << (8 * (i % 4));
  }
  *dst = make_uint4(w[0], w[1], w[2], w[3]);
  *scale = sb;
}

struct RkAppendParams {
  uint8_t* pool;
  int num_pages, P, Hkv, D;
  ChunkLayout lay;
  const int32_t* bt;
  int max_pages;
  const int32_t* start_pos;
  const int32_t* cu_new;
  int B, total_new;
  const uint16_t* k;
  const uint16_t* v;
  int32_t* status;
};

// One thread per item; the items of a (row, kv-head) are its D/64 key groups
// followed by its D/32 value groups.
__global__ void __launch_bounds__(128) rk8v4_append_kernel(const RkAppendParams p) {
  chain_wait();
  chain_release();
  const int kg = p.D / kGroup, vg = p.D / kRkVGroup, per = kg + vg;
  const int64_t items = (int64_t)p.total_new * p.Hkv * per;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rh = it / per;
    const int r = (int)(it % per);
    const int j = (int)(rh / p.Hkv), h = (int)(rh % p.Hkv);
    // sequence b of row j: cu_new[b] <= j < cu_new[b + 1]
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.cu_new + mid) <= j) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int64_t pos = (int64_t)__ldg(p.start_pos + b) + (j - __ldg(p.cu_new + b));
    if (pos < 0 || pos >= (int64_t)p.max_pages * p.P) {
      flag(p.status, NK_DEVFLAG_BAD_POS);
      continue;
    }
    const int page = __ldg(p.bt + (int64_t)b * p.max_pages + pos / p.P);
    if (page < 0 || page >= p.num_pages) {
      flag(p.status, NK_DEVFLAG_BAD_PAGE);
      continue;
    }
    const int slot = (int)(pos % p.P);
    uint8_t* chunk = p.pool + ((int64_t)page * p.Hkv + h) * p.lay.chunk;
    const int64_t row = ((int64_t)j * p.Hkv + h) * p.D;
    bool range = false;
    if (r < kg) {
      rk_key_group(reinterpret_cast<const uint4*>(p.k + row + r * kGroup),
                   reinterpret_cast<uint4*>(chunk + (int64_t)slot * p.D + r * kGroup),
                   reinterpret_cast<uint16_t*>(chunk + p.lay.ks) + slot * kg + r, range);
    } else {
      const int g = r - kg;
      rk_value_group(reinterpret_cast<const uint4*>(p.v + row + g * kRkVGroup),
                     reinterpret_cast<uint4*>(chunk + p.lay.vc + (int64_t)slot * (p.D / 2) + g * (kRkVGroup / 2)),
                     reinterpret_cast<uint16_t*>(chunk + p.lay.vs) + slot * vg + g, range);
    }
    if (range) flag(p.status, NK_DEVFLAG_RANGE);
  }
}

// Destination of row j of the batch (kv-head h): the chunk and slot, or
// nullptr after flagging a position or page id out of range.
__device__ __forceinline__ uint8_t* rk_dest(const RkAppendParams& p, int j, int h, int& slot, bool flagger) {
  int lo = 0, hi = p.B;  // sequence b of row j: cu_new[b] <= j < cu_new[b + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.cu_new + mid) <= j) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int64_t pos = (int64_t)__ldg(p.start_pos + b) + (j - __ldg(p.cu_new + b));
  if (pos < 0 || pos >= (int64_t)p.max_pages * p.P) {
    if (flagger) flag(p.status, NK_DEVFLAG_BAD_POS);
    return nullptr;
  }
  const int page = __ldg(p.bt + (int64_t)b * p.max_pages + pos / p.P);
  if (page < 0 || page >= p.num_pages) {
    if (flagger) flag(p.status, NK_DEVFLAG_BAD_PAGE);
    return nullptr;
  }
  slot = (int)(pos % p.P);
  return p.pool + ((int64_t)page * p.Hkv + h) * p.lay.chunk;
}

__device__ __forceinline__ long long shfl_xor_ll(long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)(unsigned long long)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)((unsigned long long)v >> 32), m);
  return (long long)(((unsigned long long)hi << 32) | lo);
}

// Small appends (decode and verify steps: a few rows). The thread-per-item
// kernel above then runs only a few dozen threads, each through a whole key
// group's rotation; here a warp takes a key group, lane l holding channels
// 2l and 2l + 1: the first butterfly stage runs in the lane, the five others
// across lanes by shuffle, on the same exact integer sums (so the same
// bits), then each lane rounds and codes its two outputs. A group whose
// exponents span more than 39 binades, or with an output in the fp32
// subnormal range, is rotated by lane 0 alone in the exact wide path (all of
// it, as the thread-per-item kernel does). Value groups: one thread each, in
// the warps after the key groups'.
__global__ void __launch_bounds__(128) rk8v4_append_small_kernel(const RkAppendParams p) {
  chain_wait();
  chain_release();
  const int kg = p.D / kGroup, vg = p.D / kRkVGroup;
  const int64_t nkey = (int64_t)p.total_new * p.Hkv * kg;  // key groups: one warp each
  const int64_t nval = (int64_t)p.total_new * p.Hkv * vg;  // value groups: one thread each
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= nkey) {
    const int64_t it = (gw - nkey) * 32 + lane;
    if (it >= nval) return;
    const int64_t rh = it / vg;
    const int g = (int)(it % vg), j = (int)(rh / p.Hkv), h = (int)(rh % p.Hkv);
    int slot = 0;
    uint8_t* chunk = rk_dest(p, j, h, slot, g == 0);
    if (!chunk) return;
    bool range = false;
    rk_value_group(reinterpret_cast<const uint4*>(p.v + ((int64_t)j * p.Hkv + h) * p.D + g * kRkVGroup),
                   reinterpret_cast<uint4*>(chunk + p.lay.vc + (int64_t)slot * (p.D / 2) + g * (kRkVGroup / 2)),
                   reinterpret_cast<uint16_t*>(chunk + p.lay.vs) + slot * vg + g, range);
    if (range) flag(p.status, NK_DEVFLAG_RANGE);
    return;
  }
  // one key group per warp (every lane takes the same branches up to the shuffles)
  const int64_t rh = gw / kg;
  const int r = (int)(gw % kg), j = (int)(rh / p.Hkv), h = (int)(rh % p.Hkv);
  int slot = 0;
  uint8_t* chunk = rk_dest(p, j, h, slot, r == 0 && lane == 0);
  if (!chunk) return;
  const uint16_t* src = p.k + ((int64_t)j * p.Hkv + h) * p.D + r * kGroup;
  uint8_t* dst = chunk + (int64_t)slot * p.D + r * kGroup;
  uint16_t* sdst = reinterpret_cast<uint16_t*>(chunk + p.lay.ks) + slot * kg + r;
  const uint32_t wv = __ldg(reinterpret_cast<const uint32_t*>(src) + lane);
  const uint16_t xb[2] = {(uint16_t)(wv & 0xffffu), (uint16_t)(wv >> 16)};
  int emax = 0, emin = 255;  // exponent fields of the non-zero values (subnormals count as 1)
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if ((xb[c] & 0x7fffu) == 0u) continue;
    const int e = max(1, (xb[c] >> 7) & 0xff);
    emax = max(emax, e);
    emin = min(emin, e);
  }
  emax = __reduce_max_sync(0xffffffffu, emax);
  emin = __reduce_min_sync(0xffffffffu, emin);
  bool wide = emax - emin > 39;
  float t[2] = {0.f, 0.f};
  if (!wide) {
    long long d[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t mag = xb[c] & 0x7fffu, e = mag >> 7;
      const long long m = mag == 0u ? 0ll
                                    : (long long)((mag & 0x7fu) | (e != 0u ? 0x80u : 0u))
                                          << ((e != 0u ? (int)e : 1) - emin);
      d[c] = (xb[c] & 0x8000u) ? -m : m;
    }
    {  // distance 1: channels 2l, 2l + 1
      const long long a = d[0], b = d[1];
      d[0] = a + b;
      d[1] = a - b;
    }
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {  // distance 2 hl: lane l ^ hl holds the partner
      const bool upper = (lane & hl) != 0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const long long q = shfl_xor_ll(d[c], hl);
        d[c] = upper ? q - d[c] : d[c] + q;
      }
    }
    const int k = emin - 137;  // y = d 2^k
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (d[c] == 0) continue;
      const uint32_t fb = __float_as_uint(__ll2float_rn(d[c]));  // |d| >= 1: a normal number
      const int ne = (int)((fb >> 23) & 0xffu) + k;
      if (ne >= 255)
        t[c] = __uint_as_float((fb & 0x80000000u) | 0x7f800000u);
      else if (ne >= 1)
        t[c] = __uint_as_float((uint32_t)((int)fb + k * (1 << 23)));
      else
        wide = true;  // an fp32 subnormal result: the wide path
    }
  }
  if (__any_sync(0xffffffffu, wide)) {
    if (lane == 0) {
      bool range = false;
      rk_key_group(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), sdst, range);
      if (range) flag(p.status, NK_DEVFLAG_RANGE);
    }
    return;
  }
  bool range = !__all_sync(0xffffffffu, isfinite(t[0]) && isfinite(t[1]));
  const float amax = __uint_as_float(
      __reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(fabsf(t[0]), fabsf(t[1])))));
  const uint16_t sb = rk_scale_bits(amax, 127.f, range);
  const float s = __half2float(__ushort_as_half(sb));
  reinterpret_cast<uint16_t*>(dst)[lane] =
      (uint16_t)((rk_code(t[0], s, 127) & 0xffu) | ((rk_code(t[1], s, 127) & 0xffu) << 8));
  if (lane == 0) {
    *sdst = sb;
    if (range) flag(p.status, NK_DEVFLAG_RANGE);
  }
}

constexpr int64_t kRkSmallKeyGroups = 2048;  // appends up to this many key groups take the warp-per-group kernel

cudaError_t launch_rk8v4_append(int sms, const nk_kv_pool& pool, const int32_t* bt, int max_pages,
                                const int32_t* start_pos, const int32_t* cu_new, int B, int total_new, const void* k,
                                const void* v, int32_t* status, cudaStream_t stream) {
  RkAppendParams p;
  p.pool = reinterpret_cast<uint8_t*>(pool.base_dev);
  p.num_pages = pool.num_pages;
  p.P = pool.page_size;
  p.Hkv = pool.num_kv_heads;
  p.D = pool.head_dim;
  p.lay = rk8v4_layout(p.P, p.D);
  p.bt = bt;
  p.max_pages = max_pages;
  p.start_pos = start_pos;
  p.cu_new = cu_new;
  p.B = B;
  p.total_new = total_new;
  p.k = reinterpret_cast<const uint16_t*>(k);
  p.v = reinterpret_cast<const uint16_t*>(v);
  p.status = status;
  const int64_t nkey = (int64_t)total_new * p.Hkv * (p.D / kGroup);
  if (nkey <= kRkSmallKeyGroups) {  // decode and verify steps: a warp per key group
    const int64_t warps = nkey + ((int64_t)total_new * p.Hkv * (p.D / kRkVGroup) + 31) / 32;
    const int64_t nb = (warps * 32 + 127) / 128;
    return launch_chained(rk8v4_append_small_kernel, dim3((unsigned)(nb < 1 ? 1 : nb)), dim3(128), 0, stream, p);
  }
  const int64_t items = (int64_t)total_new * p.Hkv * (p.D / kGroup + p.D / kRkVGroup);
  int64_t blocks = (items + 127) / 128;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_chained(rk8v4_append_kernel, dim3((unsigned)blocks), dim3(128), 0, stream, p);
}

// ---------------------------------------------------------------------------
// Decode attention, unstaged form (used where pages are too large for the
// staged kernel's ring, below). Same structure as the INT8 CUDA-core kernel:
// each CTA walks its segments of (sequence, kv-head, page) items; warp w
// serves query column t = w % T for pages sub, sub + nsub, ...; lane l owns channels
// [l CPL, (l + 1) CPL). The query rows are rotated once per segment (the
// butterflies of the channel bits a lane holds in registers, then those of the
// lane bits by shuffles); per key a warp forms the G dot products with the
// int8 codes, all-reduces them, applies the key's fp16 group scale and the
// online softmax (base 2), and accumulates p * Vs * (4-bit code).
// ---------------------------------------------------------------------------
constexpr int kRkWarps = 8;
constexpr int kRkMaxG = 8;

template <int CPL>
struct RkRaw {
  uint32_t k[CPL >= 4 ? CPL / 4 : 1];  // CPL int8 key codes
  uint32_t v;                          // CPL 4-bit value codes
};

template <int CPL>
__device__ __forceinline__ RkRaw<CPL> rk_load(const uint8_t* kc, const uint8_t* vc) {
  RkRaw<CPL> r;
  if constexpr (CPL == 8) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(kc));
    r.k[0] = w.x;
    r.k[1] = w.y;
    r.v = __ldg(reinterpret_cast<const unsigned int*>(vc));
  } else if constexpr (CPL == 4) {
    r.k[0] = __ldg(reinterpret_cast<const unsigned int*>(kc));
    r.v = __ldg(reinterpret_cast<const unsigned short*>(vc));
  } else {
    r.k[0] = __ldg(reinterpret_cast<const unsigned short*>(kc));
    r.v = __ldg(vc);
  }
  return r;
}

// The same codes from a page staged in shared memory (plain loads).
template <int CPL>
__device__ __forceinline__ RkRaw<CPL> rk_load_shared(const uint8_t* kc, const uint8_t* vc) {
  RkRaw<CPL> r;
  if constexpr (CPL == 8) {
    const uint2 w = *reinterpret_cast<const uint2*>(kc);
    r.k[0] = w.x;
    r.k[1] = w.y;
    r.v = *reinterpret_cast<const uint32_t*>(vc);
  } else if constexpr (CPL == 4) {
    r.k[0] = *reinterpret_cast<const uint32_t*>(kc);
    r.v = *reinterpret_cast<const uint16_t*>(vc);
  } else {
    r.k[0] = *reinterpret_cast<const uint16_t*>(kc);
    r.v = *vc;
  }
  return r;
}

template <int CPL>
__global__ void __launch_bounds__(256) decode_rk8v4_kernel(const DecodeParams p) {
  chain_wait();
  chain_release();
  extern __shared__ float smem[];
  __shared__ int pre[kMaxBatch + 1];
  __shared__ int warp_tot[8];
  constexpr int D = CPL * 32;
  constexpr int LPG = kGroup / CPL;  // lanes per 64-channel group
  const int G = p.G, T = p.T, M = G * T;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const SplitShape sh = p.shape();
  flag_bad_ctx(p);
  block_page_prefix(sh, p.ctx, p.trim, pre, warp_tot);
  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  if (W == 0) return;
  int64_t x = cta_begin(W, p.n_ctas, blockIdx.x);
  const int64_t x_end = cta_begin(W, p.n_ctas, blockIdx.x + 1);

  float* red_o = smem;                          // [8 warps][G][D]
  float* red_m = smem + kRkWarps * G * D;       // [8][G]
  float* red_l = red_m + kRkWarps * G;          // [8][G]
  const int nsub = kRkWarps / T;
  const bool active = w < nsub * T;
  const int t = w % T, sub = w / T;
  const int kgrp = (lane * CPL) / kGroup, vgrp = (lane * CPL) / kRkVGroup;

  Segment seg;
  while (next_segment(sh, pre, x, x_end, seg)) {
    const int L = p.ctx[seg.b] - p.trim;
    const int last = L - T + t;  // last key visible to column t
    float qf[kRkMaxG][CPL], o[kRkMaxG][CPL], m[kRkMaxG], l[kRkMaxG];
#pragma unroll
    for (int hg = 0; hg < kRkMaxG; ++hg) {
      m[hg] = -INFINITY;
      l[hg] = 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) { o[hg][j] = 0.f; qf[hg][j] = 0.f; }
      if (hg < G) {
        const uint16_t* qr = p.q + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * D + lane * CPL;
#pragma unroll
        for (int j = 0; j < CPL; ++j) qf[hg][j] = __uint_as_float((uint32_t)__ldg(qr + j) << 16);
      }
      // R q: channel c of a group is j + CPL (lane mod LPG); its low bits are
      // j (in registers), the high ones the lane's (by shuffles)
#pragma unroll
      for (int h = 1; h < CPL; h <<= 1)
#pragma unroll
        for (int j = 0; j < CPL; ++j)
          if ((j & h) == 0) {
            const float a = qf[hg][j], b = qf[hg][j + h];
            qf[hg][j] = a + b;
            qf[hg][j + h] = a - b;
          }
#pragma unroll
      for (int lb = 1; lb < LPG; lb <<= 1) {
        const bool upper = (lane & lb) != 0;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const float other = __shfl_xor_sync(0xffffffffu, qf[hg][j], lb);
          qf[hg][j] = upper ? other - qf[hg][j] : qf[hg][j] + other;
        }
      }
#pragma unroll
      for (int j = 0; j < CPL; ++j) qf[hg][j] *= 0.125f;
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
        const __half* ksp = reinterpret_cast<const __half*>(chunk + p.lay.ks);
        const __half* vsp = reinterpret_cast<const __half*>(chunk + p.lay.vs);
        // keys in groups of four, the next group's loads issued before the current group's math
        constexpr int KB = 4;
        RkRaw<CPL> nr[KB];
        __half nks[KB], nvs[KB];
        auto load_group = [&](int k0) {
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            const int k = min(k0 + j, kend - 1);  // clamped: a repeated key is never used
            nr[j] = rk_load<CPL>(chunk + (int64_t)k * D + lane * CPL, chunk + p.lay.vc + (int64_t)k * (D / 2) +
                                                                          lane * (CPL / 2));
            nks[j] = ksp[k * (D / kGroup) + kgrp];
            nvs[j] = vsp[k * (D / kRkVGroup) + vgrp];
          }
        };
        load_group(0);
        for (int k0 = 0; k0 < kend; k0 += KB) {
          RkRaw<CPL> cr[KB];
          float cks[KB], cvs[KB];
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            cr[j] = nr[j];
            cks[j] = __half2float(nks[j]);
            cvs[j] = __half2float(nvs[j]);
          }
          if (k0 + KB < kend) load_group(k0 + KB);
#pragma unroll
          for (int j = 0; j < KB; ++j) {
            if (k0 + j >= kend) break;
            float kc[CPL], vc[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
              kc[i] = (float)(int8_t)(cr[j].k[i / 4] >> (8 * (i % 4)));
              vc[i] = (float)((int32_t)(cr[j].v << (28 - 4 * i)) >> 28);  // sign-extended nibble i
            }
            float s[kRkMaxG];
#pragma unroll
            for (int hg = 0; hg < kRkMaxG; ++hg) {
              float acc = 0.f;
#pragma unroll
              for (int jj = 0; jj < CPL; ++jj) acc = fmaf(qf[hg][jj], kc[jj], acc);
              s[hg] = acc * cks[j];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
              for (int hg = 0; hg < kRkMaxG; ++hg) s[hg] += __shfl_xor_sync(0xffffffffu, s[hg], off);
#pragma unroll
            for (int hg = 0; hg < kRkMaxG; ++hg) {
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
              const float pv = pw * cvs[j];
#pragma unroll
              for (int jj = 0; jj < CPL; ++jj) o[hg][jj] = fmaf(pv, vc[jj], o[hg][jj]);
            }
          }
        }
      }
    }
    // merge the nsub warps of each column
#pragma unroll
    for (int hg = 0; hg < kRkMaxG; ++hg) {
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

// ---------------------------------------------------------------------------
// Staged decode, used wherever the ring below holds at least three pages. The
// CTA walks the same segments, but every (page, kv-head) chunk -- contiguous,
// 26,112 bytes at P = 64, D = 256 -- arrives in a shared-memory ring through
// one bulk asynchronous copy, issued when the last of the 8 warps releases
// the stage S pages earlier, and all the warps of the CTA work on the same
// pages (each may run up to S pages ahead of the others): warp w takes query column
// t = w % T and keys [sub KPW, (sub + 1) KPW) of the page (sub = w / T, KPW =
// P / (8 / T) rounded up). Keys are taken four at a time: the four keys' warp
// reductions are independent, so their shuffles overlap, and a row's running
// maximum moves at most once per four keys. GM >= G is the number of query
// heads the registers hold.
// ---------------------------------------------------------------------------
constexpr int kRkMaxStages = 8;
constexpr int kRkSmemBudget = 232448 - 8192;  // opt-in shared memory per block, less the static arrays

__host__ __device__ inline int rk_staged_fixed_bytes(int D, int GM) {
  return kRkWarps * GM * D * 4 + 2 * kRkWarps * GM * 4 + 128;
}

__host__ __device__ inline int rk_staged_stages(int chunk, int D, int GM) {
  int s = (kRkSmemBudget - rk_staged_fixed_bytes(D, GM)) / chunk;
  return s > kRkMaxStages ? kRkMaxStages : s;
}

template <int CPL, int GM>
__global__ void __launch_bounds__(256, 1) decode_rk8v4_staged_kernel(const DecodeParams p, int S) {
  chain_wait();
  chain_release();
  extern __shared__ uint8_t rk_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rk_smem_raw) + 127) & ~uintptr_t(127));
  __shared__ int pre[kMaxBatch + 1];
  __shared__ int warp_tot[8];
  __shared__ int stage_ok[kRkMaxStages];
  __shared__ __align__(8) uint64_t full_bar[kRkMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kRkMaxStages];  // the 8 warps are done with the stage
  __shared__ int rel_cnt[kRkMaxStages];
  __shared__ volatile int abort_flag;
  constexpr int D = CPL * 32;
  constexpr int LPG = kGroup / CPL;  // lanes per 64-channel group
  const int G = p.G, T = p.T, M = G * T;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const SplitShape sh = p.shape();
  const int chunk = (int)p.lay.chunk;
  float* red_o = reinterpret_cast<float*>(smem + (size_t)S * chunk);  // [8 warps][GM][D]
  float* red_m = red_o + kRkWarps * GM * D;                            // [8][GM]
  float* red_l = red_m + kRkWarps * GM;                                // [8][GM]
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kRkWarps);
      rel_cnt[s] = 0;
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  flag_bad_ctx(p);
  block_page_prefix(sh, p.ctx, p.trim, pre, warp_tot);  // ends with __syncthreads
  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  if (W == 0) return;
  const int64_t x_begin = cta_begin(W, p.n_ctas, blockIdx.x);
  const int64_t x_end = cta_begin(W, p.n_ctas, blockIdx.x + 1);
  const int total = (int)(x_end - x_begin);

  // chunk index (page * Hkv + head) of the CTA's page q, -1 for a page id out of range
  auto coord = [&](int q) -> int {
    const int64_t xq = x_begin + q;
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)pre[mid] * p.Hkv <= xq) lo = mid; else hi = mid;
    }
    const int pages = pre[lo + 1] - pre[lo];
    const int64_t off = xq - (int64_t)pre[lo] * p.Hkv;
    const int h = (int)(off / pages), pi = (int)(off % pages);
    const int page = __ldg(p.bt + (int64_t)lo * p.max_pages + pi);
    return (page < 0 || page >= p.num_pages) ? -1 : page * p.Hkv + h;
  };
  // one thread: load the CTA's page q into its stage
  auto issue = [&](int q) {
    const int s = q % S;
    const int z = coord(q);
    const uint32_t fb = smem_u32(&full_bar[s]);
    if (z < 0) {
      stage_ok[s] = 0;
      flag(p.status, NK_DEVFLAG_BAD_PAGE);
      mbar_arrive(fb);
      return;
    }
    stage_ok[s] = 1;
    mbar_arrive_expect_tx(fb, (uint32_t)chunk);
    bulk_load(smem_u32(smem + (size_t)s * chunk), p.pool + (int64_t)z * chunk, (uint32_t)chunk, fb);
  };
  int waited = 0;
  if (tid == 0)
    for (int q0 = 0; q0 < total && q0 < S; ++q0) issue(q0);

  const int nsub = kRkWarps / T;
  const bool active = w < nsub * T;
  const int t = w % T, sub = w / T;
  const int kpw = (p.P + nsub - 1) / nsub;
  const int kgrp = (lane * CPL) / kGroup, vgrp = (lane * CPL) / kRkVGroup;
  int q = 0;  // the CTA's page number
  int64_t x = x_begin;
  Segment seg;
  while (next_segment(sh, pre, x, x_end, seg)) {
    const int L = p.ctx[seg.b] - p.trim;
    const int last = L - T + t;  // last key visible to column t
    float qf[GM][CPL], o[GM][CPL], m[GM], l[GM];
#pragma unroll
    for (int hg = 0; hg < GM; ++hg) {
      m[hg] = -INFINITY;
      l[hg] = 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) { o[hg][j] = 0.f; qf[hg][j] = 0.f; }
      if (hg < G) {
        const uint16_t* qr = p.q + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * D + lane * CPL;
#pragma unroll
        for (int j = 0; j < CPL; ++j) qf[hg][j] = __uint_as_float((uint32_t)__ldg(qr + j) << 16);
      }
#pragma unroll
      for (int h = 1; h < CPL; h <<= 1)
#pragma unroll
        for (int j = 0; j < CPL; ++j)
          if ((j & h) == 0) {
            const float a = qf[hg][j], b = qf[hg][j + h];
            qf[hg][j] = a + b;
            qf[hg][j + h] = a - b;
          }
#pragma unroll
      for (int lb = 1; lb < LPG; lb <<= 1) {
        const bool upper = (lane & lb) != 0;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const float other = __shfl_xor_sync(0xffffffffu, qf[hg][j], lb);
          qf[hg][j] = upper ? other - qf[hg][j] : qf[hg][j] + other;
        }
      }
#pragma unroll
      for (int j = 0; j < CPL; ++j) qf[hg][j] *= 0.125f;
    }
    for (int pi = seg.page_begin; pi < seg.page_end; ++pi, ++q) {
      const int s = q % S;
      bool ok = false;
      if (!abort_flag) {
        ok = mbar_wait(smem_u32(&full_bar[s]), (uint32_t)(q / S) & 1u);
        if (ok) {
          ++waited;
        } else {
          flag(p.status, NK_DEVFLAG_TIMEOUT);
          abort_flag = 1;
        }
      }
      ok = __all_sync(0xffffffffu, ok);  // the warp's shuffles below run only if every lane has the page
      const int k_lo = sub * kpw;
      int k_hi = min(p.P, k_lo + kpw);
      k_hi = min(k_hi, last - pi * p.P + 1);
      if (active && ok && stage_ok[s] && k_lo < k_hi) {
        const uint8_t* st = smem + (size_t)s * chunk;
        const __half* ks_s = reinterpret_cast<const __half*>(st + p.lay.ks);
        const __half* vs_s = reinterpret_cast<const __half*>(st + p.lay.vs);
        for (int k0 = k_lo; k0 < k_hi; k0 += 4) {
          const int nk = min(4, k_hi - k0);
          RkRaw<CPL> raw[4];
          float sc[4][GM], vsc[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k = k0 + (j < nk ? j : nk - 1);  // a repeated key is never used
            raw[j] = rk_load_shared<CPL>(st + k * D + lane * CPL, st + p.lay.vc + k * (D / 2) + lane * (CPL / 2));
            const float ks = __half2float(ks_s[k * (D / kGroup) + kgrp]);
            vsc[j] = __half2float(vs_s[k * (D / kRkVGroup) + vgrp]);
            float kf[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) kf[i] = (float)(int8_t)(raw[j].k[i / 4] >> (8 * (i % 4)));
#pragma unroll
            for (int hg = 0; hg < GM; ++hg) {
              float acc = 0.f;
#pragma unroll
              for (int i = 0; i < CPL; ++i) acc = fmaf(qf[hg][i], kf[i], acc);
              sc[j][hg] = acc * ks;
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int hg = 0; hg < GM; ++hg) sc[j][hg] += __shfl_xor_sync(0xffffffffu, sc[j][hg], off);
#pragma unroll
          for (int hg = 0; hg < GM; ++hg) {
            if (hg >= G) break;
            float mx = m[hg];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              sc[j][hg] *= p.scale2;
              if (j < nk) mx = fmaxf(mx, sc[j][hg]);
            }
            if (mx > m[hg]) {
              const float alpha = exp2f(m[hg] - mx);  // 0 while the row is empty
              l[hg] *= alpha;
#pragma unroll
              for (int i = 0; i < CPL; ++i) o[hg][i] *= alpha;
              m[hg] = mx;
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j >= nk) break;
            float vf[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) vf[i] = (float)((int32_t)(raw[j].v << (28 - 4 * i)) >> 28);
#pragma unroll
            for (int hg = 0; hg < GM; ++hg) {
              if (hg >= G) break;
              const float pw = exp2f(sc[j][hg] - m[hg]);
              l[hg] += pw;
              const float pv = pw * vsc[j];
#pragma unroll
              for (int i = 0; i < CPL; ++i) o[hg][i] = fmaf(pv, vf[i], o[hg][i]);
            }
          }
        }
      }
      // this warp is done with stage s; the last of the 8 warps to release it
      // loads page q + S into it (warps run up to S pages apart)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&empty_bar[s]));
        if (atomicAdd(&rel_cnt[s], 1) == kRkWarps - 1) {
          rel_cnt[s] = 0;
          const int qn = q + S;
          if (qn < total && !abort_flag) {
            if (mbar_wait(smem_u32(&empty_bar[s]), (uint32_t)(q / S) & 1u)) {
              // generic-proxy reads of the stage are ordered before the bulk copy that refills it
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              issue(qn);
            } else {
              flag(p.status, NK_DEVFLAG_TIMEOUT);
              abort_flag = 1;
            }
          }
        }
      }
    }
    // merge the nsub warps of each column (as in the unstaged kernel)
#pragma unroll
    for (int hg = 0; hg < GM; ++hg) {
      if (hg >= G) break;
#pragma unroll
      for (int j = 0; j < CPL; ++j) red_o[(w * GM + hg) * D + lane * CPL + j] = o[hg][j];
      if (lane == 0) {
        red_m[w * GM + hg] = active ? m[hg] : -INFINITY;
        red_l[w * GM + hg] = active ? l[hg] : 0.f;
      }
    }
    __syncthreads();
    const int seg_slot = blockIdx.x + seg.u;
    for (int i = tid; i < M * D; i += blockDim.x) {
      const int r = i / D, c = i % D;
      const int tt = r / G, hg = r % G;
      float mx = -INFINITY;
      for (int sb = 0; sb < nsub; ++sb) mx = fmaxf(mx, red_m[(sb * T + tt) * GM + hg]);
      float lsum = 0.f, acc = 0.f;
      if (mx != -INFINITY) {
        for (int sb = 0; sb < nsub; ++sb) {
          const int ww = sb * T + tt;
          const float mw = red_m[ww * GM + hg];
          if (mw == -INFINITY) continue;
          const float f = exp2f(mw - mx);
          lsum += red_l[ww * GM + hg] * f;
          acc += red_o[(ww * GM + hg) * D + c] * f;
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
  // after a timed-out wait: let the copies that may still be in flight land
  // before the CTA exits (a page is issued only once page - S is released,
  // so at most S pages past the last one waited for)
  if (tid == 0) {
    const int end = min(total, waited + S);
    for (int qq = waited; qq < end; ++qq) (void)mbar_wait(smem_u32(&full_bar[qq % S]), (uint32_t)(qq / S) & 1u);
  }
}

static size_t rk_smem(int D, int G) { return (size_t)kRkWarps * G * (D + 2) * sizeof(float); }

int decode_rk8v4_ctas_per_sm(int D, int G) {
  int n = 0;
  const size_t smem = rk_smem(D, G);
  cudaError_t e;
  if (D == 256) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_rk8v4_kernel<8>, 256, smem);
  else if (D == 128) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_rk8v4_kernel<4>, 256, smem);
  else e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_rk8v4_kernel<2>, 256, smem);
  if (e != cudaSuccess) { (void)cudaGetLastError(); return 1; }
  return n < 1 ? 1 : n;
}

template <int CPL>
static cudaError_t launch_rk_t(const DecodeParams& p, size_t smem, cudaStream_t stream) {
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(decode_rk8v4_kernel<CPL>), (int)smem);
  if (e != cudaSuccess) return e;
  return launch_chained(decode_rk8v4_kernel<CPL>, dim3(p.n_ctas), dim3(256), smem, stream, p);
}

template <int CPL, int GM>
static cudaError_t launch_rk_staged(const DecodeParams& p, int S, cudaStream_t stream) {
  const size_t smem = (size_t)S * p.lay.chunk + rk_staged_fixed_bytes(CPL * 32, GM);
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(decode_rk8v4_staged_kernel<CPL, GM>), (int)smem);
  if (e != cudaSuccess) return e;
  return launch_chained(decode_rk8v4_staged_kernel<CPL, GM>, dim3(p.n_ctas), dim3(256), smem, stream, p, S);
}

template <int CPL>
static cudaError_t launch_rk_staged_g(const DecodeParams& p, int S, cudaStream_t stream) {
  if (p.G <= 2) return launch_rk_staged<CPL, 2>(p, S, stream);
  if (p.G <= 6) return launch_rk_staged<CPL, 6>(p, S, stream);
  return launch_rk_staged<CPL, 8>(p, S, stream);
}

cudaError_t launch_decode_rk8v4(const DecodeParams& p, cudaStream_t stream) {
  const int GM = p.G <= 2 ? 2 : (p.G <= 6 ? 6 : 8);
  const int S = rk_staged_stages((int)p.lay.chunk, p.D, GM);
  if (S >= 3) {
    if (p.D == 256) return launch_rk_staged_g<8>(p, S, stream);
    if (p.D == 128) return launch_rk_staged_g<4>(p, S, stream);
    return launch_rk_staged_g<2>(p, S, stream);
  }
  // pages too large for a ring of three: the unstaged kernel
  const size_t smem = rk_smem(p.D, p.G);
  if (p.D == 256) return launch_rk_t<8>(p, smem, stream);
  if (p.D == 128) return launch_rk_t<4>(p, smem, stream);
  return launch_rk_t<2>(p, smem, stream);
}

}  // namespace nk
