/*
 * oracle.c -- plain fp64 CPU oracle for the paged INT8 group-64 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/, the smoke check and the
 * benchmark's CPU-baseline leg; never by the CUDA product path. Shares no code
 * with it. See oracle.h for the definitions and the readings of the pages.
 *
 * Written for obviousness, not speed: each step follows the definition in the
 * order it is stated, with no blocking, fusion or reordering. The only
 * parallelism is an OpenMP loop over independent units (tokens, query rows).
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC
 */
#include "oracle.h"

#include <fenv.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GROUP 64 /* channels per quantization group ("INT8 group-64") */

static void ensure_round_to_nearest(void) {
  if (fegetround() != FE_TONEAREST) fesetround(FE_TONEAREST);
}

double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t oracle_double_to_bf16(double x) {
  /* bf16: 8 significant bits, exponent range of fp32, subnormal quantum 2^-133. */
  ensure_round_to_nearest();
  if (isnan(x)) return 0x7fc0;
  double r;
  if (x == 0.0) {
    r = x;
  } else {
    int e;
    double m = frexp(x, &e); /* x = m * 2^e, 0.5 <= |m| < 1 */
    if (e - 1 < -126) {
      r = nearbyint(ldexp(x, 133)) * ldexp(1.0, -133);
    } else {
      r = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    if (fabs(r) >= ldexp(1.0, 128)) r = copysign(INFINITY, x);
  }
  float f = (float)r; /* exact: r is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

void oracle_round_bf16(const double* x, size_t n, uint16_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = oracle_double_to_bf16(x[i]);
}

float oracle_quantize_group(const uint16_t* x, int n, int8_t* q) {
  ensure_round_to_nearest();
  /* absmax of the group (bf16 widens exactly) */
  double a = 0.0;
  for (int i = 0; i < n; ++i) {
    double v = fabs(oracle_bf16_to_double(x[i]));
    if (v > a) a = v;
  }
  /* s = a / 127 in fp32. The fp64 quotient rounded once more to fp32 is the
   * correctly rounded fp32 quotient (53 >= 2*24 + 2). */
  float s = (a == 0.0) ? 1.0f : (float)(a / 127.0);
  for (int i = 0; i < n; ++i) {
    /* fp32 quotient x / s, again exact through fp64 */
    float r = (float)(oracle_bf16_to_double(x[i]) / (double)s);
    double k = nearbyint((double)r); /* ties to even */
    if (k > 127.0) k = 127.0;
    if (k < -127.0) k = -127.0;
    q[i] = (int8_t)k;
  }
  return s;
}

size_t oracle_chunk_bytes(int page_size, int head_dim) {
  size_t P = (size_t)page_size, D = (size_t)head_dim, g = D / GROUP;
  return P * D + P * g * sizeof(float) + P * D + P * g * sizeof(float);
}

size_t oracle_pool_bytes(int num_pages, int page_size, int num_kv_heads, int head_dim) {
  return (size_t)num_pages * (size_t)num_kv_heads * oracle_chunk_bytes(page_size, head_dim);
}

/* Addresses inside one (page, head) chunk. */
typedef struct {
  int8_t* kc;
  float* ks;
  int8_t* vc;
  float* vs;
} chunk_ptrs;

static chunk_ptrs chunk_at(const uint8_t* pool, int page, int head, int num_kv_heads, int P, int D) {
  size_t g = (size_t)D / GROUP;
  uint8_t* base = (uint8_t*)pool + ((size_t)page * num_kv_heads + head) * oracle_chunk_bytes(P, D);
  chunk_ptrs c;
  c.kc = (int8_t*)base;
  c.ks = (float*)(base + (size_t)P * D);
  c.vc = (int8_t*)(base + (size_t)P * D + (size_t)P * g * sizeof(float));
  c.vs = (float*)(base + 2 * (size_t)P * D + (size_t)P * g * sizeof(float));
  return c;
}

int oracle_kv_append(uint8_t* pool, int num_pages, int page_size, int num_kv_heads, int head_dim,
                     const int32_t* block_table, int max_pages, const int32_t* start_pos,
                     const int32_t* cu_new, int B, const uint16_t* k, const uint16_t* v) {
  const int P = page_size, D = head_dim, H = num_kv_heads, g = D / GROUP;
  const int total = cu_new[B];
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (int j = 0; j < total; ++j) {
    /* which sequence owns new row j */
    int b = 0;
    while (b + 1 <= B && cu_new[b + 1] <= j) ++b;
    long pos = (long)start_pos[b] + (j - cu_new[b]);
    if (pos < 0 || pos >= (long)max_pages * P) { ++bad; continue; }
    int page = block_table[(size_t)b * max_pages + pos / P];
    if (page < 0 || page >= num_pages) { ++bad; continue; }
    int slot = (int)(pos % P);
    for (int h = 0; h < H; ++h) {
      chunk_ptrs c = chunk_at(pool, page, h, H, P, D);
      const uint16_t* krow = k + ((size_t)j * H + h) * D;
      const uint16_t* vrow = v + ((size_t)j * H + h) * D;
      for (int gr = 0; gr < g; ++gr) {
        c.ks[(size_t)slot * g + gr] = oracle_quantize_group(krow + gr * GROUP, GROUP, c.kc + (size_t)slot * D + gr * GROUP);
        c.vs[(size_t)slot * g + gr] = oracle_quantize_group(vrow + gr * GROUP, GROUP, c.vc + (size_t)slot * D + gr * GROUP);
      }
    }
  }
  return bad;
}

int oracle_attention_row(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                         int head_dim, const int32_t* block_table, int max_pages,
                         const int32_t* ctx_lens, int B, int T, int num_q_heads,
                         const uint16_t* q, double sm_scale, int b, int t, int i,
                         int key_begin, int key_end, double* o, double* lse) {
  const int P = page_size, D = head_dim, Hq = num_q_heads, H = num_kv_heads, g = D / GROUP;
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  *lse = -INFINITY;
  if (b < 0 || b >= B || t < 0 || t >= T || i < 0 || i >= Hq || Hq % H != 0) return 1;
  const int G = Hq / H;   /* q-heads per kv-head */
  const int h = i / G;    /* q-head i reads kv-head i / G */
  const long L = ctx_lens[b];
  if (L < T || L > (long)max_pages * P) return 1;
  const long last = L - T + t; /* last key this query column may see */
  long n0 = key_begin < 0 ? 0 : key_begin;
  long n1 = (long)key_end < last + 1 ? (long)key_end : last + 1;
  if (n1 <= n0) return 0;

  const uint16_t* qrow = q + (((size_t)b * T + t) * Hq + i) * D;
  double* z = (double*)malloc(sizeof(double) * (size_t)(n1 - n0));
  double* kd = (double*)malloc(sizeof(double) * (size_t)D);
  if (!z || !kd) { free(z); free(kd); return 1; }
  int err = 0;

  /* scores z_n = tau * sum_c q_c * khat_{n,c}, khat = code * scale (exact in fp64) */
  for (long n = n0; n < n1; ++n) {
    int page = block_table[(size_t)b * max_pages + n / P];
    if (page < 0 || page >= num_pages) { err = 1; break; }
    int slot = (int)(n % P);
    chunk_ptrs c = chunk_at(pool, page, h, H, P, D);
    for (int ch = 0; ch < D; ++ch)
      kd[ch] = (double)c.kc[(size_t)slot * D + ch] * (double)c.ks[(size_t)slot * g + ch / GROUP];
    double dot = 0.0;
    for (int ch = 0; ch < D; ++ch) dot += oracle_bf16_to_double(qrow[ch]) * kd[ch];
    z[n - n0] = sm_scale * dot;
  }
  if (err) { free(z); free(kd); return 1; }

  /* softmax over the visible keys, then the weighted mean of vhat */
  double m = -INFINITY;
  for (long n = n0; n < n1; ++n) if (z[n - n0] > m) m = z[n - n0];
  double l = 0.0;
  for (long n = n0; n < n1; ++n) {
    double w = exp(z[n - n0] - m);
    int page = block_table[(size_t)b * max_pages + n / P];
    int slot = (int)(n % P);
    chunk_ptrs c = chunk_at(pool, page, h, H, P, D);
    for (int ch = 0; ch < D; ++ch)
      o[ch] += w * ((double)c.vc[(size_t)slot * D + ch] * (double)c.vs[(size_t)slot * g + ch / GROUP]);
    l += w;
  }
  for (int ch = 0; ch < D; ++ch) o[ch] /= l;
  *lse = m + log(l);
  free(z);
  free(kd);
  return 0;
}

int oracle_paged_attention(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                           int head_dim, const int32_t* block_table, int max_pages,
                           const int32_t* ctx_lens, int B, int T, int num_q_heads,
                           const uint16_t* q, double sm_scale, double* out, double* lse) {
  const long rows = (long)B * T * num_q_heads;
  const int D = head_dim;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (long r = 0; r < rows; ++r) {
    int i = (int)(r % num_q_heads);
    int t = (int)((r / num_q_heads) % T);
    int b = (int)(r / ((long)num_q_heads * T));
    double row_lse;
    bad += oracle_attention_row(pool, num_pages, page_size, num_kv_heads, head_dim, block_table,
                                max_pages, ctx_lens, B, T, num_q_heads, q, sm_scale, b, t, i, 0,
                                0x7fffffff, out + (size_t)r * D, &row_lse);
    if (lse) lse[r] = row_lse;
  }
  return bad;
}

void oracle_combine(const float* part_o, const float* part_lse, int S, int R, int D, double* out) {
  for (int r = 0; r < R; ++r) {
    double m = -INFINITY;
    for (int s = 0; s < S; ++s)
      if ((double)part_lse[(size_t)s * R + r] > m) m = part_lse[(size_t)s * R + r];
    double* o = out + (size_t)r * D;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    if (m == -INFINITY) continue; /* no visible key in any split */
    double wsum = 0.0;
    for (int s = 0; s < S; ++s) {
      double ls = part_lse[(size_t)s * R + r];
      if (ls == -INFINITY) continue;
      double w = exp(ls - m);
      for (int c = 0; c < D; ++c) o[c] += w * (double)part_o[((size_t)s * R + r) * D + c];
      wsum += w;
    }
    for (int c = 0; c < D; ++c) o[c] /= wsum;
  }
}

/* ===========================================================================
 * rk8v4 ("NInfer-3090" README, "RotorQuant KV (rk8v4)"); readings in oracle.h.
 * ======================================================================== */

uint16_t oracle_double_to_f16(double x) {
  /* fp16: 11 significant bits, normal exponents -14 .. 15, subnormal quantum 2^-24. */
  ensure_round_to_nearest();
  if (isnan(x)) return 0x7e00;
  const uint16_t sign = signbit(x) ? 0x8000 : 0;
  const double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
  double r;
  if (e - 1 < -14) {
    r = nearbyint(ldexp(a, 24)) * ldexp(1.0, -24);
  } else {
    r = ldexp(nearbyint(ldexp(a, 11 - e)), e - 11);
  }
  if (r > 65504.0) return sign | 0x7c00;
  if (r < ldexp(1.0, -14)) return sign | (uint16_t)ldexp(r, 24); /* subnormal (or zero) */
  int e2;
  const double m2 = frexp(r, &e2); /* r = m2 * 2^e2 */
  const uint16_t exp_field = (uint16_t)(e2 - 1 + 15);
  const uint16_t mant = (uint16_t)ldexp(2.0 * m2 - 1.0, 10);
  return sign | (uint16_t)(exp_field << 10) | mant;
}

double oracle_f16_to_double(uint16_t bits) {
  const int e = (bits >> 10) & 0x1f, m = bits & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024 + m), e - 25);
  return (bits & 0x8000) ? -v : v;
}

/* The rotation of one key group, y = RN_fp32(H64 x / 8), follows its plain
 * definition: each output is the exact signed sum of the 64 inputs, rounded
 * once to fp32 (round to nearest, ties to even).
 *
 * Exact sum. A finite bf16 value is an integer multiple of 2^-133 (the
 * subnormal quantum): 128 + m times 2^(e - 1) units for a normal pattern
 * (exponent field e, 7-bit fraction m), m units for a subnormal one. The
 * multiples are added as base-2^16 digits held in 64-bit cells, so that no
 * partial sum is ever rounded (|x| < 2^128 and 64 terms need fewer than 268
 * bits; RK_DIGITS digits hold 320). */
#define RK_DIGITS 20

static void rk_add_term(int64_t* acc, uint16_t bits, int negate) {
  const int e = (bits >> 7) & 0xff, m = bits & 0x7f;
  const int64_t units = e == 0 ? m : 128 + m; /* times 2^shift units of 2^-133 */
  const int shift = e == 0 ? 0 : e - 1;
  const int64_t v = units << (shift % 16);     /* below 2^23 */
  const int64_t sgn = ((bits & 0x8000) != 0) != (negate != 0) ? -1 : 1;
  acc[shift / 16] += sgn * (v % 65536);
  acc[shift / 16 + 1] += sgn * (v / 65536);
}

/* Carry every cell into the next one, so that cells 0 .. RK_DIGITS-2 lie in
 * [0, 2^16) and the last one holds the sign of the whole number. */
static void rk_carry(int64_t* acc) {
  for (int k = 0; k < RK_DIGITS - 1; ++k) {
    int64_t c = acc[k] / 65536;
    if (acc[k] - c * 65536 < 0) c -= 1; /* floor division */
    acc[k] -= c * 65536;
    acc[k + 1] += c;
  }
}

static int rk_bit(const int64_t* mag, int pos) {
  return pos < 0 ? 0 : (int)((mag[pos / 16] >> (pos % 16)) & 1);
}

/* RN_fp32(S * 2^-136) for the integer S held in acc: 2^-133 units, and the
 * 1/8 of the rotation. */
static float rk_round_fp32(int64_t* acc) {
  rk_carry(acc);
  const int negative = acc[RK_DIGITS - 1] < 0;
  if (negative) {
    for (int k = 0; k < RK_DIGITS; ++k) acc[k] = -acc[k];
    rk_carry(acc);
  }
  int top = -1; /* position of the leading 1 bit of |S| */
  for (int pos = 16 * RK_DIGITS - 1; pos >= 0 && top < 0; --pos)
    if (rk_bit(acc, pos)) top = pos;
  if (top < 0) return 0.0f;
  double mant = 0.0; /* the 24 leading bits (all of them when there are fewer) */
  const int low = top - 23 > 0 ? top - 23 : 0;
  for (int pos = top; pos >= low; --pos) mant = 2.0 * mant + rk_bit(acc, pos);
  if (top >= 24) {
    const int guard = rk_bit(acc, low - 1);
    int sticky = 0;
    for (int pos = 0; pos < low - 1; ++pos) sticky |= rk_bit(acc, pos);
    if (guard && (sticky || fmod(mant, 2.0) == 1.0)) mant += 1.0; /* half up only to even */
  }
  /* mant * 2^(low - 136) is exact in double and, by construction, an fp32
   * number (or past the fp32 range, which converts to infinity) */
  const double y = ldexp(mant, low - 136);
  if (y >= ldexp(1.0, 128)) return negative ? -INFINITY : INFINITY;
  return (float)(negative ? -y : y);
}

void oracle_rk_rotate64(const uint16_t* x, float* y) {
  for (int r = 0; r < GROUP; ++r) {
    int64_t acc[RK_DIGITS];
    for (int k = 0; k < RK_DIGITS; ++k) acc[k] = 0;
    for (int j = 0; j < GROUP; ++j) rk_add_term(acc, x[j], __builtin_popcount((unsigned)(r & j)) & 1);
    y[r] = rk_round_fp32(acc);
  }
}

/* fp16 scale bits for a group absmax a and code bound qmax: RN_fp16(a / qmax),
 * 1 when that is 0, 65504 when it is past the fp16 range. */
static uint16_t rk_scale_bits(double a, double qmax) {
  uint16_t sb = oracle_double_to_f16(a / qmax);
  if ((sb & 0x7fff) == 0) sb = 0x3c00;
  else if ((sb & 0x7fff) == 0x7c00) sb = 0x7bff;
  return sb;
}

uint16_t oracle_rk_quantize_k(const float* y, int8_t* q) {
  ensure_round_to_nearest();
  double a = 0.0;
  for (int i = 0; i < GROUP; ++i) {
    const double v = fabs((double)y[i]);
    if (v > a) a = v;
  }
  const uint16_t sb = rk_scale_bits(a, 127.0);
  const double s = oracle_f16_to_double(sb);
  for (int i = 0; i < GROUP; ++i) {
    const float r = (float)((double)y[i] / s); /* the fp32 quotient (53 >= 2*24 + 2) */
    double k = nearbyint((double)r);
    if (k > 127.0) k = 127.0;
    if (k < -127.0) k = -127.0;
    q[i] = (int8_t)k;
  }
  return sb;
}

#define VGROUP 32 /* value channels per scale */

uint16_t oracle_rk_quantize_v(const uint16_t* x, uint8_t* packed) {
  ensure_round_to_nearest();
  double a = 0.0;
  for (int i = 0; i < VGROUP; ++i) {
    const double v = fabs(oracle_bf16_to_double(x[i]));
    if (v > a) a = v;
  }
  const uint16_t sb = rk_scale_bits(a, 7.0);
  const double s = oracle_f16_to_double(sb);
  int q[VGROUP];
  for (int i = 0; i < VGROUP; ++i) {
    const float r = (float)(oracle_bf16_to_double(x[i]) / s);
    double k = nearbyint((double)r);
    if (k > 7.0) k = 7.0;
    if (k < -7.0) k = -7.0;
    q[i] = (int)k;
  }
  for (int j = 0; j < VGROUP / 2; ++j) packed[j] = (uint8_t)((q[2 * j] & 0xf) | ((q[2 * j + 1] & 0xf) << 4));
  return sb;
}

size_t oracle_rk_chunk_bytes(int page_size, int head_dim) {
  size_t P = (size_t)page_size, D = (size_t)head_dim;
  return P * D + P * (D / GROUP) * 2 + P * (D / 2) + P * (D / VGROUP) * 2;
}

size_t oracle_rk_pool_bytes(int num_pages, int page_size, int num_kv_heads, int head_dim) {
  return (size_t)num_pages * (size_t)num_kv_heads * oracle_rk_chunk_bytes(page_size, head_dim);
}

typedef struct {
  int8_t* kc;   /* [P][D] */
  uint16_t* ks; /* [P][D/64] fp16 bits */
  uint8_t* vc;  /* [P][D/2] */
  uint16_t* vs; /* [P][D/32] fp16 bits */
} rk_chunk_ptrs;

static rk_chunk_ptrs rk_chunk_at(const uint8_t* pool, int page, int head, int num_kv_heads, int P, int D) {
  uint8_t* base = (uint8_t*)pool + ((size_t)page * num_kv_heads + head) * oracle_rk_chunk_bytes(P, D);
  const size_t ks = (size_t)P * D, vc = ks + (size_t)P * (D / GROUP) * 2, vs = vc + (size_t)P * (D / 2);
  rk_chunk_ptrs c;
  c.kc = (int8_t*)base;
  c.ks = (uint16_t*)(base + ks);
  c.vc = base + vc;
  c.vs = (uint16_t*)(base + vs);
  return c;
}

int oracle_rk_append(uint8_t* pool, int num_pages, int page_size, int num_kv_heads, int head_dim,
                     const int32_t* block_table, int max_pages, const int32_t* start_pos,
                     const int32_t* cu_new, int B, const uint16_t* k, const uint16_t* v) {
  const int P = page_size, D = head_dim, H = num_kv_heads;
  const int total = cu_new[B];
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (int j = 0; j < total; ++j) {
    int b = 0;
    while (b + 1 <= B && cu_new[b + 1] <= j) ++b;
    long pos = (long)start_pos[b] + (j - cu_new[b]);
    if (pos < 0 || pos >= (long)max_pages * P) { ++bad; continue; }
    int page = block_table[(size_t)b * max_pages + pos / P];
    if (page < 0 || page >= num_pages) { ++bad; continue; }
    int slot = (int)(pos % P);
    for (int h = 0; h < H; ++h) {
      rk_chunk_ptrs c = rk_chunk_at(pool, page, h, H, P, D);
      const uint16_t* krow = k + ((size_t)j * H + h) * D;
      const uint16_t* vrow = v + ((size_t)j * H + h) * D;
      for (int gr = 0; gr < D / GROUP; ++gr) {
        float y[GROUP];
        oracle_rk_rotate64(krow + gr * GROUP, y);
        c.ks[(size_t)slot * (D / GROUP) + gr] = oracle_rk_quantize_k(y, c.kc + (size_t)slot * D + gr * GROUP);
      }
      for (int gr = 0; gr < D / VGROUP; ++gr)
        c.vs[(size_t)slot * (D / VGROUP) + gr] =
            oracle_rk_quantize_v(vrow + gr * VGROUP, c.vc + (size_t)slot * (D / 2) + gr * (VGROUP / 2));
    }
  }
  return bad;
}

/* signed 4-bit code of channel ch from a packed value row */
static int rk_nibble(const uint8_t* row, int ch) {
  int n = (row[ch / 2] >> (4 * (ch & 1))) & 0xf;
  return n >= 8 ? n - 16 : n;
}

int oracle_rk_attention_row(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                            int head_dim, const int32_t* block_table, int max_pages,
                            const int32_t* ctx_lens, int B, int T, int num_q_heads,
                            const uint16_t* q, double sm_scale, int b, int t, int i,
                            int key_begin, int key_end, double* o, double* lse) {
  const int P = page_size, D = head_dim, Hq = num_q_heads, H = num_kv_heads;
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  *lse = -INFINITY;
  if (b < 0 || b >= B || t < 0 || t >= T || i < 0 || i >= Hq || Hq % H != 0) return 1;
  const int G = Hq / H;
  const int h = i / G;
  const long L = ctx_lens[b];
  if (L < T || L > (long)max_pages * P) return 1;
  const long last = L - T + t;
  long n0 = key_begin < 0 ? 0 : key_begin;
  long n1 = (long)key_end < last + 1 ? (long)key_end : last + 1;
  if (n1 <= n0) return 0;

  /* the query row in the rotated basis: (R q)_r = sum_j (-1)^popcount(r & j) q_j / 8 per group */
  const uint16_t* qrow = q + (((size_t)b * T + t) * Hq + i) * D;
  double* qr = (double*)malloc(sizeof(double) * (size_t)D);
  double* z = (double*)malloc(sizeof(double) * (size_t)(n1 - n0));
  if (!qr || !z) { free(qr); free(z); return 1; }
  for (int g0 = 0; g0 < D; g0 += GROUP)
    for (int r = 0; r < GROUP; ++r) {
      double acc = 0.0;
      for (int jj = 0; jj < GROUP; ++jj) {
        const double x = oracle_bf16_to_double(qrow[g0 + jj]);
        acc += (__builtin_popcount((unsigned)(r & jj)) & 1) ? -x : x;
      }
      qr[g0 + r] = acc / 8.0;
    }
  int err = 0;
  for (long n = n0; n < n1; ++n) {
    int page = block_table[(size_t)b * max_pages + n / P];
    if (page < 0 || page >= num_pages) { err = 1; break; }
    int slot = (int)(n % P);
    rk_chunk_ptrs c = rk_chunk_at(pool, page, h, H, P, D);
    double dot = 0.0;
    for (int ch = 0; ch < D; ++ch) {
      const double khat = (double)c.kc[(size_t)slot * D + ch] *
                          oracle_f16_to_double(c.ks[(size_t)slot * (D / GROUP) + ch / GROUP]);
      dot += qr[ch] * khat;
    }
    z[n - n0] = sm_scale * dot;
  }
  if (err) { free(qr); free(z); return 1; }
  double m = -INFINITY;
  for (long n = n0; n < n1; ++n) if (z[n - n0] > m) m = z[n - n0];
  double l = 0.0;
  for (long n = n0; n < n1; ++n) {
    double w = exp(z[n - n0] - m);
    int page = block_table[(size_t)b * max_pages + n / P];
    int slot = (int)(n % P);
    rk_chunk_ptrs c = rk_chunk_at(pool, page, h, H, P, D);
    const uint8_t* vrow = c.vc + (size_t)slot * (D / 2);
    for (int ch = 0; ch < D; ++ch)
      o[ch] += w * ((double)rk_nibble(vrow, ch) * oracle_f16_to_double(c.vs[(size_t)slot * (D / VGROUP) + ch / VGROUP]));
    l += w;
  }
  for (int ch = 0; ch < D; ++ch) o[ch] /= l;
  *lse = m + log(l);
  free(qr);
  free(z);
  return 0;
}

int oracle_rk_paged_attention(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                              int head_dim, const int32_t* block_table, int max_pages,
                              const int32_t* ctx_lens, int B, int T, int num_q_heads,
                              const uint16_t* q, double sm_scale, double* out, double* lse) {
  const long rows = (long)B * T * num_q_heads;
  const int D = head_dim;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (long r = 0; r < rows; ++r) {
    int i = (int)(r % num_q_heads);
    int t = (int)((r / num_q_heads) % T);
    int b = (int)(r / ((long)num_q_heads * T));
    double row_lse;
    bad += oracle_rk_attention_row(pool, num_pages, page_size, num_kv_heads, head_dim, block_table,
                                   max_pages, ctx_lens, B, T, num_q_heads, q, sm_scale, b, t, i, 0,
                                   0x7fffffff, out + (size_t)r * D, &row_lse);
    if (lse) lse[r] = row_lse;
  }
  return bad;
}

/* ===========================================================================
 * The pages' own INT8 layout (fp16 scales) and the bf16 baseline; readings
 * in oracle.h.
 * ======================================================================== */

uint16_t oracle_i8h_quantize_group(const uint16_t* x, int8_t* q) {
  /* the rule of the rk8v4 keys (fp16 scale of absmax / 127, fp32 quotients),
   * applied to the bf16 values as they are: no rotation */
  float y[GROUP];
  for (int i = 0; i < GROUP; ++i) y[i] = (float)oracle_bf16_to_double(x[i]);
  return oracle_rk_quantize_k(y, q);
}

size_t oracle_i8h_chunk_bytes(int page_size, int head_dim) {
  size_t P = (size_t)page_size, D = (size_t)head_dim;
  return 2 * (P * D + P * (D / GROUP) * 2);
}

size_t oracle_bf16kv_chunk_bytes(int page_size, int head_dim) {
  return 2 * (size_t)page_size * (size_t)head_dim * 2;
}

static size_t fmt_chunk_bytes(int fmt, int P, int D) {
  return fmt == 1 ? oracle_i8h_chunk_bytes(P, D) : oracle_bf16kv_chunk_bytes(P, D);
}

int oracle_fmt_append(int fmt, uint8_t* pool, int num_pages, int page_size, int num_kv_heads, int head_dim,
                      const int32_t* block_table, int max_pages, const int32_t* start_pos,
                      const int32_t* cu_new, int B, const uint16_t* k, const uint16_t* v) {
  const int P = page_size, D = head_dim, H = num_kv_heads, g = D / GROUP;
  const int total = cu_new[B];
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (int j = 0; j < total; ++j) {
    int b = 0;
    while (b + 1 <= B && cu_new[b + 1] <= j) ++b;
    long pos = (long)start_pos[b] + (j - cu_new[b]);
    if (pos < 0 || pos >= (long)max_pages * P) { ++bad; continue; }
    int page = block_table[(size_t)b * max_pages + pos / P];
    if (page < 0 || page >= num_pages) { ++bad; continue; }
    int slot = (int)(pos % P);
    for (int h = 0; h < H; ++h) {
      uint8_t* base = pool + ((size_t)page * H + h) * fmt_chunk_bytes(fmt, P, D);
      const uint16_t* krow = k + ((size_t)j * H + h) * D;
      const uint16_t* vrow = v + ((size_t)j * H + h) * D;
      if (fmt == 1) {
        /* Kc | Ks | Vc | Vs */
        const size_t half = (size_t)P * D + (size_t)P * g * 2;
        for (int gr = 0; gr < g; ++gr) {
          uint16_t sk = oracle_i8h_quantize_group(krow + gr * GROUP, (int8_t*)(base + (size_t)slot * D + gr * GROUP));
          uint16_t sv = oracle_i8h_quantize_group(vrow + gr * GROUP,
                                                  (int8_t*)(base + half + (size_t)slot * D + gr * GROUP));
          memcpy(base + (size_t)P * D + ((size_t)slot * g + gr) * 2, &sk, 2);
          memcpy(base + half + (size_t)P * D + ((size_t)slot * g + gr) * 2, &sv, 2);
        }
      } else {
        /* K | V, the bf16 rows as they are */
        memcpy(base + (size_t)slot * D * 2, krow, (size_t)D * 2);
        memcpy(base + (size_t)P * D * 2 + (size_t)slot * D * 2, vrow, (size_t)D * 2);
      }
    }
  }
  return bad;
}

/* dequantized (or widened) K and V value of channel ch of a key's slot */
static double fmt_kv(int fmt, const uint8_t* base, int P, int D, int slot, int ch, int want_v) {
  if (fmt == 1) {
    const size_t g = (size_t)D / GROUP, half = (size_t)P * D + (size_t)P * g * 2;
    const uint8_t* part = base + (want_v ? half : 0);
    uint16_t sb;
    memcpy(&sb, part + (size_t)P * D + ((size_t)slot * g + ch / GROUP) * 2, 2);
    return (double)(int8_t)part[(size_t)slot * D + ch] * oracle_f16_to_double(sb);
  }
  uint16_t bits;
  memcpy(&bits, base + (want_v ? (size_t)P * D * 2 : 0) + ((size_t)slot * D + ch) * 2, 2);
  return oracle_bf16_to_double(bits);
}

int oracle_fmt_paged_attention(int fmt, const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                               int head_dim, const int32_t* block_table, int max_pages,
                               const int32_t* ctx_lens, int B, int T, int num_q_heads,
                               const uint16_t* q, double sm_scale, double* out, double* lse) {
  const int P = page_size, D = head_dim, Hq = num_q_heads, H = num_kv_heads;
  const long rows = (long)B * T * Hq;
  int bad = 0;
  if (Hq % H != 0) return (int)rows;
  const int G = Hq / H;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (long r = 0; r < rows; ++r) {
    const int i = (int)(r % Hq), t = (int)((r / Hq) % T), b = (int)(r / ((long)Hq * T));
    const int h = i / G;
    double* o = out + (size_t)r * D;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    if (lse) lse[r] = -INFINITY;
    const long L = ctx_lens[b];
    if (L < T || L > (long)max_pages * P) { ++bad; continue; }
    const long n1 = L - T + t + 1; /* keys 0 .. L - T + t are visible */
    const uint16_t* qrow = q + (((size_t)b * T + t) * Hq + i) * D;
    double* z = (double*)malloc(sizeof(double) * (size_t)n1);
    if (!z) { ++bad; continue; }
    int err = 0;
    for (long n = 0; n < n1 && !err; ++n) {
      const int page = block_table[(size_t)b * max_pages + n / P];
      if (page < 0 || page >= num_pages) { err = 1; break; }
      const uint8_t* base = pool + ((size_t)page * H + h) * fmt_chunk_bytes(fmt, P, D);
      double dot = 0.0;
      for (int ch = 0; ch < D; ++ch) dot += oracle_bf16_to_double(qrow[ch]) * fmt_kv(fmt, base, P, D, (int)(n % P), ch, 0);
      z[n] = sm_scale * dot;
    }
    if (err) { free(z); ++bad; continue; }
    double m = -INFINITY;
    for (long n = 0; n < n1; ++n) if (z[n] > m) m = z[n];
    double l = 0.0;
    for (long n = 0; n < n1; ++n) {
      const double w = exp(z[n] - m);
      const int page = block_table[(size_t)b * max_pages + n / P];
      const uint8_t* base = pool + ((size_t)page * H + h) * fmt_chunk_bytes(fmt, P, D);
      for (int ch = 0; ch < D; ++ch) o[ch] += w * fmt_kv(fmt, base, P, D, (int)(n % P), ch, 1);
      l += w;
    }
    for (int ch = 0; ch < D; ++ch) o[ch] /= l;
    if (lse) lse[r] = m + log(l);
    free(z);
  }
  return bad;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
