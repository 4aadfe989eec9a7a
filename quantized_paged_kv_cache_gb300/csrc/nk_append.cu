// nk_append.cu -- kv_cache_append: quantize new bf16 K/V rows into int8
// 64-channel groups and scatter them into their pages.
//
// The Op that owns KV quantization and stores values from the bf16 source
// directly ("NInfer-3090" README, introduction and "RotorQuant KV (rk8v4)");
// INT8 group-64 storage ("NInfer" README, capability list). Rule per group:
//   a = max|x|, s = fp32(a / 127) (1 if a = 0), q = clamp(rne(fp32(x / s)), +-127).
//
// Two kernels. Small appends (decode and verify steps, up to 4,096 groups):
// one thread per group, loading directly. Larger ones: a bandwidth-bound
// streaming scatter, a persistent grid that streams chunks of consecutive K
// and V rows into shared memory with bulk asynchronous copies, quantizes one
// 64-channel group per thread and stores the codes with coalesced writes;
// there the group's scale and its reciprocal come from a per-block table
// indexed by the bf16 mantissa of the absmax. Both form x / s exactly from
// y = RN(1/s) by one fma refinement, so every element takes the same short
// path without a division.
#include "nk_common.cuh"
#include "nk_ptx.cuh"

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
  int p_shift, hkv_shift;  // log2 of P and Hkv when they are powers of two, else -1
};

// Per-block table of the group scale and its reciprocal by bf16 mantissa:
// for a = (1 + m/128) * 2^E, s = fp32(a / 127) = fp32((1 + m/128) / 127) * 2^E
// and RN(1/s) = RN(1/s_m) * 2^-E exactly, since scaling by a power of two
// commutes with rounding while every value stays a normal number. The table
// holds the bit patterns of s_m and RN(1/s_m); a group applies its exponent
// E by integer addition on those patterns.
struct ScaleEntry {
  uint32_t s_bits, y_bits;
};
constexpr int kMinFastExp = 40;  // biased exponent of a: below it (s < 2^-93) every element divides

// IEEE path for one element: fp32 quotient, clamp, round half to even. Kept
// out of line: only groups of magnitude below 2^-87 take it.
__device__ __noinline__ uint32_t quantize_exact(float x, float s) {
  float e = __fdiv_rn(x, s);
  e = fminf(fmaxf(e, -127.f), 127.f);
  return (uint32_t)__float2int_rn(e) & 0xffu;
}

// The 64 codes of a group from its scale s and y = RN(1/s) (the quotient
// steps described below, on pairs of values: each fp32x2 operation rounds its
// two lanes as the scalar one does).
__device__ __forceinline__ void codes64(const uint32_t (&w)[32], uint32_t (&packed)[16], float s, float y) {
  const float2 y2 = make_float2(y, y), ns2 = make_float2(-s, -s), mg2 = make_float2(12582912.f, 12582912.f);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float2 xa = make_float2(bf16_lo(w[2 * k]), bf16_hi(w[2 * k]));
    const float2 xb = make_float2(bf16_lo(w[2 * k + 1]), bf16_hi(w[2 * k + 1]));
    const float2 qa0 = __fmul2_rn(xa, y2), qb0 = __fmul2_rn(xb, y2);
    const float2 ra = __ffma2_rn(ns2, qa0, xa), rb = __ffma2_rn(ns2, qb0, xb);
    const float2 ta = __fadd2_rn(__ffma2_rn(ra, y2, qa0), mg2), tb = __fadd2_rn(__ffma2_rn(rb, y2, qb0), mg2);
    packed[k] = __byte_perm(__byte_perm(__float_as_uint(ta.x), __float_as_uint(ta.y), 0x0040),
                            __byte_perm(__float_as_uint(tb.x), __float_as_uint(tb.y), 0x0040), 0x5410);
  }
}

// Quantize one 64-channel group held as 32 raw bf16 pairs; returns the
// group's scale and writes the 64 int8 codes packed into 16 words.
//
// absmax: for finite values |x| orders like the bf16 bit pattern with the sign
// cleared, so it is a 16-bit unsigned max over the pairs. Quotient: with
// y = RN(1/s), q0 = RN(x * y) is within one ulp of x / s; the remainder
// r = x - s * q0 is exact in one fma, and RN(q0 + r * y) is the correctly
// rounded quotient (Markstein's theorem on division by fused multiply-add;
// tests/quotient_check.c also replays these steps over every bf16 (group max,
// element) pair of the exponents that matter). t = q + 1.5 * 2^23 then rounds
// q to an integer (ties to even) whose two's-complement low byte is the low
// byte of t's bits; |q| <= 127 needs no clamp.
// kTable: s and RN(1/s) from the block's table; otherwise by IEEE division
// (the same values: the table holds them for every mantissa).
template <bool kTable>
__device__ __forceinline__ float quantize64(const uint32_t (&w)[32], uint32_t (&packed)[16], const ScaleEntry* tab) {
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) m2 = __vmaxu2(m2, w[i] & 0x7fff7fffu);
  const uint32_t abits = max(m2 << 16, m2 & 0xffff0000u);  // fp32 bits of a
  const int ea = (int)(abits >> 23);
  if (abits != 0u && ea < kMinFastExp) {
    const float s = __fdiv_rn(__uint_as_float(abits), 127.f);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t wv = w[2 * k + (e >> 1)];
        word |= quantize_exact((e & 1) ? bf16_hi(wv) : bf16_lo(wv), s) << (8 * e);
      }
      packed[k] = word;
    }
    return s;
  }
  float s = 1.f, y = 1.f;  // a = 0: every code is 0
  if (abits != 0u) {
    if constexpr (kTable) {
      const ScaleEntry t = tab[(abits >> 16) & 0x7fu];
      const int sh = (ea - 127) << 23;
      s = __uint_as_float(t.s_bits + sh);
      y = __uint_as_float(t.y_bits - sh);
    } else {
      s = __fdiv_rn(__uint_as_float(abits), 127.f);
      y = __frcp_rn(s);
    }
  }
  codes64(w, packed, s, y);
  return s;
}

// The same for a group with an fp16 scale (the pages' INT8 layout):
// s = RN_fp16(a / 127) -- fp32(a / 127) rounded again to fp16 is that
// correctly rounded quotient, as for the rk8v4 keys -- stored as 1 when it
// rounds to 0 and as 65504 (with `range` set) past the fp16 maximum. The codes
// come from the same refined quotient with y = RN(1/s), replayed on the CPU
// for fp16 scales too (tests/quotient_check.c); a group whose scale is an fp16
// subnormal or saturated, where |x / s| can pass 127, divides per element and
// clamps. Returns the scale's fp16 bits.
__device__ __forceinline__ uint32_t quantize64_f16(const uint32_t (&w)[32], uint32_t (&packed)[16], bool& range) {
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) m2 = __vmaxu2(m2, w[i] & 0x7fff7fffu);
  const uint32_t abits = max(m2 << 16, m2 & 0xffff0000u);  // fp32 bits of a
  uint32_t sb = 0x3c00u;  // a = 0: scale 1, every code 0
  bool per_element = false;
  if (abits != 0u) {
    sb = __half_as_ushort(__float2half_rn(__fdiv_rn(__uint_as_float(abits), 127.f)));
    if ((sb & 0x7fffu) == 0u) {
      sb = 0x3c00u;  // below the fp16 range: |x| < 2^-17, every code 0
    } else if ((sb & 0x7fffu) >= 0x7c00u) {
      sb = 0x7bffu;
      range = true;
      per_element = true;
    } else if ((sb & 0x7c00u) == 0u) {
      per_element = true;  // subnormal scale: relative rounding beyond 2^-11
    }
  }
  const float s = __half2float(__ushort_as_half((unsigned short)sb));
  if (per_element) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t wv = w[2 * k + (e >> 1)];
        word |= quantize_exact((e & 1) ? bf16_hi(wv) : bf16_lo(wv), s) << (8 * e);
      }
      packed[k] = word;
    }
    return sb;
  }
  codes64(w, packed, s, __frcp_rn(s));
  return sb;
}

constexpr int kAppendThreads = 128;     // one 64-channel group per thread and chunk
constexpr int kAppendStages = 2;
constexpr int kAppendBlocksPerSM = 4;
constexpr int kChunkBytes = 8192;       // bf16 bytes of K (and of V) per chunk
constexpr int kDestEntries = 512;       // (row, head) destinations a block looks up at once
constexpr int kAppendSmemSeqs = 256;    // sequences whose cu_new/start_pos a block stages in shared memory

struct __align__(128) AppendSmem {
  uint8_t stage[kAppendStages][2 * kChunkBytes];  // K rows | V rows of one chunk, bf16
  int2 dest[kDestEntries];                        // per (chunk of a batch, row): (page * Hkv + head or -1, slot)
  uint64_t full[kAppendStages];
  uint64_t empty[kAppendStages];                  // the 4 warps done with a stage
  int cnt[kAppendStages];
  int abort;
  int issued;  // the highest chunk number issued so far
  ScaleEntry tab[128];
  int cu[kAppendSmemSeqs + 1];
  int start[kAppendSmemSeqs];
};

// Persistent grid, four blocks per SM: the quotient's dependent steps are
// latency-bound, and more resident warps hide them better than a deeper ring
// (measured on the 8 x 1,024-row MIX append: 2 stages x 4 blocks 12.2 us,
// 4 x 3 13.9 us, 3 x 4 13.1 us). The (row, kv-head) pairs are cut into chunks
// of R = 8 KB / (2 D) consecutive pairs; block b takes chunks b, b + grid, ...
// The K rows and the V rows of a chunk stream into a stage of a 2-deep
// shared-memory ring with two bulk copies (cp.async.bulk, completing on the
// stage's "full" mbarrier). The destinations of up to kDestEntries / R of the
// block's chunks (binary search over cu_new, block-table entry) are looked up
// together, one pair per thread, so their global loads overlap. Per chunk,
// thread t quantizes group t (K groups, then V groups), reading its 128 bytes
// in a lane-rotated order so the eight lanes of a quarter-warp hit distinct
// banks; the warp's codes then go out as whole page rows (below). There is no
// block barrier per chunk: each warp releases the stage on its "empty"
// mbarrier, and the last of the four loads the chunk S ahead into it.
template <int D, int FMT>
__global__ void __launch_bounds__(kAppendThreads, kAppendBlocksPerSM) kv_append_kernel(const AppendParams p) {
  chain_wait();
  chain_release();
  constexpr int GPR = D / kGroup;           // groups per (row, head)
  constexpr int R = kChunkBytes / (2 * D);  // (row, head) pairs per chunk
  constexpr int CB = kDestEntries / R;      // chunks per destination batch
  static_assert(R * GPR == kAppendThreads / 2, "one group per thread");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  AppendSmem& sm = *reinterpret_cast<AppendSmem*>(smem_raw);
  const int t = threadIdx.x, lane = t & 31;
  const bool staged = p.B <= kAppendSmemSeqs;
  const uint32_t npairs = (uint32_t)p.total_new * (uint32_t)p.Hkv;
  const uint32_t nchunks = (npairs + R - 1) / R;
  const uint32_t grid = gridDim.x;
  if (blockIdx.x >= nchunks) return;
  const uint32_t my_chunks = (nchunks - blockIdx.x + grid - 1) / grid;

  auto rows_of = [&](uint32_t c) { return (int)min((uint32_t)R, npairs - c * R); };
  auto issue = [&](uint32_t k) {  // chunk number k of this block into its stage
    if (k >= my_chunks) return;
    const uint32_t c = blockIdx.x + k * grid;
    const int st = (int)(k % kAppendStages);
    const uint32_t bytes = (uint32_t)rows_of(c) * D * 2;
    const uint32_t fb = smem_u32(&sm.full[st]);
    mbar_arrive_expect_tx(fb, 2 * bytes);
    const size_t off = (size_t)c * kChunkBytes;
    bulk_load(smem_u32(sm.stage[st]), reinterpret_cast<const uint8_t*>(p.k) + off, bytes, fb);
    bulk_load(smem_u32(sm.stage[st]) + kChunkBytes, reinterpret_cast<const uint8_t*>(p.v) + off, bytes, fb);
  };
  // destination of pair number `pair`: (page * Hkv + head, slot), or -1 after
  // flagging a position or page id out of range
  auto lookup = [&](uint32_t pair) {
    const uint32_t j = p.hkv_shift >= 0 ? pair >> p.hkv_shift : pair / (uint32_t)p.Hkv;
    const int h = (int)(pair - j * (uint32_t)p.Hkv);
    int lo = 0, hi = p.B;  // find b with cu_new[b] <= j < cu_new[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      const int c = staged ? sm.cu[mid] : __ldg(p.cu_new + mid);
      if (c <= (int)j) lo = mid; else hi = mid;
    }
    const int c0 = staged ? sm.cu[lo] : __ldg(p.cu_new + lo);
    const int st0 = staged ? sm.start[lo] : __ldg(p.start_pos + lo);
    const int64_t pos64 = (int64_t)st0 + ((int)j - c0);
    if (pos64 < 0 || pos64 >= (int64_t)p.max_pages * p.P || pos64 > 0x7fffffff) {
      flag(p.status, NK_DEVFLAG_BAD_POS);
      return make_int2(-1, 0);
    }
    const int pos = (int)pos64;
    const uint32_t pi = p.p_shift >= 0 ? (uint32_t)pos >> p.p_shift : (uint32_t)pos / (uint32_t)p.P;
    const int page = __ldg(p.bt + (size_t)lo * p.max_pages + pi);
    if (page < 0 || page >= p.num_pages) {
      flag(p.status, NK_DEVFLAG_BAD_PAGE);
      return make_int2(-1, 0);
    }
    const int slot = p.p_shift >= 0 ? (pos & (p.P - 1)) : (int)((uint32_t)pos % (uint32_t)p.P);
    return make_int2(page * p.Hkv + h, slot);
  };
  // destinations of the block's chunks k0 .. k0 + CB - 1 (the loads of one
  // thread's entries are independent, so they are all in flight together)
  auto lookup_batch = [&](uint32_t k0) {
#pragma unroll 4
    for (int e = t; e < kDestEntries; e += kAppendThreads) {
      const uint32_t k = k0 + e / R;
      const uint32_t pair = (blockIdx.x + k * grid) * R + e % R;
      sm.dest[e] = (k < my_chunks && pair < npairs) ? lookup(pair) : make_int2(-1, 0);
    }
  };

  if (t == 0) {
    for (int st = 0; st < kAppendStages; ++st) {
      mbar_init(smem_u32(&sm.full[st]), 1);
      mbar_init(smem_u32(&sm.empty[st]), kAppendThreads / 32);
      sm.cnt[st] = 0;
    }
    sm.abort = 0;
    sm.issued = (int)min((uint32_t)kAppendStages, my_chunks) - 1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int k = 0; k < kAppendStages; ++k) issue(k);
  }
  if (staged) {
    for (int i = t; i <= p.B; i += kAppendThreads) sm.cu[i] = __ldg(p.cu_new + i);
    for (int i = t; i < p.B; i += kAppendThreads) sm.start[i] = __ldg(p.start_pos + i);
  }
  {
    const float s_m = __fdiv_rn(1.f + (float)t * 0.0078125f, 127.f);  // t < 128
    sm.tab[t] = ScaleEntry{__float_as_uint(s_m), __float_as_uint(__frcp_rn(s_m))};
  }
  __syncthreads();

  // this thread's group in a chunk: tensor, pair row, group in the row
  const int isv = t / (R * GPR), gk = t % (R * GPR), row = gk / GPR, grp = gk % GPR;
  const int rot = lane & 7;  // 16-byte piece read first
  volatile int* abort_flag = &sm.abort;
  for (uint32_t k = 0; k < my_chunks; ++k) {
    if (k % CB == 0) {
      if (k > 0) __syncthreads();  // the previous batch's entries are no longer read
      lookup_batch(k);
      __syncthreads();
    }
    const uint32_t c = blockIdx.x + k * grid;
    const int st = (int)(k % kAppendStages);
    const uint32_t ph = (k / kAppendStages) & 1u;
    const int rows = rows_of(c);
    const int2* dest = sm.dest + (k % CB) * R;
    // after one wait has run out nothing waits any more: the chunks run
    // without data, and nothing more is issued (the copies issued so far land
    // before the block exits)
    if (!*abort_flag && !mbar_wait(smem_u32(&sm.full[st]), ph)) {
      flag(p.status, NK_DEVFLAG_TIMEOUT);
      *abort_flag = 1;
    }
    if constexpr (FMT == kFmtBf16) {
      // the rows as they are: 16-byte pieces straight from the stage into
      // their pages (one row of one tensor is D bf16 values of its page)
#pragma unroll
      for (int i = 0; i < 2 * kChunkBytes / (16 * kAppendThreads); ++i) {
        const int o = (i * kAppendThreads + t) * 16;
        const int tv = o / kChunkBytes, rem = o % kChunkBytes, r = rem / (2 * D), col = rem % (2 * D);
        const int2 dd = dest[r];
        if (r < rows && dd.x >= 0)
          *reinterpret_cast<uint4*>(p.pool + (int64_t)dd.x * p.lay.chunk + (tv ? p.lay.vc : 0) + dd.y * (2 * D) +
                                    col) = *reinterpret_cast<const uint4*>(sm.stage[st] + o);
      }
    } else {
      // load the group (pieces in rotated order), quantize
      uint32_t w[32];
      const uint8_t* src = sm.stage[st] + isv * kChunkBytes + gk * 128;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int piece = (i + rot) & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(src + piece * 16);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
      uint32_t packed[16];  // codes of the pieces in the same rotated order
      bool range = false;
      float s = 0.f;
      uint32_t sb16 = 0u;
      if constexpr (FMT == kFmtI8F16) sb16 = quantize64_f16(w, packed, range);
      else s = quantize64<true>(w, packed, sm.tab);
      // The warp's 2 KB of codes (its 2048 / D rows, lane L's group at bytes
      // 64 L) go through the part of the stage whose bf16 rows it has just
      // read, then out as whole rows: 16-byte pieces, D / 16 lanes per row, so
      // every 32-byte sector of a page row is written by one store (against
      // eight 8-byte pieces per group stored straight from each thread:
      // 13.9 against 15.2 us on the MIX append).
      uint8_t* wst = sm.stage[st] + isv * kChunkBytes + (gk - lane) * 128;
      __syncwarp();  // every lane's bf16 reads of the area are done
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int piece = (i + rot) & 7;
        *reinterpret_cast<uint2*>(wst + lane * 64 + piece * 8) = make_uint2(packed[2 * i], packed[2 * i + 1]);
      }
      // generic-proxy writes of the stage are ordered before the bulk copy that refills it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      {
        constexpr int LPR = D / 16;  // lanes per row
        constexpr int RPI = 32 / LPR;
        const int r0 = (gk - lane) / GPR;  // the warp's first row of the chunk
        const int off = (lane % LPR) * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rl = i * RPI + lane / LPR;
          const uint4 v = *reinterpret_cast<const uint4*>(wst + rl * D + off);
          const int2 dd = dest[r0 + rl];
          if (r0 + rl < rows && dd.x >= 0)
            *reinterpret_cast<uint4*>(p.pool + (int64_t)dd.x * p.lay.chunk + (isv ? p.lay.vc : 0) + dd.y * D + off) = v;
        }
      }
      // the row's GPR scales from its first group's lane, in one store
      const int2 d = dest[row];
      if constexpr (FMT == kFmtI8F16) {
        uint32_t sw[GPR];
#pragma unroll
        for (int g2 = 0; g2 < GPR; ++g2) sw[g2] = __shfl_sync(0xffffffffu, sb16, (lane & ~(GPR - 1)) + g2);
        if (row < rows && d.x >= 0) {
          uint8_t* sdst = p.pool + (int64_t)d.x * p.lay.chunk + (isv ? p.lay.vs : p.lay.ks) + d.y * GPR * 2;
          if (grp == 0) {
            if constexpr (GPR == 4) {
              *reinterpret_cast<uint2*>(sdst) = make_uint2(sw[0] | (sw[1] << 16), sw[2] | (sw[3] << 16));
            } else if constexpr (GPR == 2) {
              *reinterpret_cast<uint32_t*>(sdst) = sw[0] | (sw[1] << 16);
            } else {
              *reinterpret_cast<uint16_t*>(sdst) = (uint16_t)sw[0];
            }
          }
          if (range) flag(p.status, NK_DEVFLAG_RANGE);
        }
      } else {
        float sv[GPR];
#pragma unroll
        for (int g2 = 0; g2 < GPR; ++g2) sv[g2] = __shfl_sync(0xffffffffu, s, (lane & ~(GPR - 1)) + g2);
        if (row < rows && d.x >= 0 && grp == 0) {
          uint8_t* sdst = p.pool + (int64_t)d.x * p.lay.chunk + (isv ? p.lay.vs : p.lay.ks) + d.y * GPR * 4;
          if constexpr (GPR == 4) {
            *reinterpret_cast<float4*>(sdst) = make_float4(sv[0], sv[1], sv[2], sv[3]);
          } else if constexpr (GPR == 2) {
            *reinterpret_cast<float2*>(sdst) = make_float2(sv[0], sv[1]);
          } else {
            *reinterpret_cast<float*>(sdst) = sv[0];
          }
        }
      }
    }
    // this warp is done with the stage; the last of the four refills it
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&sm.empty[st]));
      if (atomicAdd(&sm.cnt[st], 1) == kAppendThreads / 32 - 1) {
        sm.cnt[st] = 0;
        if (k + kAppendStages < my_chunks && !*abort_flag) {
          if (mbar_wait(smem_u32(&sm.empty[st]), ph)) {
            // generic-proxy reads of the stage are ordered before the bulk copy that refills it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(k + kAppendStages);
            sm.issued = (int)(k + kAppendStages);
          } else {
            flag(p.status, NK_DEVFLAG_TIMEOUT);
            *abort_flag = 1;
          }
        }
      }
    }
  }
  // copies still in flight after a timed-out wait land before the block exits
  __syncthreads();
  if (t == 0 && *abort_flag) {
    // the last chunk issued into each stage is one of the last S issued
    for (int kk = max(0, sm.issued - kAppendStages + 1); kk <= sm.issued; ++kk)
      (void)mbar_wait(smem_u32(&sm.full[kk % kAppendStages]), (uint32_t)(kk / kAppendStages) & 1u);
  }
}

constexpr int kSmallThreads = 128;
constexpr int64_t kSmallMaxGroups = 4096;  // appends up to this many groups take the direct kernel

// Small appends (decode and verify steps: a few rows per sequence): one thread
// per 64-channel group of K or V of one (row, kv-head), nothing staged. The
// group's eight 16-byte loads go out first and the destination lookup
// (binary search over cu_new, block-table entry) runs while they are in
// flight; s = fp32(a / 127) and RN(1/s) come from IEEE division; the codes
// from the same exact quotient as the streaming kernel.
template <int D, int FMT>
__global__ void __launch_bounds__(kSmallThreads) kv_append_small_kernel(const AppendParams p) {
  chain_wait();
  chain_release();
  constexpr int GPR = D / kGroup;
  const uint32_t gid = blockIdx.x * kSmallThreads + threadIdx.x;
  const uint32_t ngroups = (uint32_t)p.total_new * (uint32_t)p.Hkv * 2u * GPR;
  const bool live = gid < ngroups;
  const int lane = threadIdx.x & 31;
  // up to 32 sequences: lane l holds cu_new[l] and start_pos[l], and the
  // search below reads them by shuffle instead of by dependent global loads
  const bool in_regs = p.B <= 32;
  int cu_l = 0, st_l = 0;
  if (in_regs) {
    cu_l = lane <= p.B ? __ldg(p.cu_new + lane) : 0x7fffffff;
    st_l = lane < p.B ? __ldg(p.start_pos + lane) : 0;
  }
  const uint32_t g = live ? gid : 0u;
  const uint32_t pair = g / (2 * GPR), isv = (g / GPR) & 1u, grp = g % GPR;
  uint32_t w[32];
  {
    const uint4* src = (isv ? p.v : p.k) + (size_t)pair * (D / 8) + grp * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 a = __ldg(src + i);
      w[4 * i] = a.x; w[4 * i + 1] = a.y; w[4 * i + 2] = a.z; w[4 * i + 3] = a.w;
    }
  }
  const bool flagger = isv == 0 && grp == 0;  // one thread per pair reports bad positions and pages
  const uint32_t j = p.hkv_shift >= 0 ? pair >> p.hkv_shift : pair / (uint32_t)p.Hkv;
  const int h = (int)(pair - j * (uint32_t)p.Hkv);
  int lo = 0, hi = p.B;  // find b with cu_new[b] <= j < cu_new[b+1]
  int c0, st0;
  if (in_regs) {
    for (int it = 0; it < 6; ++it) {  // ceil(log2(32)) + 1 rounds, the same count in every lane
      const int mid = (lo + hi) >> 1;
      const int c = __shfl_sync(0xffffffffu, cu_l, mid & 31);
      if (hi - lo > 1) {
        if (c <= (int)j) lo = mid; else hi = mid;
      }
    }
    c0 = __shfl_sync(0xffffffffu, cu_l, lo & 31);
    st0 = __shfl_sync(0xffffffffu, st_l, lo & 31);
  } else {
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.cu_new + mid) <= (int)j) lo = mid; else hi = mid;
    }
    c0 = __ldg(p.cu_new + lo);
    st0 = __ldg(p.start_pos + lo);
  }
  if (!live) return;
  const int64_t pos64 = (int64_t)st0 + ((int)j - c0);
  uint32_t packed[16];
  bool range = false;
  float s = 0.f;
  uint32_t sb16 = 0u;
  if constexpr (FMT == kFmtI8F16) sb16 = quantize64_f16(w, packed, range);
  else if constexpr (FMT == kFmtI8F32) s = quantize64<false>(w, packed, nullptr);
  if (pos64 < 0 || pos64 >= (int64_t)p.max_pages * p.P || pos64 > 0x7fffffff) {
    if (flagger) flag(p.status, NK_DEVFLAG_BAD_POS);
    return;
  }
  const int pos = (int)pos64;
  const uint32_t pi = p.p_shift >= 0 ? (uint32_t)pos >> p.p_shift : (uint32_t)pos / (uint32_t)p.P;
  const int page = __ldg(p.bt + (size_t)lo * p.max_pages + pi);
  if (page < 0 || page >= p.num_pages) {
    if (flagger) flag(p.status, NK_DEVFLAG_BAD_PAGE);
    return;
  }
  const int slot = p.p_shift >= 0 ? (pos & (p.P - 1)) : (int)((uint32_t)pos % (uint32_t)p.P);
  uint8_t* chunk = p.pool + ((int64_t)page * p.Hkv + h) * p.lay.chunk;
  if constexpr (FMT == kFmtBf16) {
    uint4* dst = reinterpret_cast<uint4*>(chunk + (isv ? p.lay.vc : 0) + slot * (2 * D) + grp * (2 * kGroup));
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(chunk + (isv ? p.lay.vc : 0) + slot * D + grp * kGroup);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
  if constexpr (FMT == kFmtI8F16) {
    *reinterpret_cast<uint16_t*>(chunk + (isv ? p.lay.vs : p.lay.ks) + (slot * GPR + grp) * 2) = (uint16_t)sb16;
    if (range) flag(p.status, NK_DEVFLAG_RANGE);
  } else {
    *reinterpret_cast<float*>(chunk + (isv ? p.lay.vs : p.lay.ks) + (slot * GPR + grp) * 4) = s;
  }
}

template <int D, int FMT>
static cudaError_t launch_append_d(int sms, const AppendParams& p, int64_t groups, int64_t pairs, cudaStream_t stream) {
  if (groups <= kSmallMaxGroups) {
    const unsigned g = (unsigned)((groups + kSmallThreads - 1) / kSmallThreads);
    return launch_chained(kv_append_small_kernel<D, FMT>, dim3(g), dim3(kSmallThreads), 0, stream, p);
  }
  if (sms < 1) sms = 1;
  const int64_t rows_per_chunk = kChunkBytes / (2 * D);
  const int64_t nchunks = (pairs + rows_per_chunk - 1) / rows_per_chunk;
  const int64_t grid = nchunks < (int64_t)sms * kAppendBlocksPerSM ? nchunks : (int64_t)sms * kAppendBlocksPerSM;
  const int smem = (int)sizeof(AppendSmem);
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kv_append_kernel<D, FMT>), smem);
  if (e != cudaSuccess) return e;
  return launch_chained(kv_append_kernel<D, FMT>, dim3((unsigned)grid), dim3(kAppendThreads), smem, stream, p);
}

template <int FMT>
static cudaError_t launch_append_fmt(int sms, const AppendParams& p, int64_t groups, int64_t pairs,
                                     cudaStream_t stream) {
  if (p.D == 256) return launch_append_d<256, FMT>(sms, p, groups, pairs, stream);
  if (p.D == 128) return launch_append_d<128, FMT>(sms, p, groups, pairs, stream);
  return launch_append_d<64, FMT>(sms, p, groups, pairs, stream);
}

cudaError_t launch_kv_append(int sms, const nk_kv_pool& pool, int fmt, const int32_t* bt, int max_pages,
                             const int32_t* start_pos, const int32_t* cu_new, int B, int total_new, const void* k,
                             const void* v, int32_t* status, cudaStream_t stream) {
  AppendParams p;
  p.pool = reinterpret_cast<uint8_t*>(pool.base_dev);
  p.num_pages = pool.num_pages;
  p.P = pool.page_size;
  p.Hkv = pool.num_kv_heads;
  p.D = pool.head_dim;
  p.lay = layout_of(fmt, p.P, p.D);
  p.bt = bt;
  p.max_pages = max_pages;
  p.start_pos = start_pos;
  p.cu_new = cu_new;
  p.B = B;
  p.total_new = total_new;
  p.k = reinterpret_cast<const uint4*>(k);
  p.v = reinterpret_cast<const uint4*>(v);
  p.status = status;
  auto log2_exact = [](int n) {
    int sh = 0;
    while ((1 << sh) < n) ++sh;
    return (1 << sh) == n ? sh : -1;
  };
  p.p_shift = log2_exact(p.P);
  p.hkv_shift = log2_exact(p.Hkv);
  const int64_t pairs = (int64_t)total_new * p.Hkv;
  if (pairs * 2 * (p.D / kGroup) >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // 32-bit numbering
  if (pairs == 0) return cudaSuccess;
  const int64_t groups = pairs * 2 * (p.D / kGroup);
  if (fmt == kFmtI8F16) return launch_append_fmt<kFmtI8F16>(sms, p, groups, pairs, stream);
  if (fmt == kFmtBf16) return launch_append_fmt<kFmtBf16>(sms, p, groups, pairs, stream);
  return launch_append_fmt<kFmtI8F32>(sms, p, groups, pairs, stream);
}

}  // namespace nk
