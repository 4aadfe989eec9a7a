// nk_decode_mma.cuh -- split-KV paged attention over the INT8 group-64 cache
// on tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulate).
//
// Attention re-reads the whole cache every step ("NInfer-3090" README,
// "Choosing a KV format"), so the kernel is built to stream pages at HBM
// speed; decode and MTP-verify rounds attend T = draft+1 columns per sequence
// ("Decode after the small-T kernels"). The dequantization happens inside the
// dot products: the int8 codes enter the MMAs exactly (as fp16), the group
// scales are applied to fp32 partial sums.
//
// CTA layout (256 threads = 8 warps, two per SM sub-partition, so a thread
// may hold up to 255 registers):
//   * Loads: per page, TMA tile loads of the K and V code tiles (128-byte
//     swizzled, [128 channels][P keys][K|V] boxes straight out of the pool by
//     physical page id) plus 1-D bulk copies of the two scale arrays land in
//     one stage of a shared-memory ring and complete on its "full" mbarrier.
//     The prologue does every global read first (context lengths into
//     shared memory, the page-coordinate cache, the first unit's Q staged
//     once per CTA), since a load issued behind this SM's page loads returns
//     only after their data; then one thread of the last warp issues the
//     first S pages in order. Afterwards the last warp to finish reading a
//     stage (elected by a shared-memory counter, after arriving on the
//     stage's "empty" mbarrier) immediately loads the page S ahead into it.
//   * Consumers: teams of CS warps. A team owns 16-key blocks of the stream
//     (block j goes to team j % NTEAMS); its CS warps split the head_dim
//     channels (DW = D/CS each, whole 64-channel groups), so each warp keeps
//     only its slice of Q (as MMA B fragments) and of the output accumulator.
//     Per block and warp:
//       QK   S^T[key][row] = K[key][ch] Q^T[ch][row], one fp32 accumulator per
//            64-channel group, scaled by Ks * sm_scale * log2(e) and summed
//            (swap-AB: keys are the MMA M dimension, the G*T query rows the N
//            dimension, so M = 24 needs no padding); K fragments come from
//            ldmatrix on the swizzled tile and are widened int8 -> fp16 with a
//            byte permute and one half2 subtract.
//       team exchange of the partial scores (CS > 1) through shared memory,
//            summed in a fixed order so every warp of the team holds identical
//            scores.
//       online softmax in base 2 with a lazy reference per row (raised, and
//            the accumulator rescaled, only when a score passes it by more
//            than 8).
//       PV   O^T[ch][row] += V^T[ch][key] P'^T[key][row] with
//            P' = p * Vs[key][group] split into fp16 hi + lo parts (two MMAs)
//            so the product keeps ~22 bits; V^T fragments come from
//            ldmatrix.trans, P'^T fragments from movmatrix of the score tile.
//     At the end of a segment (the CTA's share of one (sequence, kv-head))
//     the teams merge through shared memory in a fixed order (parked in the
//     idle ring after the CTA's last segment) and the CTA writes the bf16
//     output (whole unit) or an fp32 partial plus LSE; the next unit's Q was
//     fetched when the segment started.
// Every wait on an mbarrier is bounded; a timeout sets NK_DEVFLAG_TIMEOUT.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "nk_decode.cuh"
#include "nk_ptx.cuh"

namespace nk {
namespace mma {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kSmemLimit = 232448;  // opt-in shared memory per block on sm_100/103

struct Geometry {
  int stage_bytes;   // one page: K|V boxes, then Ks, Vs (rounded to 1 KB)
  int stages;
  int xch_off, xch_bytes;
  int merge_off, merge_bytes;
  int pre_off;
  int pid_off;
  int bar_off;
  int total;
};

__host__ __device__ inline int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Shared-memory plan. Needs the pool format, D, NT, CS, P (and B for the
// prefix array). A bf16 pool stages 2-byte K|V values and no scales.
__host__ __device__ inline Geometry geometry(int fmt, int D, int NT, int CS, int P, int B) {
  Geometry g;
  const int nteams = kConsumerWarps / CS;
  // rk8v4: D key bytes and D / 2 value bytes per key, fp16 scales per 64
  // key channels and per 32 value channels
  const int kv_bytes = fmt == kFmtRk8v4 ? 3 * P * D / 2 : 2 * P * D * (fmt == kFmtBf16 ? 2 : 1);
  const int sc_bytes = fmt == kFmtRk8v4 ? P * (D / kGroup) * 2 + P * (D / kRkVGroup) * 2
                       : (fmt == kFmtBf16 ? 0 : 2 * P * (D / kGroup) * (fmt == kFmtI8F16 ? 2 : 4));
  g.stage_bytes = round_up(kv_bytes + sc_bytes, 1024);
  g.xch_bytes = CS > 1 ? nteams * 2 * CS * NT * 4 * 32 * 4 : 0;
  const int mrows = NT * 8;
  g.merge_bytes = mrows * (D + 4) * 4 + 3 * nteams * mrows * 4 + mrows * 4;
  const int pre_bytes = round_up((2 * B + 33) * 4, 16);  // pre[B+1], warp_tot, flags, lens[B], icnt[8]
  const int pid_bytes = 1024 * 4;
  const int fixed = g.xch_bytes + g.merge_bytes + pre_bytes + pid_bytes + 8 * 2 * 8 + 1024;
  int s = (kSmemLimit - fixed) / g.stage_bytes;
  if (s > 8) s = 8;
  g.stages = s;
  int off = g.stages * g.stage_bytes;
  g.xch_off = off;
  off += g.xch_bytes;
  g.merge_off = off;
  off += g.merge_bytes;
  g.pre_off = off;
  off += pre_bytes;
  g.pid_off = off;
  off += pid_bytes;
  g.bar_off = off;
  off += 2 * 8 * 8;
  g.total = off + 1024;  // slack to align the dynamic base to 1 KB
  return g;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  // not volatile: a pure register operation, so the compiler may interleave
  // independent MMAs and hide their latency
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two signed int8 bytes of w (selected by sel, pre-biased by ^0x80808080)
// as an exact fp16 pair: 0x64XX is 1024 + XX, minus 1152 gives XX - 128.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t wb, uint32_t sel) {
  const uint32_t h = prmt(wb, 0x64646464u, sel);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6480),
                                                                                    __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Two's-complement 4-bit codes: w holds, per 16-bit half, two bytes of one
// key's value row (channels 4u .. 4u + 3, low nibble first), the low half one
// key and the high half the next. nib_lo: the low nibbles of the halves' low
// bytes as an exact fp16 pair (1024 + (n ^ 8) - 1032 = n); nib_hi: their high
// nibbles (1024 + 16 (n ^ 8), times 1/16, minus 72). w >> 8 gives the same for
// the halves' high bytes (channels 4u + 2, 4u + 3).
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) {
  const uint32_t h = (w & 0x000f000fu) ^ 0x64086408u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6408),
                                                                                    __ushort_as_half(0x6408)));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) {
  const uint32_t h = (w & 0x00f000f0u) ^ 0x64806480u;
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&h),
                            __halves2half2(__ushort_as_half(0x2c00), __ushort_as_half(0x2c00)),   // 1/16
                            __halves2half2(__ushort_as_half(0xd480), __ushort_as_half(0xd480)));  // -72
  return *reinterpret_cast<const uint32_t*>(&r);
}

// 2^x on the SFU (relative error ~2^-22); ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// Range of the fp16 MMA operands. The method is scale-free: attention of Q,
// K, V scaled by powers of two is the same attention (K) or the same output
// scaled alike (V). fp16 is not: it has a 2^-14 .. 65504 normal range. Both
// tensor-core kernels therefore carry powers of two beside their fp16 operands
// and undo them in fp32, exactly:
//   * a query row (or a warp's channel slice of it) enters the QK product as
//     q 2^e with e chosen from its largest |q|, so that it lies in
//     [2^14, 2^15); the row's fp32 scores are multiplied by 2^-e;
//   * the probability-weighted value scales P' = p Vs of a 64-channel group
//     enter the PV product as p Vs 2^-ev, and the accumulator holds O 2^-ev.
//     ev follows the exponent E of the largest Vs of the page (or 16-key
//     block): set at the first one and moved only when E - ev leaves
//     [-10, 6] -- p <= 2^8 keeps p Vs 2^-ev below 2^15, the lower bound keeps
//     the hi part of a key with p near 1 a normal fp16 number -- with the
//     accumulator rescaled by 2^(ev_old - ev_new), like the softmax
//     reference. The output is O 2^-ev times 2^ev.
// ---------------------------------------------------------------------------
// Bytes of one group scale in a pool of format fmt: fp32 for the INT8 layout
// with fp32 scales, fp16 for the pages' own INT8 layout and for rk8v4.
__host__ __device__ inline int scale_bytes(int fmt) { return (fmt == kFmtI8F16 || fmt == kFmtRk8v4) ? 2 : 4; }

// Scale number idx of a page's scale array (fp32 or fp16 elements).
__device__ __forceinline__ float ld_scale(const uint8_t* arr, int idx, int sb) {
  return sb == 2 ? __half2float(reinterpret_cast<const __half*>(arr)[idx]) : reinterpret_cast<const float*>(arr)[idx];
}

// 2^e as fp32, -126 <= e <= 127.
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// E with 2^E <= x < 2^(E+1) for a positive normal fp32 x (-127 for 0 and subnormals).
__device__ __forceinline__ int exp_of(float x) { return (int)((__float_as_uint(x) >> 23) & 0xffu) - 127; }

// Exponent that brings a query row whose largest |q| is m into [2^14, 2^15)
// (0 for a zero row; at most 2^60, so rows below 2^-46 stay smaller).
__device__ __forceinline__ int q_norm_exp(float m) {
  if (!(m > 0.f)) return 0;
  const int e = 14 - exp_of(m);
  return e > 60 ? 60 : (e < -120 ? -120 : e);
}

constexpr int kEvUnset = -1000;  // no page of the segment seen yet

// Moves the exponent ev of a group's P' when the page's largest value scale
// (exponent E) leaves ev's window; beta = 2^(ev_old - ev_new) rescales the
// accumulator (1 on the first page, whose accumulator is still zero).
__device__ __forceinline__ bool ev_update(int& ev, int E, float& beta) {
  if (ev != kEvUnset && E - ev <= 6 && E - ev >= -10) return false;
  const int ne = E > 100 ? 100 : (E < -100 ? -100 : E);
  const int d = ev == kEvUnset ? 0 : ev - ne;
  beta = d < -126 ? 0.f : pow2i(d > 127 ? 127 : d);
  ev = ne;
  return true;
}

// Byte offset of (channel chunk16 `ch16`, row) inside one K|V box region of
// a stage: boxes of 128 channels (64 for D = 64) x [K rows | V rows].
template <int D>
__device__ __forceinline__ uint32_t box_off(int P, int kv, int key, int ch16) {
  if constexpr (D == 64) {
    const int row = kv * P + key;
    return row * 64 + (((ch16 & 3) ^ ((row >> 1) & 3)) << 4);
  } else {
    const int box = ch16 >> 3;
    const int row = kv * P + key;
    return box * (2 * P * 128) + row * 128 + (((ch16 & 7) ^ (row & 7)) << 4);
  }
}

// ---------------------------------------------------------------------------
// page loads
// ---------------------------------------------------------------------------
constexpr int kPidCache = 1024;  // page coordinates cached in shared memory per CTA

// Coordinate z = page * Hkv + h of the CTA's page number q (-1 for a page id
// outside the pool), from the cache or, past it, from the block table.
__device__ __forceinline__ int page_coord(const DecodeParams& p, const SplitShape& sh, const int* pre, int64_t x_begin,
                                          int q) {
  const int64_t x = x_begin + q;
  int lo = 0, hi = sh.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)pre[mid] * sh.Hkv <= x) lo = mid; else hi = mid;
  }
  const int pages = pre[lo + 1] - pre[lo];
  const int64_t off = x - (int64_t)pre[lo] * sh.Hkv;
  const int h = (int)(off / pages), pi = (int)(off % pages);
  const int page = __ldg(p.bt + (int64_t)lo * p.max_pages + pi);
  return (page < 0 || page >= p.num_pages) ? -1 : page * p.Hkv + h;
}

// Load the CTA's page number q into its stage: TMA boxes of the K|V codes
// plus bulk copies of the two scale arrays, all completing on full_bar.
template <int D, bool BF = false>
__device__ __forceinline__ void issue_page(const DecodeParams& p, const CUtensorMap* tmap, int z, uint32_t dst,
                                           uint32_t fb) {
  const int P = p.P;
  if constexpr (BF) {
    // bf16 rows: boxes of [64 channels][P keys][K|V] (128-byte rows), no scales
    if (z < 0) {
      flag(p.status, NK_DEVFLAG_BAD_PAGE);
      mbar_arrive(fb);
      return;
    }
    mbar_arrive_expect_tx(fb, 2 * P * D * 2);
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx) tma_load_4d(dst + bx * 2 * P * 128, tmap, fb, bx * 64, 0, 0, z);
    return;
  }
  const int kv_bytes = 2 * P * D;
  const int sc_bytes = P * (D / kGroup) * scale_bytes(p.fmt);
  if (z < 0) {
    flag(p.status, NK_DEVFLAG_BAD_PAGE);
    mbar_arrive(fb);  // release the consumers; the stage keeps stale data
    return;
  }
  mbar_arrive_expect_tx(fb, kv_bytes + 2 * sc_bytes);
  if constexpr (D == 64) {
    tma_load_4d(dst, tmap, fb, 0, 0, 0, z);
  } else {
#pragma unroll
    for (int bx = 0; bx < D / 128; ++bx) tma_load_4d(dst + bx * 2 * P * 128, tmap, fb, bx * 128, 0, 0, z);
  }
  const uint8_t* chunk = p.pool + (int64_t)z * p.lay.chunk;
  bulk_load(dst + kv_bytes, chunk + p.lay.ks, sc_bytes, fb);
  bulk_load(dst + kv_bytes + sc_bytes, chunk + p.lay.vs, sc_bytes, fb);
}

// The same for an rk8v4 pool: the key codes as boxes of [128 channels][P]
// (one per 128 channels), the value codes as one box of [D / 2 bytes][P],
// then Ks and Vs (fp16) by bulk copies. Stage: K boxes | V box | Ks | Vs.
template <int D>
__device__ __forceinline__ void issue_page_rk(const DecodeParams& p, const CUtensorMap* tk, const CUtensorMap* tv, int z,
                                              uint32_t dst, uint32_t fb) {
  const int P = p.P;
  const int ks_bytes = P * (D / kGroup) * 2, vs_bytes = P * (D / kRkVGroup) * 2;
  if (z < 0) {
    flag(p.status, NK_DEVFLAG_BAD_PAGE);
    mbar_arrive(fb);
    return;
  }
  mbar_arrive_expect_tx(fb, 3 * P * D / 2 + ks_bytes + vs_bytes);
#pragma unroll
  for (int bx = 0; bx < D / 128; ++bx) tma_load_3d(dst + bx * P * 128, tk, fb, bx * 128, 0, z);
  tma_load_3d(dst + P * D, tv, fb, 0, 0, z);
  const uint8_t* chunk = p.pool + (int64_t)z * p.lay.chunk;
  bulk_load(dst + 3 * P * D / 2, chunk + p.lay.ks, ks_bytes, fb);
  bulk_load(dst + 3 * P * D / 2 + ks_bytes, chunk + p.lay.vs, vs_bytes, fb);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// BF: the pool holds bf16 rows (the unquantized layout): K and V enter the
// MMAs as they are (bf16 operands, Q bf16 too), there are no scales, and P
// enters the PV product as bf16 hi + lo.
// FMT: the pool's KvFmt (compile time, so that scale loads need no branch).
// RK: an rk8v4 pool: tmap covers the key codes and tmapv the value codes (for
// the other formats tmapv is unused); each query row is rotated by H64 / 8
// and enters the QK product as fp16 hi + lo; the 4-bit values are widened
// from their nibbles; P' carries one scale per 32 value channels.
template <int D, int NT, int CS, int FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                 const __grid_constant__ CUtensorMap tmapv,
                                                                 const DecodeParams p) {
  constexpr bool BF = FMT == kFmtBf16;
  constexpr bool RK = FMT == kFmtRk8v4;
  static_assert(!RK || D >= 128, "rk8v4: head_dim 128 or 256");
  // the tensor map is a launch parameter (no earlier kernel writes it): its
  // descriptor fetch can start before the wait for the previous kernel
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
  if constexpr (RK) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmapv)) : "memory");
  if (!p.early) chain_wait();  // (early: waits below, before the first page load)
  chain_release();
  constexpr int NTEAMS = kConsumerWarps / CS;
  constexpr int DW = D / CS;        // channels per warp
  constexpr int NCH = DW / 16;      // 16-channel chunks per warp
  constexpr int GW = DW / kGroup;   // groups per warp
  constexpr int G_ALL = D / kGroup;
  constexpr int MROWS = NT * 8;
  static_assert(DW % kGroup == 0, "a warp owns whole 64-channel groups");
  // P' groups of a warp (value channels per scale: 64, rk8v4 32) and the
  // accumulator chunks of one
  constexpr int GP = RK ? DW / kRkVGroup : GW;
  constexpr int CPG = RK ? 2 : 4;
  constexpr int GV_ALL = RK ? D / kRkVGroup : G_ALL;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geometry geo = geometry(FMT, D, NT, CS, p.P, p.B);
  const int S = geo.stages;
  constexpr int sb = (FMT == kFmtI8F16 || RK) ? 2 : 4;
  int* pre = reinterpret_cast<int*>(smem + geo.pre_off);
  int* warp_tot = pre + (p.B + 1);
  volatile int* abort_flag = pre + (p.B + 1) + 8;
  int* cnt = pre + (p.B + 1) + 9;  // [8] consumer count per stage
  int* lens = pre + (p.B + 1) + 24;  // [B] context lengths
  int* icnt = lens + p.B;            // [8] copies issued into each stage
  int* pid = reinterpret_cast<int*>(smem + geo.pid_off);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + geo.bar_off);
  uint64_t* empty_bar = full_bar + 8;
  float* xch = reinterpret_cast<float*>(smem + geo.xch_off);
  float* mo = reinterpret_cast<float*>(smem + geo.merge_off);
  float* tm_m = mo + MROWS * (D + 4);
  float* tm_l = tm_m + NTEAMS * MROWS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = p.P, BPP = P / 16;
  const int per_stage = BPP * CS;  // consumer-warp arrivals per page
  const SplitShape sh = p.shape();

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), per_stage);
      cnt[s] = 0;
      icnt[s] = 0;
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  flag_bad_ctx(p);
  block_page_prefix(sh, p.ctx, p.trim, pre, warp_tot, lens);  // ends with __syncthreads

  const int64_t W = (int64_t)pre[p.B] * p.Hkv;
  if (W == 0) {
    if (p.early) chain_wait();  // every CTA waits: the grid must not complete before its predecessor
    return;
  }
  const int64_t x_begin = cta_begin(W, p.n_ctas, blockIdx.x);
  const int64_t x_end = cta_begin(W, p.n_ctas, blockIdx.x + 1);
  const int total = (int)(x_end - x_begin);
  const uint32_t stage0 = smem_u32(smem);

  const int team = warp / CS, wit = warp % CS;  // team, warp-in-team
  const int g = lane >> 2, t4 = lane & 3;
  const int ch0 = wit * DW;                     // first channel of this warp
  const int grp0 = ch0 / kGroup;
  const int G = p.G, T = p.T, M = G * T;
  const uint32_t bias = 0x80808080u;
  // ldmatrix lane geometry: matrix mi = lane / 8, row-in-matrix = lane % 8.
  // Keys of a block start at a multiple of 16 and P is a multiple of 16, so
  // the swizzle term depends on the lane only: the per-lane byte offsets of
  // this warp's 16x16 sub-tiles are fixed for the whole kernel.
  constexpr int RB = D == 64 ? 64 : 128;  // bytes per smem row of a box
  const int lm_key = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lm_chunk = lane >> 4;
  uint32_t loff[GW][2];
#pragma unroll
  for (int gi = 0; gi < GW; ++gi)
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      const int ch16 = (ch0 >> 4) + gi * 4 + q2 * 2 + lm_chunk;
      // rk8v4 key boxes hold P rows of 128 bytes (no value rows)
      loff[gi][q2] = RK ? (uint32_t)((ch16 >> 3) * (P * 128) + lm_key * 128 + (((ch16 & 7) ^ (lm_key & 7)) << 4))
                        : box_off<D>(P, 0, lm_key, ch16);
    }
  // rk8v4 value rows: D / 2 bytes (32 channels per 16-byte chunk) after the
  // key boxes, 128-byte swizzle (64-byte at head_dim 128); matrices (keys
  // 0-7 | 8-15) x (chunks of two consecutive value groups)
  constexpr int RBV = D / 2;
  uint32_t vloff[RK ? GP / 2 : 1];
  if constexpr (RK) {
#pragma unroll
    for (int pv = 0; pv < GP / 2; ++pv) {
      const int c = (ch0 >> 5) + 2 * pv + lm_chunk;
      const int sw = RBV == 128 ? (c ^ (lm_key & 7)) : (c ^ ((lm_key >> 1) & 3));
      vloff[pv] = (uint32_t)(P * D + lm_key * RBV + (sw << 4));
    }
  }
  // bf16 stage: boxes of 64 channels, 128-byte rows (K rows, then V rows),
  // 128-byte swizzle. K fragments of a 16-channel chunk: matrices (keys 0-7 |
  // 8-15) x (channels 0-7 | 8-15); V^T fragments (transposed loads): matrices
  // (channels 0-7 | 8-15) x (keys 0-7 | 8-15).
  auto bf_off = [&](int row, int ch8) -> uint32_t {
    return (uint32_t)((ch8 >> 3) * (2 * P * 128) + row * 128 + (((ch8 & 7) ^ (row & 7)) << 4));
  };
  uint32_t kof[BF ? NCH : 1], vof[BF ? NCH : 1];
  if constexpr (BF) {
    const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      kof[c] = bf_off((mi & 1) * 8 + r8, (ch0 >> 3) + 2 * c + (mi >> 1));
      vof[c] = bf_off(P + (mi >> 1) * 8 + r8, (ch0 >> 3) + 2 * c + (mi & 1));
    }
  }

  uint32_t bq[NT][NCH][2];
  uint32_t bql[RK ? NT : 1][RK ? NCH : 1][2];  // rk8v4: the low fp16 part of the rotated rows
  float o[NCH][NT][4];
  float m_run[NT][2], l_run[NT][2];
  float sv[GP];  // 2^-ev of this warp's P' per group (0 before the segment's first block)
  int row_t[NT][2];  // verify column of each held row (T - 1 for padding rows)

  // Q fragments of this warp's channels, all rows of a segment's unit:
  // load_q fetches the raw bf16 pairs, convert_q turns them into fp16 pairs
  // scaled by a power of two per row (exact for elements within 2^31 of the
  // row's largest).
  auto load_q = [&](const Segment& sg) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = nt * 8 + g;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        uint2 raw = make_uint2(0u, 0u);
        if (r < M) {
          const int t = r / G, hg = r % G;
          const uint16_t* qr = p.q + (((int64_t)sg.b * p.qT + t) * p.Hq + sg.h * G + hg) * D + ch0 + c * 16;
          if constexpr (BF)  // the standard B layout: channels 2 t4, 2 t4 + 1 and 2 t4 + 8, 2 t4 + 9
            raw = make_uint2(*reinterpret_cast<const uint32_t*>(qr + 2 * t4),
                             *reinterpret_cast<const uint32_t*>(qr + 2 * t4 + 8));
          else
            raw = *reinterpret_cast<const uint2*>(qr + t4 * 4);
        }
        bq[nt][c][0] = raw.x;
        bq[nt][c][1] = raw.y;
      }
    }
  };
  // The first unit's Q rows, staged once per CTA in the (then idle) merge
  // buffer: one 16-byte load per thread instead of every warp loading all
  // rows; rows are padded by 16 bytes so the fragment reads hit distinct banks.
  constexpr int kQRow = D * 2 + 16;  // bytes per staged row
  static_assert(MROWS * kQRow <= MROWS * (D + 4) * 4, "staged Q fits the merge buffer");
  uint8_t* qstage = reinterpret_cast<uint8_t*>(mo);
  constexpr int QPT = (MROWS * (D / 8) + kThreads - 1) / kThreads;  // 16-byte pieces per thread
  uint4 qv[QPT];
  auto fetch_q = [&](const Segment& sg) {  // global -> registers (no wait)
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int i = tid + k * kThreads, r = i / (D / 8), c8 = i % (D / 8);
      qv[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r < M) {
        const int t = r / G, hg = r % G;
        qv[k] = *reinterpret_cast<const uint4*>(p.q + (((int64_t)sg.b * p.qT + t) * p.Hq + sg.h * G + hg) * D + c8 * 8);
      }
    }
  };
  auto stage_q = [&]() {  // registers -> shared memory
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int i = tid + k * kThreads, r = i / (D / 8), c8 = i % (D / 8);
      if (r < M) *reinterpret_cast<uint4*>(qstage + r * kQRow + c8 * 16) = qv[k];
    }
  };
  auto load_q_staged = [&]() {  // after a barrier that follows stage_q
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = nt * 8 + g;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        uint2 raw = make_uint2(0u, 0u);
        if (r < M) {
          if constexpr (BF)
            raw = make_uint2(*reinterpret_cast<const uint32_t*>(qstage + r * kQRow + (ch0 + c * 16 + 2 * t4) * 2),
                             *reinterpret_cast<const uint32_t*>(qstage + r * kQRow + (ch0 + c * 16 + 2 * t4 + 8) * 2));
          else
            raw = *reinterpret_cast<const uint2*>(qstage + r * kQRow + (ch0 + c * 16 + t4 * 4) * 2);
        }
        bq[nt][c][0] = raw.x;
        bq[nt][c][1] = raw.y;
      }
    }
  };
  // Each warp scales its channel slice of the unit's query rows by one power
  // of two 2^e (from the slice's largest |q| over all rows) before the fp16
  // conversion; kq = sm_scale log2(e) 2^-e undoes it on the partial scores
  // (folded into the key scales: no work per block).
  float kq = p.scale2;
  // rk8v4: each 64-channel group of a row becomes H64 q / 8 (butterflies in
  // fp32 over the channel-index bits: bits 0, 1 and 4, 5 are the thread's
  // own registers -- channel 16 cc + 4 t4 + 2 h + j of a group sits in
  // bq[.][4 gi + cc][h], half j -- and bits 2, 3 its t4 neighbours'), then
  // scaled like the other formats and split into fp16 hi + lo.
  auto convert_q_rk = [&]() {
    float qf[NT][GW][16];  // [row tile][group][cc * 4 + h * 2 + j]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int gi = 0; gi < GW; ++gi)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            qf[nt][gi][cc * 4 + h * 2] = bf16_lo(bq[nt][gi * 4 + cc][h]);
            qf[nt][gi][cc * 4 + h * 2 + 1] = bf16_hi(bq[nt][gi * 4 + cc][h]);
          }
    float m = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int gi = 0; gi < GW; ++gi) {
        float* v = qf[nt][gi];
        // register bits: j (stride 1), h (stride 2), cc (strides 4, 8)
#pragma unroll
        for (int st = 1; st < 16; st <<= 1)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if ((i & st) == 0) {
              const float a = v[i], b = v[i + st];
              v[i] = a + b;
              v[i + st] = a - b;
            }
        // lane bits: t4 bit 0 (channel bit 2), t4 bit 1 (channel bit 3)
#pragma unroll
        for (int lb = 1; lb <= 2; lb <<= 1) {
          const bool upper = (t4 & lb) != 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float o2 = __shfl_xor_sync(0xffffffffu, v[i], lb);
            v[i] = upper ? o2 - v[i] : v[i] + o2;
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          v[i] *= 0.125f;
          m = fmaxf(m, fabsf(v[i]));
        }
      }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = q_norm_exp(m);
    const float qs = pow2i(e);
    kq = p.scale2 * pow2i(-e);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int gi = 0; gi < GW; ++gi)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float x0 = qf[nt][gi][cc * 4 + h * 2] * qs, x1 = qf[nt][gi][cc * 4 + h * 2 + 1] * qs;
            const __half2 hh = __floats2half2_rn(x0, x1);
            const float2 hf = __half22float2(hh);
            bq[nt][gi * 4 + cc][h] = *reinterpret_cast<const uint32_t*>(&hh);
            if constexpr (RK) bql[nt][gi * 4 + cc][h] = pack_f16(x0 - hf.x, x1 - hf.y);
          }
  };
  auto convert_q = [&]() {
    kq = p.scale2;
    if constexpr (BF) return;  // bf16 operands as they are, no scaling
    if constexpr (RK) {
      convert_q_rk();
      return;
    }
    float m = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) m = fmaxf(m, fmaxf(fabsf(bf16_lo(bq[nt][c][h])), fabsf(bf16_hi(bq[nt][c][h]))));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = q_norm_exp(m);
    const float qs = pow2i(e);
    kq = p.scale2 * pow2i(-e);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          bq[nt][c][h] = pack_f16(bf16_lo(bq[nt][c][h]) * qs, bf16_hi(bq[nt][c][h]) * qs);
  };

  // Every global read of the prologue -- the first unit's Q (converted at
  // first use) and the page coordinates of the CTA's pages up to the cache
  // size -- goes out before the first page load: a load this SM issues after
  // its page loads returns only behind their data (several microseconds).
  int64_t x = x_begin;
  Segment seg;
  bool have = next_segment(sh, pre, x, x_end, seg);
  if (have) fetch_q(seg);
  const int ncache = total < kPidCache ? total : kPidCache;
  for (int q = tid; q < ncache; q += kThreads) pid[q] = page_coord(p, sh, pre, x_begin, q);
  if (have) stage_q();
  __syncthreads();
  if (p.early) chain_wait();  // the pages may hold the preceding append's rows
  // The first S pages, issued in order by one thread (the copy unit then
  // completes page 0 first). Each issue waits until the unit accepts the
  // copy, so the issuer is the last warp, whose first block is in page 1.
  if (tid == kThreads - 32) {
    const int n0 = total < S ? total : S;
    for (int q = 0; q < n0; ++q) {
      if (!p.issuable(q)) break;
      if constexpr (RK)
        issue_page_rk<D>(p, &tmap, &tmapv, pid[q], stage0 + q * geo.stage_bytes, smem_u32(&full_bar[q]));
      else
        issue_page<D, BF>(p, &tmap, pid[q], stage0 + q * geo.stage_bytes, smem_u32(&full_bar[q]));
      icnt[q] = 1;
    }
  }

  const int bpp_sh = (BPP & (BPP - 1)) == 0 ? __ffs(BPP) - 1 : -1;  // blocks per page, as a shift
  int q_cur = 0, s_cur = 0;  // last page whose stage was located, and that stage
  uint32_t par_cur = 0;
  int page_seq = 0;   // CTA page number of the current segment's first page
  int jn = team;       // next block of this team
  // With up to two row tiles the next unit's Q rows are fetched (one or two
  // 16-byte pieces per thread) at the start of the current segment -- a
  // load issued at its end would return behind the pages in flight -- and
  // staged through the merge buffer after the merge; with more tiles the
  // registers are not there, and Q loads at the segment start.
  constexpr bool kEarlyQ = NT <= 2;
  bool staged = true;  // the current unit's Q sits in the merge buffer
  while (have) {
    const int L = lens[seg.b];
    if (staged) load_q_staged();
    else load_q(seg);
    convert_q();
    if constexpr (kEarlyQ) {
      int64_t xn = x;
      Segment sn;
      if (next_segment(sh, pre, xn, x_end, sn)) fetch_q(sn);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r2 = nt * 8 + 2 * t4 + e;
        row_t[nt][e] = r2 < M ? r2 / G : T - 1;
        m_run[nt][e] = -INFINITY;
        l_run[nt][e] = 0.f;
      }
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[c][nt][k] = 0.f;
    }
#pragma unroll
    for (int gi = 0; gi < GP; ++gi) sv[gi] = BF ? 1.f : 0.f;

    // this team's blocks of the segment: CTA-wide block numbers jn = team,
    // team + NTEAMS, ... (4 blocks of 16 keys per 64-key page)
    const int seg_first = page_seq, seg_pages = seg.page_end - seg.page_begin;
    for (; jn < (seg_first + seg_pages) * BPP; jn += NTEAMS) {
      const int q = bpp_sh >= 0 ? jn >> bpp_sh : jn / BPP;  // CTA page number
      const int kb = jn - q * BPP;                           // block in page
      const int pi = seg.page_begin + (q - seg_first);
      while (q_cur < q) {  // stage and phase of page q, advanced without a division
        ++q_cur;
        if (++s_cur == S) {
          s_cur = 0;
          par_cur ^= 1u;
        }
      }
      const int s = s_cur;
      const uint32_t par = par_cur;
      const uint32_t st = stage0 + s * geo.stage_bytes;
      // [P][G_ALL] key scales (fp32 or fp16), then [P][GV_ALL] value scales
      const uint8_t* ks_s = smem + s * geo.stage_bytes + (RK ? 3 * P * D / 2 : 2 * P * D);
      const uint8_t* vs_s = ks_s + P * G_ALL * sb;
      {
        // after one wait of the CTA has run out, no wait blocks any more (the
        // blocks run without data and nothing more is issued; the end of the
        // kernel waits for the copies that were)
        if (!*abort_flag && !mbar_wait(smem_u32(&full_bar[s]), par, p.wait_cycles)) {
          if (lane == 0) flag(p.status, NK_DEVFLAG_TIMEOUT);
          *abort_flag = 1;
        }
        const int key0 = kb * 16;
        const int pos0 = pi * P + key0;  // sequence position of the block's key 0
        if (pos0 < L) {
          // ---- QK: per-group fp32 partial dot products (GW*NT independent accumulators)
          float acc[GW][NT][4];
#pragma unroll
          for (int gi = 0; gi < GW; ++gi)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int k = 0; k < 4; ++k) acc[gi][nt][k] = 0.f;
          if constexpr (BF) {
            // bf16 K fragments straight from the tile, one ldmatrix per 16 channels
#pragma unroll
            for (int gi = 0; gi < GW; ++gi)
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(st + key0 * 128 + kof[gi * 4 + cc], a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma16816_bf16(acc[gi][nt], a0, a1, a2, a3, bq[nt][gi * 4 + cc][0], bq[nt][gi * 4 + cc][1]);
              }
          } else {
            uint32_t kw[GW][4][2];  // [group][chunk][keys 0-7 | 8-15]
            const uint32_t kbase = st + key0 * RB;
#pragma unroll
            for (int gi = 0; gi < GW; ++gi)
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2)
                ldsm_x4(kbase + loff[gi][q2], kw[gi][q2 * 2][0], kw[gi][q2 * 2][1], kw[gi][q2 * 2 + 1][0],
                        kw[gi][q2 * 2 + 1][1]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int gi = 0; gi < GW; ++gi) {
                const uint32_t lo = kw[gi][cc][0] ^ bias, hi = kw[gi][cc][1] ^ bias;
                const uint32_t a0 = i8x2_to_f16x2(lo, 0x4140), a2 = i8x2_to_f16x2(lo, 0x4342);
                const uint32_t a1 = i8x2_to_f16x2(hi, 0x4140), a3 = i8x2_to_f16x2(hi, 0x4342);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma16816(acc[gi][nt], a0, a1, a2, a3, bq[nt][gi * 4 + cc][0], bq[nt][gi * 4 + cc][1]);
                if constexpr (RK) {  // the rotated rows' low parts
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma16816(acc[gi][nt], a0, a1, a2, a3, bql[nt][gi * 4 + cc][0], bql[nt][gi * 4 + cc][1]);
                }
              }
          }
          float sc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) sc[nt][k] = 0.f;
#pragma unroll
          for (int gi = 0; gi < GW; ++gi) {
            const float k0 = BF ? p.scale2 : ld_scale(ks_s, (key0 + g) * G_ALL + grp0 + gi, sb) * kq;
            const float k1 = BF ? p.scale2 : ld_scale(ks_s, (key0 + g + 8) * G_ALL + grp0 + gi, sb) * kq;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              sc[nt][0] = fmaf(k0, acc[gi][nt][0], sc[nt][0]);
              sc[nt][1] = fmaf(k0, acc[gi][nt][1], sc[nt][1]);
              sc[nt][2] = fmaf(k1, acc[gi][nt][2], sc[nt][2]);
              sc[nt][3] = fmaf(k1, acc[gi][nt][3], sc[nt][3]);
            }
          }

          // ---- team exchange: every warp of the team sums the CS partials in warp order
          if constexpr (CS > 1) {
            const int buf = (jn / NTEAMS) & 1;
            float* xb = xch + (((size_t)team * 2 + buf) * CS) * (NT * 4 * 32);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int k = 0; k < 4; ++k) xb[(wit * NT * 4 + nt * 4 + k) * 32 + lane] = sc[nt][k];
            named_bar(2 + team, CS * 32);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float sum = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < CS; ++w2) {
                  const float v = (w2 == wit) ? sc[nt][k] : xb[(w2 * NT * 4 + nt * 4 + k) * 32 + lane];
                  sum = (w2 == 0) ? v : sum + v;
                }
                sc[nt][k] = sum;
              }
          }

          // ---- causal / context mask (only blocks that reach past L - T)
          const bool need_mask = pos0 + 15 > L - T;
          bool valid0 = true, valid1 = true;
          if (need_mask) {
            valid0 = pos0 + g < L;
            valid1 = pos0 + g + 8 < L;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int key = g + (k >> 1) * 8;
                if (pos0 + key > L - T + row_t[nt][k & 1]) sc[nt][k] = -INFINITY;
              }
          }

          // ---- online softmax (base 2). The reference m_run is raised only when a
          // score passes it by more than 8 (p would exceed 2^8); the softmax
          // does not depend on the reference, so most blocks skip the row-max
          // reduction and the accumulator rescale.
          bool over = false;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) over |= sc[nt][k] > m_run[nt][k & 1] + 8.f;
          if (__any_sync(0xffffffffu, over)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float mb = fmaxf(sc[nt][e], sc[nt][e + 2]);
                mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
                mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
                mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
                const float mnew = fmaxf(m_run[nt][e], mb);
                if (mnew > m_run[nt][e]) {
                  const float alpha = ex2(m_run[nt][e] - mnew);  // 0 while the row was empty
                  l_run[nt][e] *= alpha;
#pragma unroll
                  for (int c = 0; c < NCH; ++c) {
                    o[c][nt][e] *= alpha;
                    o[c][nt][e + 2] *= alpha;
                  }
                  m_run[nt][e] = mnew;
                }
              }
          }
          float pr[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float mu0 = m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0];
            const float mu1 = m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1];
            pr[nt][0] = ex2(sc[nt][0] - mu0);
            pr[nt][1] = ex2(sc[nt][1] - mu1);
            pr[nt][2] = ex2(sc[nt][2] - mu0);
            pr[nt][3] = ex2(sc[nt][3] - mu1);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            l_run[nt][0] += pr[nt][0] + pr[nt][2];
            l_run[nt][1] += pr[nt][1] + pr[nt][3];
          }

          if constexpr (BF) {
            // ---- PV with P as bf16 hi + lo (16 significant bits) and the bf16 V^T
            uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const __nv_bfloat162 h01 = __floats2bfloat162_rn(pr[nt][0], pr[nt][1]);
              const __nv_bfloat162 h23 = __floats2bfloat162_rn(pr[nt][2], pr[nt][3]);
              const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
              const __nv_bfloat162 l01 = __floats2bfloat162_rn(pr[nt][0] - f01.x, pr[nt][1] - f01.y);
              const __nv_bfloat162 l23 = __floats2bfloat162_rn(pr[nt][2] - f23.x, pr[nt][3] - f23.y);
              bh[nt][0] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&h01));
              bh[nt][1] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&h23));
              bl[nt][0] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&l01));
              bl[nt][1] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&l23));
            }
            // slots past ctx_len may hold any bits (NaN): their V is zeroed, not
            // multiplied by p = 0. This thread's keys: 2 t4 + {0, 1} (a0, a1) and
            // 2 t4 + 8 + {0, 1} (a2, a3) of the block.
            uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
            if (need_mask) {
              const int kq = pos0 + 2 * t4;
              vmask_lo = (kq < L ? 0x0000ffffu : 0u) | (kq + 1 < L ? 0xffff0000u : 0u);
              vmask_hi = (kq + 8 < L ? 0x0000ffffu : 0u) | (kq + 9 < L ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(st + key0 * 128 + vof[c], a0, a1, a2, a3);
              a0 &= vmask_lo;
              a1 &= vmask_lo;
              a2 &= vmask_hi;
              a3 &= vmask_hi;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma16816_bf16(o[c][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma16816_bf16(o[c][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
            }
          } else {
          // ---- PV with P' = p * Vs split into fp16 hi + lo
            // P' window of each of this warp's groups (bits as in ev_update's
            // window: a Vs 2^-ev above 2^6, or one at least 2^-10); the
            // exponents move only when a group leaves it
            const int vgrp0 = RK ? ch0 / kRkVGroup : grp0;
            // the value scales of this thread's two keys (g, g + 8), once per
            // block for the window and P' (stale slots past ctx_len may hold
            // NaN scales: 0 there)
            float vsk[GP][2];
#pragma unroll
            for (int gi = 0; gi < GP; ++gi) {
              vsk[gi][0] = valid0 ? ld_scale(vs_s, (key0 + g) * GV_ALL + vgrp0 + gi, sb) : 0.f;
              vsk[gi][1] = valid1 ? ld_scale(vs_s, (key0 + g + 8) * GV_ALL + vgrp0 + gi, sb) : 0.f;
            }
            {
              uint32_t wb = 0u;
#pragma unroll
              for (int gi = 0; gi < GP; ++gi) {
                const float a0 = vsk[gi][0], a1 = vsk[gi][1];
                const float tv = fmaxf(a0, a1) * sv[gi];
                wb |= (tv > 64.f ? 1u : 0u) << gi;
                wb |= (tv >= 0.0009765625f ? 1u : 0u) << (8 + gi);
              }
              wb = __reduce_or_sync(0xffffffffu, wb);
              const uint32_t moving = ((wb & 0xffu) | (~(wb >> 8) & 0xffu)) & ((1u << GP) - 1u);
              if (moving) {
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) {
                  if (!((moving >> gi) & 1u)) continue;
                  const float a0 = vsk[gi][0], a1 = vsk[gi][1];
                  const uint32_t mxb = __reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(a0, a1)));
                  int ev = sv[gi] == 0.f ? kEvUnset : -exp_of(sv[gi]);
                  float beta;
                  if (mxb != 0u && ev_update(ev, exp_of(__uint_as_float(mxb)), beta)) {
                    sv[gi] = pow2i(-ev);
#pragma unroll
                    for (int cc = 0; cc < CPG; ++cc)
#pragma unroll
                      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int k = 0; k < 4; ++k) o[gi * CPG + cc][nt][k] *= beta;
                  }
                }
              }
            }
            // P' of group gi as the B fragments of the product (hi, lo)
            auto p_frags = [&](int gi, uint32_t (&bh)[NT][2], uint32_t (&bl)[NT][2]) {
              const float v0 = vsk[gi][0] * sv[gi], v1 = vsk[gi][1] * sv[gi];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const float q0 = pr[nt][0] * v0, q1 = pr[nt][1] * v0, q2 = pr[nt][2] * v1, q3 = pr[nt][3] * v1;
                const __half2 h01 = __floats2half2_rn(q0, q1), h23 = __floats2half2_rn(q2, q3);
                const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                const uint32_t l01 = pack_f16(q0 - f01.x, q1 - f01.y), l23 = pack_f16(q2 - f23.x, q3 - f23.y);
                bh[nt][0] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&h01));
                bh[nt][1] = movmatrix_t(*reinterpret_cast<const uint32_t*>(&h23));
                bl[nt][0] = movmatrix_t(l01);
                bl[nt][1] = movmatrix_t(l23);
              }
            };
            if constexpr (RK) {
              // Two value groups (two 16-byte chunks of 32 channels) per
              // transposed load: register vw[j][h] holds, for keys 2 t4 and
              // 2 t4 + 1 (+ 8 h), bytes 2 g and 2 g + 1 of chunk j, i.e.
              // channels 4 g .. 4 g + 3. Accumulator chunk 2 gi + u holds
              // channels 32 gi + 4 g + 2 u (rows g) and + 1 (rows g + 8).
#pragma unroll
              for (int pv = 0; pv < GP / 2; ++pv) {
                uint32_t vw[2][2];
                ldsm_x4_t(st + key0 * RBV + vloff[pv], vw[0][0], vw[0][1], vw[1][0], vw[1][1]);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const int gi = 2 * pv + j;
                  uint32_t bh[NT][2], bl[NT][2];
                  p_frags(gi, bh, bl);
                  const uint32_t w0 = vw[j][0], w1 = vw[j][1], w08 = w0 >> 8, w18 = w1 >> 8;
                  uint32_t av[2][4];
                  av[0][0] = nib_lo(w0);
                  av[0][1] = nib_hi(w0);
                  av[0][2] = nib_lo(w1);
                  av[0][3] = nib_hi(w1);
                  av[1][0] = nib_lo(w08);
                  av[1][1] = nib_hi(w08);
                  av[1][2] = nib_lo(w18);
                  av[1][3] = nib_hi(w18);
#pragma unroll
                  for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                      mma16816(o[gi * 2 + u][nt], av[u][0], av[u][1], av[u][2], av[u][3], bh[nt][0], bh[nt][1]);
#pragma unroll
                  for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                      mma16816(o[gi * 2 + u][nt], av[u][0], av[u][1], av[u][2], av[u][3], bl[nt][0], bl[nt][1]);
                }
              }
            } else {
#pragma unroll
              for (int gi = 0; gi < GW; ++gi) {
                uint32_t vw[4][2];  // [chunk][keys 0-7 | 8-15], transposed fragments
                const uint32_t vbase = st + (P + key0) * RB;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2)
                  ldsm_x4_t(vbase + loff[gi][q2], vw[q2 * 2][0], vw[q2 * 2][1], vw[q2 * 2 + 1][0], vw[q2 * 2 + 1][1]);
                uint32_t bh[NT][2], bl[NT][2];
                p_frags(gi, bh, bl);
                uint32_t av[4][4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                  const uint32_t w0 = vw[cc][0] ^ bias, w1 = vw[cc][1] ^ bias;
                  av[cc][0] = i8x2_to_f16x2(w0, 0x4240);
                  av[cc][1] = i8x2_to_f16x2(w0, 0x4341);
                  av[cc][2] = i8x2_to_f16x2(w1, 0x4240);
                  av[cc][3] = i8x2_to_f16x2(w1, 0x4341);
                }
                // all hi products first, then all lo: 4*NT independent accumulators between dependent pairs
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma16816(o[gi * 4 + cc][nt], av[cc][0], av[cc][1], av[cc][2], av[cc][3], bh[nt][0], bh[nt][1]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma16816(o[gi * 4 + cc][nt], av[cc][0], av[cc][1], av[cc][2], av[cc][3], bl[nt][0], bl[nt][1]);
              }
            }
          }
        }
        // ---- release the stage; its last reader loads the page S ahead into it
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&empty_bar[s]));
          if (atomicAdd(&cnt[s], 1) == per_stage - 1) {
            cnt[s] = 0;
            const int qn = q + S;
            if (qn < total && p.issuable(qn) && !*abort_flag) {
              // every reader arrived before its increment: the phase is complete
              if (mbar_wait(smem_u32(&empty_bar[s]), par, p.wait_cycles)) {
                const int zn = qn < kPidCache ? pid[qn] : page_coord(p, sh, pre, x_begin, qn);
                if constexpr (RK)
                  issue_page_rk<D>(p, &tmap, &tmapv, zn, st, smem_u32(&full_bar[s]));
                else
                  issue_page<D, BF>(p, &tmap, zn, st, smem_u32(&full_bar[s]));
                ++icnt[s];
              } else {
                flag(p.status, NK_DEVFLAG_TIMEOUT);
                *abort_flag = 1;
              }
            }
          }
        }
      }
    }

    page_seq += seg_pages;

    // the accumulators hold O 2^-ev per group: back to O
#pragma unroll
    for (int gi = 0; gi < GP; ++gi) {
      if (BF || sv[gi] == 0.f) continue;
      const float f = pow2i(-exp_of(sv[gi]));
#pragma unroll
      for (int cc = 0; cc < CPG; ++cc)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[gi * CPG + cc][nt][k] *= f;
    }

    const bool last_seg = x >= x_end;
    // channel (from the warp's first) of accumulator chunk c, element k: INT8
    // 16 c + 2 g + (k >> 1) (the V fragments' byte order), rk8v4
    // 32 (c >> 1) + 4 g + 2 (c & 1) + (k >> 1) (the nibble order), bf16
    // 16 c + g + 8 (k >> 1). INT8 and rk8v4 keep elements k and k + 2 in
    // adjacent channels (cpair: the first of the two).
    auto cpair = [&](int c) { return RK ? 32 * (c >> 1) + 4 * g + 2 * (c & 1) : 16 * c + 2 * g; };
    auto och = [&](int c, int k) { return BF ? 16 * c + g + 8 * (k >> 1) : cpair(c) + (k >> 1); };

    // ---- merge the teams of this segment and write the result
    // row sums: reduce the per-lane partial l over the 8 lanes of a row
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l_run[nt][e];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l_run[nt][e] = v;
      }
    __syncthreads();  // all blocks of the segment read; previous merge buffers free
    if (wit == 0 && g == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = nt * 8 + 2 * t4 + e;
          tm_m[team * MROWS + r] = m_run[nt][e];
          tm_l[team * MROWS + r] = l_run[nt][e];
        }
    }
    float* facs = tm_l + NTEAMS * MROWS;   // [NTEAMS][MROWS]: weight of a team's rows
    float* row_lse = facs + NTEAMS * MROWS;
    // After the CTA's last segment the stage ring is idle (every issued page
    // has been consumed), so each team can park its accumulator there and one
    // pass merges them; otherwise the teams add into mo one after another.
    constexpr int kSlot = MROWS * (D + 4);
    const bool parked = last_seg && (size_t)NTEAMS * kSlot * 4 <= (size_t)S * geo.stage_bytes;
    float* acc_buf = parked ? reinterpret_cast<float*>(smem) + team * kSlot : mo;
    if (parked) {
      // INT8: fragment elements k and k + 2 are adjacent channels of one row
      // (16 c + 2 g, + 1: the V fragments' byte order); bf16: channels
      // 16 c + g and 16 c + g + 8 (ldmatrix order)
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float* row = acc_buf + (nt * 8 + 2 * t4 + e) * (D + 4) + ch0;
            if constexpr (BF) {
              row[c * 16 + g] = o[c][nt][e];
              row[c * 16 + g + 8] = o[c][nt][e + 2];
            } else {
              *reinterpret_cast<float2*>(row + cpair(c)) = make_float2(o[c][nt][e], o[c][nt][e + 2]);
            }
          }
    }
    __syncthreads();
    // team weights of each row: NTEAMS consecutive lanes per row, reduced by shuffles
    for (int base = 0; base < MROWS * NTEAMS; base += kThreads) {
      if (base + warp * 32 < MROWS * NTEAMS) {  // warp-uniform
        const int j = base + tid;
        const bool act = j < MROWS * NTEAMS;
        const int r = act ? j / NTEAMS : 0, tm = j % NTEAMS;
        const float mt = act ? tm_m[tm * MROWS + r] : -INFINITY;
        float mx = mt;
#pragma unroll
        for (int o2 = 1; o2 < NTEAMS; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float wgt = (mt == -INFINITY) ? 0.f : ex2(mt - mx);
        float lsum = act ? wgt * tm_l[tm * MROWS + r] : 0.f;
#pragma unroll
        for (int o2 = 1; o2 < NTEAMS; o2 <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o2);
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        if (act) {
          facs[tm * MROWS + r] = wgt * inv;
          if (tm == 0) row_lse[r] = lsum > 0.f ? (mx + log2f(lsum)) * kLn2 : -INFINITY;
        }
      }
    }
    __syncthreads();
    if (!parked) {
      // The teams add their weighted accumulators into mo in NTEAMS rounds.
      float f[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) f[nt][e] = facs[team * MROWS + nt * 8 + 2 * t4 + e];
      if constexpr (NT <= 2) {
        // In round rd team tm takes its 16-channel chunks c with
        // c = tm + rd (mod NTEAMS): the teams of a round touch disjoint
        // chunks, and every chunk gets one team per round (fixed order).
        for (int rd = 0; rd < NTEAMS; ++rd) {
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            if (((c - team - rd) & (NTEAMS - 1)) != 0) continue;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float* row = mo + (nt * 8 + 2 * t4 + e) * (D + 4) + ch0;
                if constexpr (BF) {  // channels 16 c + g, 16 c + g + 8
                  const float p0 = rd == 0 ? 0.f : row[c * 16 + g], p1 = rd == 0 ? 0.f : row[c * 16 + g + 8];
                  row[c * 16 + g] = fmaf(o[c][nt][e], f[nt][e], p0);
                  row[c * 16 + g + 8] = fmaf(o[c][nt][e + 2], f[nt][e], p1);
                } else {
                  // fragment elements e and e + 2 are adjacent channels of one row
                  float2* dst = reinterpret_cast<float2*>(row + cpair(c));
                  const float2 prev = rd == 0 ? make_float2(0.f, 0.f) : *dst;
                  *dst = make_float2(fmaf(o[c][nt][e], f[nt][e], prev.x), fmaf(o[c][nt][e + 2], f[nt][e], prev.y));
                }
              }
          }
          __syncthreads();
        }
      } else {
        // more row tiles: team tm adds all its chunks in round tm (fewer
        // registers), all of a chunk's loads issued before its stores
        for (int tm = 0; tm < NTEAMS; ++tm) {
          if (team == tm) {
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
              float prev[NT][4];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  prev[nt][k] = (tm == 0) ? 0.f : mo[(nt * 8 + 2 * t4 + (k & 1)) * (D + 4) + ch0 + och(c, k)];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mo[(nt * 8 + 2 * t4 + (k & 1)) * (D + 4) + ch0 + och(c, k)] =
                      fmaf(o[c][nt][k], f[nt][k & 1], prev[nt][k]);
            }
          }
          __syncthreads();
        }
      }
    }
    // normalize (weights already include 1/sum) and store, 4 channels a thread
    const int64_t slot = (int64_t)blockIdx.x + seg.u;
    const float* park = reinterpret_cast<const float*>(smem);
    for (int i = tid; i < M * (D / 4); i += kThreads) {
      const int r = i / (D / 4), ch = (i % (D / 4)) * 4;
      float4 val;
      if (parked) {
        val = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int tm = 0; tm < NTEAMS; ++tm) {
          const float f = facs[tm * MROWS + r];
          const float4 v = *reinterpret_cast<const float4*>(park + tm * kSlot + r * (D + 4) + ch);
          val.x = fmaf(v.x, f, val.x);
          val.y = fmaf(v.y, f, val.y);
          val.z = fmaf(v.z, f, val.z);
          val.w = fmaf(v.w, f, val.w);
        }
      } else {
        val = *reinterpret_cast<const float4*>(mo + r * (D + 4) + ch);
      }
      if (!(isfinite(val.x) && isfinite(val.y) && isfinite(val.z) && isfinite(val.w))) flag(p.status, NK_DEVFLAG_RANGE);
      if (seg.whole) {
        const int t = r / G, hg = r % G;
        const uint32_t w0 = f32_to_bf16(val.x) | ((uint32_t)f32_to_bf16(val.y) << 16);
        const uint32_t w1 = f32_to_bf16(val.z) | ((uint32_t)f32_to_bf16(val.w) << 16);
        *reinterpret_cast<uint2*>(p.out + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * D + ch) = make_uint2(w0, w1);
      } else {
        *reinterpret_cast<float4*>(p.part_o + (slot * M + r) * D + ch) = val;
        if (ch == 0) p.part_lse[slot * M + r] = row_lse[r];
      }
    }
    have = next_segment(sh, pre, x, x_end, seg);
    staged = kEarlyQ && have;
    if (staged) {
      __syncthreads();  // the merge buffer has been read
      stage_q();
      __syncthreads();
    }
  }
  // After a timed-out wait some copies may still be in flight: the last copy
  // issued into each stage lands (bounded waits) before the CTA exits. Every
  // issue came before the last merge's barriers. Without a timeout all of
  // them were consumed already.
  if (tid == kThreads - 32) {
    for (int s2 = 0; s2 < S; ++s2)
      if (icnt[s2] > 0) (void)mbar_wait(smem_u32(&full_bar[s2]), (uint32_t)(icnt[s2] - 1) & 1u, p.wait_cycles);
  }
}

}  // namespace mma
}  // namespace nk
