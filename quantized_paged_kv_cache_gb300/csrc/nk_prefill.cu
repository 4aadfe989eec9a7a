// nk_prefill.cu -- chunked-prefill attention over the paged INT8 group-64
// cache: the T query tokens of a prefill chunk (whose K/V rows the chunk's
// kv_cache_append has already stored) attend to every cached key before them
// and causally to each other ("NInfer-4090" README, "What this fork changes":
// the INT8 attention prefill on the append shape, and the causal-tile split of
// the key blocks into unmasked interior blocks and masked boundary blocks;
// "NInfer-3090" README, "Capabilities": prefill in chunks).
//
// One CTA computes 128 query rows of one (sequence, kv-head) unit, rows
// numbered token-major (row r = token r / G, q-head r % G of the kv-head's G),
// so every K/V page a CTA stages serves all G heads of its tokens. 8 warps of
// 16 rows each, FlashAttention-style on mma.sync m16n8k16 (fp16 operands,
// fp32 accumulate):
//   QK  S[row][key] = Q[row][ch] K^T[ch][key]: A = the warp's Q rows (held in
//       registers for the whole tile, scaled by a power of two into the fp16
//       range), B = K codes widened to fp16 exactly (ldmatrix on the staged
//       page, byte permute), one fp32 accumulator per 64-channel group,
//       scaled by the keys' group scales and summed;
//   online softmax in base 2 with a lazy reference per row (raised, and the
//       accumulator rescaled, only when a score passes it by more than 8);
//   PV  O[row][ch] += P'[row][key] V[key][ch] per group, with P' = p Vs 2^-ev
//       split into fp16 hi + lo (two MMAs) and V codes widened exactly
//       (ldmatrix.trans); the score accumulators' layout is the A layout of
//       the next product, so P' needs no shuffle.
// Pages arrive as in the decode kernels (TMA boxes of the K|V codes plus bulk
// copies of the scale arrays into a shared-memory ring; the last warp to
// release a stage loads the page S ahead into it). Only the key blocks past
// the first row's causal limit take the masked path. Every wait is bounded.
//
// The fp32 accumulation inside mma.sync does not round each sum to nearest,
// and its error grows with the number of products one accumulator absorbs: a
// CTA of a long-context chunk runs every key of the sequence through one
// accumulator (2 x 8,192 MMAs at 131,072 keys). Every kFoldKeys keys each
// thread therefore folds its accumulator into a running total kept in tensor
// memory (its own lanes and columns; rounded to nearest, once per fold) and
// restarts it from zero.
#include "nk_decode_mma.cuh"

namespace nk {
namespace mma {
cudaError_t make_pool_map(const DecodeParams& p, CUtensorMap* map, int part = 0);
}

namespace pf {

using namespace mma;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = kWarps * 16;  // query rows per CTA
constexpr int kFoldKeys = 2048;     // keys per accumulator run between folds

// tensor-memory moves of 16 consecutive 32-bit columns of the thread's lane
__device__ __forceinline__ void tm_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tm_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// Q rows live in shared memory at head_dim 256 (with the output accumulator
// they would not fit the registers), padded so a fragment load hits every bank
// once per 256 bytes.
__host__ __device__ constexpr bool q_in_smem(int D) { return D == 256; }
__host__ __device__ constexpr int q_stride(int D) { return D * 2 + 32; }

struct Plan {
  int stage_bytes, stages, q_off, bar_off, total;
};

__host__ __device__ inline Plan plan(int fmt, int D, int P) {
  Plan L;
  const int kv_bytes = 2 * P * D;
  const int sc_bytes = 2 * P * (D / kGroup) * (fmt == kFmtI8F16 ? 2 : 4);
  const int q_bytes = q_in_smem(D) ? kRows * q_stride(D) : 0;
  L.stage_bytes = round_up(kv_bytes + sc_bytes, 1024);
  int s = (kSmemLimit - 1024 - 256 - q_bytes) / L.stage_bytes;
  if (s > 6) s = 6;
  L.stages = s;
  L.q_off = s * L.stage_bytes;
  L.bar_off = L.q_off + q_bytes;
  L.total = L.bar_off + 256 + 1024;
  return L;
}

// D: head dim; FMT: kFmtI8F32 or kFmtI8F16. p.n_ctas = B * Hkv * tiles, the
// tiles of a unit consecutive; p.T = the chunk's tokens.
template <int D, int FMT>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmap,
                                                              const DecodeParams p) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
  chain_wait();
  chain_release();
  constexpr int NCH = D / 16;      // 16-channel chunks
  constexpr int GW = D / kGroup;   // groups
  constexpr int sb = FMT == kFmtI8F16 ? 2 : 4;
  constexpr int RB = D == 64 ? 64 : 128;  // bytes per smem row of a box
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Plan PL = plan(FMT, D, p.P);
  const int S = PL.stages;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + PL.bar_off);
  uint64_t* empty_bar = full_bar + 8;
  int* cnt = reinterpret_cast<int*>(empty_bar + 8);  // [8]
  int* icnt = cnt + 8;                                 // [8] copies issued into each stage
  volatile int* abort_flag = icnt + 8;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int P = p.P, BPP = P / 16;
  const int G = p.G, T = p.T, MR = G * T;  // query rows of a unit
  const int tiles = (MR + kRows - 1) / kRows;
  const int u = blockIdx.x / tiles, tile = blockIdx.x % tiles;
  const int b = u / p.Hkv, h = u % p.Hkv;
  const int L = p.ctx[b];
  if (L < T || L > p.max_ctx || (int64_t)L > (int64_t)p.max_pages * P) {
    if (tile == 0 && tid == 0) flag(p.status, NK_DEVFLAG_BAD_CTX);
    return;
  }
  const int r0 = tile * kRows;                       // first row of the CTA
  const int r1 = r0 + kRows < MR ? r0 + kRows : MR;  // one past its last
  const int last_key = L - T + (r1 - 1) / G;         // largest key any row of the CTA sees
  const int npages = last_key / P + 1;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kWarps);
      cnt[s] = 0;
      icnt[s] = 0;
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // tensor memory of the folded totals: D columns, warps w and w + 4 share
  // the lanes 32 (w % 4) .. + 31 and take one half of the columns each
  uint32_t* tslot = reinterpret_cast<uint32_t*>(icnt + 9);
  constexpr uint32_t kTmCols = D;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm_base = *tslot + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(warp >> 2) * (NCH * 8);
  const uint32_t stage0 = smem_u32(smem);
  auto page_z = [&](int pi) -> int {  // pool coordinate of the unit's page pi (-1: id out of range)
    const int page = __ldg(p.bt + (int64_t)b * p.max_pages + pi);
    return (page < 0 || page >= p.num_pages) ? -1 : page * p.Hkv + h;
  };
  if (tid == 0) {
    const int n0 = npages < S ? npages : S;
    for (int q = 0; q < n0; ++q) {
      if (!p.issuable(q)) break;
      issue_page<D>(p, &tmap, page_z(q), stage0 + q * PL.stage_bytes, smem_u32(&full_bar[q]));
      icnt[q] = 1;
    }
  }

  // ---- this warp's 16 rows: Q as A fragments (channel order of the widened
  // K codes: k-index 2 t4, 2 t4 + 1 <-> channels 4 t4, 4 t4 + 1 and 2 t4 + 8,
  // 2 t4 + 9 <-> 4 t4 + 2, 4 t4 + 3 of each 16-channel chunk), scaled by one
  // power of two into the fp16 range
  const int rw = r0 + warp * 16;
  const int ra = rw + g, rb = rw + g + 8;  // this thread's rows
  constexpr bool QS = q_in_smem(D);
  uint32_t qa[QS ? 1 : NCH][4];
  float kq;  // sm_scale log2(e) 2^-e
  uint8_t* qsm = smem + PL.q_off + warp * 16 * q_stride(D);  // this warp's rows (QS)
  if constexpr (QS) {
    // 16 rows x D channels, 16-byte pieces: the warp's largest |q|, then the
    // rows scaled and converted to fp16 in place (same channel order as Q)
    constexpr int PPR = D / 8;  // pieces per row
    uint4 piece[16 * PPR / 32];
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 16 * PPR / 32; ++k) {
      const int i = lane + 32 * k, rr = i / PPR, c8 = i % PPR, r = rw + rr;
      piece[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r < r1)
        piece[k] = *reinterpret_cast<const uint4*>(p.q + (((int64_t)b * T + r / G) * p.Hq + h * G + r % G) * D + c8 * 8);
      const uint32_t w4[4] = {piece[k].x, piece[k].y, piece[k].z, piece[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w4[j])), fabsf(bf16_hi(w4[j]))));
    }
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
    const int e = q_norm_exp(m);
    const float qs = pow2i(e);
    kq = p.scale2 * pow2i(-e);
#pragma unroll
    for (int k = 0; k < 16 * PPR / 32; ++k) {
      const int i = lane + 32 * k, rr = i / PPR, c8 = i % PPR;
      const uint32_t w4[4] = {piece[k].x, piece[k].y, piece[k].z, piece[k].w};
      uint32_t hw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) hw[j] = pack_f16(bf16_lo(w4[j]) * qs, bf16_hi(w4[j]) * qs);
      *reinterpret_cast<uint4*>(qsm + rr * q_stride(D) + c8 * 16) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    __syncwarp();
  } else {
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      uint2 x = make_uint2(0u, 0u), y = make_uint2(0u, 0u);
      if (ra < r1)
        x = *reinterpret_cast<const uint2*>(p.q + (((int64_t)b * T + ra / G) * p.Hq + h * G + ra % G) * D + c * 16 +
                                            4 * t4);
      if (rb < r1)
        y = *reinterpret_cast<const uint2*>(p.q + (((int64_t)b * T + rb / G) * p.Hq + h * G + rb % G) * D + c * 16 +
                                            4 * t4);
      qa[c][0] = x.x;
      qa[c][2] = x.y;
      qa[c][1] = y.x;
      qa[c][3] = y.y;
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(qa[c][j])), fabsf(bf16_hi(qa[c][j]))));
    }
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
    const int e = q_norm_exp(m);
    const float qs = pow2i(e);
    kq = p.scale2 * pow2i(-e);
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) qa[c][j] = pack_f16(bf16_lo(qa[c][j]) * qs, bf16_hi(qa[c][j]) * qs);
  }
  // causal limits of the thread's two rows (rows past the unit see every key
  // of the CTA; they are never written)
  const int lim_a = L - T + (ra < r1 ? ra : r1 - 1) / G;
  const int lim_b = L - T + (rb < r1 ? rb : r1 - 1) / G;
  const int wlim_lo = L - T + (rw < r1 ? rw : r1 - 1) / G;  // the warp's first row: blocks past it are masked
  const int wlim_hi = L - T + ((rw + 15) < r1 ? rw + 15 : r1 - 1) / G;  // its last row: blocks past it skipped

  // ldmatrix lane offsets (as the decode kernel): matrices (keys 0-7 | 8-15) x 16-byte chunks
  const int lm_key = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lm_chunk = lane >> 4;
  uint32_t loff[GW][2];
#pragma unroll
  for (int gi = 0; gi < GW; ++gi)
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) loff[gi][q2] = box_off<D>(P, 0, lm_key, gi * 4 + q2 * 2 + lm_chunk);

  float o[NCH][2][4];  // [16-channel chunk][even | odd channels][fragment]
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[c][e][k] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float sv[GW];  // 2^-ev of the P' of each group (0: not set yet)
#pragma unroll
  for (int gi = 0; gi < GW; ++gi) sv[gi] = 0.f;
  const uint32_t bias = 0x80808080u;

  // the running total in tensor memory (once has_total), at the row
  // references tm_a, tm_b it was stored with. fold(false): total = total
  // 2^(tm - m) + o, o restarts from zero; fold(true): o = that sum, kept in
  // registers. Columns of the thread's lane: (chunk c, even|odd e, element k)
  // at 8 c + 4 e + k; elements k < 2 are row g, k >= 2 row g + 8.
  bool has_total = false;
  float tm_a = -INFINITY, tm_b = -INFINITY;
  auto fold = [&](bool final_fold) {
    const float fa = has_total && tm_a != -INFINITY ? ex2(tm_a - m_a) : 0.f;
    const float fb = has_total && tm_b != -INFINITY ? ex2(tm_b - m_b) : 0.f;
#pragma unroll
    for (int c2 = 0; c2 < NCH / 2; ++c2) {
      float v[16];
      if (has_total) tm_ld16(tm_base + c2 * 16, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float& x = o[c2 * 2 + j / 8][(j / 4) & 1][j & 3];
        const float t = has_total ? fmaf(v[j], (j & 2) ? fb : fa, x) : x;
        if (final_fold)
          x = t;
        else
          v[j] = t;
      }
      if (!final_fold) tm_st16(tm_base + c2 * 16, v);
    }
    if (!final_fold) {
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[c][e][k] = 0.f;
      has_total = true;
      tm_a = m_a;
      tm_b = m_b;
    }
  };
  const int fold_pages = P >= kFoldKeys ? 1 : kFoldKeys / P;

  int s = 0;
  uint32_t ph = 0;
  for (int q = 0; q < npages; ++q) {
    if (!*abort_flag && !mbar_wait(smem_u32(&full_bar[s]), ph, p.wait_cycles)) {
      if (lane == 0) flag(p.status, NK_DEVFLAG_TIMEOUT);
      *abort_flag = 1;
    }
    const uint32_t st = stage0 + s * PL.stage_bytes;
    const uint8_t* ks_s = smem + s * PL.stage_bytes + 2 * P * D;  // [P][GW], fp32 or fp16
    const uint8_t* vs_s = ks_s + P * GW * sb;
    for (int kb = 0; kb < BPP; ++kb) {
      const int key0 = kb * 16, pos0 = q * P + key0;
      if (pos0 <= wlim_hi) {
        // ---- QK, one accumulator per group, summed with the keys' scales
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) sc[nt][k] = 0.f;
#pragma unroll
        for (int gi = 0; gi < GW; ++gi) {
          uint32_t kw[4][2];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2)
            ldsm_x4(st + key0 * RB + loff[gi][q2], kw[q2 * 2][0], kw[q2 * 2][1], kw[q2 * 2 + 1][0], kw[q2 * 2 + 1][1]);
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[nt][k] = 0.f;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const uint32_t w = kw[cc][nt] ^ bias;
              uint32_t a0, a1, a2, a3;
              if constexpr (QS) {
                // rows g and g + 8, channels 16 c + 4 t4 .. + 3 of the warp's rows
                const int c = gi * 4 + cc;
                const uint2 x = *reinterpret_cast<const uint2*>(qsm + g * q_stride(D) + (c * 16 + 4 * t4) * 2);
                const uint2 y = *reinterpret_cast<const uint2*>(qsm + (g + 8) * q_stride(D) + (c * 16 + 4 * t4) * 2);
                a0 = x.x;
                a2 = x.y;
                a1 = y.x;
                a3 = y.y;
              } else {
                a0 = qa[gi * 4 + cc][0];
                a1 = qa[gi * 4 + cc][1];
                a2 = qa[gi * 4 + cc][2];
                a3 = qa[gi * 4 + cc][3];
              }
              mma16816(acc[nt], a0, a1, a2, a3, i8x2_to_f16x2(w, 0x4140), i8x2_to_f16x2(w, 0x4342));
            }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int kk = key0 + nt * 8 + 2 * t4;
            const float k0 = ld_scale(ks_s, kk * GW + gi, sb) * kq, k1 = ld_scale(ks_s, (kk + 1) * GW + gi, sb) * kq;
            sc[nt][0] = fmaf(k0, acc[nt][0], sc[nt][0]);
            sc[nt][1] = fmaf(k1, acc[nt][1], sc[nt][1]);
            sc[nt][2] = fmaf(k0, acc[nt][2], sc[nt][2]);
            sc[nt][3] = fmaf(k1, acc[nt][3], sc[nt][3]);
          }
        }
        // ---- causal mask: only blocks past the warp's first row's limit
        if (pos0 + 15 > wlim_lo) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int key = pos0 + nt * 8 + 2 * t4 + (k & 1);
              if (key > ((k & 2) ? lim_b : lim_a)) sc[nt][k] = -INFINITY;
            }
        }
        // ---- online softmax (base 2), lazy reference per row
        float mx_a = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx_b = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        if (__any_sync(0xffffffffu, mx_a > m_a + 8.f || mx_b > m_b + 8.f)) {
          mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
          mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
          mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
          mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
          const float na = fmaxf(m_a, mx_a), nb = fmaxf(m_b, mx_b);
          const float al_a = na > m_a ? ex2(m_a - na) : 1.f, al_b = nb > m_b ? ex2(m_b - nb) : 1.f;
          m_a = na;
          m_b = nb;
          l_a *= al_a;
          l_b *= al_b;
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              o[c][e][0] *= al_a;
              o[c][e][1] *= al_a;
              o[c][e][2] *= al_b;
              o[c][e][3] *= al_b;
            }
        }
        const float mu_a = m_a == -INFINITY ? 0.f : m_a, mu_b = m_b == -INFINITY ? 0.f : m_b;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pr[nt][0] = ex2(sc[nt][0] - mu_a);
          pr[nt][1] = ex2(sc[nt][1] - mu_a);
          pr[nt][2] = ex2(sc[nt][2] - mu_b);
          pr[nt][3] = ex2(sc[nt][3] - mu_b);
          l_a += pr[nt][0] + pr[nt][1];
          l_b += pr[nt][2] + pr[nt][3];
        }
        // ---- PV per group. The thread's keys of the A fragment: 2 t4, 2 t4 + 1
        // (n-tile 0) and 8 + 2 t4, 9 + 2 t4 (n-tile 1); keys at or past L hold
        // stale slots whose scales may be NaN: their Vs is taken as 0.
#pragma unroll
        for (int gi = 0; gi < GW; ++gi) {
          float vs[2][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int kk = key0 + nt * 8 + 2 * t4 + j;
              vs[nt][j] = pos0 + nt * 8 + 2 * t4 + j < L ? ld_scale(vs_s, kk * GW + gi, sb) : 0.f;
            }
          // P' window of the group (as the decode kernels): the exponent moves
          // only when a Vs 2^-ev passes 2^6, or none of the block's is 2^-10 or more
          {
            const float tv = fmaxf(fmaxf(vs[0][0], vs[0][1]), fmaxf(vs[1][0], vs[1][1])) * sv[gi];
            const bool up = __any_sync(0xffffffffu, tv > 64.f);
            const bool in = __any_sync(0xffffffffu, tv >= 0.0009765625f);
            if (up || !in) {
              const float vmx = fmaxf(fmaxf(vs[0][0], vs[0][1]), fmaxf(vs[1][0], vs[1][1]));
              const uint32_t mxb = __reduce_max_sync(0xffffffffu, __float_as_uint(vmx));
              int ev = sv[gi] == 0.f ? kEvUnset : -exp_of(sv[gi]);
              float beta;
              if (mxb != 0u && ev_update(ev, exp_of(__uint_as_float(mxb)), beta)) {
                sv[gi] = pow2i(-ev);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                  for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int k = 0; k < 4; ++k) o[gi * 4 + cc][e][k] *= beta;
              }
            }
          }
          uint32_t ah[4], al[4];
          {
            float pv[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              pv[nt][0] = pr[nt][0] * (vs[nt][0] * sv[gi]);
              pv[nt][1] = pr[nt][1] * (vs[nt][1] * sv[gi]);
              pv[nt][2] = pr[nt][2] * (vs[nt][0] * sv[gi]);
              pv[nt][3] = pr[nt][3] * (vs[nt][1] * sv[gi]);
            }
            // a0 = (row g, keys 2t4..), a1 = (row g+8, keys 2t4..), a2/a3 the keys + 8
            const float f[4][2] = {{pv[0][0], pv[0][1]}, {pv[0][2], pv[0][3]}, {pv[1][0], pv[1][1]}, {pv[1][2], pv[1][3]}};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __half2 hh = __floats2half2_rn(f[j][0], f[j][1]);
              const float2 hf = __half22float2(hh);
              ah[j] = *reinterpret_cast<const uint32_t*>(&hh);
              al[j] = pack_f16(f[j][0] - hf.x, f[j][1] - hf.y);
            }
          }
          uint32_t vw[4][2];  // [16-channel chunk][keys 0-7 | 8-15], transposed
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2)
            ldsm_x4_t(st + (P + key0) * RB + loff[gi][q2], vw[q2 * 2][0], vw[q2 * 2][1], vw[q2 * 2 + 1][0],
                      vw[q2 * 2 + 1][1]);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint32_t w0 = vw[cc][0] ^ bias, w1 = vw[cc][1] ^ bias;
            // even channels 16 c + 2 n, odd channels 16 c + 2 n + 1
            const uint32_t be0 = i8x2_to_f16x2(w0, 0x4240), be1 = i8x2_to_f16x2(w1, 0x4240);
            const uint32_t bo0 = i8x2_to_f16x2(w0, 0x4341), bo1 = i8x2_to_f16x2(w1, 0x4341);
            float(&oe)[4] = o[gi * 4 + cc][0];
            float(&oo)[4] = o[gi * 4 + cc][1];
            mma16816(oe, ah[0], ah[1], ah[2], ah[3], be0, be1);
            mma16816(oo, ah[0], ah[1], ah[2], ah[3], bo0, bo1);
            mma16816(oe, al[0], al[1], al[2], al[3], be0, be1);
            mma16816(oo, al[0], al[1], al[2], al[3], bo0, bo1);
          }
        }
      }
    }
    // ---- release the page's stage; the last warp to release it loads the
    // page S ahead into it
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&empty_bar[s]));
      if (atomicAdd(&cnt[s], 1) == kWarps - 1) {
        cnt[s] = 0;
        const int qn = q + S;
        if (qn < npages && p.issuable(qn) && !*abort_flag) {
          // every warp arrived before its increment: the phase is complete
          if (mbar_wait(smem_u32(&empty_bar[s]), ph, p.wait_cycles)) {
            issue_page<D>(p, &tmap, page_z(qn), st, smem_u32(&full_bar[s]));
            ++icnt[s];
          } else {
            flag(p.status, NK_DEVFLAG_TIMEOUT);
            *abort_flag = 1;
          }
        }
      }
    }
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
    if (q + 1 < npages && (q + 1) % fold_pages == 0) fold(false);
  }
  if (has_total) fold(true);

  // ---- rows: reduce the row sums over the four lanes of a row, normalize,
  // undo the P' exponents, write bf16
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
  for (int gi = 0; gi < GW; ++gi) {
    const float un = sv[gi] == 0.f ? 1.f : pow2i(-exp_of(sv[gi]));  // 2^ev
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int c = gi * 4 + cc;
      // element (e, k): row g (k < 2) or g + 8, channel 16 c + 4 t4 + 2 (k & 1) + e
      const float va[4] = {o[c][0][0] * ia * un, o[c][1][0] * ia * un, o[c][0][1] * ia * un, o[c][1][1] * ia * un};
      const float vb[4] = {o[c][0][2] * ib * un, o[c][1][2] * ib * un, o[c][0][3] * ib * un, o[c][1][3] * ib * un};
      bool fin = true;
#pragma unroll
      for (int j = 0; j < 4; ++j) fin &= isfinite(va[j]) && isfinite(vb[j]);
      if (!fin) flag(p.status, NK_DEVFLAG_RANGE);
      const int ch = c * 16 + 4 * t4;
      if (ra < r1)
        *reinterpret_cast<uint2*>(p.out + (((int64_t)b * T + ra / G) * p.Hq + h * G + ra % G) * D + ch) =
            make_uint2((uint32_t)f32_to_bf16(va[0]) | ((uint32_t)f32_to_bf16(va[1]) << 16),
                       (uint32_t)f32_to_bf16(va[2]) | ((uint32_t)f32_to_bf16(va[3]) << 16));
      if (rb < r1)
        *reinterpret_cast<uint2*>(p.out + (((int64_t)b * T + rb / G) * p.Hq + h * G + rb % G) * D + ch) =
            make_uint2((uint32_t)f32_to_bf16(vb[0]) | ((uint32_t)f32_to_bf16(vb[1]) << 16),
                       (uint32_t)f32_to_bf16(vb[2]) | ((uint32_t)f32_to_bf16(vb[3]) << 16));
    }
  }
  // after a timed-out wait: the last copy issued into each stage lands before
  // the CTA exits; every warp's tensor-memory accesses are complete (each
  // ended with its wait) before the columns are freed
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (tid == 0)
    for (int s2 = 0; s2 < S; ++s2)
      if (icnt[s2] > 0) (void)mbar_wait(smem_u32(&full_bar[s2]), (uint32_t)(icnt[s2] - 1) & 1u, p.wait_cycles);
  __syncwarp();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tslot), "r"(kTmCols) : "memory");
  }
}

template <int D, int FMT>
static cudaError_t launch_df(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  const Plan PL = plan(FMT, D, p.P);
  if (PL.stages < 2 || PL.total > kSmemLimit) return cudaErrorInvalidConfiguration;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(prefill_kernel<D, FMT>), PL.total);
  if (e != cudaSuccess) return e;
  return launch_chained(prefill_kernel<D, FMT>, dim3(p.n_ctas), dim3(kThreads), PL.total, st, map, p);
}

template <int D>
static cudaError_t launch_d(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  return p.fmt == kFmtI8F16 ? launch_df<D, kFmtI8F16>(map, p, st) : launch_df<D, kFmtI8F32>(map, p, st);
}

}  // namespace pf

bool prefill_supported(int fmt, int D, int P) {
  if (!(fmt == kFmtI8F32 || fmt == kFmtI8F16)) return false;
  if (!(D == 64 || D == 128 || D == 256) || P % 16 != 0 || P > 256) return false;
  return pf::plan(fmt, D, P).stages >= 2;
}

int prefill_rows_per_cta() { return pf::kRows; }

cudaError_t launch_prefill(const DecodeParams& p, cudaStream_t stream) {
  CUtensorMap map;
  cudaError_t e = mma::make_pool_map(p, &map);
  if (e != cudaSuccess) return e;
  if (p.D == 256) return pf::launch_d<256>(map, p, stream);
  if (p.D == 128) return pf::launch_d<128>(map, p, stream);
  return pf::launch_d<64>(map, p, stream);
}

}  // namespace nk
