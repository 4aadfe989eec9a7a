// nk_decode_tc.cu -- split-KV paged attention over the INT8 group-64 cache
// with QK^T on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory) and PV on mma.sync, for head_dim 256, 64-key pages and 9 to
// 32 query rows per kv-head (G * T).
//
// Attention re-reads the whole cache every step ("NInfer-3090" README,
// "Choosing a KV format"); decode and MTP-verify rounds attend T = draft+1
// columns per sequence ("Decode after the small-T kernels"). The int8 codes
// enter both products exactly (as fp16); the group scales are applied to fp32
// partial sums (K) and folded into the probabilities (V).
//
// CTA = 16 warps in three roles, one CTA per SM, same stream-K split over
// (sequence, kv-head, page) items as the mma.sync kernel, same TMA page ring
// (one stage = the K|V code tiles and both scale arrays of one page; the last
// of the 16 warps to release a stage loads the page S ahead into it).
//
// Convert warps 0-3 (one per tensor-memory lane quadrant), per 64-key page:
//   * thread (quadrant w, lane l) takes key k = 32 (w & 1) + l and channel
//     half c = w >> 1, widens its 128 codes to fp16 and stores them into
//     tensor-memory row 64 c + k: the page becomes a 128-row A operand whose
//     rows 0-63 hold channels 0-127 of the keys and rows 64-127 channels
//     128-255 (two tensor-memory buffers, so page j + 1 converts while the
//     scores of page j are read);
//   * QK: one thread issues 8 tcgen05.mma (M = 128, N = 2W, K = 16) into two
//     accumulators: A = groups 0|2, B = groups 1|3. The B operand stacks the
//     query rows twice, once with the channels of the first half and once
//     with those of the second (W rows each, zero padded), so lanes 0-63 of
//     columns [0, W) and lanes 64-127 of columns [W, 2W) are the per-group
//     dot products; the other quarter-blocks are unused.
// Score warps 4-7 (same key / channel-half mapping by quadrant):
//   * each thread loads its lane's two accumulator rows, applies its key's
//     two group scales (times sm_scale log2 e) and swaps half of its rows
//     with the thread holding the other channel half of the same key, so
//     quadrants 0-1 finish rows with (n mod 8) < 4 and quadrants 2-3 the rest;
//   * online softmax in base 2 with a lazy reference per row (raised only
//     when a score passes it by more than 8, agreed by the two warps of a
//     row half), P' = p * Vs[key][group] split into fp16 hi + lo, written to
//     a double-buffered shared-memory tile [group][hi|lo][8-row tile][key].
// PV warps 8-15: warp 8 + i owns channels [32 i, 32 i + 32) (group i / 2) for
//   all rows; per page it rescales its accumulators if a reference moved,
//   then O^T[ch][row] += V^T[ch][key] P'^T[key][row] with mma.sync m16n8k16
//   (swap-AB), V^T fragments from ldmatrix.trans on the TMA tile, P'
//   fragments from ldmatrix.trans on the score warps' tile (hi and lo: two
//   MMAs).
// At the end of a segment the row sums are reduced and the PV warps write
// bf16 rows (whole unit) or fp32 partials with their LSE.
// A second instance of the kernel (FOLD) adds the PV accumulators into a
// total in tensor memory every 128 pages; the host takes it when a CTA may
// run more than 512 pages of one kv-head.
// Every mbarrier wait is bounded; a timeout sets NK_DEVFLAG_TIMEOUT.
#include "nk_decode_mma.cuh"

namespace nk {
namespace mma {
cudaError_t make_pool_map(const DecodeParams& p, CUtensorMap* map, int part = 0);
}

namespace tc {

using namespace mma;

constexpr int kD = 256, kP = 64;
constexpr int kConvWarps = 4, kScoreWarps = 4, kPvWarps = 8;
constexpr int kWarps = kConvWarps + kScoreWarps + kPvWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kTmemCols = 512;
// Registers per thread: the kernel launches with 128 (512 threads, one CTA
// per SM: the whole register file). Each role's warpgroup(s) then move to
// their own share with setmaxnreg; the shares add up to the launch total, so
// no increase ever waits for registers that are not there (checked on the
// host against the compiled count before the first launch).
// The folding instance (below) gives the PV warps 8 more registers for the
// total's load/store and takes them from the convert warps.
constexpr int kLaunchRegs = 128, kRegsScore = 144;
__host__ __device__ constexpr int regs_conv(bool fold) { return fold ? 128 : 144; }
__host__ __device__ constexpr int regs_pv(bool fold) { return fold ? 120 : 112; }
static_assert(kConvWarps == 4 && kScoreWarps == 4 && kPvWarps == 8, "one warpgroup per role, two for PV");
static_assert(regs_conv(false) + kRegsScore + 2 * regs_pv(false) == 4 * kLaunchRegs, "shares = the launch's registers");
static_assert(regs_conv(true) + kRegsScore + 2 * regs_pv(true) == 4 * kLaunchRegs, "shares = the launch's registers");
// one page: the K|V code boxes, then both scale arrays (34,816 bytes with
// fp32 scales, 33,792 with fp16 ones: multiples of 1024 either way)
__host__ __device__ constexpr int stage_bytes(int sb) { return 2 * kP * kD + 2 * kP * (kD / kGroup) * sb; }
constexpr int kPidCache = 512;
constexpr int kColA = 0;      // tensor-memory columns of the two K buffers (64 each)
constexpr int kColAcc = 128;  // the two accumulator buffers (4W each)
constexpr int kQAhead = 4;    // pages before a segment's end at which the next unit's Q is prefetched
constexpr int kColTot = 384;  // the folded PV totals (32 columns per warp, two warps per lane quadrant)
// Folding: a PV accumulator restarts from zero every kFoldPages pages (8,192
// keys). The host takes the folding instance when one CTA may run more than
// kNoFoldPages pages of one kv-head through its accumulators.
constexpr int kFoldPages = 128;
constexpr int kNoFoldPages = 512;

__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);  // fp16 A/B, K-major, fp32 D
}

// K-major, 128-byte-swizzled shared-memory operand: rows of 128 bytes, 8-row
// atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3fff) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}

struct Layout {
  int stage_bytes;
  int stages;
  int off_qt, off_pbuf, off_hdr, off_xs, off_red, off_pre, off_pid, off_bar, off_tmem;
  int total;
};

__host__ __device__ inline Layout layout(int W, int NT, int sb) {
  Layout L;
  L.stage_bytes = stage_bytes(sb);
  int off = 0;
  const int qt = 2 * (2 * W) * 128;
  const int pbuf = 2 * NT * 8192;
  const int hdr = 512;
  const int xs = 2 * 2 * 64 * NT * 4 * 4;
  const int red = (2 * 4 * 32 + 2 * 32) * 4 + 4 * 4 + 32 * 4 + 64 + (16 + 4 + 8 + 16 + 4) * 4;
  const int pre = round_up((2 * kMaxBatch + 1 + 16 + 8 + 4 + 9) * 4, 16);  // pre, warp_tot, cnt, flag, lens, icnt, last MMA
  const int pid = kPidCache * 4;
  const int bar = 32 * 8;
  const int fixed = qt + pbuf + hdr + xs + red + pre + pid + bar + 16;
  int s = (kSmemLimit - 1024 - fixed) / L.stage_bytes;
  if (s > 8) s = 8;
  L.stages = s;
  off = s * L.stage_bytes;
  L.off_qt = off; off += qt;
  L.off_pbuf = off; off += pbuf;
  L.off_hdr = off; off += hdr;
  L.off_xs = off; off += xs;
  L.off_red = off; off += red;
  L.off_pre = off; off += pre;
  L.off_pid = off; off += pid;
  L.off_bar = off; off += bar;
  L.off_tmem = off; off += 16;
  L.total = off + 1024;
  return L;
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// W: padded query rows per channel half of the QK operand (16 or 32);
// NT: 8-row tiles of the PV product (ceil(G*T / 8) <= W / 8).
// SB: bytes of a group scale (4: fp32 scales; 2: the pages' fp16 scales).
// FOLD: the PV accumulators are folded into a tensor-memory total every
// kFoldPages pages.
template <int W, int NT, int SB, bool FOLD>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                const DecodeParams p) {
  // the tensor map is a launch parameter: its descriptor fetch can start
  // before the wait for the previous kernel
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
  if (!p.early) chain_wait();  // (early: waits below, before the first page load)
  chain_release();
  constexpr int NR = NT * 4;  // rows a score thread finishes (half of each 8-row tile)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int sb = SB;
  const Layout LY = layout(W, NT, sb);
  const int S = LY.stages;
  const int kStageBytes = LY.stage_bytes;
  int* pre = reinterpret_cast<int*>(smem + LY.off_pre);
  int* warp_tot = pre + (kMaxBatch + 1);
  int* cnt = warp_tot + 16;  // [8]
  volatile int* abort_flag = cnt + 8;
  int* lens = cnt + 12;  // [kMaxBatch] context lengths
  int* icnt = lens + kMaxBatch;  // [8] copies issued into each stage
  int* pid = reinterpret_cast<int*>(smem + LY.off_pid);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + LY.off_bar);
  uint64_t* empty_bar = full_bar + 8;
  uint64_t* qk_bar = empty_bar + 8;       // [2] QK MMAs of a page done
  uint64_t* accfree_bar = qk_bar + 2;     // [2] score warps done reading an accumulator buffer
  uint64_t* pfull_bar = accfree_bar + 2;  // [2]
  uint64_t* pempty_bar = pfull_bar + 2;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY.off_tmem);
  float* red_l = reinterpret_cast<float*>(smem + LY.off_red);  // [4 score warps][32]
  float* red_m = red_l + 4 * 32;                               // [4][32]
  float* lrow = red_m + 4 * 32;                                // [32]
  float* mrow = lrow + 32;                                     // [32]
  int* sflag = reinterpret_cast<int*>(mrow + 32);              // [4]
  int* row_t = sflag + 4;                                      // [32]: query column of row n (T for padding)
  float* pmx = reinterpret_cast<float*>(row_t + 32 + 16);      // [4 score warps][4 groups]: page's largest Vs
  int* evs = reinterpret_cast<int*>(pmx + 16);                 // [4]: P' exponents at a segment's end
  float* qmx = reinterpret_cast<float*>(evs + 4);              // [2 roles][4 warps]: largest |q| of the unit
  float* sva = qmx + 8;                                        // [4 score warps][4 groups]: 2^-ev of P' (0: unset)
  float* bva = sva + 16;                                       // [4 groups]: accumulator factors of a rebase
  float* xs = reinterpret_cast<float*>(smem + LY.off_xs);      // [2 pages][2 sides][64 keys][NR]
  const uint32_t qt0 = smem_u32(smem + LY.off_qt);             // two Q tiles of 2W x 128 bytes
  uint8_t* pbuf = smem + LY.off_pbuf;                          // [2][4 g][2 h][NT][64][16 B]
  float* hdr = reinterpret_cast<float*>(smem + LY.off_hdr);    // [2][alpha 32 | side flags 2 | pad]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int role = warp < kConvWarps ? 0 : (warp < kConvWarps + kScoreWarps ? 1 : 2);  // convert | score | PV
  const int quad = warp & 3;  // tensor-memory lane quadrant this warp may access
  const SplitShape sh = p.shape();
  const int G = p.G, T = p.T, M = G * T;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kWarps);
      cnt[s] = 0;
      icnt[s] = 0;
    }
    icnt[8] = -1;  // last_mma
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&qk_bar[i]), 1);
      mbar_init(smem_u32(&accfree_bar[i]), kScoreWarps);
      mbar_init(smem_u32(&pfull_bar[i]), kScoreWarps);
      mbar_init(smem_u32(&pempty_bar[i]), kPvWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < 32) row_t[tid] = tid < M ? tid / G : T;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  flag_bad_ctx(p);
  block_page_prefix(sh, p.ctx, p.trim, pre, warp_tot, lens);  // ends with __syncthreads
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t Witems = (int64_t)pre[p.B] * p.Hkv;
  const int64_t x_begin = Witems == 0 ? 0 : cta_begin(Witems, p.n_ctas, blockIdx.x);
  const int64_t x_end = Witems == 0 ? 0 : cta_begin(Witems, p.n_ctas, blockIdx.x + 1);
  const int total = (int)(x_end - x_begin);
  const uint32_t stage0 = smem_u32(smem);

  // Q rows of a unit are pulled into L1 ahead of use: a load this SM issues
  // while its page loads are in flight returns only behind their data
  // (several microseconds), so the convert warps touch a unit's Q lines
  // (M rows of 512 bytes, 128-byte lines) a few pages before they need them.
  auto prefetch_q = [&](const Segment& sg) {
    const int i = tid;  // convert-warp thread: line i & 3 of row i >> 2
    if (i < 4 * M) {
      const int n = i >> 2, t = n / G, hg = n % G;
      const uint16_t* a = p.q + (((int64_t)sg.b * p.qT + t) * p.Hq + sg.h * G + hg) * kD + (i & 3) * 64;
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
    }
  };
  // Every global read of the prologue (page coordinates up to the cache
  // size, the first unit's Q lines) goes out before the first page load.
  const int ncache = total < kPidCache ? total : kPidCache;
  for (int q = tid; q < ncache; q += kThreads) pid[q] = page_coord(p, sh, pre, x_begin, q);
  if (role == 0 && total > 0) {
    int64_t x0 = x_begin;
    Segment s0;
    if (next_segment(sh, pre, x0, x_end, s0)) prefetch_q(s0);
  }
  __syncthreads();
  if (p.early) chain_wait();  // the pages may hold the preceding append's rows
  if (tid == 0) {
    const int n0 = total < S ? total : S;
    for (int q = 0; q < n0; ++q) {
      if (!p.issuable(q)) break;
      issue_page<kD>(p, &tmap, pid[q], stage0 + q * kStageBytes, smem_u32(&full_bar[q]));
      icnt[q] = 1;
    }
  }

  // A bounded wait. After one wait of the CTA has run out (abort_flag), no
  // wait blocks any more: every role runs through its remaining pages without
  // data, no page is issued and no MMA started, and the end of the kernel
  // waits for what was issued before it releases the tensor memory.
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
    if (*abort_flag) return;
    if (!mbar_wait(smem_u32(bar), parity, p.wait_cycles)) {
      if (lane == 0) flag(p.status, NK_DEVFLAG_TIMEOUT);
      *abort_flag = 1;
    }
  };
  // A warp is done with CTA page q's stage s (phase ph); the last of all warps
  // loads page q + S into it.
  auto release_stage = [&](int q, int s, uint32_t ph) {
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&empty_bar[s]));
      if (atomicAdd(&cnt[s], 1) == kWarps - 1) {
        cnt[s] = 0;
        const int qn = q + S;
        if (qn < total && p.issuable(qn) && !*abort_flag) {
          if (mbar_wait(smem_u32(&empty_bar[s]), ph, p.wait_cycles)) {
            issue_page<kD>(p, &tmap, qn < kPidCache ? pid[qn] : page_coord(p, sh, pre, x_begin, qn),
                           stage0 + s * kStageBytes, smem_u32(&full_bar[s]));
            ++icnt[s];
          } else {
            flag(p.status, NK_DEVFLAG_TIMEOUT);
            *abort_flag = 1;
          }
        }
      }
    }
  };
  int* last_mma = icnt + 8;  // CTA page number of the last QK MMAs issued (thread 0)

  int64_t x = x_begin;
  Segment seg;
  int q0 = 0;  // CTA page number of the segment's first page
  // stage and phase of the current page, advanced page by page (no division by S)
  int s = 0;
  uint32_t ph = 0;
  auto next_stage = [&]() {
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  };
  if (role == 0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(regs_conv(FOLD)) : "memory");
    // ======================= convert warps: K codes -> tensor memory, QK MMAs
    const int half = quad >> 1, key = 32 * (quad & 1) + lane;
    while (next_segment(sh, pre, x, x_end, seg)) {
      const int npages = seg.page_end - seg.page_begin;
      // the previous segment's MMAs still read the Q tiles: wait for the last one
      if (q0 > 0) wait_bar(&qk_bar[(q0 - 1) & 1], ((q0 - 1) >> 1) & 1);
      // Q tile tb, row r: query row r % W, channels 128 (r / W) + 64 tb + [0, 64).
      // Thread (row n, quarter qq) converts channels [64 qq, 64 qq + 64) of
      // row n, scaled by the unit's power of two (q_norm_exp of the largest
      // |q| of the unit's M rows, which the score warps compute alike), into
      // tile qq & 1, row (qq >> 1) W + n.
      {
        const int n = tid >> 2, qq = tid & 3;
        uint4 raw[8];
        float m = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          raw[c] = make_uint4(0u, 0u, 0u, 0u);
          if (n < M) {
            const int t = n / G, hg = n % G;
            raw[c] = *reinterpret_cast<const uint4*>(p.q + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * kD +
                                                     64 * qq + 8 * c);
          }
          const uint32_t rw[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(rw[j])), fabsf(bf16_hi(rw[j]))));
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) qmx[quad] = m;
        named_bar(1, kConvWarps * 32);
        const float qs = pow2i(q_norm_exp(fmaxf(fmaxf(qmx[0], qmx[1]), fmaxf(qmx[2], qmx[3]))));
        if (n < W) {
          const int r = (qq >> 1) * W + n, tb = qq & 1;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t rw[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
            uint32_t hw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) hw[j] = pack_f16(bf16_lo(rw[j]) * qs, bf16_hi(rw[j]) * qs);
            *reinterpret_cast<uint4*>(smem + LY.off_qt + tb * (2 * W * 128) + r * 128 + ((c ^ (r & 7)) << 4)) =
                make_uint4(hw[0], hw[1], hw[2], hw[3]);
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q writes -> tensor-core reads
      named_bar(1, kConvWarps * 32);
      // the next unit's Q lines, kQAhead pages before this segment ends
      int64_t xn = x;
      Segment sn;
      const bool has_next = next_segment(sh, pre, xn, x_end, sn);
      const int j_pf = npages > kQAhead ? npages - kQAhead : 0;
      for (int j = 0; j < npages; ++j) {
        const int q = q0 + j;
        if (j == j_pf && has_next) prefetch_q(sn);
        // MMAs of page q - 2 (same K buffer) done, and the stores below
        // ordered after their reads of it; fenced before the wait for the
        // page's data, which usually lasts longer than the fence
        wait_bar(&qk_bar[q & 1], ((q >> 1) & 1) ^ 1);
        tc_fence_after();
        wait_bar(&full_bar[s], ph);
        const uint8_t* st = smem + s * kStageBytes;
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + kColA + (q & 1) * 64;
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          uint32_t r[32];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c = hc * 4 + c4;
            // box `half` (channels 128 half ..), K row `key`, 16-byte chunk c, 128-byte swizzle
            const uint4 w4 =
                *reinterpret_cast<const uint4*>(st + half * (2 * kP * 128) + key * 128 + ((c ^ (key & 7)) << 4));
            const uint32_t w[4] = {w4.x ^ 0x80808080u, w4.y ^ 0x80808080u, w4.z ^ 0x80808080u, w4.w ^ 0x80808080u};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              r[c4 * 8 + 2 * i] = i8x2_to_f16x2(w[i], 0x4140);
              r[c4 * 8 + 2 * i + 1] = i8x2_to_f16x2(w[i], 0x4342);
            }
          }
          tmem_st_x32(taddr + hc * 32, r);
        }
        tmem_wait_st();
        tc_fence_before();
        named_bar(1, kConvWarps * 32);
        if (tid == 0) {
          wait_bar(&accfree_bar[q & 1], ((q >> 1) & 1) ^ 1);  // scores of page q - 2 read
        }
        if (tid == 0 && !*abort_flag) {
          tc_fence_after();
          constexpr uint32_t idesc = idesc_f16_f32(128, 2 * W);
          const uint32_t acc = tmem + kColAcc + (q & 1) * (4 * W);
#pragma unroll
          for (int tb = 0; tb < 2; ++tb)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_tmem_a(acc + tb * (2 * W), tmem + kColA + (q & 1) * 64 + tb * 32 + ks * 8,
                         sdesc_sw128(qt0 + tb * (2 * W * 128) + ks * 32), idesc, ks > 0);
          mma_commit(smem_u32(&qk_bar[q & 1]));
          *last_mma = q;
        }
        release_stage(q, s, ph);
        next_stage();
      }
      q0 += npages;
    }
    // all MMAs done before the tensor memory is released
    if (q0 > 0) wait_bar(&qk_bar[(q0 - 1) & 1], ((q0 - 1) >> 1) & 1);
  } else if (role == 1) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsScore) : "memory");
    // ======================= score warps: scores, softmax, P'
    const int half = quad >> 1, key = 32 * (quad & 1) + lane;
    float m_ref[NR], l_part[NR];
    // sva[quad]: 2^-ev of the P' of the four 64-channel groups (0: not set
    // yet in the segment), a copy per warp (identical in the four), read once
    // per page
    while (next_segment(sh, pre, x, x_end, seg)) {
      const int L = lens[seg.b];
      const int npages = seg.page_end - seg.page_begin;
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        m_ref[i] = -INFINITY;
        l_part[i] = 0.f;
      }
      if (lane < 4) sva[quad * 4 + lane] = 0.f;
      float kq;  // sm_scale log2(e) 2^-e: undoes the Q tile's power of two in the scores
      {
        // the unit's power of two, from the same rows as the convert warps'
        // Q tile (so no exchange with them is needed)
        const int ts = tid - kConvWarps * 32, n = ts >> 2, qq = ts & 3;
        float m = 0.f;
        if (n < M) {
          const int t = n / G, hg = n % G;
          const uint4* src =
              reinterpret_cast<const uint4*>(p.q + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * kD + 64 * qq);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 w4 = src[c];
            const uint32_t rw[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(rw[j])), fabsf(bf16_hi(rw[j]))));
          }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) qmx[4 + quad] = m;
        named_bar(2, kScoreWarps * 32);
        kq = p.scale2 * pow2i(-q_norm_exp(fmaxf(fmaxf(qmx[4], qmx[5]), fmaxf(qmx[6], qmx[7]))));
      }
      for (int j = 0; j < npages; ++j) {
        const int q = q0 + j;
        wait_bar(&full_bar[s], ph);  // scale arrays of the page visible
        const uint8_t* st = smem + s * kStageBytes;
        const uint8_t* ks_s = st + 2 * kP * kD;           // [64 keys][4 groups], fp32 or fp16
        const uint8_t* vs_s = ks_s + kP * (kD / kGroup) * sb;
        const int pos = (seg.page_begin + j) * kP + key;
        const bool key_valid = pos < L;
        // P' window of each group, while the page's QK runs: bit g set when a
        // key's Vs 2^-ev passes 2^6 (p Vs 2^-ev could reach 2^15), bit 4 + g
        // when one is at least 2^-10; a group whose ev is not set yet has
        // neither. Slots past ctx_len may hold NaN scales: their Vs is 0.
        float vk[4];
        uint32_t wbits = 0u;
        __syncwarp();  // sva as the previous page left it
        {
          const float4 sv4 = *reinterpret_cast<const float4*>(sva + quad * 4);
          const float sv[4] = {sv4.x, sv4.y, sv4.z, sv4.w};
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            vk[g4] = key_valid ? ld_scale(vs_s, key * 4 + g4, sb) : 0.f;
            const float tv = vk[g4] * sv[g4];
            wbits |= (tv > 64.f ? 1u : 0u) << g4;
            wbits |= (tv >= 0.0009765625f ? 1u : 0u) << (4 + g4);
          }
        }
        wbits = __reduce_or_sync(0xffffffffu, wbits);
        const float ka = ld_scale(ks_s, key * 4 + 2 * half, sb) * kq;
        const float kb = ld_scale(ks_s, key * 4 + 2 * half + 1, sb) * kq;
        wait_bar(&qk_bar[q & 1], (q >> 1) & 1);
        tc_fence_after();
        // ---- this lane's accumulator rows (groups 2 half, 2 half + 1), 16 query rows at a time;
        // half of the rows go to the thread holding the other channel half of the key
        float* xq = xs + (q & 1) * (2 * 64 * NR);  // by page parity: a side rewrites it only two pages later
        float* mine = xq + (half * 64 + key) * NR;
        float sc[NR];
        {
          // every load of the page's columns in flight before the one wait
          constexpr int NC = (NT * 8 + 15) / 16;
          const uint32_t base = tmem + ((uint32_t)(quad * 32) << 16) + kColAcc + (q & 1) * (4 * W) + half * W;
          float ta[NC][16], tb[NC][16];
#pragma unroll
          for (int ci = 0; ci < NC; ++ci) {
            tmem_ld_x16(base + 16 * ci, ta[ci]);
            tmem_ld_x16(base + 2 * W + 16 * ci, tb[ci]);
          }
          tmem_wait_ld();
#pragma unroll
          for (int ci = 0; ci < NC; ++ci) {
#pragma unroll
            for (int nt2 = 0; nt2 < 2; ++nt2) {
              const int nt = 2 * ci + nt2;
              if (nt >= NT) break;
              float keep[4], send[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float lo = fmaf(kb, tb[ci][nt2 * 8 + i], ka * ta[ci][nt2 * 8 + i]);
                const float hi = fmaf(kb, tb[ci][nt2 * 8 + 4 + i], ka * ta[ci][nt2 * 8 + 4 + i]);
                keep[i] = half ? hi : lo;
                send[i] = half ? lo : hi;
                sc[nt * 4 + i] = keep[i];
              }
              *reinterpret_cast<float4*>(mine + nt * 4) = make_float4(send[0], send[1], send[2], send[3]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&accfree_bar[q & 1]));
        named_bar(2, kScoreWarps * 32);
        {
          const float* theirs = xq + ((1 - half) * 64 + key) * NR;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float4 rcv = *reinterpret_cast<const float4*>(theirs + nt * 4);
            sc[nt * 4 + 0] += rcv.x;
            sc[nt * 4 + 1] += rcv.y;
            sc[nt * 4 + 2] += rcv.z;
            sc[nt * 4 + 3] += rcv.w;
          }
        }
        // ---- causal / context mask: only pages that reach past L - T (padding rows
        // hold zero queries and are never written out, so they need no mask)
        if ((seg.page_begin + j + 1) * kP > L - T) {
          const int lim = pos - (L - T);  // visible to column t when lim <= t
#pragma unroll
          for (int i = 0; i < NR; ++i)
            if (lim > row_t[8 * (i >> 2) + 4 * half + (i & 3)]) sc[i] = -INFINITY;
        }
        // ---- lazy reference: raised when a score passes it by more than 8
        bool over = false;
#pragma unroll
        for (int i = 0; i < NR; ++i) over |= sc[i] > m_ref[i] + 8.f;
        const unsigned vote = __ballot_sync(0xffffffffu, over);
        if (lane == 0) sflag[quad] = (int)((vote != 0 ? 1u : 0u) | (wbits << 1));
        named_bar(3 + half, 64);
        const uint32_t fl = (uint32_t)(sflag[2 * half] | sflag[2 * half + 1]);
        const bool raise = (fl & 1u) != 0u;
        // groups whose ev moves: a Vs 2^-ev above the window, or none in it
        const uint32_t moving = ((fl >> 1) & 0xfu) | (~(fl >> 5) & 0xfu);
        if (moving) {  // rare: the page's largest Vs of each group moves its exponent (ev_update)
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(vk[g4]));
            if (lane == 0) pmx[quad * 4 + g4] = __uint_as_float(mx);
          }
          named_bar(3 + half, 64);
          __syncwarp();
          if (lane < 4) {  // lane g moves group g; warp 0 leaves the accumulator factors for the PV warps
            float sv = sva[quad * 4 + lane], beta = 1.f;
            if ((moving >> lane) & 1u) {
              const float mx = fmaxf(pmx[(2 * half) * 4 + lane], pmx[(2 * half + 1) * 4 + lane]);
              int ev = sv == 0.f ? kEvUnset : -exp_of(sv);
              if (mx > 0.f && ev_update(ev, exp_of(mx), beta)) sv = pow2i(-ev);
            }
            sva[quad * 4 + lane] = sv;
            if (quad == 0) bva[lane] = beta;
          }
          __syncwarp();
        }
        float al[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) al[i] = 1.f;
        if (raise) {
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            float mb = sc[i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
            if (lane == 0) red_m[quad * 32 + i] = mb;
          }
          named_bar(3 + half, 64);
#pragma unroll
          for (int i = 0; i < NR; ++i) {
            const float mb = fmaxf(red_m[(2 * half) * 32 + i], red_m[(2 * half + 1) * 32 + i]);
            const float mnew = fmaxf(m_ref[i], mb);
            if (mnew > m_ref[i]) {
              al[i] = ex2(m_ref[i] - mnew);  // 0 while the row was empty
              l_part[i] *= al[i];
              m_ref[i] = mnew;
            }
          }
        }
        // ---- probabilities, row sums, P' = p Vs split into fp16 hi + lo
        float pr[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          const float mu = m_ref[i] == -INFINITY ? 0.f : m_ref[i];
          pr[i] = ex2(sc[i] - mu);
          l_part[i] += pr[i];
        }
        wait_bar(&pempty_bar[q & 1], ((q >> 1) & 1) ^ 1);
        float* alpha = hdr + (q & 1) * 48;  // [32 alpha | 2 side flags | 2 pad | 4 beta | rebase flag]
        if ((quad & 1) == 0 && lane == 0) {
          // the PV warps rescale their accumulators by alpha (rows) and beta
          // (groups) before adding this page
#pragma unroll
          for (int i = 0; i < NR; ++i) alpha[8 * (i >> 2) + 4 * half + (i & 3)] = al[i];
          reinterpret_cast<int*>(alpha + 32)[half] = raise ? 1 : 0;
          if (half == 0) {
            if (moving) {
#pragma unroll
              for (int g4 = 0; g4 < 4; ++g4) alpha[36 + g4] = bva[g4];
            }
            reinterpret_cast<int*>(alpha + 40)[0] = moving ? 1 : 0;
          }
        }
        uint8_t* pb = pbuf + (q & 1) * (NT * 8192);
        const float4 sv4 = *reinterpret_cast<const float4*>(sva + quad * 4);
        const float svp[4] = {sv4.x, sv4.y, sv4.z, sv4.w};
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
          const float vs = vk[gq] * svp[gq];  // P' = p Vs 2^-ev
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            // hi = the value cut to 11 significant bits (exact in fp16 for
            // normal magnitudes), lo = the exact remainder rounded to fp16
            float v[4], hv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[i] = pr[nt * 4 + i] * vs;
              hv[i] = __uint_as_float(__float_as_uint(v[i]) & 0xffffe000u);
            }
            const uint32_t h01 = pack_f16(hv[0], hv[1]), h23 = pack_f16(hv[2], hv[3]);
            const uint32_t l01 = pack_f16(v[0] - hv[0], v[1] - hv[1]), l23 = pack_f16(v[2] - hv[2], v[3] - hv[3]);
            uint8_t* dst = pb + (((gq * 2 + 0) * NT + nt) * 64 + key) * 16 + half * 8;
            *reinterpret_cast<uint2*>(dst) = make_uint2(h01, h23);
            *reinterpret_cast<uint2*>(dst + NT * 64 * 16) = make_uint2(l01, l23);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&pfull_bar[q & 1]));
        release_stage(q, s, ph);
        next_stage();
      }
      q0 += npages;
      // ---- row sums of the segment: reduce l over the 64 keys of each side
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        float v = l_part[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) red_l[quad * 32 + i] = v;
      }
      named_bar(5, (kScoreWarps + kPvWarps) * 32);
      if ((quad & 1) == 0 && lane == 0) {
        // m_ref is identical across the two warps of a side
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          const int n = 8 * (i >> 2) + 4 * half + (i & 3);
          lrow[n] = red_l[quad * 32 + i] + red_l[(quad + 1) * 32 + i];
          mrow[n] = m_ref[i];
        }
        if (half == 0) {
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) evs[g4] = sva[g4] == 0.f ? kEvUnset : -exp_of(sva[g4]);
        }
      }
      named_bar(5, (kScoreWarps + kPvWarps) * 32);
      named_bar(5, (kScoreWarps + kPvWarps) * 32);  // the PV warps have read lrow / mrow
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(regs_pv(FOLD)) : "memory");
    // ======================= PV warps
    const int pw = warp - kConvWarps - kScoreWarps;
    const int g_lane = lane >> 2, t4 = lane & 3;
    const int gq = pw >> 1;  // channel group of this warp
    const int lm_key = ((lane >> 3) & 1) * 8 + (lane & 7);
    const uint32_t loff = box_off<kD>(kP, 0, lm_key, 2 * pw + (lane >> 4));
    float o[2][NT][4];
    // The fp32 sums of mma.sync are not rounded to nearest, and the error
    // they leave grows with the products one accumulator takes in. In the
    // folding instance each thread adds its accumulator every kFoldPages
    // pages into a total kept in its own tensor-memory lane and columns (one
    // rounded add per value and fold) and restarts it from zero; when the
    // row references or a group's P' exponent move, the total is rescaled in
    // place like the accumulator.
    const uint32_t tot = tmem + ((uint32_t)(quad * 32) << 16) + kColTot + (uint32_t)(pw >> 2) * 32;
    bool has_total = false;
    auto fold = [&](bool final_fold) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {  // one 8-column row tile at a time (few live registers)
        float v[8];
        tmem_ld_x8(tot + 8 * nt, v);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float& a = o[cc][nt][k];
            if (final_fold) {
              a += v[cc * 4 + k];
            } else {
              v[cc * 4 + k] += a;
              a = 0.f;
            }
          }
        if (!final_fold) tmem_st_x8(tot + 8 * nt, v);
      }
      if (!final_fold) tmem_wait_st();
    };
    // total *= beta (this warp's group) times alpha of each row (when `rows`)
    auto rescale_total = [&](const float* alpha, float beta, bool rows) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float v[8];
        tmem_ld_x8(tot + 8 * nt, v);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int k = 0; k < 4; ++k) v[cc * 4 + k] *= rows ? beta * alpha[8 * nt + 2 * t4 + (k & 1)] : beta;
        tmem_st_x8(tot + 8 * nt, v);
      }
      tmem_wait_st();
    };
    while (next_segment(sh, pre, x, x_end, seg)) {
      const int npages = seg.page_end - seg.page_begin;
      has_total = false;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[cc][nt][k] = 0.f;
      for (int j = 0; j < npages; ++j) {
        const int q = q0 + j;
        wait_bar(&full_bar[s], ph);
        wait_bar(&pfull_bar[q & 1], (q >> 1) & 1);
        const float* alpha = hdr + (q & 1) * 48;
        const int* sf = reinterpret_cast<const int*>(alpha + 32);
        if (reinterpret_cast<const int*>(alpha + 40)[0]) {  // P' exponent of a group moved
          const float bt = alpha[36 + gq];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int k = 0; k < 4; ++k) o[cc][nt][k] *= bt;
        }
        if (sf[0] | sf[1]) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float al = alpha[8 * nt + 2 * t4 + e];
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                o[cc][nt][e] *= al;
                o[cc][nt][e + 2] *= al;
              }
            }
        }
        if (FOLD && has_total) {
          const bool mv = reinterpret_cast<const int*>(alpha + 40)[0] != 0, rw = (sf[0] | sf[1]) != 0;
          if (mv || rw) rescale_total(alpha, mv ? alpha[36 + gq] : 1.f, rw);
        }
        const uint32_t st = stage0 + s * kStageBytes;
        const uint32_t pb = smem_u32(pbuf + (q & 1) * (NT * 8192));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t vw[2][2];
          ldsm_x4_t(st + (kP + kk * 16) * 128 + loff, vw[0][0], vw[0][1], vw[1][0], vw[1][1]);
          uint32_t av[2][4];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t w0 = vw[cc][0] ^ 0x80808080u, w1 = vw[cc][1] ^ 0x80808080u;
            av[cc][0] = i8x2_to_f16x2(w0, 0x4240);
            av[cc][1] = i8x2_to_f16x2(w0, 0x4341);
            av[cc][2] = i8x2_to_f16x2(w1, 0x4240);
            av[cc][3] = i8x2_to_f16x2(w1, 0x4341);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            // matrices: (hi, keys 0-7), (hi, keys 8-15), (lo, keys 0-7), (lo, keys 8-15)
            const int mi = lane >> 3;
            const uint32_t addr =
                pb + (((gq * 2 + (mi >> 1)) * NT + nt) * 64 + kk * 16 + (mi & 1) * 8 + (lane & 7)) * 16;
            uint32_t bh0, bh1, bl0, bl1;
            ldsm_x4_t(addr, bh0, bh1, bl0, bl1);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) mma16816(o[cc][nt], av[cc][0], av[cc][1], av[cc][2], av[cc][3], bh0, bh1);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) mma16816(o[cc][nt], av[cc][0], av[cc][1], av[cc][2], av[cc][3], bl0, bl1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&pempty_bar[q & 1]));
        release_stage(q, s, ph);
        next_stage();
        if (FOLD && (j + 1) % kFoldPages == 0 && j + 1 < npages) {
          if (has_total) {
            fold(false);
          } else {  // the first fold stores the accumulator as the total
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float v[8];
#pragma unroll
              for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  v[cc * 4 + k] = o[cc][nt][k];
                  o[cc][nt][k] = 0.f;
                }
              tmem_st_x8(tot + 8 * nt, v);
            }
            tmem_wait_st();
            has_total = true;
          }
        }
      }
      q0 += npages;
      if (FOLD && has_total) fold(true);
      // ---- segment result: wait for the row statistics, then write the rows
      named_bar(5, (kScoreWarps + kPvWarps) * 32);
      named_bar(5, (kScoreWarps + kPvWarps) * 32);
      const int64_t slot = (int64_t)blockIdx.x + seg.u;
      const float unscale = evs[gq] == kEvUnset ? 1.f : pow2i(evs[gq]);  // o holds O 2^-ev
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = 8 * nt + 2 * t4 + e;
          if (n >= M) continue;
          const float lsum = lrow[n];
          const float inv = lsum > 0.f ? unscale / lsum : 0.f;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = 32 * pw + 16 * cc + 2 * g_lane;
            const float v0 = o[cc][nt][e] * inv, v1 = o[cc][nt][e + 2] * inv;
            if (!isfinite(v0) || !isfinite(v1)) flag(p.status, NK_DEVFLAG_RANGE);
            if (seg.whole) {
              const int t = n / G, hg = n % G;
              *reinterpret_cast<uint32_t*>(p.out + (((int64_t)seg.b * p.qT + t) * p.Hq + seg.h * G + hg) * kD + ch) =
                  (uint32_t)f32_to_bf16(v0) | ((uint32_t)f32_to_bf16(v1) << 16);
            } else {
              *reinterpret_cast<float2*>(p.part_o + (slot * M + n) * kD + ch) = make_float2(v0, v1);
            }
          }
          if (!seg.whole && pw == 0 && g_lane == 0) {
            const float mx = mrow[n];
            p.part_lse[slot * M + n] = lsum > 0.f ? (mx + log2f(lsum)) * kLn2 : -INFINITY;
          }
        }
      named_bar(5, (kScoreWarps + kPvWarps) * 32);
    }
  }

  // release tensor memory
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    // After a timed-out wait some copies or MMAs may still be in flight:
    // the last copy issued into each stage and the last QK MMAs complete
    // (bounded waits, whatever abort_flag says) before the tensor memory is
    // released and the CTA exits. Without a timeout all of them are done.
    for (int s2 = 0; s2 < S; ++s2)
      if (icnt[s2] > 0) (void)mbar_wait(smem_u32(&full_bar[s2]), (uint32_t)(icnt[s2] - 1) & 1u, p.wait_cycles);
    const int lm = *last_mma;
    if (lm >= 0) (void)mbar_wait(smem_u32(&qk_bar[lm & 1]), (uint32_t)(lm >> 1) & 1u, p.wait_cycles);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int W, int NT, int SB, bool FOLD>
static cudaError_t launch_tsf(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  const Layout LY = layout(W, NT, SB);
  if (LY.stages < 2 || LY.total > kSmemLimit) return cudaErrorInvalidConfiguration;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(decode_tc_kernel<W, NT, SB, FOLD>), LY.total);
  if (e != cudaSuccess) return e;
  // the register shares assume the launch count they were split from
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, decode_tc_kernel<W, NT, SB, FOLD>);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
  }
  if (regs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  return launch_chained(decode_tc_kernel<W, NT, SB, FOLD>, dim3(p.n_ctas), dim3(kThreads), LY.total, st, map, p);
}

// The most pages of one kv-head a CTA may run: a CTA takes at most
// ceil(items / CTAs) consecutive (page, kv-head) items, and a kv-head of a
// sequence holds at most ceil(max_ctx / P) pages.
static int64_t max_run_pages(const DecodeParams& p) {
  const int64_t unit = ((int64_t)p.max_ctx + kP - 1) / kP;
  const int64_t items = unit * p.B * p.Hkv;
  const int64_t per_cta = (items + p.n_ctas - 1) / p.n_ctas;
  return per_cta < unit ? per_cta : unit;
}

template <int W, int NT, int SB>
static cudaError_t launch_ts(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  return max_run_pages(p) > kNoFoldPages ? launch_tsf<W, NT, SB, true>(map, p, st)
                                         : launch_tsf<W, NT, SB, false>(map, p, st);
}

template <int W, int NT>
static cudaError_t launch_t(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  return scale_bytes(p.fmt) == 2 ? launch_ts<W, NT, 2>(map, p, st) : launch_ts<W, NT, 4>(map, p, st);
}

}  // namespace tc

// At G * T <= 8 (one 8-row tile, e.g. plain decode at G = 6) the QK product is
// small and the mma.sync kernel's shorter per-page chain is faster (C1 32K:
// 34.7 us against 37.3 us for split + combine), so this kernel takes 9 to 32 rows.
bool decode_tc_supported(int fmt, int D, int T, int G, int P) {
  const int M = G * T;
  return (fmt == kFmtI8F32 || fmt == kFmtI8F16) && D == tc::kD && P == tc::kP && M > 8 && M <= 32;
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  CUtensorMap map;
  cudaError_t e = mma::make_pool_map(p, &map);
  if (e != cudaSuccess) return e;
  const int M = p.G * p.T, NT = (M + 7) / 8;
  switch (NT) {
    case 2: return tc::launch_t<16, 2>(map, p, stream);
    case 3: return tc::launch_t<32, 3>(map, p, stream);
    case 4: return tc::launch_t<32, 4>(map, p, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace nk
