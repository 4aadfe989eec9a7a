// nk_common.cuh -- shared device helpers of the CUDA library (not of the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "nk.h"

namespace nk {

constexpr int kGroup = NK_GROUP;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offsets inside one (page, kv-head) chunk:
//   Kc[P][D] int8 | Ks[P][D/64] fp32 | Vc[P][D] int8 | Vs[P][D/64] fp32
struct ChunkLayout {
  int64_t chunk;  // bytes per (page, head)
  int64_t ks;     // offset of Ks
  int64_t vc;     // offset of Vc
  int64_t vs;     // offset of Vs
  __host__ __device__ static ChunkLayout make(int P, int D) {
    ChunkLayout c;
    const int64_t g = D / kGroup;
    c.ks = (int64_t)P * D;
    c.vc = c.ks + (int64_t)P * g * 4;
    c.vs = c.vc + (int64_t)P * D;
    c.chunk = c.vs + (int64_t)P * g * 4;
    return c;
  }
};

// KV formats a pool can hold (the same nk_kv_pool struct describes each; the
// calls of a format take only pools sized for it):
//   kFmtI8F32  INT8 group-64 codes with fp32 scales (nk_kv_*);
//   kFmtI8F16  the same codes with fp16 scales, the layout whose size the
//              "NInfer-3090" README's "Choosing a KV format" table gives
//              (nk_i8f16_*);
//   kFmtBf16   the unquantized bf16 rows of the same table (nk_bf16kv_*).
enum KvFmt : int { kFmtI8F32 = 0, kFmtI8F16 = 1, kFmtBf16 = 2, kFmtRk8v4 = 3 };

// Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D] int8 | Vs[P][D/64] fp16
__host__ __device__ inline ChunkLayout i8f16_layout(int P, int D) {
  ChunkLayout c;
  const int64_t g = D / kGroup;
  c.ks = (int64_t)P * D;
  c.vc = c.ks + (int64_t)P * g * 2;
  c.vs = c.vc + (int64_t)P * D;
  c.chunk = c.vs + (int64_t)P * g * 2;
  return c;
}

// K[P][D] bf16 | V[P][D] bf16 (no scales: ks = vs = 0)
__host__ __device__ inline ChunkLayout bf16kv_layout(int P, int D) {
  ChunkLayout c;
  c.ks = 0;
  c.vc = (int64_t)P * D * 2;
  c.vs = 0;
  c.chunk = 2 * c.vc;
  return c;
}

constexpr int kRkVGroup = 32;  // rk8v4 value channels per scale

// rk8v4: Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D/2] (channel 2j in the low
// nibble of byte j, 2j + 1 in the high one) | Vs[P][D/32] fp16
__host__ __device__ inline ChunkLayout rk8v4_layout(int P, int D) {
  ChunkLayout c;
  c.ks = (int64_t)P * D;
  c.vc = c.ks + (int64_t)P * (D / kGroup) * 2;
  c.vs = c.vc + (int64_t)P * (D / 2);
  c.chunk = c.vs + (int64_t)P * (D / kRkVGroup) * 2;
  return c;
}

__host__ __device__ inline ChunkLayout layout_of(int fmt, int P, int D) {
  switch (fmt) {
    case kFmtI8F16: return i8f16_layout(P, D);
    case kFmtBf16: return bf16kv_layout(P, D);
    case kFmtRk8v4: return rk8v4_layout(P, D);
    default: return ChunkLayout::make(P, D);
  }
}

// Programmatic dependent launch. Every kernel of the library is launched
// with programmatic stream serialization (launch_chained), so it may become
// resident while the previous kernel on the stream is still running. Each one
// therefore calls chain_wait() before its first global-memory access (read or
// write) -- the decode combine kernel reads the context lengths before it,
// for the reason given there: griddepcontrol.wait returns once every prerequisite grid has
// completed and its memory operations are visible. Because every kernel waits
// in every CTA, a kernel cannot complete before its predecessor, so the order
// of the stream is kept transitively. chain_release() lets the next kernel's
// CTAs start launching (they only wait, holding no data, until this grid ends).
__device__ __forceinline__ void chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void chain_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Raises a kernel's dynamic shared-memory limit on the current device once
// (the setting persists), instead of on every launch: the host side of a
// decode step is on the critical path of a call that waits for its result.
inline cudaError_t set_smem_limit(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int device, bytes;
  };
  static std::mutex mu;
  static Entry seen[256];
  static int count = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < count; ++i)
      if (seen[i].kernel == kernel && seen[i].device == dev && seen[i].bytes >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (count < 256) seen[count++] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                  Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void flag(int32_t* status, uint32_t bits) {
  if (status) atomicOr(reinterpret_cast<unsigned int*>(status), bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------------------
// Work split shared by the decode kernels and their combine.
// Unit u = (b, h) = (u / Hkv, u % Hkv) owns ceil(ctx_len[b] / P) pages (0 if
// ctx_len[b] is invalid). Units are laid end to end into W page items; CTA c
// of n takes items [floor(c W / n), floor((c+1) W / n)). Each overlap of a CTA
// range with a unit is one segment, stored as partial slot c + u.
// ---------------------------------------------------------------------------
struct SplitShape {
  int B, Hkv, P, T, max_ctx, max_pages;
};

// Pages of a sequence of context length L (0 for an invalid length).
__device__ __forceinline__ int pages_of_len(const SplitShape& s, int L) {
  if (L < s.T || L > s.max_ctx || (int64_t)L > (int64_t)s.max_pages * s.P) return 0;
  return (L + s.P - 1) / s.P;
}

__device__ __forceinline__ int64_t cta_begin(int64_t W, int n, int c) { return (int64_t)c * W / n; }

// Largest CTA index whose range starts at or before item x (x < W).
__device__ __forceinline__ int cta_of_item(int64_t W, int n, int64_t x) {
  return (int)(((x + 1) * (int64_t)n - 1) / W);
}

}  // namespace nk

namespace nk {

constexpr int kMaxBatch = 1024;  // sequences per call (prefix sums live in shared memory)

// Block-wide exclusive prefix of per-sequence page counts:
// pre[b] = sum_{b' < b} pages(b'), pre[B] = total. Needs blockDim.x >= 256 and
// B <= kMaxBatch; every thread of the block must call it. With `lens`, the
// context lengths are also kept in shared memory (lens[b] = ctx_lens[b]), so
// the kernel reads no length from global memory after its page loads start.
// kL2Only reads the lengths at L2 (ld.global.cg), bypassing this SM's L1.
template <bool kL2Only = false>
__device__ __forceinline__ void block_page_prefix(const SplitShape& s, const int32_t* ctx_lens, int trim, int* pre,
                                                  int* warp_tot, int* lens = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int v[4];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = tid * 4 + i;
    int L = 0;
    if (b < s.B) L = (kL2Only ? __ldcg(ctx_lens + b) : ctx_lens[b]) - trim;
    v[i] = (b < s.B) ? pages_of_len(s, L) : 0;
    if (lens && b < s.B) lens[b] = L;
    sum += v[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < wid; ++w) wbase += warp_tot[w];
  int run = wbase + incl - sum;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = tid * 4 + i;
    if (b < s.B) pre[b] = run;
    run += v[i];
  }
  if (tid == blockDim.x - 1) pre[s.B] = run;
  __syncthreads();
}

// Segment of unit items handled by one CTA.
struct Segment {
  int b, h, u;           // sequence, kv-head, unit index b*Hkv + h
  int page_begin;        // first logical page of the segment within the sequence
  int page_end;          // one past the last
  bool whole;            // the segment covers the whole unit (single partial)
};

// Iterate the segments of CTA c: call first with x = cta_begin; returns false
// when the range is exhausted. `x` advances past the returned segment.
__device__ __forceinline__ bool next_segment(const SplitShape& s, const int* pre, int64_t& x, int64_t x_end,
                                             Segment& seg) {
  if (x >= x_end) return false;
  // sequence b with pre[b]*Hkv <= x < pre[b+1]*Hkv (skip empty sequences)
  int lo = 0, hi = s.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)pre[mid] * s.Hkv <= x) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int pages = pre[b + 1] - pre[b];
  const int64_t off = x - (int64_t)pre[b] * s.Hkv;
  const int h = (int)(off / pages);
  const int p0 = (int)(off % pages);
  const int64_t unit_end = (int64_t)pre[b] * s.Hkv + (int64_t)(h + 1) * pages;
  const int64_t e = unit_end < x_end ? unit_end : x_end;
  seg.b = b;
  seg.h = h;
  seg.u = b * s.Hkv + h;
  seg.page_begin = p0;
  seg.page_end = p0 + (int)(e - x);
  seg.whole = (p0 == 0) && (seg.page_end == pages);
  x = e;
  return true;
}

}  // namespace nk
