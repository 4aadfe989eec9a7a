// nk_api.cu -- the C ABI (declared in include/nk.h): argument checks, the
// work split of the decode path, and kernel launches. No allocation, no
// synchronization; every launch goes on the caller's stream.
#include <math.h>

#include <atomic>

#include "nk_decode.cuh"
#include "nk_ptx.cuh"
#include "nk_rk8v4.cuh"

namespace nk {
cudaError_t launch_kv_append(int sms, const nk_kv_pool& pool, int fmt, const int32_t* bt, int max_pages,
                             const int32_t* start_pos, const int32_t* cu_new, int B, int total_new, const void* k,
                             const void* v, int32_t* status, cudaStream_t stream);
}

using namespace nk;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// nk_test_inject_copy_stall: withheld CTA page number (-1: none) and wait limit (0: the default)
std::atomic<int> g_withhold{-1};
std::atomic<unsigned long long> g_wait_cycles{0};

bool pool_ok(const nk_kv_pool* pool, int* err) {
  if (!pool || !pool->base_dev) { *err = NK_ERR_NULL; return false; }
  const int P = pool->page_size, D = pool->head_dim;
  if (pool->num_pages < 1 || pool->num_kv_heads < 1 || P < 16 || P > 256 || P % 16 != 0 ||
      !(D == 64 || D == 128 || D == 256) || !aligned(pool->base_dev, 16)) {
    *err = NK_ERR_SHAPE;
    return false;
  }
  return true;
}

int sm_count() {
  static std::atomic<int> cached[64];  // per device; 0 = not looked up yet
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return 0; }
  if (dev >= 0 && dev < 64 && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// The longest run of one kv-head's keys a CTA of the mma.sync decode kernels
// may take: 4,096 pages of 64 keys measured 4.4e-4 to 7.0e-4 relative L2
// against the oracle (16,384 pages: 1.18e-3, past the 1e-3 tolerance).
constexpr int64_t kMaxMmaRunKeys = 262144;

int64_t max_items(int32_t B, int32_t Hkv, int32_t max_ctx, int32_t P) {
  return (int64_t)B * Hkv * ((max_ctx + P - 1) / P);
}

int32_t default_ctas(int32_t B, int32_t Hkv, int32_t max_ctx, int32_t P, int per_sm) {
  const int sms = sm_count();
  // at most two CTAs per SM: the default workspace size assumes that bound
  const int k = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
  int64_t n = (int64_t)(sms > 0 ? sms : 148) * k;
  // one sequence: a multiple of Hkv CTAs, so that no CTA's range spans two
  // kv-heads (a second segment costs a merge, a partial write and a Q load)
  if (B == 1 && Hkv > 1 && n >= Hkv) n = n / Hkv * Hkv;
  const int64_t w = max_items(B, Hkv, max_ctx, P);
  if (w < n) n = w;
  if (n < 1) n = 1;
  return (int32_t)n;
}

// Query columns per launch. A verify whose G*T rows exceed what one kernel
// holds runs as column chunks over the same pages (each chunk masks its own
// columns; the pages are read once per chunk): on the tcgen05 shapes (head
// dim 256, 64-key pages) chunks of at most 24 rows, where that kernel is
// fastest; on the mma.sync shapes at most 48 rows, fewer where a larger
// page leaves no room for them; on CUDA cores 8 columns.
int chunk_cols(bool simt, int fmt, int D, int T, int G, int P) {
  if (fmt == kFmtRk8v4) {
    // rk8v4: the tensor-core kernel where it holds the rows (up to 32 per
    // kv-head), else the CUDA-core kernel's 8 columns
    if (decode_mma_supported(fmt, D, T, G, P)) return T;
    int c = 32 / G;
    if (c < 1) c = 1;
    if (c > T) c = T;
    while (c > 1 && !decode_mma_supported(fmt, D, c, G, P)) --c;
    if (decode_mma_supported(fmt, D, c, G, P)) return c;
    return T < 8 ? T : 8;
  }
  if (simt) return T < 8 ? T : 8;
  if (decode_tc_supported(fmt, D, T, G, P)) return T;
  const bool tc_shape = D == 256 && P == 64 && fmt != kFmtBf16;  // the tcgen05 kernel's head dim, page, formats
  if (!tc_shape && decode_mma_supported(fmt, D, T, G, P)) return T;
  int c = (tc_shape ? 24 : 48) / G;
  if (c < 1) c = 1;
  if (c > T) c = T;
  while (c > 1 && !decode_tc_supported(fmt, D, c, G, P) && !decode_mma_supported(fmt, D, c, G, P)) --c;
  return c;
}

// Which split kernel a decode call runs: the tensor-core kernels or the fp32
// CUDA-core kernel on an INT8 group-64 pool (fp32 scales), the tensor-core
// kernels on a pool of the pages' INT8 layout (fp16 scales) or of bf16 rows,
// or on an rk8v4 pool the tensor-core kernel (up to 32 rows per kv-head) or
// the rk8v4 CUDA-core kernel.
enum class Path { kTensor, kSimt, kRk8v4, kTensorF16, kBf16 };

int path_fmt(Path path) {
  switch (path) {
    case Path::kTensorF16: return kFmtI8F16;
    case Path::kBf16: return kFmtBf16;
    case Path::kRk8v4: return kFmtRk8v4;
    default: return kFmtI8F32;
  }
}

// the paths on the tensor-core kernels (tcgen05 / mma.sync)
bool tensor_path(Path path) { return path == Path::kTensor || path == Path::kTensorF16 || path == Path::kBf16; }

// Checks the decode arguments and fills `p`; *empty = nothing to launch.
int prepare_decode(const nk_kv_pool* pool, const void* q, const int32_t* bt, int32_t max_pages, const int32_t* ctx,
                   int32_t B, int32_t T, int32_t Hq, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                   void* workspace, size_t workspace_bytes, void* out, int32_t* status, Path path, DecodeParams* pp,
                   bool* empty) {
  const bool simt = !tensor_path(path);
  *empty = true;
  int err = NK_OK;
  if (!pool_ok(pool, &err)) return err;
  if (B < 0 || T < 1 || T > NK_MAX_T || Hq < 1) return NK_ERR_SHAPE;
  if (B == 0) return NK_OK;
  if (!q || !bt || !ctx || !out) return NK_ERR_NULL;
  const int Hkv = pool->num_kv_heads, D = pool->head_dim, P = pool->page_size;
  if (Hq % Hkv != 0) return NK_ERR_SHAPE;
  const int G = Hq / Hkv;
  if (B > kMaxBatch) return NK_ERR_UNSUPPORTED;
  if (max_pages < 1 || max_ctx < T || (int64_t)max_ctx > (int64_t)max_pages * P) return NK_ERR_SHAPE;
  if (!isfinite(sm_scale)) return NK_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(out, 16)) return NK_ERR_SHAPE;
  const int fmt = path_fmt(path);
  const int Tc = chunk_cols(simt, fmt, D, T, G, P);
  const bool rk_tc = path == Path::kRk8v4 && decode_mma_supported(fmt, D, Tc, G, P);
  if (simt && !rk_tc) {
    if (G > 8) return NK_ERR_UNSUPPORTED;
  } else if (!rk_tc) {
    if (!decode_tc_supported(fmt, D, Tc, G, P) && !decode_mma_supported(fmt, D, Tc, G, P)) return NK_ERR_UNSUPPORTED;
  }
  const int per_sm = rk_tc ? decode_mma_ctas_per_sm(D, T, G)
                     : path == Path::kRk8v4 ? decode_rk8v4_ctas_per_sm(D, G)
                     : (simt ? decode_simt_ctas_per_sm(D, G) : decode_mma_ctas_per_sm(D, T, G));
  const int32_t n = num_ctas > 0 ? num_ctas : default_ctas(B, Hkv, max_ctx, P, per_sm);
  // The fp32 sums of mma.sync are not rounded to nearest, and their error
  // grows with the keys of one kv-head that a CTA runs through its
  // accumulators. The tcgen05 kernel folds them (its FOLD instance); the
  // mma.sync kernels do not, so a split that would give one of their CTAs
  // more than kMaxMmaRunKeys keys of one kv-head is refused. A chunked verify
  // runs its last chunk (fewer columns) on the mma.sync kernel when that
  // chunk has too few rows for the tcgen05 one.
  if (!simt || rk_tc) {
    const int Tl = T - (T - 1) / Tc * Tc;  // columns of the last chunk
    const bool mma_kernel =
        rk_tc || !decode_tc_supported(fmt, D, Tc, G, P) || !decode_tc_supported(fmt, D, Tl, G, P);
    const int64_t unit = ((int64_t)max_ctx + P - 1) / P;
    const int64_t per_cta = (max_items(B, Hkv, max_ctx, P) + n - 1) / n;
    if (mma_kernel && (per_cta < unit ? per_cta : unit) * P > kMaxMmaRunKeys) return NK_ERR_UNSUPPORTED;
  }
  const size_t need = nk_decode_workspace_bytes(B, T, Hq, Hkv, D, n);
  if (need > 0 && (!workspace || workspace_bytes < need)) return NK_ERR_WORKSPACE;
  if (workspace && !aligned(workspace, 16)) return NK_ERR_WORKSPACE;

  DecodeParams& p = *pp;
  p.pool = reinterpret_cast<const uint8_t*>(pool->base_dev);
  p.num_pages = pool->num_pages;
  p.P = P;
  p.Hkv = Hkv;
  p.D = D;
  p.lay = layout_of(fmt, P, D);
  p.fmt = fmt;
  p.q = reinterpret_cast<const uint16_t*>(q);
  p.bt = bt;
  p.max_pages = max_pages;
  p.ctx = ctx;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.G = G;
  p.sm_scale = sm_scale;
  p.scale2 = sm_scale * kLog2e;
  p.max_ctx = max_ctx;
  p.n_ctas = n;
  const int64_t slots = (int64_t)n + (int64_t)B * Hkv;
  p.part_o = reinterpret_cast<float*>(workspace);
  p.part_lse = p.part_o + slots * G * T * D;
  p.out = reinterpret_cast<uint16_t*>(out);
  p.status = status;
  p.qT = T;
  p.trim = 0;
  p.early = 0;
  const unsigned long long wc = g_wait_cycles.load(std::memory_order_relaxed);
  p.wait_cycles = wc > 0 ? wc : kWaitCycles;
  p.withhold = g_withhold.load(std::memory_order_relaxed);
  *empty = false;
  return NK_OK;
}

int launch_decode(const DecodeParams& p0, Path path, cudaStream_t st) {
  const bool simt = !tensor_path(path);
  const int Tc = chunk_cols(simt, p0.fmt, p0.D, p0.T, p0.G, p0.P);
  const int64_t slots = (int64_t)p0.n_ctas + (int64_t)p0.B * p0.Hkv;
  for (int t0 = 0; t0 < p0.T; t0 += Tc) {
    DecodeParams p = p0;
    p.T = Tc < p0.T - t0 ? Tc : p0.T - t0;
    p.qT = p0.T;
    p.trim = p0.T - t0 - p.T;  // columns after this chunk
    p.q = p0.q + (int64_t)t0 * p0.Hq * p0.D;
    p.out = p0.out + (int64_t)t0 * p0.Hq * p0.D;
    p.part_lse = p.part_o + slots * p.G * p.T * p.D;
    if (t0 > 0) p.early = 0;  // the predecessor is the previous chunk's combine
    // tensor-core path: tcgen05 QK for head_dim 256, 64-key pages and 9 to
    // 32 rows per kv-head; the mma.sync kernel for the other shapes
    cudaError_t e = path == Path::kRk8v4 ? (decode_mma_supported(p.fmt, p.D, p.T, p.G, p.P) ? launch_decode_mma(p, st)
                                                                                          : launch_decode_rk8v4(p, st))
                    : path == Path::kSimt   ? launch_decode_simt(p, st)
                    : (decode_tc_supported(p.fmt, p.D, p.T, p.G, p.P) ? launch_decode_tc(p, st)
                                                                     : launch_decode_mma(p, st));
    if (e != cudaSuccess) return NK_ERR_CUDA;
    e = launch_decode_combine(p, st);
    if (e != cudaSuccess) return NK_ERR_CUDA;
  }
  return NK_OK;
}

int paged_decode(const nk_kv_pool* pool, const void* q, const int32_t* bt, int32_t max_pages, const int32_t* ctx,
                 int32_t B, int32_t T, int32_t Hq, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                 void* workspace, size_t workspace_bytes, void* out, int32_t* status, void* stream, Path path) {
  DecodeParams p;
  bool empty = true;
  const int err = prepare_decode(pool, q, bt, max_pages, ctx, B, T, Hq, sm_scale, max_ctx, num_ctas, workspace,
                                 workspace_bytes, out, status, path, &p, &empty);
  if (err != NK_OK || empty) return err;
  return launch_decode(p, path, reinterpret_cast<cudaStream_t>(stream));
}

// Checks the append arguments; *empty = nothing to launch.
int check_append(const nk_kv_pool* pool, const int32_t* bt, int32_t max_pages, const int32_t* start_pos,
                 const int32_t* cu_new, int32_t B, int32_t total_new, const void* k, const void* v, bool* empty) {
  *empty = true;
  int err = NK_OK;
  if (!pool_ok(pool, &err)) return err;
  if (B < 0 || total_new < 0 || max_pages < 1) return NK_ERR_SHAPE;
  if (B == 0 || total_new == 0) return NK_OK;
  if (!bt || !start_pos || !cu_new || !k || !v) return NK_ERR_NULL;
  if (!aligned(k, 16) || !aligned(v, 16)) return NK_ERR_SHAPE;
  // items of one 64-channel group of K or V of one (row, kv-head), numbered in 32 bits
  if ((int64_t)total_new * pool->num_kv_heads * 2 * (pool->head_dim / 64) >= ((int64_t)1 << 31)) return NK_ERR_SHAPE;
  *empty = false;
  return NK_OK;
}

}  // namespace

extern "C" {

size_t nk_kv_chunk_bytes(int32_t page_size, int32_t head_dim) {
  if (page_size < 1 || head_dim < kGroup || head_dim % kGroup != 0) return 0;
  return (size_t)ChunkLayout::make(page_size, head_dim).chunk;
}

size_t nk_kv_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (num_pages < 0 || num_kv_heads < 1) return 0;
  return (size_t)num_pages * (size_t)num_kv_heads * nk_kv_chunk_bytes(page_size, head_dim);
}

int nk_kv_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                 const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                 const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream) {
  bool empty = true;
  const int err = check_append(pool, block_table_dev, max_pages_per_seq, start_pos_dev, cu_new_dev, B, total_new,
                               k_dev, v_dev, &empty);
  if (err != NK_OK || empty) return err;
  const cudaError_t e = launch_kv_append(sm_count(), *pool, kFmtI8F32, block_table_dev, max_pages_per_seq, start_pos_dev,
                                         cu_new_dev, B, total_new, k_dev, v_dev, status_dev,
                                         reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NK_OK : NK_ERR_CUDA;
}

int nk_decode_step(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                   const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t total_new, const void* k_dev,
                   const void* v_dev, const void* q_dev, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                   int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                   size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream) {
  bool no_append = true, no_decode = true;
  int err = check_append(pool, block_table_dev, max_pages_per_seq, start_pos_dev, cu_new_dev, B, total_new, k_dev,
                         v_dev, &no_append);
  if (err != NK_OK) return err;
  DecodeParams p;
  err = prepare_decode(pool, q_dev, block_table_dev, max_pages_per_seq, ctx_lens_dev, B, T, num_q_heads, sm_scale,
                       max_ctx, num_ctas, workspace_dev, workspace_bytes, out_dev, status_dev, Path::kTensor, &p,
                       &no_decode);
  if (err != NK_OK) return err;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!no_append) {
    const cudaError_t e = launch_kv_append(sm_count(), *pool, kFmtI8F32, block_table_dev, max_pages_per_seq, start_pos_dev,
                                           cu_new_dev, B, total_new, k_dev, v_dev, status_dev, st);
    if (e != cudaSuccess) return NK_ERR_CUDA;
  }
  if (no_decode) return NK_OK;
  // the decode's predecessor is this append, which writes only pool pages:
  // its prologue (lengths, block-table entries, Q) may overlap the append
  p.early = no_append ? 0 : 1;
  return launch_decode(p, Path::kTensor, st);
}

size_t nk_step_host_layout(int32_t B, int32_t total_new, int32_t T, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, size_t offsets[6]) {
  if (B < 1 || total_new < 0 || T < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || !offsets) return 0;
  const size_t rows = (size_t)total_new * num_kv_heads * head_dim * 2;
  const size_t qbytes = (size_t)B * T * num_q_heads * head_dim * 2;
  const size_t sizes[6] = {rows, rows, qbytes, (size_t)B * 4, (size_t)(B + 1) * 4, (size_t)B * 4};
  size_t off = 0;
  for (int i = 0; i < 6; ++i) {
    offsets[i] = off;
    off += (sizes[i] + 255) / 256 * 256;
  }
  return off;
}

int nk_decode_step_host(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                        int32_t B, int32_t total_new, int32_t T, int32_t num_q_heads, float sm_scale,
                        int32_t max_ctx, int32_t num_ctas, const void* in_host, void* staging_dev,
                        void* workspace_dev, size_t workspace_bytes, void* out_dev, void* out_host,
                        int32_t* status_dev, int32_t* status_host, void* stream) {
  int err = NK_OK;
  if (!pool_ok(pool, &err)) return err;
  if (!in_host || !staging_dev || !out_host) return NK_ERR_NULL;
  if (!aligned(staging_dev, 16)) return NK_ERR_SHAPE;
  size_t off[6];
  const size_t bytes = nk_step_host_layout(B, total_new, T, num_q_heads, pool->num_kv_heads, pool->head_dim, off);
  if (bytes == 0) return NK_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* sb = reinterpret_cast<uint8_t*>(staging_dev);
  // the step's arguments are checked (nk_decode_step) after the transfer is
  // queued; on an error nothing is launched and the call waits for the copy
  if (cudaMemcpyAsync(sb, in_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return NK_ERR_CUDA;
  err = nk_decode_step(pool, block_table_dev, max_pages_per_seq, reinterpret_cast<const int32_t*>(sb + off[3]),
                       reinterpret_cast<const int32_t*>(sb + off[4]), total_new, sb + off[0], sb + off[1], sb + off[2],
                       reinterpret_cast<const int32_t*>(sb + off[5]), B, T, num_q_heads, sm_scale, max_ctx, num_ctas,
                       workspace_dev, workspace_bytes, out_dev, status_dev, stream);
  if (err != NK_OK) {
    (void)cudaStreamSynchronize(st);
    return err;
  }
  const size_t obytes = (size_t)B * T * num_q_heads * pool->head_dim * 2;
  if (cudaMemcpyAsync(out_host, out_dev, obytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return NK_ERR_CUDA;
  if (status_dev && status_host &&
      cudaMemcpyAsync(status_host, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return NK_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? NK_OK : NK_ERR_CUDA;
}

int32_t nk_decode_default_splits(int32_t B, int32_t num_kv_heads, int32_t max_ctx, int32_t page_size) {
  if (B < 1 || num_kv_heads < 1 || max_ctx < 1 || page_size < 1) return 1;
  // one CTA per SM: the tensor-core kernels' residency (decode_mma_ctas_per_sm)
  return default_ctas(B, num_kv_heads, max_ctx, page_size, 1);
}

int32_t nk_decode_default_ctas(int32_t B, int32_t num_kv_heads, int32_t max_ctx, int32_t page_size) {
  return nk_decode_default_splits(B, num_kv_heads, max_ctx, page_size);
}

size_t nk_decode_workspace_bytes(int32_t B, int32_t T, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_ctas) {
  if (B < 1 || T < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads || head_dim < 1) return 0;
  if (num_ctas < 1) num_ctas = (sm_count() > 0 ? sm_count() : 148) * 2;
  const int64_t G = num_q_heads / num_kv_heads;
  const int64_t slots = (int64_t)num_ctas + (int64_t)B * num_kv_heads;
  const int64_t rows = slots * G * T;
  const int64_t bytes = rows * head_dim * 4 + rows * 4;
  return (size_t)((bytes + 255) / 256 * 256);
}

int nk_paged_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                         int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                         int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                         size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream) {
  return paged_decode(pool, q_dev, block_table_dev, max_pages_per_seq, ctx_lens_dev, B, T, num_q_heads, sm_scale,
                      max_ctx, num_ctas, workspace_dev, workspace_bytes, out_dev, status_dev, stream, Path::kTensor);
}

int nk_paged_decode_attn_simt(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                              int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                              int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                              void* workspace_dev, size_t workspace_bytes, void* out_dev, int32_t* status_dev,
                              void* stream) {
  return paged_decode(pool, q_dev, block_table_dev, max_pages_per_seq, ctx_lens_dev, B, T, num_q_heads, sm_scale,
                      max_ctx, num_ctas, workspace_dev, workspace_bytes, out_dev, status_dev, stream, Path::kSimt);
}

size_t nk_rk8v4_chunk_bytes(int32_t page_size, int32_t head_dim) {
  if (page_size < 1 || head_dim < kGroup || head_dim % kGroup != 0) return 0;
  return (size_t)rk8v4_layout(page_size, head_dim).chunk;
}

size_t nk_rk8v4_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (num_pages < 0 || num_kv_heads < 1) return 0;
  return (size_t)num_pages * (size_t)num_kv_heads * nk_rk8v4_chunk_bytes(page_size, head_dim);
}

int nk_rk8v4_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                    const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                    const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream) {
  bool empty = true;
  const int err = check_append(pool, block_table_dev, max_pages_per_seq, start_pos_dev, cu_new_dev, B, total_new,
                               k_dev, v_dev, &empty);
  if (err != NK_OK || empty) return err;
  const cudaError_t e = launch_rk8v4_append(sm_count(), *pool, block_table_dev, max_pages_per_seq, start_pos_dev,
                                            cu_new_dev, B, total_new, k_dev, v_dev, status_dev,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NK_OK : NK_ERR_CUDA;
}

int nk_rk8v4_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                         int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                         int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                         size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream) {
  return paged_decode(pool, q_dev, block_table_dev, max_pages_per_seq, ctx_lens_dev, B, T, num_q_heads, sm_scale,
                      max_ctx, num_ctas, workspace_dev, workspace_bytes, out_dev, status_dev, stream, Path::kRk8v4);
}

size_t nk_i8f16_chunk_bytes(int32_t page_size, int32_t head_dim) {
  if (page_size < 1 || head_dim < kGroup || head_dim % kGroup != 0) return 0;
  return (size_t)i8f16_layout(page_size, head_dim).chunk;
}

size_t nk_i8f16_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (num_pages < 0 || num_kv_heads < 1) return 0;
  return (size_t)num_pages * (size_t)num_kv_heads * nk_i8f16_chunk_bytes(page_size, head_dim);
}

size_t nk_bf16kv_chunk_bytes(int32_t page_size, int32_t head_dim) {
  if (page_size < 1 || head_dim < kGroup || head_dim % kGroup != 0) return 0;
  return (size_t)bf16kv_layout(page_size, head_dim).chunk;
}

size_t nk_bf16kv_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim) {
  if (num_pages < 0 || num_kv_heads < 1) return 0;
  return (size_t)num_pages * (size_t)num_kv_heads * nk_bf16kv_chunk_bytes(page_size, head_dim);
}

static int append_fmt(int fmt, const nk_kv_pool* pool, const int32_t* bt, int32_t max_pages, const int32_t* start_pos,
                      const int32_t* cu_new, int32_t B, int32_t total_new, const void* k, const void* v,
                      int32_t* status, void* stream) {
  bool empty = true;
  const int err = check_append(pool, bt, max_pages, start_pos, cu_new, B, total_new, k, v, &empty);
  if (err != NK_OK || empty) return err;
  const cudaError_t e = launch_kv_append(sm_count(), *pool, fmt, bt, max_pages, start_pos, cu_new, B, total_new, k, v,
                                         status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NK_OK : NK_ERR_CUDA;
}

int nk_i8f16_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                    const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                    const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream) {
  return append_fmt(kFmtI8F16, pool, block_table_dev, max_pages_per_seq, start_pos_dev, cu_new_dev, B, total_new,
                    k_dev, v_dev, status_dev, stream);
}

int nk_bf16kv_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                     const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                     const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream) {
  return append_fmt(kFmtBf16, pool, block_table_dev, max_pages_per_seq, start_pos_dev, cu_new_dev, B, total_new,
                    k_dev, v_dev, status_dev, stream);
}

int nk_i8f16_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                         int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                         int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                         size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream) {
  return paged_decode(pool, q_dev, block_table_dev, max_pages_per_seq, ctx_lens_dev, B, T, num_q_heads, sm_scale,
                      max_ctx, num_ctas, workspace_dev, workspace_bytes, out_dev, status_dev, stream, Path::kTensorF16);
}

int nk_bf16kv_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                          int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                          int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                          void* workspace_dev, size_t workspace_bytes, void* out_dev, int32_t* status_dev,
                          void* stream) {
  // The bf16 path of the mma.sync kernel ended with a GPU fault at the C1
  // decode size (32,768 keys, 152 CTAs) whose cause is not found yet; until it
  // is, no kernel is launched for a bf16 pool.
  (void)pool; (void)q_dev; (void)block_table_dev; (void)max_pages_per_seq; (void)ctx_lens_dev; (void)B; (void)T;
  (void)num_q_heads; (void)sm_scale; (void)max_ctx; (void)num_ctas; (void)workspace_dev; (void)workspace_bytes;
  (void)out_dev; (void)status_dev; (void)stream;
  return NK_ERR_UNSUPPORTED;
}

int nk_paged_prefill_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                          int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                          int32_t num_q_heads, float sm_scale, int32_t max_ctx, void* out_dev, int32_t* status_dev,
                          void* stream) {
  int err = NK_OK;
  if (!pool_ok(pool, &err)) return err;
  if (B < 0 || T < 1 || num_q_heads < 1) return NK_ERR_SHAPE;
  if (B == 0) return NK_OK;
  if (!q_dev || !block_table_dev || !ctx_lens_dev || !out_dev) return NK_ERR_NULL;
  const int Hkv = pool->num_kv_heads, D = pool->head_dim, P = pool->page_size;
  if (num_q_heads % Hkv != 0) return NK_ERR_SHAPE;
  if (max_pages_per_seq < 1 || max_ctx < T || (int64_t)max_ctx > (int64_t)max_pages_per_seq * P) return NK_ERR_SHAPE;
  if (!isfinite(sm_scale)) return NK_ERR_SHAPE;
  if (!aligned(q_dev, 16) || !aligned(out_dev, 16)) return NK_ERR_SHAPE;
  if (!prefill_supported(kFmtI8F32, D, P)) return NK_ERR_UNSUPPORTED;
  const int G = num_q_heads / Hkv;
  const int64_t tiles = ((int64_t)G * T + prefill_rows_per_cta() - 1) / prefill_rows_per_cta();
  const int64_t grid = (int64_t)B * Hkv * tiles;
  if ((int64_t)G * T >= ((int64_t)1 << 31) || grid >= ((int64_t)1 << 31)) return NK_ERR_SHAPE;
  DecodeParams p = {};
  p.pool = reinterpret_cast<const uint8_t*>(pool->base_dev);
  p.num_pages = pool->num_pages;
  p.P = P;
  p.Hkv = Hkv;
  p.D = D;
  p.lay = ChunkLayout::make(P, D);
  p.fmt = kFmtI8F32;
  p.q = reinterpret_cast<const uint16_t*>(q_dev);
  p.bt = block_table_dev;
  p.max_pages = max_pages_per_seq;
  p.ctx = ctx_lens_dev;
  p.B = B;
  p.T = T;
  p.qT = T;
  p.Hq = num_q_heads;
  p.G = G;
  p.sm_scale = sm_scale;
  p.scale2 = sm_scale * kLog2e;
  p.max_ctx = max_ctx;
  p.n_ctas = (int)grid;
  p.out = reinterpret_cast<uint16_t*>(out_dev);
  p.status = status_dev;
  const unsigned long long wc = g_wait_cycles.load(std::memory_order_relaxed);
  p.wait_cycles = wc > 0 ? wc : kWaitCycles;
  p.withhold = g_withhold.load(std::memory_order_relaxed);
  return launch_prefill(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? NK_OK : NK_ERR_CUDA;
}

int nk_attn_combine(const float* part_o_dev, const float* part_lse_dev, int32_t num_splits, int32_t rows,
                    int32_t head_dim, void* out_dev, void* stream) {
  if (num_splits < 0 || rows < 0) return NK_ERR_SHAPE;
  if (!(head_dim == 64 || head_dim == 128 || head_dim == 256)) return NK_ERR_UNSUPPORTED;
  if (rows == 0) return NK_OK;
  if (!part_o_dev || !part_lse_dev || !out_dev) return NK_ERR_NULL;
  if (!aligned(part_o_dev, 16) || !aligned(out_dev, 16)) return NK_ERR_SHAPE;
  const cudaError_t e = launch_attn_combine(part_o_dev, part_lse_dev, num_splits, rows, head_dim,
                                            reinterpret_cast<uint16_t*>(out_dev),
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NK_OK : NK_ERR_CUDA;
}

const char* nk_status_string(int code) {
  switch (code) {
    case NK_OK: return "ok";
    case NK_ERR_NULL: return "a required pointer is NULL";
    case NK_ERR_SHAPE: return "a size is out of range, inconsistent or misaligned";
    case NK_ERR_UNSUPPORTED: return "no kernel for this shape";
    case NK_ERR_WORKSPACE: return "workspace missing or too small";
    case NK_ERR_CUDA: return "a CUDA call failed";
    case NK_ERR_DEVICE_DATA: return "device-resident data out of range (see the status word)";
    case NK_ERR_TIMEOUT: return "a bounded wait on an asynchronous copy gave up";
    default: return "unknown status";
  }
}

int nk_version(void) { return 100; }

void nk_test_inject_copy_stall(int32_t withheld_page, uint64_t wait_cycles) {
  g_wait_cycles.store(withheld_page >= 0 ? wait_cycles : 0ull, std::memory_order_relaxed);
  g_withhold.store(withheld_page >= 0 ? withheld_page : -1, std::memory_order_relaxed);
}

}  // extern "C"
