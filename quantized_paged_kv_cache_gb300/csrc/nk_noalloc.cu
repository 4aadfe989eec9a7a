// nk_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand the library a scratch buffer: code running
// inside a host that owns every allocation and forbids cudaMalloc after start
// (fixed-budget serving processes, plugin hosts with strict memory
// accounting), or code that must not trigger the implicit device
// synchronization an allocation can cause. For them the split-partial scratch
// of nk_paged_decode_attn lives in one fixed-size array in device global
// memory that belongs to this library: every GPU that loads libnk.so holds it
// until the process exits.
//
// The array is shared by all calls on a device and keeps the previous call's
// contents. Nothing in it needs to start at zero: each call writes every
// partial slot it later reads. Two calls whose kernels overlap on the GPU
// (different streams, or the same array from several threads) race on it.
#include <mutex>

#include "nk_decode.cuh"

namespace {

constexpr size_t kStaticBytes = (size_t)NK_NOALLOC_MAX_WORKSPACE;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_decode_scratch[kStaticBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device; looked up once per
// device (the first call on a device does it) and kept until the process
// exits, so the entry point must not be used across a cudaDeviceReset of that
// device (the module would be reloaded at another address).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return NK_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) {
      (void)cudaGetLastError();
      return NK_ERR_CUDA;
    }
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return NK_OK;
}

}  // namespace

extern "C" int nk_paged_decode_attn_noalloc(const nk_kv_pool* pool, const void* q_dev,
                                            const int32_t* block_table_dev, int32_t max_pages_per_seq,
                                            const int32_t* ctx_lens_dev, int32_t B, int32_t T, int32_t num_q_heads,
                                            float sm_scale, int32_t max_ctx, int32_t num_ctas, void* out_dev,
                                            int32_t* status_dev, void* stream) {
  // The address lookup comes first, so that a call with B = 0 (which
  // launches nothing) sets up the current device ahead of a stream capture.
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != NK_OK) return rc;
  if (B == 0) return NK_OK;
  // The regular entry point checks the arguments, picks the same default
  // split count and returns NK_ERR_WORKSPACE when the partials of this shape
  // do not fit the array.
  return nk_paged_decode_attn(pool, q_dev, block_table_dev, max_pages_per_seq, ctx_lens_dev, B, T, num_q_heads,
                              sm_scale, max_ctx, num_ctas, scratch, kStaticBytes, out_dev, status_dev, stream);
}
