// nk_decode.cuh -- parameters and launchers shared by the decode kernels.
#pragma once

#include "nk_common.cuh"

namespace nk {

struct DecodeParams {
  const uint8_t* pool;
  int num_pages, P, Hkv, D;
  ChunkLayout lay;
  const uint16_t* q;      // bf16 [B][qT][Hq][D], already offset to this call's first column
  const int32_t* bt;      // [B][max_pages]
  int max_pages;
  const int32_t* ctx;     // [B]
  int B, T, Hq, G;
  // Column chunks of a wide verify: this launch covers T of the qT columns
  // of q / out, and every context length is read as ctx[b] - trim (the
  // columns after the chunk are left out, so the chunk's last column sees
  // keys up to its own causal limit).
  int qT, trim;
  float sm_scale;
  float scale2;           // sm_scale * log2(e)
  int max_ctx;
  int n_ctas;
  float* part_o;          // [n_ctas + B*Hkv][T*G][D]
  float* part_lse;        // [n_ctas + B*Hkv][T*G]
  uint16_t* out;          // bf16 [B][qT][Hq][D], offset like q
  int32_t* status;
  // 1: the previous kernel on the stream is this call's own append, which
  // writes only pool pages, so the split kernel reads the context lengths,
  // block-table entries and Q before waiting for it (it waits before its
  // first page load). Written before that append was launched, those inputs
  // are visible: the append itself waited for every earlier kernel before
  // this kernel could start.
  int early;
  int fmt;  // KvFmt of the pool (the rk8v4 kernel ignores it)
  // Failure-detection tests (nk_test_inject_copy_stall): every bounded wait
  // gives up after wait_cycles, and the page copies of CTA page numbers
  // >= withhold are never issued (-1: all issued).
  unsigned long long wait_cycles;
  int withhold;
  __host__ __device__ bool issuable(int q) const { return withhold < 0 || q < withhold; }
  __host__ __device__ SplitShape shape() const { return SplitShape{B, Hkv, P, T, max_ctx, max_pages}; }
};

// Flag invalid ctx lengths once (block 0 of a kernel).
__device__ __forceinline__ void flag_bad_ctx(const DecodeParams& p) {
  if (blockIdx.x != 0) return;
  for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
    const int L = p.ctx[b] - p.trim;
    if (L < p.T || L > p.max_ctx || (int64_t)L > (int64_t)p.max_pages * p.P) flag(p.status, NK_DEVFLAG_BAD_CTX);
  }
}

cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_prefill(const DecodeParams& p, cudaStream_t stream);
bool prefill_supported(int fmt, int D, int P);
int prefill_rows_per_cta();
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream);
bool decode_tc_supported(int fmt, int D, int T, int G, int P);
cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_attn_combine(const float* part_o, const float* part_lse, int S, int R, int D, uint16_t* out,
                                cudaStream_t stream);
int decode_simt_ctas_per_sm(int D, int G);
int decode_mma_ctas_per_sm(int D, int T, int G);
bool decode_mma_supported(int fmt, int D, int T, int G, int P);

}  // namespace nk
