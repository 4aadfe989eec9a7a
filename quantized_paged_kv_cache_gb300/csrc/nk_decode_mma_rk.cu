// nk_decode_mma_rk.cu -- tensor-core decode instances for the rk8v4 format
// ("NInfer-3090" README, "RotorQuant KV (rk8v4)": rotated INT8 keys with an
// INT8 tensor-core QK, 4-bit values): head_dim 128 and 256, up to 32 query
// rows per kv-head (one translation unit so they compile in parallel with
// the INT8 instances).
#include "nk_decode_mma.cuh"

namespace nk {
namespace mma {

template <int D, int NT, int CS>
static cudaError_t launch_rk_t(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, cudaStream_t st) {
  const Geometry geo = geometry(kFmtRk8v4, D, NT, CS, p.P, p.B);
  if (geo.stages < 2 || geo.total > kSmemLimit) return cudaErrorInvalidConfiguration;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(decode_mma_kernel<D, NT, CS, kFmtRk8v4>), geo.total);
  if (e != cudaSuccess) return e;
  return launch_chained(decode_mma_kernel<D, NT, CS, kFmtRk8v4>, dim3(p.n_ctas), dim3(kThreads), geo.total, st, mk,
                        mv, p);
}

// the channel splits of channel_split_rk
cudaError_t launch_rk(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, int NT, cudaStream_t st) {
  if (p.D == 256) {
    switch (NT) {
      case 1: return launch_rk_t<256, 1, 2>(mk, mv, p, st);
      case 2: return launch_rk_t<256, 2, 4>(mk, mv, p, st);
      case 3: return launch_rk_t<256, 3, 4>(mk, mv, p, st);
      case 4: return launch_rk_t<256, 4, 4>(mk, mv, p, st);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  if (p.D == 128) {
    switch (NT) {
      case 1: return launch_rk_t<128, 1, 1>(mk, mv, p, st);
      case 2: return launch_rk_t<128, 2, 2>(mk, mv, p, st);
      case 3: return launch_rk_t<128, 3, 2>(mk, mv, p, st);
      case 4: return launch_rk_t<128, 4, 2>(mk, mv, p, st);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace mma
}  // namespace nk
