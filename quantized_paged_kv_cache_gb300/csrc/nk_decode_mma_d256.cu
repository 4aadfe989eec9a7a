// nk_decode_mma_d256.cu -- tensor-core decode instances for head_dim 256
// (one translation unit per head_dim so they compile in parallel).
#include "nk_decode_mma.cuh"

namespace nk {
namespace mma {

template <int D, int NT, int CS, int FMT>
static cudaError_t launch_tb(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  const Geometry geo = geometry(FMT, D, NT, CS, p.P, p.B);
  if (geo.stages < 2 || geo.total > kSmemLimit) return cudaErrorInvalidConfiguration;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(decode_mma_kernel<D, NT, CS, FMT>), geo.total);
  if (e != cudaSuccess) return e;
  return launch_chained(decode_mma_kernel<D, NT, CS, FMT>, dim3(p.n_ctas), dim3(kThreads), geo.total, st, map, map,
                        p);
}

// INT8 pools with fp32 or fp16 scales, and bf16 pools
template <int D, int NT, int CS>
static cudaError_t launch_t(const CUtensorMap& map, const DecodeParams& p, cudaStream_t st) {
  if (p.fmt == kFmtBf16) return launch_tb<D, NT, CS, kFmtBf16>(map, p, st);
  if (p.fmt == kFmtI8F16) return launch_tb<D, NT, CS, kFmtI8F16>(map, p, st);
  return launch_tb<D, NT, CS, kFmtI8F32>(map, p, st);
}

cudaError_t launch_d256(const CUtensorMap& map, const DecodeParams& p, int NT, cudaStream_t st) {
  switch (NT) {
    case 1: return launch_t<256, 1, 1>(map, p, st);
    case 2: return launch_t<256, 2, 2>(map, p, st);
    case 3: return launch_t<256, 3, 2>(map, p, st);
    case 4: return launch_t<256, 4, 4>(map, p, st);
    case 5: return launch_t<256, 5, 4>(map, p, st);
    case 6: return launch_t<256, 6, 4>(map, p, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace mma
}  // namespace nk
