// nk_decode_mma.cu -- host side of the tensor-core decode kernel: shape
// support, the TMA descriptor of the pool, and dispatch to the instances
// compiled per head_dim (nk_decode_mma_d*.cu).
#include "nk_decode_mma.cuh"

namespace nk {
namespace mma {

// Warps per team (channel split) for a head_dim and a number of 8-row tiles:
// chosen so one warp's Q fragments and output accumulator stay near 150
// registers. rk8v4 rows carry a second (low) fp16 part, so its warps take
// narrower slices.
int channel_split(int D, int NT) {
  if (D == 256) return NT <= 1 ? 1 : (NT <= 3 ? 2 : 4);
  if (D == 128) return NT <= 3 ? 1 : 2;
  return 1;
}
int channel_split_rk(int D, int NT) {
  if (D == 256) return NT <= 1 ? 2 : 4;
  return NT <= 1 ? 1 : 2;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

// 4-D view of the pool's code bytes: [D channels][P keys][K|V][page*Hkv + h],
// boxes of [min(D,128)][P][2][1] with the matching shared-memory swizzle.
// rk8v4: part 0 = the key codes, 3-D [D][P][page * Hkv + h], boxes of
// [128][P][1]; part 1 = the value codes, [D / 2][P][page * Hkv + h] from the
// chunk's value offset, one box of [D / 2][P][1]. 128-byte swizzle (64-byte
// for 64-byte value rows).
static cudaError_t encode_rk_map(const DecodeParams& p, int part, CUtensorMap* map) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t row = part == 0 ? (cuuint64_t)p.D : (cuuint64_t)p.D / 2;
  cuuint64_t dims[3] = {row, (cuuint64_t)p.P, (cuuint64_t)p.num_pages * p.Hkv};
  cuuint64_t strides[2] = {row, (cuuint64_t)p.lay.chunk};
  cuuint32_t box[3] = {(cuuint32_t)(row < 128 ? row : 128), (cuuint32_t)p.P, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                        const_cast<uint8_t*>(p.pool + (part == 0 ? 0 : p.lay.vc)), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, row >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_pool_map(const DecodeParams& p, CUtensorMap* map, int part) {
  // the last few maps of this host thread, by pool geometry (encoding one is
  // host work on the critical path of every call)
  struct Cached {
    const void* base;
    int num_pages, P, Hkv, D, fmt, part;
    CUtensorMap map;
  };
  thread_local Cached cache[8];
  thread_local int used = 0, next = 0;
  for (int i = 0; i < used; ++i) {
    const Cached& c = cache[i];
    if (c.base == p.pool && c.num_pages == p.num_pages && c.P == p.P && c.Hkv == p.Hkv && c.D == p.D &&
        c.fmt == p.fmt && c.part == part) {
      *map = c.map;
      return cudaSuccess;
    }
  }
  if (p.fmt == kFmtRk8v4) {
    const cudaError_t e = encode_rk_map(p, part, map);
    if (e != cudaSuccess) return e;
    Cached& c = cache[next];
    c = Cached{p.pool, p.num_pages, p.P, p.Hkv, p.D, p.fmt, part, *map};
    next = (next + 1) % 8;
    if (used < 8) ++used;
    return cudaSuccess;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  // bf16 pools: 2-byte elements, boxes of 64 channels (128-byte rows)
  const bool bf = p.fmt == kFmtBf16;
  const cuuint64_t esize = bf ? 2 : 1;
  cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)p.P, 2, (cuuint64_t)p.num_pages * p.Hkv};
  cuuint64_t strides[3] = {(cuuint64_t)p.D * esize, (cuuint64_t)p.lay.vc, (cuuint64_t)p.lay.chunk};
  cuuint32_t box[4] = {(cuuint32_t)(bf ? 64 : (p.D < 128 ? p.D : 128)), (cuuint32_t)p.P, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, bf ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                        const_cast<uint8_t*>(p.pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        (p.D == 64 && !bf) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Cached& c = cache[next];
  c = Cached{p.pool, p.num_pages, p.P, p.Hkv, p.D, p.fmt, part, *map};
  next = (next + 1) % 8;
  if (used < 8) ++used;
  return cudaSuccess;
}

cudaError_t launch_d256(const CUtensorMap& map, const DecodeParams& p, int NT, cudaStream_t st);
cudaError_t launch_d128(const CUtensorMap& map, const DecodeParams& p, int NT, cudaStream_t st);
cudaError_t launch_d64(const CUtensorMap& map, const DecodeParams& p, int NT, cudaStream_t st);
cudaError_t launch_rk(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, int NT, cudaStream_t st);

}  // namespace mma

bool decode_mma_supported(int fmt, int D, int T, int G, int P) {
  const int M = G * T;
  if (M < 1 || M > 48 || P % 16 != 0 || P > 256) return false;
  if (!(D == 64 || D == 128 || D == 256)) return false;
  const int NT = (M + 7) / 8;
  if (fmt == kFmtRk8v4) {
    // rk8v4 instances: head_dim 128 or 256, up to 32 rows per kv-head
    if (D == 64 || M > 32) return false;
    return mma::geometry(fmt, D, NT, mma::channel_split_rk(D, NT), P, kMaxBatch).stages >= 2;
  }
  const mma::Geometry g = mma::geometry(fmt, D, NT, mma::channel_split(D, NT), P, kMaxBatch);
  return g.stages >= 2;
}

int decode_mma_ctas_per_sm(int, int, int) { return 1; }

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream) {
  CUtensorMap map;
  cudaError_t e = mma::make_pool_map(p, &map, 0);
  if (e != cudaSuccess) return e;
  const int NT = (p.G * p.T + 7) / 8;
  if (p.fmt == kFmtRk8v4) {
    CUtensorMap mapv;
    e = mma::make_pool_map(p, &mapv, 1);
    if (e != cudaSuccess) return e;
    return mma::launch_rk(map, mapv, p, NT, stream);
  }
  if (p.D == 256) return mma::launch_d256(map, p, NT, stream);
  if (p.D == 128) return mma::launch_d128(map, p, NT, stream);
  return mma::launch_d64(map, p, NT, stream);
}

}  // namespace nk
