// pkv_decode_mma_bf16.cu -- tensor-core decode variants for bf16 pools (head_dim 128 and 64).
#include "pkv_decode_mma.cuh"

namespace pkv {

cudaError_t launch_mma_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int cols, int shape, bool gen, cudaStream_t stream) {
  constexpr KvType KV = KvType::kBf16;
  if (p.head_dim == 128) {
    switch (shape) {
      case 0: return launch_mma_gen<KV, 128, kShapesBf16D128[0].stages, kShapesBf16D128[0].bps>(p, tk, tv, cols, gen, stream);
      case 1: return launch_mma_gen<KV, 128, kShapesBf16D128[1].stages, kShapesBf16D128[1].bps>(p, tk, tv, cols, gen, stream);
    }
  } else if (p.head_dim == 64) {
    switch (shape) {
      case 0: return launch_mma_gen<KV, 64, kShapesBf16D64[0].stages, kShapesBf16D64[0].bps>(p, tk, tv, cols, gen, stream);
      case 1: return launch_mma_gen<KV, 64, kShapesBf16D64[1].stages, kShapesBf16D64[1].bps>(p, tk, tv, cols, gen, stream);
    }
  }
  return cudaErrorInvalidValue;
}

int occupancy_mma_bf16(int head_dim, int cols, int shape, bool gen) {
  constexpr KvType KV = KvType::kBf16;
  if (head_dim == 128) {
    switch (shape) {
      case 0: return occupancy_mma_gen<KV, 128, kShapesBf16D128[0].stages, kShapesBf16D128[0].bps>(cols, gen);
      case 1: return occupancy_mma_gen<KV, 128, kShapesBf16D128[1].stages, kShapesBf16D128[1].bps>(cols, gen);
    }
  } else if (head_dim == 64) {
    switch (shape) {
      case 0: return occupancy_mma_gen<KV, 64, kShapesBf16D64[0].stages, kShapesBf16D64[0].bps>(cols, gen);
      case 1: return occupancy_mma_gen<KV, 64, kShapesBf16D64[1].stages, kShapesBf16D64[1].bps>(cols, gen);
    }
  }
  return 0;
}

}  // namespace pkv
