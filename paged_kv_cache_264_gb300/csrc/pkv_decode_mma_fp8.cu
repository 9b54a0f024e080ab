// pkv_decode_mma_fp8.cu -- tensor-core decode variants for FP8 (E4M3) pools (head_dim 128).
#include "pkv_decode_mma.cuh"

namespace pkv {

cudaError_t launch_mma_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                          int cols, int shape, bool gen, cudaStream_t stream) {
  constexpr KvType KV = KvType::kFp8;
  switch (shape) {
    case 0: return launch_mma_gen<KV, 128, kShapesQuant[0].stages, kShapesQuant[0].bps>(p, tk, tv, cols, gen, stream);
    case 1: return launch_mma_gen<KV, 128, kShapesQuant[1].stages, kShapesQuant[1].bps>(p, tk, tv, cols, gen, stream);
    case 2: return launch_mma_gen<KV, 128, kShapesQuant[2].stages, kShapesQuant[2].bps>(p, tk, tv, cols, gen, stream);
    case 3: return launch_mma_gen<KV, 128, kShapesQuant[3].stages, kShapesQuant[3].bps>(p, tk, tv, cols, gen, stream);
  }
  return cudaErrorInvalidValue;
}

int occupancy_mma_fp8(int cols, int shape, bool gen) {
  constexpr KvType KV = KvType::kFp8;
  switch (shape) {
    case 0: return occupancy_mma_gen<KV, 128, kShapesQuant[0].stages, kShapesQuant[0].bps>(cols, gen);
    case 1: return occupancy_mma_gen<KV, 128, kShapesQuant[1].stages, kShapesQuant[1].bps>(cols, gen);
    case 2: return occupancy_mma_gen<KV, 128, kShapesQuant[2].stages, kShapesQuant[2].bps>(cols, gen);
    case 3: return occupancy_mma_gen<KV, 128, kShapesQuant[3].stages, kShapesQuant[3].bps>(cols, gen);
  }
  return 0;
}

}  // namespace pkv
