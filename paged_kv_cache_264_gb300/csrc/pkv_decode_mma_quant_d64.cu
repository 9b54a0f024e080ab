// pkv_decode_mma_quant_d64.cu -- tensor-core decode variants for INT8 and FP8 (E4M3) pools
// at head_dim 64: 64-byte token rows, two to a 128-byte swizzled box row (see MmaCfg).
#include "pkv_decode_mma.cuh"

namespace pkv {

template <KvType KV>
static cudaError_t launch_d64(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int cols, int shape, bool gen, cudaStream_t stream) {
  switch (shape) {
    case 0: return launch_mma_gen<KV, 64, kShapesQuantD64[0].stages, kShapesQuantD64[0].bps>(p, tk, tv, cols, gen, stream);
    case 1: return launch_mma_gen<KV, 64, kShapesQuantD64[1].stages, kShapesQuantD64[1].bps>(p, tk, tv, cols, gen, stream);
  }
  return cudaErrorInvalidValue;
}

template <KvType KV>
static int occupancy_d64(int cols, int shape, bool gen) {
  switch (shape) {
    case 0: return occupancy_mma_gen<KV, 64, kShapesQuantD64[0].stages, kShapesQuantD64[0].bps>(cols, gen);
    case 1: return occupancy_mma_gen<KV, 64, kShapesQuantD64[1].stages, kShapesQuantD64[1].bps>(cols, gen);
  }
  return 0;
}

cudaError_t launch_mma_quant_d64(KvType kv, const DecodeParams& p, const CUtensorMap& tk,
                                 const CUtensorMap& tv, int cols, int shape, bool gen, cudaStream_t stream) {
  if (kv == KvType::kInt8) return launch_d64<KvType::kInt8>(p, tk, tv, cols, shape, gen, stream);
  if (kv == KvType::kFp8) return launch_d64<KvType::kFp8>(p, tk, tv, cols, shape, gen, stream);
  return cudaErrorInvalidValue;
}

int occupancy_mma_quant_d64(KvType kv, int cols, int shape, bool gen) {
  if (kv == KvType::kInt8) return occupancy_d64<KvType::kInt8>(cols, shape, gen);
  if (kv == KvType::kFp8) return occupancy_d64<KvType::kFp8>(cols, shape, gen);
  return 0;
}

}  // namespace pkv
