// pkv_decode_fp8.cu -- CUDA-core decode kernels for FP8 (E4M3) pools (instantiations and dispatch).
#include "pkv_decode.cuh"

namespace pkv {

// Warps per CTA and ring stages per warp for FP8 pools (the INT8 layout: one K and one V
// code tile plus 16 fp32 scales each per stage).
constexpr int kNwFp8 = 4;
constexpr int kStagesFp8D128 = 5;
constexpr int kStagesFp8D64 = 6;

template <int D, int S>
static cudaError_t dispatch_cols(const DecodeParams& p, int cols, cudaStream_t stream) {
  switch (cols) {
    case 1: return launch_decode_variant<KvType::kFp8, D, 1, kNwFp8, S>(p, stream);
    case 2: return launch_decode_variant<KvType::kFp8, D, 2, kNwFp8, S>(p, stream);
    case 4: return launch_decode_variant<KvType::kFp8, D, 4, kNwFp8, S>(p, stream);
    case 8: return launch_decode_variant<KvType::kFp8, D, 8, kNwFp8, S>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_fp8(const DecodeParams& p, int cols, cudaStream_t stream) {
  if (p.head_dim == 128) return dispatch_cols<128, kStagesFp8D128>(p, cols, stream);
  if (p.head_dim == 64) return dispatch_cols<64, kStagesFp8D64>(p, cols, stream);
  return cudaErrorInvalidValue;
}

int ctas_per_sm_fp8(int head_dim, int cols) {
  if (head_dim == 128) {
    switch (cols) {
      case 1: return ctas_per_sm_variant<KvType::kFp8, 128, 1, kNwFp8, kStagesFp8D128>();
      case 2: return ctas_per_sm_variant<KvType::kFp8, 128, 2, kNwFp8, kStagesFp8D128>();
      case 4: return ctas_per_sm_variant<KvType::kFp8, 128, 4, kNwFp8, kStagesFp8D128>();
      case 8: return ctas_per_sm_variant<KvType::kFp8, 128, 8, kNwFp8, kStagesFp8D128>();
    }
  } else if (head_dim == 64) {
    switch (cols) {
      case 1: return ctas_per_sm_variant<KvType::kFp8, 64, 1, kNwFp8, kStagesFp8D64>();
      case 2: return ctas_per_sm_variant<KvType::kFp8, 64, 2, kNwFp8, kStagesFp8D64>();
      case 4: return ctas_per_sm_variant<KvType::kFp8, 64, 4, kNwFp8, kStagesFp8D64>();
      case 8: return ctas_per_sm_variant<KvType::kFp8, 64, 8, kNwFp8, kStagesFp8D64>();
    }
  }
  return 0;
}

}  // namespace pkv
