// pkv_decode_int8.cu -- decode kernels for INT8 pools (instantiations and dispatch).
#include "pkv_decode.cuh"

namespace pkv {

// Warps per CTA and ring stages per warp for INT8 pools.  A stage holds one K and one
// V code tile plus their 16 fp32 scales each: 4224 B at head_dim 128, 2176 B at 64.
constexpr int kNwInt8 = 4;
constexpr int kStagesInt8D128 = 5;
constexpr int kStagesInt8D64 = 6;

template <int D, int S>
static cudaError_t dispatch_cols(const DecodeParams& p, int cols, cudaStream_t stream) {
  switch (cols) {
    case 1: return launch_decode_variant<KvType::kInt8, D, 1, kNwInt8, S>(p, stream);
    case 2: return launch_decode_variant<KvType::kInt8, D, 2, kNwInt8, S>(p, stream);
    case 4: return launch_decode_variant<KvType::kInt8, D, 4, kNwInt8, S>(p, stream);
    case 8: return launch_decode_variant<KvType::kInt8, D, 8, kNwInt8, S>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_int8(const DecodeParams& p, int cols, cudaStream_t stream) {
  if (p.head_dim == 128) return dispatch_cols<128, kStagesInt8D128>(p, cols, stream);
  if (p.head_dim == 64) return dispatch_cols<64, kStagesInt8D64>(p, cols, stream);
  return cudaErrorInvalidValue;
}

int ctas_per_sm_int8(int head_dim, int cols) {
  if (head_dim == 128) {
    switch (cols) {
      case 1: return ctas_per_sm_variant<KvType::kInt8, 128, 1, kNwInt8, kStagesInt8D128>();
      case 2: return ctas_per_sm_variant<KvType::kInt8, 128, 2, kNwInt8, kStagesInt8D128>();
      case 4: return ctas_per_sm_variant<KvType::kInt8, 128, 4, kNwInt8, kStagesInt8D128>();
      case 8: return ctas_per_sm_variant<KvType::kInt8, 128, 8, kNwInt8, kStagesInt8D128>();
    }
  } else if (head_dim == 64) {
    switch (cols) {
      case 1: return ctas_per_sm_variant<KvType::kInt8, 64, 1, kNwInt8, kStagesInt8D64>();
      case 2: return ctas_per_sm_variant<KvType::kInt8, 64, 2, kNwInt8, kStagesInt8D64>();
      case 4: return ctas_per_sm_variant<KvType::kInt8, 64, 4, kNwInt8, kStagesInt8D64>();
      case 8: return ctas_per_sm_variant<KvType::kInt8, 64, 8, kNwInt8, kStagesInt8D64>();
    }
  }
  return 0;
}

}  // namespace pkv
