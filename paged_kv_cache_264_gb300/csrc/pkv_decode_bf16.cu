// pkv_decode_bf16.cu -- decode kernels for bf16 pools (instantiations and dispatch), and
// the partition-merge kernel.
#include "pkv_decode.cuh"

namespace pkv {

// Warps per CTA and ring stages per warp for bf16 pools.  A stage holds one K and one V
// tile: 8 KiB at head_dim 128, 4 KiB at head_dim 64.
constexpr int kNwBf16 = 4;
constexpr int kStagesBf16D128 = 3;
constexpr int kStagesBf16D64 = 4;

template <int D, int S>
static cudaError_t dispatch_cols(const DecodeParams& p, int cols, cudaStream_t stream) {
  switch (cols) {
    case 1: return launch_decode_variant<KvType::kBf16, D, 1, kNwBf16, S>(p, stream);
    case 2: return launch_decode_variant<KvType::kBf16, D, 2, kNwBf16, S>(p, stream);
    case 4: return launch_decode_variant<KvType::kBf16, D, 4, kNwBf16, S>(p, stream);
    case 8: return launch_decode_variant<KvType::kBf16, D, 8, kNwBf16, S>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_bf16(const DecodeParams& p, int cols, cudaStream_t stream) {
  if (p.head_dim == 128) return dispatch_cols<128, kStagesBf16D128>(p, cols, stream);
  if (p.head_dim == 64) return dispatch_cols<64, kStagesBf16D64>(p, cols, stream);
  return cudaErrorInvalidValue;
}

int ctas_per_sm_bf16(int head_dim, int cols) {
  if (head_dim == 128) {
    switch (cols) {
      case 1: return ctas_per_sm_variant<KvType::kBf16, 128, 1, kNwBf16, kStagesBf16D128>();
      case 2: return ctas_per_sm_variant<KvType::kBf16, 128, 2, kNwBf16, kStagesBf16D128>();
      case 4: return ctas_per_sm_variant<KvType::kBf16, 128, 4, kNwBf16, kStagesBf16D128>();
      case 8: return ctas_per_sm_variant<KvType::kBf16, 128, 8, kNwBf16, kStagesBf16D128>();
    }
  } else if (head_dim == 64) {
    switch (cols) {
      case 1: return ctas_per_sm_variant<KvType::kBf16, 64, 1, kNwBf16, kStagesBf16D64>();
      case 2: return ctas_per_sm_variant<KvType::kBf16, 64, 2, kNwBf16, kStagesBf16D64>();
      case 4: return ctas_per_sm_variant<KvType::kBf16, 64, 4, kNwBf16, kStagesBf16D64>();
      case 8: return ctas_per_sm_variant<KvType::kBf16, 64, 8, kNwBf16, kStagesBf16D64>();
    }
  }
  return 0;
}

cudaError_t launch_lse_reduce(const DecodeParams& p, cudaStream_t stream) {
  const int64_t pairs = int64_t(p.num_seqs) * p.num_queries * p.num_q_heads;
  const int64_t grid = (pairs + 3) / 4;
  if (grid <= 0) return cudaSuccess;
  if (p.head_dim == 128)
    return launch_pdl(lse_reduce_kernel<128>, dim3(static_cast<unsigned>(grid)), dim3(128), 0, stream, p);
  if (p.head_dim == 64)
    return launch_pdl(lse_reduce_kernel<64>, dim3(static_cast<unsigned>(grid)), dim3(128), 0, stream, p);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
