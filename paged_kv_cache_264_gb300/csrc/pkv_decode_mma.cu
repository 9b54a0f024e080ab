// pkv_decode_mma.cu -- tensor-core decode variants (instantiations and dispatch).
#include "pkv_decode_mma.cuh"

namespace pkv {

// Warps per CTA, and the ring depths built per pool type.  A stage holds one K and one V
// tile: 8 KiB (bf16, head_dim 128) or 4 KiB (bf16 64, INT8 128).
constexpr int kNwMma = 4;

bool mma_supported(KvType kv, int head_dim, int group) {
  if (group != 2 && group != 4 && group != 8) return false;
  if (kv == KvType::kBf16) return head_dim == 128 || head_dim == 64;
  return head_dim == 128;
}

int mma_default_stages(KvType kv, int head_dim) {
  // Measured on GB300: shallow rings fit 3-4 CTAs per SM, which hides the per-item
  // prologue and merge better than deeper rings with 2 CTAs per SM.
  return (kv == KvType::kBf16 && head_dim == 128) ? 2 : 3;
}

bool mma_stages_built(KvType kv, int head_dim, int stages) {
  if (kv == KvType::kBf16 && head_dim == 128) return stages == 2 || stages == 3;
  return stages == 3 || stages == 6;
}

template <KvType KV, int D, int S>
static cudaError_t dispatch_g(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int group, cudaStream_t stream) {
  switch (group) {
    case 2: return launch_mma_variant<KV, D, 2, kNwMma, S>(p, tk, tv, stream);
    case 4: return launch_mma_variant<KV, D, 4, kNwMma, S>(p, tk, tv, stream);
    case 8: return launch_mma_variant<KV, D, 8, kNwMma, S>(p, tk, tv, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap* tk, const CUtensorMap* tv,
                              KvType kv, int group, int stages, cudaStream_t stream) {
  if (!mma_supported(kv, p.head_dim, group) || !mma_stages_built(kv, p.head_dim, stages))
    return cudaErrorInvalidValue;
  if (kv == KvType::kInt8)
    return stages == 3 ? dispatch_g<KvType::kInt8, 128, 3>(p, *tk, *tv, group, stream)
                       : dispatch_g<KvType::kInt8, 128, 6>(p, *tk, *tv, group, stream);
  if (p.head_dim == 128)
    return stages == 2 ? dispatch_g<KvType::kBf16, 128, 2>(p, *tk, *tv, group, stream)
                       : dispatch_g<KvType::kBf16, 128, 3>(p, *tk, *tv, group, stream);
  return stages == 3 ? dispatch_g<KvType::kBf16, 64, 3>(p, *tk, *tv, group, stream)
                     : dispatch_g<KvType::kBf16, 64, 6>(p, *tk, *tv, group, stream);
}

template <KvType KV, int D, int S>
static int occupancy(int group) {
  switch (group) {
    case 2: return mma_ctas_per_sm_variant<KV, D, 2, kNwMma, S>();
    case 4: return mma_ctas_per_sm_variant<KV, D, 4, kNwMma, S>();
    case 8: return mma_ctas_per_sm_variant<KV, D, 8, kNwMma, S>();
  }
  return 0;
}

int mma_ctas_per_sm(KvType kv, int head_dim, int group, int stages) {
  if (!mma_supported(kv, head_dim, group) || !mma_stages_built(kv, head_dim, stages)) return 0;
  static int cache[3][2][9] = {};  // [pool type][stage variant][group]
  const int ti = kv == KvType::kInt8 ? 2 : (head_dim == 128 ? 0 : 1);
  const int si = stages == mma_default_stages(kv, head_dim) ? 0 : 1;
  int& slot = cache[ti][si][group];
  if (slot) return slot;
  int n = 0;
  if (kv == KvType::kInt8)
    n = stages == 3 ? occupancy<KvType::kInt8, 128, 3>(group) : occupancy<KvType::kInt8, 128, 6>(group);
  else if (head_dim == 128)
    n = stages == 2 ? occupancy<KvType::kBf16, 128, 2>(group) : occupancy<KvType::kBf16, 128, 3>(group);
  else
    n = stages == 3 ? occupancy<KvType::kBf16, 64, 3>(group) : occupancy<KvType::kBf16, 64, 6>(group);
  slot = n;
  return n;
}

}  // namespace pkv
