// pkv_decode_mma.cu -- tensor-core decode variants (instantiations and dispatch).
#include "pkv_decode_mma.cuh"

namespace pkv {

// Warps per CTA and the built ring shapes: (stages S, blocks per stage BPS).  A block's K
// and V tiles take 8 KiB (bf16, head_dim 128) or 4 KiB (bf16 64, INT8 128).  The first
// shape listed for a pool type is its default.
constexpr int kNwMma = 4;

struct RingShape {
  int stages, bps;
};

static const RingShape kShapesBf16D128[] = {{2, 1}, {3, 1}};
static const RingShape kShapesBf16D64[] = {{3, 1}, {2, 2}};
static const RingShape kShapesInt8[] = {{3, 1}, {2, 2}, {3, 2}};  // INT8 and FP8

bool mma_supported(KvType kv, int head_dim, int cols) {
  if (cols != 2 && cols != 4 && cols != 8 && cols != 16) return false;
  if (kv == KvType::kBf16) return head_dim == 128 || head_dim == 64;
  return head_dim == 128;  // INT8, FP8
}

static int shapes_of(KvType kv, int head_dim, const RingShape** out) {
  if (kv != KvType::kBf16) { *out = kShapesInt8; return 3; }
  if (head_dim == 128) { *out = kShapesBf16D128; return 2; }
  *out = kShapesBf16D64;
  return 2;
}

// Index of the ring shape for (stages, bps), 0 meaning "default" for either; -1 if not built.
int mma_ring_shape(KvType kv, int head_dim, int stages, int bps) {
  const RingShape* sh;
  const int n = shapes_of(kv, head_dim, &sh);
  if (stages == 0 && bps == 0) return 0;
  for (int i = 0; i < n; ++i)
    if ((stages == 0 || sh[i].stages == stages) && (bps == 0 || sh[i].bps == bps)) return i;
  return -1;
}

template <KvType KV, int D, int S, int BPS>
static cudaError_t dispatch_g(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int cols, cudaStream_t stream) {
  switch (cols) {
    case 2: return launch_mma_variant<KV, D, 2, kNwMma, S, BPS>(p, tk, tv, stream);
    case 4: return launch_mma_variant<KV, D, 4, kNwMma, S, BPS>(p, tk, tv, stream);
    case 8: return launch_mma_variant<KV, D, 8, kNwMma, S, BPS>(p, tk, tv, stream);
    case 16: return launch_mma_variant<KV, D, 16, kNwMma, S, BPS>(p, tk, tv, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap* tk, const CUtensorMap* tv,
                              KvType kv, int cols, int shape, cudaStream_t stream) {
  if (!mma_supported(kv, p.head_dim, cols)) return cudaErrorInvalidValue;
  if (kv == KvType::kInt8) {
    switch (shape) {
      case 0: return dispatch_g<KvType::kInt8, 128, 3, 1>(p, *tk, *tv, cols, stream);
      case 1: return dispatch_g<KvType::kInt8, 128, 2, 2>(p, *tk, *tv, cols, stream);
      case 2: return dispatch_g<KvType::kInt8, 128, 3, 2>(p, *tk, *tv, cols, stream);
    }
  } else if (kv == KvType::kFp8) {
    switch (shape) {
      case 0: return dispatch_g<KvType::kFp8, 128, 3, 1>(p, *tk, *tv, cols, stream);
      case 1: return dispatch_g<KvType::kFp8, 128, 2, 2>(p, *tk, *tv, cols, stream);
      case 2: return dispatch_g<KvType::kFp8, 128, 3, 2>(p, *tk, *tv, cols, stream);
    }
  } else if (p.head_dim == 128) {
    switch (shape) {
      case 0: return dispatch_g<KvType::kBf16, 128, 2, 1>(p, *tk, *tv, cols, stream);
      case 1: return dispatch_g<KvType::kBf16, 128, 3, 1>(p, *tk, *tv, cols, stream);
    }
  } else {
    switch (shape) {
      case 0: return dispatch_g<KvType::kBf16, 64, 3, 1>(p, *tk, *tv, cols, stream);
      case 1: return dispatch_g<KvType::kBf16, 64, 2, 2>(p, *tk, *tv, cols, stream);
    }
  }
  return cudaErrorInvalidValue;
}

template <KvType KV, int D, int S, int BPS>
static int occupancy(int cols) {
  switch (cols) {
    case 2: return mma_ctas_per_sm_variant<KV, D, 2, kNwMma, S, BPS>();
    case 4: return mma_ctas_per_sm_variant<KV, D, 4, kNwMma, S, BPS>();
    case 8: return mma_ctas_per_sm_variant<KV, D, 8, kNwMma, S, BPS>();
    case 16: return mma_ctas_per_sm_variant<KV, D, 16, kNwMma, S, BPS>();
  }
  return 0;
}

int mma_ctas_per_sm(KvType kv, int head_dim, int cols, int shape) {
  if (!mma_supported(kv, head_dim, cols) || shape < 0 || shape > 2) return 0;
  static int cache[4][3][17] = {};  // [pool type][shape][column slots]
  const int ti = kv == KvType::kFp8 ? 3 : kv == KvType::kInt8 ? 2 : (head_dim == 128 ? 0 : 1);
  int& slot = cache[ti][shape][cols];
  if (slot) return slot;
  int n = 0;
  if (kv == KvType::kInt8) {
    n = shape == 0 ? occupancy<KvType::kInt8, 128, 3, 1>(cols)
      : shape == 1 ? occupancy<KvType::kInt8, 128, 2, 2>(cols)
                   : occupancy<KvType::kInt8, 128, 3, 2>(cols);
  } else if (kv == KvType::kFp8) {
    n = shape == 0 ? occupancy<KvType::kFp8, 128, 3, 1>(cols)
      : shape == 1 ? occupancy<KvType::kFp8, 128, 2, 2>(cols)
                   : occupancy<KvType::kFp8, 128, 3, 2>(cols);
  } else if (head_dim == 128) {
    n = shape == 0 ? occupancy<KvType::kBf16, 128, 2, 1>(cols) : occupancy<KvType::kBf16, 128, 3, 1>(cols);
  } else {
    n = shape == 0 ? occupancy<KvType::kBf16, 64, 3, 1>(cols) : occupancy<KvType::kBf16, 64, 2, 2>(cols);
  }
  slot = n;
  return n;
}

}  // namespace pkv
