// pkv_decode_mma.cu -- tensor-core decode: which variants exist and which one a call uses.
// The instantiations live in pkv_decode_mma_{bf16,int8,fp8}.cu (compiled in parallel).
#include <atomic>

#include "pkv_decode_mma.cuh"

namespace pkv {

bool mma_supported(KvType kv, int head_dim, int cols) {
  if (cols != 2 && cols != 4 && cols != 8 && cols != 16) return false;
  return head_dim == 128 || head_dim == 64;  // bf16, INT8 and FP8 pools alike
}

static int shapes_of(KvType kv, int head_dim, const RingShape** out) {
  if (kv != KvType::kBf16 && head_dim == 64) {
    *out = kShapesQuantD64;
    return int(sizeof(kShapesQuantD64) / sizeof(kShapesQuantD64[0]));
  }
  if (kv != KvType::kBf16) {
    *out = kShapesQuant;
    return int(sizeof(kShapesQuant) / sizeof(kShapesQuant[0]));
  }
  if (head_dim == 128) {
    *out = kShapesBf16D128;
    return int(sizeof(kShapesBf16D128) / sizeof(kShapesBf16D128[0]));
  }
  *out = kShapesBf16D64;
  return int(sizeof(kShapesBf16D64) / sizeof(kShapesBf16D64[0]));
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

cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap* tk, const CUtensorMap* tv,
                              KvType kv, int cols, int shape, cudaStream_t stream) {
  if (!mma_supported(kv, p.head_dim, cols)) return cudaErrorInvalidValue;
  const bool gen = mma_needs_general(p.num_queries, p.window, cols);
  if (kv != KvType::kBf16 && p.head_dim == 64) return launch_mma_quant_d64(kv, p, *tk, *tv, cols, shape, gen, stream);
  if (kv == KvType::kInt8) return launch_mma_int8(p, *tk, *tv, cols, shape, gen, stream);
  if (kv == KvType::kFp8) return launch_mma_fp8(p, *tk, *tv, cols, shape, gen, stream);
  return launch_mma_bf16(p, *tk, *tv, cols, shape, gen, stream);
}

int mma_ctas_per_sm(KvType kv, int head_dim, int cols, int shape, bool gen) {
  const RingShape* sh;
  if (!mma_supported(kv, head_dim, cols) || shape < 0 || shape >= shapes_of(kv, head_dim, &sh)) return 0;
  // [pool type][head_dim 128 | 64][shape][column slots][gen]; 0 = not yet queried (or not
  // built).  Threads may fill an entry concurrently; they store the same value.
  static std::atomic<int> cache[3][2][4][17][2];
  const int ki = static_cast<int>(kv), di = head_dim == 128 ? 0 : 1;
  std::atomic<int>& slot = cache[ki][di][shape][cols][gen ? 1 : 0];
  int n = slot.load(std::memory_order_relaxed);
  if (n) return n;
  n = kv != KvType::kBf16 && head_dim == 64 ? occupancy_mma_quant_d64(kv, cols, shape, gen)
      : kv == KvType::kInt8                 ? occupancy_mma_int8(cols, shape, gen)
      : kv == KvType::kFp8                  ? occupancy_mma_fp8(cols, shape, gen)
                                            : occupancy_mma_bf16(head_dim, cols, shape, gen);
  slot.store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace pkv
