// pkv_cache.cu -- writing new tokens' K/V into their pool slots ("reshape and cache").
//
// Each new token's key and value rows go to the slot its page table gives it
// ("Lesson 4: Model deployment and inference acceleration", section 4.2; only the new
// token's K/V are appended).  slot = slot_mapping[t]; block = slot / 16;
// offset = slot % 16; cache[block][head][offset][:] = row.
//
// bf16 pool: a straight 16-byte-vector copy, one thread per 16 bytes of a row.
// INT8 pool ("Lesson 4", section 5.3): one warp per (token, kv head), doing K and V:
// s = max|x| / 127 with IEEE fp32 division, code = round-half-even(x / s), clamped to
// [-127, 127]; the codes of one row are stored as one coalesced 32-lane write, and the
// scale next to them in the [num_blocks, Hkv, 16] scale array.
// FP8 pool (the same section names FP8 KV caches): the same with s = max|x| / 448 and the
// code the nearest E4M3 of x / s (ties to even, saturating at +-448).
#include <cuda_bf16.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kCacheThreads = 256;

__global__ void __launch_bounds__(kCacheThreads)
    cache_bf16_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                      const int32_t* __restrict__ slot_mapping, uint4* __restrict__ k_cache,
                      uint4* __restrict__ v_cache, uint32_t* err, int64_t num_tokens,
                      int64_t num_slots, int kv_heads, int chunks_per_row) {
  // chunks_per_row = head_dim * 2 / 16 sixteen-byte vectors per (token, head) row.
  griddep_wait();  // key/value/slots may come from the previous kernel in the stream
  griddep_launch_dependents();
  const int64_t total = num_tokens * kv_heads * chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t row = i / chunks_per_row;  // token * kv_heads + head
    const int c = static_cast<int>(i - row * chunks_per_row);
    const int64_t t = row / kv_heads;
    const int h = static_cast<int>(row - t * kv_heads);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0 && h == 0) set_error(err, kErrSlot);
      continue;
    }
    const int64_t block = slot / kBlockSize;
    const int64_t off = slot - block * kBlockSize;
    const int64_t dst = ((block * kv_heads + h) * kBlockSize + off) * chunks_per_row + c;
    k_cache[dst] = __ldg(key + i);
    v_cache[dst] = __ldg(value + i);
  }
}

// Quantise the D values of one row held by a warp (DPV = D / 32 per lane) and return the
// lane's packed codes (INT8, or E4M3 when kFp8).  *scale receives s on every lane.
template <int DPV, bool kFp8>
__device__ __forceinline__ uint32_t quantise_row(const float (&x)[DPV], float* scale) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < DPV; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, kFp8 ? 448.0f : 127.0f);
  *scale = s;
  if (amax == 0.0f) return 0u;
  if constexpr (kFp8) {
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < DPV; i += 2)
      packed |= e4m3x2_from_f32(__fdiv_rn(x[i], s), __fdiv_rn(x[i + 1], s)) << (8 * i);
    return packed;
  } else {
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < DPV; ++i) {
      int code = __float2int_rn(__fdiv_rn(x[i], s));
      code = min(127, max(-127, code));
      packed |= (static_cast<uint32_t>(code) & 0xffu) << (8 * i);
    }
    return packed;
  }
}

template <int D, bool kFp8>
__global__ void __launch_bounds__(kCacheThreads)
    cache_quant_kernel(const __nv_bfloat16* __restrict__ key,
                      const __nv_bfloat16* __restrict__ value,
                      const int32_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_cache,
                      uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
                      float* __restrict__ v_scale, uint32_t* err, int64_t num_tokens,
                      int64_t num_slots, int kv_heads) {
  constexpr int DPV = D / 32;  // values per lane: 4 (D=128) or 2 (D=64)
  const int lane = threadIdx.x & 31;
  griddep_wait();  // key/value/slots may come from the previous kernel in the stream
  griddep_launch_dependents();
  const int64_t rows = num_tokens * kv_heads;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    const int64_t t = row / kv_heads;
    const int h = static_cast<int>(row - t * kv_heads);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0 && h == 0) set_error(err, kErrSlot);
      continue;
    }
    const int64_t block = slot / kBlockSize;
    const int64_t off = slot - block * kBlockSize;
    const int64_t srow = (block * kv_heads + h) * kBlockSize + off;

    float kx[DPV], vx[DPV];
    const int64_t src = row * D + lane * DPV;
    if constexpr (DPV == 4) {
      const uint2 kw = __ldg(reinterpret_cast<const uint2*>(key + src));
      const uint2 vw = __ldg(reinterpret_cast<const uint2*>(value + src));
      kx[0] = bf16lo(kw.x); kx[1] = bf16hi(kw.x); kx[2] = bf16lo(kw.y); kx[3] = bf16hi(kw.y);
      vx[0] = bf16lo(vw.x); vx[1] = bf16hi(vw.x); vx[2] = bf16lo(vw.y); vx[3] = bf16hi(vw.y);
    } else {
      const uint32_t kw = __ldg(reinterpret_cast<const uint32_t*>(key + src));
      const uint32_t vw = __ldg(reinterpret_cast<const uint32_t*>(value + src));
      kx[0] = bf16lo(kw); kx[1] = bf16hi(kw);
      vx[0] = bf16lo(vw); vx[1] = bf16hi(vw);
    }
    float ks, vs;
    const uint32_t kq = quantise_row<DPV, kFp8>(kx, &ks);
    const uint32_t vq = quantise_row<DPV, kFp8>(vx, &vs);
    const int64_t dst = srow * D + lane * DPV;
    if constexpr (DPV == 4) {
      *reinterpret_cast<uint32_t*>(k_cache + dst) = kq;
      *reinterpret_cast<uint32_t*>(v_cache + dst) = vq;
    } else {
      *reinterpret_cast<uint16_t*>(k_cache + dst) = static_cast<uint16_t>(kq);
      *reinterpret_cast<uint16_t*>(v_cache + dst) = static_cast<uint16_t>(vq);
    }
    if (lane == 0) {
      k_scale[srow] = ks;
      v_scale[srow] = vs;
    }
  }
}

// Copy whole blocks (every kv head's K and V rows, and INT8/FP8 scales) from src to dst:
// the copy-on-write step of block sharing.  `pairs` is int32 [n][2] = (src, dst).  One CTA
// per (pair, 16-byte chunk range); out-of-range ids are skipped and flagged.
__global__ void __launch_bounds__(kCacheThreads)
    copy_blocks_kernel(const int32_t* __restrict__ pairs, int n, uint4* __restrict__ k_cache,
                       uint4* __restrict__ v_cache, uint4* __restrict__ k_scale,
                       uint4* __restrict__ v_scale, uint32_t* err, int64_t num_blocks,
                       int64_t chunks_per_block, int64_t scale_chunks_per_block) {
  griddep_wait();  // the pairs and the source blocks may come from earlier kernels
  griddep_launch_dependents();
  const int pi = blockIdx.y;
  if (pi >= n) return;
  const int64_t src = __ldg(pairs + 2 * pi), dst = __ldg(pairs + 2 * pi + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, kErrBlockId);
    return;
  }
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks_per_block;
       c += int64_t(gridDim.x) * blockDim.x) {
    k_cache[dst * chunks_per_block + c] = k_cache[src * chunks_per_block + c];
    v_cache[dst * chunks_per_block + c] = v_cache[src * chunks_per_block + c];
  }
  if (k_scale) {
    for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < scale_chunks_per_block;
         c += int64_t(gridDim.x) * blockDim.x) {
      k_scale[dst * scale_chunks_per_block + c] = k_scale[src * scale_chunks_per_block + c];
      v_scale[dst * scale_chunks_per_block + c] = v_scale[src * scale_chunks_per_block + c];
    }
  }
}

int grid_for(int64_t work_items, int per_block) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  return static_cast<int>(need < cap ? (need < 1 ? 1 : need) : cap);
}

}  // namespace

cudaError_t launch_cache_bf16(const CacheParams& p, cudaStream_t stream) {
  const int chunks = p.head_dim * 2 / 16;
  const int64_t total = p.num_tokens * p.kv_heads * chunks;
  return launch_pdl(cache_bf16_kernel, dim3(grid_for(total, kCacheThreads)), dim3(kCacheThreads), 0,
                    stream, static_cast<const uint4*>(p.key), static_cast<const uint4*>(p.value),
                    p.slot_mapping, static_cast<uint4*>(p.k_cache), static_cast<uint4*>(p.v_cache),
                    p.err, p.num_tokens, p.num_blocks * kBlockSize, p.kv_heads, chunks);
}

template <bool kFp8>
static cudaError_t launch_cache_quant(const CacheParams& p, cudaStream_t stream) {
  const int64_t rows = p.num_tokens * p.kv_heads;
  const int grid = grid_for(rows, kCacheThreads / 32);
  const auto* key = static_cast<const __nv_bfloat16*>(p.key);
  const auto* value = static_cast<const __nv_bfloat16*>(p.value);
  auto* kc = static_cast<uint8_t*>(p.k_cache);
  auto* vc = static_cast<uint8_t*>(p.v_cache);
  if (p.head_dim == 128)
    return launch_pdl(cache_quant_kernel<128, kFp8>, dim3(grid), dim3(kCacheThreads), 0, stream, key,
                      value, p.slot_mapping, kc, vc, p.k_scale, p.v_scale, p.err, p.num_tokens,
                      p.num_blocks * kBlockSize, p.kv_heads);
  if (p.head_dim == 64)
    return launch_pdl(cache_quant_kernel<64, kFp8>, dim3(grid), dim3(kCacheThreads), 0, stream, key,
                      value, p.slot_mapping, kc, vc, p.k_scale, p.v_scale, p.err, p.num_tokens,
                      p.num_blocks * kBlockSize, p.kv_heads);
  return cudaErrorInvalidValue;
}

cudaError_t launch_copy_blocks(const CacheParams& p, const int32_t* pairs, int n, int elem_bytes,
                               cudaStream_t stream) {
  const int64_t chunks = int64_t(p.kv_heads) * kBlockSize * p.head_dim * elem_bytes / 16;
  const int64_t scale_chunks = p.k_scale ? int64_t(p.kv_heads) * kBlockSize * 4 / 16 : 0;
  const int xblocks = static_cast<int>((chunks + kCacheThreads - 1) / kCacheThreads);
  if (n > 65535) return cudaErrorInvalidValue;
  return launch_pdl(copy_blocks_kernel, dim3(xblocks, n), dim3(kCacheThreads), 0, stream, pairs, n,
                    static_cast<uint4*>(p.k_cache), static_cast<uint4*>(p.v_cache),
                    reinterpret_cast<uint4*>(p.k_scale), reinterpret_cast<uint4*>(p.v_scale), p.err,
                    p.num_blocks, chunks, scale_chunks);
}

cudaError_t launch_cache_int8(const CacheParams& p, cudaStream_t stream) {
  return launch_cache_quant<false>(p, stream);
}

cudaError_t launch_cache_fp8(const CacheParams& p, cudaStream_t stream) {
  return launch_cache_quant<true>(p, stream);
}

}  // namespace pkv
