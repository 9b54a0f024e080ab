// pkv_decode_mma.cuh -- PagedAttention decode on the tensor cores (mma.sync) for tiles of
// 2, 4, 8 or 16 query columns per kv head (the GQA group's heads times the query tokens of
// a multi-query call; a single column, MHA decode, uses 2), head_dim 128 or 64, bf16,
// INT8 or FP8 pools.
//
// Same work decomposition and result as paged_decode_kernel (pkv_decode.cuh): one CTA
// per (sequence, kv head, context partition), NW warps taking the item's blocks in turn,
// a per-warp ring of S shared-memory stages, an online softmax and a log-sum-exp merge.
// What changes is how a 16-token block is consumed:
//
//  * Tiles arrive by TMA tensor copies (cp.async.bulk.tensor.2d) through a tensor map of
//    the pool viewed as rows of head_dim elements (two 64-byte token rows to a row for
//    INT8/FP8 at head_dim 64), in 128-byte boxes with the 128-byte swizzle, so that the
//    shared-memory reads below are free of bank conflicts.
//  * Logits for all query columns come from m16n8k16 MMAs with fp32 accumulation:
//    S[16 tokens x 8 columns] = K[16 x d] q^T[d x 8] per n-tile of 8 columns (columns past
//    the active ones are zero).  Each K fragment feeds every n-tile.  A column is one
//    (query token, head of the group) pair; with several query tokens or a sliding window
//    (the kGen variant) each column has its own causal cut and window, applied when the
//    logits are masked.
//  * The probabilities stay in registers: the accumulator fragment of S, packed to 16-bit
//    pairs and transposed with movmatrix, is exactly the B operand of the PV product
//    O^T[d x 8] += V^T[d x 16] P[16 x 8], whose A operand is V read transposed by ldmatrix.
//    The row (dims) of O^T that a lane holds and the column of its softmax state
//    coincide, so rescaling needs no data movement.  The running max is lazy: it moves
//    only when a logit passes it by more than kMaxSlack, so most stages need neither the
//    cross-lane max nor a rescale.  For bf16 pools P enters the product as bf16,
//    and the softmax sum adds those same rounded weights.
//  * INT8: codes become fp16 values 1152 + code exactly (see f16x2_biased) and both
//    products run in fp16; the constant 1152 is taken out afterwards: from the logits as
//    1152 * sum_d q_d per column, and from O^T as 1152 times the running sum of P per
//    column.  q is scaled by a power of two into fp16 range (exact for bf16 values), the
//    K scale multiplies the fp32 logits, and the V scale is folded into P together with a
//    power-of-two block exponent that keeps P in [0, 2): O^T is kept in units of 2^E and E
//    only grows, like the running max, so the rescale stays rare.  FP8 (E4M3) pools take
//    the same path with the hardware E4M3 -> fp16 conversion and no offset.  Codes come
//    through ldmatrix on the tile seen as byte pairs: plain for K (four dims of a token per
//    register, the dims of a k-step permuted alike in K and q) and transposed for V (two
//    tokens' codes of two dims per register).
//  * Without the general masks the block loop is unrolled over the S ring stages, so that
//    a stage's shared-memory addresses are per-lane registers plus immediates.
#pragma once

#include <limits.h>

#include "pkv_decode.cuh"

namespace pkv {

template <KvType KV, int D, int NC, int NW, int S, int BPS>
struct MmaCfg {
  static constexpr int kNT = NC > 8 ? NC / 8 : 1;     // n-tiles of 8 query columns
  static constexpr int kEsz = KvTraits<KV>::kElemBytes;
  static constexpr bool kQuant = KvTraits<KV>::kQuant;
  static constexpr bool kFp8 = KV == KvType::kFp8;     // E4M3 codes (else INT8 when kQuant)
  static constexpr int kRowBytes = D * kEsz;           // one token row of one tile
  // 64-byte token rows (INT8/FP8 at head_dim 64) travel two to a 128-byte box row, so that
  // every tile keeps the 128-byte swizzle: token t is box row t / 2, bytes 64 (t % 2) on.
  static constexpr bool kPairRows = kRowBytes == 64;
  static constexpr int kBoxCols = 128 / kEsz;          // elements in a 128-byte box row
  static constexpr int kBoxRows = kPairRows ? kBlockSize / 2 : kBlockSize;
  static constexpr int kBoxes = kPairRows ? 1 : kRowBytes / 128;  // boxes per tile
  static constexpr int kBoxBytes = kBoxRows * 128;     // 2 KiB (1 KiB for pair rows), 1 KiB aligned
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * BPS * kTileBytes;   // BPS K tiles, then BPS V tiles
  static constexpr int kScaleStage = kQuant ? 2 * BPS * kBlockSize * 4 : 0;  // K then V scales
  static constexpr int kKSteps = D / 16;
  static constexpr int kMTiles = D / 16;
  static constexpr int kThreads = NW * 32;
  static constexpr size_t kRingBytes = size_t(NW) * S * kStageBytes;
  static constexpr size_t kScaleOff = kRingBytes;
  static constexpr size_t kBarOff = align_up(kScaleOff + size_t(NW) * S * kScaleStage, 16);
  static constexpr size_t kTableOff = kBarOff + size_t(NW) * S * 8;
  static size_t smem_bytes(int partition_blocks, int sched_seqs) {
    return 1024 /* alignment slack */ + kTableOff + size_t(partition_cap(partition_blocks)) * 4 +
           sched_smem_bytes(sched_seqs, kThreads);
  }

  static_assert(kRowBytes % 128 == 0 || kPairRows, "rows must be whole 128-byte swizzle spans or pairs");
  static_assert(!kQuant || D == 128 || D == 64, "INT8/FP8 tensor-core path is built for head_dim 64 and 128");
  static_assert(!kPairRows || kQuant, "pair rows are the quantised head_dim 64 layout");
  static_assert(NC == 2 || NC == 4 || NC == 8 || NC == 16, "2, 4, 8 or 16 query columns");
  static_assert(BPS == 1 || BPS == 2, "one or two blocks per ring stage");
  static_assert(size_t(NC) * record_stride(D) * 4 <= size_t(S) * kStageBytes, "merge record fits the ring");
};

// Warps per CTA and the built ring shapes: (stages S, blocks per stage BPS).  A block's K
// and V tiles take 8 KiB (bf16, head_dim 128), 4 KiB (bf16 64, INT8/FP8 128) or 2 KiB
// (INT8/FP8 64).  The first shape listed for a pool type is its default.
constexpr int kNwMma = 4;
struct RingShape {
  int stages, bps;
};
constexpr RingShape kShapesBf16D128[] = {{2, 1}, {3, 1}};
constexpr RingShape kShapesBf16D64[] = {{3, 1}, {2, 2}};
// INT8 and FP8.  Measured on GB300 (int8_cb / fp8_cb, microseconds per call, median of 3
// interleaved runs): 3x1 168.2 / 162.0, 2x1 169.6 / 162.1, 2x2 172.1 / -, 3x2 ~250 / ~246.
// Forcing more CTAs per SM through launch bounds (fewer registers) never helped.
constexpr RingShape kShapesQuant[] = {{3, 1}, {2, 1}, {2, 2}, {3, 2}};
// INT8 and FP8 at head_dim 64 (2 KiB per block).  Measured on GB300 (int8_cb lengths at
// head_dim 64, microseconds per call): 2x2 122.8, 3x1 138.2 (the CUDA-core kernel: 246.0).
constexpr RingShape kShapesQuantD64[] = {{2, 2}, {3, 1}};

// Launch / occupancy of one pool type's variants (defined in pkv_decode_mma_<type>.cu):
// cols = column slots (2, 4, 8, 16), shape = index into the type's shape list, gen = kGen.
cudaError_t launch_mma_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int cols, int shape, bool gen, cudaStream_t stream);
cudaError_t launch_mma_int8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int cols, int shape, bool gen, cudaStream_t stream);
cudaError_t launch_mma_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           int cols, int shape, bool gen, cudaStream_t stream);
int occupancy_mma_bf16(int head_dim, int cols, int shape, bool gen);
int occupancy_mma_int8(int cols, int shape, bool gen);
int occupancy_mma_fp8(int cols, int shape, bool gen);
// INT8 / FP8 pools at head_dim 64 (pkv_decode_mma_quant_d64.cu).
cudaError_t launch_mma_quant_d64(KvType kv, const DecodeParams& p, const CUtensorMap& tk,
                                 const CUtensorMap& tv, int cols, int shape, bool gen, cudaStream_t stream);
int occupancy_mma_quant_d64(KvType kv, int cols, int shape, bool gen);

// Byte offset of 16-byte chunk `c` of token row `t` in a tile whose 128-byte boxes were
// written with the 128-byte swizzle (chunk index xor row index mod 8).
__device__ __forceinline__ int swz_off(int t, int c) {
  return (c >> 3) * 2048 + t * 128 + (((c & 7) ^ (t & 7)) << 4);
}

// The same for a tile of 64-byte token rows held two to a 128-byte box row: token t is box
// row t / 2, its chunk c (0..3) is chunk 4 (t % 2) + c of that row before the swizzle.  The
// 8 tokens of an ldmatrix matrix then cover the 8 chunk positions of 4 box rows, so the
// reads stay free of bank conflicts.
__device__ __forceinline__ int swz_off_pair(int t, int c) {
  const int r = t >> 1;
  return r * 128 + (((((t & 1) << 2) | c) ^ (r & 7)) << 4);
}

// A ring stage known at compile time (the stage of an unrolled loop body), a loop over
// 0..N-1 of them, and a stage known only at run time.
template <int N>
struct IntC {
  static constexpr int value = N;
};
struct StageRt {
  int value;
};
template <int N, int I = 0, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(IntC<I>{});
    static_for<N, I + 1>(f);
  }
}

// kGen: the general masks (causal cuts of several query tokens, a sliding window).  Without
// it a column sees every context token, the only mask is the context end, and the kernel
// carries none of that arithmetic (the INT8 and FP8 paths are instruction-bound).
// INT8/FP8 tiles of up to 8 columns with one block per stage are held to 128 registers
// (4 CTAs per SM), the compiler's own choice for most of them, which the 8-column tiles
// otherwise exceed (168); every other variant keeps the compiler's choice.
template <KvType KV, int D, int NC, int NW, int S, int BPS, bool kGen>
__global__ void __launch_bounds__(NW * 32, (KvTraits<KV>::kQuant && NC <= 8 && BPS == 1) ? 4 : 0)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using C = MmaCfg<KV, D, NC, NW, S, BPS>;
  constexpr int NT = C::kNT;
  constexpr uint32_t kFull = 0xffffffffu;
  griddep_wait();  // inputs may come from the previous kernel in the stream
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2;  // fragment row group
  const int gj = lane & 3;   // fragment column pair

  int* tbl = reinterpret_cast<int*>(smem + C::kTableOff);
  const SchedSmem ss = sched_smem(smem + C::kTableOff + size_t(partition_cap(p.partition_blocks)) * 4,
                                  p.persistent ? p.num_seqs : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff) + warp * S;
  unsigned char* ring = smem + size_t(warp) * S * C::kStageBytes;
  float* scl = reinterpret_cast<float*>(smem + C::kScaleOff) + warp * S * (C::kScaleStage / 4);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(bars + s, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tensor_map(&tmap_k);
    prefetch_tensor_map(&tmap_v);
  }
  const int P = p.partition_blocks;
  // Blocks this warp has consumed over all its items: stage and phase counter.  Without
  // the general masks it is a multiple of S whenever an item starts, so that the stage of
  // each unrolled step of the block loop is a compile-time constant and every
  // shared-memory address below is a per-lane register plus an immediate.
  uint32_t kb = 0;

  // ldmatrix row assignment: lane gives the row address of matrix lane / 8.
  const int mi = lane >> 3;
  // K (A of S) and quantised V: matrices (token rows 0-7 | 8-15) x (16-byte chunk lo | hi).
  const int tok_k = (lane & 7) + (mi & 1) * 8;
  const int ck = mi >> 1;
  // bf16 V^T (A of O^T, transposed load): matrices (chunk lo | hi) x (token rows 0-7 | 8-15).
  const int tok_v = (lane & 7) + (mi >> 1) * 8;
  const int cv = mi & 1;
  // Row addresses in stage 0 of the ring for the 16-byte chunk pair m of a 128-byte box
  // row (chunks 2m, 2m+1 before the swizzle): the 128-byte swizzle puts chunk c of row t at
  // c ^ (t & 7).  A stage, a tile and a later box add constants.
  const uint32_t ring_a = smem_addr(ring);
  uint32_t kaddr[4];
#pragma unroll
  for (int m2 = 0; m2 < 4; ++m2)
    kaddr[m2] = ring_a + (C::kPairRows ? swz_off_pair(tok_k, ((2 * m2) | ck) & 3) : swz_off(tok_k, (2 * m2) | ck));
  const uint32_t scl_a = smem_addr(scl) + gi * 4;  // this lane's token row gi in the scales

  for (int item = first_item<C::kThreads>(p, ss); item >= 0;) {
  const int ticket = prefetch_ticket(p);
  ItemInfo it;
  locate_unit(p, ss, item, it);
  // Without a window the item's table slice starts at block part * P whatever the
  // context length, so the length and the slice's first kThreads entries are requested
  // together (one global-memory round trip instead of two).  Entries past the context
  // still lie inside the table row (part * P < max_blocks_per_seq) and are never used.
  const int32_t* trow0 = p.block_tables + size_t(it.b) * p.max_blocks_per_seq + it.part * P;
  int tpre = 0;
  if (!kGen && int(threadIdx.x) < min(partition_cap(P), p.max_blocks_per_seq - it.part * P))
    tpre = __ldg(trow0 + threadIdx.x);
  if (locate_len(p, __ldg(p.context_lens + it.b), it)) {
  const int b = it.b, kvh = it.kvh, part = it.part, nparts = it.nparts, T = it.T;
  if (it.bad_len) {
    write_bad_len<NC, D, C::kThreads>(p, it);
  } else {
  const int nblk = (T + kBlockSize - 1) / kBlockSize;
  const int blk0 = (kGen ? first_block(p, T) : 0) + part * P;
  const int nb_item = (part == nparts - 1 ? nblk : min(nblk, blk0 + P)) - blk0;  // the last takes the rest
  const int32_t* trow = p.block_tables + size_t(b) * p.max_blocks_per_seq + blk0;
  if constexpr (!kGen) {
    if (int(threadIdx.x) < nb_item) tbl[threadIdx.x] = tpre;
    for (int i = threadIdx.x + C::kThreads; i < nb_item; i += C::kThreads) tbl[i] = __ldg(trow + i);
  } else {
    for (int i = threadIdx.x; i < nb_item; i += C::kThreads) tbl[i] = __ldg(trow + i);
  }
  // The previous item's merge record sits in the rings (generic-proxy stores and loads);
  // order those accesses before this item's tensor / bulk copies (async proxy) refill them.
  fence_proxy_async_smem();
  __syncthreads();

  // The item's blocks are taken BPS at a time (one ring stage); warp w takes stages
  // w, w + NW, ... of the item.
  const int nst = (nb_item + BPS - 1) / BPS;
  const int nw = warp < nst ? (nst - 1 - warp) / NW + 1 : 0;
  // Tiles are read once, unless the kv head's columns are split into chunks: then the
  // other chunks' CTAs read them again right away, so keep them in L2.
  const uint64_t policy = p.chunks > 1 ? l2_evict_last_policy() : l2_evict_first_policy();

  // Fetch the warp's k-th stage of the item.  The whole warp runs this with warp-uniform
  // values; one elected lane issues the copies.
  auto issue = [&](auto s_c, int k) {
    const int s = s_c.value;  // (kb + k) % S
    unsigned char* st = ring + s * C::kStageBytes;
    float* sc = scl + s * (C::kScaleStage / 4);
    const int ib0 = (warp + k * NW) * BPS;
    int tiles[BPS];
    uint32_t bytes = 0;
#pragma unroll
    for (int j = 0; j < BPS; ++j) {
      tiles[j] = -1;
      if (ib0 + j >= nb_item) continue;
      const int phys = tbl[ib0 + j];
      if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) set_error(p.err, kErrBlockId);
        continue;
      }
      tiles[j] = phys * p.kv_heads + kvh;  // pools with tensor maps have < 2^27 tiles
      bytes += 2 * C::kTileBytes + (C::kQuant ? 2 * kBlockSize * 4 : 0);
    }
    if (!elect_one()) return;
    if (bytes == 0) {
      mbar_arrive(bars + s);  // complete the phase with no data; the blocks are skipped
      return;
    }
    mbar_arrive_expect_tx(bars + s, bytes);
#pragma unroll
    for (int j = 0; j < BPS; ++j) {
      if (tiles[j] < 0) continue;
      const int row = tiles[j] * C::kBoxRows;  // row of the tensor map's view of the pool
#pragma unroll
      for (int x = 0; x < C::kBoxes; ++x) {
        tma_load_2d(st + j * C::kTileBytes + x * C::kBoxBytes, &tmap_k, x * C::kBoxCols, row,
                    bars + s, policy);
        tma_load_2d(st + (BPS + j) * C::kTileBytes + x * C::kBoxBytes, &tmap_v, x * C::kBoxCols,
                    row, bars + s, policy);
      }
      if constexpr (C::kQuant) {
        bulk_copy_g2s(sc + j * kBlockSize, p.k_scale + int64_t(tiles[j]) * kBlockSize,
                      kBlockSize * 4, bars + s, policy);
        bulk_copy_g2s(sc + (BPS + j) * kBlockSize, p.v_scale + int64_t(tiles[j]) * kBlockSize,
                      kBlockSize * 4, bars + s, policy);
      }
    }
  };
  {
    if constexpr (kGen) {
      for (int k = 0; k < S && k < nw; ++k) issue(StageRt{int((kb + k) % S)}, k);
    } else {
      static_for<S>([&](auto s_c) {  // kb is a multiple of S: stage k for the k-th
        constexpr int k = decltype(s_c)::value;
        if (k < nw) issue(s_c, k);
      });
    }
  }

  // ---- q as the B operand of S = K q^T: in n-tile nt, lane (gi, gj) holds column
  //      8nt + gi, k pairs 2gj, 2gj+8.
  const int c0 = it.chunk * NC;  // first query column of this item's chunk
  const int ncols = chunk_cols(p, c0, NC);
  const auto* qall = static_cast<const __nv_bfloat16*>(p.q);
  uint32_t qf[C::kKSteps][NT][2];
  float logit_factor = p.scale_log2;
  float kbias[NT][2];  // INT8: 1152 * sum_d q_d for columns 8nt + 2gj, 8nt + 2gj + 1
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) kbias[nt][0] = kbias[nt][1] = 0.0f;
  if constexpr (!C::kQuant) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = 8 * nt + gi;
      const bool act = c < ncols;
      const __nv_bfloat16* qb = qall + col_row(p, b, kvh, c0 + c) * D;  // read only when active
#pragma unroll
      for (int s = 0; s < C::kKSteps; ++s) {
        qf[s][nt][0] = qf[s][nt][1] = 0u;
        if (act) {
          qf[s][nt][0] = __ldg(reinterpret_cast<const uint32_t*>(qb + 16 * s + 2 * gj));
          qf[s][nt][1] = __ldg(reinterpret_cast<const uint32_t*>(qb + 16 * s + 2 * gj + 8));
        }
      }
    }
  } else {
    // fp16 operands: bring q into fp16 range with a power of two (exact for bf16 values);
    // its inverse goes into the logit factor.  Lane (gi, gj) loads dims 16s + 4gj .. +3 of
    // column 8nt + gi for k-step s (the permutation used for K below), so the warp holds
    // every active column once and reduces max |q| from registers.
    uint2 raw[NT][C::kKSteps];
    float amax = 0.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = 8 * nt + gi;
      const __nv_bfloat16* qb = qall + col_row(p, b, kvh, c0 + c) * D + 4 * gj;  // read only when active
#pragma unroll
      for (int s = 0; s < C::kKSteps; ++s) {
        raw[nt][s] = make_uint2(0u, 0u);
        if (c < ncols) raw[nt][s] = __ldg(reinterpret_cast<const uint2*>(qb + 16 * s));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16lo(raw[nt][s].x)), fabsf(bf16hi(raw[nt][s].x))),
                                 fmaxf(fabsf(bf16lo(raw[nt][s].y)), fabsf(bf16hi(raw[nt][s].y)))));
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    int e = 0;
    if (amax > 0.0f) e = min(100, max(-100, int((__float_as_uint(amax) >> 23) & 0xff) - 127 - 14));
    const float qs = __uint_as_float(uint32_t(127 - e) << 23);
    logit_factor = p.scale_log2 * __uint_as_float(uint32_t(127 + e) << 23);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int s = 0; s < C::kKSteps; ++s) {
        qf[s][nt][0] = pack_f16x2(bf16lo(raw[nt][s].x) * qs, bf16hi(raw[nt][s].x) * qs);
        qf[s][nt][1] = pack_f16x2(bf16lo(raw[nt][s].y) * qs, bf16hi(raw[nt][s].y) * qs);
      }
      // INT8 K codes enter the product as 1152 + code: S' = S + 1152 * sum_d q_d.  Sum the
      // fp16 values exactly as the MMA sees them, per column.
      float qsum = 0.0f;
#pragma unroll
      for (int s = 0; s < C::kKSteps; ++s) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&qf[s][nt][0]));
        const float2 c2 = __half22float2(*reinterpret_cast<const __half2*>(&qf[s][nt][1]));
        qsum += (a.x + a.y) + (c2.x + c2.y);
      }
      qsum += __shfl_xor_sync(kFull, qsum, 1);
      qsum += __shfl_xor_sync(kFull, qsum, 2);  // lanes of row gi now hold column 8nt+gi's sum
      if constexpr (!C::kFp8) {
        kbias[nt][0] = 1152.0f * __shfl_sync(kFull, qsum, 4 * (2 * gj));
        kbias[nt][1] = 1152.0f * __shfl_sync(kFull, qsum, 4 * (2 * gj + 1));
      }
    }
  }
  // Causal cuts of the accumulator columns 8nt + 2gj and 8nt + 2gj + 1.
  int cut[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    cut[nt][0] = kGen ? col_cut(p, c0 + 8 * nt + 2 * gj) : 0;
    cut[nt][1] = kGen ? col_cut(p, c0 + 8 * nt + 2 * gj + 1) : 0;
  }

  float o[C::kMTiles][NT][4];
#pragma unroll
  for (int t = 0; t < C::kMTiles; ++t)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[t][nt][0] = o[t][nt][1] = o[t][nt][2] = o[t][nt][3] = 0.0f;
  // Softmax state of columns 8nt + 2gj ([nt][0]) and 8nt + 2gj + 1 ([nt][1]).
  float m[NT][2], l[NT][2];
  // INT8: running sum of P' per column (units of 2^e_run), for the V bias.  An MMA with an
  // all-ones A operand forms it from the same fp16 P' as the PV product, in the layout
  // of an O^T fragment (every row holds its column's sum).
  float psum[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = kMaxFloor;
    l[nt][0] = l[nt][1] = 0.0f;
    psum[nt][0] = psum[nt][1] = psum[nt][2] = psum[nt][3] = 0.0f;
  }
  int e_run = INT_MIN;  // quantised pools: O^T is kept in units of 2^e_run
  float pe = 1.0f;       // 2^-e_run
  float pe_next = 0.0f;  // 2^(e_run + 1): a V scale at or above it moves e_run

  int failed_at = -1;
  // One block-loop step: the warp's k-th stage of the item, in ring stage s = k % S, whose
  // barrier phase has parity ph.
  auto step = [&](auto s_c, int k, uint32_t ph) {
    const int s = s_c.value;
    const int kSt = s * C::kStageBytes;  // byte offset of the stage in the ring
    const int kScl = s * C::kScaleStage;  // byte offset of its scales
    const bool ok = __all_sync(kFull, mbar_wait_bounded(bars + s, ph));
    if (!ok) {
      failed_at = k;
      if (lane == 0) set_error(p.err, kErrTimeout);
      return;
    }
    const int ib0 = (warp + k * NW) * BPS;
    int vt[BPS];   // tokens of block j inside the context (0: absent block)
    int rem[BPS];  // context tokens from block j's first token on (0: absent block)
    int tlo[BPS];  // tokens of block j before every query's window (0 without kGen)
    bool any = false;
#pragma unroll
    for (int j = 0; j < BPS; ++j) {
      vt[j] = 0;
      rem[j] = 0;
      if (ib0 + j < nb_item) {
        const int phys = tbl[ib0 + j];
        if (phys >= 0 && phys < p.num_blocks) {
          rem[j] = T - (blk0 + ib0 + j) * kBlockSize;
          vt[j] = min(kBlockSize, rem[j]);
        }
      }
      tlo[j] = kGen ? max(0, rem[j] - (p.num_queries - 1) - p.window) : 0;
      any |= vt[j] > 0;
    }
    if (any) {
      // ---- S_j = K_j q^T (fp32) per block j and n-tile nt:
      //      sacc[j][nt] = {S[gi][c0], S[gi][c1], S[gi+8][c0], S[gi+8][c1]},
      //      c0 = 8nt + 2gj, c1 = c0 + 1
      float sacc[BPS][NT][4];
#pragma unroll
      for (int j = 0; j < BPS; ++j) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sacc[j][nt][0] = sacc[j][nt][1] = sacc[j][nt][2] = sacc[j][nt][3] = 0.0f;
        if (vt[j] == 0) continue;
        const int kKt = kSt + j * C::kTileBytes;  // K tile j
        // Two accumulators (even and odd k-steps) halve the dependent MMA chain.
        float acc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc2[nt][0] = acc2[nt][1] = acc2[nt][2] = acc2[nt][3] = 0.0f;
        if constexpr (!C::kQuant) {
#pragma unroll
          for (int s2 = 0; s2 < C::kKSteps; ++s2) {
            uint32_t a[4];
            ldmatrix_x4(a, kaddr[s2 & 3] + (kKt + (s2 >> 2) * 2048));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16_16816((s2 & 1) ? acc2[nt] : sacc[j][nt], a, qf[s2][nt][0], qf[s2][nt][1]);
          }
        } else {
          // ldmatrix on the tile seen as pairs of bytes: matrix (tokens 0-7 | 8-15) x
          // 16-byte chunk 2x + (0 | 1) gives lane (gi, gj) the codes of dims 16c + 4gj .. +3
          // (chunk c = 2x + h) of token gi (register 2h) and gi + 8 (register 2h + 1).
          // K-step c pairs dims 16c + 4gj + {0,1} with k slots 2gj, 2gj+1 and + {2,3} with
          // 2gj+8, 2gj+9.
#pragma unroll
          for (int x = 0; x < C::kKSteps / 2; ++x) {
            uint32_t w[4];
            ldmatrix_x4(w, kaddr[x] + kKt);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int s2 = 2 * x + h;
              uint32_t a[4];
              if constexpr (C::kFp8) {
                f16x2x2_from_e4m3x4(w[2 * h], a[0], a[2]);
                f16x2x2_from_e4m3x4(w[2 * h + 1], a[1], a[3]);
              } else {
                const uint32_t ua = w[2 * h] ^ 0x80808080u, ub = w[2 * h + 1] ^ 0x80808080u;
                a[0] = f16x2_biased(ua, 0x4140u);
                a[1] = f16x2_biased(ub, 0x4140u);
                a[2] = f16x2_biased(ua, 0x4342u);
                a[3] = f16x2_biased(ub, 0x4342u);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_f16_16816(h ? acc2[nt] : sacc[j][nt], a, qf[s2][nt][0], qf[s2][nt][1]);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sacc[j][nt][i] += acc2[nt][i];
      }

      // ---- logits in log2 units, masked past the context, each column's causal cut and
      //      window (and for absent blocks, whose rem is 0)
      float sc[BPS][NT][4];
      float bm[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) bm[nt][0] = bm[nt][1] = -INFINITY;
#pragma unroll
      for (int j = 0; j < BPS; ++j) {
        float f0 = logit_factor, f1 = logit_factor;
        if constexpr (C::kQuant) {
          if (vt[j] > 0) {
            f0 *= lds_f32(scl_a + (kScl + j * kBlockSize * 4));
            f1 *= lds_f32(scl_a + (kScl + j * kBlockSize * 4 + 32));
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          sc[j][nt][0] = (sacc[j][nt][0] - kbias[nt][0]) * f0;
          sc[j][nt][1] = (sacc[j][nt][1] - kbias[nt][1]) * f0;
          sc[j][nt][2] = (sacc[j][nt][2] - kbias[nt][0]) * f1;
          sc[j][nt][3] = (sacc[j][nt][3] - kbias[nt][1]) * f1;
          if constexpr (kGen) {  // (token gi | gi + 8) x (column 8nt + 2gj | + 1) visible
            const int lim0 = rem[j] - cut[nt][0], lim1 = rem[j] - cut[nt][1];
            if (!visible(lim0, gi, p.window)) sc[j][nt][0] = -INFINITY;
            if (!visible(lim1, gi, p.window)) sc[j][nt][1] = -INFINITY;
            if (!visible(lim0, gi + 8, p.window)) sc[j][nt][2] = -INFINITY;
            if (!visible(lim1, gi + 8, p.window)) sc[j][nt][3] = -INFINITY;
          }
        }
        // Without the general masks only a block that the context ends in (the item's last;
        // the test is the same for the whole warp) has tokens to mask.
        if (!kGen && vt[j] < kBlockSize) {
          const bool h0 = gi >= vt[j], h1 = gi + 8 >= vt[j];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (h0) sc[j][nt][0] = sc[j][nt][1] = -INFINITY;
            if (h1) sc[j][nt][2] = sc[j][nt][3] = -INFINITY;
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          bm[nt][0] = fmaxf(bm[nt][0], fmaxf(sc[j][nt][0], sc[j][nt][2]));
          bm[nt][1] = fmaxf(bm[nt][1], fmaxf(sc[j][nt][1], sc[j][nt][3]));
        }
      }

      // ---- online softmax for this lane's columns over the stage's tokens.  The running
      //      max moves only when a logit passes it by more than kMaxSlack (log2 units):
      //      until then the probabilities are taken against the old max and may reach
      //      2^kMaxSlack, which fp32 sums and the 16-bit P operand hold with their usual
      //      relative precision.  Most stages thus skip the cross-lane max and the rescale.
      bool grow = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        grow |= (bm[nt][0] > m[nt][0] + kMaxSlack) | (bm[nt][1] > m[nt][1] + kMaxSlack);
      float r[NT][2];  // rescale factors of the running sums
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) r[nt][0] = r[nt][1] = 1.0f;
      bool rescale = __any_sync(kFull, grow);
      if (rescale) {
#pragma unroll
        for (int ofs = 4; ofs < 32; ofs <<= 1)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            bm[nt][0] = fmaxf(bm[nt][0], __shfl_xor_sync(kFull, bm[nt][0], ofs));
            bm[nt][1] = fmaxf(bm[nt][1], __shfl_xor_sync(kFull, bm[nt][1], ofs));
          }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const float mu = fmaxf(m[nt][c], bm[nt][c]);  // finite, see kMaxFloor
            r[nt][c] = fast_exp2(m[nt][c] - mu);
            m[nt][c] = mu;
          }
      }
      float pr[BPS][NT][4];
      float ps[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) ps[nt][0] = ps[nt][1] = 0.0f;
#pragma unroll
      for (int j = 0; j < BPS; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pr[j][nt][0] = fast_exp2(sc[j][nt][0] - m[nt][0]);
          pr[j][nt][1] = fast_exp2(sc[j][nt][1] - m[nt][1]);
          pr[j][nt][2] = fast_exp2(sc[j][nt][2] - m[nt][0]);
          pr[j][nt][3] = fast_exp2(sc[j][nt][3] - m[nt][1]);
        }

      uint32_t x01[BPS][NT], x23[BPS][NT];
      if constexpr (!C::kQuant) {
        // P enters the PV product as bf16 (8 significant bits); the softmax sum takes the
        // same rounded weights, so that numerator and denominator agree (summing the fp32
        // weights instead leaves a systematic relative error of up to 2^-9 in the output).
#pragma unroll
        for (int j = 0; j < BPS; ++j)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            x01[j][nt] = pack_bf16x2(pr[j][nt][0], pr[j][nt][1]);
            x23[j][nt] = pack_bf16x2(pr[j][nt][2], pr[j][nt][3]);
            ps[nt][0] += bf16lo(x01[j][nt]) + bf16lo(x23[j][nt]);
            ps[nt][1] += bf16hi(x01[j][nt]) + bf16hi(x23[j][nt]);
          }
      } else {
        // fp16 P' (11 significant bits) carries the V scale too; the sum stays on the fp32
        // weights, whose rounding in P' is 4x finer than bf16's.
#pragma unroll
        for (int j = 0; j < BPS; ++j)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            ps[nt][0] += pr[j][nt][0] + pr[j][nt][2];
            ps[nt][1] += pr[j][nt][1] + pr[j][nt][3];
          }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        l[nt][0] = fmaf(l[nt][0], r[nt][0], ps[nt][0]);
        l[nt][1] = fmaf(l[nt][1], r[nt][1], ps[nt][1]);
      }
      if constexpr (C::kQuant) {
        float sv[BPS][2];
        float svm = 0.0f;
#pragma unroll
        for (int j = 0; j < BPS; ++j) {
          // scales of tokens outside [tlo, vt) may be anything: their weight is 0 anyway
          sv[j][0] = lds_f32(scl_a + (kScl + (BPS + j) * kBlockSize * 4));
          sv[j][1] = lds_f32(scl_a + (kScl + (BPS + j) * kBlockSize * 4 + 32));
          if (kGen || vt[j] < kBlockSize) {
            const unsigned span = unsigned(vt[j] - tlo[j]);
            if (unsigned(gi - tlo[j]) >= span) sv[j][0] = 0.0f;
            if (unsigned(gi + 8 - tlo[j]) >= span) sv[j][1] = 0.0f;
          }
          svm = fmaxf(svm, fmaxf(sv[j][0], sv[j][1]));
        }
        // The exponent E only grows: it moves when some scale reaches 2^(E+1) (and at the
        // first stage), and then to the exponent of the largest scale of the stage.
        if (__any_sync(kFull, e_run == INT_MIN || svm >= pe_next)) {
#pragma unroll
          for (int ofs = 4; ofs < 32; ofs <<= 1) svm = fmaxf(svm, __shfl_xor_sync(kFull, svm, ofs));
          const int eb = int((__float_as_uint(svm) >> 23) & 0xff) - 127;  // floor(log2 svm)
          const int e_new = min(126, e_run == INT_MIN ? eb : max(e_run, eb));
          if (e_run != INT_MIN && e_new != e_run) {
            const float f = pow2i(max(-126, e_run - e_new));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              r[nt][0] *= f;
              r[nt][1] *= f;
            }
            rescale = true;
          }
          e_run = e_new;
          pe = pow2i(-e_new);
          pe_next = e_new >= 126 ? INFINITY : pow2i(e_new + 1);
        }
#pragma unroll
        for (int j = 0; j < BPS; ++j) {
          const float w0 = sv[j][0] * pe, w1 = sv[j][1] * pe;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            x01[j][nt] = pack_f16x2(pr[j][nt][0] * w0, pr[j][nt][1] * w0);
            x23[j][nt] = pack_f16x2(pr[j][nt][2] * w1, pr[j][nt][3] * w1);
          }
        }
      }
      if (rescale) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int t = 0; t < C::kMTiles; ++t) {
            o[t][nt][0] *= r[nt][0]; o[t][nt][1] *= r[nt][1];
            o[t][nt][2] *= r[nt][0]; o[t][nt][3] *= r[nt][1];
          }
          psum[nt][0] *= r[nt][0]; psum[nt][1] *= r[nt][1];
          psum[nt][2] *= r[nt][0]; psum[nt][3] *= r[nt][1];
        }
      }

      // ---- O^T += V_j^T P_j.  P_j as the B operand: in n-tile nt lane (gi, gj) needs
      //      P_j[tokens 2gj, 2gj+1 (+8)][column 8nt + gi], the transpose of what it holds.
#pragma unroll
      for (int j = 0; j < BPS; ++j) {
        if (vt[j] == 0) continue;
        uint32_t pb0[NT], pb1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pb0[nt] = movmatrix_trans(x01[j][nt]);
          pb1[nt] = movmatrix_trans(x23[j][nt]);
        }
        const int kVt = kSt + (BPS + j) * C::kTileBytes;  // V tile j
        if constexpr (!C::kQuant) {
          // Slots past the context in the last block, and before every query's window in
          // the first, may hold anything, NaN included, and 0 * NaN would poison the sum:
          // zero those tokens' V.  Lane (gi, gj) holds tokens 2gj, 2gj+1 in A registers 0-1
          // and 2gj+8, 2gj+9 in registers 2-3 (low half first).
          const bool tail = vt[j] < kBlockSize || tlo[j] > 0;
          const unsigned span = unsigned(vt[j] - tlo[j]);
          const uint32_t mlo = (unsigned(2 * gj - tlo[j]) < span ? 0x0000ffffu : 0u) |
                               (unsigned(2 * gj + 1 - tlo[j]) < span ? 0xffff0000u : 0u);
          const uint32_t mhi = (unsigned(2 * gj + 8 - tlo[j]) < span ? 0x0000ffffu : 0u) |
                               (unsigned(2 * gj + 9 - tlo[j]) < span ? 0xffff0000u : 0u);
#pragma unroll
          for (int t = 0; t < C::kMTiles; ++t) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, ring_a + kVt + swz_off(tok_v, 2 * t + cv));
            if (tail) {
              a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[t][nt], a, pb0[nt], pb1[nt]);
          }
        } else {
          // INT8 codes are always finite and masked tokens have a zero weight in P; E4M3 has
          // NaN codes, so an FP8 block's tokens outside [tlo, vt) are zeroed in the fragment
          // as for bf16.
          // ldmatrix.trans on the tile seen as pairs of bytes: matrix (tokens 0-7 | 8-15) x
          // 16-byte column 2x + (0 | 1) gives lane (gi, gj) the bytes [t d, t d+1, t' d,
          // t' d+1] of tokens t = 2gj, t' = 2gj + 1 (+8 in the second matrix) and dims
          // d = 16t + 2gi, d + 1 of m-tile t: row gi is dim 16t + 2gi, row gi + 8 is
          // 16t + 2gi + 1.  One byte permutation per fp16 pair then builds the A operand.
          const unsigned span8 = unsigned(vt[j] - tlo[j]);
          const uint32_t mlo8 = (unsigned(2 * gj - tlo[j]) < span8 ? 0x0000ffffu : 0u) |
                                (unsigned(2 * gj + 1 - tlo[j]) < span8 ? 0xffff0000u : 0u);
          const uint32_t mhi8 = (unsigned(2 * gj + 8 - tlo[j]) < span8 ? 0x0000ffffu : 0u) |
                                (unsigned(2 * gj + 9 - tlo[j]) < span8 ? 0xffff0000u : 0u);
#pragma unroll
          for (int x = 0; x < C::kMTiles / 2; ++x) {
            uint32_t w[4];
            ldmatrix_x4_trans(w, kaddr[x] + kVt);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int t = 2 * x + h;
              uint32_t lo = w[2 * h], hi = w[2 * h + 1];  // tokens 2gj, 2gj+1 | 2gj+8, 2gj+9
              uint32_t a[4];
              if constexpr (C::kFp8) {
                f16x2x2_from_e4m3x4(__byte_perm(lo, 0u, 0x3120u), a[0], a[1]);
                f16x2x2_from_e4m3x4(__byte_perm(hi, 0u, 0x3120u), a[2], a[3]);
                if (vt[j] < kBlockSize || tlo[j] > 0) {
                  a[0] &= mlo8; a[1] &= mlo8; a[2] &= mhi8; a[3] &= mhi8;
                }
              } else {
                lo ^= 0x80808080u;
                hi ^= 0x80808080u;
                a[0] = f16x2_biased(lo, 0x4240u);
                a[1] = f16x2_biased(lo, 0x4341u);
                a[2] = f16x2_biased(hi, 0x4240u);
                a[3] = f16x2_biased(hi, 0x4341u);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o[t][nt], a, pb0[nt], pb1[nt]);
            }
          }
          if constexpr (!C::kFp8) {
            const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};  // fp16 1.0
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16_16816(psum[nt], ones, pb0[nt], pb1[nt]);
          }
        }
      }
    }
    __syncwarp();
    if (k + S < nw) {
      fence_proxy_async_smem();
      issue(s_c, k + S);
    }
  };
  if constexpr (kGen) {
    // The general masks carry more per-block state: a rolled loop is faster here, and kb
    // need not be a multiple of S.
    for (int k = 0; k < nw && failed_at < 0; ++k) step(StageRt{int((kb + k) % S)}, k, ((kb + k) / S) & 1u);
  } else {
    uint32_t ph = (kb / S) & 1u;  // parity of the current round of S stages
    for (int k0 = 0; k0 < nw && failed_at < 0; k0 += S) {
      static_for<S>([&](auto s_c) {
        constexpr int s = decltype(s_c)::value;
        if (failed_at < 0 && k0 + s < nw) step(s_c, k0 + s, ph);
      });
      ph ^= 1u;
    }
  }
  if (failed_at >= 0) {
    // Let the copies in flight land (bounded) before the ring holds the merge record; the
    // CTA then takes no further items.
    for (int k = failed_at; k < nw && k < failed_at + S; ++k)
      (void)mbar_wait_bounded(bars + ((kb + k) % S), ((kb + k) / S) & 1);
    if (lane == 0 && p.persistent) ss.slot[1] = 1;
    __syncwarp();
  }
  kb += failed_at >= 0 ? min(nw, failed_at + S) : nw;
  if (!kGen && failed_at < 0) {
    // Back to a multiple of S: complete the phases of the stages this item left unused.
    for (; kb % S != 0; ++kb) {
      if (lane == 0) mbar_arrive(bars + kb % S);
      __syncwarp();
      (void)mbar_wait_bounded(bars + kb % S, (kb / S) & 1);
    }
  }

  // ---- this warp's state -> merge record [NC][record_stride(D)] in its ring
#pragma unroll
  for (int ofs = 4; ofs < 32; ofs <<= 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      l[nt][0] += __shfl_xor_sync(kFull, l[nt][0], ofs);
      l[nt][1] += __shfl_xor_sync(kFull, l[nt][1], ofs);
    }
  float oscale = 1.0f;
  if constexpr (C::kQuant) {
    oscale = e_run == INT_MIN ? 0.0f : pow2i(max(-126, e_run));
    if constexpr (!C::kFp8) {
      // INT8 V codes entered as 1152 + code: O'^T = O^T + 1152 * sum_t P'_t for every dim.
#pragma unroll
      for (int t = 0; t < C::kMTiles; ++t)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[t][nt][i] = fmaf(-1152.0f, psum[nt][i], o[t][nt][i]);
    }
  }
  float* rec = reinterpret_cast<float*>(ring);
  constexpr int kRec = record_stride(D);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h0 = 8 * nt + 2 * gj, h1 = h0 + 1;
    if (gi == 0) {
      if (h0 < NC) { rec[h0 * kRec] = m[nt][0]; rec[h0 * kRec + 1] = l[nt][0]; }
      if (h1 < NC) { rec[h1 * kRec] = m[nt][1]; rec[h1 * kRec + 1] = l[nt][1]; }
    }
#pragma unroll
    for (int t = 0; t < C::kMTiles; ++t) {
      if constexpr (C::kQuant) {
        // rows gi and gi + 8 of the O^T fragment are dims 16t + 2gi and 16t + 2gi + 1:
        // one 8-byte store per column (the record's columns start at even floats)
        const int d0 = 16 * t + 2 * gi;
        if (h0 < NC)
          *reinterpret_cast<float2*>(rec + h0 * kRec + 2 + d0) =
              make_float2(o[t][nt][0] * oscale, o[t][nt][2] * oscale);
        if (h1 < NC)
          *reinterpret_cast<float2*>(rec + h1 * kRec + 2 + d0) =
              make_float2(o[t][nt][1] * oscale, o[t][nt][3] * oscale);
      } else {
        const int d0 = 16 * t + gi, d1 = d0 + 8;
        if (h0 < NC) {
          rec[h0 * kRec + 2 + d0] = o[t][nt][0];
          rec[h0 * kRec + 2 + d1] = o[t][nt][2];
        }
        if (h1 < NC) {
          rec[h1 * kRec + 2 + d0] = o[t][nt][1];
          rec[h1 * kRec + 2 + d1] = o[t][nt][3];
        }
      }
    }
  }
  __syncthreads();
  merge_warp_records<NC, D, NW>(smem, size_t(S) * C::kStageBytes, p, b, kvh, c0, part, nparts);
  }  // valid context length
  }  // item located
  item = next_item(p, ss, ticket);
  }  // items
  // The next kernel's CTAs may launch once every CTA of this one has passed here: a
  // trigger at the start let a grid that leaves CTA slots free (the one-wave window
  // plan) have the next call's CTAs placed early and unevenly across the SMs.
  griddep_launch_dependents();
  finish_items(p);
}

template <KvType KV, int D, int NC, int NW, int S, int BPS, bool kGen>
cudaError_t launch_mma_variant(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
  using C = MmaCfg<KV, D, NC, NW, S, BPS>;
  auto kern = paged_decode_mma_kernel<KV, D, NC, NW, S, BPS, kGen>;
  static std::atomic<bool> attr_done[64];  // per device: the shared-memory limit is raised
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::smem_bytes(kMaxPartitionBlocks, kMaxSchedSeqs)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_relaxed);
  }
  const int64_t grid =
      p.persistent ? int64_t(p.grid) : int64_t(p.max_parts) * p.num_seqs * p.kv_heads * p.chunks;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads),
                    C::smem_bytes(p.partition_blocks, p.persistent ? p.num_seqs : 0), stream, tk, tv, p);
}

template <KvType KV, int D, int NC, int NW, int S, int BPS, bool kGen>
int mma_ctas_per_sm_variant() {
  using C = MmaCfg<KV, D, NC, NW, S, BPS>;
  auto kern = paged_decode_mma_kernel<KV, D, NC, NW, S, BPS, kGen>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(C::smem_bytes(kMaxPartitionBlocks, kMaxSchedSeqs)));
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::kThreads, C::smem_bytes(64, 256)) !=
      cudaSuccess)
    return 0;
  return n;
}

// Column-slot dispatch for one (pool type, head_dim, ring shape, kGen).  Plain decode has
// at most 8 columns (a GQA group), so 16 columns exist only with kGen, and only where the
// 16-column merge record fits a warp's ring.  Combinations not built report 0 CTAs per SM
// (the plan turns that into "unsupported").
template <KvType KV, int D, int S, int BPS>
constexpr bool mma_record_fits(int nc) {
  return size_t(nc) * record_stride(D) * 4 <= size_t(S) * MmaCfg<KV, D, 2, kNwMma, S, BPS>::kStageBytes;
}

template <KvType KV, int D, int S, int BPS, bool kGen>
cudaError_t launch_mma_cols(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int cols, cudaStream_t stream) {
  switch (cols) {
    case 2: return launch_mma_variant<KV, D, 2, kNwMma, S, BPS, kGen>(p, tk, tv, stream);
    case 4: return launch_mma_variant<KV, D, 4, kNwMma, S, BPS, kGen>(p, tk, tv, stream);
    case 8: return launch_mma_variant<KV, D, 8, kNwMma, S, BPS, kGen>(p, tk, tv, stream);
    case 16:
      if constexpr (kGen && mma_record_fits<KV, D, S, BPS>(16))
        return launch_mma_variant<KV, D, 16, kNwMma, S, BPS, kGen>(p, tk, tv, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <KvType KV, int D, int S, int BPS, bool kGen>
int occupancy_mma_cols(int cols) {
  switch (cols) {
    case 2: return mma_ctas_per_sm_variant<KV, D, 2, kNwMma, S, BPS, kGen>();
    case 4: return mma_ctas_per_sm_variant<KV, D, 4, kNwMma, S, BPS, kGen>();
    case 8: return mma_ctas_per_sm_variant<KV, D, 8, kNwMma, S, BPS, kGen>();
    case 16:
      if constexpr (kGen && mma_record_fits<KV, D, S, BPS>(16))
        return mma_ctas_per_sm_variant<KV, D, 16, kNwMma, S, BPS, kGen>();
      return 0;
  }
  return 0;
}

template <KvType KV, int D, int S, int BPS>
cudaError_t launch_mma_gen(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           int cols, bool gen, cudaStream_t stream) {
  return gen ? launch_mma_cols<KV, D, S, BPS, true>(p, tk, tv, cols, stream)
             : launch_mma_cols<KV, D, S, BPS, false>(p, tk, tv, cols, stream);
}

template <KvType KV, int D, int S, int BPS>
int occupancy_mma_gen(int cols, bool gen) {
  return gen ? occupancy_mma_cols<KV, D, S, BPS, true>(cols) : occupancy_mma_cols<KV, D, S, BPS, false>(cols);
}

}  // namespace pkv
