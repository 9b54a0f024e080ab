// pkv_decode.cuh -- PagedAttention decode on the CUDA cores (paged_decode_kernel), the
// work scheduling and partition merge shared with the tensor-core kernel
// (pkv_decode_mma.cuh), for sm_103a.  The tensor-core kernel is the automatic choice for
// every built shape; this one computes the same function and can be forced.
//
// What is computed ("Lesson 4: Model deployment and inference acceleration", 4.2,
// attention-invariance equation): for sequence b and query head h,
//     out[b][h] = sum_{t < T_b} softmax_t(scale * q[b][h] . K_b[t]) V_b[t],
// where token t of sequence b sits in physical block block_tables[b][t / 16] at offset
// t % 16 of a [num_blocks, Hkv, 16, D] pool, and q head h reads kv head h / G with
// G = Hq / Hkv (contiguous GQA groups; "LLM/MLLM inference optimisation", 2.3).
//
// Work decomposition.  A work item is (sequence b, kv head, context partition p); the
// partition covers P consecutive logical blocks.  One CTA of NW warps runs one item and
// serves all query columns of its kv head (the G query heads of the group, times the query
// tokens of a multi-query call; template parameter G counts column slots), so each K/V
// block is read from HBM once per group.  Warp w takes the item's blocks w, w + NW, ...;
// each warp owns a ring of S shared-memory stages, and one elected lane fills a stage with
// one bulk asynchronous copy per tile (the [phys][kvh] K tile and V tile are each one
// contiguous 16*D-element run, so no tensor map is needed), completing on the stage's
// mbarrier.  The block table slice of the item is staged in shared memory first.
//
// Per block a warp computes 16 tokens x G columns of logits with fp32 FMAs: lanes split
// a token's D dims (DPL dims each) and hold q for all G columns in registers; a
// transposed butterfly reduces the G partial dot products across the lanes of a token
// so that each lane ends with one column's logit.  The online softmax ("LLM/MLLM inference
// optimisation", 3.2: running max and running sum) rescales the running state by
// exp(m_old - m_new) per block; logits are kept in log2 units (scale * log2 e is folded
// into q) so that exp2 is the only exponential.  Probabilities go through a small
// per-warp shared array to the PV layout, where each lane owns D/32 output dims of all
// G columns.  At the end of the item the NW warp states merge in shared memory; a
// single-partition sequence writes bf16 output directly, otherwise the item writes its
// partial (max, sum, accumulator) and a second kernel merges the partitions with the
// same log-sum-exp algebra.
//
// INT8 pools: logit = (scale * log2 e) * s_K[t] * sum_c q_c code_c, and the PV weight of
// token t is p_t * s_V[t]; codes are widened to fp32 exactly (see i8_from_flipped).
// FP8 (E4M3) pools work the same way with the hardware E4M3 -> fp16 conversion.
//
// Several query tokens per sequence (verifying k draft tokens in one pass; "Lesson 4", 5.2
// "Speculative Decoding"): the k queries are the sequence's last k positions and query i
// sees tokens t < T_b - (k - 1 - i).  A CTA then serves group * k query columns of its kv
// head -- column c is query c / group of head kvh * group + c % group -- so each K/V block
// is still read once, and each column carries its own causal cut.  With k = 1 this is the
// plain decode above.
//
// Sliding window ("LLM/MLLM inference optimisation", 2.3: keep only the most recent window
// of the cache): a query at position p sees tokens p - W + 1 .. p.  A sequence's work then
// starts at the first block any of its queries sees; earlier blocks are never read (their
// table entries may be -1), and tokens of that first block before the window are masked
// and their V zeroed, since their slots may hold anything.
//
// Masking: tokens t >= T_b of the last block get logit -inf and are excluded from the
// PV loop, so whatever bytes sit in unused slots are never used.  Block ids outside
// [0, num_blocks) are skipped (no copy) and flagged in the device error word.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "pkv_device.cuh"

namespace pkv {

constexpr int kMaxPartitionBlocks = 1024;  // largest P

template <KvType KV>
struct KvTraits;
template <>
struct KvTraits<KvType::kBf16> {
  static constexpr int kElemBytes = 2;
  static constexpr bool kQuant = false;
};
template <>
struct KvTraits<KvType::kInt8> {
  static constexpr int kElemBytes = 1;
  static constexpr bool kQuant = true;
};
template <>
struct KvTraits<KvType::kFp8> {
  static constexpr int kElemBytes = 1;
  static constexpr bool kQuant = true;
};

// Four 1-byte codes of a word -> fp32 values (INT8 or E4M3), exactly.
template <KvType KV>
__device__ __forceinline__ void dequant4(uint32_t w, float (&f)[4]) {
  if constexpr (KV == KvType::kFp8) {
    e4m3x4_to_f32(w, f);
  } else {
    const uint32_t u = w ^ 0x80808080u;
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = i8_from_flipped(u, i);
  }
}

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Floats per query column in a warp's merge record: running max, sum, D accumulators and
// two of padding.  With a stride of D + 4 (4 mod 16), the tensor-core kernel's transposed
// record writes -- lane (gi, gj) writes column 2gj (+1), dims 16t + 2gi (+1) or 16t + gi
// (+8) -- land in distinct banks (a stride of D + 2 put two to four lanes on one bank).
constexpr int record_stride(int d) { return d + 4; }

// Shared memory of the persistent-grid scheduler: the batch's partition prefix sum
// (num_seqs + 1 ints), two control ints and one scan slot per thread.
__host__ __device__ constexpr size_t sched_smem_bytes(int num_seqs, int threads) {
  return (size_t(num_seqs) + 1 + 2 + threads) * 4;
}

template <KvType KV, int D, int G, int NW, int S>
struct DecodeCfg {
  static constexpr int kEsz = KvTraits<KV>::kElemBytes;
  static constexpr bool kQuant = KvTraits<KV>::kQuant;
  static constexpr int kTileBytes = kBlockSize * D * kEsz;         // one K (or V) tile
  static constexpr int kScaleBytes = kQuant ? kBlockSize * 4 : 0;  // one fp32 scale tile
  static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes;
  static constexpr int kDPL = (G <= 4) ? 16 : 8;  // QK: dims per lane
  static constexpr int kLPT = D / kDPL;           // QK: lanes per token
  static constexpr int kTPP = 32 / kLPT;          // QK: tokens per pass
  static constexpr int kPasses = kBlockSize / kTPP;
  static constexpr int kDup = kLPT / G;            // lanes holding the same (token, column) logit
  static constexpr int kDPV = D / 32;             // PV: dims per lane
  static constexpr int kThreads = NW * 32;
  static constexpr bool kSwapHalves = !kQuant && kDPL == 16;

  static constexpr size_t kRingBytes = size_t(NW) * S * kStageBytes;
  static constexpr size_t kProbOff = kRingBytes;  // float [NW][17][G]: 16 p rows + alpha row
  static constexpr size_t kProbBytes = size_t(NW) * 17 * G * 4;
  static constexpr size_t kBarOff = align_up(kProbOff + kProbBytes, 16);
  static constexpr size_t kTableOff = kBarOff + size_t(NW) * S * 8;
  static size_t smem_bytes(int partition_blocks, int sched_seqs) {
    return kTableOff + size_t(partition_cap(partition_blocks)) * 4 + sched_smem_bytes(sched_seqs, kThreads);
  }

  static_assert(D % 32 == 0 && (D == 64 || D == 128), "head_dim 64 or 128");
  static_assert(kLPT >= G && kLPT <= 32, "a token's lanes must cover the group");
  static_assert(kTPP * kPasses == kBlockSize, "passes must cover the block");
  static_assert(size_t(G) * record_stride(D) * 4 <= size_t(kStageBytes), "merge record fits a stage");
  static_assert(kTileBytes % 16 == 0 && kStageBytes % 16 == 0, "bulk copies need 16 B");
};

// Transposed butterfly: NG partial sums per lane, lanes at xor-distance O, O/2, ... 1
// belong to one token.  While more than one head remains, each step swaps half of the
// heads with the partner lane, so the number of shuffles is about NG instead of
// NG * log2(lanes).  At the end v[0] holds the full dot product for head
// (lane % LPT) / (LPT / G).
template <int NG, int O>
struct HeadReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (NG > 1) {
      constexpr int H = NG / 2;
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = upper ? v[i] : v[i + H];
        const float keep = upper ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      HeadReduce<H, O / 2>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      HeadReduce<1, O / 2>::run(v, lane);
    }
  }
};

template <int G, int NQ>
__device__ __forceinline__ void fma_bf16x8(float (&part)[G], const float (&qr)[G][NQ], int base,
                                           const uint4 w) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float k0 = bf16lo(ws[i]);
    const float k1 = bf16hi(ws[i]);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      part[g] = fmaf(qr[g][base + 2 * i], k0, part[g]);
      part[g] = fmaf(qr[g][base + 2 * i + 1], k1, part[g]);
    }
  }
}

template <KvType KV, int G, int NQ>
__device__ __forceinline__ void fma_code4(float (&part)[G], const float (&qr)[G][NQ], int base,
                                          uint32_t w) {
  float k[4];
  dequant4<KV>(w, k);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int g = 0; g < G; ++g) part[g] = fmaf(qr[g][base + i], k[i], part[g]);
  }
}

// ---------------------------------------------------------------- work scheduling
//
// A work item is (sequence b, kv head, partition).  Two ways to map CTAs to items:
//  * classic grid (large batches): one CTA per (partition slot, sequence, kv head), where
//    slots past a sequence's own partition count exit at once;
//  * persistent grid (batches up to kMaxSchedSeqs sequences): a few CTAs per SM build, in
//    shared memory, the prefix sum of every sequence's partition count and take items from
//    a ticket counter in global memory, one item ahead, until the tickets run out.  The
//    last CTA to finish resets the counters to zero for the next call.  Nothing waits on
//    another CTA.
// A sequence whose context length is out of range counts as one item that writes zeros.

struct ItemInfo {
  int b, kvh, chunk, part, nparts, T;  // chunk: which slice of the kv head's query columns
  bool bad_len;
};

// Shared-memory tail after the block-table slice: cum[B + 1] | slot[2] | scan[NT].
struct SchedSmem {
  int* cum;
  int* slot;  // [0]: current item, [1]: abort flag
  int* scan;
};

__device__ __forceinline__ SchedSmem sched_smem(unsigned char* tail, int num_seqs) {
  int* base = reinterpret_cast<int*>(tail);
  return SchedSmem{base, base + num_seqs + 1, base + num_seqs + 3};
}

// First logical block of a T-token sequence that some query sees (0 without a window).
__device__ __forceinline__ int first_block(const DecodeParams& p, int T) {
  const int lo = T - (p.num_queries - 1) - p.window;  // first query's first visible token
  return lo > 0 ? lo / kBlockSize : 0;
}

__device__ __forceinline__ int seq_parts(const DecodeParams& p, int T) {
  if (T < p.num_queries || T > p.max_context_len) return 1;
  const int nblk = (T + kBlockSize - 1) / kBlockSize - first_block(p, T);
  return partition_count(nblk, p.partition_blocks);
}

// Whether token t of a block is visible to a column: lim = the column's visible tokens
// counted from the block's first token (context minus causal cut minus block start);
// visible iff lim - W <= t < lim, one unsigned compare.
__device__ __forceinline__ bool visible(int lim, int t, int window) {
  return unsigned(lim - 1 - t) < unsigned(window);
}

// First item of this CTA, or -1.  Builds the prefix sum in persistent mode.  Ends with a
// barrier (so it also publishes the mbarrier initialisation done before it).
template <int NT>
__device__ __forceinline__ int first_item(const DecodeParams& p, const SchedSmem& ss) {
  if (!p.persistent) {
    __syncthreads();
    return blockIdx.x;
  }
  const int B = p.num_seqs;
  const int per = (B + NT - 1) / NT;
  const int lo = min(B, int(threadIdx.x) * per);
  const int hi = min(B, lo + per);
  int sum = 0;
  for (int b = lo; b < hi; ++b) {
    const int c = seq_parts(p, __ldg(p.context_lens + b));
    ss.cum[b + 1] = c;
    sum += c;
  }
  ss.scan[threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < NT; ++i) {
      const int v = ss.scan[i];
      ss.scan[i] = run;
      run += v;
    }
    ss.cum[0] = 0;
    ss.slot[0] = static_cast<int>(atomicAdd(p.sched, 1u));
    ss.slot[1] = 0;
  }
  __syncthreads();
  int run = ss.scan[threadIdx.x];
  for (int b = lo; b < hi; ++b) {
    run += ss.cum[b + 1];
    ss.cum[b + 1] = run;
  }
  __syncthreads();
  const int item = ss.slot[0];
  return item < ss.cum[B] * (p.kv_heads * p.chunks) ? item : -1;
}

// Ticket for the item after this one (thread 0 fetches it now; its value is used at the
// end of the item, so the atomic's latency overlaps the item's work).
__device__ __forceinline__ int prefetch_ticket(const DecodeParams& p) {
  return (p.persistent && threadIdx.x == 0) ? static_cast<int>(atomicAdd(p.sched, 1u)) : 0;
}

__device__ __forceinline__ int next_item(const DecodeParams& p, const SchedSmem& ss, int ticket) {
  if (!p.persistent) return -1;
  __syncthreads();  // this item's shared memory is free again
  if (threadIdx.x == 0) ss.slot[0] = ticket;
  __syncthreads();
  const int item = ss.slot[0];
  if (ss.slot[1]) return -1;  // a bounded wait gave up: stop taking work
  return item < ss.cum[p.num_seqs] * (p.kv_heads * p.chunks) ? item : -1;
}

__device__ __forceinline__ void finish_items(const DecodeParams& p) {
  if (!p.persistent || threadIdx.x != 0) return;
  __threadfence();
  if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
    atomicExch(p.sched, 0u);
    atomicExch(p.sched + 1, 0u);
  }
}

// (b, kv head, column chunk, partition) of an item, which need no context length.  A
// sequence has kv_heads * chunks work units; the chunks of one kv head are adjacent, so
// they tend to run together and share the head's K/V blocks in L2.
__device__ __forceinline__ void locate_unit(const DecodeParams& p, const SchedSmem& ss, int item,
                                            ItemInfo& it) {
  const int ups = p.kv_heads * p.chunks;  // work units per sequence
  int v;
  if (p.persistent) {
    const int u = item / ups;
    v = item - u * ups;
    int lo = 0, hi = p.num_seqs;  // cum[lo] <= u < cum[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ss.cum[mid] <= u) lo = mid; else hi = mid;
    }
    it.b = lo;
    it.part = u - ss.cum[lo];
  } else {
    const int units = p.num_seqs * ups;
    it.part = item / units;
    const int rem = item - it.part * units;
    it.b = rem / ups;
    v = rem - it.b * ups;
  }
  it.kvh = v / p.chunks;
  it.chunk = v - it.kvh * p.chunks;
}

// The rest of an item once its sequence's context length T is known; false for an idle
// classic-grid slot.
__device__ __forceinline__ bool locate_len(const DecodeParams& p, int T, ItemInfo& it) {
  it.T = T;
  it.bad_len = it.T < p.num_queries || it.T > p.max_context_len;
  it.nparts = seq_parts(p, it.T);
  return it.part < it.nparts;
}

__device__ __forceinline__ bool locate_item(const DecodeParams& p, const SchedSmem& ss, int item,
                                            ItemInfo& it) {
  locate_unit(p, ss, item, it);
  return locate_len(p, __ldg(p.context_lens + it.b), it);
}

// Query token of column c and, in *g, its head within the group: c / group and c % group
// (a shift and a mask when the group is a power of two).
__device__ __forceinline__ int col_query(const DecodeParams& p, int c, int* g) {
  const int qi = p.group_log2 >= 0 ? c >> p.group_log2 : c / p.group;
  *g = c - qi * p.group;
  return qi;
}

// Row of q / out (in units of head_dim elements) that query column c of (b, kvh) reads
// and writes: query token c / group of head kvh * group + c % group.
__device__ __forceinline__ size_t col_row(const DecodeParams& p, int b, int kvh, int c) {
  int g;
  const int qi = col_query(p, c, &g);
  return (size_t(b) * p.num_queries + qi) * p.num_q_heads + size_t(kvh) * p.group + g;
}

// Tokens of the sequence hidden from column c by the causal cut: query qi sits k - 1 - qi
// positions before the newest token.  Columns past group * k get 0 (never written).
__device__ __forceinline__ int col_cut(const DecodeParams& p, int c) {
  int g;
  const int qi = col_query(p, c, &g);
  return qi < p.num_queries ? p.num_queries - 1 - qi : 0;
}

// Start value of a running max.  A finite floor rather than -inf: a query column can see
// no token of a whole block (all behind its causal cut), and with a finite start its
// rescale factor exp2(m_old - m_new) is 1 and its probabilities exp2(-inf - m) are 0
// without a special case; once a real logit arrives exp2(kMaxFloor - m) underflows to 0.
constexpr float kMaxFloor = -3.402823466e38f;

// Headroom of a lazily updated running max, in log2 units: a kernel may keep its max while
// new logits stay within kMaxSlack above it, so probabilities reach at most 2^kMaxSlack.
constexpr float kMaxSlack = 8.0f;

// Query columns in the chunk that starts at column c0 (NC slots; the last chunk may be short).
__device__ __forceinline__ int chunk_cols(const DecodeParams& p, int c0, int nc) {
  return min(nc, p.group * p.num_queries - c0);
}

// Zero output and an error bit for a sequence with an out-of-range context length.
template <int NC, int D, int NT>
__device__ __forceinline__ void write_bad_len(const DecodeParams& p, const ItemInfo& it) {
  if (it.part != 0) return;
  auto* out = static_cast<__nv_bfloat16*>(p.out);
  const int c0 = it.chunk * NC;
  const int ncols = chunk_cols(p, c0, NC);
  for (int i = threadIdx.x; i < NC * D; i += NT) {
    const int c = i / D;
    if (c < ncols) out[col_row(p, it.b, it.kvh, c0 + c) * D + (i - c * D)] = __float2bfloat16_rn(0.0f);
  }
  if (threadIdx.x == 0) set_error(p.err, kErrContextLen);
}

// Merge the NW per-warp states of one work item by log-sum-exp and write the bf16 output
// (single-partition sequences) or the item's partial (m, l, acc) to the workspace.  Warp w's
// record is [NC][record_stride(D)] floats (running max in log2 units, sum, accumulator) per query
// column at smem + w * warp_stride; record column c is query column c0 + c.  Each thread
// takes kE consecutive dims of one column, so that the column's weights 2^(m_w - M) are
// formed once per thread and the reads and writes are vectors (out and the workspace are
// 16-byte aligned, and kE divides D).
template <int NC, int D, int NW>
__device__ __forceinline__ void merge_warp_records(const unsigned char* smem, size_t warp_stride,
                                                   const DecodeParams& p, int b, int kvh, int c0,
                                                   int part, int nparts) {
  constexpr int kThreads = NW * 32;
  constexpr int kE = NC * D > kThreads ? NC * D / kThreads : 1;  // dims per thread
  constexpr int kTpc = D / kE;                                    // threads per column
  static_assert(kE * kThreads >= NC * D && D % kE == 0 && (kE == 1 || kE % 2 == 0),
                "merge layout");
  const int g = threadIdx.x / kTpc;
  const int d0 = (threadIdx.x - g * kTpc) * kE;
  if (g >= chunk_cols(p, c0, NC)) return;  // an inactive column, or a thread past NC * D
  float mw[NW];
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    mw[w] = reinterpret_cast<const float*>(smem + size_t(w) * warp_stride)[g * record_stride(D)];
    M = fmaxf(M, mw[w]);
  }
  float L = 0.0f;
  float acc[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) acc[e] = 0.0f;
  if (M != -INFINITY) {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* r = reinterpret_cast<const float*>(smem + size_t(w) * warp_stride) + g * record_stride(D);
      const float f = fast_exp2(mw[w] - M);
      L = fmaf(f, r[1], L);
      if constexpr (kE == 1) {
        acc[0] = fmaf(f, r[2 + d0], acc[0]);
      } else {
#pragma unroll
        for (int e = 0; e < kE; e += 2) {  // record columns start at an even float
          const float2 v = *reinterpret_cast<const float2*>(r + 2 + d0 + e);
          acc[e] = fmaf(f, v.x, acc[e]);
          acc[e + 1] = fmaf(f, v.y, acc[e + 1]);
        }
      }
    }
  }
  const size_t row = col_row(p, b, kvh, c0 + g);
  if (nparts == 1) {
    auto* out = static_cast<__nv_bfloat16*>(p.out) + row * D + d0;
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    if constexpr (kE == 1) {
      out[0] = __float2bfloat16_rn(acc[0] * inv);
    } else {
      uint32_t packed[kE / 2];
#pragma unroll
      for (int e = 0; e < kE; e += 2) packed[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
      if constexpr (kE % 8 == 0) {
#pragma unroll
        for (int e = 0; e < kE / 2; e += 4)
          *reinterpret_cast<uint4*>(out + 2 * e) = make_uint4(packed[e], packed[e + 1], packed[e + 2], packed[e + 3]);
      } else if constexpr (kE == 4) {
        *reinterpret_cast<uint2*>(out) = make_uint2(packed[0], packed[1]);
      } else {
        *reinterpret_cast<uint32_t*>(out) = packed[0];
      }
    }
  } else {
    const size_t pi = row * p.max_parts + part;
    float* ws = p.ws_acc + pi * D + d0;
    if constexpr (kE % 4 == 0) {
#pragma unroll
      for (int e = 0; e < kE; e += 4)
        *reinterpret_cast<float4*>(ws + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    } else if constexpr (kE == 2) {
      *reinterpret_cast<float2*>(ws) = make_float2(acc[0], acc[1]);
    } else {
      ws[0] = acc[0];
    }
    if (d0 == 0) {
      p.ws_ml[2 * pi] = M;
      p.ws_ml[2 * pi + 1] = L;
    }
  }
}

template <KvType KV, int D, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32)
    paged_decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<KV, D, G, NW, S>;
  constexpr uint32_t kFull = 0xffffffffu;
  extern __shared__ __align__(128) unsigned char smem[];
  griddep_wait();  // inputs may come from the previous kernel in the stream

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int* tbl = reinterpret_cast<int*>(smem + C::kTableOff);
  const SchedSmem ss = sched_smem(smem + C::kTableOff + size_t(partition_cap(p.partition_blocks)) * 4,
                                  p.persistent ? p.num_seqs : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff) + warp * S;
  unsigned char* ring = smem + size_t(warp) * S * C::kStageBytes;
  float* prob = reinterpret_cast<float*>(smem + C::kProbOff) + warp * 17 * G;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(bars + s, 1);
    fence_barrier_init();
  }
  const int P = p.partition_blocks;
  uint32_t kb = 0;  // blocks this warp has consumed over all its items: stage and phase counter

  for (int item = first_item<C::kThreads>(p, ss); item >= 0;) {
  const int ticket = prefetch_ticket(p);
  ItemInfo it;
  if (locate_item(p, ss, item, it)) {
  const int b = it.b, kvh = it.kvh, part = it.part, nparts = it.nparts, T = it.T;
  if (it.bad_len) {
    write_bad_len<G, D, C::kThreads>(p, it);
  } else {
  const int nblk = (T + kBlockSize - 1) / kBlockSize;
  const int blk0 = first_block(p, T) + part * P;
  const int nb_item = (part == nparts - 1 ? nblk : min(nblk, blk0 + P)) - blk0;  // the last takes the rest
  const int32_t* trow = p.block_tables + size_t(b) * p.max_blocks_per_seq + blk0;
  for (int i = threadIdx.x; i < nb_item; i += C::kThreads) tbl[i] = __ldg(trow + i);
  // The previous item's merge record sits in the rings (generic-proxy stores and loads);
  // order those accesses before this item's tensor / bulk copies (async proxy) refill them.
  fence_proxy_async_smem();
  __syncthreads();

  // Blocks of this warp: item blocks warp, warp + NW, ...
  const int nw = warp < nb_item ? (nb_item - 1 - warp) / NW + 1 : 0;
  const uint64_t policy = l2_evict_first_policy();
  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);

  // Fetch the warp's k-th block of the item: the whole warp runs this with warp-uniform
  // values, one elected lane issues the copies.
  auto issue = [&](int k) {
    const int s = (kb + k) % S;
    unsigned char* st = ring + size_t(s) * C::kStageBytes;
    const int phys = tbl[warp + k * NW];
    if (!elect_one()) return;
    if (phys < 0 || phys >= p.num_blocks) {
      set_error(p.err, kErrBlockId);
      mbar_arrive(bars + s);  // complete the phase with no data; the block is skipped
      return;
    }
    const int64_t tile = int64_t(phys) * p.kv_heads + kvh;
    mbar_arrive_expect_tx(bars + s, C::kStageBytes);
    bulk_copy_g2s(st, kbase + tile * C::kTileBytes, C::kTileBytes, bars + s, policy);
    bulk_copy_g2s(st + C::kTileBytes, vbase + tile * C::kTileBytes, C::kTileBytes, bars + s,
                  policy);
    if constexpr (C::kQuant) {
      bulk_copy_g2s(st + 2 * C::kTileBytes,
                    reinterpret_cast<const char*>(p.k_scale) + tile * C::kScaleBytes,
                    C::kScaleBytes, bars + s, policy);
      bulk_copy_g2s(st + 2 * C::kTileBytes + C::kScaleBytes,
                    reinterpret_cast<const char*>(p.v_scale) + tile * C::kScaleBytes,
                    C::kScaleBytes, bars + s, policy);
    }
  };
  for (int k = 0; k < S && k < nw; ++k) issue(k);

  // ---- q for this lane's dims of all G query columns, pre-multiplied by scale * log2(e)
  const int tok = lane / C::kLPT;    // token within a pass
  const int chunk = lane % C::kLPT;  // which DPL-dim slice of the row
  const int sw = C::kSwapHalves ? ((lane >> 2) & 1) : 0;
  const int c0 = it.chunk * G;  // first query column of this item's chunk
  const int ncols = chunk_cols(p, c0, G);
  float qr[G][C::kDPL];
  {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const auto* qrow = static_cast<const __nv_bfloat16*>(p.q) + col_row(p, b, kvh, c0 + g) * D;
      const uint4* src = reinterpret_cast<const uint4*>(qrow + chunk * C::kDPL);
#pragma unroll
      for (int h = 0; h < C::kDPL / 8; ++h) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);  // inactive columns: q = 0, never written out
        if (g < ncols) w = __ldg(src + (h ^ sw));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qr[g][8 * h + 2 * i] = bf16lo(ws[i]) * p.scale_log2;
          qr[g][8 * h + 2 * i + 1] = bf16hi(ws[i]) * p.scale_log2;
        }
      }
    }
  }

  const int g_lane = (lane % C::kLPT) / C::kDup;  // column whose logit this lane ends with
  const bool store_lane = (lane % C::kDup) == 0;
  const int cut = col_cut(p, c0 + g_lane);         // its causal cut (0 for a single query)
  float m_run = kMaxFloor;
  float l_run = 0.0f;
  float acc[G][C::kDPV];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < C::kDPV; ++i) acc[g][i] = 0.0f;

  int failed_at = -1;
  for (int k = 0; k < nw; ++k) {
    const int s = (kb + k) % S;
    const bool ok = __all_sync(kFull, mbar_wait_bounded(bars + s, ((kb + k) / S) & 1));
    if (!ok) {
      failed_at = k;
      if (lane == 0) set_error(p.err, kErrTimeout);
      break;
    }
    const int ib = warp + k * NW;
    const int phys = tbl[ib];
    const bool valid = phys >= 0 && phys < p.num_blocks;
    const int vt = valid ? min(kBlockSize, T - (blk0 + ib) * kBlockSize) : 0;
    if (vt > 0) {
      // tokens of this block that column g_lane may see: lim - W <= t < lim; tokens before
      // t_lo are seen by no column (window) and take no part in PV
      const int rem = T - (blk0 + ib) * kBlockSize;
      const int lim = rem - cut;
      const int t_lo = max(0, rem - (p.num_queries - 1) - p.window);
      const unsigned char* st = ring + size_t(s) * C::kStageBytes;
      const unsigned char* ktile = st;
      const unsigned char* vtile = st + C::kTileBytes;
      const float* kscale = reinterpret_cast<const float*>(st + 2 * C::kTileBytes);
      const float* vscale = kscale + kBlockSize;

      // ---- logits (log2 units)
      float sc[C::kPasses];
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        const int t = ps * C::kTPP + tok;
        const unsigned char* row = ktile + (t * D + chunk * C::kDPL) * C::kEsz;
        float part_g[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part_g[g] = 0.0f;
        if constexpr (!C::kQuant) {
#pragma unroll
          for (int h = 0; h < C::kDPL / 8; ++h)
            fma_bf16x8<G, C::kDPL>(part_g, qr, 8 * h,
                                   *reinterpret_cast<const uint4*>(row + 16 * (h ^ sw)));
        } else if constexpr (C::kDPL == 16) {
          const uint4 w = *reinterpret_cast<const uint4*>(row);
          fma_code4<KV, G, C::kDPL>(part_g, qr, 0, w.x);
          fma_code4<KV, G, C::kDPL>(part_g, qr, 4, w.y);
          fma_code4<KV, G, C::kDPL>(part_g, qr, 8, w.z);
          fma_code4<KV, G, C::kDPL>(part_g, qr, 12, w.w);
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(row);
          fma_code4<KV, G, C::kDPL>(part_g, qr, 0, w.x);
          fma_code4<KV, G, C::kDPL>(part_g, qr, 4, w.y);
        }
        HeadReduce<G, C::kLPT / 2>::run(part_g, lane);
        float logit = part_g[0];
        if constexpr (C::kQuant) logit *= kscale[t];
        sc[ps] = visible(lim, t, p.window) ? logit : -INFINITY;
      }

      // ---- online softmax update for head g_lane
      float bm = sc[0];
#pragma unroll
      for (int ps = 1; ps < C::kPasses; ++ps) bm = fmaxf(bm, sc[ps]);
#pragma unroll
      for (int o = C::kLPT; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, o));
      const float m_new = fmaxf(m_run, bm);
      const float alpha = fast_exp2(m_run - m_new);
      m_run = m_new;
      float psum = 0.0f;
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        const int t = ps * C::kTPP + tok;
        const float pr = fast_exp2(sc[ps] - m_new);
        psum += pr;
        if (store_lane) {
          float w = pr;
          if constexpr (C::kQuant) w = (t < vt && t >= t_lo) ? pr * vscale[t] : 0.0f;
          prob[t * G + g_lane] = w;
        }
      }
      l_run = l_run * alpha + (store_lane ? psum : 0.0f);
      if (store_lane && tok == 0) prob[kBlockSize * G + g_lane] = alpha;
      __syncwarp();

      // ---- PV: acc[g][lane dims] = alpha_g * acc + sum_t p[t][g] * v[t][lane dims]
      float al[G];
#pragma unroll
      for (int g = 0; g < G; ++g) al[g] = prob[kBlockSize * G + g];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < C::kDPV; ++i) acc[g][i] *= al[g];
#pragma unroll 4
      for (int t = t_lo; t < vt; ++t) {
        float pv[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int g4 = 0; g4 < G / 4; ++g4) {
            const float4 v4 = reinterpret_cast<const float4*>(prob + t * G)[g4];
            pv[4 * g4] = v4.x; pv[4 * g4 + 1] = v4.y; pv[4 * g4 + 2] = v4.z; pv[4 * g4 + 3] = v4.w;
          }
        } else if constexpr (G == 2) {
          const float2 v2 = reinterpret_cast<const float2*>(prob + t * G)[0];
          pv[0] = v2.x; pv[1] = v2.y;
        } else {
          pv[0] = prob[t];
        }
        float vf[C::kDPV];
        const unsigned char* vrow = vtile + (t * D + lane * C::kDPV) * C::kEsz;
        if constexpr (!C::kQuant && C::kDPV == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vrow);
          vf[0] = bf16lo(w.x); vf[1] = bf16hi(w.x); vf[2] = bf16lo(w.y); vf[3] = bf16hi(w.y);
        } else if constexpr (!C::kQuant) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow);
          vf[0] = bf16lo(w); vf[1] = bf16hi(w);
        } else if constexpr (C::kDPV == 4) {
          dequant4<KV>(*reinterpret_cast<const uint32_t*>(vrow), vf);
        } else {
          float v4[4];
          dequant4<KV>(uint32_t(*reinterpret_cast<const uint16_t*>(vrow)), v4);
          vf[0] = v4[0];
          vf[1] = v4[1];
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int i = 0; i < C::kDPV; ++i) acc[g][i] = fmaf(pv[g], vf[i], acc[g][i]);
      }
    }
    __syncwarp();  // every lane is done with this stage and with `prob`
    if (k + S < nw) {
      fence_proxy_async_smem();
      issue(k + S);
    }
  }
  if (failed_at >= 0) {
    // Let the copies still in flight into this warp's ring land (bounded) before the
    // ring is reused for the merge record; their data is not used.  The CTA then takes no
    // further items.
    for (int k = failed_at; k < nw && k < failed_at + S; ++k)
      (void)mbar_wait_bounded(bars + ((kb + k) % S), ((kb + k) / S) & 1);
    if (lane == 0 && p.persistent) ss.slot[1] = 1;
    __syncwarp();
  }
  kb += failed_at >= 0 ? min(nw, failed_at + S) : nw;

  // ---- this warp's softmax sum per head, then its merge record in its ring stage 0
#pragma unroll
  for (int o = C::kLPT; o < 32; o <<= 1) l_run += __shfl_xor_sync(kFull, l_run, o);
  float* rec = reinterpret_cast<float*>(ring);  // [G][record_stride(D)]: max, sum, accumulator
  constexpr int kRec = record_stride(D);
  if (lane < C::kLPT && store_lane) {
    rec[g_lane * kRec] = m_run;
    rec[g_lane * kRec + 1] = l_run;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < C::kDPV; ++i) rec[g * kRec + 2 + lane * C::kDPV + i] = acc[g][i];
  __syncthreads();

  merge_warp_records<G, D, NW>(smem, size_t(S) * C::kStageBytes, p, b, kvh, c0, part, nparts);
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

// Merge the partitions of every split sequence: M = max_p m_p, L = sum_p 2^(m_p - M) l_p,
// out = sum_p 2^(m_p - M) acc_p / L.  One warp per (sequence, query token, query head).
template <int D>
__global__ void __launch_bounds__(128) lse_reduce_kernel(const DecodeParams p) {
  constexpr int kDPV = D / 32;
  constexpr int kAhead = 4;  // partitions whose accumulators are loaded before T is known
  constexpr uint32_t kFull = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  griddep_wait();  // the partials come from the decode kernel just before
  const int gw = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);  // row of [B, k, Hq]
  if (gw >= p.num_seqs * p.num_queries * p.num_q_heads) return;
  const int b = gw / (p.num_queries * p.num_q_heads);
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + size_t(gw) * p.max_parts;
  const float* src = p.ws_acc + size_t(gw) * p.max_parts * D + lane * kDPV;

  // The length, this lane's (m, l) and the first kAhead partitions' accumulators are all
  // requested before any of them is used, so the row costs one global-memory round trip
  // instead of three.  Slots past the row's partition count (the workspace has max_parts
  // per row) hold stale values; they are loaded but never used.
  const int T = __ldg(p.context_lens + b);
  float2 mine = make_float2(-INFINITY, 0.0f);
  if (lane < p.max_parts) mine = ml[lane];
  float v[kAhead][kDPV];
#pragma unroll
  for (int u = 0; u < kAhead; ++u) {
    if (u < p.max_parts) {
      if constexpr (kDPV == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src + size_t(u) * D);
        v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src + size_t(u) * D);
        v[u][0] = x.x; v[u][1] = x.y;
      }
    }
  }
  if (T < p.num_queries || T > p.max_context_len) return;  // the decode kernel wrote zeros
  const int nparts = seq_parts(p, T);
  if (nparts <= 1) return;  // written directly by the decode kernel
  if (lane >= nparts) mine = make_float2(-INFINITY, 0.0f);

  // Lane i holds partitions i, i + 32, ...; the weight 2^(m_p - M) of a lane's first
  // partition stays in a register for the accumulator pass.
  float M = mine.x;
  for (int i = lane + 32; i < nparts; i += 32) M = fmaxf(M, ml[i].x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float L = 0.0f;
  float a[kDPV];
#pragma unroll
  for (int i = 0; i < kDPV; ++i) a[i] = 0.0f;
  if (M != -INFINITY) {
    const float f_mine = lane < nparts ? exp2f(mine.x - M) : 0.0f;
    L = f_mine * mine.y;
    for (int i = lane + 32; i < nparts; i += 32) {
      const float2 w = ml[i];
      L = fmaf(exp2f(w.x - M), w.y, L);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const float f = __shfl_sync(kFull, f_mine, u);
      if (u < nparts) {
#pragma unroll
        for (int c = 0; c < kDPV; ++c) a[c] = fmaf(f, v[u][c], a[c]);
      }
    }
    int i = kAhead;
    for (; i + 4 <= nparts; i += 4) {  // four partitions' loads in flight
      float f[4];
      float w[4][kDPV];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pi = i + u;
        f[u] = pi < 32 ? __shfl_sync(kFull, f_mine, pi) : exp2f(ml[pi].x - M);
        if constexpr (kDPV == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + size_t(pi) * D);
          w[u][0] = x.x; w[u][1] = x.y; w[u][2] = x.z; w[u][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src + size_t(pi) * D);
          w[u][0] = x.x; w[u][1] = x.y;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < kDPV; ++c) a[c] = fmaf(f[u], w[u][c], a[c]);
    }
    for (; i < nparts; ++i) {
      const float f = i < 32 ? __shfl_sync(kFull, f_mine, i) : exp2f(ml[i].x - M);
#pragma unroll
      for (int c = 0; c < kDPV; ++c) a[c] = fmaf(f, src[size_t(i) * D + c], a[c]);
    }
  }
  auto* out = static_cast<__nv_bfloat16*>(p.out) + size_t(gw) * D + lane * kDPV;
#pragma unroll
  for (int i = 0; i < kDPV; ++i) out[i] = __float2bfloat16_rn(L > 0.0f ? a[i] / L : 0.0f);
}

// ---- launch helpers
template <KvType KV, int D, int G, int NW, int S>
cudaError_t launch_decode_variant(const DecodeParams& p, cudaStream_t stream) {
  using C = DecodeCfg<KV, D, G, NW, S>;
  auto kern = paged_decode_kernel<KV, D, G, NW, S>;
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
                    C::smem_bytes(p.partition_blocks, p.persistent ? p.num_seqs : 0), stream, p);
}

template <KvType KV, int D, int G, int NW, int S>
int ctas_per_sm_variant() {
  using C = DecodeCfg<KV, D, G, NW, S>;
  auto kern = paged_decode_kernel<KV, D, G, NW, S>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(C::smem_bytes(kMaxPartitionBlocks, kMaxSchedSeqs)));
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::kThreads, C::smem_bytes(64, 256)) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace pkv
