// Paged decode attention for sm_103a.
//
// What it computes ("vLLM ve Triton ile maliyet optimizasyonu", section 03):
// scaled dot-product attention of each sequence's single new query against
// its K/V, which the kernel gathers from scattered 16-token blocks by
// following the block table.  Grouped-query attention ("Yerel LLM
// sistemlerinde backpressure ve olcekleme", section "KV butcesi"): the G
// query heads of one KV head are processed together, so every K/V tile is
// read from HBM once per group, not once per query head.
//
// Three kernels per call, all on the caller's stream:
//   1. prep   (1 CTA)    clamps lengths, cuts every sequence into 512-token
//                        partitions, lists them (full partitions first) in
//                        the workspace and resets the work counters;
//   2. attend (persistent, two CTAs per SM)
//                        one work item = (partition, KV head).  Warp 0
//                        schedules: it takes items from an atomic counter as
//                        slots of a two-slot item ring free up and stages each
//                        item's partition record, block ids and query rows
//                        there.  Warp 1 (one thread; FP8: warps 1 and 2,
//                        alternate stages) streams each block's K and V tiles
//                        into a ring of shared-memory stages with TMA
//                        (128-byte swizzle), completion on mbarriers, without
//                        ever waiting on global memory.  Four consumer warps
//                        own the ring stages (block g of the CTA's stream to
//                        warp g % 4), each keeping an online softmax (running
//                        max and sum, fp32) for the G heads; at the end of an
//                        item each hands its state to a combiner warp, which
//                        folds the four and writes either the final output
//                        (one partition) or the partition's (max, sum,
//                        unnormalised output), while the consumers go on;
//   3. merge  (grid-stride) combines the partitions of split sequences:
//                        one CTA per (sequence, KV head), slices of
//                        partitions merged with a running maximum.
//
// Two math variants for the per-block QK^T / softmax / PV step, selected at
// run time for the A/B measurement:
//   FMA  CUDA-core fp32 FMAs; scores reduced and broadcast with warp shuffles;
//   MMA  mma.sync m16n8k16 (16 tokens x 8 heads x 16 dims): S^T = K Q^T, then
//        O^T += V^T P with P moved into operand layout by movmatrix.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

struct ItemInfo {
  int32_t b, h, p, len, nparts, nblk, g0, part, start, pad0;
  float k_scale, v_scale;  // FP8 caches: the KV head's dequantisation scales
};

// The scheduler stages each item's G query rows in shared memory, one row per
// query head, rows padded by 16 bytes so that the consumers' fragment loads
// (8 rows x 4 lanes) fall in distinct banks.
template <int D>
struct QStage {
  static constexpr int kRow = D + 8;                 // elements per staged row
  static constexpr int kChunks = D * 2 / 16;         // 16-byte chunks per row
  static constexpr int kSlotBytes = 8 * kRow * 2;    // up to G = 8 rows
};

struct DecodeParams {
  const void* q;
  void* out;
  const int32_t* tables;
  const int32_t* seq_lens;
  WsHeader* ws;
  PartInfo* parts;
  int2* seq_first;
  MergeInfo* split;
  int4* seq_prefix;   // per sequence: first prefix partial, group size, chunks, prefix tokens
  int4* group_info;   // per group: prefix partial base, item base, chunks, row tiles
  int32_t* group_bad; // per group: shared prefix rejected
  int4* pitems;       // shared-prefix work items (group, chunk, row tile)
  const int32_t* group_off;     // [num_groups + 1] or null
  const int32_t* group_prefix;  // [num_groups] or null
  int32_t num_groups;
  const float* k_scale;         // FP8 caches: per KV head dequantisation scales
  const float* v_scale;
  float2* ml;
  float* acc;
  int64_t max_parts;  // partition records the workspace holds
  int64_t max_rows;   // partial-result rows it holds (partitions + shared-prefix chunks)
  int64_t max_pitems; // shared-prefix work items it holds
  int64_t num_blocks;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t max_seq_len;
  int32_t hq, hkv, G;
  float scale_log2;
};

// ---------------------------------------------------------------------------
// 1. prep

__device__ __forceinline__ int clamp_len(const DecodeParams& P, int b) {
  int L = P.seq_lens[b];
  if (L < 0 || L > P.max_seq_len) {
    atomicOr(&P.ws->error_bits, kErrSeqLen);
    L = L < 0 ? 0 : P.max_seq_len;
  }
  return L;
}

// Exclusive scan over the 1024 threads of the block; *total = sum.

// Group of sequence b: the last g with group_off[g] <= b.
__device__ __forceinline__ int group_of(const DecodeParams& P, int b) {
  int lo = 0, hi = P.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.group_off[mid] <= b) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Partition size: the largest of 512, 1024, 2048 tokens that still leaves at
// least `target_full_items` full-partition work items, so long sequences make
// fewer partials to merge while the persistent grid stays balanced.  Partial
// (tail) partitions are ordered longest first by a counting sort on their
// size, so the dynamic work queue ends on the shortest items.
//
// Grouped decode: sequences come in contiguous groups whose members share
// their first `prefix` tokens (whole blocks).  The attention kernel then only
// covers each member's own tokens [prefix, len); the prefix is cut into
// 256-token chunks handled once per (group, KV head) by the prefix kernel for
// all members together.  A group whose prefix is not a multiple of 16 or
// longer than one of its members is flagged and decoded without sharing.
constexpr int kMergeThreads = 512;  // split merge CTA: 512 / columns thread groups share the partials
constexpr int kPrepCache = 4096;  // sequences whose (length, start) prep keeps in shared memory
// dynamic shared memory of the prep kernel: per cached sequence (length,
// first token), first full-partition record, partitions
constexpr size_t kPrepSmem = kPrepCache * (sizeof(int2) + 2 * sizeof(int));

// Threads of the prep kernel: one per sequence up to 256 (a loop over
// sequences per thread would chain their loads), 1024 beyond.  Measured on
// the 256-sequence batch: 4.7 us with 256 threads, 5.5 with 1024, 10.5 with 64.
inline int prep_threads(int num_seqs) { return num_seqs <= 256 ? 256 : 1024; }

__global__ void __launch_bounds__(1024) prep_kernel(DecodeParams P, int row_uint4,
                                                    int target_full_items, int force_pt) {
  extern __shared__ int4 prep_smem[];
  int2* s_ls = reinterpret_cast<int2*>(prep_smem);      // (clamped length, first token of the partitions)
  int* s_first = reinterpret_cast<int*>(s_ls + kPrepCache);
  int* s_np = s_first + kPrepCache;
  __shared__ int sw[32];
  __shared__ int s_full[3];
  __shared__ int s_hist[kMaxPartBlocks + 1];
  __shared__ int s_nsplit, s_total_tail, s_groups_ok;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();  // the attention kernel may set up while the plan is made
  if (tid == 0) {
    P.ws->error_bits = 0;
    s_full[0] = s_full[1] = s_full[2] = 0;
    s_nsplit = 0;
    s_groups_ok = 1;
  }
  for (int i = tid; i <= kMaxPartBlocks; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int ng = P.num_groups;
  if (ng > 0) {
    for (int g = tid; g < ng; g += blockDim.x) {
      const int a = P.group_off[g], e = P.group_off[g + 1];
      if (a < 0 || e < a || e > P.num_seqs || (g == 0 && a != 0) || (g == ng - 1 && e != P.num_seqs))
        s_groups_ok = 0;
      P.group_bad[g] = 0;
    }
  }
  if (ng > 0) __syncthreads();  // (ng is the same for every thread)
  const bool use_groups = ng > 0 && s_groups_ok;
  if (ng > 0 && !use_groups && tid == 0) atomicOr(&P.ws->error_bits, kErrGroup);
  if (use_groups) {
    for (int b = tid; b < P.num_seqs; b += blockDim.x) {
      const int g = group_of(P, b);
      const int pre = P.group_prefix[g];
      if (pre < 0 || pre % kBlock != 0 || pre > clamp_len(P, b)) {
        atomicOr(&P.group_bad[g], 1);
        atomicOr(&P.ws->error_bits, kErrGroup);
      }
    }
    __syncthreads();
    // first token of the attention kernel's partitions for each sequence,
    // kept in seq_prefix[b].w (rewritten in full in pass B)
    for (int b = tid; b < P.num_seqs; b += blockDim.x) {
      const int g = group_of(P, b);
      P.seq_prefix[b] = make_int4(g, 0, 0, P.group_bad[g] ? 0 : P.group_prefix[g]);
    }
    __syncthreads();
  }
  const bool cached = P.num_seqs <= kPrepCache;
  if (cached) {
    for (int b = tid; b < P.num_seqs; b += blockDim.x)
      s_ls[b] = make_int2(clamp_len(P, b), use_groups ? P.seq_prefix[b].w : 0);
    __syncthreads();
  }
  auto seq_len = [&](int b) -> int { return cached ? s_ls[b].x : clamp_len(P, b); };
  auto suffix_start = [&](int b) -> int {
    return cached ? s_ls[b].y : (use_groups ? P.seq_prefix[b].w : 0);
  };
  // pass A: full partitions for each candidate size
  int f1 = 0, f2 = 0, f4 = 0;
  for (int b = tid; b < P.num_seqs; b += blockDim.x) {
    const int n = seq_len(b) - suffix_start(b);
    f1 += n / kPartTokens;
    f2 += n / (2 * kPartTokens);
    f4 += n / (4 * kPartTokens);
  }
  // one shared atomic per warp: 1024 same-address atomics would serialise
  f1 = __reduce_add_sync(0xffffffffu, f1);
  f2 = __reduce_add_sync(0xffffffffu, f2);
  f4 = __reduce_add_sync(0xffffffffu, f4);
  if ((tid & 31) == 0) {
    atomicAdd(&s_full[0], f1);
    atomicAdd(&s_full[1], f2);
    atomicAdd(&s_full[2], f4);
  }
  __syncthreads();
  // force_pt (512 / 1024 / 2048, or 0 to choose) fixes the size instead
  int pt = kPartTokens, total_full = s_full[0];
  if (force_pt == 4 * kPartTokens ||
      (force_pt == 0 && static_cast<int64_t>(s_full[2]) * P.hkv >= target_full_items)) {
    pt = 4 * kPartTokens;
    total_full = s_full[2];
  } else if (force_pt == 2 * kPartTokens ||
             (force_pt == 0 && static_cast<int64_t>(s_full[1]) * P.hkv >= target_full_items)) {
    pt = 2 * kPartTokens;
    total_full = s_full[1];
  }
  // tails by size (blocks), then start offsets in descending size order
  for (int b = tid; b < P.num_seqs; b += blockDim.x) {
    const int r = (seq_len(b) - suffix_start(b)) % pt;
    if (r) atomicAdd(&s_hist[(r + kBlock - 1) / kBlock], 1);
  }
  __syncthreads();
  {  // start offsets in descending size order: a scan over the reversed bins
    const int nbins = pt / kBlock;  // <= 128
    int carry = 0;
    for (int base = 0; base < nbins; base += blockDim.x) {
      const int i = base + tid;
      const int sz = nbins - i;
      const int c = i < nbins ? s_hist[sz] : 0;
      int total;
      const int off = block_exclusive_scan(c, sw, &total);
      if (i < nbins) s_hist[sz] = carry + off;
      carry += total;
    }
    if (tid == 0) s_total_tail = carry;
  }
  __syncthreads();
  const int n_suffix = total_full + s_total_tail;
  // groups: prefix chunks, row tiles, partial and work-item bases
  int n_pitems = 0;
  if (use_groups) {
    int carry_r = 0, carry_i = 0;
    for (int base = 0; base < ng; base += blockDim.x) {
      const int g = base + tid;
      int nch = 0, M = 0, nt = 0;
      if (g < ng) {
        M = P.group_off[g + 1] - P.group_off[g];
        const int pre = P.group_bad[g] ? 0 : P.group_prefix[g];
        nch = (pre > 0 && M > 0) ? (pre + kPrefixChunkTokens - 1) / kPrefixChunkTokens : 0;
        nt = (M * P.G + kPrefixRows - 1) / kPrefixRows;
      }
      int tot_r, tot_i;
      const int ro = block_exclusive_scan(nch * M, sw, &tot_r);
      const int io = block_exclusive_scan(nch * nt, sw, &tot_i);
      if (g < ng) {
        P.group_info[g] = make_int4(n_suffix + carry_r + ro, carry_i + io, nch, nt);
        for (int c = 0; c < nch; ++c)
          for (int t = 0; t < nt; ++t) P.pitems[carry_i + io + c * nt + t] = make_int4(g, c, t, 0);
      }
      carry_r += tot_r;
      carry_i += tot_i;
    }
    n_pitems = carry_i;
  }
  __syncthreads();
  // pass B: full partitions in sequence order, tails at their sorted slots
  int carry_full = 0;
  for (int base = 0; base < P.num_seqs; base += blockDim.x) {
    const int b = base + tid;
    int L = 0, st = 0;
    if (b < P.num_seqs) {
      L = seq_len(b);
      st = suffix_start(b);
    }
    const int nfull = (L - st) / pt;
    const int r = (L - st) % pt;
    int tot_f;
    const int fo = block_exclusive_scan(nfull, sw, &tot_f);
    bool need_merge = false;
    MergeInfo mi{};
    if (b < P.num_seqs) {
      int4 sp = make_int4(0, 0, 0, st);
      if (use_groups) {
        const int g = P.seq_prefix[b].x;
        const int4 gi = P.group_info[g];
        if (gi.z > 0) {
          const int M = P.group_off[g + 1] - P.group_off[g];
          sp = make_int4(gi.x + (b - P.group_off[g]), M, gi.z, st);
        }
      }
      P.seq_prefix[b] = sp;
      const int nparts = nfull + (r != 0) + sp.z;
      const int first = carry_full + fo;
      const int tail_idx = r ? total_full + atomicAdd(&s_hist[(r + kBlock - 1) / kBlock], 1) : -1;
      P.seq_first[b] = make_int2(first, tail_idx);
      if (cached) {  // the full-partition records are written below, by every thread
        s_first[b] = first;
        s_np[b] = nparts;
      } else {
        for (int p = 0; p < nfull; ++p) P.parts[first + p] = PartInfo{b, p, L, nparts, st, 0, 0, 0};
      }
      if (r) P.parts[tail_idx] = PartInfo{b, nfull, L, nparts, st, 0, 0, 0};
      need_merge = nparts > 1 || sp.z > 0;
      mi = MergeInfo{b, first, tail_idx, nfull, nfull + (r != 0), sp.x, sp.y, sp.z};
    }
    // one shared atomic per warp for the merge-record slots
    const unsigned mm = __ballot_sync(0xffffffffu, need_merge);
    int slot0 = 0;
    if ((tid & 31) == 0 && mm) slot0 = atomicAdd(&s_nsplit, __popc(mm));
    slot0 = __shfl_sync(0xffffffffu, slot0, 0);
    if (need_merge) P.split[slot0 + __popc(mm & ((1u << (tid & 31)) - 1u))] = mi;
    carry_full += tot_f;
  }
  __syncthreads();
  if (cached) {
    // Full-partition records r = 0 .. total_full-1, consecutive threads on
    // consecutive records (coalesced): record r belongs to the last sequence
    // whose first record is <= r (sequences without full partitions share
    // the next one's first index and are passed over).
    for (int rr = tid; rr < total_full; rr += blockDim.x) {
      int lo = 0, hi = P.num_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_first[mid] <= rr) lo = mid;
        else hi = mid - 1;
      }
      const int2 ls = s_ls[lo];
      P.parts[rr] = PartInfo{lo, rr - s_first[lo], ls.x, s_np[lo], ls.y, 0, 0, 0};
    }
  }
  if (tid == 0) {
    P.ws->n_parts = n_suffix;
    P.ws->n_suffix_parts = n_suffix;
    P.ws->n_items = n_suffix * P.hkv;
    P.ws->next_item = 0;
    P.ws->n_split = s_nsplit;
    P.ws->next_split = 0;
    P.ws->part_tokens = pt;
    P.ws->n_pitems = n_pitems;
  }
}

// ---------------------------------------------------------------------------
// 2. attend

template <int D>
struct Tile {
  static constexpr int kHalfBytes = 16 * 64 * 2;             // 16 rows x 64 dims, 2048 B apart
  static constexpr int kHalves = D / 64;                     // 64-dim halves per K (or V) tile
  static constexpr int kKVBytes = kHalves * kHalfBytes;      // one K (or V) tile: one 3-D box
  static constexpr int kStageBytes = 2 * kKVBytes;           // K then V
};

// Shared-memory address of 16-byte chunk c (0 .. D/8-1) of token row r.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t tile, int r, int c) {
  return tile + (c >> 3) * 2048 + swz128(r, c & 7);
}

template <int D, int NC>
struct MergeSlot {
  float acc[NC][8][D + 4];
  float m[NC][8];
  float l[NC][8];
};

// ---- MMA math ----------------------------------------------------------------

template <typename T, int D>
struct MmaState {
  uint32_t qb[D / 16][2];
  float m[2], l[2];
  float o[D / 16][4];

  __device__ __forceinline__ void begin(const DecodeParams& P, const ItemInfo& it, int lane, float*,
                                        const T* qs) {
    const int g = lane >> 2, t = lane & 3;
    const T* q = qs + g * QStage<D>::kRow;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if (g < P.G) {
        qb[ks][0] = *reinterpret_cast<const uint32_t*>(q + 16 * ks + 2 * t);
        qb[ks][1] = *reinterpret_cast<const uint32_t*>(q + 16 * ks + 2 * t + 8);
      } else {
        qb[ks][0] = qb[ks][1] = 0u;
      }
    }
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  }

  __device__ __forceinline__ void block(uint32_t sK, uint32_t sV, int nvalid, float scale_log2,
                                        int lane, float*) {
    const int g = lane >> 2, t = lane & 3;
    float s[4];
    // S^T[token][head] = sum_d K[token][d] Q[head][d], as four independent
    // accumulation chains (the dependent mma latency of a block is then two
    // products at head_dim 128 instead of eight)
    {
      constexpr int kChains = D / 16 < 4 ? D / 16 : 4;
      float sp[kChains][4];
#pragma unroll
      for (int c = 0; c < kChains; ++c) sp[c][0] = sp[c][1] = sp[c][2] = sp[c][3] = 0.f;
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int cofs = lane >> 4;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(a0, a1, a2, a3, chunk_addr(sK, r, 2 * ks + cofs));
        Mma<T>::run(sp[ks % kChains], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float acc = sp[0][e];
#pragma unroll
        for (int c = 1; c < kChains; ++c) acc += sp[c][e];
        s[e] = acc;
      }
    }
    // s[0]: (token g, head 2t)  s[1]: (g, 2t+1)  s[2]: (g+8, 2t)  s[3]: (g+8, 2t+1)
    const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
    const float x0 = v0 ? s[0] * scale_log2 : -INFINITY;
    const float x1 = v0 ? s[1] * scale_log2 : -INFINITY;
    const float x2 = v1 ? s[2] * scale_log2 : -INFINITY;
    const float x3 = v1 ? s[3] * scale_log2 : -INFINITY;
    // Lazy rescaling: the reference maximum m moves only when some score of
    // the block exceeds it by more than 2^8 (log2 units), so the weights
    // stay below 256 -- inside the range of the 16-bit P operand -- and most
    // blocks need neither the block maximum (a shuffle reduction over the
    // token rows) nor the rescale of l and o.  Exact either way: l and o are
    // always relative to the same m.  Each lane tests its own scores; the
    // decision is a vote over the warp.
    float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
    if (__any_sync(0xffffffffu, bm0 > m[0] + 8.f || bm1 > m[1] + 8.f)) {
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {  // block maximum (finite: nvalid >= 1)
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o2));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o2));
      }
      const float mn0 = fmaxf(m[0], bm0), mn1 = fmaxf(m[1], bm1);
      const float al0 = exp2f(m[0] - mn0), al1 = exp2f(m[1] - mn1);
      l[0] *= al0;
      l[1] *= al1;
      m[0] = mn0;
      m[1] = mn1;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    const float p0 = exp2f(x0 - m[0]), p1 = exp2f(x1 - m[1]);
    const float p2 = exp2f(x2 - m[0]), p3 = exp2f(x3 - m[1]);
    l[0] += p0 + p2;
    l[1] += p1 + p3;
    // P[token][head] (accumulator layout) -> B operand (token = k, head = n)
    const uint32_t b0 = movmatrix_trans(pack2<T>(p0, p1));
    const uint32_t b1 = movmatrix_trans(pack2<T>(p2, p3));
    const int r = (lane & 7) + (lane >> 4) * 8;
    const int cofs = (lane >> 3) & 1;
    if (nvalid == 16) {  // a full block: every V row is a token
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(a0, a1, a2, a3, chunk_addr(sV, r, 2 * mt + cofs));
        Mma<T>::run(o[mt], a0, a1, a2, a3, b0, b1);
      }
    } else {
      // Rows past the sequence end may hold anything (NaN included): zero
      // them in the V operand so 0 * garbage cannot reach the sum.
      const uint32_t mk0 = (2 * t < nvalid ? 0x0000ffffu : 0u) | (2 * t + 1 < nvalid ? 0xffff0000u : 0u);
      const uint32_t mk1 = (2 * t + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * t + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(a0, a1, a2, a3, chunk_addr(sV, r, 2 * mt + cofs));
        Mma<T>::run(o[mt], a0 & mk0, a1 & mk0, a2 & mk1, a3 & mk1, b0, b1);
      }
    }
  }

  template <int NC>
  __device__ __forceinline__ void store(MergeSlot<D, NC>& ms, int w, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float L0 = l[0], L1 = l[1];
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
      L0 += __shfl_xor_sync(0xffffffffu, L0, o2);
      L1 += __shfl_xor_sync(0xffffffffu, L1, o2);
    }
    if (g == 0) {
      ms.m[w][2 * t] = m[0];
      ms.m[w][2 * t + 1] = m[1];
      ms.l[w][2 * t] = L0;
      ms.l[w][2 * t + 1] = L1;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      ms.acc[w][2 * t][16 * mt + g] = o[mt][0];
      ms.acc[w][2 * t + 1][16 * mt + g] = o[mt][1];
      ms.acc[w][2 * t][16 * mt + g + 8] = o[mt][2];
      ms.acc[w][2 * t + 1][16 * mt + g + 8] = o[mt][3];
    }
  }
};

// ---- FMA math ----------------------------------------------------------------
// QK lanes: token = lane & 15, head half = lane >> 4 (HPG heads each).
// PV lanes: 16-byte chunk c = lane % (D/8), head group = lane / (D/8).
// Per-warp scratch (fp32): q[8][D] scaled by scale*log2(e), p[8][16], alpha[8].

template <int D>
struct FmaScratch {
  static constexpr int kFloats = 8 * D + 8 * 16 + 8;
};

template <typename T, int D, int HPG>
struct FmaState {
  static constexpr int kChunks = D / 8;
  static constexpr int kGroups = 32 / kChunks;                 // PV head groups
  static constexpr int HPV = (HPG * 2 + kGroups - 1) / kGroups;  // PV heads per lane
  float m[HPG], l[HPG];
  float acc[HPV][8];
  int G;

  __device__ __forceinline__ void begin(const DecodeParams& P, const ItemInfo& it, int lane,
                                        float* scr, const T* qs) {
    G = P.G;
    for (int e = lane; e < P.G * D; e += 32)
      scr[e] = to_float<T>(qs[(e / D) * QStage<D>::kRow + e % D]) * P.scale_log2;
#pragma unroll
    for (int j = 0; j < HPG; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < HPV; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    __syncwarp();
  }

  __device__ __forceinline__ void block(uint32_t sK, uint32_t sV, int nvalid, float,
                                        int lane, float* scr) {
    float* qs = scr;
    float* ps = scr + 8 * D;
    float* as = ps + 8 * 16;
    const int tok = lane & 15, hh = lane >> 4;
    float s[HPG];
#pragma unroll
    for (int j = 0; j < HPG; ++j) s[j] = 0.f;
#pragma unroll 4
    for (int c = 0; c < kChunks; ++c) {
      uint4 kv;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(kv.x), "=r"(kv.y), "=r"(kv.z), "=r"(kv.w)
                   : "r"(chunk_addr(sK, tok, c)));
      const float2 k0 = unpack2<T>(kv.x), k1 = unpack2<T>(kv.y);
      const float2 k2 = unpack2<T>(kv.z), k3 = unpack2<T>(kv.w);
#pragma unroll
      for (int j = 0; j < HPG; ++j) {
        const int head = hh * HPG + j;
        if (head < G) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + head * D + 8 * c);
          const float4 qc = *reinterpret_cast<const float4*>(qs + head * D + 8 * c + 4);
          float a = s[j];
          a = fmaf(qa.x, k0.x, a);
          a = fmaf(qa.y, k0.y, a);
          a = fmaf(qa.z, k1.x, a);
          a = fmaf(qa.w, k1.y, a);
          a = fmaf(qc.x, k2.x, a);
          a = fmaf(qc.y, k2.y, a);
          a = fmaf(qc.z, k3.x, a);
          a = fmaf(qc.w, k3.y, a);
          s[j] = a;
        }
      }
    }
    const bool valid = tok < nvalid;
#pragma unroll
    for (int j = 0; j < HPG; ++j) {
      const int head = hh * HPG + j;
      float x = valid ? s[j] : -INFINITY;
      float bm = x;
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o2));
      const float mn = fmaxf(m[j], bm);
      const float al = exp2f(m[j] - mn);
      const float p = exp2f(x - mn);
      l[j] = l[j] * al + p;
      m[j] = mn;
      if (head < G) {
        ps[head * 16 + tok] = p;
        if (tok == 0) as[head] = al;
      }
    }
    __syncwarp();
    const int c = lane % kChunks, hg = lane / kChunks;
#pragma unroll
    for (int j = 0; j < HPV; ++j) {
      const int head = hg * HPV + j;
      if (head < G) {
        const float al = as[head];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] *= al;
      }
    }
    for (int r = 0; r < nvalid; ++r) {
      uint4 vv;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(vv.x), "=r"(vv.y), "=r"(vv.z), "=r"(vv.w)
                   : "r"(chunk_addr(sV, r, c)));
      const float2 v0 = unpack2<T>(vv.x), v1 = unpack2<T>(vv.y);
      const float2 v2 = unpack2<T>(vv.z), v3 = unpack2<T>(vv.w);
#pragma unroll
      for (int j = 0; j < HPV; ++j) {
        const int head = hg * HPV + j;
        if (head < G) {
          const float p = ps[head * 16 + r];
          acc[j][0] = fmaf(p, v0.x, acc[j][0]);
          acc[j][1] = fmaf(p, v0.y, acc[j][1]);
          acc[j][2] = fmaf(p, v1.x, acc[j][2]);
          acc[j][3] = fmaf(p, v1.y, acc[j][3]);
          acc[j][4] = fmaf(p, v2.x, acc[j][4]);
          acc[j][5] = fmaf(p, v2.y, acc[j][5]);
          acc[j][6] = fmaf(p, v3.x, acc[j][6]);
          acc[j][7] = fmaf(p, v3.y, acc[j][7]);
        }
      }
    }
    __syncwarp();
  }

  template <int NC>
  __device__ __forceinline__ void store(MergeSlot<D, NC>& ms, int w, int lane) {
    const int tok = lane & 15, hh = lane >> 4;
#pragma unroll
    for (int j = 0; j < HPG; ++j) {
      float L = l[j];
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
      const int head = hh * HPG + j;
      if (tok == 0 && head < 8) {
        ms.m[w][head] = head < G ? m[j] : -INFINITY;
        ms.l[w][head] = head < G ? L : 0.f;
      }
    }
    const int c = lane % kChunks, hg = lane / kChunks;
#pragma unroll
    for (int j = 0; j < HPV; ++j) {
      const int head = hg * HPV + j;
      if (head < G) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ms.acc[w][head][8 * c + e] = acc[j][e];
      }
    }
  }
};

// ---- FP8 math ------------------------------------------------------------------
// Caches hold E4M3 bytes: K tiles [16 tokens][D] (128-byte swizzle), V tiles
// dimension-major [D][16 tokens].  ldmatrix on byte rows hands each lane four
// consecutive bytes per 8x8 matrix of 16-bit cells; cvt.f16x2.e4m3x2 turns
// them into fp16 exactly.  The four bytes land on the mma fragment slots
// (k = 2t, 2t+1, 2t+8, 2t+9), so both reductions run in a permuted order:
//   QK: k slot (2t, 2t+1, 2t+8, 2t+9) <-> head_dim (4t .. 4t+3) of the 16-dim
//       step; q is loaded in that order.  A-row r of the K operand is token
//       sigma(r) (chosen by the ldmatrix row addresses), sigma = (0 1 4 5 8 9
//       12 13 | 2 3 6 7 10 11 14 15), so that after movmatrix the P operand's
//       k slots hold tokens 4t .. 4t+3 --
//   PV: exactly the tokens the V rows deliver in those slots.
// The scales fold in: scores use scale * k_scale[h], outputs are * v_scale[h].

__device__ __forceinline__ int fp8_sigma(int r) {
  return r < 8 ? 4 * (r >> 1) + (r & 1) : 4 * ((r - 8) >> 1) + 2 + (r & 1);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T, int D>
struct Fp8State {
  uint32_t qb[D / 16][2];
  float m[2], l[2];
  float o[D / 16][4];
  float sl, vs;

  __device__ __forceinline__ void begin(const DecodeParams& P, const ItemInfo& it, int lane, float*,
                                        const T* qs) {
    const int g = lane >> 2, t = lane & 3;
    const T* q = qs + g * QStage<D>::kRow;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if (g < P.G) {
        const uint2 w = *reinterpret_cast<const uint2*>(q + 16 * ks + 4 * t);
        const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y);
        qb[ks][0] = pack_half2(a.x, a.y);
        qb[ks][1] = pack_half2(b.x, b.y);
      } else {
        qb[ks][0] = qb[ks][1] = 0u;
      }
    }
    sl = P.scale_log2 * it.k_scale;
    vs = it.v_scale;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  }

  __device__ __forceinline__ void block(uint32_t sK, uint32_t sV, int nvalid, float, int lane,
                                        float*) {
    const int g = lane >> 2, t = lane & 3;
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    {
      // four independent accumulation chains (one per 32-dim step) keep the
      // dependent mma latency of a block to one product
      float sp[D / 32][4];
      const int tok = fp8_sigma((lane & 7) + 8 * ((lane >> 3) & 1));
      const int cofs = lane >> 4;
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(r0, r1, r2, r3, sK + swz128(tok, 2 * kk + cofs));
        uint32_t a0, a2, a1, a3, b0, b2, b1, b3;
        e4m3x4_to_half2x2(r0, &a0, &a2);
        e4m3x4_to_half2x2(r1, &a1, &a3);
        e4m3x4_to_half2x2(r2, &b0, &b2);
        e4m3x4_to_half2x2(r3, &b1, &b3);
        sp[kk][0] = sp[kk][1] = sp[kk][2] = sp[kk][3] = 0.f;
        Mma<__half>::run(sp[kk], a0, a1, a2, a3, qb[2 * kk][0], qb[2 * kk][1]);
        Mma<__half>::run(sp[kk], b0, b1, b2, b3, qb[2 * kk + 1][0], qb[2 * kk + 1][1]);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) s[c] = (sp[0][c] + sp[1][c]) + (sp[2][c] + sp[3][c]);
    }
    const bool v0 = fp8_sigma(g) < nvalid, v1 = fp8_sigma(g + 8) < nvalid;
    const float x0 = v0 ? s[0] * sl : -INFINITY;
    const float x1 = v0 ? s[1] * sl : -INFINITY;
    const float x2 = v1 ? s[2] * sl : -INFINITY;
    const float x3 = v1 ? s[3] * sl : -INFINITY;
    // Lazy rescaling, as for the 16-bit caches: the reference maximum m
    // moves only when some score of the block exceeds it by more than 2^8,
    // so the weights stay below 256 (inside the fp16 P operand's range) and
    // most blocks need neither the block maximum nor the rescale of l and o.
    // Each lane tests its own scores; the decision is a vote over the warp.
    float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
    if (__any_sync(0xffffffffu, bm0 > m[0] + 8.f || bm1 > m[1] + 8.f)) {
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {  // block maximum
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o2));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o2));
      }
      const float mn0 = fmaxf(m[0], bm0), mn1 = fmaxf(m[1], bm1);
      const float al0 = exp2f(m[0] - mn0), al1 = exp2f(m[1] - mn1);
      l[0] *= al0;
      l[1] *= al1;
      m[0] = mn0;
      m[1] = mn1;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    const float p0 = exp2f(x0 - m[0]), p1 = exp2f(x1 - m[1]);
    const float p2 = exp2f(x2 - m[0]), p3 = exp2f(x3 - m[1]);
    l[0] += p0 + p2;
    l[1] += p1 + p3;
    const uint32_t b0 = movmatrix_trans(pack_half2(p0, p1));
    const uint32_t b1 = movmatrix_trans(pack_half2(p2, p3));
    const int row = (lane & 7) + 8 * ((lane >> 3) & 1) + 16 * (lane >> 4);
    if (nvalid == 16) {  // a full block: every V row is a token
#pragma unroll
      for (int mm = 0; mm < D / 32; ++mm) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(r0, r1, r2, r3, sV + (32 * mm + row) * 16);
        uint32_t a0, a2, a1, a3, c0, c2, c1, c3;
        e4m3x4_to_half2x2(r0, &a0, &a2);
        e4m3x4_to_half2x2(r1, &a1, &a3);
        e4m3x4_to_half2x2(r2, &c0, &c2);
        e4m3x4_to_half2x2(r3, &c1, &c3);
        Mma<__half>::run(o[2 * mm], a0, a1, a2, a3, b0, b1);
        Mma<__half>::run(o[2 * mm + 1], c0, c1, c2, c3, b0, b1);
      }
    } else {
      // Rows past the sequence end may hold anything (NaN included): zero
      // them in the operand so 0 * garbage cannot reach the sum.
      const uint32_t mk0 = (4 * t < nvalid ? 0x0000ffffu : 0u) | (4 * t + 1 < nvalid ? 0xffff0000u : 0u);
      const uint32_t mk1 = (4 * t + 2 < nvalid ? 0x0000ffffu : 0u) | (4 * t + 3 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
      for (int mm = 0; mm < D / 32; ++mm) {
        uint32_t r0, r1, r2, r3;
        ldmatrix_x4(r0, r1, r2, r3, sV + (32 * mm + row) * 16);
        uint32_t a0, a2, a1, a3, c0, c2, c1, c3;
        e4m3x4_to_half2x2(r0, &a0, &a2);
        e4m3x4_to_half2x2(r1, &a1, &a3);
        e4m3x4_to_half2x2(r2, &c0, &c2);
        e4m3x4_to_half2x2(r3, &c1, &c3);
        Mma<__half>::run(o[2 * mm], a0 & mk0, a1 & mk0, a2 & mk1, a3 & mk1, b0, b1);
        Mma<__half>::run(o[2 * mm + 1], c0 & mk0, c1 & mk0, c2 & mk1, c3 & mk1, b0, b1);
      }
    }
  }

  template <int NC>
  __device__ __forceinline__ void store(MergeSlot<D, NC>& ms, int w, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float L0 = l[0], L1 = l[1];
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
      L0 += __shfl_xor_sync(0xffffffffu, L0, o2);
      L1 += __shfl_xor_sync(0xffffffffu, L1, o2);
    }
    if (g == 0) {
      ms.m[w][2 * t] = m[0];
      ms.m[w][2 * t + 1] = m[1];
      ms.l[w][2 * t] = L0;
      ms.l[w][2 * t + 1] = L1;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      ms.acc[w][2 * t][16 * mt + g] = o[mt][0] * vs;
      ms.acc[w][2 * t + 1][16 * mt + g] = o[mt][1] * vs;
      ms.acc[w][2 * t][16 * mt + g + 8] = o[mt][2] * vs;
      ms.acc[w][2 * t + 1][16 * mt + g + 8] = o[mt][3] * vs;
    }
  }
};

constexpr size_t align_up_c(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <typename T, int D, int NC, int S, bool kFma, bool kFp8 = false>
struct AttendCfg {
  static_assert(S % NC == 0, "within an item, each ring stage must be consumed by one warp");
  // copy warps: FP8 stages (4 KB as two 2 KB boxes) drain faster than one
  // thread issues their copies, so two warps issue alternate stages
  static constexpr int kIss = kFp8 ? 2 : 1;
  static_assert(S % kIss == 0, "each ring stage must be refilled by one copy warp");
  // scheduler, copy warps, NC consumers, combiner
  static constexpr int kThreads = 32 * (NC + 2 + kIss);
  static_assert((NC & (NC - 1)) == 0 && NC * 8 <= 32, "the combiner holds one lane per (residue, head)");
  static constexpr int kKBytes = kFp8 ? kBlock * D : Tile<D>::kKVBytes;  // K part of a stage
  static constexpr int kStageBytes = kFp8 ? 2 * kBlock * D : Tile<D>::kStageBytes;
  static constexpr size_t kStagesOff = 0;
  static constexpr size_t kMergeOff = static_cast<size_t>(S) * kStageBytes;
  static constexpr size_t kScrOff = kMergeOff + 2 * sizeof(MergeSlot<D, NC>);
  static constexpr size_t kScrBytes = kFma ? NC * FmaScratch<D>::kFloats * sizeof(float) : 0;
  static constexpr size_t kBarOff = align_up_c(kScrOff + kScrBytes, 16);
  // full[S], empty[S], item_full[2], item_empty[2], merge_full[2], merge_empty[2]
  static constexpr size_t kInfoOff = kBarOff + (2 * S + 8) * sizeof(uint64_t);
  static constexpr size_t kIdsOff = kInfoOff + 2 * sizeof(ItemInfo);
  static constexpr size_t kQOff = kIdsOff + 2 * kMaxPartBlocks * sizeof(int32_t);
  static constexpr size_t kAbortOff = kQOff + 2 * QStage<D>::kSlotBytes;
  static_assert(kQOff % 16 == 0 && QStage<D>::kSlotBytes % 16 == 0, "16-byte staged query rows");
  static constexpr size_t kBytes = kAbortOff + 16 + 1024;  // + slack to 1024-align the base
};

template <typename T, int D, int NC, int S, bool kFma, int HPG, bool kFp8>
__device__ __forceinline__ void attend_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                            const DecodeParams& P) {
  using Cfg = AttendCfg<T, D, NC, S, kFma, kFp8>;
  using State = typename std::conditional<
      kFp8, Fp8State<T, D>,
      typename std::conditional<kFma, FmaState<T, D, HPG>, MmaState<T, D>>::type>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem + Cfg::kStagesOff;
  MergeSlot<D, NC>* merge = reinterpret_cast<MergeSlot<D, NC>*>(smem + Cfg::kMergeOff);
  float* scratch = reinterpret_cast<float*>(smem + Cfg::kScrOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  uint64_t* empty = full + S;
  uint64_t* item_full = empty + S;
  uint64_t* item_empty = item_full + 2;
  uint64_t* merge_full = item_empty + 2;
  uint64_t* merge_empty = merge_full + 2;
  ItemInfo* info = reinterpret_cast<ItemInfo*>(smem + Cfg::kInfoOff);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + Cfg::kIdsOff);
  uint8_t* qstage = smem + Cfg::kQOff;  // two slots of staged query rows
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kAbortOff);
  int* err = &P.ws->error_bits;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&item_full[s], 1);
      mbar_init(&item_empty[s], NC + Cfg::kIss + 1);  // consumers, copy threads, combiner
      mbar_init(&merge_full[s], NC);
      mbar_init(&merge_empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  pdl_wait();               // the plan, q and the caches are ready from here on

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler
    // Takes work items from the atomic counter as item-ring slots free up and
    // stages each item's partition record, block ids and query rows there, so
    // the TMA warp never waits on global memory between items.  The plan may be one a
    // caller reuses from an earlier call (PA_DECODE_REUSE_PLAN), so it is not
    // trusted: an item count beyond the workspace's capacity is cut, a record
    // that is not a partition of this call's sequences is skipped, and a
    // length that differs from seq_lens marks the plan stale; each is flagged
    // (kErrPlan) and no index leaves its buffer.
    // The first item is blockIdx.x: its record is loaded together with the
    // header (one round trip at the kernel's start, not two; the grid is at
    // most the workspace's item capacity, so the record is inside it).
    const int4* rec0 = reinterpret_cast<const int4*>(P.parts + static_cast<int>(blockIdx.x) / P.hkv);
    const int4 r0a = __ldcg(rec0), r0b = __ldcg(rec0 + 1);
    const int pt = *reinterpret_cast<volatile int32_t*>(&P.ws->part_tokens);
    const bool pt_ok = pt == kPartTokens || pt == 2 * kPartTokens || pt == 4 * kPartTokens;
    int32_t n_items = *reinterpret_cast<volatile int32_t*>(&P.ws->n_items);
    if (!pt_ok || n_items < 0 || n_items > P.max_parts * P.hkv) {
      if (lane == 0) atomicOr(err, kErrPlan);
      n_items = pt_ok ? static_cast<int32_t>(min(static_cast<int64_t>(max(n_items, 0)),
                                                 P.max_parts * P.hkv))
                      : 0;
    }
    uint32_t g = 0;  // blocks of this CTA's stream before the next item
    // Item blockIdx.x is this CTA's first (no atomic on the critical path of
    // the kernel's start); the work counter hands out the rest from gridDim.x.
    bool first = true;
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&item_empty[slot], ((it >> 1) & 1) ^ 1, abort_flag, err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      int item, part = 0, h = 0, first_tok = 0, nblk = 0;
      PartInfo pi;
      for (;;) {  // the next item whose record is a partition of this call
        // claimed only now that its slot is free: near the end of the queue a
        // CTA then holds one item fewer than it would claiming one ahead
        int claimed = 0;
        if (lane == 0) {
          if (first) {
            claimed = static_cast<int>(blockIdx.x);
          } else {
            const int r = atomicAdd(&P.ws->next_item, 1);
            // a counter the last call did not leave at 0 never yields a
            // wrapped index (a negative one is flagged below)
            claimed = r < 0 ? -1 : (r > INT32_MAX - static_cast<int>(gridDim.x) ? n_items
                                                                             : static_cast<int>(gridDim.x) + r);
          }
        }
        first = false;
        item = __shfl_sync(0xffffffffu, claimed, 0);
        if (item < 0) {  // the work counter itself was not reset: no item is taken
          if (lane == 0) atomicOr(err, kErrPlan);
          item = n_items;
        }
        if (item >= n_items) break;
        part = item / P.hkv;
        h = item - part * P.hkv;
        if (it == 0 && item == static_cast<int>(blockIdx.x))
          pi = PartInfo{r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
        else
          pi = P.parts[part];
        const int64_t ft = static_cast<int64_t>(pi.start) + static_cast<int64_t>(pi.p) * pt;
        if (pi.b >= 0 && pi.b < P.num_seqs && pi.len > 0 && pi.len <= P.max_seq_len &&
            pi.start >= 0 && pi.start % kBlock == 0 && pi.p >= 0 && pi.nparts >= 1 && ft < pi.len) {
          first_tok = static_cast<int>(ft);
          nblk = min(pt / kBlock, (pi.len - first_tok + kBlock - 1) / kBlock);
          break;
        }
        if (lane == 0) atomicOr(err, kErrPlan);
      }
      if (item >= n_items) {
        if (lane == 0) {
          info[slot].b = -1;
          mbar_arrive(&item_full[slot]);
          // The merge kernel may be scheduled once every CTA's queue is empty
          // (it waits for this grid before reading anything).  Not earlier:
          // its CTAs would sit resident beside this kernel's CTAs through the
          // whole stream and slow them down.
          pdl_launch_dependents();
        }
        break;
      }
      // the item's block ids, its G query rows and (FP8) the KV head's
      // scales: every load issued before any store, one round trip in all
      const int32_t* trow = P.tables + static_cast<int64_t>(pi.b) * P.max_blocks + first_tok / kBlock;
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          static_cast<const T*>(P.q) + (static_cast<int64_t>(pi.b) * P.hq + h * P.G) * D);
      const int nq = P.G * QStage<D>::kChunks;
      constexpr int kIdIt = kMaxPartBlocks / 32, kQIt = 8 * QStage<D>::kChunks / 32;
      int32_t idv[kIdIt];
      uint4 qv[kQIt];
#pragma unroll
      for (int k = 0; k < kIdIt; ++k) {
        const int j = lane + 32 * k;
        idv[k] = j < nblk ? trow[j] : 0;
      }
#pragma unroll
      for (int k = 0; k < kQIt; ++k) {
        const int c = lane + 32 * k;
        if (c < nq) qv[k] = qsrc[c];
      }
      float ksc = 0.f, vsc = 0.f;
      if (kFp8 && lane == 0) {
        ksc = P.k_scale[h];
        vsc = P.v_scale[h];
      }
#pragma unroll
      for (int k = 0; k < kIdIt; ++k) {
        const int j = lane + 32 * k;
        if (j < nblk) {
          int32_t id = idv[k];
          if (id < 0 || id >= P.num_blocks) {
            atomicOr(err, kErrBlockId);
            id = -1;
          }
          ids[slot * kMaxPartBlocks + j] = id;
        }
      }
      uint8_t* qdst = qstage + slot * QStage<D>::kSlotBytes;
#pragma unroll
      for (int k = 0; k < kQIt; ++k) {
        const int c = lane + 32 * k;
        if (c < nq) {
          const int row = c / QStage<D>::kChunks, ch = c - row * QStage<D>::kChunks;
          *reinterpret_cast<uint4*>(qdst + row * QStage<D>::kRow * 2 + ch * 16) = qv[k];
        }
      }
      __syncwarp();
      if (lane == 0) {
        info[slot] = ItemInfo{pi.b, h, pi.p, pi.len, pi.nparts, nblk, static_cast<int32_t>(g), part,
                              pi.start, 0, ksc, vsc};
        mbar_arrive(&item_full[slot]);
        // a plan made for other lengths is flagged (after the item is out: the
        // check costs a global load the copies need not wait for)
        int L = P.seq_lens[pi.b];
        L = L < 0 ? 0 : min(L, P.max_seq_len);
        if (L != pi.len) atomicOr(err, kErrPlan);
      }
      g += nblk;
    }
    return;
  }

  if (warp <= Cfg::kIss) {
    // ---------------------------------------------------------------- TMA
    // One thread per copy warp streams the blocks into the stage ring; with
    // two copy warps, warp 1 + i issues the blocks g with g % 2 == i of the
    // CTA's block stream, so each stage is refilled by one thread, in order.
    if (lane != 0) return;
    const uint32_t iss = static_cast<uint32_t>(warp - 1);
    const int64_t y_oob = P.num_blocks * P.hkv * kBlock;  // one past the pool: reads as zeros
    uint32_t g = 0;  // blocks issued by this CTA
    bool ok = true;
    for (uint32_t it = 0; ok; ++it) {
      const int slot = it & 1;
      ok = mbar_wait(&item_full[slot], (it >> 1) & 1, abort_flag, err);
      if (!ok) break;
      const ItemInfo inf = info[slot];
      if (inf.b < 0) {
        mbar_arrive(&item_empty[slot]);
        break;
      }
      for (int j = 0; j < inf.nblk; ++j, ++g) {
        if (g % Cfg::kIss != iss) continue;  // the other copy warp's stage
        const int st = g % S;
        ok = mbar_wait(&empty[st], ((g / S) & 1) ^ 1, abort_flag, err);
        if (!ok) break;
        const int32_t id = ids[slot * kMaxPartBlocks + j];
        const int32_t y = static_cast<int32_t>(id < 0 ? y_oob : (static_cast<int64_t>(id) * P.hkv + inf.h) * kBlock);
        uint8_t* dst = stages + static_cast<size_t>(st) * Cfg::kStageBytes;
        mbar_arrive_expect_tx(&full[st], Cfg::kStageBytes);
        if constexpr (kFp8) {
          // K and V tiles: one box of 16 rows x D bytes each (V's rows are
          // groups of D/16 dimensions of 16 tokens)
          tma_load_2d(dst, &tm_k, 0, y, &full[st]);
          tma_load_2d(dst + Cfg::kKBytes, &tm_v, 0, y, &full[st]);
        } else {
          // one 3-D box per K (V) tile: both 64-dim halves
          tma_load_3d(dst, &tm_k, 0, y, 0, &full[st]);
          tma_load_3d(dst + Tile<D>::kKVBytes, &tm_v, 0, y, 0, &full[st]);
        }
      }
      if (ok) mbar_arrive(&item_empty[slot]);
    }
    if (!ok) {
      // Abort: let the copies this CTA issued land before it exits.
      const uint32_t lo = g > static_cast<uint32_t>(S) ? g - S : 0;
      for (uint32_t k = lo; k < g; ++k) {
        if (k % Cfg::kIss != iss) continue;
        unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&full[k % S], (k / S) & 1) &&
               global_timer_ns() - t0 < kWaitLimitNs / 4) {
        }
      }
    }
    return;
  }

  if (warp == Cfg::kIss + 1 + NC) {
    // ------------------------------------------------------------ combiner
    // Folds the NC consumer states of each item, in item order, into the
    // output (one partition) or the partition's (max, sum, unnormalised
    // output); the consumers meanwhile go on with the next item.  Residue
    // class k of the item's blocks (j % NC == k) was summed by consumer
    // (g0 + k) % NC; the classes are folded in the order k = 0 .. NC-1, so the
    // arithmetic does not depend on where the item fell in the CTA's stream.
    const int G = P.G;
    for (uint32_t it = 0;; ++it) {
      const int slot = it & 1;
      bool ok = mbar_wait(&item_full[slot], (it >> 1) & 1, abort_flag, err);
      if (!__all_sync(0xffffffffu, ok)) break;
      const ItemInfo inf = info[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      if (inf.b < 0) break;
      ok = mbar_wait(&merge_full[slot], (it >> 1) & 1, abort_flag, err);
      if (!__all_sync(0xffffffffu, ok)) break;
      const MergeSlot<D, NC>& ms = merge[slot];
      // lane (k, hd) = (lane >> 3, lane & 7): residue class k's maximum and sum
      // for head hd; the head's largest maximum, the class weights and the
      // sum over the classes (in class order) by lane (0, hd)
      const int kk = lane >> 3, hh = lane & 7;
      const int wk_slot = static_cast<int>((static_cast<uint32_t>(inf.g0) + kk) & (NC - 1));
      const float mk = (kk < NC && hh < G) ? ms.m[wk_slot][hh] : -INFINITY;
      const float lk = (kk < NC && hh < G) ? ms.l[wk_slot][hh] : 0.f;
      float wts[NC];
      float M = -INFINITY, Lsum = 0.f;
#pragma unroll
      for (int k = 0; k < NC; ++k) M = fmaxf(M, __shfl_sync(0xffffffffu, mk, k * 8 + hh));
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        wts[k] = exp2f(__shfl_sync(0xffffffffu, mk, k * 8 + hh) - M);
        Lsum = fmaf(__shfl_sync(0xffffffffu, lk, k * 8 + hh), wts[k], Lsum);
      }
      const int head0 = inf.h * G;
      const bool single = inf.nparts == 1;
      const uint64_t pol_last = l2_policy_evict_last();  // the merge reads the partials back
      constexpr int kD4 = D / 4;
      for (int base = 0; base < G * kD4; base += 32) {  // whole warp each round (shuffles)
        const int idx = base + lane;
        const int hd = min(idx / kD4, G - 1), d4 = idx - (idx / kD4) * kD4;
        const float Mh = __shfl_sync(0xffffffffu, M, hd);
        const float Lh = __shfl_sync(0xffffffffu, Lsum, hd);
        float wh[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) wh[k] = __shfl_sync(0xffffffffu, wts[k], hd);
        if (idx >= G * kD4) continue;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          const int ws = static_cast<int>((static_cast<uint32_t>(inf.g0) + k) & (NC - 1));
          const float4 a = *reinterpret_cast<const float4*>(&ms.acc[ws][hd][4 * d4]);
          O.x = fmaf(a.x, wh[k], O.x);
          O.y = fmaf(a.y, wh[k], O.y);
          O.z = fmaf(a.z, wh[k], O.z);
          O.w = fmaf(a.w, wh[k], O.w);
        }
        const int64_t row = static_cast<int64_t>(inf.b) * P.hq + head0 + hd;
        if (single) {
          uint2 pk;
          pk.x = pack2<T>(O.x / Lh, O.y / Lh);
          pk.y = pack2<T>(O.z / Lh, O.w / Lh);
          *reinterpret_cast<uint2*>(static_cast<T*>(P.out) + row * D + 4 * d4) = pk;
        } else {
          const int64_t prow = static_cast<int64_t>(inf.part) * P.hq + head0 + hd;
          st_global_hint(reinterpret_cast<float4*>(P.acc + prow * D + 4 * d4), O, pol_last);
          if (d4 == 0) P.ml[prow] = make_float2(Mh, Lh);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&merge_empty[slot]);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int w = warp - 1 - Cfg::kIss;
  const int pt = *reinterpret_cast<volatile int32_t*>(&P.ws->part_tokens);
  float* scr = scratch + (kFma ? w * FmaScratch<D>::kFloats : 0);
  State st;
  for (uint32_t it = 0;; ++it) {
    const int slot = it & 1;
    bool ok = mbar_wait(&item_full[slot], (it >> 1) & 1, abort_flag, err);
    if (!__all_sync(0xffffffffu, ok)) break;
    const ItemInfo inf = info[slot];
    // the staged query rows are read before the slot is handed back
    if (inf.b >= 0)
      st.begin(P, inf, lane, scr,
               reinterpret_cast<const T*>(qstage + slot * QStage<D>::kSlotBytes));
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[slot]);
    if (inf.b < 0) break;

    bool alive = true;
    // Block g of the CTA's stream goes to consumer g % NC: with S a multiple
    // of NC every ring stage has one consumer, which waits for each of its
    // rounds only after releasing the one before, so a parity wait can never
    // be satisfied by an older phase of its stage, and no barrier between
    // items is needed.  Within an item the blocks j with j % NC == k (one
    // residue class) are summed by one warp in order, whichever warp it is.
    const int j0 = static_cast<int>((static_cast<uint32_t>(w) - static_cast<uint32_t>(inf.g0)) & (NC - 1));
    for (int j = j0; j < inf.nblk; j += NC) {
      const uint32_t gg = inf.g0 + j;
      const int s = gg % S;
      ok = mbar_wait(&full[s], (gg / S) & 1, abort_flag, err);
      if (!__all_sync(0xffffffffu, ok)) {
        alive = false;
        break;
      }
      const uint32_t sK = smem_u32(stages + static_cast<size_t>(s) * Cfg::kStageBytes);
      const int nvalid = min(kBlock, inf.len - (inf.start + inf.p * pt + j * kBlock));
      st.block(sK, sK + Cfg::kKBytes, nvalid, P.scale_log2, lane, scr);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!alive) break;

    // hand the state to the combiner (double-buffered by item parity) and go on
    ok = mbar_wait(&merge_empty[slot], ((it >> 1) & 1) ^ 1, abort_flag, err);
    if (!__all_sync(0xffffffffu, ok)) break;
    st.template store<NC>(merge[slot], w, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&merge_full[slot]);
  }
}

// The tensor maps live in kernel parameter space (__grid_constant__); the body
// takes their addresses for the copies.
template <typename T, int D, int NC, int S, bool kFma, int HPG>
__global__ void __launch_bounds__(32 * (NC + 3))
    attend_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams P) {
  attend_body<T, D, NC, S, kFma, HPG, false>(tm_k, tm_v, P);
}

// FP8 caches: two copy warps, two CTAs per SM (16 stages of 4 KB each).  One
// copy thread per CTA left the FP8 kernel short of copies in flight at this
// tile size (316 vs 309 us on the Llama-3-70B-shaped batch).
template <typename T, int D, int NC, int S>
__global__ void __launch_bounds__(32 * (NC + 4), 2)
    attend_fp8_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeParams P) {
  attend_body<T, D, NC, S, false, 1, true>(tm_k, tm_v, P);
}

// ---------------------------------------------------------------------------
// 3. merge of split sequences
//
// One CTA per (sequence with several partial results, KV head).  The prep
// kernel leaves everything a merge needs in one MergeInfo record.  Thread
// (c, s) owns float4 column c of the G x D block (kCols columns, a partial
// is one fully coalesced G*D*4-byte read) and the partials p = s, s + kSplit,
// ... of the sequence, U of them in flight, folded with a running maximum
// (the online rule used inside a partition); the kMergeSplit partial states
// of a column are then combined through shared memory.  Splitting the
// partials over 512 / kCols thread groups cuts the chain of dependent load
// rounds of a long sequence (64 partials at G = 4: 8 rounds -> 2).

template <typename T, int D, int kCols, int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads >= 1024 ? 1 : (kThreads >= 512 ? 2 : 512 / kThreads))
    merge_kernel(const DecodeParams P) {
  constexpr int U = kThreads >= 512 ? 6 : 8;  // partials in flight per thread (no spills)
  constexpr int kMergeSplit = kThreads / kCols;
  __shared__ float4 s_o[kMergeSplit][kCols];
  __shared__ float2 s_ml[kMergeSplit][kCols];
  pdl_wait();
  pdl_launch_dependents();
  // The first work unit's record is loaded together with the count (the
  // grid is at most num_seqs x hkv, so the record is inside the array).
  const int wi0 = static_cast<int>(blockIdx.x);
  MergeInfo mi0{};
  if (P.num_seqs > 0) mi0 = P.split[min(wi0 / P.hkv, P.num_seqs - 1)];
  // the merge records may come from a reused plan: a count beyond the
  // workspace and records that do not fit it are skipped and flagged
  int n_split = *reinterpret_cast<volatile int32_t*>(&P.ws->n_split);
  if (n_split < 0 || n_split > P.num_seqs) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&P.ws->error_bits, kErrPlan);
    n_split = n_split < 0 ? 0 : P.num_seqs;
  }
  const int n_work = n_split * P.hkv;
  const int G = P.G;
  const int n4 = G * D / 4;
  const int t = threadIdx.x;
  const int c = t % kCols, sp = t / kCols;
  const float4* acc4 = reinterpret_cast<const float4*>(P.acc);
  // the attention kernel has finished: its work counter is reset here, so
  // that a later call may reuse this workspace's plan without the prep kernel
  if (blockIdx.x == 0 && t == 0) P.ws->next_item = 0;
  for (int wi = blockIdx.x; wi < n_work; wi += gridDim.x) {
    const MergeInfo mi = wi == wi0 ? mi0 : P.split[wi / P.hkv];
    const int h = wi - (wi / P.hkv) * P.hkv;
    const int64_t head0 = static_cast<int64_t>(h) * G;
    // every count is bounded by the workspace before it is used (int64 sums:
    // no record can overflow them), so every partial index stays inside it
    const int64_t nfull = mi.nfull, nsuf = mi.nsuf, nchunks = mi.nchunks;
    const bool fits =
        mi.b >= 0 && mi.b < P.num_seqs && nfull >= 0 && nfull <= P.max_parts &&
        (nsuf == nfull || nsuf == nfull + 1) && nchunks >= 0 && nchunks <= P.max_rows &&
        nsuf + nchunks >= 1 &&
        (nfull == 0 || (mi.first_full >= 0 && mi.first_full + nfull <= P.max_parts)) &&
        (nsuf == nfull || (mi.tail >= 0 && mi.tail < P.max_parts)) &&
        (nchunks == 0 ||
         (mi.pfirst >= 0 && mi.pstride >= 1 && mi.pfirst + (nchunks - 1) * mi.pstride < P.max_rows));
    if (!fits) {
      if (t == 0) atomicOr(&P.ws->error_bits, kErrPlan);
      continue;
    }
    const int nparts = mi.nsuf + mi.nchunks;
    const bool col = c < n4;
    const int gk = min(4 * c / D, 7);
    float m = -INFINITY, l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = sp; p0 < nparts; p0 += U * kMergeSplit) {
      float4 a[U];
      float2 ml[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int p = p0 + u * kMergeSplit;
        if (col && p < nparts) {
          const int64_t idx =
              p < mi.nsuf ? (p < mi.nfull ? mi.first_full + p : mi.tail)
                          : static_cast<int64_t>(mi.pfirst) + static_cast<int64_t>(p - mi.nsuf) * mi.pstride;
          a[u] = __ldcg(&acc4[(idx * P.hq + head0) * (D / 4) + c]);
          ml[u] = __ldcg(&P.ml[idx * P.hq + head0 + gk]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (col && p0 + u * kMergeSplit < nparts) {
          const float mn = fmaxf(m, ml[u].x);
          const float al = exp2f(m - mn), wg = exp2f(ml[u].x - mn);
          l = fmaf(l, al, ml[u].y * wg);
          o.x = fmaf(o.x, al, a[u].x * wg);
          o.y = fmaf(o.y, al, a[u].y * wg);
          o.z = fmaf(o.z, al, a[u].z * wg);
          o.w = fmaf(o.w, al, a[u].w * wg);
          m = mn;
        }
      }
    }
    s_o[sp][c] = o;
    s_ml[sp][c] = make_float2(m, l);
    __syncthreads();
    if (sp == 0 && col) {
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kMergeSplit; ++k) M = fmaxf(M, s_ml[k][c].x);
      float Lsum = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kMergeSplit; ++k) {
        const float wk = exp2f(s_ml[k][c].x - M);  // 0 for a group without partials
        const float4 ok = s_o[k][c];
        Lsum = fmaf(s_ml[k][c].y, wk, Lsum);
        O.x = fmaf(ok.x, wk, O.x);
        O.y = fmaf(ok.y, wk, O.y);
        O.z = fmaf(ok.z, wk, O.z);
        O.w = fmaf(ok.w, wk, O.w);
      }
      const float inv = 1.f / Lsum;
      T* dst = static_cast<T*>(P.out) + (static_cast<int64_t>(mi.b) * P.hq + head0) * D + 4 * c;
      uint2 pk;
      pk.x = pack2<T>(O.x * inv, O.y * inv);
      pk.y = pack2<T>(O.z * inv, O.w * inv);
      *reinterpret_cast<uint2*>(dst) = pk;
    }
    __syncthreads();  // s_o / s_ml are rewritten for the next work unit
  }
  // the empty softmax of a zero-length sequence: its output is defined as 0
  // (after the merges, whose loads need not wait behind these)
  for (int b = blockIdx.x * kThreads + t; b < P.num_seqs; b += gridDim.x * kThreads) {
    int L = P.seq_lens[b];
    if (L <= 0) {
      uint4* o = reinterpret_cast<uint4*>(static_cast<T*>(P.out) + static_cast<int64_t>(b) * P.hq * D);
      for (int i = 0; i < P.hq * D * 2 / 16; ++i) o[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// 4. shared-prefix attention (grouped decode)
//
// One work item = (group, 256-token chunk of the shared prefix, tile of 128
// query rows, KV head).  The members of a group share the prefix's physical
// blocks, so the chunk's K and V tiles are loaded once (TMA, 128-byte
// swizzle) and every member's G query heads attend to them together: a real
// [128 rows x head_dim] x [head_dim x 16 tokens] product per block, on the
// tensor cores (mma.sync m16n8k16; eight warps, 16 query rows each, Q kept in
// registers, P reused from the score accumulators as the PV operand).  Each
// row's (max, sum, unnormalised output) over the chunk is a partial result
// that the merge kernel folds into the member's output.

constexpr int kPrefixWarps = kPrefixRows / 16;

template <int D>
struct PrefixCfg {
  static constexpr int kStageBytes = Tile<D>::kStageBytes;
  static constexpr size_t kBytes = static_cast<size_t>(kPrefixChunkBlocks) * kStageBytes + 64 + 1024;
};

template <typename T, int D>
__global__ void __launch_bounds__(kPrefixWarps * 32)
    prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams P) {
  using Cfg = PrefixCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kPrefixChunkBlocks * Cfg::kStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 1);
  int* err = &P.ws->error_bits;
  int n_pitems = *reinterpret_cast<volatile int32_t*>(&P.ws->n_pitems);
  if (n_pitems < 0 || n_pitems > P.max_pitems) {  // a reused plan that does not fit
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, kErrPlan);
    n_pitems = n_pitems < 0 ? 0 : static_cast<int>(P.max_pitems);
  }
  const int n_work = n_pitems * P.hkv;
  if (blockIdx.x >= n_work) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = P.G;
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t y_oob = P.num_blocks * P.hkv * kBlock;
  uint32_t n_local = 0;  // items this CTA has loaded (the barrier's phase)
  for (int wi = blockIdx.x; wi < n_work; wi += gridDim.x) {
    const int4 item = P.pitems[wi / P.hkv];
    const int h = wi - (wi / P.hkv) * P.hkv;
    const int grp = item.x, chunk = item.y, tile = item.z;
    // the item may come from a reused plan: one that does not describe a
    // chunk of this call's groups inside the workspace is skipped (uniformly:
    // every thread reads the same values)
    if (grp < 0 || grp >= P.num_groups || chunk < 0 || tile < 0) {
      if (tid == 0) atomicOr(err, kErrPlan);
      continue;
    }
    const int off = P.group_off[grp];
    const int64_t M64 = static_cast<int64_t>(P.group_off[grp + 1]) - off;
    const int4 gi = P.group_info[grp];
    const int pre = P.group_prefix[grp];
    const int64_t nblk64 = min(static_cast<int64_t>(kPrefixChunkBlocks),
                               static_cast<int64_t>(pre / kBlock) - static_cast<int64_t>(chunk) * kPrefixChunkBlocks);
    if (off < 0 || M64 < 1 || off + M64 > P.num_seqs || pre <= 0 || pre % kBlock != 0 || nblk64 < 1 ||
        static_cast<int64_t>(chunk) * kPrefixChunkBlocks + nblk64 > P.max_blocks ||
        static_cast<int64_t>(tile) * kPrefixRows >= M64 * G || gi.x < 0 ||
        static_cast<int64_t>(gi.x) + (static_cast<int64_t>(chunk) + 1) * M64 > P.max_rows) {
      if (tid == 0) atomicOr(err, kErrPlan);
      continue;
    }
    const int M = static_cast<int>(M64), nblk = static_cast<int>(nblk64);
    if (tid == 0) {
      // the prefix blocks are those of the group's first member
      const int32_t* trow = P.tables + static_cast<int64_t>(off) * P.max_blocks + chunk * kPrefixChunkBlocks;
      mbar_arrive_expect_tx(bar, nblk * Cfg::kStageBytes);
      for (int j = 0; j < nblk; ++j) {
        int32_t id = trow[j];
        if (id < 0 || id >= P.num_blocks) {
          atomicOr(err, kErrBlockId);
          id = -1;
        }
        const int32_t y = static_cast<int32_t>(id < 0 ? y_oob : (static_cast<int64_t>(id) * P.hkv + h) * kBlock);
        uint8_t* dst = smem + static_cast<size_t>(j) * Cfg::kStageBytes;
        tma_load_3d(dst, &tm_k, 0, y, 0, bar);
        tma_load_3d(dst + Tile<D>::kKVBytes, &tm_v, 0, y, 0, bar);
      }
    }
    // this warp's 16 query rows: row r -> member r / G, head r % G
    const int r0 = tile * kPrefixRows + warp * 16 + g, r1 = r0 + 8;
    const int m0 = r0 / G, m1 = r1 / G;
    const bool ok0 = m0 < M, ok1 = m1 < M;
    const T* q0 = static_cast<const T*>(P.q) + ((static_cast<int64_t>(off) + m0) * P.hq + h * G + r0 % G) * D;
    const T* q1 = static_cast<const T*>(P.q) + ((static_cast<int64_t>(off) + m1) * P.hq + h * G + r1 % G) * D;
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + 16 * ks + 2 * t) : 0u;
      qa[ks][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + 16 * ks + 2 * t) : 0u;
      qa[ks][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + 16 * ks + 2 * t + 8) : 0u;
      qa[ks][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + 16 * ks + 2 * t + 8) : 0u;
    }
    bool ok = mbar_wait(bar, n_local & 1, abort_flag, err);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) {  // let this CTA's copies land before it leaves
        unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(bar, n_local & 1) && global_timer_ns() - t0 < kWaitLimitNs / 4) {
        }
      }
      return;
    }
    float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    for (int j = 0; j < nblk; ++j) {
      const uint32_t sK = smem_u32(smem + static_cast<size_t>(j) * Cfg::kStageBytes);
      const uint32_t sV = sK + Tile<D>::kKVBytes;
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
        const int cofs = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b00, b01, b10, b11;
          ldmatrix_x4(b00, b01, b10, b11, chunk_addr(sK, tok, 2 * ks + cofs));
          Mma<T>::run(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
          Mma<T>::run(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
        }
      }
      // rows g (s*[0], s*[1]) and g + 8 (s*[2], s*[3]); tokens 2t, 2t+1 (+8 for s1)
      float x[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        x[e][0] = s0[2 * e] * P.scale_log2;
        x[e][1] = s0[2 * e + 1] * P.scale_log2;
        x[e][2] = s1[2 * e] * P.scale_log2;
        x[e][3] = s1[2 * e + 1] * P.scale_log2;
      }
      float pr[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float bm = fmaxf(fmaxf(x[e][0], x[e][1]), fmaxf(x[e][2], x[e][3]));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        const float mn = fmaxf(mr[e], bm);
        const float al = exp2f(mr[e] - mn);
#pragma unroll
        for (int c = 0; c < 4; ++c) pr[e][c] = exp2f(x[e][c] - mn);
        lr[e] = lr[e] * al + (pr[e][0] + pr[e][1] + pr[e][2] + pr[e][3]);
        mr[e] = mn;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          o[nd][2 * e] *= al;
          o[nd][2 * e + 1] *= al;
        }
      }
      const uint32_t pa0 = pack2<T>(pr[0][0], pr[0][1]), pa1 = pack2<T>(pr[1][0], pr[1][1]);
      const uint32_t pa2 = pack2<T>(pr[0][2], pr[0][3]), pa3 = pack2<T>(pr[1][2], pr[1][3]);
      {
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int cofs = lane >> 4;
#pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
          uint32_t b00, b01, b10, b11;
          ldmatrix_x4_trans(b00, b01, b10, b11, chunk_addr(sV, tok, nd + cofs));
          Mma<T>::run(o[nd], pa0, pa1, pa2, pa3, b00, b01);
          Mma<T>::run(o[nd + 1], pa0, pa1, pa2, pa3, b10, b11);
        }
      }
    }
    // partial results of this chunk for the warp's rows
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float L = lr[e];
      L += __shfl_xor_sync(0xffffffffu, L, 1);
      L += __shfl_xor_sync(0xffffffffu, L, 2);
      const int r = e ? r1 : r0;
      const int m = r / G;
      if (m < M) {
        const int64_t prow = (static_cast<int64_t>(gi.x) + static_cast<int64_t>(chunk) * M + m) * P.hq +
                             h * G + r % G;
        float* dst = P.acc + prow * D;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd)
          *reinterpret_cast<float2*>(dst + 8 * nd + 2 * t) = make_float2(o[nd][2 * e], o[nd][2 * e + 1]);
        if (t == 0) P.ml[prow] = make_float2(mr[e], L);
      }
    }
    // every warp is done with the stages before the next item's copies
    __syncthreads();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    ++n_local;
  }
}

// ---------------------------------------------------------------------------
// Host side.

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn(std::string* why) {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  if (!fn && why) *why = "cuTensorMapEncodeTiled is not available from the driver";
  return fn;
}

// FP8 caches: K as rows of D bytes (box 16 rows, 128-byte swizzle); V tiles
// are contiguous, read as 16 rows of D bytes without swizzle (ldmatrix reads
// its 16-byte dimension rows conflict-free).
bool encode_fp8_maps(CUtensorMap* mk, CUtensorMap* mv, const void* kbase, const void* vbase,
                     int64_t num_blocks, int hkv, int D, std::string* why) {
  EncodeTiledFn fn = get_encode_fn(why);
  if (!fn) return false;
  const cuuint32_t estr[2] = {1, 1};
  cuuint64_t kd[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_blocks) * hkv * kBlock};
  cuuint64_t ks[1] = {static_cast<cuuint64_t>(D)};
  cuuint32_t kb[2] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(kBlock)};
  CUresult r = fn(mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kbase), kd, ks, kb, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    // A V tile (D dims x 16 bytes) is one contiguous run of 16 * D bytes; it is
    // described as 16 rows of D bytes so TMA moves it in 16 long requests.
    cuuint64_t vd[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_blocks) * hkv * kBlock};
    cuuint64_t vs[1] = {static_cast<cuuint64_t>(D)};
    cuuint32_t vb[2] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(kBlock)};
    r = fn(mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(vbase), vd, vs, vb, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled (FP8) failed with CUresult " + std::to_string(static_cast<int>(r));
    return false;
  }
  return true;
}

}  // namespace

void* tensor_map_encoder(std::string* why) { return reinterpret_cast<void*>(get_encode_fn(why)); }

// The 16-bit caches as a 2-D tensor of token rows (one 16 x 64 box per
// block and 64-dim half): the prefill kernel's chunk layout puts a block's
// halves 16 KB apart, so it copies them separately.
bool encode_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv, int D,
                      std::string* why) {
  EncodeTiledFn fn = get_encode_fn(why);
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(num_blocks) * hkv * kBlock};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlock)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (why) *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
    return false;
  }
  return true;
}

// The 16-bit caches as a 3-D tensor for the decode kernels: (64 dims of one
// half, token rows, halves), so that one box of 64 x 16 x D/64 moves a whole
// (block, KV head) tile, its halves 2048 bytes apart as two 2-D boxes would
// put them (the 128-byte swizzle phase is the token row either way).
bool encode_cache_map3(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv, int D,
                       std::string* why) {
  EncodeTiledFn fn = get_encode_fn(why);
  if (!fn) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(num_blocks) * hkv * kBlock,
                        static_cast<cuuint64_t>(D / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBlock), static_cast<cuuint32_t>(D / 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (why) *why = "cuTensorMapEncodeTiled (3-D) failed with CUresult " + std::to_string(static_cast<int>(r));
    return false;
  }
  return true;
}

namespace {

struct LaunchShape {
  int grid;
  size_t smem;
};

template <typename T, int D, int NC, int S, bool kFma, int HPG, bool kFp8 = false>
bool launch_attend(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& P,
                   int64_t max_items, cudaStream_t stream, std::string* why) {
  using Cfg = AttendCfg<T, D, NC, S, kFma, kFp8>;
  void (*kern)(CUtensorMap, CUtensorMap, DecodeParams);
  if constexpr (kFp8) {
    kern = attend_fp8_kernel<T, D, NC, S>;
  } else {
    kern = attend_kernel<T, D, NC, S, kFma, HPG>;
  }
  static int occ_cache[64] = {0};  // per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  const int slot = dev & 63;
  if (occ_cache[slot] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kBytes));
    if (e != cudaSuccess) {
      *why = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return false;
    }
    int per_sm = 0, sms = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::kThreads, Cfg::kBytes);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (per_sm < 1) per_sm = 1;
    occ_cache[slot] = per_sm * sms;
  }
  int64_t grid = occ_cache[slot];
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(Cfg::kThreads),
                             Cfg::kBytes, stream, tk, tv, P);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("attend launch: ") + cudaGetErrorString(e);
    return false;
  }
  return true;
}

template <typename T, int D>
bool dispatch_attend(int variant, int G, const CUtensorMap& tk, const CUtensorMap& tv,
                     const DecodeParams& P, int64_t max_items, cudaStream_t s, std::string* why) {
  constexpr int NC = 4;
  if (variant == 1) {
    constexpr int S = 4;  // the FMA variant also keeps q, p in shared memory
    if (G <= 2) return launch_attend<T, D, NC, S, true, 1>(tk, tv, P, max_items, s, why);
    if (G <= 4) return launch_attend<T, D, NC, S, true, 2>(tk, tv, P, max_items, s, why);
    return launch_attend<T, D, NC, S, true, 4>(tk, tv, P, max_items, s, why);
  }
  constexpr int S = 8;
  return launch_attend<T, D, NC, S, false, 1>(tk, tv, P, max_items, s, why);
}

}  // namespace

// One side stream and a fork/join event pair per device, created on first
// use and kept for the process.  Reusing the events is safe as long as one
// call's record-then-wait sequence is not interleaved with another's (a
// stream wait uses the record that precedes it): a grouped decode holds the
// device's `use` lock from the fork record until its stream has waited on
// the join, so host threads calling it concurrently take turns there.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex use;
};

SideStream* side_stream(std::string* why) {
  static SideStream sides[64];
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) {
    *why = "device ordinal out of range";
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  SideStream& ss = sides[dev];
  if (!ss.stream) {
    cudaError_t e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      *why = std::string("side stream: ") + cudaGetErrorString(e);
      if (ss.join) cudaEventDestroy(ss.join);
      if (ss.fork) cudaEventDestroy(ss.fork);
      if (ss.stream) cudaStreamDestroy(ss.stream);
      ss.stream = nullptr;
      ss.fork = ss.join = nullptr;
      return nullptr;
    }
  }
  return &ss;
}

template <typename T, int D>
bool launch_prefix(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& P, int n_sm,
                   cudaStream_t stream, std::string* why) {
  using Cfg = PrefixCfg<D>;
  auto kern = prefix_kernel<T, D>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kBytes));
    if (e != cudaSuccess) {
      *why = std::string("cudaFuncSetAttribute (prefix): ") + cudaGetErrorString(e);
      return false;
    }
    attr_set[dev & 63] = true;
  }
  kern<<<static_cast<unsigned>(2 * n_sm), kPrefixWarps * 32, Cfg::kBytes, stream>>>(tk, tv, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("prefix launch: ") + cudaGetErrorString(e);
    return false;
  }
  return true;
}

// Merge kernel for kThreads = one group of kCols threads, 512 or 1024.
template <typename T, int D, int kCols>
cudaError_t launch_merge(int threads, dim3 grid, cudaStream_t s, const DecodeParams& P) {
  if (threads == 1024) return launch_pdl(merge_kernel<T, D, kCols, 1024>, grid, dim3(1024), 0, s, P);
  if (threads == kMergeThreads)
    return launch_pdl(merge_kernel<T, D, kCols, kMergeThreads>, grid, dim3(kMergeThreads), 0, s, P);
  return launch_pdl(merge_kernel<T, D, kCols, kCols>, grid, dim3(kCols), 0, s, P);
}

int decode_launch(const DecodeArgs& a, std::string* why) {
  const bool grouped = a.num_groups > 0;
  const WsLayout L = ws_layout(a.num_seqs, a.num_q_heads, a.head_dim, a.max_seq_len, grouped);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  DecodeParams P;
  P.q = a.q;
  P.out = a.out;
  P.tables = a.block_tables;
  P.seq_lens = a.seq_lens;
  P.ws = reinterpret_cast<WsHeader*>(ws);
  P.parts = reinterpret_cast<PartInfo*>(ws + L.off_parts);
  P.seq_first = reinterpret_cast<int2*>(ws + L.off_seq_first);
  P.split = reinterpret_cast<MergeInfo*>(ws + L.off_split);
  P.seq_prefix = reinterpret_cast<int4*>(ws + L.off_seq_prefix);
  P.group_info = reinterpret_cast<int4*>(ws + L.off_group);
  P.group_bad = reinterpret_cast<int32_t*>(ws + L.off_group_bad);
  P.pitems = reinterpret_cast<int4*>(ws + L.off_pitems);
  P.group_off = a.group_off;
  P.group_prefix = a.group_prefix;
  P.num_groups = grouped ? a.num_groups : 0;
  P.ml = reinterpret_cast<float2*>(ws + L.off_ml);
  P.acc = reinterpret_cast<float*>(ws + L.off_acc);
  P.max_parts = L.max_parts;
  P.max_rows = L.max_parts + L.max_prefix;
  P.max_pitems = L.max_prefix;
  P.num_blocks = a.num_blocks;
  P.max_blocks = a.max_blocks_per_seq;
  P.num_seqs = a.num_seqs;
  P.max_seq_len = a.max_seq_len;
  P.hq = a.num_q_heads;
  P.hkv = a.num_kv_heads;
  P.G = a.num_q_heads / a.num_kv_heads;
  P.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);

  P.k_scale = a.k_scale;
  P.v_scale = a.v_scale;
  CUtensorMap tk, tv;
  if (a.fp8) {
    if (!encode_fp8_maps(&tk, &tv, a.k_cache, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, why))
      return 5;
  } else if (!encode_cache_map3(&tk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, why) ||
             !encode_cache_map3(&tv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, why)) {
    return 5;
  }

  cudaStream_t s = static_cast<cudaStream_t>(a.stream);
  const int row_uint4 = a.num_q_heads * a.head_dim * 2 / 16;
  cudaEvent_t join_after_attend = nullptr;
  std::unique_lock<std::mutex> side_lock;  // held from the fork record to the wait on the join
  int dev0 = 0, n_sm = 0;
  cudaGetDevice(&dev0);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev0);
  // 8 full-partition items per attention CTA (two CTAs per SM)
  // the plan (partition list, merge records, counters) depends only on the
  // lengths, tables and shapes: a caller may reuse the workspace's plan
  if (!a.reuse_plan) {
    static bool prep_attr[64] = {false};
    cudaError_t e = cudaSuccess;
    if (!prep_attr[dev0 & 63]) {
      e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kPrepSmem));
      if (e == cudaSuccess) prep_attr[dev0 & 63] = true;
    }
    if (e == cudaSuccess)
      e = launch_pdl(prep_kernel, dim3(1), dim3(prep_threads(a.num_seqs)), kPrepSmem, s, P, row_uint4,
                     16 * n_sm, static_cast<int>(a.partition_tokens));
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
      *why = std::string("prep launch: ") + cudaGetErrorString(e);
      return 5;
    }
  }
  if (grouped) {
    // The prefix kernel moves little data and is mostly latency: it runs on a
    // library-owned side stream forked from and joined back into the
    // caller's stream with events, so it overlaps the attention kernel.
    SideStream* side = side_stream(why);
    if (!side) return 5;
    side_lock = std::unique_lock<std::mutex>(side->use);
    cudaEventRecord(side->fork, s);
    cudaStreamWaitEvent(side->stream, side->fork, 0);
    bool okp = a.dtype == 1
                   ? (a.head_dim == 128 ? launch_prefix<__nv_bfloat16, 128>(tk, tv, P, n_sm, side->stream, why)
                                        : launch_prefix<__nv_bfloat16, 64>(tk, tv, P, n_sm, side->stream, why))
                   : (a.head_dim == 128 ? launch_prefix<__half, 128>(tk, tv, P, n_sm, side->stream, why)
                                        : launch_prefix<__half, 64>(tk, tv, P, n_sm, side->stream, why));
    if (!okp) return 5;
    cudaEventRecord(side->join, side->stream);
    join_after_attend = side->join;
  }
  if (a.ev_before) cudaEventRecord(static_cast<cudaEvent_t>(a.ev_before), s);
  const int64_t max_items = L.max_parts * a.num_kv_heads;
  const int variant = a.variant == 0 ? 2 : a.variant;
  bool ok;
  if (a.fp8) {  // head_dim 128 only; 16 stages of 4 KB, two copy warps, two CTAs per SM
    ok = a.dtype == 1
             ? launch_attend<__nv_bfloat16, 128, 4, 16, false, 1, true>(tk, tv, P, max_items, s, why)
             : launch_attend<__half, 128, 4, 16, false, 1, true>(tk, tv, P, max_items, s, why);
  } else if (a.dtype == 1) {
    ok = a.head_dim == 128
             ? dispatch_attend<__nv_bfloat16, 128>(variant, P.G, tk, tv, P, max_items, s, why)
             : dispatch_attend<__nv_bfloat16, 64>(variant, P.G, tk, tv, P, max_items, s, why);
  } else {
    ok = a.head_dim == 128 ? dispatch_attend<__half, 128>(variant, P.G, tk, tv, P, max_items, s, why)
                           : dispatch_attend<__half, 64>(variant, P.G, tk, tv, P, max_items, s, why);
  }
  if (!ok) return 5;
  if (a.ev_after) cudaEventRecord(static_cast<cudaEvent_t>(a.ev_after), s);
  if (join_after_attend) cudaStreamWaitEvent(s, join_after_attend, 0);
  if (side_lock.owns_lock()) side_lock.unlock();

  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one column of threads per float4 column of the G x D block (256 for G = 8
  // at head_dim 128, else 128), 512 threads in all; a whole batch's merges
  // fit in one wave
  // Sequences of at most 8 partitions (of 512 tokens, the smallest) are
  // merged by one thread group each, many CTAs per SM; longer ones by
  // 512-thread CTAs whose groups share the partials.
  const bool wide = P.G * a.head_dim / 4 > 128;
  const bool split = (static_cast<int64_t>(a.max_seq_len) + kPartTokens - 1) / kPartTokens > 8;
  // Long sequences: 512 threads, the thread groups sharing a sequence's
  // partials; 1024 (twice the groups: one round of loads for 64 partials)
  // when the (sequence, KV head) units fit one CTA per SM.
  const int64_t units = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  const int mthreads = split ? (units <= sms ? 1024 : kMergeThreads) : (wide ? 256 : 128);
  int64_t mgrid = units;
  const int mres = mthreads >= 1024 ? 1 : (mthreads >= 512 ? 2 : 512 / mthreads);  // resident per SM
  if (mgrid > sms * mres) mgrid = sms * mres;
  if (mgrid < 1) mgrid = 1;
  const dim3 mg(static_cast<unsigned>(mgrid));
  cudaError_t e;
  if (a.dtype == 1) {
    if (a.head_dim == 128)
      e = wide ? launch_merge<__nv_bfloat16, 128, 256>(mthreads, mg, s, P)
               : launch_merge<__nv_bfloat16, 128, 128>(mthreads, mg, s, P);
    else
      e = launch_merge<__nv_bfloat16, 64, 128>(mthreads, mg, s, P);
  } else {
    if (a.head_dim == 128)
      e = wide ? launch_merge<__half, 128, 256>(mthreads, mg, s, P)
               : launch_merge<__half, 128, 128>(mthreads, mg, s, P);
    else
      e = launch_merge<__half, 64, 128>(mthreads, mg, s, P);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("merge launch: ") + cudaGetErrorString(e);
    return 5;
  }
  return 0;
}

size_t decode_workspace_bytes(int64_t num_seqs, int64_t num_q_heads, int64_t head_dim,
                              int64_t max_seq_len, bool grouped) {
  return ws_layout(num_seqs, num_q_heads, head_dim, max_seq_len, grouped).total;
}

}  // namespace pa
