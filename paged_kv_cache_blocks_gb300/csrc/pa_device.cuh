// Device-side building blocks shared by the libpa kernels (sm_103a):
// mbarriers with bounded waits, TMA tile loads, ldmatrix / movmatrix / mma,
// 16-bit <-> fp32 conversions, and the decode workspace layout.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace pa {

constexpr int kBlock = 16;          // tokens per KV block
constexpr int kPartTokens = 512;    // smallest decode partition (tokens)
constexpr int kMaxPartMult = 4;     // partitions are 512, 1024 or 2048 tokens
constexpr int kMaxPartBlocks = kPartTokens * kMaxPartMult / kBlock;

// Device error bits (mirrored by PA_DEVERR_* in pa.h).
constexpr int kErrSeqLen = 1;
constexpr int kErrBlockId = 2;
constexpr int kErrTimeout = 4;
constexpr int kErrGroup = 8;

// A wait that has not completed after this long gives up (ns of globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// Decode workspace layout (caller-owned device memory, 256-byte aligned).
struct WsHeader {
  int32_t error_bits;
  int32_t n_parts;      // partitions of all sequences
  int32_t n_items;      // n_parts * num_kv_heads
  int32_t next_item;    // dynamic work counter of the attention kernel
  int32_t n_split;      // sequences with more than one partition
  int32_t next_split;   // dynamic work counter of the merge kernel
  int32_t part_tokens;  // tokens per partition chosen for this call
  int32_t n_pitems;     // shared-prefix work items (grouped decode)
  int32_t n_suffix_parts;  // partitions of the attention kernel (= n_parts)
  int32_t pad[55];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// Per partition: sequence, partition index, clamped length, partial results of
// the sequence, first token the partitions cover (after a shared prefix).
struct PartInfo {
  int32_t b, p, len, nparts, start, pad0, pad1, pad2;
};

// Everything the merge needs about one sequence with several partial results:
// its partitions are first_full .. first_full+nfull-1, then tail (if nsuf >
// nfull), then the shared-prefix chunks pfirst + c * pstride, c < nchunks.
struct MergeInfo {
  int32_t b, first_full, tail, nfull, nsuf, pfirst, pstride, nchunks;
};

// Shared-prefix chunks of grouped decode: 16 blocks (256 tokens) each.
constexpr int kPrefixChunkBlocks = 16;
constexpr int kPrefixChunkTokens = kPrefixChunkBlocks * kBlock;
constexpr int kPrefixRows = 128;  // query rows (members x heads) per prefix work item

struct WsLayout {
  size_t off_parts;       // PartInfo[max_parts]
  size_t off_seq_first;   // int2[num_seqs]: first full partition, tail partition (-1: none)
  size_t off_split;       // MergeInfo[num_seqs]: sequences whose partial results need a merge
  size_t off_seq_prefix;  // int4[num_seqs]: first prefix partial, group size, chunks, prefix tokens
  size_t off_group;       // int4[num_seqs]: per group: partial base, item base, chunks, row tiles
  size_t off_group_bad;   // int32[num_seqs]: per group: shared prefix rejected
  size_t off_pitems;      // int4[max_pitems]: (group, chunk, row tile)
  size_t off_ml;          // float2[(max_parts + max_prefix) * num_q_heads]: (max, sum)
  size_t off_acc;         // float[(max_parts + max_prefix) * num_q_heads * head_dim]
  size_t total;
  int64_t max_parts;      // attention-kernel partitions
  int64_t max_prefix;     // shared-prefix partial rows (grouped decode only)
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int64_t num_seqs, int64_t num_q_heads, int64_t head_dim,
                          int64_t max_seq_len, bool grouped = false) {
  WsLayout L;
  int64_t per_seq = (max_seq_len + kPartTokens - 1) / kPartTokens;
  if (per_seq < 1) per_seq = 1;
  L.max_parts = num_seqs * per_seq;
  L.max_prefix = grouped ? num_seqs * ((max_seq_len + kPrefixChunkTokens - 1) / kPrefixChunkTokens)
                         : 0;
  const int64_t rows = L.max_parts + L.max_prefix;
  size_t o = sizeof(WsHeader);
  L.off_parts = o;       o = align_up(o + sizeof(PartInfo) * L.max_parts, 256);
  L.off_seq_first = o;   o = align_up(o + sizeof(int2) * num_seqs, 256);
  L.off_split = o;       o = align_up(o + sizeof(MergeInfo) * num_seqs, 256);
  L.off_seq_prefix = o;  o = align_up(o + sizeof(int4) * num_seqs, 256);
  L.off_group = o;       o = align_up(o + (grouped ? sizeof(int4) * num_seqs : 0), 256);
  L.off_group_bad = o;   o = align_up(o + (grouped ? sizeof(int32_t) * num_seqs : 0), 256);
  L.off_pitems = o;      o = align_up(o + sizeof(int4) * L.max_prefix, 256);
  L.off_ml = o;          o = align_up(o + sizeof(float2) * rows * num_q_heads, 256);
  L.off_acc = o;         o = align_up(o + sizeof(float) * rows * num_q_heads * head_dim, 256);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// PTX helpers.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete.  Gives up after kWaitLimitNs
// or when *abort becomes non-zero; returns false then (and sets the flags).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err_bits) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(err_bits, kErrTimeout);
      return false;
    }
  }
}

// 2-D tiled TMA load of one box into shared memory, completion on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <typename T>
struct Mma;

template <>
struct Mma<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};

template <>
struct Mma<__half> {
  __device__ __forceinline__ static void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
};

// Two E4M3 bytes (low byte -> low half) -> two fp16, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint16_t x) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(x));
  return d;
}

// Two fp32 -> two E4M3 bytes (lo -> low byte), round to nearest even,
// saturated to +-448.
__device__ __forceinline__ uint16_t float2_to_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two fp32 -> one packed pair of 16-bit values (lo in the low half), RNE.
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One packed pair -> two fp32.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t x);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  return __half22float2(h);
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_float<__half>(float x) {
  return __float2half_rn(x);
}

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float to_float<__half>(__half x) {
  return __half2float(x);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a TMA box of
// rows of 128 bytes written with the 128-byte swizzle (box base 1024-aligned).
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// Exclusive prefix sum of one int per thread over the whole CTA; *total gets
// the sum.  sw: 32 ints of shared scratch.  Every thread must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sw, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sw[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? sw[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    sw[lane] = t;
  }
  __syncthreads();
  int res = (w ? sw[w - 1] : 0) + x - v;
  *total = sw[nw - 1];
  __syncthreads();
  return res;
}

// Tensor map over a 16-bit cache [num_blocks][hkv][16][D] viewed as rows of D
// elements: box 64 elements x 16 rows, 128-byte swizzle.
bool encode_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv, int D,
                      std::string* why);

}  // namespace pa
