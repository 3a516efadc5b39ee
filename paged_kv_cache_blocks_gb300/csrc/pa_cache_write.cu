// Cache write and copy-on-write block copy for sm_103a.
//
// Cache write: scatter each new token's K and V rows into the
// paged cache through the slot mapping ("vLLM Nedir? PagedAttention ile
// Production LLM Serving", section "Bir istek motorun icinde", step 2;
// "vLLM ve Triton ile maliyet optimizasyonu", section 03, steps 1-3).
//
// One thread per 16-byte chunk of a (token, KV head) row; blockIdx.y picks K
// or V.  Loads and stores are 16-byte vectors, consecutive threads touch
// consecutive chunks of a row, so both sides are fully coalesced.  The work
// is a few hundred KB per step, so the kernel is launch- and latency-bound.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
    cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                       const int64_t* __restrict__ slot_mapping, int64_t n_chunks, int chunks_per_token,
                       int chunks_per_row, int hkv, uint4* __restrict__ k_cache,
                       uint4* __restrict__ v_cache, int64_t num_blocks) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_chunks) return;
  const int64_t t = i / chunks_per_token;
  const int rem = static_cast<int>(i - t * chunks_per_token);
  const int h = rem / chunks_per_row;
  const int c = rem - h * chunks_per_row;
  // the chunk is loaded together with its token's slot (its index does not
  // depend on the slot): one round trip to global memory, not two
  const uint4 val = blockIdx.y == 0 ? k[i] : v[i];
  const int64_t s = slot_mapping[t];
  if (s < 0) return;                      // padding token
  const int64_t blk = s / kBlock;
  if (blk >= num_blocks) return;          // outside the pool: not written
  const int64_t off = s - blk * kBlock;
  const int64_t dst = ((blk * hkv + h) * kBlock + off) * chunks_per_row + c;
  (blockIdx.y == 0 ? k_cache : v_cache)[dst] = val;
}

int cache_write_launch(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                       int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                       int64_t num_blocks, void* stream, std::string* why) {
  const int chunks_per_row = head_dim * 2 / 16;
  const int chunks_per_token = chunks_per_row * num_kv_heads;
  const int64_t n_chunks = static_cast<int64_t>(num_tokens) * chunks_per_token;
  if (n_chunks == 0) return 0;
  const int threads = 256;
  const int64_t blocks = (n_chunks + threads - 1) / threads;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  cudaError_t e = launch_pdl(cache_write_kernel, grid, dim3(threads), 0,
                             static_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                             static_cast<const uint4*>(v), slot_mapping, n_chunks, chunks_per_token,
                             chunks_per_row, num_kv_heads, static_cast<uint4*>(k_cache),
                             static_cast<uint4*>(v_cache), num_blocks);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("cache_write launch: ") + cudaGetErrorString(e);
    return 5;
  }
  return 0;
}

// FP8 cache write: the same scatter, each value quantised to E4M3 as
// E4M3(fp32(x) * fp32(1 / scale[h])) (round to nearest even, saturated).
// K rows stay token-major ([block][head][16][D]); V is stored dimension-major
// ([block][head][D][16]) so the decode kernel can feed it to the tensor cores
// without a transpose.  One thread per 8 values of a (token, head) row.
template <typename T>
__global__ void __launch_bounds__(256)
    cache_write_fp8_kernel(const T* __restrict__ k, const T* __restrict__ v,
                           const int64_t* __restrict__ slot_mapping, int64_t n_chunks, int hkv, int D,
                           const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                           uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                           int64_t num_blocks) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_chunks) return;
  const int cpr = D / 8;
  const int64_t t = i / (static_cast<int64_t>(hkv) * cpr);
  const int rem = static_cast<int>(i - t * hkv * cpr);
  const int h = rem / cpr, c = rem - h * cpr;
  const int64_t s = slot_mapping[t];
  if (s < 0) return;
  const int64_t blk = s / kBlock;
  if (blk >= num_blocks) return;
  const int64_t off = s - blk * kBlock;
  const float ik = 1.0f / k_scale[h], iv = 1.0f / v_scale[h];
  const uint4 kv = *reinterpret_cast<const uint4*>(k + (t * hkv + h) * D + 8 * c);
  const uint4 vv = *reinterpret_cast<const uint4*>(v + (t * hkv + h) * D + 8 * c);
  const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
  uint16_t kq[4], vq[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 a = unpack2<T>(kw[e]), b = unpack2<T>(vw[e]);
    kq[e] = float2_to_e4m3x2(a.x * ik, a.y * ik);
    vq[e] = float2_to_e4m3x2(b.x * iv, b.y * iv);
  }
  uint2 kout;
  kout.x = static_cast<uint32_t>(kq[0]) | (static_cast<uint32_t>(kq[1]) << 16);
  kout.y = static_cast<uint32_t>(kq[2]) | (static_cast<uint32_t>(kq[3]) << 16);
  *reinterpret_cast<uint2*>(k_cache + ((blk * hkv + h) * kBlock + off) * D + 8 * c) = kout;
  uint8_t* vrow = v_cache + ((blk * hkv + h) * D + 8 * c) * kBlock + off;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    vrow[(2 * e) * kBlock] = static_cast<uint8_t>(vq[e] & 0xff);
    vrow[(2 * e + 1) * kBlock] = static_cast<uint8_t>(vq[e] >> 8);
  }
}

int cache_write_fp8_launch(const void* k, const void* v, const int64_t* slot_mapping,
                           int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                           const float* k_scale, const float* v_scale, void* k_cache, void* v_cache,
                           int64_t num_blocks, int32_t dtype, void* stream, std::string* why) {
  const int64_t n_chunks = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 8);
  if (n_chunks == 0) return 0;
  const int64_t blocks = (n_chunks + 255) / 256;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == 1)
    cache_write_fp8_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), slot_mapping,
        n_chunks, num_kv_heads, head_dim, k_scale, v_scale, static_cast<uint8_t*>(k_cache),
        static_cast<uint8_t*>(v_cache), num_blocks);
  else
    cache_write_fp8_kernel<__half><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __half*>(k), static_cast<const __half*>(v), slot_mapping, n_chunks,
        num_kv_heads, head_dim, k_scale, v_scale, static_cast<uint8_t*>(k_cache),
        static_cast<uint8_t*>(v_cache), num_blocks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("cache_write_fp8 launch: ") + cudaGetErrorString(e);
    return 5;
  }
  return 0;
}

// Copy-on-write block copy ("vLLM ve Triton ile maliyet optimizasyonu",
// section 03: a shared block is copied when one holder writes into it).
// One CTA per (pair, K or V): the whole block -- every KV head's 16 rows -- is
// contiguous in the [num_blocks][num_kv_heads][16][head_dim] layout, so each
// CTA streams it with 16-byte loads and stores, eight loads in flight per
// thread before their stores (source and destination are different blocks).
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                       int64_t num_blocks, int chunks_per_block) {
  constexpr int kBatch = 8;
  const int i = blockIdx.x;
  const int32_t s = src[i], d = dst[i];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks || s == d) return;
  uint4* cache = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* from = cache + static_cast<int64_t>(s) * chunks_per_block;
  uint4* to = cache + static_cast<int64_t>(d) * chunks_per_block;
  for (int base = threadIdx.x; base < chunks_per_block; base += kBatch * blockDim.x) {
    uint4 r[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int c = base + j * blockDim.x;
      if (c < chunks_per_block) r[j] = from[c];
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int c = base + j * blockDim.x;
      if (c < chunks_per_block) to[c] = r[j];
    }
  }
}

int copy_blocks_launch(void* k_cache, void* v_cache, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, const int32_t* src, const int32_t* dst, int32_t n_pairs,
                       void* stream, std::string* why) {
  if (n_pairs == 0) return 0;
  const int chunks_per_block = num_kv_heads * kBlock * head_dim * 2 / 16;
  dim3 grid(static_cast<unsigned>(n_pairs), 2);
  copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src, dst, num_blocks,
      chunks_per_block);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("copy_blocks launch: ") + cudaGetErrorString(e);
    return 5;
  }
  return 0;
}

}  // namespace pa
