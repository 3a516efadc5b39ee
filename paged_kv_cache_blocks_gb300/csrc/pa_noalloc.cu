// pa_decode_noalloc: decode attention for callers that cannot allocate GPU
// memory.  Some callers cannot call cudaMalloc or hand over a workspace:
// code that runs where allocating is not allowed or not safe (inside a
// fixed memory budget planned ahead of time, from a plugin or callback that
// owns no device memory, or next to a caching allocator that must not see
// foreign allocations).  This entry point gives them the same decode with
// no allocation at all: its scratch lives in one statically sized device
// array that the CUDA module holds for as long as the library is loaded.
//
// The array is shared by every call on a device.  Each decode starts by
// rewriting everything it reads from the scratch (its partition list and
// counters), so no clearing is needed between calls, but two calls whose
// kernels overlap on the GPU (different streams, no ordering) race on it.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per device

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Looked up
// once per device (host code only sees a host-side stand-in for the symbol);
// the first call on a device loads the module and must not happen during
// stream capture.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    pa::set_error(std::string("pa_decode_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
    return PA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    pa::set_error("pa_decode_noalloc: device ordinal out of range");
    return PA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      pa::set_error(std::string("pa_decode_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      return PA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(const void* d_q, const void* d_k_cache, const void* d_v_cache,
                                 int64_t num_blocks, const int32_t* d_block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
                                 int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, float scale, int32_t dtype,
                                 void* d_out, void* stream) {
  if (num_seqs > 0 && num_q_heads > 0 && head_dim > 0 && max_blocks_per_seq > 0) {
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * PA_BLOCK_SIZE;
    const int32_t msl = max_seq_len > 0 ? max_seq_len : static_cast<int32_t>(cap > INT32_MAX ? INT32_MAX : cap);
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, msl);
    if (need > kScratchBytes) {
      pa::set_error("pa_decode_noalloc: this batch needs " + std::to_string(need) +
                    " bytes of scratch, more than the fixed " + std::to_string(kScratchBytes) +
                    " bytes (64 MiB); use pa_decode with a caller-provided workspace");
      return PA_ERR_INVALID;
    }
  }
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc != PA_OK) return rc;
  return pa_decode(d_q, d_k_cache, d_v_cache, num_blocks, d_block_tables, max_blocks_per_seq,
                   d_seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, scale,
                   dtype, d_out, ws, kScratchBytes, stream);
}
