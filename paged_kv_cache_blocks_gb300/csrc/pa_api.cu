// C ABI of libpa: argument checks, error strings and dispatch to the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {
thread_local std::string g_last_error;
}

void set_error(const std::string& msg) { g_last_error = msg; }

}  // namespace pa

namespace {

int fail(int code, const std::string& msg) {
  pa::set_error(msg);
  return code;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_head_dim(int32_t d) { return d == 64 || d == 128; }

// An NVTX range around one library call, visible to Nsight tools (no cost
// beyond a function-pointer check when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Shapes of the decode call that last planned into a workspace (keyed by
// device and workspace address).  A call with PA_DECODE_REUSE_PLAN is refused
// unless its workspace holds a plan made for the same shapes, so a stale or
// foreign workspace never reaches the kernels as a plan.  A prefill on the
// workspace, or a planning call that fails, drops the record.
struct PlanShape {
  int32_t num_seqs, max_blocks_per_seq, max_seq_len, num_q_heads, num_kv_heads, head_dim,
      num_groups;
  bool operator==(const PlanShape& o) const {
    return num_seqs == o.num_seqs && max_blocks_per_seq == o.max_blocks_per_seq &&
           max_seq_len == o.max_seq_len && num_q_heads == o.num_q_heads &&
           num_kv_heads == o.num_kv_heads && head_dim == o.head_dim && num_groups == o.num_groups;
  }
};
using PlanKey = std::pair<int, uintptr_t>;
constexpr size_t kMaxPlanRecords = 4096;  // beyond this the oldest-keyed records are dropped
std::mutex g_plan_mu;
std::map<PlanKey, PlanShape> g_plans;

PlanKey plan_key(const void* ws) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  return PlanKey(dev, reinterpret_cast<uintptr_t>(ws));
}

bool plan_matches(const void* ws, const PlanShape& shape) {
  const PlanKey k = plan_key(ws);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  auto it = g_plans.find(k);
  return it != g_plans.end() && it->second == shape;
}

void plan_forget(const void* ws) {
  const PlanKey k = plan_key(ws);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plans.erase(k);
}

void plan_record(const void* ws, const PlanShape& shape) {
  const PlanKey k = plan_key(ws);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (g_plans.size() >= kMaxPlanRecords && g_plans.find(k) == g_plans.end())
    g_plans.erase(g_plans.begin());
  g_plans[k] = shape;
}

}  // namespace

extern "C" {

const char* pa_last_error_string(void) { return pa::g_last_error.c_str(); }

const char* pa_version(void) { return "libpa 0.1 (sm_103a)"; }

int pa_cache_write(const void* d_k, const void* d_v, const int64_t* d_slot_mapping, int32_t num_tokens,
                   int32_t num_kv_heads, int32_t head_dim, void* d_k_cache, void* d_v_cache,
                   int64_t num_blocks, int32_t dtype, void* stream) {
  NvtxRange nvtx("pa_cache_write");
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "pa_cache_write: num_tokens < 0");
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_cache_write: dtype");
  if (!supported_head_dim(head_dim))
    return fail(PA_ERR_UNSUPPORTED, "pa_cache_write: head_dim must be 64 or 128");
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID, "pa_cache_write: num_kv_heads and num_blocks must be > 0");
  if (num_tokens == 0) return PA_OK;
  if (!d_k || !d_v || !d_slot_mapping || !d_k_cache || !d_v_cache)
    return fail(PA_ERR_INVALID, "pa_cache_write: NULL pointer");
  if (!aligned(d_k, 16) || !aligned(d_v, 16) || !aligned(d_k_cache, 16) || !aligned(d_v_cache, 16) ||
      !aligned(d_slot_mapping, 8))
    return fail(PA_ERR_INVALID, "pa_cache_write: k, v and caches must be 16-byte aligned");
  std::string why;
  int rc = pa::cache_write_launch(d_k, d_v, d_slot_mapping, num_tokens, num_kv_heads, head_dim,
                                  d_k_cache, d_v_cache, num_blocks, stream, &why);
  return rc ? fail(rc, why) : PA_OK;
}

int pa_cache_write_fp8(const void* d_k, const void* d_v, const int64_t* d_slot_mapping,
                       int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                       const float* d_k_scale, const float* d_v_scale, void* d_k_cache8,
                       void* d_v_cache8, int64_t num_blocks, int32_t dtype, void* stream) {
  NvtxRange nvtx("pa_cache_write_fp8");
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "pa_cache_write_fp8: num_tokens < 0");
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_cache_write_fp8: dtype");
  if (head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "pa_cache_write_fp8: head_dim must be 128");
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID, "pa_cache_write_fp8: num_kv_heads and num_blocks must be > 0");
  if (num_tokens == 0) return PA_OK;
  if (!d_k || !d_v || !d_slot_mapping || !d_k_cache8 || !d_v_cache8 || !d_k_scale || !d_v_scale)
    return fail(PA_ERR_INVALID, "pa_cache_write_fp8: NULL pointer");
  if (!aligned(d_k, 16) || !aligned(d_v, 16) || !aligned(d_k_cache8, 16) || !aligned(d_v_cache8, 16) ||
      !aligned(d_slot_mapping, 8) || !aligned(d_k_scale, 4) || !aligned(d_v_scale, 4))
    return fail(PA_ERR_INVALID, "pa_cache_write_fp8: k, v and caches must be 16-byte aligned");
  std::string why;
  int rc = pa::cache_write_fp8_launch(d_k, d_v, d_slot_mapping, num_tokens, num_kv_heads, head_dim,
                                      d_k_scale, d_v_scale, d_k_cache8, d_v_cache8, num_blocks, dtype,
                                      stream, &why);
  return rc ? fail(rc, why) : PA_OK;
}

int pa_copy_blocks(void* d_k_cache, void* d_v_cache, int64_t num_blocks, int32_t num_kv_heads,
                   int32_t head_dim, const int32_t* d_src, const int32_t* d_dst, int32_t n_pairs,
                   void* stream) {
  NvtxRange nvtx("pa_copy_blocks");
  if (n_pairs < 0) return fail(PA_ERR_INVALID, "pa_copy_blocks: n_pairs < 0");
  if (!supported_head_dim(head_dim))
    return fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: head_dim must be 64 or 128");
  if (num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID, "pa_copy_blocks: num_kv_heads and num_blocks must be > 0");
  if (n_pairs == 0) return PA_OK;
  if (!d_k_cache || !d_v_cache || !d_src || !d_dst)
    return fail(PA_ERR_INVALID, "pa_copy_blocks: NULL pointer");
  if (!aligned(d_k_cache, 16) || !aligned(d_v_cache, 16) || !aligned(d_src, 4) || !aligned(d_dst, 4))
    return fail(PA_ERR_INVALID, "pa_copy_blocks: caches must be 16-byte aligned");
  std::string why;
  int rc = pa::copy_blocks_launch(d_k_cache, d_v_cache, num_blocks, num_kv_heads, head_dim, d_src,
                                  d_dst, n_pairs, stream, &why);
  return rc ? fail(rc, why) : PA_OK;
}

size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_seq_len) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return pa::decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len);
}

}  // extern "C"

namespace {

int decode_common(const void* d_q, const void* d_k_cache, const void* d_v_cache, int64_t num_blocks,
                  const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
                  int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                  int32_t head_dim, float scale, int32_t dtype, void* d_out, void* d_workspace,
                  size_t workspace_bytes, void* stream, const pa_decode_opts* opts,
                  const int32_t* d_group_offsets, const int32_t* d_group_prefix_tokens,
                  int32_t num_groups, const float* d_k_scale = nullptr,
                  const float* d_v_scale = nullptr) {
  const bool fp8 = d_k_scale != nullptr;
  if (num_seqs < 0) return fail(PA_ERR_INVALID, "pa_decode: num_seqs < 0");
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_decode: dtype");
  if (!supported_head_dim(head_dim))
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: head_dim must be 64 or 128");
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "pa_decode: num_q_heads must be a positive multiple of num_kv_heads");
  const int32_t G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: query heads per KV head must be 1, 2, 4 or 8");
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID, "pa_decode: num_blocks and max_blocks_per_seq must be > 0");
  if (num_blocks * num_kv_heads * PA_BLOCK_SIZE > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: num_blocks * num_kv_heads * 16 must be < 2^31");
  if (fp8 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: head_dim must be 128");
  if (fp8 && num_blocks * num_kv_heads * head_dim > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: num_blocks * num_kv_heads * 128 must be < 2^31");
  if (fp8 && (!d_v_scale || !aligned(d_k_scale, 4) || !aligned(d_v_scale, 4)))
    return fail(PA_ERR_INVALID, "pa_decode_fp8: k_scale and v_scale must be device float arrays");
  if (static_cast<int64_t>(max_blocks_per_seq) * PA_BLOCK_SIZE > INT32_MAX)
    return fail(PA_ERR_INVALID, "pa_decode: max_blocks_per_seq too large");
  const int32_t cap = max_blocks_per_seq * PA_BLOCK_SIZE;
  if (max_seq_len <= 0) max_seq_len = cap;
  if (max_seq_len > cap)
    return fail(PA_ERR_INVALID, "pa_decode: max_seq_len exceeds max_blocks_per_seq * 16");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "pa_decode: scale is not finite");
  if (opts && (opts->variant < 0 || opts->variant > 2))
    return fail(PA_ERR_INVALID, "pa_decode: opts->variant must be 0, 1 or 2");
  if (opts && (opts->flags & ~PA_DECODE_REUSE_PLAN))
    return fail(PA_ERR_INVALID, "pa_decode: unknown opts->flags bits");
  if (opts && opts->partition_tokens != 0 && opts->partition_tokens != pa::kPartTokens &&
      opts->partition_tokens != 2 * pa::kPartTokens && opts->partition_tokens != 4 * pa::kPartTokens)
    return fail(PA_ERR_INVALID, "pa_decode: opts->partition_tokens must be 0, 512, 1024 or 2048");
  if (num_seqs == 0) return PA_OK;
  const int64_t per_seq_parts = (max_seq_len + pa::kPartTokens - 1) / pa::kPartTokens;
  if (static_cast<int64_t>(num_seqs) * per_seq_parts * num_kv_heads > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: too many partitions for one call");
  if (!d_q || !d_k_cache || !d_v_cache || !d_block_tables || !d_seq_lens || !d_out || !d_workspace)
    return fail(PA_ERR_INVALID, "pa_decode: NULL pointer");
  if (!aligned(d_k_cache, 16) || !aligned(d_v_cache, 16) || !aligned(d_q, 16) || !aligned(d_out, 16) ||
      !aligned(d_workspace, 256) || !aligned(d_block_tables, 4) || !aligned(d_seq_lens, 4))
    return fail(PA_ERR_INVALID,
                "pa_decode: q, out and caches must be 16-byte aligned, the workspace 256-byte aligned");
  if (num_groups < 0 || num_groups > num_seqs)
    return fail(PA_ERR_INVALID, "pa_decode_grouped: num_groups must be in [1, num_seqs]");
  if (num_groups > 0 && (!d_group_offsets || !d_group_prefix_tokens))
    return fail(PA_ERR_INVALID, "pa_decode_grouped: NULL group array");
  const size_t need = pa::decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len,
                                                 num_groups > 0);
  if (workspace_bytes < need)
    return fail(PA_ERR_INVALID, num_groups > 0
                                    ? "pa_decode_grouped: workspace smaller than pa_decode_grouped_workspace_bytes()"
                                    : "pa_decode: workspace smaller than pa_decode_workspace_bytes()");

  const bool reuse = opts && (opts->flags & PA_DECODE_REUSE_PLAN);
  const PlanShape shape{num_seqs, max_blocks_per_seq, max_seq_len, num_q_heads, num_kv_heads,
                        head_dim, num_groups};
  if (reuse && !plan_matches(d_workspace, shape))
    return fail(PA_ERR_INVALID,
                "pa_decode: PA_DECODE_REUSE_PLAN needs a workspace planned by a decode call "
                "with the same num_seqs, max_blocks_per_seq, max_seq_len, head counts, head_dim "
                "and groups");
  if (!reuse) plan_forget(d_workspace);

  pa::DecodeArgs a;
  a.q = d_q;
  a.k_cache = d_k_cache;
  a.v_cache = d_v_cache;
  a.num_blocks = num_blocks;
  a.block_tables = d_block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.seq_lens = d_seq_lens;
  a.num_seqs = num_seqs;
  a.max_seq_len = max_seq_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.dtype = dtype;
  a.out = d_out;
  a.workspace = d_workspace;
  a.stream = stream;
  a.variant = opts ? opts->variant : 0;
  a.ev_before = opts ? opts->event_before_main : nullptr;
  a.ev_after = opts ? opts->event_after_main : nullptr;
  a.reuse_plan = reuse;
  a.partition_tokens = opts ? opts->partition_tokens : 0;
  a.group_off = d_group_offsets;
  a.group_prefix = d_group_prefix_tokens;
  a.num_groups = num_groups;
  a.fp8 = fp8;
  a.k_scale = d_k_scale;
  a.v_scale = d_v_scale;
  std::string why;
  int rc = pa::decode_launch(a, &why);
  if (rc) {
    plan_forget(d_workspace);
    return fail(rc, why);
  }
  if (!reuse) plan_record(d_workspace, shape);
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_decode_ex(const void* d_q, const void* d_k_cache, const void* d_v_cache, int64_t num_blocks,
                 const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
                 int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                 int32_t head_dim, float scale, int32_t dtype, void* d_out, void* d_workspace,
                 size_t workspace_bytes, void* stream, const pa_decode_opts* opts) {
  NvtxRange nvtx("pa_decode");
  return decode_common(d_q, d_k_cache, d_v_cache, num_blocks, d_block_tables, max_blocks_per_seq,
                       d_seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, scale,
                       dtype, d_out, d_workspace, workspace_bytes, stream, opts, nullptr, nullptr, 0);
}

size_t pa_decode_grouped_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                         int32_t max_seq_len) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return pa::decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len, true);
}

int pa_decode_fp8(const void* d_q, const void* d_k_cache8, const void* d_v_cache8,
                  const float* d_k_scale, const float* d_v_scale, int64_t num_blocks,
                  const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
                  int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                  int32_t head_dim, float scale, int32_t dtype, void* d_out, void* d_workspace,
                  size_t workspace_bytes, void* stream, const pa_decode_opts* opts) {
  NvtxRange nvtx("pa_decode_fp8");
  if (!d_k_scale) return fail(PA_ERR_INVALID, "pa_decode_fp8: NULL k_scale");
  if (opts && opts->variant == 1)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: only the tensor-core variant exists");
  return decode_common(d_q, d_k_cache8, d_v_cache8, num_blocks, d_block_tables, max_blocks_per_seq,
                       d_seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, scale,
                       dtype, d_out, d_workspace, workspace_bytes, stream, opts, nullptr, nullptr,
                       0, d_k_scale, d_v_scale);
}

int pa_decode_grouped(const void* d_q, const void* d_k_cache, const void* d_v_cache,
                      int64_t num_blocks, const int32_t* d_block_tables, int32_t max_blocks_per_seq,
                      const int32_t* d_seq_lens, int32_t num_seqs, int32_t max_seq_len,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                      int32_t dtype, const int32_t* d_group_offsets,
                      const int32_t* d_group_prefix_tokens, int32_t num_groups, void* d_out,
                      void* d_workspace, size_t workspace_bytes, void* stream,
                      const pa_decode_opts* opts) {
  NvtxRange nvtx("pa_decode_grouped");
  if (num_groups <= 0 && num_seqs > 0)
    return fail(PA_ERR_INVALID, "pa_decode_grouped: num_groups must be >= 1");
  return decode_common(d_q, d_k_cache, d_v_cache, num_blocks, d_block_tables, max_blocks_per_seq,
                       d_seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, scale,
                       dtype, d_out, d_workspace, workspace_bytes, stream, opts, d_group_offsets,
                       d_group_prefix_tokens, num_groups);
}

int pa_decode(const void* d_q, const void* d_k_cache, const void* d_v_cache, int64_t num_blocks,
              const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
              int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
              int32_t head_dim, float scale, int32_t dtype, void* d_out, void* d_workspace,
              size_t workspace_bytes, void* stream) {
  return pa_decode_ex(d_q, d_k_cache, d_v_cache, num_blocks, d_block_tables, max_blocks_per_seq,
                      d_seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, scale,
                      dtype, d_out, d_workspace, workspace_bytes, stream, nullptr);
}

size_t pa_prefill_workspace_bytes(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                  int32_t num_kv_heads) {
  if (num_seqs < 0 || num_q_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  return pa::prefill_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads);
}

int pa_prefill(const void* d_q, const void* d_k_cache, const void* d_v_cache, int64_t num_blocks,
               const int32_t* d_block_tables, int32_t max_blocks_per_seq, const int32_t* d_seq_lens,
               const int32_t* d_q_offsets, int32_t num_seqs, int32_t num_q_tokens,
               int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
               float scale, int32_t dtype, void* d_out, void* d_workspace, size_t workspace_bytes,
               void* stream, const pa_decode_opts* opts) {
  NvtxRange nvtx("pa_prefill");
  if (num_seqs < 0 || num_q_tokens < 0)
    return fail(PA_ERR_INVALID, "pa_prefill: num_seqs and num_q_tokens must be >= 0");
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_prefill: dtype");
  if (!supported_head_dim(head_dim))
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill: head_dim must be 64 or 128");
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "pa_prefill: num_q_heads must be a positive multiple of num_kv_heads");
  const int32_t G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill: query heads per KV head must be 1, 2, 4 or 8");
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID, "pa_prefill: num_blocks and max_blocks_per_seq must be > 0");
  if (num_blocks * num_kv_heads * PA_BLOCK_SIZE > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill: num_blocks * num_kv_heads * 16 must be < 2^31");
  if (static_cast<int64_t>(max_blocks_per_seq) * PA_BLOCK_SIZE > INT32_MAX)
    return fail(PA_ERR_INVALID, "pa_prefill: max_blocks_per_seq too large");
  const int32_t cap = max_blocks_per_seq * PA_BLOCK_SIZE;
  if (max_seq_len <= 0) max_seq_len = cap;
  if (max_seq_len > cap)
    return fail(PA_ERR_INVALID, "pa_prefill: max_seq_len exceeds max_blocks_per_seq * 16");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "pa_prefill: scale is not finite");
  if (opts && opts->variant != 0 && opts->variant != 2 && opts->variant != 3)
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill: variant must be 0 (auto), 2 (mma.sync) or 3 (tcgen05)");
  if (opts && (opts->flags != 0 || opts->partition_tokens != 0))
    return fail(PA_ERR_INVALID, "pa_prefill: opts->flags and opts->partition_tokens must be 0");
  if (opts && opts->variant == 3 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill: the tcgen05 variant needs head_dim 128");
  if (num_seqs == 0 || num_q_tokens == 0) return PA_OK;
  if (!d_q || !d_k_cache || !d_v_cache || !d_block_tables || !d_seq_lens || !d_q_offsets || !d_out ||
      !d_workspace)
    return fail(PA_ERR_INVALID, "pa_prefill: NULL pointer");
  if (!aligned(d_k_cache, 16) || !aligned(d_v_cache, 16) || !aligned(d_q, 16) || !aligned(d_out, 16) ||
      !aligned(d_workspace, 256) || !aligned(d_block_tables, 4) || !aligned(d_seq_lens, 4) ||
      !aligned(d_q_offsets, 4))
    return fail(PA_ERR_INVALID,
                "pa_prefill: q, out and caches must be 16-byte aligned, the workspace 256-byte aligned");
  if (workspace_bytes < pa::prefill_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads))
    return fail(PA_ERR_INVALID, "pa_prefill: workspace smaller than pa_prefill_workspace_bytes()");
  pa::PrefillArgs a;
  a.q = d_q;
  a.k_cache = d_k_cache;
  a.v_cache = d_v_cache;
  a.num_blocks = num_blocks;
  a.block_tables = d_block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.seq_lens = d_seq_lens;
  a.q_offsets = d_q_offsets;
  a.num_seqs = num_seqs;
  a.num_q_tokens = num_q_tokens;
  a.max_seq_len = max_seq_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.scale = scale;
  a.dtype = dtype;
  a.out = d_out;
  a.workspace = d_workspace;
  a.stream = stream;
  a.ev_before = opts ? opts->event_before_main : nullptr;
  a.ev_after = opts ? opts->event_after_main : nullptr;
  a.variant = opts ? opts->variant : 0;
  plan_forget(d_workspace);  // the prefill overwrites the workspace
  std::string why;
  int rc = pa::prefill_launch(a, &why);
  return rc ? fail(rc, why) : PA_OK;
}

int pa_decode_check(const void* d_workspace, void* stream, int32_t* error_bits) {
  NvtxRange nvtx("pa_decode_check");
  if (!d_workspace || !error_bits) return fail(PA_ERR_INVALID, "pa_decode_check: NULL argument");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("pa_decode_check: ") + cudaGetErrorString(e));
  int32_t bits = 0;
  e = cudaMemcpy(&bits, d_workspace, sizeof(bits), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("pa_decode_check: ") + cudaGetErrorString(e));
  *error_bits = bits;
  if (bits) return fail(PA_ERR_DEVICE, "pa_decode_check: the device flagged bad input (see error bits)");
  return PA_OK;
}

}  // extern "C"
