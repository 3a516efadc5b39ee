// Internal host-side interfaces between the C ABI layer and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <string>

namespace pa {

// Sets the calling thread's message for pa_last_error_string().
void set_error(const std::string& msg);

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* seq_lens;
  int32_t num_seqs;
  int32_t max_seq_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  float scale;
  int32_t dtype;
  void* out;
  void* workspace;
  void* stream;
  int32_t variant;
  void* ev_before;
  void* ev_after;
  const int32_t* group_off = nullptr;     // grouped decode: [num_groups + 1] (device)
  const int32_t* group_prefix = nullptr;  // [num_groups] shared prefix tokens (device)
  int32_t num_groups = 0;
  bool fp8 = false;                       // E4M3 caches (K token-major, V dim-major)
  const float* k_scale = nullptr;         // [num_kv_heads] (device), FP8 only
  const float* v_scale = nullptr;
  bool reuse_plan = false;                // skip the prep kernel: the workspace holds the plan
  int32_t partition_tokens = 0;           // 0: chosen by the prep kernel; else 512 / 1024 / 2048
};

// Both return 0 on success or a pa_status code, with *why set on failure.
int decode_launch(const DecodeArgs& a, std::string* why);
size_t decode_workspace_bytes(int64_t num_seqs, int64_t num_q_heads, int64_t head_dim,
                              int64_t max_seq_len, bool grouped = false);

struct PrefillArgs {
  const void* q;              // [num_q_tokens][num_q_heads][head_dim]
  const void* k_cache;
  const void* v_cache;
  int64_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* seq_lens;
  const int32_t* q_offsets;   // [num_seqs + 1]
  int32_t num_seqs;
  int32_t num_q_tokens;
  int32_t max_seq_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  float scale;
  int32_t dtype;
  void* out;
  void* workspace;
  void* stream;
  void* ev_before;
  void* ev_after;
  int32_t variant = 0;        // 0 auto, 2 mma.sync, 3 tcgen05 (head_dim 128)
};

int prefill_launch(const PrefillArgs& a, std::string* why);
size_t prefill_workspace_bytes(int64_t num_seqs, int64_t num_q_tokens, int64_t num_q_heads,
                               int64_t num_kv_heads);

int cache_write_launch(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                       int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                       int64_t num_blocks, void* stream, std::string* why);

int cache_write_fp8_launch(const void* k, const void* v, const int64_t* slot_mapping,
                           int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                           const float* k_scale, const float* v_scale, void* k_cache, void* v_cache,
                           int64_t num_blocks, int32_t dtype, void* stream, std::string* why);

int copy_blocks_launch(void* k_cache, void* v_cache, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, const int32_t* src, const int32_t* dst, int32_t n_pairs,
                       void* stream, std::string* why);

}  // namespace pa
