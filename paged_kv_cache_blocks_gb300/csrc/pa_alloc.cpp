// Host-side paged KV block allocator (C ABI in pa.h).
//
// Fixed 16-token blocks handed out from a free queue only when a sequence's
// current block is full, ref-counted sharing of blocks between sequences and
// copy-on-write of a shared block on the first write into it:
//   "vLLM Nedir? PagedAttention ile Production LLM Serving", sections
//   "PagedAttention" and "Bir istek motorun icinde" (steps 2 and 5);
//   "vLLM ve Triton ile maliyet optimizasyonu", section 03 (step 3 and the
//   copy-on-write paragraph).
// Where the pages leave a policy open (queue order, all-or-nothing append,
// fork of a partly covered block) this follows the readings listed in pa.h.
#include <deque>
#include <new>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  int32_t num_blocks = 0;
  int32_t block_size = PA_BLOCK_SIZE;
  std::deque<int32_t> free_q;
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_id = 0;
};

namespace {

int fail(int code, const std::string& msg) {
  pa::set_error(msg);
  return code;
}

// Blocks sequence s takes from the free queue for `tokens` more tokens.
int64_t blocks_needed(const pa_alloc& a, const pa_alloc::Seq& s, int64_t tokens, bool* cow) {
  const int64_t bs = a.block_size;
  int64_t need = 0;
  *cow = false;
  if (tokens > 0 && !s.table.empty() && s.len % bs != 0 && a.ref[s.table.back()] > 1) {
    *cow = true;
    need += 1;
  }
  const int64_t have = static_cast<int64_t>(s.table.size()) * bs;
  const int64_t extra = s.len + tokens - have;
  if (extra > 0) need += (extra + bs - 1) / bs;
  return need;
}

}  // namespace

extern "C" {

int pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                    pa_alloc_t** out) {
  if (!out) return fail(PA_ERR_INVALID, "pa_alloc_create: out is NULL");
  *out = nullptr;
  if (num_blocks <= 0) return fail(PA_ERR_INVALID, "pa_alloc_create: num_blocks must be > 0");
  if (block_size != PA_BLOCK_SIZE)
    return fail(PA_ERR_UNSUPPORTED, "pa_alloc_create: block_size must be 16");
  pa_alloc* a = new (std::nothrow) pa_alloc;
  if (!a) return fail(PA_ERR_OOM, "pa_alloc_create: host allocation failed");
  a->num_blocks = num_blocks;
  a->ref.assign(num_blocks, 0);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete a;
        return fail(PA_ERR_INVALID, "pa_alloc_create: free_order is not a permutation of 0..num_blocks-1");
      }
      seen[b] = 1;
      a->free_q.push_back(b);
    }
  } else {
    for (int32_t i = 0; i < num_blocks; ++i) a->free_q.push_back(i);
  }
  *out = a;
  return PA_OK;
}

void pa_alloc_destroy(pa_alloc_t* a) { delete a; }

int pa_seq_create(pa_alloc_t* a, int64_t* seq_id_out) {
  if (!a || !seq_id_out) return fail(PA_ERR_INVALID, "pa_seq_create: NULL argument");
  const int64_t id = a->next_id++;
  a->seqs.emplace(id, pa_alloc::Seq{});
  *seq_id_out = id;
  return PA_OK;
}

int pa_seq_fork(pa_alloc_t* a, int64_t parent, int32_t prefix_tokens, int64_t* child_out) {
  if (!a || !child_out) return fail(PA_ERR_INVALID, "pa_seq_fork: NULL argument");
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return fail(PA_ERR_INVALID, "pa_seq_fork: unknown parent sequence");
  if (prefix_tokens < 0 || prefix_tokens > it->second.len)
    return fail(PA_ERR_INVALID, "pa_seq_fork: prefix_tokens outside [0, parent length]");
  const int64_t nblk = (prefix_tokens + a->block_size - 1) / a->block_size;
  pa_alloc::Seq child;
  child.table.assign(it->second.table.begin(), it->second.table.begin() + nblk);
  child.len = prefix_tokens;
  for (int32_t b : child.table) a->ref[b] += 1;
  const int64_t id = a->next_id++;
  a->seqs.emplace(id, std::move(child));
  *child_out = id;
  return PA_OK;
}

int pa_seq_free(pa_alloc_t* a, int64_t seq_id) {
  if (!a) return fail(PA_ERR_INVALID, "pa_seq_free: NULL allocator");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return fail(PA_ERR_INVALID, "pa_seq_free: unknown or already freed sequence");
  for (int32_t b : it->second.table) {
    if (--a->ref[b] == 0) a->free_q.push_back(b);
  }
  a->seqs.erase(it);
  return PA_OK;
}

int pa_seq_append_slots(pa_alloc_t* a, const int64_t* seq_ids, int32_t n_seqs, int32_t tokens_each,
                        int64_t* slot_mapping_out, int32_t* cow_src_out, int32_t* cow_dst_out,
                        int32_t cow_capacity, int32_t* n_cow_out, int32_t* block_table_io,
                        int32_t max_blocks, int32_t* seq_lens_io) {
  if (!a) return fail(PA_ERR_INVALID, "pa_seq_append_slots: NULL allocator");
  if (n_seqs < 0 || tokens_each < 0)
    return fail(PA_ERR_INVALID, "pa_seq_append_slots: negative count");
  if (n_seqs > 0 && (!seq_ids || (tokens_each > 0 && !slot_mapping_out)))
    return fail(PA_ERR_INVALID, "pa_seq_append_slots: NULL array");
  if (block_table_io && max_blocks <= 0)
    return fail(PA_ERR_INVALID, "pa_seq_append_slots: max_blocks must be > 0 with a table");
  // Validate everything before changing anything.
  std::vector<pa_alloc::Seq*> seqs(n_seqs);
  std::unordered_set<int64_t> seen;
  int64_t need = 0, n_cow = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end()) return fail(PA_ERR_INVALID, "pa_seq_append_slots: unknown sequence");
    if (!seen.insert(seq_ids[i]).second)
      return fail(PA_ERR_INVALID, "pa_seq_append_slots: a sequence appears twice");
    seqs[i] = &it->second;
    bool cow = false;
    need += blocks_needed(*a, *seqs[i], tokens_each, &cow);
    n_cow += cow;
    if (block_table_io) {
      const int64_t after = (seqs[i]->len + tokens_each + a->block_size - 1) / a->block_size;
      if (after > max_blocks)
        return fail(PA_ERR_INVALID, "pa_seq_append_slots: a table row would exceed max_blocks");
    }
  }
  // A write into a block other sequences still hold must be preceded by a
  // copy; a call that cannot report the copy would write into the shared block.
  if (n_cow > 0 && (!cow_src_out || !cow_dst_out || n_cow > cow_capacity))
    return fail(PA_ERR_SHARED_WRITE,
                "pa_seq_append_slots: a write would land in a shared block and the copy-on-write "
                "pairs exceed cow_capacity");
  if (need > static_cast<int64_t>(a->free_q.size()))
    return fail(PA_ERR_OOM, "pa_seq_append_slots: free queue cannot cover the request");

  const int64_t bs = a->block_size;
  int64_t k = 0;
  int32_t c = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    pa_alloc::Seq& s = *seqs[i];
    int32_t* row = block_table_io ? block_table_io + static_cast<int64_t>(i) * max_blocks : nullptr;
    for (int32_t n = 0; n < tokens_each; ++n) {
      const int64_t pos = s.len;
      const int64_t j = pos / bs, off = pos % bs;
      if (j == static_cast<int64_t>(s.table.size())) {  // current block is full
        const int32_t b = a->free_q.front();
        a->free_q.pop_front();
        a->ref[b] = 1;
        s.table.push_back(b);
        if (row) row[j] = b;
      } else if (a->ref[s.table[j]] > 1) {               // first write into a shared block
        const int32_t src = s.table[j];
        const int32_t dst = a->free_q.front();
        a->free_q.pop_front();
        a->ref[dst] = 1;
        a->ref[src] -= 1;
        s.table[j] = dst;
        cow_src_out[c] = src;
        cow_dst_out[c] = dst;
        ++c;
        if (row) row[j] = dst;
      }
      slot_mapping_out[k++] = static_cast<int64_t>(s.table[j]) * bs + off;
      s.len = pos + 1;
    }
    if (seq_lens_io) seq_lens_io[i] = static_cast<int32_t>(s.len);
  }
  if (n_cow_out) *n_cow_out = c;
  return PA_OK;
}

int pa_seq_block_table(pa_alloc_t* a, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                       int32_t* table_out, int32_t* seq_lens_out) {
  if (!a) return fail(PA_ERR_INVALID, "pa_seq_block_table: NULL allocator");
  if (n < 0 || max_blocks <= 0) return fail(PA_ERR_INVALID, "pa_seq_block_table: bad sizes");
  if (n > 0 && (!seq_ids || !table_out)) return fail(PA_ERR_INVALID, "pa_seq_block_table: NULL array");
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end()) return fail(PA_ERR_INVALID, "pa_seq_block_table: unknown sequence");
    if (static_cast<int64_t>(it->second.table.size()) > max_blocks)
      return fail(PA_ERR_INVALID, "pa_seq_block_table: a row exceeds max_blocks");
  }
  for (int32_t i = 0; i < n; ++i) {
    const pa_alloc::Seq& s = a->seqs.find(seq_ids[i])->second;
    int32_t* row = table_out + static_cast<int64_t>(i) * max_blocks;
    const int32_t nb = static_cast<int32_t>(s.table.size());
    for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < nb ? s.table[j] : -1;
    if (seq_lens_out) seq_lens_out[i] = static_cast<int32_t>(s.len);
  }
  return PA_OK;
}

int pa_alloc_stats(pa_alloc_t* a, pa_stats_t* out) {
  if (!a || !out) return fail(PA_ERR_INVALID, "pa_alloc_stats: NULL argument");
  pa_stats_t st{};
  st.num_blocks = a->num_blocks;
  st.free_blocks = static_cast<int64_t>(a->free_q.size());
  for (int32_t r : a->ref) {
    st.used_blocks += r > 0;
    st.shared_blocks += r > 1;
    st.refs += r;
  }
  st.seqs = static_cast<int64_t>(a->seqs.size());
  for (const auto& kv : a->seqs)
    st.frag_tokens += static_cast<int64_t>(kv.second.table.size()) * a->block_size - kv.second.len;
  *out = st;
  return PA_OK;
}

}  // extern "C"
