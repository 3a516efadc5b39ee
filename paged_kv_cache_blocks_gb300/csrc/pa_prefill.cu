// Multi-query paged attention (chunked prefill) for sm_103a.
//
// What it computes: a long prompt is prefilled in pieces that fit a step's
// token budget, each iteration together with the running sequences' decode
// tokens ("Yerel LLM sistemlerinde backpressure ve olcekleme", section
// "4. Prefill ve decode"; "vLLM Nedir? PagedAttention ile Production LLM
// Serving", section "Chunked prefill").  Sequence b holds L_b tokens in its
// blocks once its piece's K/V are written; the piece is the last Q_b of
// them, so query j sits at position L_b - Q_b + j and attends causally to
// tokens 0 .. L_b - Q_b + j.  A decode token is a piece of one.  Scaled
// dot-product attention with grouped-query heads as in the decode kernels.
//
// Two kernels on the caller's stream:
//   1. prefill_prep (1 CTA)  validates the pieces, cuts every piece into
//                            tiles of 16 * NW query rows (a row = one query
//                            token x one of the G heads of a KV head) and
//                            lists them in the workspace by descending number
//                            of key blocks (longest first);
//   2. prefill_tc (head_dim 128, tcgen05; described below) or prefill
//      (mma.sync; persistent, one CTA per SM)
//                            one work item = (KV head, tile), taken from an
//                            atomic counter, KV-head-major so that the CTAs
//                            running together share their K/V in L2.  Warp NW
//                            streams the key blocks 0 .. (last position)/16
//                            with TMA into a ring of shared-memory stages
//                            (128-byte swizzle, mbarriers); each of the NW
//                            consumer warps owns 16 query rows with Q in
//                            registers and runs S = Q K^T and O += P V on
//                            mma.sync m16n8k16 for every block (P reused from
//                            the score accumulators), online softmax in fp32,
//                            the causal mask on the blocks that cross a row's
//                            position, and writes its rows' outputs.
#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

struct PrefillHeader {
  int32_t error_bits;
  int32_t n_entries;   // tiles of all pieces
  int32_t next_item;   // dynamic work counter
  int32_t pad[61];
};
static_assert(sizeof(PrefillHeader) == 256, "header is one 256-byte line");

constexpr int kPrefillBins = 1024;  // key-length bins of the longest-first order

struct PrefillParams {
  const void* q;        // [num_q_tokens][hq][D]
  void* out;            // same shape
  const int32_t* tables;
  const int32_t* seq_lens;
  const int32_t* q_off;  // [num_seqs + 1]
  PrefillHeader* ws;
  int4* entries;         // (sequence, tile, key blocks, 0), longest first
  int64_t num_blocks;
  int max_blocks, num_seqs, num_q_tokens, max_seq_len, hq, hkv, G;
  int tile_tokens;       // query tokens per tile = 16 * NW / G
  int max_entries;       // capacity of `entries`
  float scale_log2;
};

// Validated view of sequence b: clamped length, first query token, piece
// length.  Bad input is flagged and clamped so no access leaves its buffer.
struct PieceView {
  int L, q0, n;
};

__device__ __forceinline__ PieceView piece_view(const PrefillParams& P, int b, bool flag) {
  int L = P.seq_lens[b];
  int a = P.q_off[b], e = P.q_off[b + 1];
  bool bad = false;
  if (L < 0 || L > P.max_seq_len) {
    bad = true;
    L = L < 0 ? 0 : P.max_seq_len;
  }
  if (a < 0 || a > P.num_q_tokens || e < a || e > P.num_q_tokens || (b == 0 && a != 0)) bad = true;
  a = min(max(a, 0), P.num_q_tokens);
  e = min(max(e, a), P.num_q_tokens);
  if (e - a > L) bad = true;  // a piece longer than its sequence
  if (bad && flag) atomicOr(&P.ws->error_bits, kErrSeqLen);
  return PieceView{L, a, e - a};
}

// Key blocks a tile needs: up to the position of its last query token.
__device__ __forceinline__ int tile_key_blocks(const PieceView& v, int tile, int tile_tokens) {
  const int last = min((tile + 1) * tile_tokens, v.n) - 1;
  const int maxpos = min(v.L - v.n + last, v.L - 1);
  return maxpos < 0 ? 0 : (maxpos + kBlock) / kBlock;
}

constexpr int kPrepSeqs = 4096;   // sequences whose tile offsets the prep keeps in shared memory

__global__ void __launch_bounds__(1024) prefill_prep_kernel(PrefillParams P) {
  __shared__ int sw[32];
  __shared__ int s_hist[kPrefillBins];
  __shared__ int s_first[kPrepSeqs + 1];   // first global tile index of each sequence
  __shared__ int s_shift;
  const int tid = threadIdx.x, nthr = blockDim.x;
  if (tid == 0) {
    P.ws->error_bits = 0;
    int sh = 0;
    while ((P.max_blocks >> sh) >= kPrefillBins) ++sh;
    s_shift = sh;
  }
  for (int i = tid; i < kPrefillBins; i += nthr) s_hist[i] = 0;
  __syncthreads();
  const int shift = s_shift;
  if (P.num_seqs <= kPrepSeqs) {
    // one thread per (sequence, tile): the tile counts' prefix sum in shared
    // memory maps a global tile index back to its sequence (binary search),
    // so a long piece's tiles spread over all threads
    const int per = (P.num_seqs + nthr - 1) / nthr;   // <= 4 sequences per thread
    const int b0 = tid * per;
    int cnt = 0;
    for (int k = 0; k < per; ++k) {
      const int b = b0 + k;
      if (b < P.num_seqs) {
        const PieceView v = piece_view(P, b, true);   // flags bad input once per sequence
        const int nt = (v.n + P.tile_tokens - 1) / P.tile_tokens;
        s_first[b] = nt;                                // count for now
        cnt += nt;
      }
    }
    __syncthreads();
    int total_tiles = 0;
    int run = block_exclusive_scan(cnt, sw, &total_tiles);
    for (int k = 0; k < per; ++k) {
      const int b = b0 + k;
      if (b < P.num_seqs) {
        const int nt = s_first[b];
        s_first[b] = run;
        run += nt;
      }
    }
    if (tid == 0) s_first[P.num_seqs] = total_tiles;
    __syncthreads();
    auto locate = [&](int g, int* tile) -> int {   // sequence of global tile g
      int lo = 0, hi = P.num_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_first[mid] <= g) lo = mid;
        else hi = mid - 1;
      }
      *tile = g - s_first[lo];
      return lo;
    };
    for (int g = tid; g < total_tiles; g += nthr) {
      int t;
      const int b = locate(g, &t);
      const PieceView v = piece_view(P, b, false);
      atomicAdd(&s_hist[min(tile_key_blocks(v, t, P.tile_tokens) >> shift, kPrefillBins - 1)], 1);
    }
    __syncthreads();
    // start offsets in descending bin order: a scan over the reversed bins
    int total = 0;
    const int c = tid < kPrefillBins ? s_hist[kPrefillBins - 1 - tid] : 0;
    const int off = block_exclusive_scan(c, sw, &total);
    if (tid < kPrefillBins) s_hist[kPrefillBins - 1 - tid] = off;
    __syncthreads();
    for (int g = tid; g < total_tiles; g += nthr) {
      int t;
      const int b = locate(g, &t);
      const PieceView v = piece_view(P, b, false);
      const int kb = tile_key_blocks(v, t, P.tile_tokens);
      const int slot = atomicAdd(&s_hist[min(kb >> shift, kPrefillBins - 1)], 1);
      // overlapping pieces (offsets out of order, already flagged) cannot
      // overflow the list: records past its capacity are dropped
      if (slot < P.max_entries) P.entries[slot] = make_int4(b, t, kb, 0);
    }
    if (tid == 0) {
      if (total > P.max_entries) atomicOr(&P.ws->error_bits, kErrSeqLen);
      P.ws->n_entries = min(total, P.max_entries);
      P.ws->next_item = 0;
    }
    return;
  }
  // many sequences: one thread per sequence walks its tiles
  for (int b = tid; b < P.num_seqs; b += nthr) {
    const PieceView v = piece_view(P, b, true);
    const int nt = (v.n + P.tile_tokens - 1) / P.tile_tokens;
    for (int t = 0; t < nt; ++t)
      atomicAdd(&s_hist[min(tile_key_blocks(v, t, P.tile_tokens) >> shift, kPrefillBins - 1)], 1);
  }
  __syncthreads();
  // start offsets in descending bin order: a scan over the reversed bins
  int total = 0;
  const int c = tid < kPrefillBins ? s_hist[kPrefillBins - 1 - tid] : 0;
  const int off = block_exclusive_scan(c, sw, &total);
  if (tid < kPrefillBins) s_hist[kPrefillBins - 1 - tid] = off;
  __syncthreads();
  for (int b = tid; b < P.num_seqs; b += nthr) {
    const PieceView v = piece_view(P, b, false);
    const int nt = (v.n + P.tile_tokens - 1) / P.tile_tokens;
    for (int t = 0; t < nt; ++t) {
      const int kb = tile_key_blocks(v, t, P.tile_tokens);
      const int slot = atomicAdd(&s_hist[min(kb >> shift, kPrefillBins - 1)], 1);
      if (slot < P.max_entries) P.entries[slot] = make_int4(b, t, kb, 0);
    }
  }
  if (tid == 0) {
    if (total > P.max_entries) atomicOr(&P.ws->error_bits, kErrSeqLen);
    P.ws->n_entries = min(total, P.max_entries);
    P.ws->next_item = 0;
  }
}

template <int D>
struct PrefillTile {
  static constexpr int kHalfBytes = 16 * 64 * 2;         // one 16 x 64 box
  static constexpr int kHalves = D / 64;
  static constexpr int kKVBytes = kHalves * kHalfBytes;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kKVBytes;       // K then V
};

__device__ __forceinline__ uint32_t tile_chunk(uint32_t tile, int r, int c) {
  return tile + (c >> 3) * 2048 + swz128(r, c & 7);
}

template <int D, int NW, int S>
struct PrefillCfg {
  static constexpr int kThreads = 32 * (NW + 1);
  static constexpr int kStageBytes = PrefillTile<D>::kStageBytes;
  // stages, full + empty barriers, item slot, abort flag; 1 KB for alignment
  static constexpr size_t kBytes = static_cast<size_t>(S) * kStageBytes + 2 * S * 8 + 16 + 1024;
};

template <typename T, int D, int NW, int S>
__global__ void __launch_bounds__(32 * (NW + 1), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const PrefillParams P) {
  using Cfg = PrefillCfg<D, NW, S>;
  using Tl = PrefillTile<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  volatile int* s_item = reinterpret_cast<volatile int*>(empty + S);
  volatile int* abort_flag = s_item + 1;
  int* err = &P.ws->error_bits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = P.G;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == NW && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  const int n_entries = *reinterpret_cast<volatile int32_t*>(&P.ws->n_entries);
  const int n_work = n_entries * P.hkv;
  const int64_t y_oob = P.num_blocks * P.hkv * kBlock;
  uint32_t u_base = 0;    // key blocks this CTA has streamed so far (ring position)
  uint32_t u_issued = 0;  // producer: uses of the ring whose copies were issued
  while (true) {
    if (tid == 0) *s_item = atomicAdd(&P.ws->next_item, 1);
    __syncthreads();
    const int wi = *s_item;
    if (wi >= n_work || *abort_flag) break;
    const int h = wi / n_entries;
    const int4 ent = P.entries[wi - h * n_entries];
    const int b = ent.x, tile = ent.y, nkb = ent.z;
    const PieceView v = piece_view(P, b, false);
    if (warp == NW) {
      // ---- producer: key blocks 0 .. nkb-1 of (b, h) into the ring ----
      const int32_t* trow = P.tables + static_cast<int64_t>(b) * P.max_blocks;
      int32_t ids = 0;
      for (int j = 0; j < nkb; ++j) {
        if ((j & 31) == 0) {
          const int jj = j + lane;
          int32_t id = jj < nkb ? trow[jj] : 0;
          if (jj < nkb && (id < 0 || id >= P.num_blocks)) {
            atomicOr(err, kErrBlockId);
            id = -1;
          }
          ids = id;
        }
        const int32_t id = __shfl_sync(0xffffffffu, ids, j & 31);
        const uint32_t u = u_base + j;
        const int s = u % S;
        bool ok = true;
        if (u >= S) ok = mbar_wait(&empty[s], ((u / S) - 1) & 1, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
          const int32_t y = static_cast<int32_t>(id < 0 ? y_oob : (static_cast<int64_t>(id) * P.hkv + h) * kBlock);
          uint8_t* dst = smem + static_cast<size_t>(s) * Cfg::kStageBytes;
#pragma unroll
          for (int hf = 0; hf < Tl::kHalves; ++hf) {
            tma_load_2d(dst + hf * Tl::kHalfBytes, &tm_k, hf * 64, y, &full[s]);
            tma_load_2d(dst + Tl::kKVBytes + hf * Tl::kHalfBytes, &tm_v, hf * 64, y, &full[s]);
          }
        }
        u_issued = u + 1;
      }
    } else {
      // ---- consumer warp: 16 query rows (row r -> token r / G, head r % G) ----
      const int base = v.L - v.n;                      // position of the piece's first token
      const int tok_w0 = tile * P.tile_tokens + (warp * 16) / G;
      const int tok_w1 = min(tile * P.tile_tokens + (warp * 16 + 15) / G, v.n - 1);
      const int wmax = min(base + tok_w1, v.L - 1);    // the warp's last position
      const bool active = tok_w0 < v.n && wmax >= 0;
      const int wmin = base + tok_w0;
      const int r0 = warp * 16 + g, r1 = r0 + 8;
      const int tq0 = tile * P.tile_tokens + r0 / G, tq1 = tile * P.tile_tokens + r1 / G;
      const int pos0 = base + tq0, pos1 = base + tq1;
      const bool ok0 = tq0 < v.n && pos0 >= 0, ok1 = tq1 < v.n && pos1 >= 0;
      const int lim0 = ok0 ? pos0 : wmax, lim1 = ok1 ? pos1 : wmax;  // last key each row sees
      const T* q0p = static_cast<const T*>(P.q) + ((static_cast<int64_t>(v.q0) + tq0) * P.hq + h * G + r0 % G) * D;
      const T* q1p = static_cast<const T*>(P.q) + ((static_cast<int64_t>(v.q0) + tq1) * P.hq + h * G + r1 % G) * D;
      uint32_t qa[D / 16][4];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + 16 * ks + 2 * t) : 0u;
        qa[ks][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + 16 * ks + 2 * t) : 0u;
        qa[ks][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0p + 16 * ks + 2 * t + 8) : 0u;
        qa[ks][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1p + 16 * ks + 2 * t + 8) : 0u;
      }
      float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
      float o[D / 8][4];
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
      bool alive = true;
      for (int j = 0; j < nkb; ++j) {
        const uint32_t u = u_base + j;
        const int s = u % S;
        alive = mbar_wait(&full[s], (u / S) & 1, abort_flag, err);
        if (!__all_sync(0xffffffffu, alive)) {
          alive = false;
          break;
        }
        const int k0 = j * kBlock;
        if (active && k0 <= wmax) {
          const uint32_t sK = smem_u32(smem + static_cast<size_t>(s) * Cfg::kStageBytes);
          const uint32_t sV = sK + Tl::kKVBytes;
          float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
          {
            const int tok = (lane & 7) + ((lane >> 4) << 3);
            const int cofs = (lane >> 3) & 1;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              uint32_t b00, b01, b10, b11;
              ldmatrix_x4(b00, b01, b10, b11, tile_chunk(sK, tok, 2 * ks + cofs));
              Mma<T>::run(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
              Mma<T>::run(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
            }
          }
          // row g: s*[0], s*[1]; row g + 8: s*[2], s*[3]; keys 2t, 2t+1 (+8 for s1)
          const bool edge = k0 + kBlock - 1 > wmin || k0 + kBlock > v.L;
          float x[2][4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            x[e][0] = s0[2 * e] * P.scale_log2;
            x[e][1] = s0[2 * e + 1] * P.scale_log2;
            x[e][2] = s1[2 * e] * P.scale_log2;
            x[e][3] = s1[2 * e + 1] * P.scale_log2;
          }
          if (edge) {  // causal mask (and the block's tail past the sequence)
            const int kk[4] = {k0 + 2 * t, k0 + 2 * t + 1, k0 + 8 + 2 * t, k0 + 9 + 2 * t};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (kk[c] > lim0) x[0][c] = -INFINITY;
              if (kk[c] > lim1) x[1][c] = -INFINITY;
            }
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
          // V rows past the sequence end may hold anything (NaN): zero them
          // in the operand so that 0 * NaN never enters the sums
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (k0 + kBlock > v.L) {
            mlo = (k0 + 2 * t < v.L ? 0x0000ffffu : 0u) | (k0 + 2 * t + 1 < v.L ? 0xffff0000u : 0u);
            mhi = (k0 + 8 + 2 * t < v.L ? 0x0000ffffu : 0u) | (k0 + 9 + 2 * t < v.L ? 0xffff0000u : 0u);
          }
          {
            const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
            const int cofs = lane >> 4;
#pragma unroll
            for (int nd = 0; nd < D / 8; nd += 2) {
              uint32_t b00, b01, b10, b11;
              ldmatrix_x4_trans(b00, b01, b10, b11, tile_chunk(sV, tok, nd + cofs));
              Mma<T>::run(o[nd], pa0, pa1, pa2, pa3, b00 & mlo, b01 & mhi);
              Mma<T>::run(o[nd + 1], pa0, pa1, pa2, pa3, b10 & mlo, b11 & mhi);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (alive) {
        // this warp's rows: out = o / l, one rounding to T
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float L = lr[e];
          L += __shfl_xor_sync(0xffffffffu, L, 1);
          L += __shfl_xor_sync(0xffffffffu, L, 2);
          const int tq = e ? tq1 : tq0;
          const int r = e ? r1 : r0;
          const bool rv = e ? ok1 : ok0;
          if (tq < v.n) {
            const float inv = (rv && L > 0.f) ? 1.0f / L : 0.f;
            T* dst = static_cast<T*>(P.out) + ((static_cast<int64_t>(v.q0) + tq) * P.hq + h * G + r % G) * D;
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd)
              *reinterpret_cast<uint32_t*>(dst + 8 * nd + 2 * t) =
                  pack2<T>(o[nd][2 * e] * inv, o[nd][2 * e + 1] * inv);
          }
        }
      }
    }
    u_base += nkb;
    __syncthreads();
  }
  if (*abort_flag && warp == NW && lane == 0) {
    // let this CTA's copies in flight land before it leaves: the last use of
    // each stage completes after every earlier one
    const unsigned long long t0 = global_timer_ns();
    for (int s = 0; s < S; ++s) {
      if (u_issued <= static_cast<uint32_t>(s)) break;
      const uint32_t last = u_issued - 1 - ((u_issued - 1 - s) % S);
      while (!mbar_try_wait(&full[s], (last / S) & 1) && global_timer_ns() - t0 < kWaitLimitNs / 4) {
      }
    }
  }
}

// ---------------------------------------------------------------------------
// tcgen05 version (head_dim 128).  One work item = (KV head, tile of 128 query
// rows) as above.  Per CTA (one per SM, 14 warps):
//   warps 8-11  producers: warp 8 takes items from the atomic counter,
//               publishes them in a two-slot item ring and TMA-loads the
//               tile's Q (128 rows x 128 dims, one 3-D box of tokens x heads
//               x dims) into shared memory; all four load the key blocks in
//               chunks of 8 blocks = 128 keys (K one chunk ahead of V) into
//               three-stage K and V rings, each warp issuing the copies of
//               two blocks (K and V of a chunk are 128 swizzled rows per
//               64-dim half, so one descriptor spans the chunk).  TMA issue
//               from one warp is too slow for a chunk;
//   warp 12     allocates the tensor memory (S | P | O0 | O1 | Q); one thread
//               issues S = Q K^T (M 128, N 128 keys, K 128 dims) for chunk
//               c+1 as soon as the softmax of chunk c has read S;
//   warp 13     one thread issues, per key half hk, O_hk += P[:, 64 hk ..]
//               V[64 hk .., :] (M 128, N 128 dims, K 64 keys) once that
//               half's softmax warps have written P.  Issuing a product
//               blocks the thread about as long as the product runs, hence
//               two issuers.  Both products take their A operand (Q, P) from
//               tensor memory, which runs them at the full rate where an A
//               operand in shared memory halves it; tcgen05.commit signals
//               each result on an mbarrier;
//   warps 0-7   two threads per query row (its tensor-memory lane): warp w
//               takes keys 0-63 of every chunk, warp w + 4 keys 64-127.  At
//               the start of an item each moves its 64 dims of the Q row from
//               shared to tensor memory; per chunk it reads its 64 scores,
//               applies the scale and the causal mask, runs an online softmax
//               in fp32 with its own running maximum (moved only when it
//               grows by more than 2^8: the exact result either way, fewer
//               rescales of its O), scale-and-subtract and row sums on the
//               packed two-lane fp32 FMA / add, and writes its P as 16-bit
//               values, two per column.  The halves never wait for each other
//               inside an item; at its end they exchange (maximum, sum) and
//               each writes 64 dims of (O0 2^(m0-m) + O1 2^(m1-m)) / l.
// The softmax warpgroups take registers the producer warpgroup gives back
// (setmaxnreg), so that nothing spills.
// Every wait is bounded; a timeout flags PA_DEVERR_TIMEOUT and the CTA
// drains its copies and tensor-core work before freeing tensor memory.

// One 32-bit tensor-memory column of this thread's lane, stored / loaded
// and waited for in the same statement.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(__float_as_uint(v))
      : "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}

struct TcCfg {
  static constexpr int kHalf = 128 * 128;           // 128 rows x 64 16-bit values
  static constexpr int kQBytes = 2 * kHalf;          // Q tile, head_dim 128
  static constexpr int kChunkBytes = 2 * kHalf;      // K (or V) of one chunk of 128 keys
  static constexpr int kChunkBlocks = 8;
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 3;
  static constexpr size_t kOffQ = 0;
  static constexpr size_t kOffK = kOffQ + kQBytes;
  static constexpr size_t kOffV = kOffK + static_cast<size_t>(kKStages) * kChunkBytes;
  static constexpr size_t kOffBar = kOffV + static_cast<size_t>(kVStages) * kChunkBytes;
  static constexpr size_t kBytes = kOffBar + 512 + 1024;
  static constexpr int kSoftmaxWarps = 8;            // warpgroups 0 and 1: key halves 0 and 1
  static constexpr int kProducerWarp0 = 8;           // warpgroup 2
  static constexpr int kProducerWarps = 4;           // one per SM sub-partition: TMA issue
                                                     // from one warp is too slow for a chunk
  static constexpr int kMmaWarp = 12;                // warps 12 (S) and 13 (PV)
  static constexpr int kMmaWarps = 2;
  static constexpr int kThreads = 32 * (kMmaWarp + kMmaWarps);
  // registers per thread: 128 at launch (four warps on one sub-partition);
  // the producers drop to 64 and the softmax threads rise to 160:
  // 256 x 160 + 128 x 64 + 64 x 128 = 57344 <= 448 x 128 = 57344
  static constexpr int kRegsLaunch = 128, kRegsProducer = 64, kRegsSoftmax = 160;
  // tensor memory: S (128 fp32 columns) | P (128 16-bit values per row in 64
  // columns, keys 0-63 then 64-127) | O0 | O1 (128 fp32 columns each: the
  // products over keys 0-63 and 64-127 of every chunk, each half with its own
  // running maximum) | Q (128 16-bit values per row in 64 columns)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColP = 128, kColO = 192, kColQ = 448;
};
static_assert(TcCfg::kBytes <= 232448, "shared memory of one CTA");
static_assert(TcCfg::kColQ + 64 <= TcCfg::kTmemCols, "tensor-memory columns");
static_assert(TcCfg::kColO + 256 <= TcCfg::kColQ, "tensor-memory columns of O0 and O1");
static_assert(32 * (TcCfg::kSoftmaxWarps * TcCfg::kRegsSoftmax + TcCfg::kProducerWarps * TcCfg::kRegsProducer +
                    TcCfg::kMmaWarps * TcCfg::kRegsLaunch) <= TcCfg::kThreads * TcCfg::kRegsLaunch,
              "register split within the registers the CTA is launched with");

// Barrier indices, laid out from the ring sizes; every ring of n slots has
// one barrier per slot, so that a parity wait never meets a phase n uses
// ahead.
enum TcBar : int {
  kKFull = 0,
  kKEmpty = kKFull + TcCfg::kKStages,
  kVFull = kKEmpty + TcCfg::kKStages,
  kVEmpty = kVFull + TcCfg::kVStages,
  kSFull = kVEmpty + TcCfg::kVStages,
  kSFree = kSFull + 1,
  kPFull = kSFree + 1,        // [key half]
  kODone = kPFull + 2,        // [key half]
  kQFull = kODone + 2,
  kQTmem = kQFull + 1,
  kItemFull = kQTmem + 1,     // [item slot]
  kItemEmpty = kItemFull + 2,
  kDrain = kItemEmpty + 2,
  kXFull = kDrain + 1,        // [quarter][slot]: the two threads of a row published a value (epilogue)
  kNumTcBars = kXFull + 8
};
static_assert(kNumTcBars * 8 + 16 <= 512, "barrier region");

template <typename T>
__global__ void __launch_bounds__(TcCfg::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams P) {
  using C = TcCfg;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  volatile int* s_items = reinterpret_cast<volatile int*>(bar + kNumTcBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + kNumTcBars + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + kNumTcBars + 2);
  int* err = &P.ws->error_bits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G;
  if (tid == 0) {
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&bar[kKFull + i], C::kProducerWarps);
      mbar_init(&bar[kKEmpty + i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&bar[kVFull + i], C::kProducerWarps);
      mbar_init(&bar[kVEmpty + i], 1);
    }
    mbar_init(&bar[kSFull], 1);
    mbar_init(&bar[kSFree], C::kSoftmaxWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kPFull + i], C::kSoftmaxWarps / 2);   // per key half
      mbar_init(&bar[kODone + i], 1);
      mbar_init(&bar[kItemFull + i], 1);
      // helpers (3), MMA issuers (2), softmax (4)
      mbar_init(&bar[kItemEmpty + i], C::kProducerWarps - 1 + C::kMmaWarps + C::kSoftmaxWarps);
    }
    mbar_init(&bar[kQFull], 1);
    mbar_init(&bar[kQTmem], C::kSoftmaxWarps);
    mbar_init(&bar[kDrain], C::kMmaWarps);
    for (int i = 0; i < 8; ++i) mbar_init(&bar[kXFull + i], 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kProducerWarp0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == C::kMmaWarp) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int n_entries = *reinterpret_cast<volatile int32_t*>(&P.ws->n_entries);
  const int n_work = n_entries * P.hkv;

  if (warp >= C::kProducerWarp0 && warp < C::kMmaWarp) {
    // ------------------------------------------------------------ producers
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsProducer));
    // Warp 4 takes items from the atomic counter and publishes them; all
    // four producer warps read block ids 32 at a time (one coalesced load)
    // and each issues the copies of blocks p and p + 4 of every chunk
    // (lanes 0..3: block p / p + 4, dims 0-63 / 64-127), arming the stage
    // barrier for its own 8 KB.
    const int pw = warp - C::kProducerWarp0;
    const int64_t y_oob = P.num_blocks * P.hkv * kBlock;
    uint32_t it = 0, cc = 0;
    bool ok = true;
    auto wait = [&](int idx, uint32_t parity) {
      if (ok) ok = mbar_wait(&bar[idx], parity, abort_flag, err);
      ok = __all_sync(0xffffffffu, ok);
      return ok;
    };
    const int my_blk = pw + 4 * (lane & 1), my_hf = (lane >> 1) & 1;
    while (ok) {
      const int slot = it & 1;
      int wi = 0;
      if (pw == 0) {
        if (lane == 0) wi = atomicAdd(&P.ws->next_item, 1);
        wi = __shfl_sync(0xffffffffu, wi, 0);
        if (*abort_flag) wi = n_work;
        if (it >= 2 && !wait(kItemEmpty + slot, ((it >> 1) - 1) & 1)) break;
        if (lane == 0) {
          s_items[slot] = wi < n_work ? wi : -1;
          mbar_arrive(&bar[kItemFull + slot]);
        }
        if (wi >= n_work) break;
      } else {
        if (!wait(kItemFull + slot, (it >> 1) & 1)) break;
        wi = s_items[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kItemEmpty + slot]);
        if (wi < 0) break;
      }
      const int h = wi / n_entries;
      const int4 ent = P.entries[wi - h * n_entries];
      const int b = ent.x, tile = ent.y, nkb = ent.z;
      if (pw == 0) {
        // the softmax warps moved the previous item's Q into tensor memory
        const PieceView v = piece_view(P, b, false);
        if (it >= 1 && !wait(kQTmem, (it - 1) & 1)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar[kQFull], C::kQBytes);
          const int z = v.q0 + tile * P.tile_tokens;
          tma_load_3d(sQ, &tm_q, 0, h * G, z, &bar[kQFull]);
          tma_load_3d(sQ + C::kHalf, &tm_q, 64, h * G, z, &bar[kQFull]);
        }
      }
      const int32_t* trow = P.tables + static_cast<int64_t>(b) * P.max_blocks;
      const int nch = (nkb + C::kChunkBlocks - 1) / C::kChunkBlocks;
      // K runs one chunk ahead of V: S of chunk c needs K(c) one step before
      // O += P V needs V(c)
      int32_t ids = 0, yk = 0, yprev = 0;   // lanes 0..3: the row of this lane's block
      for (int c = 0; c <= nch && ok; ++c) {
        if (c < nch) {
          if ((c & 3) == 0) {   // ids of chunks c .. c + 3
            const int blk = c * C::kChunkBlocks + lane;
            int32_t id = blk < nkb ? trow[blk] : -1;   // past the tile's keys: zero fill
            if (blk < nkb && (id < 0 || id >= P.num_blocks)) {
              if (pw == 0) atomicOr(err, kErrBlockId);
              id = -1;
            }
            ids = id;
          }
          const int32_t id = __shfl_sync(0xffffffffu, ids, (c & 3) * C::kChunkBlocks + my_blk);
          yk = static_cast<int32_t>(id < 0 ? y_oob : (static_cast<int64_t>(id) * P.hkv + h) * kBlock);
          const uint32_t x = cc + c;
          const int ks = x % C::kKStages;
          if (x >= C::kKStages && !wait(kKEmpty + ks, ((x / C::kKStages) - 1) & 1)) break;
          if (lane == 0) mbar_arrive_expect_tx(&bar[kKFull + ks], C::kChunkBytes / C::kProducerWarps);
          __syncwarp();
          if (lane < 4)
            tma_load_2d(smem + C::kOffK + static_cast<size_t>(ks) * C::kChunkBytes + my_hf * C::kHalf + my_blk * 2048,
                        &tm_k, my_hf * 64, yk, &bar[kKFull + ks]);
        }
        if (c >= 1) {
          const uint32_t x = cc + c - 1;
          const int vs = x % C::kVStages;
          if (x >= C::kVStages && !wait(kVEmpty + vs, ((x / C::kVStages) - 1) & 1)) break;
          if (lane == 0) mbar_arrive_expect_tx(&bar[kVFull + vs], C::kChunkBytes / C::kProducerWarps);
          __syncwarp();
          if (lane < 4)
            tma_load_2d(smem + C::kOffV + static_cast<size_t>(vs) * C::kChunkBytes + my_hf * C::kHalf + my_blk * 2048,
                        &tm_v, my_hf * 64, yprev, &bar[kVFull + vs]);
        }
        yprev = yk;
      }
      cc += nch;
      ++it;
    }
  } else if (warp >= C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuers
    // lane 0 of warp 8 issues the S products, lane 0 of warp 9 the PV
    // products: issuing blocks a thread about as long as the product runs,
    // so with one issuer its waits and commits sat between the products;
    // with two, each one's bookkeeping overlaps the other's products
    if (lane == 0) {
      const bool pv_role = warp == C::kMmaWarp + 1;
      constexpr int kBf = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
      constexpr uint32_t id_s = umma_idesc_f16(kBf, 0, 128, 128);
      constexpr uint32_t id_o = umma_idesc_f16(kBf, 1, 128, 128);
      // shared-memory descriptors of the K and V rings; an MMA's operand is
      // the base plus a constant byte offset (>> 4 in the start-address field)
      const uint64_t dK0 = umma_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
      // V is MN-major (dims contiguous): one N = 128 product spans its two
      // 64-dim atoms, C::kHalf bytes apart (the leading byte offset); one
      // 128-wide product runs at the full rate where two 64-wide ones do not
      const uint64_t dV0 = umma_desc_sw128(smem_u32(smem + C::kOffV), C::kHalf, 1024);
      uint32_t it = 0, cc = 0;
      bool ok = true;
      auto wait = [&](int idx, uint32_t parity) {
        if (ok) ok = mbar_wait_sleep(&bar[idx], parity, abort_flag, err);
        return ok;
      };
      while (ok) {
        const int slot = it & 1;
        if (!wait(kItemFull + slot, (it >> 1) & 1)) break;
        const int wi = s_items[slot];
        mbar_arrive(&bar[kItemEmpty + slot]);
        if (wi < 0) break;
        const int h = wi / n_entries;
        const int nkb = P.entries[wi - h * n_entries].z;
        const int nch = (nkb + C::kChunkBlocks - 1) / C::kChunkBlocks;
        if (!pv_role) {
          // S of chunk x into the single S buffer once the softmax has read
          // S of chunk x - 1: A = Q from tensor memory (16 dims = 8 packed
          // columns per step), B = K (K-major, 32 bytes per step inside a
          // 128-byte row)
          if (!wait(kQTmem, it & 1)) break;   // this item's Q is in tensor memory
          for (int c = 0; c < nch && ok; ++c, ++cc) {
            const int kst = cc % C::kKStages;
            if (!wait(kKFull + kst, (cc / C::kKStages) & 1)) break;
            if (cc >= 1 && !wait(kSFree, (cc - 1) & 1)) break;
            tc_fence_after();
            const uint64_t dK = dK0 + (static_cast<uint64_t>(kst) * C::kChunkBytes >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_f16_ts(tbase + C::kColS, tbase + C::kColQ + 8 * ks,
                          dK + (((ks >> 2) * C::kHalf + (ks & 3) * 32) >> 4), id_s, ks > 0);
            umma_commit(&bar[kSFull]);
            umma_commit(&bar[kKEmpty + kst]);
          }
        } else {
          // O += P V of chunk x: A = P from tensor memory (16 keys = 8
          // packed columns per step), B = V (MN-major)
          for (int c = 0; c < nch && ok; ++c, ++cc) {
            const int vs = cc % C::kVStages;
            if (!wait(kVFull + vs, (cc / C::kVStages) & 1)) break;
            const uint64_t dV = dV0 + (static_cast<uint64_t>(vs) * C::kChunkBytes >> 4);
            // key half hk: O_hk += P[:, 64 hk ..] V[64 hk .., :] once that half's
            // softmax warps wrote their P
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
              if (!wait(kPFull + hk, cc & 1)) break;
              tc_fence_after();
#pragma unroll
              for (int ks = 4 * hk; ks < 4 * hk + 4; ++ks)
                umma_f16_ts(tbase + C::kColO + 128 * hk, tbase + C::kColP + 8 * ks, dV + ((ks * 2048) >> 4),
                            id_o, c > 0 || ks > 4 * hk);
              umma_commit(&bar[kODone + hk]);
            }
            if (!ok) break;
            umma_commit(&bar[kVEmpty + vs]);
          }
        }
        ++it;
      }
      // every product issued has completed before tensor memory is freed
      umma_commit(&bar[kDrain]);
      const unsigned long long t0 = global_timer_ns();
      while (!mbar_try_wait(&bar[kDrain], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // two threads per query row: warp w (w < 4) takes keys 0-63 of every
    // chunk, warp w + 4 keys 64-127, in the same tensor-memory lane quarter.
    // Each keeps its own running maximum and sum and its own O (O0, O1), so
    // the two never wait for each other inside an item; at its end they
    // exchange (maximum, sum) once and each writes 64 of the 128 output
    // dims of the combined result.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsSoftmax));
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(32 * quarter) << 16);
    const uint32_t o_mine = lane_addr + C::kColO + 128 * half;
    uint32_t it = 0, cc = 0, xk = 0;
    bool ok = true;
    auto wait = [&](int idx, uint32_t parity) {
      if (ok) ok = mbar_wait(&bar[idx], parity, abort_flag, err);
      ok = __all_sync(0xffffffffu, ok);
      return ok;
    };
    // one value with the row's other thread, through two tensor-memory
    // columns of the S buffer (free at an epilogue: the next item's first S
    // waits for its Q, which these warps write after the epilogue); a slot
    // is rewritten two exchanges later, after the partner passed the
    // exchange between
    auto exchange = [&](float mine) -> float {
      const uint32_t xs = xk & 1;
      tmem_st1(lane_addr + C::kColS + 2 * xs + half, mine);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kXFull + 2 * quarter + xs]);
      wait(kXFull + 2 * quarter + xs, (xk >> 1) & 1);
      tc_fence_after();
      const float other = tmem_ld1(lane_addr + C::kColS + 2 * xs + (half ^ 1));
      ++xk;
      return other;
    };
    while (ok) {
      const int slot = it & 1;
      if (!wait(kItemFull + slot, (it >> 1) & 1)) break;
      const int wi = s_items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kItemEmpty + slot]);
      if (wi < 0) break;
      const int h = wi / n_entries;
      const int4 ent = P.entries[wi - h * n_entries];
      const int b = ent.x, tile = ent.y, nkb = ent.z;
      const PieceView v = piece_view(P, b, false);
      const int nch = (nkb + C::kChunkBlocks - 1) / C::kChunkBlocks;
      const int tok = tile * P.tile_tokens + row / G;
      const int pos = v.L - v.n + tok;
      const bool valid = tok < v.n && pos >= 0;
      const int lim = valid ? pos : -1;
      // this thread's 64 dims of the Q row -> tensor memory (the previous
      // item's products, which read the old Q, completed before its
      // epilogue).  The TMA box put row `row` at row * 128 bytes of each
      // 64-dim half, its 16-byte pieces permuted by the 128-byte swizzle
      // (piece j at j ^ (row & 7)).
      if (!wait(kQFull, it & 1)) break;
      {
        uint32_t qw[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 u = *reinterpret_cast<const uint4*>(sQ + half * C::kHalf + row * 128 + ((j ^ (row & 7)) << 4));
          qw[4 * j] = u.x;
          qw[4 * j + 1] = u.y;
          qw[4 * j + 2] = u.z;
          qw[4 * j + 3] = u.w;
        }
        tmem_st32u(lane_addr + C::kColQ + 32 * half, qw);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kQTmem]);
      float m_ref = -INFINITY, l = 0.f;   // this key half's reference maximum and sum
      for (int c = 0; c < nch; ++c, ++cc) {
        if (!wait(kSFull, cc & 1)) break;
        tc_fence_after();
        const int kc = c * 128, k0 = kc + 64 * half;
        float t[64];
        tmem_ld64(lane_addr + C::kColS + 64 * half, t);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kSFree]);
        if (!__all_sync(0xffffffffu, k0 + 63 <= lim)) {   // causal mask / tail: -inf
#pragma unroll
          for (int i = 0; i < 64; ++i) t[i] = k0 + i <= lim ? t[i] : -INFINITY;
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // 4 chains for ILP
#pragma unroll
        for (int i = 0; i < 64; ++i) m4[i & 3] = fmaxf(m4[i & 3], t[i]);
        // the scale is positive, so it commutes with the maximum
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * P.scale_log2;
        const bool need = mx > m_ref + 8.f;
        const float new_ref = need ? mx : m_ref;
        const float mu = new_ref == -INFINITY ? 0.f : new_ref;
        const float alpha = need ? exp2f(m_ref - new_ref) : 1.f;
        // p = 2^(s * scale - mu) as 16-bit, two per column, into this half's
        // 32 columns of P, once the previous chunk's product over this half
        // has read them; row sum in fp32 (pairs on the packed two-lane FMA/add)
        const float2 sc2 = make_float2(P.scale_log2, P.scale_log2), nm2 = make_float2(-mu, -mu);
        float2 r2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 x = fma2(make_float2(t[2 * i], t[2 * i + 1]), sc2, nm2);
          const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          r2[i & 3] = add2(r2[i & 3], p);
          pk[i] = pack2<T>(p.x, p.y);
        }
        if (cc >= 1 && !wait(kODone + half, (cc - 1) & 1)) break;
        tc_fence_after();
        tmem_st32u(lane_addr + C::kColP + 32 * half, pk);
        r2[0] = add2(add2(r2[0], r2[1]), add2(r2[2], r2[3]));
        l = l * alpha + (r2[0].x + r2[0].y);
        if (c > 0 && __any_sync(0xffffffffu, need)) {
          // this half's O holds the previous chunk's product (waited above)
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float o32[32];
            tmem_ld32(o_mine + cb * 32, o32);
#pragma unroll
            for (int i = 0; i < 32; ++i) o32[i] *= alpha;
            tmem_st32(o_mine + cb * 32, o32);
          }
        }
        // V rows past the sequence end (the last block's tail) may hold
        // anything, NaN included: zero them so that 0 * NaN never enters O
        if (kc + 128 > v.L) {
          // the chunk's V copies have landed before their rows are overwritten
          const int vs = cc % C::kVStages;
          if (!wait(kVFull + vs, (cc / C::kVStages) & 1)) break;
          // this half's product reads only keys 64 half .. 64 half + 63 of the
          // chunk, and waits only for this half's warps: they zero those rows
          const int z0 = max(max(v.L, kc) - kc, 64 * half);
          const int z1 = min(min(kc + 128, nkb * kBlock) - kc, 64 * half + 64);
          uint8_t* sV = smem + C::kOffV + static_cast<size_t>(vs) * C::kChunkBytes;
          for (int i = row; i < (z1 - z0) * 16; i += 128) {   // 16 x 16 B per key row
            const int key = z0 + (i >> 4), part = i & 15;
            *reinterpret_cast<uint4*>(sV + (part >> 3) * C::kHalf + key * 128 + (part & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();   // the zeros before the tensor cores read V
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kPFull + half]);
        m_ref = new_ref;
      }
      if (!ok) break;
      // epilogue: combine the halves, out = (O0 2^(m0 - m) + O1 2^(m1 - m)) /
      // (l0 2^(m0 - m) + l1 2^(m1 - m)) with m the larger maximum; each thread
      // writes 64 of the 128 dims, one rounding to T
      const float m_other = exchange(m_ref);
      const float l_other = exchange(l);
      if (!ok) break;
      if (nch > 0) {
        if (!wait(kODone + 0, (cc - 1) & 1)) break;
        if (!wait(kODone + 1, (cc - 1) & 1)) break;
      }
      tc_fence_after();
      {
        const float m0 = half == 0 ? m_ref : m_other, m1 = half == 0 ? m_other : m_ref;
        const float l0 = half == 0 ? l : l_other, l1 = half == 0 ? l_other : l;
        const float mm = fmaxf(m0, m1);
        const float w0 = mm == -INFINITY ? 0.f : exp2f(m0 - mm);
        const float w1 = mm == -INFINITY ? 0.f : exp2f(m1 - mm);
        const float lsum = l0 * w0 + l1 * w1;
        const float inv = (valid && lsum > 0.f) ? 1.0f / lsum : 0.f;
        const float a0 = w0 * inv, a1 = w1 * inv;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(P.out) +
                                              ((static_cast<int64_t>(v.q0) + tok) * P.hq + h * G + row % G) * D +
                                              64 * half);
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
          float x32[32], y32[32];
          if (nch > 0) {   // uniform over the warp: every lane takes part in the loads
            tmem_ld32(lane_addr + C::kColO + 64 * half + cb * 32, x32);
            tmem_ld32(lane_addr + C::kColO + 128 + 64 * half + cb * 32, y32);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) x32[i] = y32[i] = 0.f;
          }
          if (tok < v.n) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              float o8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) o8[e] = fmaf(x32[8 * q4 + e], a0, y32[8 * q4 + e] * a1);
              dst[cb * 4 + q4] = make_uint4(pack2<T>(o8[0], o8[1]), pack2<T>(o8[2], o8[3]),
                                            pack2<T>(o8[4], o8[5]), pack2<T>(o8[6], o8[7]));
            }
          }
        }
      }
      tc_fence_before();
      ++it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // copies still in flight land before the CTA leaves: a copy takes
    // microseconds, so every thread waits 200 us of global time
    const unsigned long long t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

namespace {

constexpr int kPrefillWarps = 8;
constexpr int kPrefillStages = 16;

template <typename T, int D>
bool launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& P,
                    int64_t max_work, cudaStream_t s, std::string* why) {
  using Cfg = PrefillCfg<D, kPrefillWarps, kPrefillStages>;
  auto kern = prefill_kernel<T, D, kPrefillWarps, kPrefillStages>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::kBytes));
  if (e != cudaSuccess) {
    *why = std::string("cudaFuncSetAttribute (prefill): ") + cudaGetErrorString(e);
    return false;
  }
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::kThreads, Cfg::kBytes);
  if (per_sm < 1) per_sm = 1;
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid > max_work) grid = max_work;
  if (grid < 1) grid = 1;
  kern<<<static_cast<unsigned>(grid), Cfg::kThreads, Cfg::kBytes, s>>>(tk, tv, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("prefill launch: ") + cudaGetErrorString(e);
    return false;
  }
  return true;
}

int64_t max_entries(int64_t num_seqs, int64_t num_q_tokens, int64_t tile_tokens) {
  return num_q_tokens / tile_tokens + num_seqs + 1;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// q [Tq][hq][D] as a 3-D tensor (dims, heads, tokens); one box = the G heads
// of a KV head for 128 / G tokens and 64 dims: 128 rows of 128 bytes in the
// order (token, head), 128-byte swizzle.
bool encode_q_map(CUtensorMap* m, const void* q, int64_t Tq, int hq, int G, int D,
                  std::string* why) {
  EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder(why));
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(hq),
                        static_cast<cuuint64_t>(Tq)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(hq) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled (q) failed with CUresult " + std::to_string(static_cast<int>(r));
    return false;
  }
  return true;
}

template <typename T>
bool launch_prefill_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const PrefillParams& P, int64_t max_work, cudaStream_t s, std::string* why) {
  auto kern = prefill_tc_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(TcCfg::kBytes));
  if (e != cudaSuccess) {
    *why = std::string("cudaFuncSetAttribute (prefill tc): ") + cudaGetErrorString(e);
    return false;
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one CTA per SM: its shared memory rules out a second one, and each CTA
  // holds all 512 tensor-memory columns
  int64_t grid = sms;
  if (grid > max_work) grid = max_work;
  if (grid < 1) grid = 1;
  kern<<<static_cast<unsigned>(grid), TcCfg::kThreads, TcCfg::kBytes, s>>>(tq, tk, tv, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("prefill tc launch: ") + cudaGetErrorString(e);
    return false;
  }
  return true;
}

}  // namespace

size_t prefill_workspace_bytes(int64_t num_seqs, int64_t num_q_tokens, int64_t num_q_heads,
                               int64_t num_kv_heads) {
  const int64_t G = num_q_heads / num_kv_heads;
  const int64_t tile_tokens = 16 * kPrefillWarps / G;
  return sizeof(PrefillHeader) + align_up(sizeof(int4) * max_entries(num_seqs, num_q_tokens, tile_tokens), 256);
}

int prefill_launch(const PrefillArgs& a, std::string* why) {
  PrefillParams P;
  P.q = a.q;
  P.out = a.out;
  P.tables = a.block_tables;
  P.seq_lens = a.seq_lens;
  P.q_off = a.q_offsets;
  P.ws = static_cast<PrefillHeader*>(a.workspace);
  P.entries = reinterpret_cast<int4*>(static_cast<uint8_t*>(a.workspace) + sizeof(PrefillHeader));
  P.num_blocks = a.num_blocks;
  P.max_blocks = a.max_blocks_per_seq;
  P.num_seqs = a.num_seqs;
  P.num_q_tokens = a.num_q_tokens;
  P.max_seq_len = a.max_seq_len;
  P.hq = a.num_q_heads;
  P.hkv = a.num_kv_heads;
  P.G = a.num_q_heads / a.num_kv_heads;
  P.tile_tokens = 16 * kPrefillWarps / P.G;
  P.max_entries = static_cast<int>(max_entries(a.num_seqs, a.num_q_tokens, P.tile_tokens));
  P.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  CUtensorMap tk, tv;
  if (!encode_cache_map(&tk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, why) ||
      !encode_cache_map(&tv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, why))
    return 5;
  cudaStream_t s = static_cast<cudaStream_t>(a.stream);
  prefill_prep_kernel<<<1, 1024, 0, s>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = std::string("prefill prep launch: ") + cudaGetErrorString(e);
    return 5;
  }
  const int64_t max_work = max_entries(a.num_seqs, a.num_q_tokens, P.tile_tokens) * a.num_kv_heads;
  // variant 0: tcgen05 at head_dim 128, else mma.sync; 2: mma.sync; 3: tcgen05
  const bool tc = a.variant == 3 || (a.variant == 0 && a.head_dim == 128);
  CUtensorMap tq;
  if (tc && !encode_q_map(&tq, a.q, a.num_q_tokens, a.num_q_heads, P.G, a.head_dim, why)) return 5;
  if (a.ev_before) cudaEventRecord(static_cast<cudaEvent_t>(a.ev_before), s);
  bool ok;
  if (tc)
    ok = a.dtype == 1 ? launch_prefill_tc<__nv_bfloat16>(tq, tk, tv, P, max_work, s, why)
                      : launch_prefill_tc<__half>(tq, tk, tv, P, max_work, s, why);
  else
    ok = a.dtype == 1
             ? (a.head_dim == 128 ? launch_prefill<__nv_bfloat16, 128>(tk, tv, P, max_work, s, why)
                                  : launch_prefill<__nv_bfloat16, 64>(tk, tv, P, max_work, s, why))
             : (a.head_dim == 128 ? launch_prefill<__half, 128>(tk, tv, P, max_work, s, why)
                                  : launch_prefill<__half, 64>(tk, tv, P, max_work, s, why));
  if (!ok) return 5;
  if (a.ev_after) cudaEventRecord(static_cast<cudaEvent_t>(a.ev_after), s);
  return 0;
}

}  // namespace pa
