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
//   2. prefill (persistent, one CTA per SM)
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

__global__ void __launch_bounds__(1024) prefill_prep_kernel(PrefillParams P) {
  __shared__ int sw[32];
  __shared__ int s_hist[kPrefillBins];
  __shared__ int s_shift;
  const int tid = threadIdx.x;
  if (tid == 0) {
    P.ws->error_bits = 0;
    int sh = 0;
    while ((P.max_blocks >> sh) >= kPrefillBins) ++sh;
    s_shift = sh;
  }
  for (int i = tid; i < kPrefillBins; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int shift = s_shift;
  for (int b = tid; b < P.num_seqs; b += blockDim.x) {
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
  for (int b = tid; b < P.num_seqs; b += blockDim.x) {
    const PieceView v = piece_view(P, b, false);
    const int nt = (v.n + P.tile_tokens - 1) / P.tile_tokens;
    for (int t = 0; t < nt; ++t) {
      const int kb = tile_key_blocks(v, t, P.tile_tokens);
      const int slot = atomicAdd(&s_hist[min(kb >> shift, kPrefillBins - 1)], 1);
      // overlapping pieces (offsets out of order, already flagged) cannot
      // overflow the list: records past its capacity are dropped
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
  if (a.ev_before) cudaEventRecord(static_cast<cudaEvent_t>(a.ev_before), s);
  bool ok = a.dtype == 1
                ? (a.head_dim == 128 ? launch_prefill<__nv_bfloat16, 128>(tk, tv, P, max_work, s, why)
                                     : launch_prefill<__nv_bfloat16, 64>(tk, tv, P, max_work, s, why))
                : (a.head_dim == 128 ? launch_prefill<__half, 128>(tk, tv, P, max_work, s, why)
                                     : launch_prefill<__half, 64>(tk, tv, P, max_work, s, why));
  if (!ok) return 5;
  if (a.ev_after) cudaEventRecord(static_cast<cudaEvent_t>(a.ev_after), s);
  return 0;
}

}  // namespace pa
