// ep_layout.cu -- layout of the routing: per-expert / per-rank histograms,
// aligned exclusive prefix sums, deterministic destination slots and
// recv_src_metadata (EPHandle fields of "DeepEP overall architecture
// analysis"; the counting role of its "notify warps" in the Dispatch data flow
// figure).
//
// Rows of one expert are ordered by the flat index t*K+k, so the slot of an
// entry is psum_expert[e] + (number of earlier entries routed to e): a stable
// counting sort.  Three launches, the last two with programmatic dependent
// launch so that each is scheduled while its predecessor drains:
//
//   count  one CTA per chunk of kLayoutTPC tokens.  The chunk's ids are staged
//          in shared memory with one coalesced load and every pass runs from
//          there.  Per-warp histograms over contiguous runs of entries use
//          shared-memory atomics; an exclusive scan across the warps gives each
//          warp its start per expert, and a pass over 32-entry batches that
//          combines lanes carrying the same expert with __match_any_sync gives
//          each entry its stable rank in the chunk.  Tokens per rank: each
//          entry ORs its rank bit into its token's mask, then warp ballots
//          count the set bits.  The chunk's column totals (E experts + W ranks)
//          go to a column-major [E+W][C] table.
//   spine  a warp per column scans the C chunk totals (chunk offsets and
//          column totals).
//   slots  every CTA rebuilds the aligned exclusive prefix over the experts
//          from the column totals (E values, cheaper than another launch) and
//          CTA 0 writes the counts, the prefix sums and the number of receive
//          rows.  One CTA per chunk turns ranks into slots (dst_slot), sorts the
//          chunk's entries by (expert, rank) in shared memory and writes their
//          metadata rows through a flat index: the rows of one expert from one
//          chunk are contiguous, so consecutive threads write consecutive words.
//          Every CTA also writes -1 into its share of the rows that receive
//          nothing (expert padding and [R, capacity)).
//
// Non-expand layout (EPHandle do_expand = false): one row per (token,
// destination rank).  count and spine are shared (the rank columns of the
// table already count each chunk's tokens per rank); a second slots kernel
// places rank r's tokens in ascending order from psum_rank[r] on, using warp
// ballots over the tokens' rank masks for the position inside the chunk.
// No kernel waits on another CTA.
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

constexpr int kCountThreads = kLayoutCountWarps * 32;
constexpr int kSpineWarps = 8;
constexpr int kSlotThreads = 256;

__device__ __forceinline__ int expert_of(int64_t v, int E) {
  return (v >= 0 && v < E) ? static_cast<int>(v) : -1;
}

// Rank of expert e, e / Epr, as a multiply-high with the magic number of
// RankMagic (0 when Epr == 1).
__device__ __forceinline__ int rank_of(int e, uint32_t magic) {
  return magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(e), magic)) : e;
}

// Let the next kernel of the stream (launched with programmatic stream
// serialisation) be scheduled; it waits for this grid's completion itself.
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the preceding grid of the stream has completed and its writes are visible.
__device__ __forceinline__ void wait_for_preceding_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Block-wide exclusive scan of align(v[e], A) for e in [0, n) into out[0..n]
// (out[n] = total).  warp_tot needs 33 words.  All threads must call it.
__device__ void block_exclusive_scan(const int32_t* v, int n, int A, int32_t* out,
                                     int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  const int V = (n + nthr - 1) / nthr;
  const int beg = min(n, tid * V), end = min(n, beg + V);
  int sum = 0;
  for (int e = beg; e < end; ++e) sum += (v[e] + A - 1) / A * A;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nwarp ? warp_tot[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nwarp) warp_tot[lane] = s - w;  // exclusive warp offsets
    if (lane == nwarp - 1) warp_tot[32] = s;  // grand total
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - sum;
  for (int e = beg; e < end; ++e) {
    out[e] = run;
    run += (v[e] + A - 1) / A * A;
  }
  if (tid == 0) out[n] = warp_tot[32];
  __syncthreads();
}

// ---------------------------------------------------------------- count

template <int KC>
__global__ void __launch_bounds__(kCountThreads) ep_layout_count_kernel(LayoutParams p) {
  constexpr int NW = kLayoutCountWarps;
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, W = p.world_size;
  const int EW = E + W;
  const int C = p.num_chunks;
  extern __shared__ int32_t sm[];
  int32_t* whist = sm;                                     // [NW][EW]
  int32_t* ids = whist + NW * EW;                          // [TPC*K] expert ids, -1 = skip

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int t0 = c * kLayoutTPC;
  const int ntok = min(p.num_tokens, t0 + kLayoutTPC) - t0;
  const int nent = ntok * K;
  const int64_t* topk = p.topk_idx + static_cast<int64_t>(t0) * K;

  allow_dependents();
  bool bad = false;
  int32_t* clone = p.topk_i32 ? p.topk_i32 + static_cast<int64_t>(t0) * K : nullptr;
  for (int i = tid; i < nent; i += kCountThreads) {
    const int64_t v = topk[i];
    const int e = expert_of(v, E);
    bad |= (e < 0 && v != -1);
    ids[i] = e;
    if (clone) clone[i] = e;
  }
  for (int i = tid; i < NW * EW; i += kCountThreads) whist[i] = 0;
  __syncthreads();

  // per-warp histogram over a contiguous run of entries (whole 32-entry batches)
  const int per_warp = (((nent + NW - 1) / NW) + 31) & ~31;
  const int wbeg = warp * per_warp;
  const int wend = min(nent, wbeg + per_warp);
  int32_t* wh = whist + warp * EW;
  for (int i = wbeg + lane; i < wend; i += 32) {
    const int e = ids[i];
    if (e >= 0) atomicAdd(&wh[e], 1);
  }
  // tokens per rank: each thread builds its token's rank mask in registers
  // (no atomics: all K entries of a token would hit one word), warp ballots count
  for (int tl0 = warp * 32; tl0 < ntok; tl0 += kCountThreads) {
    const int tl = tl0 + lane;
    unsigned long long mask = 0ull;
    if (tl < ntok)
      for (int k = 0; k < K; ++k) {
        const int e = ids[tl * K + k];
        if (e >= 0) mask |= 1ull << rank_of(e, p.epr_magic);
      }
    for (int r = 0; r < W; ++r) {
      const int n = __popc(__ballot_sync(0xffffffffu, (mask >> r) & 1ull));
      if (lane == 0 && n) atomicAdd(&whist[E + r], n);
    }
  }
  __syncthreads();

  // exclusive scan across warps per column; the column total is the chunk's count
  for (int j = tid; j < EW; j += kCountThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int v = whist[w * EW + j];
      whist[w * EW + j] = run;
      run += v;
    }
    p.chunk_hist[static_cast<int64_t>(j) * C + c] = run;
  }
  __syncthreads();

  // stable rank of each entry within the chunk (the expand layout's slots)
  int32_t* local = p.dst_slot + static_cast<int64_t>(t0) * K;
  for (int i = wbeg; i < wend && !p.no_expand; i += 32) {
    const int idx = i + lane;
    const int e = idx < wend ? ids[idx] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int base = e >= 0 ? wh[e] : 0;
    const int rank = base + __popc(peers & lanemask_lt());
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wh[e] = base + __popc(peers);
    __syncwarp();
    if (idx < wend) local[idx] = e >= 0 ? rank : -1;
  }
  if (bad) atomicOr(p.err, kErrBadExpert);
}

// ---------------------------------------------------------------- spine

// A warp per column j of the [E+W][C] table: exclusive scan over the C chunks
// (each lane a contiguous run of chunks, kept in registers when short).
__global__ void __launch_bounds__(kSpineWarps * 32) ep_layout_spine_kernel(LayoutParams p) {
  const int EW = p.num_experts + p.world_size;
  const int C = p.num_chunks;
  const int j = blockIdx.x * kSpineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  allow_dependents();
  wait_for_preceding_grid();
  if (j >= EW) return;
  const int32_t* in = p.chunk_hist + static_cast<int64_t>(j) * C;
  int32_t* out = p.chunk_off + static_cast<int64_t>(j) * C;
  constexpr int kRegRun = 8;
  const int V = (C + 31) / 32;
  const int cbeg = min(C, lane * V), cend = min(C, cbeg + V);
  int sum = 0;
  int reg[kRegRun];
  if (V <= kRegRun) {
#pragma unroll
    for (int u = 0; u < kRegRun; ++u) {
      reg[u] = cbeg + u < cend ? in[cbeg + u] : 0;
      sum += reg[u];
    }
  } else {
    for (int c = cbeg; c < cend; ++c) sum += in[c];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;
  if (V <= kRegRun) {
#pragma unroll
    for (int u = 0; u < kRegRun; ++u)
      if (cbeg + u < cend) {
        out[cbeg + u] = run;
        run += reg[u];
      }
  } else {
    for (int c = cbeg; c < cend; ++c) {
      const int v = in[c];
      out[c] = run;
      run += v;
    }
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) p.col_total[j] = total;
}

// ---------------------------------------------------------------- slots

template <int KC>
__global__ void __launch_bounds__(kSlotThreads) ep_layout_slots_kernel(LayoutParams p) {
  constexpr int KM = KC ? KC : kMaxTopk;
  const int K = KC ? KC : p.topk;
  const int KW = K + 2;  // metadata row width
  const int E = p.num_experts, C = p.num_chunks;
  const int T = p.max_tok_per_rank;
  extern __shared__ int32_t sm[];
  int32_t* psum_s = sm;                   // [E+1]
  int32_t* cnt_s = psum_s + E + 1;        // [E]
  int32_t* cl = cnt_s + E;                // [E]   this chunk's count per expert
  int32_t* co = cl + E;                   // [E]   chunk_off of this chunk per expert
  int32_t* cx = co + E;                   // [E+1] exclusive scan of cl over experts
  int32_t* warp_tot = cx + E + 1;         // [33]
  int32_t* slots_s = warp_tot + 33;       // [TPC*K]
  int32_t* sorted = slots_s + kLayoutTPC * K;  // [TPC*K] entries ordered by (expert, rank)
  int32_t* src = sorted + kLayoutTPC * K;      // [2*TPC] {t / T, t mod T} per token

  const int c = blockIdx.x;
  const bool has_tokens = c < C;
  wait_for_preceding_grid();
  for (int e = threadIdx.x; e < E; e += kSlotThreads) {
    cnt_s[e] = p.col_total[e];
    if (has_tokens) {
      cl[e] = p.chunk_hist[static_cast<int64_t>(e) * C + c];
      co[e] = p.chunk_off[static_cast<int64_t>(e) * C + c];
    }
  }
  __syncthreads();
  // the aligned exclusive prefix over experts (every CTA; E values)
  block_exclusive_scan(cnt_s, E, p.alignment, psum_s, warp_tot);
  if (c == 0) {
    const int W = p.world_size;
    for (int e = threadIdx.x; e <= E; e += kSlotThreads) {
      p.psum_expert[e] = psum_s[e];
      if (e < E) p.cnt[e] = cnt_s[e];
    }
    for (int r = threadIdx.x; r <= W; r += kSlotThreads) {
      p.psum_rank[r] = psum_s[r * p.num_expert_per_rank];
      if (r < W) p.tok_per_rank[r] = p.col_total[E + r];
    }
    if (threadIdx.x == 0) *p.num_recv = psum_s[E];
  }
  if (has_tokens) block_exclusive_scan(cl, E, 1, cx, warp_tot);  // uniform per CTA

  const int t0 = c * kLayoutTPC;
  const int ntok = has_tokens ? min(p.num_tokens, t0 + kLayoutTPC) - t0 : 0;
  if (threadIdx.x < ntok) {
    const int tl = threadIdx.x, t = t0 + tl;
    const int64_t* row = p.topk_idx + static_cast<int64_t>(t) * K;
    int32_t* ds = p.dst_slot + static_cast<int64_t>(t) * K;
    int32_t slot[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k < K) {
        const int e = expert_of(row[k], E);
        const int loc = ds[k];
        slot[k] = e >= 0 ? psum_s[e] + co[e] + loc : -1;
        if (e >= 0) sorted[cx[e] + loc] = tl * K + k;
      }
    }
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (k < K) {
        ds[k] = slot[k];
        slots_s[tl * K + k] = slot[k];
      }
    const int r = t / T;
    src[2 * tl] = r;
    src[2 * tl + 1] = t - r * T;
  }
  __syncthreads();

  // metadata rows of this chunk, in (expert, rank) order: flat words f of the
  // concatenated rows; rows of one expert are contiguous in memory.
  if (has_tokens) {
    const int nvalid = cx[E];
    if ((KW & 1) == 0) {
      // even row width: word pairs (8-byte stores; rows start 8-byte aligned)
      const int hw = KW / 2;
      for (int f = threadIdx.x; f < nvalid * hw; f += kSlotThreads) {
        const int q = f / hw, c2 = f - q * hw;
        const int entry = sorted[q];
        const int tl = entry / K;
        const int2 v = c2 == 0 ? make_int2(src[2 * tl], src[2 * tl + 1])
                               : make_int2(slots_s[tl * K + 2 * c2 - 2], slots_s[tl * K + 2 * c2 - 1]);
        reinterpret_cast<int2*>(p.meta + static_cast<int64_t>(slots_s[entry]) * KW)[c2] = v;
      }
    } else {
      for (int f = threadIdx.x; f < nvalid * KW; f += kSlotThreads) {
        const int q = f / KW, col = f - q * KW;
        const int entry = sorted[q];
        const int tl = entry / K;
        const int v = col < 2 ? src[2 * tl + col] : slots_s[tl * K + col - 2];
        p.meta[static_cast<int64_t>(slots_s[entry]) * KW + col] = v;
      }
    }
  }

  // rows that receive nothing: the padding of experts e = c, c + grid, ... and
  // this CTA's slice of [R, capacity)
  for (int e = c; e < E; e += gridDim.x) {
    const int64_t beg = static_cast<int64_t>(psum_s[e] + cnt_s[e]) * KW;
    const int64_t end = static_cast<int64_t>(psum_s[e + 1]) * KW;
    for (int64_t f = beg + threadIdx.x; f < end; f += kSlotThreads) p.meta[f] = -1;
  }
  const int64_t tail_beg = static_cast<int64_t>(psum_s[E]) * KW;
  const int64_t tail_words = p.rcap * KW - tail_beg;
  const int64_t per = (tail_words + gridDim.x - 1) / gridDim.x;
  const int64_t sbeg = tail_beg + per * c;
  const int64_t send = sbeg + per < p.rcap * KW ? sbeg + per : p.rcap * KW;
  for (int64_t f = sbeg + threadIdx.x; f < send; f += kSlotThreads) p.meta[f] = -1;
}

// ---------------------------------------------------------------- slots, non-expand

constexpr int kTokenWarps = kLayoutTPC / 32;

// Exclusive scan of v[r] over r < n <= 64 by one warp (two values per lane)
// into out[0..n] (out[n] = total).
__device__ __forceinline__ void warp_scan64(const int32_t* v, int n, int32_t* out) {
  const int lane = threadIdx.x & 31;
  const int r0 = 2 * lane, r1 = r0 + 1;
  const int v0 = r0 < n ? v[r0] : 0, v1 = r1 < n ? v[r1] : 0;
  int incl = v0 + v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int ex = incl - v0 - v1;
  if (r0 < n) out[r0] = ex;
  if (r1 < n) out[r1] = ex + v0;
  if (lane == 31) out[n] = incl;
}

// Rank r's rows are its tokens in ascending order: the row of (t, r) is
// psum_rank[r] + chunk_off[r][chunk] + (tokens of the chunk before t that reach
// r).  Threads 0..127 own the chunk's tokens; each rank's positions come from
// a ballot per token warp and an exclusive scan over the four warps.
template <int KC>
__global__ void __launch_bounds__(kSlotThreads) ep_layout_slots_ne_kernel(LayoutParams p) {
  constexpr int KM = KC ? KC : kMaxTopk;
  constexpr int TW = kTokenWarps;
  const int K = KC ? KC : p.topk;
  const int KW = K + 2;
  const int E = p.num_experts, W = p.world_size, C = p.num_chunks;
  const int T = p.max_tok_per_rank;
  const int RM = K < W ? K : W;            // rows per token at most
  extern __shared__ int32_t sm[];
  int2* sorted = reinterpret_cast<int2*>(sm);          // [TPC*RM] (token, row) by (rank, token)
  int32_t* prank = sm + 2 * kLayoutTPC * RM;          // [W+1] exclusive prefix of tokens per rank
  int32_t* tpr = prank + W + 1;                        // [W]   tokens per rank
  int32_t* rcl = tpr + W;                              // [W]   this chunk's tokens per rank
  int32_t* rbase = rcl + W;                            // [W]   first row of this chunk per rank
  int32_t* rcx = rbase + W;                            // [W+1] exclusive scan of rcl over ranks
  int32_t* woff = rcx + W + 1;                         // [TW][W] per-warp counts, then offsets
  int32_t* warp_tot = woff + TW * W;                   // [33]
  int32_t* dslot = warp_tot + 33;                      // [TPC*K] row of each (t, k)
  int32_t* src = dslot + kLayoutTPC * K;               // [2*TPC] {t / T, t mod T}
  int32_t* cnt_s = src + 2 * kLayoutTPC;               // [E]   (CTA 0)
  int32_t* psum_s = cnt_s + E;                         // [E+1] (CTA 0)

  const int c = blockIdx.x;
  const bool has_tokens = c < C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  wait_for_preceding_grid();
  for (int r = tid; r < W; r += kSlotThreads) {
    tpr[r] = p.col_total[E + r];
    if (has_tokens) {
      rcl[r] = p.chunk_hist[static_cast<int64_t>(E + r) * C + c];
      rbase[r] = p.chunk_off[static_cast<int64_t>(E + r) * C + c];
    }
  }
  __syncthreads();
  if (warp == 0) warp_scan64(tpr, W, prank);
  if (warp == 1 && has_tokens) warp_scan64(rcl, W, rcx);
  __syncthreads();
  for (int r = tid; r < W && has_tokens; r += kSlotThreads) rbase[r] += prank[r];

  if (c == 0) {  // the counts and prefix sums (the expert ones as in the expand layout)
    for (int e = tid; e < E; e += kSlotThreads) cnt_s[e] = p.col_total[e];
    __syncthreads();
    block_exclusive_scan(cnt_s, E, p.alignment, psum_s, warp_tot);
    for (int e = tid; e <= E; e += kSlotThreads) {
      p.psum_expert[e] = psum_s[e];
      if (e < E) p.cnt[e] = cnt_s[e];
    }
    for (int r = tid; r <= W; r += kSlotThreads) {
      p.psum_rank[r] = prank[r];
      if (r < W) p.tok_per_rank[r] = tpr[r];
    }
    if (tid == 0) *p.num_recv = prank[W];
  }

  const int t0 = c * kLayoutTPC;
  const int ntok = has_tokens ? min(p.num_tokens, t0 + kLayoutTPC) - t0 : 0;
  const int tl = tid;                      // token of this thread (token warps only)
  unsigned long long mask = 0ull;
  int rk[KM];                              // rank of each entry, -1 when skipped
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    rk[k] = -1;
    if (k < K && warp < TW && tl < ntok) {
      const int e = expert_of(p.topk_idx[static_cast<int64_t>(t0 + tl) * K + k], E);
      if (e >= 0) {
        rk[k] = rank_of(e, p.epr_magic);
        mask |= 1ull << rk[k];
      }
    }
  }
  if (warp < TW)
    for (int r = 0; r < W; ++r) {
      const unsigned b = __ballot_sync(0xffffffffu, (mask >> r) & 1ull);
      if (lane == 0) woff[warp * W + r] = __popc(b);
    }
  __syncthreads();
  for (int r = tid; r < W; r += kSlotThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < TW; ++w) {
      const int v = woff[w * W + r];
      woff[w * W + r] = run;
      run += v;
    }
  }
  __syncthreads();

  if (warp < TW && has_tokens) {
    int32_t* ss = p.send_slot + static_cast<int64_t>(t0 + tl) * K;
    int j = 0;
    for (int r = 0; r < W; ++r) {
      const bool has = (mask >> r) & 1ull;
      const unsigned b = __ballot_sync(0xffffffffu, has);
      if (has) {
        const int pos = woff[warp * W + r] + __popc(b & lanemask_lt());
        const int row = rbase[r] + pos;
        ss[j++] = row;
        sorted[rcx[r] + pos] = make_int2(tl, row);
#pragma unroll
        for (int k = 0; k < KM; ++k)
          if (k < K && rk[k] == r) dslot[tl * K + k] = row;
      }
    }
    if (tl < ntok) {
      for (; j < K; ++j) ss[j] = -1;
      int32_t* ds = p.dst_slot + static_cast<int64_t>(t0 + tl) * K;
#pragma unroll
      for (int k = 0; k < KM; ++k)
        if (k < K) {
          if (rk[k] < 0) dslot[tl * K + k] = -1;
          ds[k] = dslot[tl * K + k];
        }
      const int t = t0 + tl, sr = t / T;
      src[2 * tl] = sr;
      src[2 * tl + 1] = t - sr * T;
    }
  }
  __syncthreads();

  // metadata rows of this chunk in (rank, token) order: the rows of one rank
  // from one chunk are contiguous, so consecutive threads write consecutive words
  if (has_tokens) {
    const int nvalid = rcx[W];
    if ((KW & 1) == 0) {
      const int hw = KW / 2;
      for (int f = tid; f < nvalid * hw; f += kSlotThreads) {
        const int q = f / hw, c2 = f - q * hw;
        const int2 e = sorted[q];
        const int2 v = c2 == 0 ? make_int2(src[2 * e.x], src[2 * e.x + 1])
                               : make_int2(dslot[e.x * K + 2 * c2 - 2], dslot[e.x * K + 2 * c2 - 1]);
        reinterpret_cast<int2*>(p.meta + static_cast<int64_t>(e.y) * KW)[c2] = v;
      }
    } else {
      for (int f = tid; f < nvalid * KW; f += kSlotThreads) {
        const int q = f / KW, col = f - q * KW;
        const int2 e = sorted[q];
        const int v = col < 2 ? src[2 * e.x + col] : dslot[e.x * K + col - 2];
        p.meta[static_cast<int64_t>(e.y) * KW + col] = v;
      }
    }
  }

  // this CTA's slice of the rows that receive nothing, [R, capacity)
  const int64_t tail_beg = static_cast<int64_t>(prank[W]) * KW;
  const int64_t tail_words = p.rcap * KW - tail_beg;
  const int64_t per = (tail_words + gridDim.x - 1) / gridDim.x;
  const int64_t sbeg = tail_beg + per * c;
  const int64_t send = sbeg + per < p.rcap * KW ? sbeg + per : p.rcap * KW;
  for (int64_t f = sbeg + tid; f < send; f += kSlotThreads) p.meta[f] = -1;
}

// ---------------------------------------------------------------- launch

template <class Kern>
cudaError_t launch_dependent(Kern kernel, int grid, int block, size_t smem, cudaStream_t s,
                             const LayoutParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

size_t count_smem(int topk, int cols) {
  return sizeof(int32_t) * (static_cast<size_t>(kLayoutCountWarps) * cols +
                            static_cast<size_t>(kLayoutTPC) * topk);
}

size_t slots_smem(int E, int topk) {
  return sizeof(int32_t) * (5 * static_cast<size_t>(E) + 2 + 33 + 2 * kLayoutTPC * topk +
                            2 * kLayoutTPC);
}

size_t slots_ne_smem(int E, int W, int topk) {
  const size_t rm = static_cast<size_t>(topk < W ? topk : W);
  return sizeof(int32_t) * (2 * kLayoutTPC * rm + 5 * static_cast<size_t>(W) + 2 +
                            static_cast<size_t>(kTokenWarps) * W + 33 +
                            static_cast<size_t>(kLayoutTPC) * topk + 2 * kLayoutTPC +
                            2 * static_cast<size_t>(E) + 1);
}

template <int KC, bool NE>
cudaError_t launch_layout(const LayoutParams& p, const LaunchGeom& g, cudaStream_t s) {
  const int EW = p.num_experts + p.world_size;
  if (p.num_chunks > 0)
    ep_layout_count_kernel<KC><<<p.num_chunks, kCountThreads, count_smem(p.topk, EW), s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_dependent(ep_layout_spine_kernel, (EW + kSpineWarps - 1) / kSpineWarps,
                       kSpineWarps * 32, 0, s, p);
  if (e != cudaSuccess) return e;
  const int grid = p.num_chunks > g.num_sms ? p.num_chunks : g.num_sms;
  if constexpr (NE)
    return launch_dependent(ep_layout_slots_ne_kernel<KC>, grid, kSlotThreads,
                            slots_ne_smem(p.num_experts, p.world_size, p.topk), s, p);
  else
    return launch_dependent(ep_layout_slots_kernel<KC>, grid, kSlotThreads,
                            slots_smem(p.num_experts, p.topk), s, p);
}

// Shared-memory limits are set to what the largest launch can need (every E+W
// and, for the generic variant, every top-k the library accepts), so that
// handles with different shapes never lower them for each other.
template <int KC, bool NE>
cudaError_t prepare_layout(int, int, int, LaunchGeom* g) {
  const int kmax = KC ? KC : kMaxTopk;
  cudaError_t e = cudaFuncSetAttribute(ep_layout_count_kernel<KC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(count_smem(kmax, kMaxExperts + kMaxWorld)));
  if (e != cudaSuccess) return e;
  if constexpr (NE)
    e = cudaFuncSetAttribute(ep_layout_slots_ne_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(slots_ne_smem(kMaxExperts, kMaxWorld, kmax)));
  else
    e = cudaFuncSetAttribute(ep_layout_slots_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(slots_smem(kMaxExperts, kmax)));
  if (e != cudaSuccess) return e;
  g->blocks_per_sm = 1;
  return cudaSuccess;
}

}  // namespace

int64_t LayoutScratchInts(int max_chunks, int columns) {
  return 2LL * columns * (max_chunks > 0 ? max_chunks : 1) + columns;
}

void BindLayoutScratch(LayoutParams* p, int32_t* base, int max_chunks, int columns) {
  const int64_t cap = max_chunks > 0 ? max_chunks : 1;
  p->chunk_hist = base;
  p->chunk_off = base + static_cast<int64_t>(columns) * cap;
  p->col_total = p->chunk_off + static_cast<int64_t>(columns) * cap;
}

uint32_t RankMagic(int num_expert_per_rank) {
  // m = floor(2^32 / d) + 1 gives umulhi(e, m) = floor(e/d + e*(d - 2^32 mod d)/(d*2^32)):
  // the added term is below 2^-21 while e/d is at least 1/d >= 2^-11 short of the
  // next integer, so the result is e / d for every e < 2^11 and 2 <= d <= 2^11.
  if (num_expert_per_rank <= 1) return 0u;
  return static_cast<uint32_t>((1ull << 32) / static_cast<uint64_t>(num_expert_per_rank) + 1ull);
}

Variant<LayoutLaunch> FindLayout(int topk, bool no_expand) {
  if (no_expand) switch (topk) {
      case 4: return {"ep_layout_nonexpand_k4", launch_layout<4, true>, prepare_layout<4, true>};
      case 6: return {"ep_layout_nonexpand_k6", launch_layout<6, true>, prepare_layout<6, true>};
      case 8: return {"ep_layout_nonexpand_k8", launch_layout<8, true>, prepare_layout<8, true>};
      default: return {"ep_layout_nonexpand_generic", launch_layout<0, true>, prepare_layout<0, true>};
    }
  switch (topk) {
    case 4: return {"ep_layout_k4", launch_layout<4, false>, prepare_layout<4, false>};
    case 6: return {"ep_layout_k6", launch_layout<6, false>, prepare_layout<6, false>};
    case 8: return {"ep_layout_k8", launch_layout<8, false>, prepare_layout<8, false>};
    default: return {"ep_layout_generic", launch_layout<0, false>, prepare_layout<0, false>};
  }
}

}  // namespace epg
