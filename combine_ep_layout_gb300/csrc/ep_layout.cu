// ep_layout.cu -- layout of the routing: per-expert / per-rank histograms,
// aligned exclusive prefix sums, deterministic destination slots and
// recv_src_metadata (EPHandle fields of "DeepEP overall architecture
// analysis"; the counting role of its "notify warps" in the Dispatch data flow
// figure).
//
// Rows of one expert are ordered by the flat index t*K+k, so the slot of an
// entry is psum_expert[e] + (number of earlier entries routed to e): a stable
// counting sort.  The tokens are cut into ranges, one per CTA; each range is
// counted (count_tokens), the ranges' counts are scanned, and each range
// writes its slots and metadata.  Three ways to run that, by batch size:
//
// Counting (the same device code everywhere): a range's entries, flat index
// (t - t0)*K + k, are cut into one run of whole 32-entry batches per warp;
// each lane loads its ids straight into registers.  Per batch the lanes that
// carry the same expert find each other (one ballot per bit of the expert
// id), so one pass gives each warp's histogram (a row private to the warp)
// and every entry's rank among its warp's earlier entries of that expert.  A thread per column
// then scans the 16 warps' counts (each warp's start, the range's total);
// tokens per rank come from per-token rank masks counted with ballots.
//
// Large batches, three launches (the last two with programmatic dependent
// launch so that each is scheduled while its predecessor drains; the last
// one, like the single-launch kernels, lets the dispatch that follows be
// scheduled early too):
//   count  one CTA per chunk of kLayoutTPC tokens: the ranks go to dst_slot,
//          the chunk's column totals (E experts + W ranks) to a row-major
//          [C][E+W] table and a column-major copy.
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
// Small batches (up to kClusterCtas * kClusterMaxTPB tokens), one launch: a
// single thread-block cluster, one CTA per token range.  Each CTA counts its
// range into shared memory; after a cluster barrier every CTA reads the other
// CTAs' column totals through distributed shared memory (its offset inside
// each column is the sum over the CTAs before it), and goes on to the slots
// and metadata of its range without another launch.  A second cluster barrier
// keeps every CTA's shared memory alive until the others have read it.
//
// Mid-size batches (as many ranges as a cooperative grid keeps resident), one
// launch: the fused kernel counts each range like the cluster kernel, but
// exchanges the column totals through L2 -- a row per range and atomic sums
// per superchunk of 16 ranges -- around one grid barrier (split into arrive
// and wait, with the range's local sort in between), then finishes its range
// with the same device code.  This is the single-pass form of the
// counting the pages give the "notify warps" of the Dispatch data flow
// figure: no count / scan / slots kernel boundaries, ranks kept on chip.
//
// Non-expand layout (EPHandle do_expand = false): one row per (token,
// destination rank).  The counting is shared (the rank columns already count
// each range's tokens per rank); the slots step places rank r's tokens in
// ascending order from psum_rank[r] on, using warp ballots over the tokens'
// rank masks for the position inside the range.
//
// Waits: the cluster barriers, which every thread of every CTA of the cluster
// reaches unconditionally, and the fused kernel's grid barrier, whose wait is
// bounded by %globaltimer (LayoutParams::wait_ns): a CTA that gives up records
// device error value 2 (bit 1) and returns.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

constexpr int kCountThreads = kLayoutCountWarps * 32;
// Resident count CTAs per SM asked of the compiler (at most 42 registers): the
// 256 chunks of a 32768-token batch then run in one wave.  (The runtime-top-k
// variant carries up to 16 ids per thread and asks for 2.)
constexpr int kCountMinBlocks = 3;
constexpr int kSpineWarps = 8;
constexpr int kSlotThreads = 512;
constexpr int kClusterThreads = kCountThreads;   // the cluster kernel counts like count
constexpr int kClusterCtas = 8;                  // portable cluster size
constexpr int kClusterMaxTPB = 2 * kLayoutTPC;   // tokens per CTA of the cluster kernel
// The cluster kernel is used when its padding and tail rows are few (at most
// this many rows to fill with -1 on kClusterCtas SMs) and its shared memory fits.
constexpr int64_t kClusterMaxFillRows = 1 << 16;
constexpr size_t kClusterMaxSmem = 160 * 1024;

__device__ __forceinline__ int expert_of(int64_t v, int E) {
  return (v >= 0 && v < E) ? static_cast<int>(v) : -1;
}

// Rank of expert e, e / Epr, as a multiply-high with the magic number of
// RankMagic (0 when Epr == 1).
__device__ __forceinline__ int rank_of(int e, uint32_t magic) {
  return magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(e), magic)) : e;
}

// ---- thread-block cluster primitives (sm_90 and later) ----------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Arrive at the cluster barrier (release: this thread's shared-memory writes
// become visible to the cluster) / wait for every thread of the cluster to
// arrive (acquire).  Every thread of every CTA executes both, warp-converged.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive without releasing anything: for a signal that publishes no writes
// (no fence on the way).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Load the int32 at the same shared-memory offset as `local` in CTA `rank` of
// the cluster (distributed shared memory).
__device__ __forceinline__ int32_t ld_cluster_shared(const int32_t* local, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  int32_t v;
  asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// ---- scans --------------------------------------------------------------------

// v rounded up to a multiple of A.  P2: A is a power of two (a mask); the
// callers test that once per scan, so no element pays for a division it does
// not need.
template <bool P2>
__device__ __forceinline__ int align_to(int v, int A) {
  return P2 ? (v + A - 1) & -A : (v + A - 1) / A * A;
}

// Block-wide exclusive scan of align(v[e], A) for e in [0, n) into out[0..n]
// (out[n] = total).  warp_tot needs 33 words.  All threads must call it.
template <bool P2>
__device__ void block_exclusive_scan_a(const int32_t* v, int n, int A, int32_t* out, int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  const int V = (n + nthr - 1) / nthr;
  const int beg = min(n, tid * V), end = min(n, beg + V);
  int sum = 0;
  for (int e = beg; e < end; ++e) sum += align_to<P2>(v[e], A);
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
    run += align_to<P2>(v[e], A);
  }
  if (tid == 0) out[n] = warp_tot[32];
  __syncthreads();
}

__device__ void block_exclusive_scan(const int32_t* v, int n, int A, int32_t* out, int32_t* warp_tot) {
  if ((A & (A - 1)) == 0) block_exclusive_scan_a<true>(v, n, A, out, warp_tot);
  else block_exclusive_scan_a<false>(v, n, A, out, warp_tot);
}

// Exclusive scan of align(v[e], A) for e in [0, n) by one warp (ceil(n/32)
// consecutive values per lane) into out[0..n] (out[n] = total).
template <bool P2>
__device__ __forceinline__ void warp_exclusive_scan_a(const int32_t* v, int n, int A, int32_t* out) {
  const int lane = threadIdx.x & 31;
  const int V = (n + 31) / 32;
  const int beg = min(n, lane * V), end = min(n, beg + V);
  int sum = 0;
  int incl;
  if (V <= 16) {  // the lane's values in registers, all loads in flight at once
    int x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      x[u] = beg + u < end ? align_to<P2>(v[beg + u], A) : 0;
      sum += x[u];
    }
    incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (beg + u < end) {
        out[beg + u] = run;
        run += x[u];
      }
  } else {
    for (int e = beg; e < end; ++e) sum += align_to<P2>(v[e], A);
    incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int e = beg; e < end; ++e) {
      out[e] = run;
      run += align_to<P2>(v[e], A);
    }
  }
  if (lane == 31) out[n] = incl;
}

__device__ __forceinline__ void warp_exclusive_scan(const int32_t* v, int n, int A, int32_t* out) {
  if ((A & (A - 1)) == 0) warp_exclusive_scan_a<true>(v, n, A, out);
  else warp_exclusive_scan_a<false>(v, n, A, out);
}

// Two exclusive scans over the E <= blockDim.x experts at once, from values
// the threads hold in registers (thread e: a = expert e's total, rounded up
// to A into out_a; b = its count, into out_b; E+1 outputs each).  All threads
// call; one block barrier inside, a second before returning so that both
// outputs are visible.  warp_tot needs 2 * (blockDim.x / 32) words.
__device__ void dual_block_scan(int a, int b, int A, int E, int32_t* out_a, int32_t* out_b,
                                int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  const bool p2 = (A & (A - 1)) == 0;
  const int va = tid < E ? (p2 ? align_to<true>(a, A) : align_to<false>(a, A)) : 0;
  const int vb = tid < E ? b : 0;
  int ia = va, ib = vb;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, ia, o);
    const int yb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += ya;
      ib += yb;
    }
  }
  if (lane == 31) {
    warp_tot[warp] = ia;
    warp_tot[nwarp + warp] = ib;
  }
  __syncthreads();
  int ba = 0, bb = 0;
  for (int w = 0; w < warp; ++w) {
    ba += warp_tot[w];
    bb += warp_tot[nwarp + w];
  }
  if (tid < E) {
    out_a[tid] = ba + ia - va;
    out_b[tid] = bb + ib - vb;
  }
  if (tid == E - 1) {
    out_a[E] = ba + ia;
    out_b[E] = bb + ib;
  }
  __syncthreads();
}

// Expert counts up to this many are scanned by single warps (no block barriers
// inside the scan; at most 16 values per lane); larger ones by the whole block.
constexpr int kWarpScanMax = 512;

// The two exclusive scans over the E experts: align(a[e], A) into out_a and,
// when b is non-null, b[e] into out_b (E+1 outputs each).  All threads call;
// the results are visible to the whole CTA on return.  For E <= kWarpScanMax
// warps 0 and 1 scan one array each, at the same time, behind one barrier.
__device__ void expert_scans(const int32_t* a, int A, int32_t* out_a, const int32_t* b,
                             int32_t* out_b, int E, int32_t* warp_tot) {
  if (E <= kWarpScanMax) {
    const int warp = threadIdx.x >> 5;
    if (warp == 0) warp_exclusive_scan(a, E, A, out_a);
    else if (warp == 1 && b != nullptr) warp_exclusive_scan(b, E, 1, out_b);
    __syncthreads();
  } else {
    block_exclusive_scan(a, E, A, out_a, warp_tot);
    if (b != nullptr) block_exclusive_scan(b, E, 1, out_b, warp_tot);
  }
}

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

// ---------------------------------------------------------------- count

// Batches of 32 entries a warp of a counting CTA walks at most: ranges of up to
// kClusterMaxTPB tokens, kLayoutCountWarps warps.
template <int KC>
constexpr int CountBatches() {
  return ((kClusterMaxTPB * (KC ? KC : kMaxTopk) + kLayoutCountWarps - 1) / kLayoutCountWarps + 31) / 32;
}

// What a counting thread keeps in registers for the slot pass of the same CTA:
// the expert of its entry in each batch (-1: none) and the entry's rank among
// the earlier entries of that expert in its warp's run.
template <int KC>
struct CountRegs {
  int e[CountBatches<KC>()];
  int loc[CountBatches<KC>()];
};

// The lanes of the calling warp whose key equals this lane's, for keys below
// 2^nbits: the AND over the key's bits of the ballot of lanes that share that
// bit.  The same mask as __match_any_sync on the key, which costs about twice
// as much on this GPU (measured: ~820 cycles for 16 warps' match.any against
// ~440 for six ballots and ~545 for eight, in a loop of one CTA of 16 warps).
constexpr int kBallotKeyBits = 9;
__device__ __forceinline__ unsigned peers_by_ballots(int key, int nbits) {
  unsigned peers = 0xffffffffu;
#pragma unroll
  for (int bit = 0; bit < kBallotKeyBits; ++bit) {
    if (bit < nbits) {  // uniform across the warp
      const bool set = (key >> bit) & 1;
      const unsigned bb = __ballot_sync(0xffffffffu, set);
      peers &= set ? bb : ~bb;
    }
  }
  return peers;
}

// Token rank masks are OR-reduced over each token's lanes with shuffles when
// K is a power of two that divides 32 (then a 32-entry batch holds whole
// tokens); otherwise each entry sets its bit with a shared-memory atomic.
template <int KC>
constexpr bool ShuffleMasks() { return KC != 0 && 32 % KC == 0; }

// Count the tokens [t0, t0 + ntok) of this CTA (kCountThreads threads, all of
// which call this).  The range's entries, flat index i = (t - t0)*K + k, are cut
// into one contiguous run of whole 32-entry batches per warp.  For each batch
// the lanes that carry the same expert find each other (ballots over the bits
// of the expert id, or __match_any_sync for more than 511 experts):
// an entry's rank among its run's earlier entries of its expert is the warp's
// running count of that expert (the warp's own row of whist, which only that
// warp touches until the barrier) plus the lanes of its group below it.  One
// pass therefore gives the warp's histogram and every entry's stable rank in
// the run.  Tokens per rank: each token's rank mask (bit r: an expert on rank
// r) goes to tmask[t - t0], and after the barrier ballots count each rank's
// bit.  On return (after one block barrier; the caller barriers again before
// reading them):
//   whist [NW][E+W]  each warp's exclusive start per expert (a scan over the warps)
//   colcnt [E+W]     the range's entries per expert, then tokens per rank
//   ids [ntok*K]     the staged expert ids (-1: skipped), when non-null
//   regs             per batch: expert and rank within the warp's run
// A range entry's rank among all the range's entries of expert e is
// whist[warp][e] + regs.loc[b].
template <int KC>
__device__ void count_tokens(const LayoutParams& p, int t0, int ntok, int32_t* whist,
                             unsigned long long* tmask, int32_t* colcnt, int32_t* ids,
                             CountRegs<KC>& regs) {
  constexpr int NW = kLayoutCountWarps;
  constexpr int NB = CountBatches<KC>();
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, W = p.world_size;
  const int EW = E + W;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nent = ntok * K;
  const int per_warp = (((nent + NW - 1) / NW) + 31) & ~31;
  const int wbeg = warp * per_warp;
  const int wend = min(nent, wbeg + per_warp);
  const int64_t* topk = p.topk_idx + static_cast<int64_t>(t0) * K;
  int32_t* clone = p.topk_i32 ? p.topk_i32 + static_cast<int64_t>(t0) * K : nullptr;

  // all of the warp's ids in flight at once
  int64_t raw[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int i = wbeg + b * 32 + lane;
    raw[b] = (b * 32 < per_warp && i < wend) ? topk[i] : -1;
  }
  int32_t* wh = whist + warp * EW;
  for (int j = lane; j < EW; j += 32) wh[j] = 0;
  if constexpr (!ShuffleMasks<KC>()) {
    for (int t = tid; t < ntok; t += kCountThreads) tmask[t] = 0ull;
    __syncthreads();
  }
  __syncwarp();

  bool bad = false;
  // the key of a lane: its expert, E when skipped; matched by one ballot per
  // key bit when that takes at most kBallotKeyBits ballots, else by match.any
  const int kb = 32 - __clz(E);
  const int key_bits = kb <= kBallotKeyBits ? kb : 0;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b * 32 >= per_warp) break;  // warp-uniform: the run's batches are done
    const int i = wbeg + b * 32 + lane;
    const bool in = i < wend;
    const int e = in ? expert_of(raw[b], E) : -1;
    bad |= in && e < 0 && raw[b] != -1;
    if (in) {
      if (ids) ids[i] = e;
      if (clone) clone[i] = e;
    }
    const unsigned peers = key_bits ? peers_by_ballots(e >= 0 ? e : E, key_bits)
                                    : __match_any_sync(0xffffffffu, e);
    const int base = e >= 0 ? wh[e] : 0;
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wh[e] = base + __popc(peers);
    __syncwarp();
    regs.e[b] = e;
    regs.loc[b] = base + __popc(peers & lanemask_lt());
    unsigned long long m = e >= 0 ? 1ull << rank_of(e, p.epr_magic) : 0ull;
    if constexpr (ShuffleMasks<KC>()) {
#pragma unroll
      for (int o = 1; o < KC; o <<= 1) m |= __shfl_xor_sync(0xffffffffu, m, o);
      if (in && i % KC == 0) tmask[i / KC] = m;
    } else {
      if (m) atomicOr(&tmask[i / K], m);
    }
  }
  if (bad) atomicOr(p.err, kErrBadExpert);
  __syncthreads();

  // per expert, a thread scans its column of the 16 warps' counts: each warp's
  // start and the range's total (consecutive threads touch consecutive words:
  // no bank conflicts; eight loads in flight before the first add)
  for (int j = tid; j < E; j += kCountThreads) {
    int run = 0;
#pragma unroll
    for (int w0 = 0; w0 < NW; w0 += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = whist[(w0 + u) * EW + j];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        whist[(w0 + u) * EW + j] = run;
        run += v[u];
      }
    }
    colcnt[j] = run;
  }
  // tokens per rank: count each rank's bit over the token masks
  for (int r = warp; r < W; r += NW) {
    int c = 0;
    for (int t = lane; t - lane < ntok; t += 32) {
      const unsigned long long m = t < ntok ? tmask[t] : 0ull;
      c += __popc(__ballot_sync(0xffffffffu, (m >> r) & 1ull));
    }
    if (lane == 0) colcnt[E + r] = c;
  }
}

// Each counted entry's rank among all of its range's entries of its expert
// (the slots' offset inside the range), written to loc[i] (-1 when skipped).
// After a barrier that follows count_tokens.
template <int KC>
__device__ __forceinline__ void write_range_ranks(int ntok, int K, const int32_t* whist, int EW,
                                                  const CountRegs<KC>& regs, int32_t* loc) {
  constexpr int NW = kLayoutCountWarps;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nent = ntok * K;
  const int per_warp = (((nent + NW - 1) / NW) + 31) & ~31;
  const int wbeg = warp * per_warp;
  const int wend = min(nent, wbeg + per_warp);
#pragma unroll
  for (int b = 0; b < CountBatches<KC>(); ++b) {
    if (b * 32 >= per_warp) break;
    const int i = wbeg + b * 32 + lane;
    if (i < wend) {
      const int e = regs.e[b];
      loc[i] = e >= 0 ? whist[warp * EW + e] + regs.loc[b] : -1;
    }
  }
}

// Shared-memory words of the counting scratch (whist, tmask as 64-bit words,
// colcnt) for E+W columns and up to tpb tokens.
__host__ __device__ constexpr int CountSmemWords(int EW, int tpb) {
  return kLayoutCountWarps * EW + 2 * tpb + EW;
}

template <int KC>
__global__ void __launch_bounds__(kCountThreads, KC ? kCountMinBlocks : 2) ep_layout_count_kernel(LayoutParams p) {
  const int K = KC ? KC : p.topk;
  const int EW = p.num_experts + p.world_size;
  extern __shared__ __align__(16) int32_t sm[];
  auto* tmask = reinterpret_cast<unsigned long long*>(sm);   // [TPC]
  int32_t* whist = sm + 2 * kLayoutTPC;                      // [NW][EW]
  int32_t* colcnt = whist + kLayoutCountWarps * EW;          // [EW]
  const int c = blockIdx.x;
  const int t0 = c * kLayoutTPC;
  const int ntok = min(p.num_tokens, t0 + kLayoutTPC) - t0;
  allow_dependent_grids();
  CountRegs<KC> regs;
  count_tokens<KC>(p, t0, ntok, whist, tmask, colcnt, nullptr, regs);
  __syncthreads();
  // the range ranks go to dst_slot, which the slots kernel turns into slots
  if (!p.no_expand)
    write_range_ranks<KC>(ntok, K, whist, EW, regs, p.dst_slot + static_cast<int64_t>(t0) * K);
  // the range's column totals: a contiguous row of the [C][E+W] table (read
  // by the slots kernel) and a column entry of the [E+W][C] copy (read by the
  // spine, one column per warp)
  for (int j = threadIdx.x; j < EW; j += kCountThreads) {
    p.chunk_hist[static_cast<int64_t>(c) * EW + j] = colcnt[j];
    p.chunk_hist_cols[static_cast<int64_t>(j) * p.num_chunks + c] = colcnt[j];
  }
}

// ---------------------------------------------------------------- spine

// A warp per column j of the [C][E+W] table: exclusive scan over the C chunks
// (each lane a contiguous run of chunks, kept in registers when short).
__global__ void __launch_bounds__(kSpineWarps * 32) ep_layout_spine_kernel(LayoutParams p) {
  const int EW = p.num_experts + p.world_size;
  const int C = p.num_chunks;
  const int j = blockIdx.x * kSpineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  allow_dependent_grids();
  grid_dependency_wait();
  if (j >= EW) return;
  // column j: read contiguously from the [E+W][C] copy, written into the
  // row-major [C][E+W] offsets table that the slots kernel reads by rows
  const int32_t* in = p.chunk_hist_cols + static_cast<int64_t>(j) * C;
  int32_t* out = p.chunk_off + j;
  const int64_t ld = EW;
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
        out[(cbeg + u) * ld] = run;
        run += reg[u];
      }
  } else {
    for (int c = cbeg; c < cend; ++c) {
      const int v = in[c];
      out[c * ld] = run;
      run += v;
    }
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) p.col_total[j] = total;
}

// ---------------------------------------------------------------- slots (expand)

// CTA 0's outputs: counts, aligned expert prefix, rank prefix at each rank's
// first expert, tokens per rank, number of receive rows.
__device__ void write_outputs_expand(const LayoutParams& p, const int32_t* cnt_s,
                                     const int32_t* psum_s, const int32_t* tpr) {
  const int E = p.num_experts, W = p.world_size;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    p.psum_expert[e] = psum_s[e];
    if (e < E) p.cnt[e] = cnt_s[e];
  }
  for (int r = threadIdx.x; r <= W; r += blockDim.x) {
    p.psum_rank[r] = psum_s[r * p.num_expert_per_rank];
    if (r < W) p.tok_per_rank[r] = tpr[r];
  }
  if (threadIdx.x == 0) *p.num_recv = psum_s[E];
}

template <int KC>
__device__ void write_metadata_rows(const LayoutParams& p, int nvalid, const int32_t* sorted,
                                    const int32_t* slots_s, const int32_t* src);

// Slots and metadata of the tokens [t0, t0 + ntok) of this CTA (expand
// layout; all threads call, entry i = (t - t0)*K + k spread over all of them).
// psum_s [E+1] is the aligned expert prefix, co[E] the range's offset inside
// each expert's rows, cx[E+1] the exclusive scan over experts of the range's
// counts, loc[i] the entry's rank among the range's entries of its expert
// (may alias p.dst_slot of the range, which is overwritten with the slots),
// ids[i] the staged expert ids or nullptr (then read from topk_idx).
// Scratch: slots_s and sorted [ntok*K], src [2*ntok]; slots_s and src 8-byte
// aligned (the metadata rows are read from them as word pairs).
template <int KC>
__device__ void slots_expand_tokens(const LayoutParams& p, int t0, int ntok, const int32_t* psum_s,
                                    const int32_t* co, const int32_t* cx, const int32_t* loc,
                                    const int32_t* ids, int32_t* slots_s, int32_t* sorted,
                                    int32_t* src) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, T = p.max_tok_per_rank;
  const int nthr = blockDim.x;
  const int nent = ntok * K;
  int32_t* ds = p.dst_slot + static_cast<int64_t>(t0) * K;
  const int64_t* topk = p.topk_idx + static_cast<int64_t>(t0) * K;
  for (int i = threadIdx.x; i < nent; i += nthr) {
    const int e = ids ? ids[i] : expert_of(topk[i], E);
    const int l = loc[i];  // read before ds[i] (possibly the same word) is overwritten
    const int slot = e >= 0 ? psum_s[e] + co[e] + l : -1;
    if (e >= 0) sorted[cx[e] + l] = i;
    ds[i] = slot;
    slots_s[i] = slot;
  }
  for (int tl = threadIdx.x; tl < ntok; tl += nthr) {
    const int t = t0 + tl, r = t / T;
    src[2 * tl] = r;
    src[2 * tl + 1] = t - r * T;
  }
  __syncthreads();
  write_metadata_rows<KC>(p, cx[E], sorted, slots_s, src);
}

// The metadata rows of a range, in (expert, rank) order: sorted[q] is the entry
// of the range's q-th row (nvalid rows), slots_s[i] entry i's slot and src the
// tokens' {t / T, t mod T} (both 8-byte aligned).  Flat words f of the
// concatenated rows: rows of one expert are contiguous in memory, so
// consecutive threads write consecutive words.  (One row per thread instead
// measured 29% slower at prefill: the stores lose their coalescing.)  All
// threads call, after a barrier that makes the inputs visible.
template <int KC>
__device__ void write_metadata_rows(const LayoutParams& p, int nvalid, const int32_t* sorted,
                                    const int32_t* slots_s, const int32_t* src) {
  const int K = KC ? KC : p.topk;
  const int KW = K + 2;  // metadata row width
  const int nthr = blockDim.x;
  if ((KW & 1) == 0) {
    // even row width: word pairs (8-byte stores; rows start 8-byte aligned)
    const int hw = KW / 2;
    for (int f = threadIdx.x; f < nvalid * hw; f += nthr) {
      const int q = f / hw, c2 = f - q * hw;
      const int entry = sorted[q];
      const int tl = entry / K;
      // one 8-byte load per word pair (src and slots_s are 8-byte aligned, K even)
      const int2 v = *reinterpret_cast<const int2*>(c2 == 0 ? src + 2 * tl : slots_s + tl * K + 2 * c2 - 2);
      reinterpret_cast<int2*>(p.meta + static_cast<int64_t>(slots_s[entry]) * KW)[c2] = v;
    }
  } else {
    for (int f = threadIdx.x; f < nvalid * KW; f += nthr) {
      const int q = f / KW, col = f - q * KW;
      const int entry = sorted[q];
      const int tl = entry / K;
      const int v = col < 2 ? src[2 * tl + col] : slots_s[tl * K + col - 2];
      p.meta[static_cast<int64_t>(slots_s[entry]) * KW + col] = v;
    }
  }
}

// -1 into the rows that receive nothing, share `part` of `parts`: the padding
// rows of the experts (cnt_s non-null: expand layout; a warp per expert, none
// when A == 1) and a slice of [R, capacity).
__device__ void fill_unreceived(const LayoutParams& p, const int32_t* psum_s, const int32_t* cnt_s,
                                int R, int part, int parts) {
  const int KW = p.topk + 2;
  const int nthr = blockDim.x;
  if (cnt_s != nullptr && p.alignment > 1) {
    // a warp per expert, experts dealt round-robin over the CTAs first (CTA
    // `part` takes experts part, part + parts, ...), so that the padding is
    // spread over the grid instead of loading its first CTAs
    const int lane = threadIdx.x & 31, nwarp = nthr >> 5;
    for (int e = part + (threadIdx.x >> 5) * parts; e < p.num_experts; e += parts * nwarp) {
      const int64_t beg = static_cast<int64_t>(psum_s[e] + cnt_s[e]) * KW;
      const int64_t end = static_cast<int64_t>(psum_s[e + 1]) * KW;
      for (int64_t f = beg + lane; f < end; f += 32) p.meta[f] = -1;
    }
  }
  const int64_t tail_beg = static_cast<int64_t>(R) * KW;
  const int64_t tail_words = p.rcap * KW - tail_beg;
  const int64_t per = (tail_words + parts - 1) / parts;
  const int64_t sbeg = tail_beg + per * part;
  const int64_t send = sbeg + per < p.rcap * KW ? sbeg + per : p.rcap * KW;
  for (int64_t f = sbeg + threadIdx.x; f < send; f += nthr) p.meta[f] = -1;
}

template <int KC>
__global__ void __launch_bounds__(kSlotThreads, 1) ep_layout_slots_kernel(LayoutParams p) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, C = p.num_chunks;
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* psum_s = sm;                   // [E+1]
  int32_t* cnt_s = psum_s + E + 1;        // [E]
  int32_t* cl = cnt_s + E;                // [E]   this chunk's count per expert
  int32_t* co = cl + E;                   // [E]   chunk_off of this chunk per expert
  int32_t* cx = co + E;                   // [E+1] exclusive scan of cl over experts
  int32_t* warp_tot = cx + E + 1;         // [33]
  int32_t* slots_s = warp_tot + 33 + ((5 * E + 35) & 1);   // [TPC*K], 8-byte aligned
  int32_t* sorted = slots_s + kLayoutTPC * K;  // [TPC*K] entries ordered by (expert, rank)
  int32_t* src = sorted + kLayoutTPC * K;      // [2*TPC] {t / T, t mod T} per token

  const int c = blockIdx.x;
  const bool has_tokens = c < C;
  allow_dependent_grids();   // the dispatch that follows may be scheduled now
  grid_dependency_wait();
  const int64_t row = static_cast<int64_t>(c) * (E + p.world_size);  // this chunk's table row
  for (int e = threadIdx.x; e < E; e += kSlotThreads) {
    cnt_s[e] = p.col_total[e];
    if (has_tokens) {
      cl[e] = p.chunk_hist[row + e];
      co[e] = p.chunk_off[row + e];
    }
  }
  __syncthreads();
  // the aligned exclusive prefix over experts (every CTA; E values) and the
  // scan of this chunk's counts
  expert_scans(cnt_s, p.alignment, psum_s, has_tokens ? cl : nullptr, cx, E, warp_tot);
  if (c == 0) write_outputs_expand(p, cnt_s, psum_s, p.col_total + E);
  if (has_tokens) {  // uniform per CTA
    const int t0 = c * kLayoutTPC;
    const int ntok = min(p.num_tokens, t0 + kLayoutTPC) - t0;
    slots_expand_tokens<KC>(p, t0, ntok, psum_s, co, cx, p.dst_slot + static_cast<int64_t>(t0) * K,
                            nullptr, slots_s, sorted, src);
  }
  fill_unreceived(p, psum_s, cnt_s, psum_s[E], c, gridDim.x);
}

// ---------------------------------------------------------------- slots (non-expand)

// Rank r's rows are its tokens in ascending order: the row of (t, r) is
// psum_rank[r] + (the range's offset in rank r) + (tokens of the range before
// t that reach r).  Token warps (threads < tpb, tpb a multiple of 32, token
// t0 + i owned by thread i) take each rank's positions from a ballot per warp
// and an exclusive scan over the token warps.  rbase[W] = psum_rank[r] + the
// range's offset, rcx[W+1] = exclusive scan over ranks of the range's tokens
// per rank; scratch: woff [tpb/32][W], dslot [tpb*K], src [2*tpb], sorted
// [tpb*min(K, W)] (8-byte aligned).  All threads call.
template <int KC>
__device__ void slots_nonexpand_tokens(const LayoutParams& p, int t0, int ntok, int tpb,
                                       const int32_t* rbase, const int32_t* rcx, const int32_t* ids,
                                       int32_t* woff, int32_t* dslot, int32_t* src, int2* sorted) {
  constexpr int KM = KC ? KC : kMaxTopk;
  const int K = KC ? KC : p.topk;
  const int KW = K + 2;
  const int E = p.num_experts, W = p.world_size, T = p.max_tok_per_rank;
  const int TW = tpb / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x;
  const int tl = tid;                      // token of this thread (token warps only)
  unsigned long long mask = 0ull;
  int rk[KM];                              // rank of each entry, -1 when skipped
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    rk[k] = -1;
    if (k < K && warp < TW && tl < ntok) {
      const int e = ids ? ids[tl * K + k]
                        : expert_of(p.topk_idx[static_cast<int64_t>(t0 + tl) * K + k], E);
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
  for (int r = tid; r < W; r += nthr) {
    int run = 0;
    for (int w = 0; w < TW; ++w) {
      const int v = woff[w * W + r];
      woff[w * W + r] = run;
      run += v;
    }
  }
  __syncthreads();

  if (warp < TW) {
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

  // metadata rows of this range in (rank, token) order: the rows of one rank
  // from one range are contiguous, so consecutive threads write consecutive words
  const int nvalid = rcx[W];
  if ((KW & 1) == 0) {
    const int hw = KW / 2;
    for (int f = tid; f < nvalid * hw; f += nthr) {
      const int q = f / hw, c2 = f - q * hw;
      const int2 e = sorted[q];
      const int2 v = c2 == 0 ? make_int2(src[2 * e.x], src[2 * e.x + 1])
                             : make_int2(dslot[e.x * K + 2 * c2 - 2], dslot[e.x * K + 2 * c2 - 1]);
      reinterpret_cast<int2*>(p.meta + static_cast<int64_t>(e.y) * KW)[c2] = v;
    }
  } else {
    for (int f = tid; f < nvalid * KW; f += nthr) {
      const int q = f / KW, col = f - q * KW;
      const int2 e = sorted[q];
      const int v = col < 2 ? src[2 * e.x + col] : dslot[e.x * K + col - 2];
      p.meta[static_cast<int64_t>(e.y) * KW + col] = v;
    }
  }
}

// CTA 0's outputs of the non-expand layout: counts and aligned expert prefix
// (as in the expand layout; psum_s already scanned), tokens per rank and their
// exclusive prefix, rows.
__device__ void write_outputs_nonexpand(const LayoutParams& p, const int32_t* cnt_s,
                                        const int32_t* psum_s, const int32_t* prank,
                                        const int32_t* tpr) {
  const int E = p.num_experts, W = p.world_size;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    p.psum_expert[e] = psum_s[e];
    if (e < E) p.cnt[e] = cnt_s[e];
  }
  for (int r = threadIdx.x; r <= W; r += blockDim.x) {
    p.psum_rank[r] = prank[r];
    if (r < W) p.tok_per_rank[r] = tpr[r];
  }
  if (threadIdx.x == 0) *p.num_recv = prank[W];
}

// Shared-memory words of slots_nonexpand_tokens' scratch for tpb tokens.
__host__ __device__ constexpr int NonExpandScratchWords(int tpb, int K, int W) {
  return 2 * tpb * (K < W ? K : W) + (((tpb / 32) * W + 1) & ~1) + tpb * K + 2 * tpb;
}

template <int KC>
__global__ void __launch_bounds__(kSlotThreads, 1) ep_layout_slots_ne_kernel(LayoutParams p) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, W = p.world_size, C = p.num_chunks;
  const int RM = K < W ? K : W;
  extern __shared__ __align__(16) int32_t sm[];
  int2* sorted = reinterpret_cast<int2*>(sm);          // [TPC*RM]
  int32_t* woff = sm + 2 * kLayoutTPC * RM;            // [TPC/32][W]
  int32_t* dslot = woff + (kLayoutTPC / 32) * W;       // [TPC*K]
  int32_t* src = dslot + kLayoutTPC * K;               // [2*TPC]
  int32_t* prank = src + 2 * kLayoutTPC;               // [W+1] exclusive prefix of tokens per rank
  int32_t* tpr = prank + W + 1;                        // [W]   tokens per rank
  int32_t* rcl = tpr + W;                              // [W]   this chunk's tokens per rank
  int32_t* rbase = rcl + W;                            // [W]   first row of this chunk per rank
  int32_t* rcx = rbase + W;                            // [W+1] exclusive scan of rcl over ranks
  int32_t* warp_tot = rcx + W + 1;                     // [33]
  int32_t* cnt_s = warp_tot + 33;                      // [E]   (CTA 0)
  int32_t* psum_s = cnt_s + E;                         // [E+1] (CTA 0)

  const int c = blockIdx.x;
  const bool has_tokens = c < C;
  const int tid = threadIdx.x, warp = tid >> 5;
  allow_dependent_grids();   // the dispatch that follows may be scheduled now
  grid_dependency_wait();
  const int64_t row = static_cast<int64_t>(c) * (E + W);  // this chunk's table row
  for (int r = tid; r < W; r += kSlotThreads) {
    tpr[r] = p.col_total[E + r];
    if (has_tokens) {
      rcl[r] = p.chunk_hist[row + E + r];
      rbase[r] = p.chunk_off[row + E + r];
    }
  }
  __syncthreads();
  if (warp == 0) warp_scan64(tpr, W, prank);
  if (warp == 1 && has_tokens) warp_scan64(rcl, W, rcx);
  __syncthreads();
  for (int r = tid; r < W && has_tokens; r += kSlotThreads) rbase[r] += prank[r];

  if (c == 0) {
    for (int e = tid; e < E; e += kSlotThreads) cnt_s[e] = p.col_total[e];
    __syncthreads();
    expert_scans(cnt_s, p.alignment, psum_s, nullptr, nullptr, E, warp_tot);
    write_outputs_nonexpand(p, cnt_s, psum_s, prank, tpr);
  }
  if (has_tokens) {  // uniform per CTA
    __syncthreads();
    const int t0 = c * kLayoutTPC;
    const int ntok = min(p.num_tokens, t0 + kLayoutTPC) - t0;
    slots_nonexpand_tokens<KC>(p, t0, ntok, kLayoutTPC, rbase, rcx, nullptr, woff, dslot, src,
                               sorted);
  }
  fill_unreceived(p, nullptr, nullptr, prank[W], c, gridDim.x);
}

// ---------------------------------------------------------------- cluster (small batches)

// Words of shared memory of the cluster kernel for E experts, W ranks, top-k K
// and tpb tokens per CTA (the carve-up at the top of the kernel).
__host__ __device__ constexpr int ClusterSmemWords(int E, int W, int K, int tpb, bool ne) {
  const int EW = E + W;
  return (ne ? NonExpandScratchWords(tpb, K, W) : 0)      // non-expand scratch (first: int2)
         + 2 * tpb                                        // tmask (64-bit words)
         + kLayoutCountWarps * EW + 3 * EW + (EW & 1)     // whist, colcnt, tot, off (+ pad to even)
         + tpb * K                                        // ids
         + (ne ? 0 : 3 * tpb * K + 2 * tpb)               // loc, slots_s, sorted, src (expand)
         + 2 * (E + 1) + 33                               // psum_s, cx, warp_tot
         + (W + 1) + W + (W + 1)                          // prank, rbase, rcx
         + 4;                                             // misc
}

// Shared memory of one token range of the single-launch kernels (cluster and
// fused), carved out of `sm` for tpb tokens (ClusterSmemWords words).
struct RangeSmem {
  int2* sorted_ne;               // NE: [tpb*RM] (rank, token) rows in (rank, token) order
  int32_t* woff;                 // NE: [tpb/32][W]
  int32_t* dslot;                // NE: [tpb*K]
  int32_t* src_ne;               // NE: [2*tpb]
  unsigned long long* tmask;     // [tpb] (8-byte aligned: even offset)
  int32_t* whist;                // [NW][EW]
  int32_t* colcnt;               // [EW] this range's totals (read remotely by the cluster kernel)
  int32_t* tot;                  // [EW] totals over all ranges
  int32_t* off;                  // [EW] sum over the ranges before this one
  int32_t* ids;                  // [tpb*K]
  int32_t* loc;                  // expand: [tpb*K]
  int32_t* slots_s;              // expand: [tpb*K]
  int32_t* sorted;               // expand: [tpb*K]
  int32_t* src;                  // expand: [2*tpb]
  int32_t* psum_s;               // [E+1]
  int32_t* cx;                   // [E+1]
  int32_t* warp_tot;             // [33]
  int32_t* prank;                // [W+1]
  int32_t* rbase;                // [W]
  int32_t* rcx;                  // [W+1]
  int32_t* misc;                 // [4]
};

template <bool NE>
__device__ __forceinline__ RangeSmem carve_range_smem(int32_t* sm, int E, int W, int K, int tpb) {
  const int EW = E + W;
  RangeSmem r{};
  int32_t* base = sm;
  r.sorted_ne = reinterpret_cast<int2*>(sm);
  if constexpr (NE) {
    const int RM = K < W ? K : W;
    r.woff = sm + 2 * tpb * RM;
    r.dslot = r.woff + (((tpb / 32) * W + 1) & ~1);   // even: tmask below stays 8-byte aligned
    r.src_ne = r.dslot + tpb * K;
    base = r.src_ne + 2 * tpb;
  }
  r.tmask = reinterpret_cast<unsigned long long*>(base);
  base += 2 * tpb;
  r.whist = base;
  r.colcnt = r.whist + kLayoutCountWarps * EW;
  r.tot = r.colcnt + EW;
  r.off = r.tot + EW;
  r.ids = r.off + EW + (EW & 1);   // even offset: slots_s and src below are 8-byte aligned
  r.loc = r.ids + tpb * K;
  r.slots_s = r.loc + (NE ? 0 : tpb * K);
  r.sorted = r.slots_s + (NE ? 0 : tpb * K);
  r.src = r.sorted + (NE ? 0 : tpb * K);
  r.psum_s = r.src + (NE ? 0 : 2 * tpb);
  r.cx = r.psum_s + E + 1;
  r.warp_tot = r.cx + E + 1;
  r.prank = r.warp_tot + 33;
  r.rbase = r.prank + W + 1;
  r.rcx = r.rbase + W;
  r.misc = r.rcx + W + 1;
  return r;
}

// Local half of an expand range's slot pass (E <= kWarpScanMax), which needs nothing from the
// other ranges: cx = exclusive scan over experts of the range's counts, the
// entries ordered by (expert, rank) (sorted[cx[e] + loc[i]] = i) and each
// token's {t / T, t mod T}.  The fused kernel runs it between arriving at its
// grid barrier and waiting on it, while the other ranges are still counting.
// All threads call, after a barrier that makes colcnt and loc visible.
template <int KC>
__device__ void presort_expand_range(const LayoutParams& p, const RangeSmem& r, int t0, int ntok) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, T = p.max_tok_per_rank;
  // every warp but the last (whose lane 0 is arriving at the grid barrier, an
  // atomic round trip through L2) takes part; they meet at named barrier 1
  const int nthr = blockDim.x - 32, nent = ntok * K;
  if (threadIdx.x >= nthr) return;
  if ((threadIdx.x >> 5) == 0) warp_exclusive_scan(r.colcnt, E, 1, r.cx);   // E <= kWarpScanMax
  asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
  for (int i = threadIdx.x; i < nent; i += nthr) {
    const int e = r.ids[i];
    if (e >= 0) r.sorted[r.cx[e] + r.loc[i]] = i;
  }
  for (int tl = threadIdx.x; tl < ntok; tl += nthr) {
    const int t = t0 + tl, q = t / T;
    r.src[2 * tl] = q;
    r.src[2 * tl + 1] = t - q * T;
  }
}

// The rest of an expand range (E <= kWarpScanMax) once presort_expand_range has
// run and r.tot (totals over all ranges), r.off (the sum over the ranges
// before this one) and r.psum_s (the aligned prefix over experts) are known:
// CTA 0's outputs, the slots, the metadata rows and this range's share of the
// rows that receive nothing.  All threads call, after a barrier that makes
// them visible.
template <int KC>
__device__ void finish_expand_presorted(const LayoutParams& p, const RangeSmem& r, int me, int nranges,
                                        int t0, int ntok) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts;
  const int nthr = blockDim.x, nent = ntok * K;
  if (me == 0) write_outputs_expand(p, r.tot, r.psum_s, r.tot + E);
  int32_t* ds = p.dst_slot + static_cast<int64_t>(t0) * K;
  for (int i = threadIdx.x; i < nent; i += nthr) {
    const int e = r.ids[i];
    const int slot = e >= 0 ? r.psum_s[e] + r.off[e] + r.loc[i] : -1;
    ds[i] = slot;
    r.slots_s[i] = slot;
  }
  __syncthreads();
  write_metadata_rows<KC>(p, r.cx[E], r.sorted, r.slots_s, r.src);
  fill_unreceived(p, r.psum_s, r.tot, r.psum_s[E], me, nranges);
}

// The rest of a range once r.tot (totals over all ranges) and r.off (the sum
// over the ranges before this one) are known, for range `me` of `nranges`:
// prefix sums, CTA 0's outputs, slots, metadata and this range's share of the
// rows that receive nothing.  All threads call, after a barrier that makes
// tot and off visible.
template <int KC, bool NE>
__device__ void finish_range(const LayoutParams& p, const RangeSmem& r, int me, int nranges, int t0,
                             int ntok, int tpb) {
  const int E = p.num_experts, W = p.world_size;
  if constexpr (!NE) {
    expert_scans(r.tot, p.alignment, r.psum_s, r.colcnt, r.cx, E, r.warp_tot);
    if (me == 0) write_outputs_expand(p, r.tot, r.psum_s, r.tot + E);
    slots_expand_tokens<KC>(p, t0, ntok, r.psum_s, r.off, r.cx, r.loc, r.ids, r.slots_s, r.sorted, r.src);
    fill_unreceived(p, r.psum_s, r.tot, r.psum_s[E], me, nranges);
  } else {
    // rank prefix, this range's rank scan and (range 0, few experts) the expert
    // prefix on three warps behind one barrier
    const int warp = threadIdx.x >> 5;
    const bool warp_psum = E <= kWarpScanMax;
    if (warp == 0) warp_scan64(r.tot + E, W, r.prank);
    else if (warp == 1) warp_scan64(r.colcnt + E, W, r.rcx);
    else if (warp == 2 && me == 0 && warp_psum) warp_exclusive_scan(r.tot, E, p.alignment, r.psum_s);
    __syncthreads();
    if (me == 0 && !warp_psum) block_exclusive_scan(r.tot, E, p.alignment, r.psum_s, r.warp_tot);
    for (int q = threadIdx.x; q < W; q += blockDim.x) r.rbase[q] = r.prank[q] + r.off[E + q];
    if (me == 0) write_outputs_nonexpand(p, r.tot, r.psum_s, r.prank, r.tot + E);
    // rbase is read after slots_nonexpand_tokens' first barrier
    slots_nonexpand_tokens<KC>(p, t0, ntok, tpb, r.rbase, r.rcx, r.ids, r.woff, r.dslot, r.src_ne,
                               r.sorted_ne);
    fill_unreceived(p, nullptr, nullptr, r.prank[W], me, nranges);
  }
}

template <int KC, bool NE>
__global__ void __launch_bounds__(kClusterThreads, 1) ep_layout_cluster_kernel(LayoutParams p, int tpb) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, W = p.world_size, EW = E + W;
  extern __shared__ __align__(16) int32_t sm[];
  const RangeSmem r = carve_range_smem<NE>(sm, E, W, K, tpb);

  const uint32_t me = cluster_ctarank(), ncta = cluster_nctarank();
  allow_dependent_grids();   // the dispatch that follows may be scheduled now
  const int t0 = static_cast<int>(me) * tpb;
  const int ntok = max(0, min(p.num_tokens, t0 + tpb) - t0);
  CountRegs<KC> regs;
  count_tokens<KC>(p, t0, ntok, r.whist, r.tmask, r.colcnt, r.ids, regs);

  // every CTA's column totals are complete: gather the cluster's totals and
  // this CTA's offsets from the other CTAs' shared memory.  (The CTAs of a
  // cluster finish counting together, so there is no wait here to hide the
  // range's local work behind, as the fused kernel does: measured slower.)
  cluster_arrive();
  cluster_wait();
  if constexpr (!NE) write_range_ranks<KC>(ntok, K, r.whist, EW, regs, r.loc);
  int own_total = 0, own_count = 0;   // thread e's expert column: cluster total, own count
  for (int j = threadIdx.x; j < EW; j += kClusterThreads) {
    int v[kClusterCtas];
#pragma unroll
    for (int b = 0; b < kClusterCtas; ++b)  // all remote loads in flight together
      v[b] = b >= static_cast<int>(ncta) ? 0
           : b == static_cast<int>(me)   ? r.colcnt[j]
                                         : ld_cluster_shared(r.colcnt + j, static_cast<uint32_t>(b));
    int t = 0, o = 0;
#pragma unroll
    for (int b = 0; b < kClusterCtas; ++b) {
      o += b < static_cast<int>(me) ? v[b] : 0;
      t += v[b];
    }
    r.tot[j] = t;
    r.off[j] = o;
    if (j == static_cast<int>(threadIdx.x)) {
      own_total = t;
      own_count = r.colcnt[j];
    }
  }
  cluster_arrive_relaxed();  // this CTA is done reading remote shared memory
  if (!NE && E <= kWarpScanMax) {
    // both scans over experts from the threads' own values in registers:
    // psum_s (aligned cluster totals) and cx (this range's counts)
    dual_block_scan(own_total, own_count, p.alignment, E, r.psum_s, r.cx, r.warp_tot);
    if (me == 0) write_outputs_expand(p, r.tot, r.psum_s, r.tot + E);
    slots_expand_tokens<KC>(p, t0, ntok, r.psum_s, r.off, r.cx, r.loc, r.ids, r.slots_s, r.sorted, r.src);
    fill_unreceived(p, r.psum_s, r.tot, r.psum_s[E], static_cast<int>(me), static_cast<int>(ncta));
  } else {
    __syncthreads();
    finish_range<KC, NE>(p, r, static_cast<int>(me), static_cast<int>(ncta), t0, ntok, tpb);
  }
  // keep this CTA's shared memory until every CTA has finished reading it
  cluster_wait();
}

// ---------------------------------------------------------------- fused (one launch, mid-size batches)

// Global-memory exchange of the single-launch layout for batches beyond one
// cluster: a cooperative grid (every CTA resident at once), one token range
// per CTA.  Each CTA counts its range exactly as the cluster kernel does, then
// publishes its column totals twice: as a row of 16-bit counts in the range
// table [C][EW8], and, by atomic adds, into the row of its superchunk (the
// kFusedSuper consecutive ranges it belongs to) of the superchunk table
// [S][EW8].  After one grid barrier a CTA has everything in L2: the totals
// (sum of the S superchunk rows), and its offset in each column (the
// superchunk rows before its own plus the range rows of its superchunk before
// it): at most S + kFusedSuper - 1 values per column instead of one per
// range.  Its ranks are still in registers and its ids in shared memory, so
// it goes straight on to slots and metadata.
//
// The superchunk table is double-buffered by launch parity: a launch adds
// into buffer (launches so far & 1) and zeroes the other one for the next
// launch.
// Integer adds commute, so the sums do not depend on the order of the atomics.

constexpr int kFusedSuper = 16;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* a) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* a) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ int4 ld_cg_v4(const int4* a) {
  int4 v;
  asm volatile("ld.global.cg.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(a));
  return v;
}

// Words of the fused kernel's staging area (after the range's shared memory):
// S superchunk rows of EW8 int32 and up to kFusedSuper - 1 range rows of EW8
// 16-bit counts.
__host__ __device__ constexpr int FusedStageWords(int S, int EW8) {
  return S * EW8 + (kFusedSuper / 2) * EW8;
}

// Barrier over the nctas CTAs of a cooperative grid, in two halves so that a
// CTA can do local work between arriving and waiting; every thread of every
// CTA calls both.  bar[0] counts arrivals and only grows (modulo 2^32); bar[1]
// is its value when this launch began and bar[2] the number of launches so
// far, both read by each CTA before it arrives (they change only after every
// CTA has arrived: the last arrival sets them for the next launch).  A CTA
// arrives with one atomic add and waits (acquire) until the counter reaches
// bar[1] + nctas.  The state stays consistent for the next launch whatever
// the grid size, also when a wait gives up: every CTA arrives exactly once.
struct GridArrival {
  unsigned target;  // counter value once every CTA has arrived
  bool last;        // this CTA arrived last (thread 0's value)
};

// The arriving (and later waiting) thread: lane 0 of the CTA's last warp, so
// that the fence and the atomic round trip of the arrival stall no warp that
// the local work between the halves uses.
__device__ __forceinline__ bool is_arriving_thread() { return threadIdx.x == blockDim.x - 32; }

__device__ GridArrival fused_grid_arrive(unsigned* bar, unsigned base, unsigned gen, unsigned nctas) {
  __syncthreads();  // this CTA's writes are done
  GridArrival a{base + nctas, false};
  if (is_arriving_thread()) {
    __threadfence();  // ... and visible at gpu scope before the arrival
    const unsigned arrival = atomicAdd(bar, 1u);
    if (arrival == a.target - 1u) {
      bar[1] = a.target;  // the next launch's base and count (read after this kernel)
      bar[2] = gen + 1u;
      a.last = true;
      __threadfence();  // order this CTA's later reads after every arrival it observed
    }
  }
  return a;
}

// The waiting half, bounded by wait_ns (the deadline is checked before each
// test, so wait_ns = 0 gives up at once unless this CTA arrived last); returns
// false, for every thread of the CTA, when this CTA's wait gave up.
__device__ bool fused_grid_wait(const unsigned* bar, const GridArrival& a, uint64_t wait_ns,
                                int32_t* ok_s) {
  if (is_arriving_thread()) {
    int ok = 1;
    if (!a.last) {
      const uint64_t t0 = global_ns();
      for (;;) {
        if (global_ns() - t0 >= wait_ns) {
          ok = 0;
          break;
        }
        if (static_cast<int>(ld_acquire_gpu(bar) - a.target) >= 0) break;
      }
    }
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

template <int KC, bool NE>
__global__ void __launch_bounds__(kCountThreads, 2) ep_layout_fused_kernel(LayoutParams p) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, W = p.world_size, EW = E + W;
  const int EW8 = (EW + 7) & ~7;
  const int tpb = p.fused_tpb;
  extern __shared__ __align__(16) int32_t sm[];
  const RangeSmem r = carve_range_smem<NE>(sm, E, W, K, tpb);
  const int c = blockIdx.x, C = gridDim.x;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int t0 = c * tpb;
  const int ntok = max(0, min(p.num_tokens, t0 + tpb) - t0);
  if (tid == 0) {
    r.misc[0] = static_cast<int32_t>(ld_relaxed_gpu(p.fused_bar + 1));   // barrier base
    r.misc[2] = static_cast<int32_t>(ld_relaxed_gpu(p.fused_bar + 2));   // launches so far
  }
  allow_dependent_grids();   // the dispatch that follows may be scheduled now
  CountRegs<KC> regs;
  count_tokens<KC>(p, t0, ntok, r.whist, r.tmask, r.colcnt, r.ids, regs);
  __syncthreads();
  if constexpr (!NE) write_range_ranks<KC>(ntok, K, r.whist, EW, regs, r.loc);

  // publish this range's column totals
  const unsigned base = static_cast<unsigned>(r.misc[0]);
  const unsigned gen = static_cast<unsigned>(r.misc[2]);
  const int64_t sup_words = static_cast<int64_t>(p.fused_super_rows) * EW8;
  int32_t* sup = p.fused_super + (gen & 1u) * sup_words;
  int32_t* sup_next = p.fused_super + ((gen & 1u) ^ 1u) * sup_words;
  // (CTAs past the last range of tokens only fill padding: nothing to publish,
  // and no range reads their rows)
  const int CR = (p.num_tokens + tpb - 1) / tpb;
  const int s = c / kFusedSuper;
  if (c < CR) {
    uint32_t* row = reinterpret_cast<uint32_t*>(p.fused_rows + static_cast<int64_t>(c) * EW8);
    for (int j2 = tid; j2 < EW8 / 2; j2 += nthr) {
      const int j = 2 * j2;
      const uint32_t lo = j < EW ? static_cast<uint32_t>(r.colcnt[j]) : 0u;
      const uint32_t hi = j + 1 < EW ? static_cast<uint32_t>(r.colcnt[j + 1]) : 0u;
      row[j2] = lo | (hi << 16);
    }
    for (int j = tid; j < EW; j += nthr) {
      const int v = r.colcnt[j];
      if (v) atomicAdd(sup + static_cast<int64_t>(s) * EW8 + j, v);
    }
  }
  for (int64_t f = static_cast<int64_t>(c) * nthr + tid; f < sup_words; f += static_cast<int64_t>(C) * nthr)
    sup_next[f] = 0;  // the next launch's buffer

  // the range's local work runs between arriving and waiting (up to 512 experts)
  const bool presort = !NE && E <= kWarpScanMax;
  const GridArrival arrival = fused_grid_arrive(p.fused_bar, base, gen, static_cast<unsigned>(C));
  if (presort) presort_expand_range<KC>(p, r, t0, ntok);
  if (!fused_grid_wait(p.fused_bar, arrival, p.wait_ns, r.misc + 1)) {
    if (tid == 0) atomicOr(p.err, kErrTimeout);
    return;  // uniform per CTA
  }

  // totals and this range's offsets.  The superchunk rows and the range rows
  // of this superchunk before this range were written by other CTAs in this
  // launch: they are staged in shared memory with 16-byte .cg loads (L2, never
  // the non-coherent path), all in flight at once, then summed per column.
  const int S = (CR + kFusedSuper - 1) / kFusedSuper;
  const int c_lo = s * kFusedSuper;
  const int nrow = max(0, (c < CR ? c : CR) - c_lo);
  int32_t* st_sup = sm + ((ClusterSmemWords(E, W, K, tpb, NE) + 3) & ~3);     // [S][EW8], 16-byte aligned
  const uint16_t* st_rows = reinterpret_cast<const uint16_t*>(st_sup + S * EW8);   // [nrow][EW8]
  {
    const int n_sup4 = S * EW8 / 4, n4 = n_sup4 + nrow * EW8 / 8;
    const int4* gs = reinterpret_cast<const int4*>(sup);
    const int4* gr = reinterpret_cast<const int4*>(p.fused_rows + static_cast<int64_t>(c_lo) * EW8);
    int4* st4 = reinterpret_cast<int4*>(st_sup);
    for (int f0 = tid; f0 < n4; f0 += 4 * nthr) {
      int4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = f0 + u * nthr;
        if (f < n4) a[u] = ld_cg_v4(f < n_sup4 ? gs + f : gr + (f - n_sup4));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = f0 + u * nthr;
        if (f < n4) st4[f] = a[u];   // the range rows follow the superchunk rows
      }
    }
  }
  __syncthreads();
  int own_total = 0;   // thread e's expert column total (e < E)
  for (int j = tid; j < EW; j += nthr) {
    int pre = 0, all = 0;
    for (int s2 = 0; s2 < S; ++s2) {
      const int v = st_sup[s2 * EW8 + j];
      all += v;
      pre += s2 < s ? v : 0;
    }
    for (int q = 0; q < nrow; ++q) pre += st_rows[q * EW8 + j];
    r.tot[j] = all;
    r.off[j] = pre;
    if (j == tid) own_total = all;
  }
  if (presort) {
    // the aligned exclusive prefix over experts straight from the threads'
    // own totals (thread e holds expert e; E <= kWarpScanMax = blockDim.x), a
    // block scan instead of a single warp's pass over E values in shared memory
    const int A = p.alignment;
    const bool p2 = (A & (A - 1)) == 0;
    const int v = tid < E ? (p2 ? align_to<true>(own_total, A) : align_to<false>(own_total, A)) : 0;
    const int lane = tid & 31, warp = tid >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) r.warp_tot[warp] = incl;
    __syncthreads();   // also makes tot and off visible
    int base = 0;
    for (int w = 0; w < warp; ++w) base += r.warp_tot[w];
    if (tid < E) r.psum_s[tid] = base + incl - v;
    if (tid == E - 1) r.psum_s[E] = base + incl;
    __syncthreads();
    finish_expand_presorted<KC>(p, r, c, C, t0, ntok);
  } else {
    __syncthreads();
    finish_range<KC, NE>(p, r, c, C, t0, ntok, tpb);
  }
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

size_t count_smem(int, int cols) {
  return sizeof(int32_t) * static_cast<size_t>(CountSmemWords(cols, kLayoutTPC));
}

size_t slots_smem(int E, int topk) {
  return sizeof(int32_t) * (5 * static_cast<size_t>(E) + 2 + 34 + 2 * kLayoutTPC * topk +
                            2 * kLayoutTPC);
}

size_t slots_ne_smem(int E, int W, int topk) {
  return sizeof(int32_t) * (static_cast<size_t>(NonExpandScratchWords(kLayoutTPC, topk, W)) +
                            5 * static_cast<size_t>(W) + 2 + 33 + 2 * static_cast<size_t>(E) + 1);
}

size_t cluster_smem(int E, int W, int topk, int tpb, bool ne) {
  return sizeof(int32_t) * static_cast<size_t>(ClusterSmemWords(E, W, topk, tpb, ne));
}

// Tokens per CTA of the cluster kernel for this launch, or 0 when the batch is
// served by the three-launch path.
int cluster_tpb(const LayoutParams& p, const LaunchGeom& g) {
  if (!g.cluster_ok || p.num_tokens <= 0 || p.num_tokens > kClusterCtas * kClusterMaxTPB) return 0;
  const int64_t fill = p.rcap - static_cast<int64_t>(p.num_tokens) * p.topk;
  if (fill > kClusterMaxFillRows) return 0;
  const int tpb = p.num_tokens <= kClusterCtas * kLayoutTPC ? kLayoutTPC : kClusterMaxTPB;
  if (cluster_smem(p.num_experts, p.world_size, p.topk, tpb, p.no_expand != 0) > kClusterMaxSmem)
    return 0;
  return tpb;
}

template <int KC, bool NE>
cudaError_t launch_cluster(const LayoutParams& p, int tpb, cudaStream_t s) {
  const int ncta = (p.num_tokens + tpb - 1) / tpb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncta);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = cluster_smem(p.num_experts, p.world_size, p.topk, tpb, NE);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ncta);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ep_layout_cluster_kernel<KC, NE>, p, tpb);
}

// Rows of -1 one CTA of the fused kernel fills at most; batches with more
// padding than their ranges cover get extra CTAs with no tokens.
constexpr int64_t kFusedFillPerCta = 8192;

// Geometry of the fused kernel for this launch (tpb = 0: it does not serve
// it -- no fused state (the allocation-free entry point), switched off, more
// ranges than the state holds, more CTAs than a cooperative grid keeps
// resident, or more
// shared memory than the cluster kernel's limit).  The grid has one CTA per
// range of tpb tokens, and at least one per kFusedFillPerCta rows to fill.
struct FusedGeom {
  int tpb = 0;
  int ctas = 0;
  size_t smem = 0;
};

// Dynamic shared memory of a fused launch: the range's share plus the staging
// area for S superchunk rows.
size_t fused_smem(int E, int W, int K, int tpb, bool ne, int S) {
  const int EW8 = (E + W + 7) & ~7;
  return sizeof(int32_t) * (((static_cast<size_t>(ClusterSmemWords(E, W, K, tpb, ne)) + 3) & ~static_cast<size_t>(3)) +
                            static_cast<size_t>(FusedStageWords(S, EW8)));
}

FusedGeom fused_geom(const LayoutParams& p, const LaunchGeom& g) {
  FusedGeom f;
  if (p.fused_bar == nullptr || g.fused_blocks_per_sm <= 0 || p.num_tokens <= 0) return f;
  // Unless pinned: the fewest tokens per CTA (a multiple of 32, from kLayoutTPC
  // to kClusterMaxTPB) that give at most one range per SM, so that the
  // metadata stores of the tail phase are spread over as many SMs as possible
  // without two ranges sharing one.  Measured at 32768 tokens on 152 SMs (cold):
  // 256 ranges of 128 tokens 18.4 us, 128 of 256 18.4 us, 147 of 224 17.2 us,
  // 171 of 192 20.5 us.
  int tpb = g.fused_tpb;
  if (tpb == 0) {
    const int per_sm = (p.num_tokens + g.num_sms - 1) / g.num_sms;
    tpb = (per_sm + 31) / 32 * 32;
    tpb = tpb < kLayoutTPC ? kLayoutTPC : (tpb > kClusterMaxTPB ? kClusterMaxTPB : tpb);
  }
  const int64_t ranges = (p.num_tokens + tpb - 1) / tpb;
  const int64_t fill = p.rcap - static_cast<int64_t>(p.num_tokens) * p.topk;
  const int64_t fill_ctas = (fill + kFusedFillPerCta - 1) / kFusedFillPerCta;
  const int64_t ctas = ranges > fill_ctas ? ranges : fill_ctas;
  if (ranges > p.fused_max_ranges || ctas > static_cast<int64_t>(g.fused_blocks_per_sm) * g.num_sms)
    return f;
  const int S = static_cast<int>((ranges + kFusedSuper - 1) / kFusedSuper);
  if (S > g.fused_max_super) return f;   // beyond the staging the occupancy was computed for
  const size_t smem = fused_smem(p.num_experts, p.world_size, p.topk, tpb, p.no_expand != 0, S);
  if (smem > kClusterMaxSmem) return f;
  f.tpb = tpb;
  f.ctas = static_cast<int>(ctas);
  f.smem = smem;
  return f;
}

template <int KC, bool NE>
cudaError_t launch_fused(LayoutParams p, const FusedGeom& f, cudaStream_t s) {
  p.fused_tpb = f.tpb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(f.ctas));
  cfg.blockDim = dim3(kCountThreads);
  cfg.dynamicSmemBytes = f.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once: the grid barrier's premise
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ep_layout_fused_kernel<KC, NE>, p);
}

template <int KC, bool NE>
cudaError_t launch_layout(const LayoutParams& p, const LaunchGeom& g, cudaStream_t s) {
  const int tpb = cluster_tpb(p, g);
  if (tpb > 0) return launch_cluster<KC, NE>(p, tpb, s);
  const FusedGeom f = fused_geom(p, g);
  if (f.tpb > 0) return launch_fused<KC, NE>(p, f, s);
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
// handles with different shapes never lower them for each other.  The cluster
// kernel's limit is kClusterMaxSmem (larger requests take the three-launch
// path); it is used only if a cluster of kClusterCtas CTAs with that much
// shared memory can be resident, and not when EP_GB300_LAYOUT_CLUSTER=0.
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
  g->cluster_ok = 0;
  g->fused_blocks_per_sm = 0;
  e = cudaFuncSetAttribute(ep_layout_cluster_kernel<KC, NE>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kClusterMaxSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ep_layout_fused_kernel<KC, NE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kClusterMaxSmem));
  if (e != cudaSuccess) return e;
  // tokens per CTA of the fused kernel pinned by EP_GB300_LAYOUT_FUSED_TPB (a
  // multiple of 32 from 64 to 256); 0: chosen per launch from the batch size
  const char* tenv = std::getenv("EP_GB300_LAYOUT_FUSED_TPB");
  const int t = tenv ? std::atoi(tenv) : 0;
  g->fused_tpb = (t >= 64 && t <= kClusterMaxTPB && t % 32 == 0) ? t : 0;
  const char* fenv = std::getenv("EP_GB300_LAYOUT_FUSED");
  // superchunk rows staged at most: enough for two resident CTAs per SM
  g->fused_max_super = (2 * g->num_sms + kFusedSuper - 1) / kFusedSuper;
  if (g->layout_experts > 0 && !(fenv != nullptr && fenv[0] == '0')) {
    // resident CTAs per SM at the largest range and staging the fused kernel takes
    const size_t smem = fused_smem(g->layout_experts, g->layout_world, kmax, 256, NE, g->fused_max_super);
    int n = 0;
    if (smem <= kClusterMaxSmem &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ep_layout_fused_kernel<KC, NE>, kCountThreads,
                                                      smem) == cudaSuccess)
      g->fused_blocks_per_sm = n;
    cudaGetLastError();
  }
  const char* env = std::getenv("EP_GB300_LAYOUT_CLUSTER");
  if (env != nullptr && env[0] == '0') return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kClusterCtas);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = kClusterMaxSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, ep_layout_cluster_kernel<KC, NE>, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();  // not schedulable as a cluster here: the three-launch path serves
    return cudaSuccess;
  }
  g->cluster_ok = clusters > 0 ? 1 : 0;
  return cudaSuccess;
}

}  // namespace

LayoutPath LayoutPathOf(const LayoutParams& p, const LaunchGeom& g) {
  if (cluster_tpb(p, g) > 0) return LayoutPath::kCluster;
  if (fused_geom(p, g).tpb > 0) return LayoutPath::kFused;
  return LayoutPath::kLaunches;
}

int64_t LayoutScratchInts(int max_chunks, int columns) {
  return 3LL * columns * (max_chunks > 0 ? max_chunks : 1) + columns;
}

void BindLayoutScratch(LayoutParams* p, int32_t* base, int max_chunks, int columns) {
  const int64_t cap = max_chunks > 0 ? max_chunks : 1;
  p->chunk_hist = base;
  p->chunk_hist_cols = base + static_cast<int64_t>(columns) * cap;
  p->chunk_off = p->chunk_hist_cols + static_cast<int64_t>(columns) * cap;
  p->col_total = p->chunk_off + static_cast<int64_t>(columns) * cap;
}

namespace {
constexpr int kFusedMaxRanges = 1024;   // above any cooperative grid of 512-thread CTAs on one GPU
int fused_ranges(int max_chunks) {
  const int r = 2 * (max_chunks > 0 ? max_chunks : 1);   // ranges of 64 tokens at the smallest
  return r < kFusedMaxRanges ? r : kFusedMaxRanges;
}
}  // namespace

int64_t LayoutFusedStateInts(int max_chunks, int columns) {
  const int64_t R = fused_ranges(max_chunks);
  const int64_t S = (R + kFusedSuper - 1) / kFusedSuper;
  const int64_t EW8 = (columns + 7) & ~7;
  const int64_t rows_words = ((R * EW8 + 1) / 2 + 63) & ~int64_t{63};
  return 64 + 2 * S * EW8 + rows_words;
}

void BindLayoutFusedState(LayoutParams* p, int32_t* base, int max_chunks, int columns) {
  const int R = fused_ranges(max_chunks);
  const int S = (R + kFusedSuper - 1) / kFusedSuper;
  const int64_t EW8 = (columns + 7) & ~7;
  p->fused_bar = reinterpret_cast<uint32_t*>(base);
  p->fused_super = base + 64;
  p->fused_rows = reinterpret_cast<uint16_t*>(base + 64 + 2 * S * EW8);
  p->fused_super_rows = S;
  p->fused_max_ranges = R;
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
