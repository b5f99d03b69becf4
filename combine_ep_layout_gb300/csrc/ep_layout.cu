// ep_layout.cu -- layout of the routing: per-expert / per-rank histograms,
// aligned exclusive prefix sums, deterministic destination slots and
// recv_src_metadata (EPHandle fields of "DeepEP overall architecture
// analysis"; the counting role of its "notify warps" in the Dispatch data flow
// figure).
//
// Rows of one expert are ordered by the flat index t*K+k, so the slot of an
// entry is psum_expert[e] + (number of earlier entries routed to e): a stable
// counting sort.  Three launches, no device-side waiting:
//
//   count  one CTA per chunk of kLayoutTPC tokens.  Each warp histograms a
//          contiguous run of the chunk's entries in shared memory, combining
//          lanes that carry the same expert with __match_any_sync (one update
//          per distinct expert per 32 entries, which keeps hot experts of a
//          skewed routing from serialising).  An exclusive scan across the
//          warps gives each warp its start per expert; a second pass over the
//          same entries gives each entry its stable rank within the chunk.
//          The chunk's column totals (E experts + W ranks) go to a
//          column-major [E+W][C] table.
//   spine  one warp per column: exclusive scan over the C chunks.
//   slots  each CTA rebuilds the aligned exclusive prefix over experts from
//          the column totals (E values, cheaper than another launch), then
//          turns every entry's in-chunk rank into its slot and writes the
//          metadata rows; extra CTAs write -1 into every row that receives
//          nothing.
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

constexpr int kCountThreads = kLayoutCountWarps * 32;
constexpr int kSpineWarps = 8;
constexpr int kSlotThreads = kLayoutTPC;  // one token per thread

__device__ __forceinline__ int expert_of(int64_t v, int E) {
  return (v >= 0 && v < E) ? static_cast<int>(v) : -1;
}

template <int KC>
__global__ void __launch_bounds__(kCountThreads) ep_layout_count_kernel(LayoutParams p) {
  constexpr int NW = kLayoutCountWarps;
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts;
  const int EW = E + p.world_size;
  const int C = p.num_chunks;
  extern __shared__ int32_t whist[];  // [NW][EW] per-warp counts, then per-warp starts

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int t0 = c * kLayoutTPC;
  const int t1 = min(p.num_tokens, t0 + kLayoutTPC);
  const int nent = (t1 - t0) * K;
  const int64_t* topk = p.topk_idx + static_cast<int64_t>(t0) * K;

  for (int i = tid; i < NW * EW; i += kCountThreads) whist[i] = 0;
  __syncthreads();

  // contiguous run of entries per warp, whole 32-entry batches
  const int per_warp = (((nent + NW - 1) / NW) + 31) & ~31;
  const int wbeg = warp * per_warp;
  const int wend = min(nent, wbeg + per_warp);
  int32_t* wh = whist + warp * EW;

  bool bad = false;
  for (int i = wbeg; i < wend; i += 32) {
    const int idx = i + lane;
    int e = -1;
    if (idx < wend) {
      const int64_t v = topk[idx];
      e = expert_of(v, E);
      bad |= (e < 0 && v != -1);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
    __syncwarp();
  }

  // tokens that touch each rank (a token counts once per rank)
  const int Epr = p.num_expert_per_rank;
  for (int t = t0 + tid; t < t1; t += kCountThreads) {
    uint64_t mask = 0;
    const int64_t* row = p.topk_idx + static_cast<int64_t>(t) * K;
    for (int k = 0; k < K; ++k) {
      const int e = expert_of(row[k], E);
      if (e >= 0) mask |= 1ull << (e / Epr);
    }
    while (mask) {
      const int r = __ffsll(static_cast<long long>(mask)) - 1;
      mask &= mask - 1;
      atomicAdd(&whist[E + r], 1);
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

  // stable rank of each entry within the chunk
  int32_t* local = p.dst_slot + static_cast<int64_t>(t0) * K;
  for (int i = wbeg; i < wend; i += 32) {
    const int idx = i + lane;
    const int e = idx < wend ? expert_of(topk[idx], E) : -1;
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

// One warp per column j of the [E+W][C] table: exclusive scan over chunks.
__global__ void __launch_bounds__(kSpineWarps * 32) ep_layout_spine_kernel(LayoutParams p) {
  const int EW = p.num_experts + p.world_size;
  const int C = p.num_chunks;
  const int j = blockIdx.x * kSpineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= EW) return;
  const int32_t* in = p.chunk_hist + static_cast<int64_t>(j) * C;
  int32_t* out = p.chunk_off + static_cast<int64_t>(j) * C;
  const int V = (C + 31) / 32;  // a contiguous run of chunks per lane
  const int cbeg = min(C, lane * V), cend = min(C, cbeg + V);
  int sum = 0;
  for (int c = cbeg; c < cend; ++c) sum += in[c];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;
  for (int c = cbeg; c < cend; ++c) {
    const int v = in[c];
    out[c] = run;
    run += v;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) p.col_total[j] = total;
}

// Block-wide exclusive scan of align(cnt[e]) for e in [0, E) into psum[0..E].
__device__ void aligned_exclusive_scan(const int32_t* __restrict__ cnt, int E, int A,
                                       int32_t* psum, int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  const int V = (E + nthr - 1) / nthr;
  const int beg = min(E, tid * V), end = min(E, beg + V);
  int sum = 0;
  for (int e = beg; e < end; ++e) sum += (cnt[e] + A - 1) / A * A;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < nwarp ? warp_tot[lane] : 0;
    int s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nwarp) warp_tot[lane] = s - v;  // exclusive warp offsets
    if (lane == nwarp - 1) warp_tot[32] = s;  // grand total
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - sum;
  for (int e = beg; e < end; ++e) {
    psum[e] = run;
    run += (cnt[e] + A - 1) / A * A;
  }
  if (tid == 0) psum[E] = warp_tot[32];
  __syncthreads();
}

template <int KC>
__global__ void __launch_bounds__(kSlotThreads) ep_layout_slots_kernel(LayoutParams p) {
  const int K = KC ? KC : p.topk;
  const int E = p.num_experts, W = p.world_size, C = p.num_chunks;
  const int Epr = p.num_expert_per_rank, T = p.max_tok_per_rank;
  extern __shared__ int32_t sm[];
  int32_t* cnt_s = sm;               // [E]
  int32_t* psum_s = sm + E;          // [E+1]
  int32_t* warp_tot = psum_s + E + 1;  // [33]

  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = p.col_total[e];
  __syncthreads();
  aligned_exclusive_scan(cnt_s, E, p.alignment, psum_s, warp_tot);

  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      p.psum_expert[e] = psum_s[e];
      if (e < E) p.cnt[e] = cnt_s[e];
    }
    for (int r = threadIdx.x; r <= W; r += blockDim.x) {
      p.psum_rank[r] = psum_s[r * Epr];
      if (r < W) p.tok_per_rank[r] = p.col_total[E + r];
    }
    if (threadIdx.x == 0) *p.num_recv = psum_s[E];
  }

  const int KW = K + 2;  // metadata row width
  if (static_cast<int>(blockIdx.x) < C) {
    const int c = blockIdx.x;
    const int t = c * kLayoutTPC + threadIdx.x;
    if (t >= p.num_tokens) return;
    int32_t slot[KC ? KC : kMaxTopk];
    const int64_t* row = p.topk_idx + static_cast<int64_t>(t) * K;
    int32_t* ds = p.dst_slot + static_cast<int64_t>(t) * K;
#pragma unroll
    for (int k = 0; k < (KC ? KC : kMaxTopk); ++k) {
      if (k < K) {
        const int e = expert_of(row[k], E);
        const int loc = ds[k];
        slot[k] = e >= 0 ? psum_s[e] + p.chunk_off[static_cast<int64_t>(e) * C + c] + loc : -1;
      }
    }
#pragma unroll
    for (int k = 0; k < (KC ? KC : kMaxTopk); ++k)
      if (k < K) ds[k] = slot[k];
    const int src_rank = t / T, src_local = t - src_rank * T;
#pragma unroll
    for (int k = 0; k < (KC ? KC : kMaxTopk); ++k) {
      if (k >= K || slot[k] < 0) continue;
      int32_t* m = p.meta + static_cast<int64_t>(slot[k]) * KW;
      if ((KW & 1) == 0) {  // 8-byte aligned rows: paired stores
        int2* m2 = reinterpret_cast<int2*>(m);
        m2[0] = make_int2(src_rank, src_local);
#pragma unroll
        for (int j = 0; j < (KC ? KC : kMaxTopk); j += 2)
          if (j < K) m2[1 + j / 2] = make_int2(slot[j], slot[j + 1]);
      } else {
        m[0] = src_rank;
        m[1] = src_local;
#pragma unroll
        for (int j = 0; j < (KC ? KC : kMaxTopk); ++j)
          if (j < K) m[2 + j] = slot[j];
      }
    }
  } else {
    // rows that receive nothing: padding inside an expert segment, and [R, rcap)
    const int64_t nfill = static_cast<int64_t>(gridDim.x - C) * blockDim.x;
    for (int64_t r = static_cast<int64_t>(blockIdx.x - C) * blockDim.x + threadIdx.x; r < p.rcap;
         r += nfill) {
      // largest e in [0, E] with psum_s[e] <= r
      int lo = 0, hi = E;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (psum_s[mid] <= r) lo = mid; else hi = mid - 1;
      }
      const bool pad = (lo == E) || (r >= psum_s[lo] + cnt_s[lo]);
      if (!pad) continue;
      int32_t* m = p.meta + r * KW;
      for (int j = 0; j < KW; ++j) m[j] = -1;
    }
  }
}

template <int KC>
cudaError_t launch_layout(const LayoutParams& p, const LaunchGeom& g, cudaStream_t s) {
  const int EW = p.num_experts + p.world_size;
  if (p.num_chunks > 0) {
    const size_t smem = sizeof(int32_t) * kLayoutCountWarps * EW;
    ep_layout_count_kernel<KC><<<p.num_chunks, kCountThreads, smem, s>>>(p);
  }
  ep_layout_spine_kernel<<<(EW + kSpineWarps - 1) / kSpineWarps, kSpineWarps * 32, 0, s>>>(p);
  const int64_t fill_ctas = (p.rcap + kSlotThreads * 8 - 1) / (kSlotThreads * 8);
  const int nfill = static_cast<int>(fill_ctas < 1 ? 1 : (fill_ctas > 2 * g.num_sms ? 2 * g.num_sms
                                                                                     : fill_ctas));
  const size_t smem2 = sizeof(int32_t) * (2 * p.num_experts + 1 + 33);
  ep_layout_slots_kernel<KC><<<p.num_chunks + nfill, kSlotThreads, smem2, s>>>(p);
  return cudaGetLastError();
}

template <int KC>
cudaError_t prepare_layout(int /*hidden*/, int /*topk*/, int num_experts_plus_ranks,
                           LaunchGeom* g) {
  const int smem = static_cast<int>(sizeof(int32_t)) * kLayoutCountWarps * num_experts_plus_ranks;
  cudaError_t e = cudaFuncSetAttribute(ep_layout_count_kernel<KC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  g->blocks_per_sm = 1;
  return cudaSuccess;
}

}  // namespace

size_t LayoutScratchBytes(int max_chunks, int columns) {
  // chunk_hist [columns][C] + chunk_off [columns][C] + col_total [columns]
  return sizeof(int32_t) * (2 * static_cast<size_t>(columns) * (max_chunks > 0 ? max_chunks : 1) +
                            static_cast<size_t>(columns));
}

Variant<LayoutLaunch> FindLayout(int topk) {
  switch (topk) {
    case 4: return {"ep_layout_k4", launch_layout<4>, prepare_layout<4>};
    case 6: return {"ep_layout_k6", launch_layout<6>, prepare_layout<6>};
    case 8: return {"ep_layout_k8", launch_layout<8>, prepare_layout<8>};
    default: return {"ep_layout_generic", launch_layout<0>, prepare_layout<0>};
  }
}

}  // namespace epg
