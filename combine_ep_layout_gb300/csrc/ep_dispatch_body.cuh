// ep_dispatch_body.cuh -- device code of the dispatch kernels (row copy for
// the bf16 / fp32 / packed-fp4 transports, fused FP8 cast, routing
// forwarding).  Included by ep_dispatch.cu, which instantiates the compiled
// variants, and rendered into the run-time specialisations (ep_jit.cpp); it
// therefore includes only headers NVRTC can compile.
#pragma once

#include "ep_cfg.hpp"
#include "ep_types.cuh"

namespace epg {

// ---- vector access ---------------------------------------------------------

template <int V>
__device__ __forceinline__ void load_stream(const void* p, Vec<V>& r) {
  if constexpr (V == 8) {
    asm volatile("ld.global.cg.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                   "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p));
  } else {
    asm volatile("ld.global.cg.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "l"(p));
  }
}

template <int V>
__device__ __forceinline__ void store(void* p, const Vec<V>& r) {
  if constexpr (V == 8) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r.w[0]),
                 "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "r"(r.w[4]), "r"(r.w[5]), "r"(r.w[6]),
                 "r"(r.w[7])
                 : "memory");
  } else {
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.w[0]), "r"(r.w[1]),
                 "r"(r.w[2]), "r"(r.w[3])
                 : "memory");
  }
}

// ---- geometry ----------------------------------------------------------------

// Threads per CTA of the copy kernel (RB row bytes, V words per vector) and of
// the FP8 kernel (HC channels) when each row is split over S CTAs; 0 row bytes /
// channels: the runtime-shape variant, kRowMaxThreads threads walking the row
// in a loop.
constexpr int CopyThreads(int rb, int v, int s = 1) {
  return rb ? (RowThreads(rb / (4 * v) / s) ? RowThreads(rb / (4 * v) / s) : kRowMaxThreads)
            : kRowMaxThreads;
}
constexpr int Fp8Threads(int hc, int v, int s = 1) {
  return hc ? (RowThreads(2 * hc / (4 * v) / s) ? RowThreads(2 * hc / (4 * v) / s) : kRowMaxThreads)
            : kRowMaxThreads;
}

// A row of `vectors` vectors can be split over s CTAs when each slice is a
// whole number of `unit`-vector groups held by a compile-time geometry.
constexpr bool Splittable(int vectors, int unit, int s) {
  return vectors > 0 && vectors % (s * unit) == 0 && RowThreads(vectors / s) != 0;
}

// Forward the routing with the rows (the dispatch copy epilogue's
// recv_topk_weights / recv_topk_idx).  Expand layout: row dst_slot[t][k] gets
// topk_weights[t][k] and the expert id of (t, k).  Non-expand layout: each row
// s of the token gets K entries, (id, weight) of the entries it carries
// (entry_slot[t][k] == s) and (-1, 0) for the others.
__device__ __forceinline__ void forward_routing(const DispatchParams& p, int t, int K,
                                                const int32_t* sl) {
  if (p.recv_topk_weights == nullptr && p.recv_topk_idx == nullptr) return;
  if (p.entry_slot != nullptr) {
    const int32_t* es = p.entry_slot + static_cast<int64_t>(t) * K;
    for (int i = threadIdx.x; i < K * K; i += blockDim.x) {
      const int j = i / K, k = i - j * K;
      const int32_t d = sl[j];
      if (d < 0) continue;
      const bool mine = es[k] == d;
      const int64_t src = static_cast<int64_t>(t) * K + k;
      const int64_t dst = static_cast<int64_t>(d) * K + k;
      if (p.recv_topk_weights) p.recv_topk_weights[dst] = mine ? p.topk_weights[src] : 0.0f;
      if (p.recv_topk_idx) p.recv_topk_idx[dst] = mine ? p.topk_i32[src] : -1;
    }
    return;
  }
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const int32_t d = sl[k];
    if (d < 0) continue;
    const int64_t i = static_cast<int64_t>(t) * K + k;
    if (p.recv_topk_weights) p.recv_topk_weights[d] = p.topk_weights[i];
    if (p.recv_topk_idx) p.recv_topk_idx[d] = p.topk_i32[i];
  }
}

// The K slots of a token (sl) as the compiled row kernels read them.  With row
// slices (S > 1: small batches, one short-lived wave) lane k of each warp loads
// slot k up front, in flight with the row's loads, and the store loop takes it
// from that lane: one round trip instead of K dependent ones between the stores
// (decode, 1024 tokens: FP8 dispatch 16.9 -> 14.3 us, bf16 20.9 -> 20.5 us).
// With one CTA per row (large batches) slot k is loaded right before its
// stores: that pacing of each CTA's stores measured 1.2% faster at 32768 tokens
// (627 vs 635 us, bf16) than issuing all of them at once.  All lanes of the
// warp call both (the row kernels' CTAs are whole warps); K <= kMaxTopk (16).
static_assert(kMaxTopk <= 32, "a warp holds one slot per lane");
template <int S>
struct RowSlots {
  int32_t lane_slot = -1;
  __device__ __forceinline__ RowSlots(const int32_t* sl, int K) {
    if constexpr (S > 1) {
      const int lane = threadIdx.x & 31;
      if (lane < K) lane_slot = ld_coherent(sl + lane);
    }
  }
  __device__ __forceinline__ int32_t at(const int32_t* sl, int k) const {
    if constexpr (S > 1) return __shfl_sync(0xffffffffu, lane_slot, k);
    else return ld_coherent(sl + k);
  }
};

// ---- copy (bf16, fp32 and packed-fp4 transports) ------------------------------

// S > 1 (compiled row geometries only): each row is split into S contiguous
// slices, CTA b copying slice b % S of token b / S.
template <int RB, int KC, int V, int S = 1>
__device__ __forceinline__ void dispatch_copy_body(const DispatchParams& p) {
  constexpr int UNIT = 4 * V;  // bytes per vector
  constexpr int KM = KC ? KC : kMaxTopk;
  const int K = KC ? KC : p.topk;
  const int row = RB ? RB : p.row_bytes;
  const int t = S == 1 ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) / S;
  const uint8_t* xr = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t) * row;
  uint8_t* rx = static_cast<uint8_t*>(p.recv_x);
  const int32_t* sl = p.dst_slot + static_cast<int64_t>(t) * K;

  constexpr int CH = RB ? RB / UNIT / S : 0;  // vectors of this CTA's slice
  constexpr int T = RB ? RowThreads(CH) : 0;
  static_assert(S == 1 || (RB != 0 && Splittable(RB / UNIT, 1, S)), "row slices need a compiled geometry");
  const int64_t base = (S == 1 || RB == 0) ? 0 : static_cast<int64_t>(blockIdx.x % S) * CH * UNIT;
  // x is not an output of the layout: warm L2 with this CTA's part of the row
  // while the preceding grid drains, then wait for that grid (dst_slot)
  if (threadIdx.x == 0) prefetch_l2(xr + base, RB ? CH * UNIT : row);
  allow_dependent_grids();
  grid_dependency_wait();
  if constexpr (T != 0) {
    constexpr int PER = CH / T;
    const RowSlots<S> slots(sl, K);
    Vec<V> v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u)
      load_stream<V>(xr + base + static_cast<int64_t>(threadIdx.x + u * T) * UNIT, v[u]);
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k >= K) break;
      const int32_t d = slots.at(sl, k);
      if (d < 0) continue;
      uint8_t* dr = rx + static_cast<int64_t>(d) * row + base;
#pragma unroll
      for (int u = 0; u < PER; ++u) store<V>(dr + static_cast<int64_t>(threadIdx.x + u * T) * UNIT, v[u]);
    }
  } else {
    const int chunks = row / UNIT;
    const int nt = blockDim.x;
    int32_t d[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) d[k] = k < K ? ld_coherent(sl + k) : -1;
    for (int c0 = threadIdx.x; c0 < chunks; c0 += 2 * nt) {
      const int c1 = c0 + nt;
      Vec<V> a, b;
      load_stream<V>(xr + static_cast<int64_t>(c0) * UNIT, a);
      if (c1 < chunks) load_stream<V>(xr + static_cast<int64_t>(c1) * UNIT, b);
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (d[k] < 0) continue;
        uint8_t* dr = rx + static_cast<int64_t>(d[k]) * row;
        store<V>(dr + static_cast<int64_t>(c0) * UNIT, a);
        if (c1 < chunks) store<V>(dr + static_cast<int64_t>(c1) * UNIT, b);
      }
    }
  }
  if (S == 1 || blockIdx.x % S == 0) forward_routing(p, t, K, sl);
}

// ---- FP8 --------------------------------------------------------------------

// Two fp32 values to packed e4m3 (round to nearest even, saturate to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise the 2V bf16 values of one vector with the scale of its 128-channel
// group; `lanes` consecutive lanes (a power of two) hold the group.  Every lane
// of the warp must call this (the reduction is a full-warp shuffle).
template <int V>
__device__ __forceinline__ void quantise(const Vec<V>& in, int lanes, uint32_t (&q)[V / 2],
                                         float& scale) {
  float f[2 * V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    f[2 * i] = __uint_as_float(in.w[i] << 16);
    f[2 * i + 1] = __uint_as_float(in.w[i] & 0xffff0000u);
  }
  uint32_t a = 0;
#pragma unroll
  for (int i = 0; i < 2 * V; ++i) {
    uint32_t b = __float_as_uint(f[i]) & 0x7fffffffu;
    b = b > 0x7f800000u ? 0u : b;  // NaN does not take part in the maximum
    a = b > a ? b : a;
  }
  for (int o = 1; o < lanes; o <<= 1) {
    const uint32_t other = __shfl_xor_sync(0xffffffffu, a, o);
    a = other > a ? other : a;
  }
  scale = 0.0f;
#pragma unroll
  for (int i = 0; i < V / 2; ++i) q[i] = 0u;
  if (a != 0u) {
    scale = __fdiv_rn(__uint_as_float(a), 448.0f);
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      const float r0 = __fdiv_rn(f[4 * i], scale), r1 = __fdiv_rn(f[4 * i + 1], scale);
      const float r2 = __fdiv_rn(f[4 * i + 2], scale), r3 = __fdiv_rn(f[4 * i + 3], scale);
      q[i] = cvt_e4m3x2(r0, r1) | (cvt_e4m3x2(r2, r3) << 16);
    }
  }
}

template <int V>
__device__ __forceinline__ void store_q(void* p, const uint32_t (&q)[V / 2]) {
  if constexpr (V == 8) {
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(q[0]), "r"(q[1]), "r"(q[2]),
                 "r"(q[3])
                 : "memory");
  } else {
    asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(q[0]), "r"(q[1]) : "memory");
  }
}

// S > 1 (compiled geometries only): each row is split into S slices of whole
// 128-channel groups, CTA b quantising slice b % S of token b / S.
template <int HC, int KC, int V, int S = 1>
__device__ __forceinline__ void dispatch_fp8_body(const DispatchParams& p) {
  constexpr int UNIT = 4 * V;            // input bytes per vector (2V channels)
  constexpr int LANES = 128 / (2 * V);   // lanes per 128-channel group
  constexpr int KM = KC ? KC : kMaxTopk;
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const int G = H / kScaleGroup;
  const int t = S == 1 ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) / S;
  const uint8_t* xr = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t) * 2 * H;
  uint8_t* rq = static_cast<uint8_t*>(p.recv_x);
  float* rs = p.recv_scales;
  const int32_t* sl = p.dst_slot + static_cast<int64_t>(t) * K;
  const bool leader = (threadIdx.x % LANES) == 0;

  constexpr int CH = HC ? 2 * HC / UNIT / S : 0;  // vectors of this CTA's slice
  constexpr int T = HC ? RowThreads(CH) : 0;
  static_assert(S == 1 || (HC != 0 && Splittable(2 * HC / UNIT, LANES, S)),
                "row slices need a compiled geometry of whole scale groups");
  const int cs = (S == 1 || HC == 0) ? 0 : static_cast<int>(blockIdx.x % S) * CH;  // first vector of the slice
  // x is not an output of the layout: warm L2 with this CTA's part of the row
  // while the preceding grid drains, then wait for that grid (dst_slot)
  if (threadIdx.x == 0)
    prefetch_l2(xr + static_cast<int64_t>(cs) * UNIT, HC ? CH * UNIT : 2 * H);
  allow_dependent_grids();
  grid_dependency_wait();
  if constexpr (T != 0) {
    constexpr int PER = CH / T;
    const RowSlots<S> slots(sl, K);
    Vec<V> v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u)
      load_stream<V>(xr + static_cast<int64_t>(cs + threadIdx.x + u * T) * UNIT, v[u]);
    uint32_t q[PER][V / 2];
    float s[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) quantise<V>(v[u], LANES, q[u], s[u]);
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k >= K) break;
      const int32_t d = slots.at(sl, k);
      if (d < 0) continue;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int c = cs + threadIdx.x + u * T;
        store_q<V>(rq + static_cast<int64_t>(d) * H + static_cast<int64_t>(c) * (2 * V), q[u]);
        if (leader) rs[static_cast<int64_t>(d) * G + c / LANES] = s[u];
      }
    }
  } else {
    const int chunks = 2 * H / UNIT;
    int32_t d[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) d[k] = k < K ? ld_coherent(sl + k) : -1;
    // uniform trip count (blockDim is a multiple of 32): the shuffles see every lane
    for (int c0 = 0; c0 < chunks; c0 += blockDim.x) {
      const int c = c0 + threadIdx.x;
      const bool in = c < chunks;
      Vec<V> v;
#pragma unroll
      for (int i = 0; i < V; ++i) v.w[i] = 0u;
      if (in) load_stream<V>(xr + static_cast<int64_t>(c) * UNIT, v);
      uint32_t q[V / 2];
      float s;
      quantise<V>(v, LANES, q, s);
      if (!in) continue;
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (d[k] < 0) continue;
        store_q<V>(rq + static_cast<int64_t>(d[k]) * H + static_cast<int64_t>(c) * (2 * V), q);
        if (leader) rs[static_cast<int64_t>(d[k]) * G + c / LANES] = s;
      }
    }
  }
  if (S == 1 || blockIdx.x % S == 0) forward_routing(p, t, K, sl);
}

}  // namespace epg
