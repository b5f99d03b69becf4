// ep_dispatch.cu -- dispatch: scatter each token row to its K receive rows
// ("Dispatch data flow" of "DeepEP overall architecture analysis": pack token
// data + scale factors, then copy into recv_x; "MORI JIT v2" §3.7: the
// transport dtype is a property of the copy, not arithmetic).
//
// On one GPU the pages' two hops (symmetric buffer, then copy epilogue) fold
// into one pass: read x[t] once, write it K times.  One CTA per token: every
// thread loads its whole share of the row first (all loads of the row in
// flight at once), then writes it to the K destination rows.  Accesses are
// 32 bytes per thread (the 256-bit ld/st of the sm_100 family) when the row
// and the buffers are 32-byte aligned, 16 bytes otherwise.
//
// Design note: a cp.async.bulk (TMA) ring that staged each row in shared
// memory and issued K bulk stores moved the same bytes with one thread per CTA,
// but saturated at ~6.0 TB/s on the prefill shape at every ring depth and CTA
// count tried; the register copy with many CTAs per SM reaches ~6.8 TB/s,
// above the device's pure-write rate, because the loads overlap the stores.
//
//   copy: bf16, fp32 and packed-fp4 (Fp4x2: H channels in H/2 bytes) rows
//         are moved as bytes, unchanged.
//   FP8:  each 128-channel group is held by 8 (32-byte) or 16 (16-byte)
//         consecutive lanes; amax is reduced across them with shuffles, the
//         scale is amax/448 (IEEE division), values are x/s (IEEE division)
//         converted with cvt.rn.satfinite.e4m3x2.f32, once per token, and the
//         bytes plus the scale are written to every destination row.
// Optionally each destination row also receives the routing it came with
// (its expert id and the token's weight for it), as the pages' dispatch copy
// epilogue fills recv_topk_idx / recv_topk_weights.
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

// ---- vector access ---------------------------------------------------------

template <int V>
struct Vec {
  uint32_t w[V];
};

template <int V>
__device__ __forceinline__ void load_stream(const void* p, Vec<V>& r) {
  if constexpr (V == 8) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                   "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p));
  } else {
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
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

// Threads per CTA for a row of `chunks` vectors: the largest multiple of 32 that
// divides it and is at most 256 (so every thread owns the same number of
// vectors, at most 8); 0 when there is none (the row is then walked in a loop).
constexpr int threads_for(int chunks) {
  for (int t = 256; t >= 32; t -= 32)
    if (chunks % t == 0 && chunks / t <= 8) return t;
  return 0;
}

constexpr int kMaxThreads = 256;

// CTA size of the loop path: enough threads for `per_iter` vectors per thread
// per iteration, a multiple of 32, at most kMaxThreads.
inline int loop_block(int chunks, int per_iter) {
  int t = (chunks + per_iter - 1) / per_iter;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > kMaxThreads ? kMaxThreads : t);
}

// Forward the routing with the rows (the dispatch copy epilogue's
// recv_topk_weights / recv_topk_idx): row dst_slot[t][k] gets topk_weights[t][k]
// and the expert id of (t, k).
__device__ __forceinline__ void forward_routing(const DispatchParams& p, int t, int K,
                                                const int32_t* sl) {
  if (p.recv_topk_weights == nullptr && p.recv_topk_idx == nullptr) return;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const int32_t d = sl[k];
    if (d < 0) continue;
    const int64_t i = static_cast<int64_t>(t) * K + k;
    if (p.recv_topk_weights) p.recv_topk_weights[d] = p.topk_weights[i];
    if (p.recv_topk_idx) p.recv_topk_idx[d] = p.topk_i32[i];
  }
}

// ---- copy (bf16, fp32 and packed-fp4 transports) ------------------------------

template <int RB, int KC, int V>
__global__ void __launch_bounds__(RB ? (threads_for(RB / (4 * V)) ? threads_for(RB / (4 * V))
                                                                  : kMaxThreads)
                                     : kMaxThreads)
    ep_dispatch_copy_kernel(DispatchParams p) {
  constexpr int UNIT = 4 * V;  // bytes per vector
  constexpr int KM = KC ? KC : kMaxTopk;
  const int K = KC ? KC : p.topk;
  const int row = RB ? RB : p.row_bytes;
  const int t = blockIdx.x;
  const uint8_t* xr = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t) * row;
  uint8_t* rx = static_cast<uint8_t*>(p.recv_x);
  const int32_t* sl = p.dst_slot + static_cast<int64_t>(t) * K;

  constexpr int CH = RB ? RB / UNIT : 0;
  constexpr int T = RB ? threads_for(CH) : 0;
  if constexpr (T != 0) {
    constexpr int PER = CH / T;
    Vec<V> v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u)
      load_stream<V>(xr + static_cast<int64_t>(threadIdx.x + u * T) * UNIT, v[u]);
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k >= K) break;
      const int32_t d = __ldg(sl + k);
      if (d < 0) continue;
      uint8_t* dr = rx + static_cast<int64_t>(d) * row;
#pragma unroll
      for (int u = 0; u < PER; ++u) store<V>(dr + static_cast<int64_t>(threadIdx.x + u * T) * UNIT, v[u]);
    }
  } else {
    const int chunks = row / UNIT;
    const int nt = blockDim.x;
    int32_t d[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) d[k] = k < K ? __ldg(sl + k) : -1;
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
  forward_routing(p, t, K, sl);
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

template <int HC, int KC, int V>
__global__ void __launch_bounds__(HC ? (threads_for(2 * HC / (4 * V)) ? threads_for(2 * HC / (4 * V))
                                                                      : kMaxThreads)
                                     : kMaxThreads)
    ep_dispatch_fp8_kernel(DispatchParams p) {
  constexpr int UNIT = 4 * V;            // input bytes per vector (2V channels)
  constexpr int LANES = 128 / (2 * V);   // lanes per 128-channel group
  constexpr int KM = KC ? KC : kMaxTopk;
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const int G = H / kScaleGroup;
  const int t = blockIdx.x;
  const uint8_t* xr = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t) * 2 * H;
  uint8_t* rq = static_cast<uint8_t*>(p.recv_x);
  float* rs = p.recv_scales;
  const int32_t* sl = p.dst_slot + static_cast<int64_t>(t) * K;
  const bool leader = (threadIdx.x % LANES) == 0;

  constexpr int CH = HC ? 2 * HC / UNIT : 0;
  constexpr int T = HC ? threads_for(CH) : 0;
  if constexpr (T != 0) {
    constexpr int PER = CH / T;
    Vec<V> v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u)
      load_stream<V>(xr + static_cast<int64_t>(threadIdx.x + u * T) * UNIT, v[u]);
    uint32_t q[PER][V / 2];
    float s[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) quantise<V>(v[u], LANES, q[u], s[u]);
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k >= K) break;
      const int32_t d = __ldg(sl + k);
      if (d < 0) continue;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int c = threadIdx.x + u * T;
        store_q<V>(rq + static_cast<int64_t>(d) * H + static_cast<int64_t>(c) * (2 * V), q[u]);
        if (leader) rs[static_cast<int64_t>(d) * G + c / LANES] = s[u];
      }
    }
  } else {
    const int chunks = 2 * H / UNIT;
    int32_t d[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) d[k] = k < K ? __ldg(sl + k) : -1;
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
  forward_routing(p, t, K, sl);
}

// ---- launchers -------------------------------------------------------------

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

template <int RB, int KC, int V>
int copy_block(int row_bytes) {
  constexpr int T = RB ? threads_for(RB / (4 * V)) : 0;
  return T ? T : loop_block(row_bytes / (4 * V), 2);
}

template <int RB, int KC>
cudaError_t launch_copy(const DispatchParams& p, const LaunchGeom&, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  // 32-byte vectors when every row start is 32-byte aligned
  if (p.row_bytes % 32 == 0 && aligned32(p.x) && aligned32(p.recv_x))
    ep_dispatch_copy_kernel<RB, KC, 8><<<p.num_tokens, copy_block<RB, KC, 8>(p.row_bytes), 0, s>>>(p);
  else
    ep_dispatch_copy_kernel<RB, KC, 4><<<p.num_tokens, copy_block<RB, KC, 4>(p.row_bytes), 0, s>>>(p);
  return cudaGetLastError();
}

template <int RB, int KC>
cudaError_t prepare_copy(int, int, int, LaunchGeom* g) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_dispatch_copy_kernel<RB, KC, 8>, kMaxThreads, 0);
}

template <int HC, int KC, int V>
int fp8_block(int hidden) {
  constexpr int T = HC ? threads_for(2 * HC / (4 * V)) : 0;
  return T ? T : loop_block(2 * hidden / (4 * V), 1);
}

template <int HC, int KC>
cudaError_t launch_fp8(const DispatchParams& p, const LaunchGeom&, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  // hidden % 128 == 0 here, so 32-byte input vectors only need an aligned x
  if (aligned32(p.x))
    ep_dispatch_fp8_kernel<HC, KC, 8><<<p.num_tokens, fp8_block<HC, KC, 8>(p.hidden), 0, s>>>(p);
  else
    ep_dispatch_fp8_kernel<HC, KC, 4><<<p.num_tokens, fp8_block<HC, KC, 4>(p.hidden), 0, s>>>(p);
  return cudaGetLastError();
}

template <int HC, int KC>
cudaError_t prepare_fp8(int, int, int, LaunchGeom* g) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_dispatch_fp8_kernel<HC, KC, 8>, kMaxThreads, 0);
}

}  // namespace

Variant<DispatchLaunch> FindDispatch(int hidden, int topk, EpDType dtype) {
  switch (dtype) {
    case EpDType::Bf16:
#define EPG_CASE(H, K)                                                            \
  if (hidden == H && topk == K)                                                   \
    return {"ep_dispatch_bf16_h" #H "_k" #K, launch_copy<2 * H, K>, prepare_copy<2 * H, K>};
      EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
      return {"ep_dispatch_bf16_generic", launch_copy<0, 0>, prepare_copy<0, 0>};
    case EpDType::Fp32:
#define EPG_CASE(H, K)                                                            \
  if (hidden == H && topk == K)                                                   \
    return {"ep_dispatch_fp32_h" #H "_k" #K, launch_copy<4 * H, K>, prepare_copy<4 * H, K>};
      EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
      return {"ep_dispatch_fp32_generic", launch_copy<0, 0>, prepare_copy<0, 0>};
    case EpDType::Fp4x2:
#define EPG_CASE(H, K)                                                            \
  if (hidden == H && topk == K)                                                   \
    return {"ep_dispatch_fp4x2_h" #H "_k" #K, launch_copy<H / 2, K>, prepare_copy<H / 2, K>};
      EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
      return {"ep_dispatch_fp4x2_generic", launch_copy<0, 0>, prepare_copy<0, 0>};
    case EpDType::Fp8:
#define EPG_CASE(H, K)                                                         \
  if (hidden == H && topk == K)                                                \
    return {"ep_dispatch_fp8_h" #H "_k" #K, launch_fp8<H, K>, prepare_fp8<H, K>};
      EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
      return {"ep_dispatch_fp8_generic", launch_fp8<0, 0>, prepare_fp8<0, 0>};
  }
  return {nullptr, nullptr, nullptr};
}

}  // namespace epg
