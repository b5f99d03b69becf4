// ep_combine.cu -- combine: per token, the weighted reduce of its K expert
// output rows back to token order ("Combine data flow" of "DeepEP overall
// architecture analysis": reduce from the buffer weighted by topk_weights and
// write back; "MORI JIT v2" §3.7 / §5: combine reduces bf16 with fp32
// accumulation).
//
// out[t][c] = bf16_rn(fold over k ascending of acc = fmaf(w[t][k], y[slot][c], acc)),
// acc = +0.0f, masked k skipped.  The order is fixed, so the result is
// bit-for-bit reproducible.
//
// Optionally a bf16 bias [N, H] is added after the fold (one fp32 addition,
// the "+ bias" of the pages' combine epilogue) and the output is fp32 instead
// of bf16.
//
// One CTA per token; each thread owns 32-byte (16 channels) column chunks --
// 16-byte chunks when a buffer is only 16-byte aligned -- and issues the loads
// of all K rows for a chunk before folding them, so K row fetches are in
// flight per thread.  Expert rows are read exactly once, so the loads bypass
// L1.  (An evict-first L2 hint on these loads measured ~3% slower on the
// prefill shape, so none is given.)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

constexpr int kCombineThreads = 128;

template <int V>
struct Vec {
  uint32_t w[V];
};

template <int V>
__device__ __forceinline__ void ld_stream(const void* p, Vec<V>& r) {
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
__device__ __forceinline__ void st_stream(void* p, const Vec<V>& r) {
  if constexpr (V == 8) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r.w[0]),
                 "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "r"(r.w[4]), "r"(r.w[5]), "r"(r.w[6]),
                 "r"(r.w[7])
                 : "memory");
  } else {
    asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.w[0]), "r"(r.w[1]),
                 "r"(r.w[2]), "r"(r.w[3])
                 : "memory");
  }
}

template <int V>
__device__ __forceinline__ void fold(float (&acc)[2 * V], const Vec<V>& v, float w, bool weighted) {
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const float lo = __uint_as_float(v.w[i] << 16);
    const float hi = __uint_as_float(v.w[i] & 0xffff0000u);
    if (weighted) {
      acc[2 * i] = __fmaf_rn(w, lo, acc[2 * i]);
      acc[2 * i + 1] = __fmaf_rn(w, hi, acc[2 * i + 1]);
    } else {
      acc[2 * i] = __fadd_rn(acc[2 * i], lo);
      acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], hi);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <int V>
__device__ __forceinline__ void st_f32(void* p, const float (&acc)[2 * V]) {
  // 2V fp32 values: two vectors of V words
  Vec<V> a, b;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    a.w[i] = __float_as_uint(acc[i]);
    b.w[i] = __float_as_uint(acc[V + i]);
  }
  st_stream<V>(p, a);
  st_stream<V>(static_cast<uint8_t*>(p) + 4 * V, b);
}

template <int HC, int KC, bool WEIGHTED, int V, bool BIAS, bool F32>
__global__ void __launch_bounds__(kCombineThreads) ep_combine_kernel(CombineParams p) {
  constexpr int KM = KC ? KC : kMaxTopk;
  constexpr int UNIT = 4 * V;  // bytes of bf16 per chunk (2V channels)
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const int row = 2 * H;
  const int chunks = row / UNIT;
  const int t = blockIdx.x;

  int32_t slot[KM];
  float w[KM];
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    slot[k] = -1;
    w[k] = 1.0f;
    if (k < K) {
      slot[k] = __ldg(p.dst_slot + static_cast<int64_t>(t) * K + k);
      if (WEIGHTED) w[k] = __ldg(p.weights + static_cast<int64_t>(t) * K + k);
    }
  }
  const uint8_t* y = static_cast<const uint8_t*>(p.y);
  const uint8_t* bias = BIAS ? static_cast<const uint8_t*>(p.bias) + static_cast<int64_t>(t) * row
                             : nullptr;
  uint8_t* out = static_cast<uint8_t*>(p.out) + static_cast<int64_t>(t) * (F32 ? 2 * row : row);
  for (int c = threadIdx.x; c < chunks; c += kCombineThreads) {
    Vec<V> v[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (slot[k] >= 0)
        ld_stream<V>(y + static_cast<int64_t>(slot[k]) * row + static_cast<int64_t>(c) * UNIT, v[k]);
    Vec<V> bv;
    if (BIAS) ld_stream<V>(bias + static_cast<int64_t>(c) * UNIT, bv);
    float acc[2 * V];
#pragma unroll
    for (int i = 0; i < 2 * V; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (slot[k] >= 0) fold<V>(acc, v[k], w[k], WEIGHTED);
    if (BIAS) fold<V>(acc, bv, 1.0f, false);  // one fp32 addition after the fold
    if (F32) {
      st_f32<V>(out + static_cast<int64_t>(c) * 2 * UNIT, acc);
    } else {
      Vec<V> o;
#pragma unroll
      for (int i = 0; i < V; ++i) o.w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
      st_stream<V>(out + static_cast<int64_t>(c) * UNIT, o);
    }
  }
}

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

template <int HC, int KC, bool WEIGHTED, int V>
cudaError_t launch_flags(const CombineParams& p, cudaStream_t s) {
  const bool bias = p.bias != nullptr, f32 = p.out_f32 != 0;
  if (bias && f32)
    ep_combine_kernel<HC, KC, WEIGHTED, V, true, true><<<p.num_tokens, kCombineThreads, 0, s>>>(p);
  else if (bias)
    ep_combine_kernel<HC, KC, WEIGHTED, V, true, false><<<p.num_tokens, kCombineThreads, 0, s>>>(p);
  else if (f32)
    ep_combine_kernel<HC, KC, WEIGHTED, V, false, true><<<p.num_tokens, kCombineThreads, 0, s>>>(p);
  else
    ep_combine_kernel<HC, KC, WEIGHTED, V, false, false><<<p.num_tokens, kCombineThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int HC, int KC, bool WEIGHTED>
cudaError_t launch_combine(const CombineParams& p, const LaunchGeom&, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  // 32-byte chunks when every row start is 32-byte aligned; otherwise the
  // generic variant with 16-byte chunks
  const bool v8 = p.hidden % 16 == 0 && aligned32(p.y) && aligned32(p.out) &&
                  (p.bias == nullptr || aligned32(p.bias));
  if (v8) return launch_flags<HC, KC, WEIGHTED, 8>(p, s);
  return launch_flags<0, 0, WEIGHTED, 4>(p, s);
}

template <int HC, int KC, bool WEIGHTED>
cudaError_t prepare_combine(int, int, int, LaunchGeom* g) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_combine_kernel<HC, KC, WEIGHTED, 8, false, false>, kCombineThreads, 0);
}

}  // namespace

Variant<CombineLaunch> FindCombine(int hidden, int topk, bool use_weights) {
  if (use_weights) {
#define EPG_CASE(H, K)                                                                  \
  if (hidden == H && topk == K)                                                         \
    return {"ep_combine_w_h" #H "_k" #K, launch_combine<H, K, true>, prepare_combine<H, K, true>};
    EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
    return {"ep_combine_w_generic", launch_combine<0, 0, true>, prepare_combine<0, 0, true>};
  }
#define EPG_CASE(H, K)                                                                    \
  if (hidden == H && topk == K)                                                           \
    return {"ep_combine_h" #H "_k" #K, launch_combine<H, K, false>, prepare_combine<H, K, false>};
  EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
  return {"ep_combine_generic", launch_combine<0, 0, false>, prepare_combine<0, 0, false>};
}

}  // namespace epg
