// ep_combine_body.cuh -- device code of the combine kernel (weighted fold of
// the K expert rows in fixed k order, optional bias, bf16 or fp32 output).
// Included by ep_combine.cu, which instantiates the compiled variants, and
// rendered into the run-time specialisations (ep_jit.cpp); it therefore
// includes only headers NVRTC can compile.
#pragma once

#include "ep_cfg.hpp"
#include "ep_types.cuh"

namespace epg {

constexpr int kCombineThreads = 128;

template <int V>
__device__ __forceinline__ void ld_stream(const void* p, Vec<V>& r) {
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

// Two fp32 values to packed bf16 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
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

// a[k] for a runtime k of a small register array (a compile-time unrolled
// select, so the array stays in registers)
template <int N, class T>
__device__ __forceinline__ T pick(const T (&a)[N], int k) {
  T r = a[0];
#pragma unroll
  for (int i = 1; i < N; ++i) r = k == i ? a[i] : r;
  return r;
}
template <int N>
__device__ __forceinline__ int32_t slot_at(const int32_t (&a)[N], int k) { return pick<N>(a, k); }
template <int N>
__device__ __forceinline__ float w_at(const float (&a)[N], int k) { return pick<N>(a, k); }

template <int HC, int KC, bool WEIGHTED, int V, bool BIAS, bool F32>
__device__ __forceinline__ void combine_body(const CombineParams& p) {
  constexpr int KM = KC ? KC : kMaxTopk;
  constexpr int UNIT = 4 * V;  // bytes of bf16 per chunk (2V channels)
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const int row = 2 * H;
  const int chunks = row / UNIT;
  const int t = blockIdx.x;
  // every input here may be an output of the preceding grid (dst_slot of the
  // layout, y of the expert step): nothing is read before it has completed
  allow_dependent_grids();
  grid_dependency_wait();

  int32_t slot[KM];
  float w[KM];
  bool all = true;  // every entry of the token is routed
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    slot[k] = -1;
    w[k] = 1.0f;
    if (k < K) {
      slot[k] = ld_coherent(p.dst_slot + static_cast<int64_t>(t) * K + k);
      if (WEIGHTED) w[k] = ld_coherent(p.weights + static_cast<int64_t>(t) * K + k);
      all &= slot[k] >= 0;
    }
  }
  const uint8_t* y = static_cast<const uint8_t*>(p.y);
  const uint8_t* bias = BIAS ? static_cast<const uint8_t*>(p.bias) + static_cast<int64_t>(t) * row
                             : nullptr;
  uint8_t* out = static_cast<uint8_t*>(p.out) + static_cast<int64_t>(t) * (F32 ? 2 * row : row);
  // bias (one fp32 addition after the fold) and the store of one chunk
  auto finish = [&](int c, float (&acc)[2 * V]) {
    if (BIAS) {
      Vec<V> bv;
      ld_stream<V>(bias + static_cast<int64_t>(c) * UNIT, bv);
      fold<V>(acc, bv, 1.0f, false);
    }
    if (F32) {
      st_f32<V>(out + static_cast<int64_t>(c) * 2 * UNIT, acc);
    } else {
      Vec<V> o;
#pragma unroll
      for (int i = 0; i < V; ++i) o.w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
      st_stream<V>(out + static_cast<int64_t>(c) * UNIT, o);
    }
  };
  if (KC != 0 && all) {
    // the common case, a token with all K entries routed: every row load of a
    // chunk in flight and no per-entry branch.  (Branches around the loads make
    // the compiler keep all K loaded vectors live at once: 96-128 registers
    // instead of ~56, hence fewer resident CTAs; a decode batch of 1024 tokens
    // then needs a second, latency-bound wave.)
    for (int c = threadIdx.x; c < chunks; c += kCombineThreads) {
      Vec<V> v[KM];
#pragma unroll
      for (int k = 0; k < KM; ++k)
        ld_stream<V>(y + static_cast<int64_t>(slot[k]) * row + static_cast<int64_t>(c) * UNIT, v[k]);
      float acc[2 * V];
#pragma unroll
      for (int i = 0; i < 2 * V; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int k = 0; k < KM; ++k) fold<V>(acc, v[k], w[k], WEIGHTED);
      finish(c, acc);
    }
  } else {
    // tokens with a masked entry, and the runtime-top-k variant: the routed
    // rows in k order, four loads in flight at a time
    for (int c = threadIdx.x; c < chunks; c += kCombineThreads) {
      float acc[2 * V];
#pragma unroll
      for (int i = 0; i < 2 * V; ++i) acc[i] = 0.0f;
#pragma unroll 1
      for (int k0 = 0; k0 < K; k0 += 4) {
        Vec<V> v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = k0 + u;
          const int32_t sk = k < K ? slot_at(slot, k) : -1;
          if (sk >= 0) ld_stream<V>(y + static_cast<int64_t>(sk) * row + static_cast<int64_t>(c) * UNIT, v[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = k0 + u;
          if (k < K && slot_at(slot, k) >= 0) fold<V>(acc, v[u], w_at(w, k), WEIGHTED);
        }
      }
      finish(c, acc);
    }
  }
}

}  // namespace epg
