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
// One CTA per token; each thread owns 16-byte column chunks (8 channels) and
// issues the loads of all K rows for a chunk before reducing them, so K row
// fetches are in flight per thread.  Expert rows are read exactly once, so the
// loads bypass L1 and carry an evict-first L2 hint.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

constexpr int kCombineThreads = 128;

__device__ __forceinline__ uint4 ld_stream(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void fold8(float (&acc)[8], const uint4& v, float w, bool weighted) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(u[i] << 16);
    const float hi = __uint_as_float(u[i] & 0xffff0000u);
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

template <int HC, int KC, bool WEIGHTED>
__global__ void __launch_bounds__(kCombineThreads) ep_combine_kernel(CombineParams p) {
  constexpr int KM = KC ? KC : kMaxTopk;
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const int chunks = H / 8;  // 16-byte chunks per row
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
  const uint4* y = static_cast<const uint4*>(p.y);
  uint4* out = static_cast<uint4*>(p.out) + static_cast<int64_t>(t) * chunks;
  const uint64_t pol = policy_evict_first();

  for (int c = threadIdx.x; c < chunks; c += kCombineThreads) {
    uint4 v[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (slot[k] >= 0) v[k] = ld_stream(y + static_cast<int64_t>(slot[k]) * chunks + c, pol);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < KM; ++k)
      if (slot[k] >= 0) fold8(acc, v[k], w[k], WEIGHTED);
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    __stcs(out + c, o);
  }
}

template <int HC, int KC, bool WEIGHTED>
cudaError_t launch_combine(const CombineParams& p, const LaunchGeom&, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  ep_combine_kernel<HC, KC, WEIGHTED><<<p.num_tokens, kCombineThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int HC, int KC, bool WEIGHTED>
cudaError_t prepare_combine(int, int, int, LaunchGeom* g) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_combine_kernel<HC, KC, WEIGHTED>, kCombineThreads, 0);
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
