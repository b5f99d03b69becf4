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
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_combine_body.cuh"
#include "ep_kernels.hpp"

namespace epg {

namespace {

template <int HC, int KC, bool WEIGHTED, int V, bool BIAS, bool F32>
__global__ void __launch_bounds__(kCombineThreads) ep_combine_kernel(CombineParams p) {
  combine_body<HC, KC, WEIGHTED, V, BIAS, F32>(p);
}

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

template <int HC, int KC, bool WEIGHTED, int V>
cudaError_t launch_flags(const CombineParams& p, cudaStream_t s, int pdl) {
  const bool bias = p.bias != nullptr, f32 = p.out_f32 != 0;
  const int n = p.num_tokens;
  if (bias && f32)
    return LaunchData(ep_combine_kernel<HC, KC, WEIGHTED, V, true, true>, n, kCombineThreads, s, p, pdl);
  if (bias)
    return LaunchData(ep_combine_kernel<HC, KC, WEIGHTED, V, true, false>, n, kCombineThreads, s, p, pdl);
  if (f32)
    return LaunchData(ep_combine_kernel<HC, KC, WEIGHTED, V, false, true>, n, kCombineThreads, s, p, pdl);
  return LaunchData(ep_combine_kernel<HC, KC, WEIGHTED, V, false, false>, n, kCombineThreads, s, p, pdl);
}

template <int HC, int KC, bool WEIGHTED>
cudaError_t launch_combine(const CombineParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  // 32-byte chunks when every row start is 32-byte aligned; otherwise the
  // generic variant with 16-byte chunks
  const bool v8 = p.hidden % 16 == 0 && aligned32(p.y) && aligned32(p.out) &&
                  (p.bias == nullptr || aligned32(p.bias));
  if (v8) return launch_flags<HC, KC, WEIGHTED, 8>(p, s, g.pdl);
  return launch_flags<0, 0, WEIGHTED, 4>(p, s, g.pdl);
}

template <int HC, int KC, bool WEIGHTED>
cudaError_t prepare_combine(int, int, int, LaunchGeom* g) {
  g->pdl = PdlEnabled() ? 1 : 0;
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
