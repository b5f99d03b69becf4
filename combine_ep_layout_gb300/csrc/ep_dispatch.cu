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
//
// Small batches split each row over two CTAs (the geometry table below), so
// that a batch that fills less than a wave of the GPU still keeps every SM's
// loads and stores in flight.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "ep_cfg.hpp"
#include "ep_dispatch_body.cuh"
#include "ep_kernels.hpp"

namespace epg {

namespace {

template <int RB, int KC, int V, int S>
__global__ void __launch_bounds__(CopyThreads(RB, V, S), CopyMinBlocks(RB, V, S))
    ep_dispatch_copy_kernel(DispatchParams p) {
  dispatch_copy_body<RB, KC, V, S>(p);
}

// The explicit minimum of one resident CTA leaves the register budget to the
// kernel's needs (39-47 registers): with the thread bound alone ptxas held some
// variants to 32 registers and moved values to local memory (a 4-byte spill and
// 8-24 byte stack frames).
template <int HC, int KC, int V, int S>
__global__ void __launch_bounds__(Fp8Threads(HC, V, S), 1) ep_dispatch_fp8_kernel(DispatchParams p) {
  dispatch_fp8_body<HC, KC, V, S>(p);
}

// ---- geometry tuning table ---------------------------------------------------
//
// Token-count buckets -> CTAs per token row for the compiled row kernels ("MORI
// JIT v2" §5.1: a geometry table per kernel keyed by the number of tokens).  From
// a sweep on GB300 at hidden 7168, top-8, cold buffers: splitting each row over
// two CTAs moved 1024 tokens in 23.4 us instead of 24.4 us and 2048 tokens in
// 44.0 us instead of 44.9 us; from 8192 tokens on one CTA per row is as fast
// (162 us either way; at 32768 tokens within 0.5 %).  Combine has one geometry:
// none of the sweep's alternatives beat it.
struct SliceBucket {
  int max_tokens;
  int slices;
};
constexpr SliceBucket kDispatchSlices[] = {{2048, 2}, {1 << 30, 1}};

inline int row_slices(int num_tokens, const LaunchGeom& g) {
  if (g.row_slices > 0) return g.row_slices;
  for (const SliceBucket& b : kDispatchSlices)
    if (num_tokens <= b.max_tokens) return b.slices;
  return 1;
}

// EP_GB300_DISPATCH_SLICES=1|2 pins the table's choice (for benchmarking).
inline int slices_override() {
  const char* env = std::getenv("EP_GB300_DISPATCH_SLICES");
  if (env == nullptr) return 0;
  const int v = std::atoi(env);
  return v == 1 || v == 2 ? v : 0;
}

// CTA size of the loop path: enough threads for `per_iter` vectors per thread
// per iteration, a multiple of 32, at most kRowMaxThreads.
inline int loop_block(int chunks, int per_iter) {
  int t = (chunks + per_iter - 1) / per_iter;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > kRowMaxThreads ? kRowMaxThreads : t);
}

// ---- launchers -------------------------------------------------------------

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

template <int RB, int KC, int V, int S>
int copy_block(int row_bytes) {
  constexpr int T = RB ? RowThreads(RB / (4 * V) / S) : 0;
  return T ? T : loop_block(row_bytes / (4 * V), 2);
}

template <int RB, int KC>
cudaError_t launch_copy(const DispatchParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  // 32-byte vectors when every row start is 32-byte aligned
  if (p.row_bytes % 32 == 0 && aligned32(p.x) && aligned32(p.recv_x)) {
    if constexpr (RB != 0 && Splittable(RB / 32, 1, 2)) {
      if (row_slices(p.num_tokens, g) == 2)
        return LaunchData(ep_dispatch_copy_kernel<RB, KC, 8, 2>, 2 * p.num_tokens,
                          copy_block<RB, KC, 8, 2>(p.row_bytes), s, p, g.pdl);
    }
    return LaunchData(ep_dispatch_copy_kernel<RB, KC, 8, 1>, p.num_tokens,
                      copy_block<RB, KC, 8, 1>(p.row_bytes), s, p, g.pdl);
  }
  return LaunchData(ep_dispatch_copy_kernel<RB, KC, 4, 1>, p.num_tokens,
                    copy_block<RB, KC, 4, 1>(p.row_bytes), s, p, g.pdl);
}

template <int RB, int KC>
cudaError_t prepare_copy(int, int, int, LaunchGeom* g) {
  g->row_slices = slices_override();
  g->pdl = PdlEnabled() ? 1 : 0;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_dispatch_copy_kernel<RB, KC, 8, 1>, kRowMaxThreads, 0);
}

template <int HC, int KC, int V, int S>
int fp8_block(int hidden) {
  constexpr int T = HC ? RowThreads(2 * HC / (4 * V) / S) : 0;
  return T ? T : loop_block(2 * hidden / (4 * V), 1);
}

template <int HC, int KC>
cudaError_t launch_fp8(const DispatchParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  // hidden % 128 == 0 here, so 32-byte input vectors only need an aligned x
  if (aligned32(p.x)) {
    if constexpr (HC != 0 && Splittable(2 * HC / 32, 128 / 16, 2)) {
      if (row_slices(p.num_tokens, g) == 2)
        return LaunchData(ep_dispatch_fp8_kernel<HC, KC, 8, 2>, 2 * p.num_tokens,
                          fp8_block<HC, KC, 8, 2>(p.hidden), s, p, g.pdl);
    }
    return LaunchData(ep_dispatch_fp8_kernel<HC, KC, 8, 1>, p.num_tokens,
                      fp8_block<HC, KC, 8, 1>(p.hidden), s, p, g.pdl);
  }
  return LaunchData(ep_dispatch_fp8_kernel<HC, KC, 4, 1>, p.num_tokens,
                    fp8_block<HC, KC, 4, 1>(p.hidden), s, p, g.pdl);
}

template <int HC, int KC>
cudaError_t prepare_fp8(int, int, int, LaunchGeom* g) {
  g->row_slices = slices_override();
  g->pdl = PdlEnabled() ? 1 : 0;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_dispatch_fp8_kernel<HC, KC, 8, 1>, kRowMaxThreads, 0);
}

}  // namespace

bool PdlEnabled() {
  const char* env = std::getenv("EP_GB300_PDL");
  return env == nullptr || env[0] != '0';
}

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
