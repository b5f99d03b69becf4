// ep_types.cuh -- parameter blocks the data kernels take by value, the
// device error bits and the programmatic-dependent-launch helpers.  Compiled by
// the host compiler, nvcc and NVRTC alike, so it includes nothing but the
// configuration header and keeps device code behind __CUDACC__.
#pragma once

#include "ep_cfg.hpp"

namespace epg {

// Device error bits (sticky, read and cleared by ep_handle_status).
constexpr int32_t kErrBadExpert = 1;   // value 1 (bit 0): a topk id outside [-1, E) was skipped
constexpr int32_t kErrTimeout = 2;     // value 2 (bit 1): a kernel gave up a bounded wait

#if defined(__CUDACC__)
// ---- programmatic dependent launch (sm_90 and later) --------------------------
//
// A kernel launched with programmatic stream serialisation may be scheduled
// while the preceding kernel of its stream is still running.  Such a kernel
// calls grid_dependency_wait() before its first access to memory that a
// preceding kernel may have written (and before any store): the wait returns
// once the preceding grid has completed and its writes are visible.  Launched
// without the attribute, the wait returns at once.  allow_dependent_grids()
// lets the next kernel of the stream be scheduled as soon as every CTA of this
// grid has called it (or exited); that kernel still waits for this grid's
// completion itself.

__device__ __forceinline__ void allow_dependent_grids() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Loads in kernels launched with programmatic stream serialisation.  Such a
// kernel is alive while its predecessor still writes, so the non-coherent
// read-only path (ld.global.nc / __ldg), whose contract is data that stays
// unchanged for the reading kernel's whole lifetime, must not serve anything
// a predecessor may produce: a replayed graph read stale dst_slot / row lines
// through it.  These loads are cached in L2 only (.cg), which is where the
// predecessor's writes are visible once grid_dependency_wait() has returned.
__device__ __forceinline__ int32_t ld_coherent(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_coherent(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// Ask the TMA unit to bring `bytes` (a multiple of 16, 16-byte aligned address)
// of global memory into L2.  A hint only: no data reaches the thread, so it is
// safe on memory another kernel may still be writing.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
#endif

// V 32-bit words moved by one vector access (V = 4: 16 bytes, V = 8: 32 bytes).
template <int V>
struct Vec {
  uint32_t w[V];
};

struct DispatchParams {
  const void* x;             // [N, row_bytes] (bf16 for FP8 dispatch)
  void* recv_x;              // [Rcap, row_bytes] (e4m3 [Rcap, H] for FP8)
  float* recv_scales;        // fp32 [Rcap, H/128] (FP8 only)
  const int32_t* dst_slot;   // [N, K]
  int num_tokens;
  int hidden;
  int topk;
  int row_bytes;             // bytes of one transported row (copy transports)
  int32_t* err;
  // routing forwarded with the rows (both nullptr: not forwarded)
  const float* topk_weights;   // fp32 [N, K]
  const int32_t* topk_i32;     // int32 [N, K] expert ids (the handle's clone)
  float* recv_topk_weights;    // fp32 [Rcap] (non-expand: [Rcap, K]) or nullptr
  int32_t* recv_topk_idx;      // int32 [Rcap] (non-expand: [Rcap, K]) or nullptr
  // non-expand layout: dst_slot above holds the token's distinct rows and this
  // the row of each (t, k); nullptr for the expand layout
  const int32_t* entry_slot;   // [N, K]
  // bound of one wait on the TMA dispatch's mbarriers (ns; 0: give up at the
  // first test that finds the copy still in flight)
  uint64_t wait_ns;
};

// Default bound of a bounded device-side wait: one second.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

struct CombineParams {
  const void* y;             // bf16 [Rcap, H]
  const float* weights;      // fp32 [N, K] or nullptr
  const void* bias;          // bf16 [N, H] or nullptr
  void* out;                 // bf16 or fp32 [N, H]
  const int32_t* dst_slot;   // [N, K]
  int num_tokens;
  int hidden;
  int topk;
  int out_f32;               // 1: fp32 output, 0: bf16
  int32_t* err;              // device error word (the TMA combine's timeouts)
  uint64_t wait_ns;          // bound of one wait on the TMA combine's mbarrier
};

}  // namespace epg
