// ep_types.cuh -- parameter blocks the data kernels take by value, and the
// device error bits.  Compiled by the host compiler, nvcc and NVRTC alike, so
// it includes nothing but the configuration header.
#pragma once

#include "ep_cfg.hpp"

namespace epg {

// Device error bits (sticky, read and cleared by ep_handle_status).
constexpr int32_t kErrBadExpert = 1;   // a topk id outside [-1, E) was skipped
constexpr int32_t kErrTimeout = 2;     // reserved: a kernel gave up a bounded wait

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
};

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
};

}  // namespace epg
