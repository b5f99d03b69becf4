// ep_kernels.hpp -- host-side interface between the C ABI (ep_api.cu) and the
// kernel translation units.  Each kernel file exposes a registry lookup that
// maps a runtime shape to the launcher of a compiled variant (a
// specialisation from EPG_SHAPE_LIST, or the generic one), with the variant's
// descriptive name ("MORI JIT v2" §3.3: the entry name carries the shape).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_types.cuh"

namespace epg {


struct LayoutParams {
  const int64_t* topk_idx;   // [N, K]
  int num_tokens;            // N
  int topk;                  // K
  int world_size;            // W
  int max_tok_per_rank;      // T
  int num_expert_per_rank;   // Epr
  int num_experts;           // E
  int alignment;             // A
  int64_t rcap;              // receive capacity (rows of meta)
  int no_expand;             // 1: one row per (token, rank) (EPHandle do_expand = false)
  int num_chunks;            // C = ceil(N / kLayoutTPC)
  // outputs (handle)
  int32_t* cnt;              // [E]
  int32_t* tok_per_rank;     // [W]
  int32_t* psum_expert;      // [E+1]
  int32_t* psum_rank;        // [W+1]
  int32_t* num_recv;         // [1]
  int32_t* dst_slot;         // [N, K]
  int32_t* send_slot;        // [N, K] non-expand: the token's distinct rows, ascending
  int32_t* meta;             // [rcap, K+2]
  int32_t* err;              // [1]
  int32_t* topk_i32;         // [N, K] clone of the ids (-1 where skipped), or nullptr
  uint32_t epr_magic;        // RankMagic(num_expert_per_rank)
  // scratch (BindLayoutScratch): per-chunk column histograms, row-major [C][E+W]
  // (a chunk's row is contiguous: written by count, read by slots), the same
  // counts column-major [E+W][C] (a column is contiguous: read by the spine),
  // and the exclusive prefix over chunks, row-major [C][E+W]
  int32_t* chunk_hist;
  int32_t* chunk_hist_cols;
  int32_t* chunk_off;
  int32_t* col_total;        // [E+W]
  // state of the single-launch fused layout (BindLayoutFusedState; all nullptr:
  // that path is not used).  EW8 = E+W rounded up to a multiple of 8.
  uint32_t* fused_bar;       // [3] grid-barrier arrivals, their count when the launch began, launches so far
  int32_t* fused_super;      // [2][fused_super_rows][EW8] superchunk sums, by launch parity
  uint16_t* fused_rows;      // [max chunks][EW8] per-range column counts
  int fused_super_rows;      // superchunk rows of one parity
  int fused_max_ranges;      // ranges (CTAs) the state holds
  int fused_tpb;             // tokens per CTA of the fused kernel (set by the launcher)
  uint64_t wait_ns;          // bound of the fused kernel's grid-barrier wait
};

// Launch geometry of a variant on the current device, filled by its prepare
// function when a handle is built.
struct LaunchGeom {
  int num_sms;        // SMs of the device
  int blocks_per_sm;  // resident CTAs per SM for the variant's block and shared memory
  int cluster_ok;     // layout: the single-launch cluster kernel can be scheduled
  int row_slices;     // dispatch: CTAs per token row forced by EP_GB300_DISPATCH_SLICES (0: table)
  int pdl;            // dispatch / combine: launched with programmatic stream serialisation
  // layout only: experts and ranks of the handle (set before prepare; 0 when
  // unknown) and the fused kernel's resident CTAs per SM for them (0: that path
  // is off, by EP_GB300_LAYOUT_FUSED=0 or because it does not fit)
  int layout_experts;
  int layout_world;
  int fused_blocks_per_sm;
  int fused_tpb;      // tokens per CTA of the fused kernel (0: chosen per launch)
  int fused_max_super;  // superchunk rows the fused kernel's staging is sized for
};

// Programmatic dependent launch of the data kernels, unless EP_GB300_PDL=0
// (read when a handle is built; for A/B measurements).
bool PdlEnabled();

// Launch `kernel(p)` on `s`, with programmatic stream serialisation when `pdl`:
// the kernel may then be scheduled while the preceding kernel of the stream
// drains; it waits for that kernel's completion (grid_dependency_wait) before
// it touches memory.
template <class P>
cudaError_t LaunchData(void (*kernel)(P), int grid, int block, cudaStream_t s, const P& p, int pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

using LayoutLaunch = cudaError_t (*)(const LayoutParams&, const LaunchGeom&, cudaStream_t);
using DispatchLaunch = cudaError_t (*)(const DispatchParams&, const LaunchGeom&, cudaStream_t);
using CombineLaunch = cudaError_t (*)(const CombineParams&, const LaunchGeom&, cudaStream_t);
// Per-device set-up of a variant (shared-memory opt-in, occupancy).  `aux` is
// E+W for the layout and unused elsewhere.
using PrepareFn = cudaError_t (*)(int hidden, int topk, int aux, LaunchGeom* geom);

template <class F>
struct Variant {
  const char* name;
  F launch;
  PrepareFn prepare;
};

Variant<LayoutLaunch> FindLayout(int topk, bool no_expand);
// Which kernels a layout launch with these parameters runs: the single-launch
// cluster kernel (small batches), the single-launch fused kernel (a
// cooperative grid, mid-size batches) or count / spine / slots.
enum class LayoutPath { kLaunches = 0, kCluster = 1, kFused = 2 };
LayoutPath LayoutPathOf(const LayoutParams& p, const LaunchGeom& g);
Variant<DispatchLaunch> FindDispatch(int hidden, int topk, EpDType dtype);
// The dispatch that stages rows through shared memory with TMA bulk copies
// (byte-copy transports; null launch when the dtype or the row size is not
// served), requested by EP_GB300_DISPATCH_TMA=1.
Variant<DispatchLaunch> FindDispatchTma(EpDType dtype, int row_bytes);
bool DispatchTmaRequested();
// Bound of a device-side wait in ns: EP_GB300_WAIT_NS, else kDefaultWaitNs.
uint64_t WaitLimitNs();
Variant<CombineLaunch> FindCombine(int hidden, int topk, bool use_weights);
// The combine that stages the K expert rows of a token through shared memory
// with TMA bulk copies (bf16 output, no bias; null launch when the row cannot
// be cut into 16-byte pieces), requested by EP_GB300_COMBINE_TMA=1.
Variant<CombineLaunch> FindCombineTma(int hidden, int topk, bool use_weights);
bool CombineTmaRequested();

// int32 words of layout scratch for up to max_chunks chunks and `columns` = E+W
// columns: [chunk_hist] [chunk_hist_cols] [chunk_off], each columns x max_chunks,
// then [columns] totals.
int64_t LayoutScratchInts(int max_chunks, int columns);
// Point p's scratch fields into `base` (LayoutScratchInts(max_chunks, columns) words).
void BindLayoutScratch(LayoutParams* p, int32_t* base, int max_chunks, int columns);
// int32 words of the fused layout's state for up to max_chunks ranges of
// kLayoutTPC tokens and `columns` = E+W columns (0 when max_chunks exceeds
// what a cooperative grid can hold: that path is then never taken).
int64_t LayoutFusedStateInts(int max_chunks, int columns);
// Point p's fused-state fields into `base` (LayoutFusedStateInts words, zeroed
// once when allocated; the kernel keeps it consistent from launch to launch).
void BindLayoutFusedState(LayoutParams* p, int32_t* base, int max_chunks, int columns);
// Magic multiplier for dividing an expert id by num_expert_per_rank on the device.
uint32_t RankMagic(int num_expert_per_rank);

// Record `msg` as the calling thread's ep_last_error() and return `code`
// (for entry points defined outside ep_api.cpp).
int RecordError(int code, const char* msg);

}  // namespace epg
