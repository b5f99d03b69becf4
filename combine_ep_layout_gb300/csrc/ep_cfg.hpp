// ep_cfg.hpp -- compile-time configuration of the kernels and the arithmetic
// that host and device share.
//
// Mirrors the design of "MORI JIT v2" §3.1-§3.5: the configuration is one
// named struct used as a non-type template parameter, the kernel's switches
// are `if constexpr` on its fields, and the same constexpr functions size the
// launches on the host and index memory on the device.  Like that page's
// header, this one includes no CUDA header and uses plain constexpr (no
// __host__ __device__), so a host-only compiler accepts it (a test compiles
// it with g++).
//
// What is compile-time here and why: hidden size and top-k set the trip counts
// of the row-copy and reduce loops and every stride the kernels divide or
// multiply by ("MORI JIT v2" §8: integer divides 41 -> 3 and 57 -> 10 once the
// shape is a compile-time constant); dtype and useWeights select code paths.
// World size, tokens per rank, experts and alignment stay runtime arguments:
// they only enter the layout, which is integer work on a few MB.
#pragma once

#if defined(__CUDACC_RTC__)
// NVRTC compiles the kernel bodies at run time without the C library headers.
typedef signed char int8_t;
typedef unsigned char uint8_t;
typedef short int16_t;
typedef unsigned short uint16_t;
typedef int int32_t;
typedef unsigned int uint32_t;
typedef long long int64_t;
typedef unsigned long long uint64_t;
typedef unsigned long long uintptr_t;
#else
#include <cstdint>
#endif

namespace epg {

// Transport dtype ("MORI JIT v2" §3.7 numbering).
enum class EpDType : int { Bf16 = 0, Fp32 = 1, Fp8 = 2, Fp4x2 = 3 };

// The compile-time shape of one kernel variant.  hidden == 0 or topk == 0
// means "runtime value" (the generic variant that serves shapes for which no
// specialisation was compiled).
struct EpShape {
  int hidden;       // H, channels per row
  int topk;         // K
  EpDType dtype;    // dispatch transport dtype (combine always reduces bf16)
  bool useWeights;  // combine: weighted by topk_weights
};

// Field-count guard: adding a field to EpShape without revisiting the variant
// naming and registry below stops this from compiling (a structured binding
// must name every member).
constexpr int EpShapeFieldCount() {
  auto [h, k, d, w] = EpShape{0, 0, EpDType::Bf16, false};
  (void)h; (void)k; (void)d; (void)w;
  return 4;
}
static_assert(EpShapeFieldCount() == 4, "EpShape changed: update the variant table and names");

// ---- shared arithmetic ------------------------------------------------------

constexpr int kScaleGroup = 128;   // channels per FP8 scale

constexpr int64_t RowBytes(int hidden, EpDType dt) {
  return dt == EpDType::Bf16 ? 2LL * hidden
       : dt == EpDType::Fp32 ? 4LL * hidden
       : dt == EpDType::Fp8  ? 1LL * hidden
                             : (hidden + 1) / 2;
}

constexpr int ScaleGroups(int hidden) { return hidden / kScaleGroup; }

constexpr int64_t AlignUp(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Rows of the receive buffer for any routing of max_tokens tokens.
constexpr int64_t RecvCapacity(int64_t max_tokens, int topk, int num_experts, int alignment) {
  return max_tokens * topk + (int64_t)num_experts * (alignment - 1);
}

// Rows of the non-expand receive buffer (one per (token, destination rank)):
// a token reaches at most min(K, W) ranks.
constexpr int64_t RecvCapacityNonExpand(int64_t max_tokens, int topk, int world_size) {
  return max_tokens * (topk < world_size ? topk : world_size);
}

// Threads per CTA of the row kernels for a row of `chunks` vectors: the largest
// multiple of 32 that divides it and is at most 256 (every thread owns the same
// number of vectors, at most 8); 0 when there is none (the row is walked in a
// loop by kRowLoopThreads-or-fewer threads).
constexpr int kRowMaxThreads = 256;
constexpr int RowThreads(int chunks) {
  for (int t = kRowMaxThreads; t >= 32; t -= 32)
    if (chunks % t == 0 && chunks / t <= 8) return t;
  return 0;
}

// Minimum resident CTAs per SM asked of the compiler for the copy kernel of
// rows of rb bytes (v words per vector, s CTAs per row).  When a thread holds at
// most 16 words of the row, 32 registers suffice and the whole SM (65536
// registers) can be filled; stating that keeps the compiler from trading a
// register for a spill.  The count is capped at the SM's 32 resident CTAs
// (small rows take small CTAs).  Larger per-thread shares, and the loop
// variant, are left to the compiler (1).
constexpr int kMaxCtasPerSm = 32;
constexpr int CopyMinBlocks(int rb, int v, int s = 1) {
  return rb && RowThreads(rb / (4 * v) / s) &&
                 (rb / (4 * v) / s / RowThreads(rb / (4 * v) / s)) * v <= 16
             ? (65536 / (32 * RowThreads(rb / (4 * v) / s)) < kMaxCtasPerSm
                    ? 65536 / (32 * RowThreads(rb / (4 * v) / s))
                    : kMaxCtasPerSm)
             : 1;
}

// Layout chunking: the count and slot kernels give each CTA kLayoutTPC tokens.
constexpr int kLayoutTPC = 128;
constexpr int kLayoutCountWarps = 16;
constexpr int NumLayoutChunks(int num_tokens) { return (num_tokens + kLayoutTPC - 1) / kLayoutTPC; }

// Limits checked when a handle is built ("MORI JIT v2" §3.5: a configuration
// that cannot be served is a construction-time error).
constexpr int kMaxWorld = 64;       // rank sets are 64-bit masks
constexpr int kMaxExperts = 2048;   // per-warp histograms live in shared memory
constexpr int kMaxTopk = 16;
constexpr int kMaxAlignment = 4096;
constexpr int kMaxHidden = 32768;   // a bf16 row must fit twice in shared memory
constexpr int64_t kMaxTokens = 1LL << 24;

// The specialisations compiled into the library: (hidden, topk) pairs.  Each
// one is instantiated for bf16 dispatch, FP8 dispatch and both combine modes.
// Shapes outside the list run the generic variant of the same kernels.
#define EPG_SHAPE_LIST(X) \
  X(1024, 4)              \
  X(2048, 8)              \
  X(4096, 6)              \
  X(4096, 8)              \
  X(5120, 8)              \
  X(6144, 8)              \
  X(7168, 4)              \
  X(7168, 6)              \
  X(7168, 8)              \
  X(8192, 8)

}  // namespace epg
