// ep_combine_tma.cu -- combine with each token's K expert rows staged in
// shared memory by the TMA unit (cp.async.bulk), for bf16 output without bias
// ("Combine data flow" of "DeepEP overall architecture analysis": gather the
// expert outputs of a token and reduce them weighted by topk_weights).
// Selected with EP_GB300_COMBINE_TMA=1 when a handle is built; the register
// combine of ep_combine.cu stays the default and serves the bias and fp32
// outputs.
//
// One CTA per (token, piece of its row): the row is cut into P equal pieces,
// P the smallest power of two for which the K pieces of one token take at most
// kCombineTmaStageBytes of shared memory, so that many CTAs per SM keep their
// copies in flight while others fold.  Thread 0 issues one bulk copy per
// routed entry (its piece of that expert row), all completing on one
// mbarrier, and waits on it, bounded by %globaltimer (CombineParams::wait_ns);
// after a block barrier every thread folds the K pieces from shared memory in
// k order with the register combine's arithmetic (fp32 fmaf from +0, masked
// entries skipped, bf16 round to nearest even) and stores its 16-byte output
// vectors.  A CTA whose wait gives up records kErrTimeout (value 2) in the
// device error word, lets its copies land (again bounded) and stores nothing.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "ep_cfg.hpp"
#include "ep_combine_body.cuh"
#include "ep_kernels.hpp"
#include "ep_tma.cuh"

namespace epg {
namespace {

using namespace tma;

// 128 threads and at most 16 KB of pieces per CTA (the prefill row of 14336
// bytes in 8 pieces of 1792): measured best of 64 / 128 / 256 threads and
// 4-120 KB per CTA (prefill combine 606 us at 16 KB, 647 at 32 KB, 762 at
// 8 KB; 256 threads: 761 at 16 KB, 614 at 32 KB).
constexpr int kCombineTmaThreads = 128;
constexpr int kCombineTmaStageBytes = 16 * 1024;

// Pieces per row for rows of row_bytes and K entries (0: no cut gives 16-byte
// pieces that fit).
int combine_pieces(int row_bytes, int K) {
  for (int P = 1; P <= row_bytes / 16; P *= 2) {
    if (row_bytes % P != 0 || (row_bytes / P) % 16 != 0) return 0;
    if (static_cast<int64_t>(K) * (row_bytes / P) <= kCombineTmaStageBytes) return P;
  }
  return 0;
}

__global__ void __launch_bounds__(kCombineTmaThreads) ep_combine_tma_kernel(CombineParams p, int P, int piece) {
  extern __shared__ __align__(128) uint8_t stage[];   // [K][piece]
  __shared__ int32_t slot_s[kMaxTopk];
  __shared__ float w_s[kMaxTopk];
  __shared__ __align__(8) uint64_t bar_s;
  const int K = p.topk;
  const int t = static_cast<int>(blockIdx.x) / P;
  const int q = static_cast<int>(blockIdx.x) - t * P;
  const bool weighted = p.weights != nullptr;
  const uint32_t bar = smem_u32(&bar_s);
  // y, dst_slot and the weights may be outputs of the preceding grid
  allow_dependent_grids();
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init_fence();
  }
  if (static_cast<int>(threadIdx.x) < K) {
    slot_s[threadIdx.x] = ld_coherent(p.dst_slot + static_cast<int64_t>(t) * K + threadIdx.x);
    w_s[threadIdx.x] = weighted ? ld_coherent(p.weights + static_cast<int64_t>(t) * K + threadIdx.x) : 1.0f;
  }
  __syncthreads();  // the mbarrier is initialised; slots and weights are visible
  const int64_t row = 2 * static_cast<int64_t>(p.hidden);
  if (threadIdx.x == 0) {
    uint32_t bytes = 0;
    for (int k = 0; k < K; ++k) bytes += slot_s[k] >= 0 ? static_cast<uint32_t>(piece) : 0u;
    mbar_expect_tx(bar, bytes);
    const uint8_t* y = static_cast<const uint8_t*>(p.y) + static_cast<int64_t>(q) * piece;
    for (int k = 0; k < K; ++k)
      if (slot_s[k] >= 0)
        bulk_load(smem_u32(stage + k * piece), y + static_cast<int64_t>(slot_s[k]) * row,
                  static_cast<uint32_t>(piece), bar);
  }
  // thread 0 waits for the copies; the block barrier then orders every
  // thread's reads of the staged pieces after the copies' completion
  const bool ok = threadIdx.x != 0 || mbar_wait_bounded(bar, 0, p.wait_ns);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) {
      atomicOr(p.err, kErrTimeout);
      mbar_wait_bounded(bar, 0, kDrainNs);  // no copy may still write into this CTA's shared memory
    }
    return;
  }
  uint8_t* out = static_cast<uint8_t*>(p.out) + static_cast<int64_t>(t) * row + static_cast<int64_t>(q) * piece;
  for (int v = threadIdx.x; v < piece / 16; v += kCombineTmaThreads) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int k = 0; k < K; ++k) {
      if (slot_s[k] < 0) continue;
      const uint4 u = *reinterpret_cast<const uint4*>(stage + k * piece + v * 16);
      Vec<4> r;
      r.w[0] = u.x;
      r.w[1] = u.y;
      r.w[2] = u.z;
      r.w[3] = u.w;
      fold<4>(acc, r, w_s[k], weighted);
    }
    Vec<4> o;
#pragma unroll
    for (int i = 0; i < 4; ++i) o.w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    st_stream<4>(out + v * 16, o);
  }
}

cudaError_t launch_combine_tma(const CombineParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  const int row = 2 * p.hidden;
  const int P = combine_pieces(row, p.topk);
  if (P == 0) return cudaErrorInvalidConfiguration;   // FindCombineTma serves no such shape
  const int piece = row / P;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.num_tokens) * static_cast<unsigned>(P));
  cfg.blockDim = dim3(kCombineTmaThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.topk) * piece;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, ep_combine_tma_kernel, p, P, piece);
}

cudaError_t prepare_combine_tma(int, int, int, LaunchGeom* g) {
  g->pdl = PdlEnabled() ? 1 : 0;
  cudaError_t e = cudaFuncSetAttribute(ep_combine_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kCombineTmaStageBytes);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g->blocks_per_sm, ep_combine_tma_kernel,
                                                       kCombineTmaThreads, kCombineTmaStageBytes);
}

}  // namespace

bool CombineTmaRequested() {
  const char* env = std::getenv("EP_GB300_COMBINE_TMA");
  return env != nullptr && env[0] == '1';
}

Variant<CombineLaunch> FindCombineTma(int hidden, int topk, bool use_weights) {
  if (combine_pieces(2 * hidden, topk) == 0) return {nullptr, nullptr, nullptr};
  return {use_weights ? "ep_combine_tma_w" : "ep_combine_tma", launch_combine_tma, prepare_combine_tma};
}

}  // namespace epg
