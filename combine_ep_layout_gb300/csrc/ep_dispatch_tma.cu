// ep_dispatch_tma.cu -- dispatch with the rows staged through shared memory by
// the TMA unit (cp.async.bulk), for the byte-copy transports (bf16, fp32,
// packed fp4).  Selected with EP_GB300_DISPATCH_TMA=1 when a handle is built;
// the register copy of ep_dispatch.cu is the default because it is faster on
// GB300 (the TMA ring levels off near 6.0 TB/s on the prefill shape, the
// register copy reaches the device's copy rate).
//
// One warp per CTA and a grid of (SMs x resident CTAs), each CTA taking a
// contiguous run of tokens.  Lane 0 keeps a ring of S row buffers in shared
// memory: a bulk load brings token j's row in (completion counted on the
// stage's mbarrier), then K bulk stores copy the buffer to the token's K
// receive rows (one bulk group per token).  A stage is refilled with token
// j - 1 + S once the stores of token j - 1 have finished reading it, so one
// token's stores and S - 1 loads are in flight behind the current token.
//
// Every wait on an mbarrier is bounded by %globaltimer (DispatchParams::wait_ns):
// past the limit the kernel records kErrTimeout (value 2) in the device error
// word, waits (again bounded) for the loads it has issued so that no copy is
// left writing into its shared memory, drains its stores and returns.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "ep_cfg.hpp"
#include "ep_dispatch_body.cuh"
#include "ep_kernels.hpp"
#include "ep_tma.cuh"

namespace epg {
namespace {

constexpr int kTmaMaxStages = 4;
constexpr size_t kTmaSmemLimit = 227 * 1024;      // dynamic shared memory a CTA may opt into

using namespace tma;

constexpr uint32_t AlignRow(uint32_t row) { return (row + 127u) & ~127u; }

// Ring stages for rows of row_bytes: as many as fit (at most kTmaMaxStages);
// fewer than 2 cannot keep a load ahead of the stores (then 0: not served).
int tma_stages(int row_bytes) {
  const size_t per = AlignRow(static_cast<uint32_t>(row_bytes)) + 8;
  int st = static_cast<int>(kTmaSmemLimit / per);
  st = st > kTmaMaxStages ? kTmaMaxStages : st;
  return st >= 2 ? st : 0;
}

size_t tma_smem(int row_bytes, int stages) {
  return static_cast<size_t>(AlignRow(static_cast<uint32_t>(row_bytes))) * stages + 8 * stages;
}

__global__ void __launch_bounds__(32, 1) ep_dispatch_tma_kernel(DispatchParams p, int per, int S) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x;
  const uint32_t row = static_cast<uint32_t>(p.row_bytes);
  const uint32_t stride = AlignRow(row);
  const uint32_t bufs = smem_u32(smem);
  const uint32_t bars = bufs + stride * S;
  const int K = p.topk;
  const int t0 = blockIdx.x * per;
  const int n = min(p.num_tokens, t0 + per) - t0;
  if (n <= 0) return;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
    mbar_init_fence();
  }
  __syncwarp();
  allow_dependent_grids();
  grid_dependency_wait();  // dst_slot (and x) may be outputs of the preceding grid

  const uint8_t* x = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t0) * row;
  uint8_t* rx = static_cast<uint8_t*>(p.recv_x);
  int issued = 0;  // loads issued (tokens [0, issued) of the run)
  auto load = [&](int j) {
    const uint32_t bar = bars + 8 * (j % S);
    mbar_expect_tx(bar, row);
    bulk_load(bufs + stride * (j % S), x + static_cast<int64_t>(j) * row, row, bar);
  };
  if (lane == 0)
    for (int j = 0; j < min(n, S); ++j) load(j);
  issued = min(n, S);

  int j = 0;
  bool timed_out = false;
  for (; j < n; ++j) {
    const int s = j % S;
    const uint32_t parity = static_cast<uint32_t>(j / S) & 1u;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(bars + 8 * s, parity, p.wait_ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      timed_out = true;
      break;
    }
    const int t = t0 + j;
    const int32_t d = lane < K ? ld_coherent(p.dst_slot + static_cast<int64_t>(t) * K + lane) : -1;
    for (int k = 0; k < K; ++k) {
      const int32_t dk = __shfl_sync(0xffffffffu, d, k);
      if (lane == 0 && dk >= 0) bulk_store(rx + static_cast<int64_t>(dk) * row, bufs + stride * s, row);
    }
    if (lane == 0) {
      bulk_commit();
      // token j - 1's stores have read their stage: refill it
      const int next = j - 1 + S;
      if (j >= 1 && next < n) {
        bulk_wait_read<1>();
        load(next);
      }
    }
    if (j >= 1 && j - 1 + S < n) ++issued;
    forward_routing(p, t, K, p.dst_slot + static_cast<int64_t>(t) * K);
  }
  if (timed_out) {
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      // no load may still be writing into this CTA's shared memory when it exits
      for (int jj = j; jj < issued; ++jj)
        mbar_wait_bounded(bars + 8 * (jj % S), static_cast<uint32_t>(jj / S) & 1u, kDrainNs);
    }
    __syncwarp();
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

cudaError_t launch_tma(const DispatchParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  const int slots = g.num_sms * (g.blocks_per_sm > 0 ? g.blocks_per_sm : 1);
  const int per = (p.num_tokens + slots - 1) / slots;
  const int grid = (p.num_tokens + per - 1) / per;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(32);
  const int stages = tma_stages(p.row_bytes);
  cfg.dynamicSmemBytes = tma_smem(p.row_bytes, stages);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, ep_dispatch_tma_kernel, p, per, stages);
}

cudaError_t prepare_tma(int, int, int row_bytes, LaunchGeom* g) {
  g->pdl = PdlEnabled() ? 1 : 0;
  const size_t smem = tma_smem(row_bytes, tma_stages(row_bytes));
  cudaError_t e = cudaFuncSetAttribute(ep_dispatch_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g->blocks_per_sm, ep_dispatch_tma_kernel, 32, smem);
}

}  // namespace

bool DispatchTmaRequested() {
  const char* env = std::getenv("EP_GB300_DISPATCH_TMA");
  return env != nullptr && env[0] == '1';
}

uint64_t WaitLimitNs() {
  const char* env = std::getenv("EP_GB300_WAIT_NS");
  if (env == nullptr || env[0] == '\0') return kDefaultWaitNs;
  return std::strtoull(env, nullptr, 10);
}

Variant<DispatchLaunch> FindDispatchTma(EpDType dtype, int row_bytes) {
  if (tma_stages(row_bytes) == 0) return {nullptr, nullptr, nullptr};
  switch (dtype) {
    case EpDType::Bf16: return {"ep_dispatch_tma_bf16", launch_tma, prepare_tma};
    case EpDType::Fp32: return {"ep_dispatch_tma_fp32", launch_tma, prepare_tma};
    case EpDType::Fp4x2: return {"ep_dispatch_tma_fp4x2", launch_tma, prepare_tma};
    default: return {nullptr, nullptr, nullptr};
  }
}

}  // namespace epg
