// ep_layout_noalloc.cu -- the layout for callers that cannot allocate device
// memory.
//
// ep_handle_create allocates (cudaMallocAsync) the handle's outputs and the
// layout's scratch: per-chunk expert/rank histograms and their prefix sums
// over chunks.  Some callers cannot make that call.  A framework that hands
// all device memory to its own caching pool may not allow an extra cudaMalloc
// beside it.  A serving loop that has to keep its memory fixed after start-up
// may not allocate per request.  Code that is only given buffers, with no
// allocator in reach, cannot allocate at all.  ep_layout_noalloc serves
// them.  The caller passes every output buffer.  The scratch is one
// fixed-size array compiled into this file as a file-scope __device__
// variable.  Nothing here calls cudaMalloc, cudaFree or any library routine
// that allocates.
//
// The array costs every GPU that loads the library kNoAllocScratchInts * 4
// bytes (1 MiB) until the process exits.  Its device address is looked up per
// device (cudaGetSymbolAddress, with that device current) by the first call
// made while that device is current; the same set-up also sets the layout
// kernels' shared-memory limit, so that first call should come before any
// stream capture.  The set-up is recorded only when it succeeds (a failed one
// is retried by the next call) and is tied to the device's current CUDA
// context: after cudaDeviceReset, or under another context, it runs again,
// so no call launches with an address or a limit of a context that is gone.
//
// All calls share the one array and it keeps whatever the last call left
// there.  The layout kernels write every scratch entry they later read, so no
// part of it has to start at zero.  Two calls that can run at the same time on
// the GPU (different streams, no ordering between them) overwrite each
// other's scratch and give wrong results: order them, e.g. on one stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "ep_cfg.hpp"
#include "ep_gb300.h"
#include "ep_kernels.hpp"

namespace epg {
namespace {

constexpr int64_t kNoAllocScratchInts = 1 << 18;  // 262144 int32 = 1 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

struct DeviceSetup {
  bool done = false;
  unsigned long long ctx_id = 0;  // CUDA context the set-up was made in
  int32_t* scratch = nullptr;     // device address of g_noalloc_scratch in that context
  int num_sms = 0;
  int cluster_ok = 1;             // every layout variant can run its single-launch cluster kernel
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kNoAllocMaxDevices];

// Unique id of the calling thread's current CUDA context (cuCtxGetCurrent +
// cuCtxGetId, reached through the runtime so that nothing links the driver
// library directly).  A new context -- after cudaDeviceReset, say -- has a new id.
cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
    if (e != cudaSuccess) return e;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess) return e;
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    get_current = reinterpret_cast<GetCurrent>(f1);
    get_id = reinterpret_cast<GetId>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Per-device set-up, with that device current: the scratch address and the
// layout kernels' shared-memory opt-in.  Fills *s only when every step succeeds.
cudaError_t setup_device(int dev, unsigned long long ctx_id, DeviceSetup* s) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // shared-memory opt-in of every layout variant, sized for the largest E+W
  int cluster_ok = 1;
  const int topks[] = {4, 6, 8, 0};
  for (int k : topks) {
    LaunchGeom g{sms, 1};
    if ((e = FindLayout(k, false).prepare(0, k, kMaxExperts + kMaxWorld, &g)) != cudaSuccess) return e;
    cluster_ok &= g.cluster_ok;
  }
  s->scratch = static_cast<int32_t*>(p);
  s->num_sms = sms;
  s->cluster_ok = cluster_ok;
  s->ctx_id = ctx_id;
  s->done = true;
  return cudaSuccess;
}

int err_cuda(cudaError_t e, const char* what) {
  char buf[256];
  std::snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return RecordError(EP_ECUDA, buf);
}

}  // namespace
}  // namespace epg

using namespace epg;

extern "C" int ep_layout_noalloc(const ep_cfg_t* cfg, const int64_t* topk_idx, int32_t num_tokens,
                                 int32_t* num_unaligned_per_expert, int32_t* num_tokens_per_rank,
                                 int32_t* psum_per_expert, int32_t* psum_per_rank,
                                 int32_t* num_recv, int32_t* dst_slot, int32_t* recv_src_metadata,
                                 int32_t* device_error, ep_stream_t stream) noexcept {
  try {
    const int64_t rcap = ep_recv_capacity(cfg);  // validates cfg and records the message
    if (rcap < 0) return static_cast<int>(rcap);
    if (cfg->no_expand)
      return RecordError(EP_EUNSUPPORTED, "ep_layout_noalloc serves the expand layout only");
    const int W = cfg->world_size, E = W * cfg->num_expert_per_rank, K = cfg->num_expert_per_token;
    const int64_t max_tokens = static_cast<int64_t>(W) * cfg->max_tok_per_rank;
    if (num_tokens < 0 || num_tokens > max_tokens)
      return RecordError(EP_EINVAL, "num_tokens must be in [0, world_size*max_tok_per_rank]");
    const int cols = E + W;
    const int C = NumLayoutChunks(num_tokens);
    const int64_t need = LayoutScratchInts(C, cols);
    if (need > kNoAllocScratchInts) {
      char buf[320];
      std::snprintf(buf, sizeof buf,
                    "ep_layout_noalloc: %d tokens over %d experts + %d ranks need %lld int32 of "
                    "scratch (3*(E+W)*ceil(N/%d) + (E+W)); the static scratch holds %lld",
                    num_tokens, E, W, static_cast<long long>(need), kLayoutTPC,
                    static_cast<long long>(kNoAllocScratchInts));
      return RecordError(EP_EINVAL, buf);
    }
    if (!num_unaligned_per_expert || !num_tokens_per_rank || !psum_per_expert || !psum_per_rank ||
        !num_recv || !recv_src_metadata || !device_error || (num_tokens > 0 && (!topk_idx || !dst_slot)))
      return RecordError(EP_EINVAL, "ep_layout_noalloc: an input or output pointer is NULL");
    if (num_tokens > 0 && (reinterpret_cast<uintptr_t>(topk_idx) & 7u))
      return RecordError(EP_EINVAL, "topk_idx must be 8-byte aligned");
    if ((K + 2) % 2 == 0 && (reinterpret_cast<uintptr_t>(recv_src_metadata) & 7u))
      return RecordError(EP_EINVAL, "recv_src_metadata must be 8-byte aligned");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return err_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoAllocMaxDevices)
      return RecordError(EP_EUNSUPPORTED, "ep_layout_noalloc: device ordinal above 63");
    unsigned long long ctx_id = 0;
    if ((e = current_context_id(&ctx_id)) != cudaSuccess) return err_cuda(e, "current CUDA context");
    DeviceSetup setup;
    {
      std::lock_guard<std::mutex> lock(g_setup_mutex);
      DeviceSetup* s = &g_setup[dev];
      if (!s->done || s->ctx_id != ctx_id) {
        DeviceSetup fresh;
        if ((e = setup_device(dev, ctx_id, &fresh)) != cudaSuccess) {
          cudaGetLastError();
          return err_cuda(e, "ep_layout_noalloc set-up");
        }
        *s = fresh;
      }
      setup = *s;
    }

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((e = cudaMemsetAsync(device_error, 0, sizeof(int32_t), st)) != cudaSuccess)
      return err_cuda(e, "cudaMemsetAsync");
    const int Cs = C > 0 ? C : 1;
    LayoutParams p{};
    p.topk_idx = topk_idx;
    p.num_tokens = num_tokens;
    p.topk = K;
    p.world_size = W;
    p.max_tok_per_rank = cfg->max_tok_per_rank;
    p.num_expert_per_rank = cfg->num_expert_per_rank;
    p.num_experts = E;
    p.alignment = cfg->expert_alignment;
    p.rcap = rcap;
    p.num_chunks = C;
    p.cnt = num_unaligned_per_expert;
    p.tok_per_rank = num_tokens_per_rank;
    p.psum_expert = psum_per_expert;
    p.psum_rank = psum_per_rank;
    p.num_recv = num_recv;
    p.dst_slot = dst_slot;
    p.meta = recv_src_metadata;
    p.err = device_error;
    p.epr_magic = RankMagic(cfg->num_expert_per_rank);
    BindLayoutScratch(&p, setup.scratch, Cs, cols);
    const LaunchGeom g{setup.num_sms, 1, setup.cluster_ok, 0};
    if ((e = FindLayout(K, false).launch(p, g, st)) != cudaSuccess) return err_cuda(e, "layout launch");
    return EP_OK;
  } catch (...) {
    return RecordError(EP_EINVAL, "unknown exception");
  }
}
