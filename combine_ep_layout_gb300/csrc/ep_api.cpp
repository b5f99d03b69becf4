// ep_api.cpp -- the C ABI of libep_gb300.so (declared in include/ep_gb300.h).
//
// Conventions from "MORI JIT v2": every entry point is noexcept and reports
// errors as a negative return code plus a thread-local message (§6: an
// exception crossing extern "C" would take the interpreter down); a
// configuration the kernels cannot serve is rejected when the handle is built
// (§3.5, §5 "capability gate at construction, before allocation"); the
// variant for a configuration is picked from a table of compiled
// specialisations keyed by its shape (§5.1), never compiled on the hot path.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <exception>
#include <string>

#include "ep_cfg.hpp"
#include "ep_gb300.h"
#include "ep_jit.hpp"
#include "ep_kernels.hpp"

using namespace epg;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(EP_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                            cudaGetErrorString(e) + ")");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks of "MORI JIT v2" §3.5 (token bytes 16-byte aligned; receive capacity
// covers the worst case) plus this library's own limits.
int validate(const ep_cfg_t* c) {
  if (!c) return fail(EP_EINVAL, "cfg is NULL");
  if (c->world_size < 1 || c->world_size > kMaxWorld)
    return fail(EP_EINVAL, "world_size must be in [1, 64]");
  if (c->max_tok_per_rank < 1) return fail(EP_EINVAL, "max_tok_per_rank must be >= 1");
  const int64_t max_tokens = static_cast<int64_t>(c->world_size) * c->max_tok_per_rank;
  if (max_tokens > kMaxTokens) return fail(EP_EINVAL, "world_size*max_tok_per_rank exceeds 2^24");
  if (c->num_expert_per_rank < 1) return fail(EP_EINVAL, "num_expert_per_rank must be >= 1");
  const int64_t E = static_cast<int64_t>(c->world_size) * c->num_expert_per_rank;
  if (E > kMaxExperts) return fail(EP_EINVAL, "world_size*num_expert_per_rank exceeds 2048");
  if (c->num_expert_per_token < 1 || c->num_expert_per_token > kMaxTopk)
    return fail(EP_EINVAL, "num_expert_per_token must be in [1, 16]");
  if (c->expert_alignment < 1 || c->expert_alignment > kMaxAlignment)
    return fail(EP_EINVAL, "expert_alignment must be in [1, 4096]");
  if (c->hidden_dim < 8 || c->hidden_dim > kMaxHidden || c->hidden_dim % 8 != 0)
    return fail(EP_EINVAL, "hidden_dim must be a multiple of 8 in [8, 32768] (16-byte rows)");
  if (c->use_weights != 0 && c->use_weights != 1) return fail(EP_EINVAL, "use_weights must be 0 or 1");
  if (c->no_expand != 0 && c->no_expand != 1) return fail(EP_EINVAL, "no_expand must be 0 or 1");
  if (c->no_expand && c->use_weights)
    return fail(EP_EINVAL,
                "the non-expand layout combines rank rows unweighted: use_weights must be 0 with no_expand");
  switch (c->dispatch_dtype) {
    case EP_BF16: break;
    case EP_FP8_E4M3:
      if (c->hidden_dim % kScaleGroup != 0)
        return fail(EP_EINVAL, "FP8 dispatch needs hidden_dim % 128 == 0 (one scale per 128 channels)");
      break;
    case EP_FP32: break;
    case EP_FP4X2:
      if (c->hidden_dim % 32 != 0)
        return fail(EP_EINVAL, "FP4x2 transport needs hidden_dim % 32 == 0 (16-byte rows of H/2 bytes)");
      break;
    default: return fail(EP_EINVAL, "unknown dispatch_dtype");
  }
  const int64_t rcap = RecvCapacity(max_tokens, c->num_expert_per_token, static_cast<int>(E),
                                    c->expert_alignment);
  if (rcap > INT32_MAX) return fail(EP_EINVAL, "receive capacity exceeds int32 rows");
  return EP_OK;
}

// Receive rows of a valid configuration: per (token, expert) plus padding for
// the expand layout, per (token, rank) for the non-expand layout.
int64_t recv_rows(const ep_cfg_t* c) {
  const int64_t max_tokens = static_cast<int64_t>(c->world_size) * c->max_tok_per_rank;
  if (c->no_expand) return RecvCapacityNonExpand(max_tokens, c->num_expert_per_token, c->world_size);
  return RecvCapacity(max_tokens, c->num_expert_per_token, c->world_size * c->num_expert_per_rank,
                      c->expert_alignment);
}

}  // namespace

int epg::RecordError(int code, const char* msg) { return fail(code, msg ? msg : ""); }

struct ep_handle {
  ep_cfg_t cfg;
  int device = -1;
  int W = 0, T = 0, Epr = 0, E = 0, K = 0, H = 0, A = 0;
  int64_t max_tokens = 0, rcap = 0;
  int max_chunks = 0;
  int num_tokens = 0;
  cudaStream_t last_stream = nullptr;  // stream of the last call that enqueued work
  bool launched = false;               // some call enqueued work on last_stream
  // private non-blocking stream on which the metadata block is allocated,
  // cleared and freed (stream-ordered allocator: no device-wide synchronisation)
  cudaStream_t own_stream = nullptr;
  void* block = nullptr;
  bool no_expand = false;
  // non-null: this handle uses the routing of that handle's ep_layout (its own
  // metadata pointers below stay null)
  ep_handle* src = nullptr;
  int32_t *cnt = nullptr, *tok_per_rank = nullptr, *psum_expert = nullptr, *psum_rank = nullptr,
          *num_recv = nullptr, *err = nullptr, *dst_slot = nullptr, *meta = nullptr,
          *topk_i32 = nullptr, *scratch = nullptr, *fused = nullptr;
  // rows each token is written to / read from: dst_slot for the expand layout,
  // the token's distinct rank rows for the non-expand one
  int32_t* send_slot = nullptr;
  Variant<LayoutLaunch> layout{};
  std::string layout_ran;  // kernel name of the last ep_layout (cluster, fused or three launches)
  Variant<DispatchLaunch> dispatch{};
  Variant<CombineLaunch> combine{};
  Variant<CombineLaunch> combine_tma{};   // EP_GB300_COMBINE_TMA=1: rows staged by TMA (bf16 out, no bias)
  LaunchGeom g_layout{}, g_dispatch{}, g_combine{}, g_combine_tma{};
  uint64_t wait_ns = kDefaultWaitNs;  // bound of a device-side wait (EP_GB300_WAIT_NS)
  // run-time specialisations for shapes outside the compiled table (function
  // null when not used); they serve 32-byte-aligned buffers, the compiled
  // generic variant everything else
  jit::Kernel jit_dispatch, jit_combine;
};

namespace {

bool is_generic(const char* name) {
  const size_t n = std::strlen(name);
  return n >= 8 && std::strcmp(name + n - 8, "_generic") == 0;
}

jit::Request dispatch_request(const ep_cfg_t* c) {
  const EpDType dt = static_cast<EpDType>(c->dispatch_dtype);
  if (dt == EpDType::Fp8)
    return {jit::Request::kFp8, 0, c->hidden_dim, c->num_expert_per_token, false};
  return {jit::Request::kCopy, static_cast<int>(RowBytes(c->hidden_dim, dt)), c->hidden_dim,
          c->num_expert_per_token, false};
}

jit::Request combine_request(const ep_cfg_t* c) {
  return {jit::Request::kCombine, 0, c->hidden_dim, c->num_expert_per_token, c->use_weights != 0};
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// The handle whose ep_layout produced the routing h uses.
const ep_handle* owner(const ep_handle* h) { return h->src ? h->src : h; }

int check_device(const ep_handle* h) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(EP_EINVAL, "the current device is not the device the handle was created on");
  return EP_OK;
}

// ep_handle_create (src null) and ep_handle_create_shared (src: the handle
// whose layout the new one uses; nothing of the layout is allocated).
int create_handle(const ep_cfg_t* cfg, ep_handle* src, ep_handle_t* out) {
  try {
    if (!out) return fail(EP_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = validate(cfg);
    if (rc != EP_OK) return rc;
    if (src) {
      const ep_cfg_t& c = src->cfg;
      if (cfg->world_size != c.world_size || cfg->max_tok_per_rank != c.max_tok_per_rank ||
          cfg->num_expert_per_rank != c.num_expert_per_rank ||
          cfg->num_expert_per_token != c.num_expert_per_token ||
          cfg->expert_alignment != c.expert_alignment || cfg->no_expand != c.no_expand)
        return fail(EP_EINVAL,
                    "a shared layout needs the world_size, max_tok_per_rank, num_expert_per_rank, "
                    "num_expert_per_token, expert_alignment and no_expand of layout_src");
      if ((rc = check_device(src)) != EP_OK) return rc;
    }
    ep_handle* h = new ep_handle();
    h->src = src;
    h->cfg = *cfg;
    h->W = cfg->world_size;
    h->T = cfg->max_tok_per_rank;
    h->Epr = cfg->num_expert_per_rank;
    h->E = h->W * h->Epr;
    h->K = cfg->num_expert_per_token;
    h->H = cfg->hidden_dim;
    h->A = cfg->expert_alignment;
    h->max_tokens = static_cast<int64_t>(h->W) * h->T;
    h->no_expand = cfg->no_expand != 0;
    h->rcap = recv_rows(cfg);
    h->max_chunks = NumLayoutChunks(static_cast<int>(h->max_tokens));

    auto bail = [&](int code) {
      if (h->block) {
        cudaFreeAsync(h->block, h->own_stream);
        cudaStreamSynchronize(h->own_stream);
      }
      if (h->own_stream) cudaStreamDestroy(h->own_stream);
      delete h;
      return code;
    };
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) return bail(fail_cuda(e, "cudaGetDevice"));
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) return bail(fail_cuda(e, "cudaDeviceGetAttribute"));

    const EpDType dt = static_cast<EpDType>(cfg->dispatch_dtype);
    const int row_bytes = static_cast<int>(RowBytes(h->H, dt));
    h->layout = FindLayout(h->K, h->no_expand);
    h->dispatch = FindDispatch(h->H, h->K, dt);
    if (DispatchTmaRequested()) {  // rows staged through shared memory by TMA bulk copies
      const Variant<DispatchLaunch> tma = FindDispatchTma(dt, row_bytes);
      if (tma.launch) h->dispatch = tma;
    }
    h->wait_ns = WaitLimitNs();
    h->combine = FindCombine(h->H, h->K, cfg->use_weights != 0);
    if (!h->dispatch.launch) return bail(fail(EP_EUNSUPPORTED, "no dispatch kernel for this dtype"));
    h->g_layout.num_sms = h->g_dispatch.num_sms = h->g_combine.num_sms = sms;
    const int cols = h->E + h->W;
    h->g_layout.layout_experts = h->E;
    h->g_layout.layout_world = h->W;
    if ((e = h->layout.prepare(h->H, h->K, cols, &h->g_layout)) != cudaSuccess)
      return bail(fail_cuda(e, "layout kernel set-up"));
    if ((e = h->dispatch.prepare(h->H, h->K, row_bytes, &h->g_dispatch)) != cudaSuccess)
      return bail(fail_cuda(e, "dispatch kernel set-up"));
    if (h->g_dispatch.blocks_per_sm < 1)
      return bail(fail(EP_EUNSUPPORTED, "dispatch kernel does not fit on an SM for this hidden_dim"));
    if ((e = h->combine.prepare(h->H, h->K, 0, &h->g_combine)) != cudaSuccess)
      return bail(fail_cuda(e, "combine kernel set-up"));
    if (CombineTmaRequested()) {  // expert rows staged through shared memory by TMA bulk copies
      h->combine_tma = FindCombineTma(h->H, h->K, cfg->use_weights != 0);
      h->g_combine_tma.num_sms = sms;
      if (h->combine_tma.launch &&
          (e = h->combine_tma.prepare(h->H, h->K, 0, &h->g_combine_tma)) != cudaSuccess)
        return bail(fail_cuda(e, "TMA combine kernel set-up"));
    }
    // shapes outside the compiled table: specialise at run time when possible;
    // when not (no NVRTC, switched off), the compiled generic variants serve
    if (jit::Enabled()) {
      std::string why;
      const jit::Request dr = dispatch_request(cfg), cr = combine_request(cfg);
      if (is_generic(h->dispatch.name) && jit::Worthwhile(dr)) jit::Load(dr, &h->jit_dispatch, &why);
      if (is_generic(h->combine.name) && jit::Worthwhile(cr)) jit::Load(cr, &h->jit_combine, &why);
    }

    if (src) {  // the routing, its metadata and the error word are src's
      *out = h;
      return EP_OK;
    }
    // one allocation, 256-byte aligned sub-buffers
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t n_small = al(4 * (h->E + h->W + (h->E + 1) + (h->W + 1) + 2));
    const size_t n_slot = al(4 * static_cast<size_t>(h->max_tokens) * h->K);  // dst_slot, and the id clone
    const size_t n_meta = al(4 * static_cast<size_t>(h->rcap) * (h->K + 2));
    const size_t n_scr = al(sizeof(int32_t) * static_cast<size_t>(LayoutScratchInts(h->max_chunks, cols)));
    const size_t n_send = h->no_expand ? n_slot : 0;
    const size_t n_fused = al(sizeof(int32_t) * static_cast<size_t>(LayoutFusedStateInts(h->max_chunks, cols)));
    const size_t total = n_small + 2 * n_slot + n_meta + n_scr + n_send + n_fused;
    // Stream-ordered allocation on a private non-blocking stream: creating a
    // handle waits for nothing but its own clearing memset, never for work on
    // the caller's other streams (cudaMalloc and cudaDeviceSynchronize may wait
    // for the whole device).
    if ((e = cudaStreamCreateWithFlags(&h->own_stream, cudaStreamNonBlocking)) != cudaSuccess)
      return bail(fail_cuda(e, "cudaStreamCreateWithFlags"));
    e = cudaMallocAsync(&h->block, total, h->own_stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      h->block = nullptr;
      return bail(fail(EP_ENOMEM, std::string("cudaMallocAsync of the handle's metadata failed: ") +
                                      cudaGetErrorString(e)));
    }
    char* b = static_cast<char*>(h->block);
    int32_t* s = reinterpret_cast<int32_t*>(b);
    h->cnt = s;
    h->tok_per_rank = h->cnt + h->E;
    h->psum_expert = h->tok_per_rank + h->W;
    h->psum_rank = h->psum_expert + h->E + 1;
    h->num_recv = h->psum_rank + h->W + 1;
    h->err = h->num_recv + 1;
    h->dst_slot = reinterpret_cast<int32_t*>(b + n_small);
    h->topk_i32 = reinterpret_cast<int32_t*>(b + n_small + n_slot);
    h->meta = reinterpret_cast<int32_t*>(b + n_small + 2 * n_slot);
    h->scratch = reinterpret_cast<int32_t*>(b + n_small + 2 * n_slot + n_meta);
    h->send_slot = h->no_expand ? reinterpret_cast<int32_t*>(b + n_small + 2 * n_slot + n_meta + n_scr)
                                : h->dst_slot;
    h->fused = reinterpret_cast<int32_t*>(b + n_small + 2 * n_slot + n_meta + n_scr + n_send);
    if ((e = cudaMemsetAsync(h->block, 0, total, h->own_stream)) != cudaSuccess)
      return bail(fail_cuda(e, "cudaMemsetAsync"));
    // the block is ready for any stream once this returns
    if ((e = cudaStreamSynchronize(h->own_stream)) != cudaSuccess)
      return bail(fail_cuda(e, "cudaStreamSynchronize"));
    *out = h;
    return EP_OK;
  } catch (const std::exception& ex) {
    return fail(EP_EINVAL, ex.what());
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

}  // namespace

extern "C" {

int64_t ep_recv_capacity(const ep_cfg_t* cfg) noexcept {
  try {
    int rc = validate(cfg);
    if (rc != EP_OK && rc != EP_EUNSUPPORTED) return rc;
    return recv_rows(cfg);
  } catch (const std::exception& ex) {
    return fail(EP_EINVAL, ex.what());
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

int ep_handle_create(const ep_cfg_t* cfg, ep_handle_t* out) noexcept {
  return create_handle(cfg, nullptr, out);
}

int ep_handle_create_shared(const ep_cfg_t* cfg, ep_handle_t layout_src, ep_handle_t* out) noexcept {
  if (out) *out = nullptr;
  if (!layout_src) return fail(EP_EINVAL, "layout_src is NULL");
  return create_handle(cfg, layout_src->src ? layout_src->src : layout_src, out);
}

int ep_layout(ep_handle_t h, const int64_t* topk_idx, int32_t num_tokens, ep_stream_t stream) noexcept {
  try {
    if (!h) return fail(EP_EINVAL, "handle is NULL");
    if (h->src)
      return fail(EP_EINVAL, "this handle uses the layout of another handle: call ep_layout on that one");
    if (num_tokens < 0 || num_tokens > h->max_tokens)
      return fail(EP_EINVAL, "num_tokens must be in [0, world_size*max_tok_per_rank]");
    if (num_tokens > 0 && !topk_idx) return fail(EP_EINVAL, "topk_idx is NULL");
    if (num_tokens > 0 && (reinterpret_cast<uintptr_t>(topk_idx) & 7u))
      return fail(EP_EINVAL, "topk_idx must be 8-byte aligned");
    int rc = check_device(h);
    if (rc != EP_OK) return rc;
    LayoutParams p{};
    p.topk_idx = topk_idx;
    p.num_tokens = num_tokens;
    p.topk = h->K;
    p.world_size = h->W;
    p.max_tok_per_rank = h->T;
    p.num_expert_per_rank = h->Epr;
    p.num_experts = h->E;
    p.alignment = h->A;
    p.rcap = h->rcap;
    p.no_expand = h->no_expand ? 1 : 0;
    p.num_chunks = NumLayoutChunks(num_tokens);
    p.cnt = h->cnt;
    p.tok_per_rank = h->tok_per_rank;
    p.psum_expert = h->psum_expert;
    p.psum_rank = h->psum_rank;
    p.num_recv = h->num_recv;
    p.dst_slot = h->dst_slot;
    p.send_slot = h->send_slot;
    p.meta = h->meta;
    p.err = h->err;
    p.topk_i32 = h->topk_i32;
    p.epr_magic = RankMagic(h->Epr);
    BindLayoutScratch(&p, h->scratch, h->max_chunks, h->E + h->W);
    BindLayoutFusedState(&p, h->fused, h->max_chunks, h->E + h->W);
    p.wait_ns = h->wait_ns;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const LayoutPath path = LayoutPathOf(p, h->g_layout);
    cudaError_t e = h->layout.launch(p, h->g_layout, s);
    if (e != cudaSuccess) return fail_cuda(e, "layout launch");
    h->layout_ran = h->layout.name;
    if (path == LayoutPath::kCluster)
      h->layout_ran.insert(h->layout_ran.rfind('_'), "_cluster");  // ..._cluster_k8
    else if (path == LayoutPath::kFused)
      h->layout_ran.insert(h->layout_ran.rfind('_'), "_fused");    // ..._fused_k8
    h->num_tokens = num_tokens;
    h->last_stream = s;
    h->launched = true;
    return EP_OK;
  } catch (const std::exception& ex) {
    return fail(EP_EINVAL, ex.what());
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

int ep_dispatch(ep_handle_t h, const void* x, void* recv_x, float* recv_scales,
                ep_stream_t stream) noexcept {
  return ep_dispatch_fwd(h, x, recv_x, recv_scales, nullptr, nullptr, nullptr, stream);
}

int ep_dispatch_fwd(ep_handle_t h, const void* x, void* recv_x, float* recv_scales,
                    const float* topk_weights, float* recv_topk_weights, int32_t* recv_topk_idx,
                    ep_stream_t stream) noexcept {
  try {
    if (!h) return fail(EP_EINVAL, "handle is NULL");
    const bool fp8 = h->cfg.dispatch_dtype == EP_FP8_E4M3;
    if (fp8 && !recv_scales) return fail(EP_EINVAL, "FP8 dispatch needs recv_scales");
    if (!fp8 && recv_scales) return fail(EP_EINVAL, "recv_scales is only written by FP8 dispatch");
    if (recv_topk_weights && !topk_weights)
      return fail(EP_EINVAL, "recv_topk_weights needs topk_weights");
    const ep_handle* o = owner(h);
    if (o->num_tokens > 0) {
      if (!x || !recv_x) return fail(EP_EINVAL, "x / recv_x is NULL");
      if (!aligned16(x) || !aligned16(recv_x) || (recv_scales && !aligned16(recv_scales)))
        return fail(EP_EINVAL, "x, recv_x and recv_scales must be 16-byte aligned");
      if ((topk_weights && (reinterpret_cast<uintptr_t>(topk_weights) & 3u)) ||
          (recv_topk_weights && (reinterpret_cast<uintptr_t>(recv_topk_weights) & 3u)) ||
          (recv_topk_idx && (reinterpret_cast<uintptr_t>(recv_topk_idx) & 3u)))
        return fail(EP_EINVAL, "weights and ids must be 4-byte aligned");
    }
    int rc = check_device(h);
    if (rc != EP_OK) return rc;
    DispatchParams p{};
    p.x = x;
    p.recv_x = recv_x;
    p.recv_scales = recv_scales;
    p.dst_slot = o->send_slot;
    p.entry_slot = o->no_expand ? o->dst_slot : nullptr;
    p.num_tokens = o->num_tokens;
    p.hidden = h->H;
    p.topk = h->K;
    p.row_bytes = static_cast<int>(RowBytes(h->H, static_cast<EpDType>(h->cfg.dispatch_dtype)));
    p.err = o->err;
    p.topk_weights = topk_weights;
    p.topk_i32 = o->topk_i32;
    p.recv_topk_weights = recv_topk_weights;
    p.recv_topk_idx = recv_topk_idx;
    p.wait_ns = h->wait_ns;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool jit_ok = h->jit_dispatch.function && aligned32(x) && aligned32(recv_x);
    cudaError_t e = jit_ok ? jit::Launch(h->jit_dispatch, p.num_tokens, &p, s)
                           : h->dispatch.launch(p, h->g_dispatch, s);
    if (e != cudaSuccess) return fail_cuda(e, "dispatch launch");
    h->last_stream = s;
    h->launched = true;
    return EP_OK;
  } catch (const std::exception& ex) {
    return fail(EP_EINVAL, ex.what());
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

int ep_combine(ep_handle_t h, const void* y, const float* topk_weights, void* out,
               ep_stream_t stream) noexcept {
  return ep_combine_ex(h, y, topk_weights, nullptr, out, EP_BF16, stream);
}

int ep_combine_ex(ep_handle_t h, const void* y, const float* topk_weights, const void* bias,
                  void* out, int32_t out_dtype, ep_stream_t stream) noexcept {
  try {
    if (!h) return fail(EP_EINVAL, "handle is NULL");
    if (out_dtype != EP_BF16 && out_dtype != EP_FP32)
      return fail(EP_EINVAL, "combine output dtype must be EP_BF16 or EP_FP32");
    const bool weighted = h->cfg.use_weights != 0;
    const ep_handle* o = owner(h);
    if (o->num_tokens > 0) {
      if (!y || !out) return fail(EP_EINVAL, "y / out is NULL");
      if (weighted && !topk_weights) return fail(EP_EINVAL, "use_weights is set but topk_weights is NULL");
      if (!aligned16(y) || !aligned16(out) || (bias && !aligned16(bias)))
        return fail(EP_EINVAL, "y, bias and out must be 16-byte aligned");
      if (weighted && (reinterpret_cast<uintptr_t>(topk_weights) & 3u))
        return fail(EP_EINVAL, "topk_weights must be 4-byte aligned");
    }
    int rc = check_device(h);
    if (rc != EP_OK) return rc;
    CombineParams p{};
    p.y = y;
    p.weights = weighted ? topk_weights : nullptr;
    p.bias = bias;
    p.out = out;
    p.dst_slot = o->send_slot;
    p.num_tokens = o->num_tokens;
    p.hidden = h->H;
    p.topk = h->K;
    p.out_f32 = out_dtype == EP_FP32 ? 1 : 0;
    p.err = o->err;
    p.wait_ns = h->wait_ns;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the TMA combine (EP_GB300_COMBINE_TMA=1) serves the plain bf16 combine
    const bool tma_ok = h->combine_tma.launch && !bias && p.out_f32 == 0;
    const bool jit_ok = h->jit_combine.function && !bias && p.out_f32 == 0 && aligned32(y) &&
                        aligned32(out);
    cudaError_t e = tma_ok   ? h->combine_tma.launch(p, h->g_combine_tma, s)
                    : jit_ok ? jit::Launch(h->jit_combine, p.num_tokens, &p, s)
                             : h->combine.launch(p, h->g_combine, s);
    if (e != cudaSuccess) return fail_cuda(e, "combine launch");
    h->last_stream = s;
    h->launched = true;
    return EP_OK;
  } catch (const std::exception& ex) {
    return fail(EP_EINVAL, ex.what());
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

void ep_handle_free(ep_handle_t h) noexcept {
  try {
    if (!h) return;
    // the handle's work on its last stream finishes before its memory goes
    if (h->launched) cudaStreamSynchronize(h->last_stream);
    if (h->block) {
      cudaFreeAsync(h->block, h->own_stream);
      cudaStreamSynchronize(h->own_stream);
    }
    if (h->own_stream) cudaStreamDestroy(h->own_stream);
    delete h;
  } catch (...) {
  }
}

int ep_handle_get(ep_handle_t h, int32_t field, void** dev_ptr, int64_t* numel) noexcept {
  try {
    if (!h || !dev_ptr || !numel) return fail(EP_EINVAL, "NULL argument");
    h = const_cast<ep_handle*>(owner(h));  // a shared handle shows its layout_src's fields
    switch (field) {
      case EP_FIELD_NUM_UNALIGNED_PER_EXPERT: *dev_ptr = h->cnt; *numel = h->E; break;
      case EP_FIELD_NUM_TOKENS_PER_RANK: *dev_ptr = h->tok_per_rank; *numel = h->W; break;
      case EP_FIELD_PSUM_PER_EXPERT: *dev_ptr = h->psum_expert; *numel = h->E + 1; break;
      case EP_FIELD_PSUM_PER_RANK: *dev_ptr = h->psum_rank; *numel = h->W + 1; break;
      case EP_FIELD_DST_SLOT:
        *dev_ptr = h->dst_slot;
        *numel = static_cast<int64_t>(h->num_tokens) * h->K;
        break;
      case EP_FIELD_RECV_SRC_METADATA: *dev_ptr = h->meta; *numel = h->rcap * (h->K + 2); break;
      case EP_FIELD_NUM_RECV: *dev_ptr = h->num_recv; *numel = 1; break;
      case EP_FIELD_DEVICE_ERROR: *dev_ptr = h->err; *numel = 1; break;
      case EP_FIELD_TOPK_IDX:
        *dev_ptr = h->topk_i32;
        *numel = static_cast<int64_t>(h->num_tokens) * h->K;
        break;
      case EP_FIELD_SEND_SLOT:
        *dev_ptr = h->send_slot;
        *numel = static_cast<int64_t>(h->num_tokens) * h->K;
        break;
      default: return fail(EP_EINVAL, "unknown field");
    }
    return EP_OK;
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

int ep_handle_status(ep_handle_t h, int32_t* device_error) noexcept {
  try {
    if (!h || !device_error) return fail(EP_EINVAL, "NULL argument");
    int rc = check_device(h);
    if (rc != EP_OK) return rc;
    // read and clear the error word in order on the handle's last stream and
    // wait for that stream only (other streams of the process keep running)
    const cudaStream_t s = h->last_stream;
    int32_t v = 0;
    int32_t* err = owner(h)->err;
    cudaError_t e = cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync");
    if ((e = cudaMemsetAsync(err, 0, sizeof v, s)) != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    *device_error = v;
    return EP_OK;
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

int ep_handle_variant(ep_handle_t h, int32_t step, char* buf, int32_t len) noexcept {
  try {
    if (!h || !buf || len < 1) return fail(EP_EINVAL, "NULL argument");
    const ep_handle* o = owner(h);
    const char* name = step == 0 ? (o->layout_ran.empty() ? o->layout.name : o->layout_ran.c_str())
                     : step == 1 ? (h->jit_dispatch.function ? h->jit_dispatch.name.c_str()
                                                             : h->dispatch.name)
                     : step == 2 ? (h->combine_tma.launch ? h->combine_tma.name
                                    : h->jit_combine.function ? h->jit_combine.name.c_str()
                                                              : h->combine.name)
                                 : nullptr;
    if (!name) return fail(EP_EINVAL, "step must be 0, 1 or 2");
    std::snprintf(buf, static_cast<size_t>(len), "%s", name);
    return EP_OK;
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

int ep_jit_precompile(const ep_cfg_t* cfg, const char* arch, char* report, int32_t len) noexcept {
  try {
    int rc = validate(cfg);
    if (rc != EP_OK) return rc;
    std::string rep;
    int compiled_now = 0;
    const std::string a = arch && *arch ? arch : "sm_103a";
    const Variant<DispatchLaunch> dv =
        FindDispatch(cfg->hidden_dim, cfg->num_expert_per_token,
                     static_cast<EpDType>(cfg->dispatch_dtype));
    const Variant<CombineLaunch> cv =
        FindCombine(cfg->hidden_dim, cfg->num_expert_per_token, cfg->use_weights != 0);
    const jit::Request reqs[2] = {dispatch_request(cfg), combine_request(cfg)};
    const char* names[2] = {dv.name, cv.name};
    for (int i = 0; i < 2; ++i) {
      if (!is_generic(names[i])) {
        rep += std::string(names[i]) + " compiled-in\n";
        continue;
      }
      if (!jit::Worthwhile(reqs[i])) {
        rep += std::string(names[i]) + " generic\n";
        continue;
      }
      bool compiled = false;
      std::string dir, err;
      if (!jit::Prepare(reqs[i], a, &compiled, &dir, &err))
        return fail(err.find("not available") != std::string::npos ? EP_EUNSUPPORTED : EP_ECUDA, err);
      compiled_now += compiled ? 1 : 0;
      rep += jit::EntryName(reqs[i]) + (compiled ? " compiled " : " cached ") + dir + "\n";
    }
    if (report && len > 0) std::snprintf(report, static_cast<size_t>(len), "%s", rep.c_str());
    return compiled_now;
  } catch (const std::exception& ex) {
    return fail(EP_EINVAL, ex.what());
  } catch (...) {
    return fail(EP_EINVAL, "unknown exception");
  }
}

const char* ep_last_error(void) noexcept { return g_last_error.c_str(); }

}  // extern "C"
