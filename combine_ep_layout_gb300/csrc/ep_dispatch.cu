// ep_dispatch.cu -- dispatch: scatter each token row to its K receive rows
// ("Dispatch data flow" of "DeepEP overall architecture analysis": pack token
// data + scale factors, then copy into recv_x; "MORI JIT v2" §3.7: the
// transport dtype is a property of the copy, not arithmetic).
//
// On one GPU the pages' two hops (symmetric buffer, then copy epilogue) fold
// into one pass: read x[t] once, write it K times.  The copy never touches
// registers: the TMA unit moves whole rows with cp.async.bulk, global ->
// shared (one load per token) and shared -> global (K stores per token).
//
//   bf16: one warp per CTA; lane 0 drives an S-stage ring of row buffers.
//         Loads run up to S-1 tokens ahead; a stage is refilled once the bulk
//         stores of its previous token have finished reading it
//         (cp.async.bulk.wait_group.read).
//   FP8:  one producer warp (loads and stores) and kFp8ConsumerWarps
//         consumer warps that turn the staged bf16 row into e4m3 bytes and
//         per-128-channel fp32 scales in shared memory, once per token; the
//         producer then stores the same bytes to all K rows.  full / ready /
//         empty mbarriers per stage order the three roles.
//
// Persistent grid: (#SMs x resident CTAs) CTAs, each with a contiguous run of
// tokens whose K slots it stages in shared memory first.  Every wait is
// bounded; on a timeout a kernel sets kErrTimeout, drains its own copies and
// returns.
#include <cuda_runtime.h>

#include <cstdint>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"
#include "ep_ptx.cuh"

namespace epg {

namespace {

constexpr int kBf16Stages = 4;
constexpr int kFp8Stages = 3;
constexpr int kFp8ConsumerWarps = 4;
constexpr int kSlotCap = 2048;  // int32 slots staged per CTA (8 KB)

__host__ __device__ constexpr uint32_t align128(uint32_t v) { return (v + 127u) & ~127u; }

struct Bf16Smem {
  uint32_t row;        // row bytes
  uint32_t row_pad;    // row stride in shared memory
  uint32_t bars;       // offset of S mbarriers
  uint32_t slots;      // offset of the slot table
  uint32_t total;
};

__host__ __device__ constexpr Bf16Smem bf16_smem(int hidden) {
  const uint32_t row = 2u * hidden;
  const uint32_t rp = align128(row);
  const uint32_t bars = rp * kBf16Stages;
  const uint32_t slots = bars + 8u * kBf16Stages;
  return {row, rp, bars, slots, slots + 4u * kSlotCap};
}

template <int HC, int KC>
__global__ void __launch_bounds__(32) ep_dispatch_bf16_kernel(DispatchParams p, int tokens_per_cta) {
  constexpr int S = kBf16Stages;
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const Bf16Smem L = bf16_smem(H);
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* slots = reinterpret_cast<int32_t*>(smem + L.slots);

  const int lane = threadIdx.x;
  const int t0 = blockIdx.x * tokens_per_cta;
  const int t1 = min(p.num_tokens, t0 + tokens_per_cta);
  if (t0 >= t1) return;
  const int n = t1 - t0;
  for (int i = lane; i < n * K; i += 32) slots[i] = p.dst_slot[static_cast<int64_t>(t0) * K + i];
  const uint32_t rows0 = smem_addr(smem);
  const uint32_t bar0 = smem_addr(smem + L.bars);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane != 0) return;

  const uint8_t* xb = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t0) * L.row;
  uint8_t* rx = static_cast<uint8_t*>(p.recv_x);
  const uint64_t pol_x = policy_evict_first();
  int issued = 0;
  auto issue_load = [&](int j) {
    const int s = j % S;
    mbar_arrive_expect_tx(bar0 + 8 * s, L.row);
    bulk_g2s_hint(rows0 + s * L.row_pad, xb + static_cast<int64_t>(j) * L.row, L.row, bar0 + 8 * s,
                  pol_x);
    ++issued;
  };
  const int pro = n < S ? n : S;
  for (int j = 0; j < pro; ++j) issue_load(j);

  int j = 0;
  for (; j < n; ++j) {
    const int s = j % S;
    if (!mbar_wait(bar0 + 8 * s, (j / S) & 1)) break;
    const int32_t* sl = slots + j * K;
#pragma unroll
    for (int k = 0; k < (KC ? KC : kMaxTopk); ++k) {
      if (k >= K) break;
      const int32_t d = sl[k];
      if (d >= 0) bulk_s2g(rx + static_cast<int64_t>(d) * L.row, rows0 + s * L.row_pad, L.row);
    }
    bulk_commit();
    if (j >= 1 && j - 1 + S < n) {
      bulk_wait_read<1>();  // the stores of token j-1 have read their stage
      issue_load(j - 1 + S);
    }
  }
  if (j < n) {  // timed out: report, then let our own loads land before leaving
    atomicOr(p.err, kErrTimeout);
    for (int jj = j; jj < issued; ++jj) mbar_wait(bar0 + 8 * (jj % S), (jj / S) & 1);
  }
  bulk_wait_all<0>();
}

struct Fp8Smem {
  uint32_t in_row, in_pad;   // bf16 input row
  uint32_t q_row, q_pad;     // e4m3 row
  uint32_t sc_row, sc_pad;   // scales row
  uint32_t in, q, sc;        // region offsets
  uint32_t bars;             // full[S], ready[S], empty[S]
  uint32_t slots;
  uint32_t total;
};

__host__ __device__ constexpr Fp8Smem fp8_smem(int hidden) {
  const uint32_t in_row = 2u * hidden, q_row = hidden, sc_row = 4u * (hidden / kScaleGroup);
  const uint32_t in_pad = align128(in_row), q_pad = align128(q_row), sc_pad = align128(sc_row);
  const uint32_t in = 0, q = in + kFp8Stages * in_pad, sc = q + kFp8Stages * q_pad;
  const uint32_t bars = sc + kFp8Stages * sc_pad;
  const uint32_t slots = bars + 8u * 3 * kFp8Stages;
  return {in_row, in_pad, q_row, q_pad, sc_row, sc_pad, in, q, sc, bars, slots,
          slots + 4u * kSlotCap};
}

// Two fp32 values to packed e4m3 (round to nearest even, saturate to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int HC, int KC>
__global__ void __launch_bounds__(32 * (1 + kFp8ConsumerWarps))
    ep_dispatch_fp8_kernel(DispatchParams p, int tokens_per_cta) {
  constexpr int S = kFp8Stages;
  constexpr int NC = kFp8ConsumerWarps;
  const int H = HC ? HC : p.hidden;
  const int K = KC ? KC : p.topk;
  const int G = H / kScaleGroup;
  const Fp8Smem L = fp8_smem(H);
  const bool sc_bulk = (L.sc_row % 16u) == 0;
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* slots = reinterpret_cast<int32_t*>(smem + L.slots);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * tokens_per_cta;
  const int t1 = min(p.num_tokens, t0 + tokens_per_cta);
  if (t0 >= t1) return;
  const int n = t1 - t0;
  for (int i = tid; i < n * K; i += blockDim.x) slots[i] = p.dst_slot[static_cast<int64_t>(t0) * K + i];
  const uint32_t full0 = smem_addr(smem + L.bars);
  const uint32_t ready0 = full0 + 8 * S;
  const uint32_t empty0 = ready0 + 8 * S;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(ready0 + 8 * s, NC);
      mbar_init(empty0 + 8 * s, 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  uint8_t* rq = static_cast<uint8_t*>(p.recv_x);
  float* rs = p.recv_scales;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    const uint8_t* xb = static_cast<const uint8_t*>(p.x) + static_cast<int64_t>(t0) * L.in_row;
    const uint32_t in0 = smem_addr(smem + L.in), q0 = smem_addr(smem + L.q),
                   sc0 = smem_addr(smem + L.sc);
    const uint64_t pol_x = policy_evict_first();
    int issued = 0;
    auto issue_load = [&](int j) {
      const int s = j % S;
      mbar_arrive_expect_tx(full0 + 8 * s, L.in_row);
      bulk_g2s_hint(in0 + s * L.in_pad, xb + static_cast<int64_t>(j) * L.in_row, L.in_row,
                    full0 + 8 * s, pol_x);
      ++issued;
    };
    const int pro = n < S ? n : S;
    for (int j = 0; j < pro; ++j) issue_load(j);
    int j = 0;
    for (; j < n; ++j) {
      const int s = j % S;
      if (!mbar_wait(ready0 + 8 * s, (j / S) & 1)) break;
      const int32_t* sl = slots + j * K;
#pragma unroll
      for (int k = 0; k < (KC ? KC : kMaxTopk); ++k) {
        if (k >= K) break;
        const int32_t d = sl[k];
        if (d < 0) continue;
        bulk_s2g(rq + static_cast<int64_t>(d) * L.q_row, q0 + s * L.q_pad, L.q_row);
        if (sc_bulk)
          bulk_s2g(reinterpret_cast<uint8_t*>(rs) + static_cast<int64_t>(d) * L.sc_row,
                   sc0 + s * L.sc_pad, L.sc_row);
      }
      bulk_commit();
      if (j + S < n) issue_load(j + S);  // consumers are done with the input stage
      if (j >= 1) {
        bulk_wait_read<1>();               // stores of token j-1 have read their stage
        mbar_arrive(empty0 + 8 * ((j - 1) % S));
      }
    }
    if (j < n) {
      atomicOr(p.err, kErrTimeout);
      for (int jj = j; jj < issued; ++jj) mbar_wait(full0 + 8 * (jj % S), (jj / S) & 1);
    }
    bulk_wait_all<0>();
    return;
  }

  // ---------------- consumers: bf16 -> e4m3 + scales ----------------
  const int cw = warp - 1;
  for (int j = 0; j < n; ++j) {
    const int s = j % S;
    if (!mbar_wait(full0 + 8 * s, (j / S) & 1)) { atomicOr(p.err, kErrTimeout); return; }
    if (j >= S && !mbar_wait(empty0 + 8 * s, ((j / S) - 1) & 1)) {
      atomicOr(p.err, kErrTimeout);
      return;
    }
    const uint8_t* in_s = smem + L.in + s * L.in_pad;
    uint8_t* q_s = smem + L.q + s * L.q_pad;
    float* sc_s = reinterpret_cast<float*>(smem + L.sc + s * L.sc_pad);
    for (int g = cw; g < G; g += NC) {
      const uint2 raw = *reinterpret_cast<const uint2*>(in_s + g * 256 + lane * 8);
      float f[4];
      f[0] = __uint_as_float(raw.x << 16);
      f[1] = __uint_as_float(raw.x & 0xffff0000u);
      f[2] = __uint_as_float(raw.y << 16);
      f[3] = __uint_as_float(raw.y & 0xffff0000u);
      uint32_t a = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t b = __float_as_uint(f[i]) & 0x7fffffffu;
        b = b > 0x7f800000u ? 0u : b;  // NaN does not take part in the maximum
        a = b > a ? b : a;
      }
      a = __reduce_max_sync(0xffffffffu, a);
      float sc = 0.0f;
      uint32_t q4 = 0;
      if (a != 0u) {
        sc = __fdiv_rn(__uint_as_float(a), 448.0f);
        const float r0 = __fdiv_rn(f[0], sc), r1 = __fdiv_rn(f[1], sc);
        const float r2 = __fdiv_rn(f[2], sc), r3 = __fdiv_rn(f[3], sc);
        q4 = cvt_e4m3x2(r0, r1) | (cvt_e4m3x2(r2, r3) << 16);
      }
      *reinterpret_cast<uint32_t*>(q_s + g * 128 + lane * 4) = q4;
      if (lane == 0) {
        sc_s[g] = sc;
        if (!sc_bulk) {
          const int32_t* sl = slots + j * K;
          for (int k = 0; k < K; ++k)
            if (sl[k] >= 0) rs[static_cast<int64_t>(sl[k]) * G + g] = sc;
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(ready0 + 8 * s);
  }
}

// Persistent grid: CTAs resident at once, each with a contiguous run of tokens,
// no more than kSlotCap / K tokens per CTA.
inline void persistent_split(int num_tokens, int topk, const LaunchGeom& g, int* grid, int* per) {
  const int resident = g.num_sms * (g.blocks_per_sm > 0 ? g.blocks_per_sm : 1);
  int tpc = (num_tokens + resident - 1) / resident;
  const int cap = kSlotCap / topk;
  if (tpc > cap) tpc = cap;
  if (tpc < 1) tpc = 1;
  *per = tpc;
  *grid = (num_tokens + tpc - 1) / tpc;
}

template <int HC, int KC>
cudaError_t launch_bf16(const DispatchParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  int grid, per;
  persistent_split(p.num_tokens, p.topk, g, &grid, &per);
  const Bf16Smem L = bf16_smem(p.hidden);
  ep_dispatch_bf16_kernel<HC, KC><<<grid, 32, L.total, s>>>(p, per);
  return cudaGetLastError();
}

template <int HC, int KC>
cudaError_t prepare_bf16(int hidden, int, int, LaunchGeom* g) {
  const Bf16Smem L = bf16_smem(hidden);
  cudaError_t e = cudaFuncSetAttribute(ep_dispatch_bf16_kernel<HC, KC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g->blocks_per_sm,
                                                       ep_dispatch_bf16_kernel<HC, KC>, 32, L.total);
}

template <int HC, int KC>
cudaError_t launch_fp8(const DispatchParams& p, const LaunchGeom& g, cudaStream_t s) {
  if (p.num_tokens == 0) return cudaSuccess;
  int grid, per;
  persistent_split(p.num_tokens, p.topk, g, &grid, &per);
  const Fp8Smem L = fp8_smem(p.hidden);
  ep_dispatch_fp8_kernel<HC, KC><<<grid, 32 * (1 + kFp8ConsumerWarps), L.total, s>>>(p, per);
  return cudaGetLastError();
}

template <int HC, int KC>
cudaError_t prepare_fp8(int hidden, int, int, LaunchGeom* g) {
  const Fp8Smem L = fp8_smem(hidden);
  cudaError_t e = cudaFuncSetAttribute(ep_dispatch_fp8_kernel<HC, KC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g->blocks_per_sm, ep_dispatch_fp8_kernel<HC, KC>, 32 * (1 + kFp8ConsumerWarps), L.total);
}

}  // namespace

Variant<DispatchLaunch> FindDispatch(int hidden, int topk, EpDType dtype) {
  if (dtype == EpDType::Bf16) {
#define EPG_CASE(H, K)                                                         \
  if (hidden == H && topk == K)                                                \
    return {"ep_dispatch_bf16_h" #H "_k" #K, launch_bf16<H, K>, prepare_bf16<H, K>};
    EPG_SHAPE_LIST(EPG_CASE)
#undef EPG_CASE
    return {"ep_dispatch_bf16_generic", launch_bf16<0, 0>, prepare_bf16<0, 0>};
  }
  if (dtype == EpDType::Fp8) {
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
