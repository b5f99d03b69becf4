"""CPU oracle for the MoE expert-parallel layout / dispatch / combine path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The product library never calls it
and shares no code with it; the CUDA path fails loudly when its own extension
is missing instead of falling back here.

The arithmetic lives in plain C (ep_oracle.c, single-threaded, no fast-math,
no contraction).  This module only marshals numpy arrays into it.  bf16 values
travel as their uint16 bit patterns, e4m3 values as uint8 codes.

Parity status: every routine here is pinned by the CPU tests in
tests/test_oracle_*.py (brute force on tiny inputs, an independent stable-sort
formulation, invariants, exhaustive e4m3 checks against torch's float8_e4m3fn
cast, closed-form combine cases, error bounds).
"""
import ctypes
import numpy as np

from .build import build_oracle

_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def lib():
    """Load (building first if needed) liboracle_ep.so."""
    global _lib
    if _lib is not None:
        return _lib
    L = ctypes.CDLL(build_oracle())
    c = ctypes
    L.oracle_recv_capacity.restype = c.c_int64
    L.oracle_recv_capacity.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int]
    L.oracle_layout.restype = c.c_int
    L.oracle_layout.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                _i64p, c.c_int, _i32p, _i32p, _i32p, _i32p,
                                _i32p, _i32p, c.c_int64, _i32p, _i32p]
    L.oracle_dispatch_bf16.restype = None
    L.oracle_dispatch_bf16.argtypes = [c.c_int, c.c_int, c.c_int, _u16p, _i32p, _u16p]
    L.oracle_dispatch_fp8.restype = None
    L.oracle_dispatch_fp8.argtypes = [c.c_int, c.c_int, c.c_int, _u16p, _i32p, _u8p, _f32p]
    L.oracle_quant_fp8_row.restype = None
    L.oracle_quant_fp8_row.argtypes = [c.c_int, _u16p, _u8p, _f32p]
    L.oracle_combine.restype = None
    L.oracle_combine.argtypes = [c.c_int, c.c_int, c.c_int, _u16p, _i32p, c.c_void_p, _u16p]
    L.oracle_e4m3_encode_array.restype = None
    L.oracle_e4m3_encode_array.argtypes = [c.c_int64, _f32p, _u8p]
    L.oracle_e4m3_decode_array.restype = None
    L.oracle_e4m3_decode_array.argtypes = [c.c_int64, _u8p, _f64p]
    L.oracle_f32_to_bf16_array.restype = None
    L.oracle_f32_to_bf16_array.argtypes = [c.c_int64, _f32p, _u16p]
    L.oracle_dispatch_bytes.restype = None
    L.oracle_dispatch_bytes.argtypes = [c.c_int, c.c_int64, c.c_int, _u8p, _i32p, _u8p]
    L.oracle_forward_routing.restype = None
    L.oracle_forward_routing.argtypes = [c.c_int, c.c_int, _i64p, c.c_void_p, _i32p, c.c_void_p,
                                         c.c_void_p]
    L.oracle_combine_ex.restype = None
    L.oracle_combine_ex.argtypes = [c.c_int, c.c_int, c.c_int, _u16p, _i32p, c.c_void_p,
                                    c.c_void_p, c.c_void_p, c.c_void_p]
    L.oracle_recv_capacity_nonexpand.restype = c.c_int64
    L.oracle_recv_capacity_nonexpand.argtypes = [c.c_int, c.c_int, c.c_int]
    L.oracle_layout_nonexpand.restype = c.c_int
    L.oracle_layout_nonexpand.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                          _i64p, c.c_int, _i32p, _i32p, _i32p, _i32p,
                                          _i32p, _i32p, _i32p, c.c_int64, _i32p, _i32p]
    L.oracle_forward_routing_nonexpand.restype = None
    L.oracle_forward_routing_nonexpand.argtypes = [c.c_int, c.c_int, _i64p, c.c_void_p, _i32p,
                                                   _i32p, c.c_void_p, c.c_void_p]
    _lib = L
    return L


def recv_capacity(max_tokens, topk, num_experts, alignment):
    """Rows a receive buffer needs for any routing of max_tokens tokens."""
    return int(lib().oracle_recv_capacity(max_tokens, topk, num_experts, alignment))


def layout(topk_idx, world_size, max_tok_per_rank, num_expert_per_rank,
           alignment, rcap=None):
    """Layout of topk_idx (int64 [N, K]).  Returns a dict of numpy arrays:
    cnt [E], tok_per_rank [W], psum_expert [E+1], psum_rank [W+1],
    dst_slot [N, K], meta [rcap, K+2], num_recv (int), err (int), rcap (int)."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    N, K = topk_idx.shape
    W, T, Epr, A = world_size, max_tok_per_rank, num_expert_per_rank, alignment
    E = W * Epr
    if rcap is None:
        rcap = recv_capacity(W * T, K, E, A)
    out = dict(
        cnt=np.zeros(E, np.int32), tok_per_rank=np.zeros(W, np.int32),
        psum_expert=np.zeros(E + 1, np.int32), psum_rank=np.zeros(W + 1, np.int32),
        dst_slot=np.zeros((N, K), np.int32), meta=np.zeros((rcap, K + 2), np.int32),
    )
    num_recv = np.zeros(1, np.int32)
    err = np.zeros(1, np.int32)
    rc = lib().oracle_layout(W, T, Epr, K, A, topk_idx.reshape(-1), N,
                             out["cnt"], out["tok_per_rank"], out["psum_expert"],
                             out["psum_rank"], out["dst_slot"].reshape(-1),
                             out["meta"].reshape(-1), rcap, num_recv, err)
    if rc != 0:
        raise ValueError("oracle layout: receive capacity exceeded")
    out["num_recv"] = int(num_recv[0])
    out["err"] = int(err[0])
    out["rcap"] = int(rcap)
    return out


def dispatch_bf16(x_bits, dst_slot, recv_x):
    """recv_x[dst_slot[t, k]] = x[t] in place; x_bits / recv_x are uint16."""
    N, H = x_bits.shape
    K = dst_slot.shape[1]
    assert recv_x.dtype == np.uint16 and recv_x.shape[1] == H and recv_x.flags.c_contiguous
    lib().oracle_dispatch_bf16(N, H, K, np.ascontiguousarray(x_bits),
                               np.ascontiguousarray(dst_slot, dtype=np.int32), recv_x)
    return recv_x


def dispatch_fp8(x_bits, dst_slot, recv_x, recv_scales):
    """FP8 dispatch in place: recv_x uint8 [rows, H], recv_scales fp32 [rows, H/128]."""
    N, H = x_bits.shape
    K = dst_slot.shape[1]
    assert H % 128 == 0
    assert recv_x.dtype == np.uint8 and recv_x.flags.c_contiguous
    assert recv_scales.dtype == np.float32 and recv_scales.flags.c_contiguous
    lib().oracle_dispatch_fp8(N, H, K, np.ascontiguousarray(x_bits),
                              np.ascontiguousarray(dst_slot, dtype=np.int32),
                              recv_x, recv_scales)
    return recv_x, recv_scales


def quant_fp8_row(x_row_bits):
    """Quantise one bf16 row: returns (e4m3 codes uint8 [H], scales fp32 [H/128])."""
    x_row_bits = np.ascontiguousarray(x_row_bits, dtype=np.uint16)
    H = x_row_bits.shape[0]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.float32)
    lib().oracle_quant_fp8_row(H, x_row_bits, q, s)
    return q, s


def combine(y_bits, dst_slot, weights=None):
    """out[t] = bf16(sum_k w[t,k] * y[dst_slot[t,k]]) with the fixed fma order.
    y_bits uint16 [rows, H]; weights fp32 [N, K] or None. Returns uint16 [N, H]."""
    dst_slot = np.ascontiguousarray(dst_slot, dtype=np.int32)
    N, K = dst_slot.shape
    H = y_bits.shape[1]
    out = np.zeros((N, H), np.uint16)
    wp = None
    if weights is not None:
        weights = np.ascontiguousarray(weights, dtype=np.float32)
        assert weights.shape == (N, K)
        wp = weights.ctypes.data_as(ctypes.c_void_p)
    lib().oracle_combine(N, H, K, np.ascontiguousarray(y_bits), dst_slot, wp, out)
    return out


def e4m3_encode(v):
    """fp32 array -> e4m3 codes (round to nearest even, saturate to +-448)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, np.uint8)
    lib().oracle_e4m3_encode_array(v.size, v.reshape(-1), out.reshape(-1))
    return out


def e4m3_decode(c):
    """e4m3 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.zeros(c.shape, np.float64)
    lib().oracle_e4m3_decode_array(c.size, c.reshape(-1), out.reshape(-1))
    return out


def f32_to_bf16(v):
    """fp32 array -> bf16 bit patterns (round to nearest even)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, np.uint16)
    lib().oracle_f32_to_bf16_array(v.size, v.reshape(-1), out.reshape(-1))
    return out


def _vp(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def dispatch_bytes(x_bytes, dst_slot, recv):
    """recv[dst_slot[t, k]] = x[t] as raw bytes; x_bytes uint8 [N, row_bytes],
    recv uint8 [rows, row_bytes], in place."""
    x_bytes = np.ascontiguousarray(x_bytes, dtype=np.uint8)
    N, rb = x_bytes.shape
    K = dst_slot.shape[1]
    assert recv.dtype == np.uint8 and recv.shape[1] == rb and recv.flags.c_contiguous
    lib().oracle_dispatch_bytes(N, rb, K, x_bytes, np.ascontiguousarray(dst_slot, np.int32), recv)
    return recv


def forward_routing(topk_idx, weights, dst_slot, recv_w=None, recv_idx=None):
    """recv_w[dst_slot[t, k]] = weights[t, k]; recv_idx[dst_slot[t, k]] = topk_idx[t, k]
    (in place; either output may be None)."""
    topk_idx = np.ascontiguousarray(topk_idx, np.int64)
    N, K = topk_idx.shape
    w = None if weights is None else np.ascontiguousarray(weights, np.float32)
    for a, dt in ((recv_w, np.float32), (recv_idx, np.int32)):
        assert a is None or (a.dtype == dt and a.flags.c_contiguous)
    lib().oracle_forward_routing(N, K, topk_idx, _vp(w), np.ascontiguousarray(dst_slot, np.int32),
                                 _vp(recv_w), _vp(recv_idx))


def combine_ex(y_bits, dst_slot, weights=None, bias_bits=None, out_dtype="bf16"):
    """Combine + optional bf16 bias [N, H]; returns uint16 bf16 bits or float32 [N, H]."""
    dst_slot = np.ascontiguousarray(dst_slot, dtype=np.int32)
    N, K = dst_slot.shape
    H = y_bits.shape[1]
    w = None if weights is None else np.ascontiguousarray(weights, np.float32)
    b = None if bias_bits is None else np.ascontiguousarray(bias_bits, np.uint16)
    assert b is None or b.shape == (N, H)
    if out_dtype == "fp32":
        out = np.zeros((N, H), np.float32)
        lib().oracle_combine_ex(N, H, K, np.ascontiguousarray(y_bits), dst_slot, _vp(w), _vp(b),
                                None, _vp(out))
    else:
        out = np.zeros((N, H), np.uint16)
        lib().oracle_combine_ex(N, H, K, np.ascontiguousarray(y_bits), dst_slot, _vp(w), _vp(b),
                                _vp(out), None)
    return out


def recv_capacity_nonexpand(max_tokens, topk, world_size):
    """Rows a non-expand receive buffer needs: one per (token, rank), min(K, W) per token."""
    return int(lib().oracle_recv_capacity_nonexpand(max_tokens, topk, world_size))


def layout_nonexpand(topk_idx, world_size, max_tok_per_rank, num_expert_per_rank,
                     alignment, rcap=None):
    """Non-expand layout (one receive row per (token, destination rank)).  Same
    keys as layout(), plus send_slot [N, K] (the token's distinct rows,
    ascending, then -1); psum_rank / num_recv / meta describe the rank rows."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    N, K = topk_idx.shape
    W, T, Epr, A = world_size, max_tok_per_rank, num_expert_per_rank, alignment
    E = W * Epr
    if rcap is None:
        rcap = recv_capacity_nonexpand(W * T, K, W)
    out = dict(
        cnt=np.zeros(E, np.int32), tok_per_rank=np.zeros(W, np.int32),
        psum_expert=np.zeros(E + 1, np.int32), psum_rank=np.zeros(W + 1, np.int32),
        dst_slot=np.zeros((N, K), np.int32), send_slot=np.zeros((N, K), np.int32),
        meta=np.zeros((rcap, K + 2), np.int32),
    )
    num_recv = np.zeros(1, np.int32)
    err = np.zeros(1, np.int32)
    rc = lib().oracle_layout_nonexpand(W, T, Epr, K, A, topk_idx.reshape(-1), N,
                                       out["cnt"], out["tok_per_rank"], out["psum_expert"],
                                       out["psum_rank"], out["dst_slot"].reshape(-1),
                                       out["send_slot"].reshape(-1), out["meta"].reshape(-1),
                                       rcap, num_recv, err)
    if rc != 0:
        raise ValueError("oracle non-expand layout: receive capacity exceeded")
    out["num_recv"] = int(num_recv[0])
    out["err"] = int(err[0])
    out["rcap"] = int(rcap)
    return out


def forward_routing_nonexpand(topk_idx, weights, dst_slot, send_slot, recv_w=None, recv_idx=None):
    """K-wide routing rows of the non-expand layout, in place: recv_w fp32 [rows, K],
    recv_idx int32 [rows, K] (either may be None)."""
    topk_idx = np.ascontiguousarray(topk_idx, np.int64)
    N, K = topk_idx.shape
    w = None if weights is None else np.ascontiguousarray(weights, np.float32)
    for a, dt in ((recv_w, np.float32), (recv_idx, np.int32)):
        assert a is None or (a.dtype == dt and a.flags.c_contiguous and a.shape[-1] == K)
    lib().oracle_forward_routing_nonexpand(N, K, topk_idx, _vp(w),
                                           np.ascontiguousarray(dst_slot, np.int32),
                                           np.ascontiguousarray(send_slot, np.int32),
                                           _vp(recv_w), _vp(recv_idx))
