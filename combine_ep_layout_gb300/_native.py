"""ctypes binding of libep_gb300.so (include/ep_gb300.h).

Argument marshalling only: every step of layout / dispatch / combine runs in
the library's CUDA kernels.  There is no other implementation behind these
functions; if the library is missing they raise instead of computing anything.
Tensors are torch CUDA tensors passed by data pointer; the stream defaults to
torch's current stream on the tensor's device.
"""
import ctypes
import os
import re

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libep_gb300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "ep_gb300.h")

EP_BF16, EP_FP32, EP_FP8_E4M3, EP_FP4X2 = 0, 1, 2, 3
EP_OK, EP_EINVAL, EP_EUNSUPPORTED, EP_ECUDA, EP_ENOMEM = 0, -1, -2, -3, -4
(FIELD_NUM_UNALIGNED_PER_EXPERT, FIELD_NUM_TOKENS_PER_RANK, FIELD_PSUM_PER_EXPERT,
 FIELD_PSUM_PER_RANK, FIELD_DST_SLOT, FIELD_RECV_SRC_METADATA, FIELD_NUM_RECV,
 FIELD_DEVICE_ERROR, FIELD_TOPK_IDX, FIELD_SEND_SLOT) = range(10)
ERR_BAD_EXPERT, ERR_TIMEOUT = 1, 2

_DTYPES = {"bf16": EP_BF16, "fp32": EP_FP32, "fp8": EP_FP8_E4M3, "fp8_e4m3": EP_FP8_E4M3,
           "fp4x2": EP_FP4X2}


class ep_cfg_t(ctypes.Structure):
    _fields_ = [("world_size", ctypes.c_int32), ("hidden_dim", ctypes.c_int32),
                ("max_tok_per_rank", ctypes.c_int32), ("num_expert_per_rank", ctypes.c_int32),
                ("num_expert_per_token", ctypes.c_int32), ("expert_alignment", ctypes.c_int32),
                ("dispatch_dtype", ctypes.c_int32), ("use_weights", ctypes.c_int32),
                ("no_expand", ctypes.c_int32)]


class EpError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("ep error %d: %s" % (code, msg))
        self.code = code


_lib = None


def load_library():
    """Load libep_gb300.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libep_gb300.so is not built (%s); run __graft_entry__.build() or "
                          "python combine_ep_layout_gb300/build.py" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    c = ctypes
    vp, i32, i64 = c.c_void_p, c.c_int32, c.c_int64
    L.ep_recv_capacity.restype = i64
    L.ep_recv_capacity.argtypes = [c.POINTER(ep_cfg_t)]
    L.ep_handle_create.restype = c.c_int
    L.ep_handle_create.argtypes = [c.POINTER(ep_cfg_t), c.POINTER(vp)]
    L.ep_handle_create_shared.restype = c.c_int
    L.ep_handle_create_shared.argtypes = [c.POINTER(ep_cfg_t), vp, c.POINTER(vp)]
    L.ep_layout.restype = c.c_int
    L.ep_layout.argtypes = [vp, vp, i32, vp]
    L.ep_dispatch.restype = c.c_int
    L.ep_dispatch.argtypes = [vp, vp, vp, vp, vp]
    L.ep_combine.restype = c.c_int
    L.ep_combine.argtypes = [vp, vp, vp, vp, vp]
    L.ep_dispatch_fwd.restype = c.c_int
    L.ep_dispatch_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    L.ep_combine_ex.restype = c.c_int
    L.ep_combine_ex.argtypes = [vp, vp, vp, vp, vp, i32, vp]
    L.ep_handle_free.restype = None
    L.ep_handle_free.argtypes = [vp]
    L.ep_handle_get.restype = c.c_int
    L.ep_handle_get.argtypes = [vp, i32, c.POINTER(vp), c.POINTER(i64)]
    L.ep_handle_status.restype = c.c_int
    L.ep_handle_status.argtypes = [vp, c.POINTER(i32)]
    L.ep_handle_variant.restype = c.c_int
    L.ep_handle_variant.argtypes = [vp, i32, c.c_char_p, i32]
    L.ep_last_error.restype = c.c_char_p
    L.ep_last_error.argtypes = []
    L.ep_jit_precompile.restype = c.c_int
    L.ep_jit_precompile.argtypes = [c.POINTER(ep_cfg_t), c.c_char_p, c.c_char_p, i32]
    L.ep_layout_noalloc.restype = c.c_int
    L.ep_layout_noalloc.argtypes = [c.POINTER(ep_cfg_t), vp, i32] + [vp] * 8 + [vp]
    _lib = L
    return L


def declared_symbols():
    """Names of the functions include/ep_gb300.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[\w\s\*]*?\b(ep_\w+)\s*\(", text, flags=re.M)))


def ep_last_error():
    return load_library().ep_last_error().decode()


def _check(rc):
    if rc != EP_OK:
        raise EpError(rc, ep_last_error())


def make_cfg(world_size, hidden_dim, max_tok_per_rank, num_expert_per_rank, num_expert_per_token,
             expert_alignment=1, dispatch_dtype="bf16", use_weights=True, no_expand=False):
    dt = _DTYPES[dispatch_dtype] if isinstance(dispatch_dtype, str) else int(dispatch_dtype)
    return ep_cfg_t(world_size, hidden_dim, max_tok_per_rank, num_expert_per_rank,
                    num_expert_per_token, expert_alignment, dt, int(bool(use_weights)),
                    int(bool(no_expand)))


def ep_recv_capacity(cfg):
    r = load_library().ep_recv_capacity(ctypes.byref(cfg))
    if r < 0:
        raise EpError(int(r), ep_last_error())
    return int(r)


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _require(cond, msg):
    """Argument checks that survive python -O (unlike assert)."""
    if not cond:
        raise ValueError(msg)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


class _DevArray:
    """A raw device buffer of int32, exposed to torch via __cuda_array_interface__."""

    def __init__(self, ptr, shape):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<i4",
                                         "data": (int(ptr), False), "version": 3,
                                         "strides": None}


class EpHandle:
    """Owner of an ep_handle_t; methods mirror the C entry points."""

    def __init__(self, cfg, layout_of=None):
        """layout_of: another EpHandle whose layout this one uses
        (ep_handle_create_shared); it must outlive this handle."""
        self.cfg = cfg
        self.device = torch.cuda.current_device()
        h = ctypes.c_void_p()
        if layout_of is None:
            _check(load_library().ep_handle_create(ctypes.byref(cfg), ctypes.byref(h)))
        else:
            _check(load_library().ep_handle_create_shared(ctypes.byref(cfg), layout_of.ptr,
                                                          ctypes.byref(h)))
        self._layout_of = layout_of          # keeps the layout's owner alive
        self._h = h
        self.recv_capacity = ep_recv_capacity(cfg)
        self.num_tokens = 0

    @property
    def ptr(self):
        if self._h is None:
            raise EpError(EP_EINVAL, "handle already freed")
        return self._h

    def layout(self, topk_idx, num_tokens=None, stream=None):
        _require(topk_idx.dtype == torch.int64 and topk_idx.is_cuda and topk_idx.is_contiguous(),
                 "topk_idx must be a contiguous int64 CUDA tensor")
        _require(topk_idx.dim() == 2 and topk_idx.shape[1] == self.cfg.num_expert_per_token,
                 "topk_idx must be [num_tokens, num_expert_per_token]")
        n = topk_idx.shape[0] if num_tokens is None else int(num_tokens)
        _check(load_library().ep_layout(self.ptr, _ptr(topk_idx) if n else None, n,
                                        _stream_ptr(stream, self.device)))
        self.num_tokens = n

    def dispatch(self, x, recv_x, recv_scales=None, topk_weights=None, recv_topk_weights=None,
                 recv_topk_idx=None, stream=None):
        """ep_dispatch, or ep_dispatch_fwd when recv_topk_weights / recv_topk_idx are given."""
        _require(x.is_cuda and x.is_contiguous() and recv_x.is_contiguous(),
                 "x and recv_x must be contiguous CUDA tensors")
        for t in (recv_scales, topk_weights, recv_topk_weights, recv_topk_idx):
            _require(t is None or t.is_contiguous(), "optional dispatch tensors must be contiguous")
        L = load_library()
        st = _stream_ptr(stream, self.device)
        if recv_topk_weights is None and recv_topk_idx is None:
            _check(L.ep_dispatch(self.ptr, _ptr(x), _ptr(recv_x), _ptr(recv_scales), st))
        else:
            _check(L.ep_dispatch_fwd(self.ptr, _ptr(x), _ptr(recv_x), _ptr(recv_scales),
                                     _ptr(topk_weights), _ptr(recv_topk_weights),
                                     _ptr(recv_topk_idx), st))

    def combine(self, y, topk_weights, out, bias=None, stream=None):
        """ep_combine, or ep_combine_ex when a bias is given or out is fp32."""
        _require(y.is_cuda and y.is_contiguous() and out.is_contiguous(),
                 "y and out must be contiguous CUDA tensors")
        _require(topk_weights is None or topk_weights.is_contiguous(),
                 "topk_weights must be contiguous")
        _require(bias is None or (bias.dtype == torch.bfloat16 and bias.is_contiguous()),
                 "bias must be a contiguous bf16 tensor")
        _require(out.dtype in (torch.bfloat16, torch.float32), "out must be bf16 or fp32")
        L = load_library()
        st = _stream_ptr(stream, self.device)
        if bias is None and out.dtype == torch.bfloat16:
            _check(L.ep_combine(self.ptr, _ptr(y), _ptr(topk_weights), _ptr(out), st))
        else:
            odt = EP_FP32 if out.dtype == torch.float32 else EP_BF16
            _check(L.ep_combine_ex(self.ptr, _ptr(y), _ptr(topk_weights), _ptr(bias), _ptr(out),
                                   odt, st))

    def field(self, field):
        """A torch int32 view (no copy) of one handle field on the handle's device;
        valid until the handle is freed, and overwritten by the next layout."""
        p, n = ctypes.c_void_p(), ctypes.c_int64()
        _check(load_library().ep_handle_get(self.ptr, field, ctypes.byref(p), ctypes.byref(n)))
        K = self.cfg.num_expert_per_token
        shape = (n.value,)
        if field in (FIELD_DST_SLOT, FIELD_SEND_SLOT):
            shape = (n.value // K, K)
        elif field == FIELD_TOPK_IDX:
            shape = (n.value // K, K)
        elif field == FIELD_RECV_SRC_METADATA:
            shape = (n.value // (K + 2), K + 2)
        dev = torch.device("cuda", self.device)
        if n.value == 0:
            return torch.zeros(shape, dtype=torch.int32, device=dev)
        return torch.as_tensor(_DevArray(p.value or 0, shape), device=dev)

    def status(self):
        v = ctypes.c_int32()
        _check(load_library().ep_handle_status(self.ptr, ctypes.byref(v)))
        return v.value

    def variant(self, step):
        buf = ctypes.create_string_buffer(128)
        _check(load_library().ep_handle_variant(self.ptr, step, buf, 128))
        return buf.value.decode()

    def free(self):
        if self._h is not None:
            load_library().ep_handle_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


# Function-style API with the C names.
def ep_handle_create(cfg):
    return EpHandle(cfg)


def ep_handle_create_shared(cfg, layout_src):
    return EpHandle(cfg, layout_of=layout_src)


def ep_layout(h, topk_idx, num_tokens=None, stream=None):
    h.layout(topk_idx, num_tokens, stream)


def ep_dispatch(h, x, recv_x, recv_scales=None, stream=None):
    h.dispatch(x, recv_x, recv_scales, stream=stream)


def ep_dispatch_fwd(h, x, recv_x, recv_scales, topk_weights, recv_topk_weights, recv_topk_idx,
                    stream=None):
    h.dispatch(x, recv_x, recv_scales, topk_weights, recv_topk_weights, recv_topk_idx, stream)


def ep_combine(h, y, topk_weights, out, stream=None):
    h.combine(y, topk_weights, out, stream=stream)


def ep_combine_ex(h, y, topk_weights, bias, out, stream=None):
    h.combine(y, topk_weights, out, bias, stream)


def ep_handle_free(h):
    h.free()


def ep_handle_get(h, field):
    return h.field(field)


def ep_handle_status(h):
    return h.status()


def ep_handle_variant(h, step):
    return h.variant(step)


NOALLOC_OUTPUTS = ("num_unaligned_per_expert", "num_tokens_per_rank", "psum_per_expert",
                   "psum_per_rank", "num_recv", "dst_slot", "recv_src_metadata", "device_error")


def ep_layout_noalloc(cfg, topk_idx, out, stream=None):
    """Layout into caller-owned int32 CUDA tensors (dict keyed by NOALLOC_OUTPUTS);
    the library allocates nothing for this call."""
    n = topk_idx.shape[0]
    _require(topk_idx.dtype == torch.int64 and topk_idx.is_cuda and topk_idx.is_contiguous(),
             "topk_idx must be a contiguous int64 CUDA tensor")
    for k in NOALLOC_OUTPUTS:
        _require(out[k].dtype == torch.int32 and out[k].is_cuda and out[k].is_contiguous(),
                 "%s must be a contiguous int32 CUDA tensor" % k)
    _check(load_library().ep_layout_noalloc(
        ctypes.byref(cfg), _ptr(topk_idx) if n else None, n,
        *[_ptr(out[k]) for k in NOALLOC_OUTPUTS], _stream_ptr(stream, topk_idx.device)))


def ep_jit_precompile(cfg, arch=None):
    """Compile (or find in the disk cache) the run-time specialisations cfg would
    use; returns (number compiled now, report lines).  Needs NVRTC, not a GPU."""
    buf = ctypes.create_string_buffer(8192)
    rc = load_library().ep_jit_precompile(ctypes.byref(cfg), arch.encode() if arch else None,
                                          buf, 8192)
    if rc < 0:
        raise EpError(rc, ep_last_error())
    return rc, buf.value.decode().splitlines()
