"""Seeded synthetic inputs for the MoE expert-parallel layout / dispatch / combine path.

This module only draws inputs.  It holds none of the method's arithmetic; the
CUDA library and the CPU oracle both take its outputs as given.

Recipes (one seed per workload, offset per array):
  x            bf16 of N(0,1) fp32 draws (torch generator on the target device)
  topk_idx     int64 [N, K]; "uniform": K distinct experts, uniform without
               replacement (first K of a random permutation of the E experts);
               "zipf": K draws without replacement with P(e) proportional to
               (e+1)^-s, renormalised over the experts not yet drawn
  topk_weights fp32 [N, K], softmax over the K chosen experts of N(0,1) logits
  y            bf16 of N(0,1) for expert outputs; rows that hold no token may
               be set to bf16 NaN so that any read of them poisons a result
"""
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    world_size: int          # W logical ranks
    max_tok_per_rank: int    # T
    num_tokens: int          # N <= W*T
    hidden: int              # H
    num_expert_per_rank: int # Epr, E = W*Epr
    topk: int                # K
    alignment: int           # A (1 = no padding)
    dispatch_dtype: str      # "bf16" or "fp8"
    use_weights: bool
    routing: str = "uniform" # "uniform" or "zipf"
    zipf_s: float = 0.0
    seed: int = 0xEB00

    @property
    def num_experts(self):
        return self.world_size * self.num_expert_per_rank

    @property
    def recv_capacity(self):
        return (self.world_size * self.max_tok_per_rank * self.topk
                + self.num_experts * (self.alignment - 1))

    def with_(self, **kw):
        return replace(self, **kw)


WORKLOADS = {
    # 128 tokens, hidden 1024, 32 experts over 4 logical ranks, top-4, no padding
    "tiny": Workload("tiny", 4, 32, 128, 1024, 8, 4, 1, "bf16", True, seed=0xEB00),
    # 8 ranks x 128 tokens, hidden 7168, 64 experts, top-8
    "decode": Workload("decode", 8, 128, 1024, 7168, 8, 8, 1, "bf16", True, seed=0xEB01),
    # 8 ranks x 4096 tokens, hidden 7168, 256 experts, top-8, alignment 128
    "prefill_bf16": Workload("prefill_bf16", 8, 4096, 32768, 7168, 32, 8, 128, "bf16", True,
                             seed=0xEB02),
    # the same shape, dispatch cast to e4m3 with per-128 fp32 scales
    "prefill_fp8": Workload("prefill_fp8", 8, 4096, 32768, 7168, 32, 8, 128, "fp8", True,
                            seed=0xEB03),
    # 16384 tokens, hidden 4096, 128 experts over 8 ranks, top-6 Zipf(1.2), alignment 64
    "skewed": Workload("skewed", 8, 2048, 16384, 4096, 16, 6, 64, "bf16", True,
                       routing="zipf", zipf_s=1.2, seed=0xEB04),
}


def _gen(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gen_topk(wl: Workload, seed_offset: int = 1, mask_frac: float = 0.0):
    """topk_idx int64 [N, K] on the CPU; with mask_frac > 0 that fraction of the
    entries is replaced by -1 (masked)."""
    g = _gen(wl.seed * 16 + seed_offset)
    N, E, K = wl.num_tokens, wl.num_experts, wl.topk
    if N == 0:
        return torch.zeros((0, K), dtype=torch.int64)
    if wl.routing == "uniform":
        keys = torch.rand((N, E), generator=g)
        idx = keys.argsort(dim=1)[:, :K].contiguous()
    elif wl.routing == "zipf":
        p = torch.arange(1, E + 1, dtype=torch.float64).pow(-wl.zipf_s)
        idx = torch.multinomial(p.expand(N, E), K, replacement=False, generator=g)
    else:
        raise ValueError(wl.routing)
    idx = idx.to(torch.int64)
    if mask_frac > 0:
        m = torch.rand((N, K), generator=g) < mask_frac
        idx[m] = -1
    return idx.contiguous()


def gen_weights(wl: Workload, seed_offset: int = 2):
    """topk_weights fp32 [N, K] on the CPU: softmax of N(0,1) logits."""
    g = _gen(wl.seed * 16 + seed_offset)
    logits = torch.randn((wl.num_tokens, wl.topk), generator=g, dtype=torch.float64)
    return torch.softmax(logits, dim=1).to(torch.float32).contiguous()


def gen_bf16_normal(rows: int, cols: int, seed: int, device="cpu"):
    """bf16 [rows, cols] of N(0,1) draws made on `device`."""
    g = _gen(seed, device)
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    step = max(1, (1 << 26) // max(cols, 1))      # bounded fp32 temporaries
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = torch.randn((r1 - r0, cols), generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def gen_x(wl: Workload, device="cpu", seed_offset: int = 3):
    """Token activations x, bf16 [N, H]."""
    return gen_bf16_normal(wl.num_tokens, wl.hidden, wl.seed * 16 + seed_offset, device)


def gen_y(wl: Workload, valid_rows=None, device="cpu", seed_offset: int = 4):
    """Expert outputs y, bf16 [Rcap, H]; rows where valid_rows is False are NaN."""
    y = gen_bf16_normal(wl.recv_capacity, wl.hidden, wl.seed * 16 + seed_offset, device)
    if valid_rows is not None:
        v = torch.as_tensor(valid_rows, device=device)
        y[~v] = float("nan")
    return y


def make_case(name_or_wl, device="cpu", mask_frac: float = 0.0):
    """Inputs of one workload: dict(wl, topk_idx (cpu), topk_weights (cpu), x (device))."""
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    return dict(wl=wl, topk_idx=gen_topk(wl, mask_frac=mask_frac),
                topk_weights=gen_weights(wl), x=gen_x(wl, device))


def bits16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
