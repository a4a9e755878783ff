"""Seeded synthetic inputs for kernelised linear attention.

This module holds random-number generation only (no attention arithmetic):
it is the single piece shared by the CUDA path's tests/bench and the oracle.

Recipe: one CPU ``torch.Generator`` seeded with ``seed`` draws fp32 N(0, 1)
tensors in the order Q, K, V; each is multiplied by ``scale`` and then cast to
the requested dtype (round-to-nearest-even for bf16).  Layout is the library's:
Q, K [B, H, N, D], V [B, H, N, M], row-major.

The named workloads below are the shapes of the image-pixel autoregression
and long-sequence experiments of "Transformers are RNNs" (sec. 4.1.2 sweeps
N = 2^9 .. 2^16; sec. 4.2.2 generates CIFAR-10 images as N = 3072 pixels),
with synthetic values standing in for the datasets.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    op: str            # "causal" | "noncausal" | "decode"
    B: int
    H: int
    N: int             # tokens per sequence (decode: prefill length)
    D: int
    M: int
    dtype: torch.dtype
    scale: float       # multiplies N(0, 1) draws
    chunk: int = 0     # causal chunk length (0 = library default)
    steps: int = 0     # decode: sequential steps after the prefill
    seed: int = 0
    variant: tuple = ()  # (feature map, nu, norm, update) of a variant workload; () = elu + 1

    @property
    def tokens(self) -> int:
        return self.B * self.N


WORKLOADS = {
    "causal_tiny_f32": Workload("causal_tiny_f32", "causal", 1, 1, 64, 16, 16, torch.float32, 1.0, 0, 0, 1001),
    "noncausal_b8h8n4096d64": Workload("noncausal_b8h8n4096d64", "noncausal", 8, 8, 4096, 64, 64,
                                       torch.bfloat16, 1.0, 0, 0, 1002),
    # The causal workloads are configured with chunk C = 64.  The library takes
    # the chunk length as a hint: its tensor-core path groups the same sums by
    # 128 rows (one tcgen05 M = 128 tile), the same computation in exact
    # arithmetic (chunk-length invariance is a parity test).
    "causal_b16h8n3072d64": Workload("causal_b16h8n3072d64", "causal", 16, 8, 3072, 64, 64,
                                     torch.bfloat16, 1.0 / math.sqrt(64), 64, 0, 1003),
    "causal_b1h16n65536d128": Workload("causal_b1h16n65536d128", "causal", 1, 16, 65536, 128, 128,
                                       torch.bfloat16, 1.0 / math.sqrt(128), 64, 0, 1004),
    "decode_b256h16d64": Workload("decode_b256h16d64", "decode", 256, 16, 1024, 64, 64,
                                  torch.bfloat16, 1.0, 0, 4096, 1005),
    # Variants on the training shape: the delta rule with sum-normalised elu + 1
    # features, and the sum rule with sum-normalised DPFP-1 features (F = 128).
    "delta_b16h8n3072d64": Workload("delta_b16h8n3072d64", "causal_variant", 16, 8, 3072, 64, 64,
                                    torch.bfloat16, 1.0 / math.sqrt(64), 0, 0, 1006, ("elu1", 1, "sum", "delta")),
    "dpfp_b16h8n3072d64": Workload("dpfp_b16h8n3072d64", "causal_variant", 16, 8, 3072, 64, 64,
                                   torch.bfloat16, 1.0 / math.sqrt(64), 0, 0, 1007, ("dpfp", 1, "sum", "sum")),
}


def betas(B, H, N, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Per-token interpolation weights of the delta rule, [B, H, N], drawn
    uniform on [0, 1) and cast to dtype."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    return torch.rand((B, H, N), generator=g, dtype=torch.float32, device=device).to(dtype).contiguous()


def qkv(B, H, N, D, M, dtype=torch.bfloat16, scale=1.0, seed=0, device="cpu"):
    """Q, K [B,H,N,D] and V [B,H,N,M], drawn Q then K then V.

    On the CPU (the default, used by every parity test) the values are the
    CPU generator's; ``device="cuda..."`` draws with that device's generator
    instead (a different, equally seeded stream, used only for timing)."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    out = []
    for shape in ((B, H, N, D), (B, H, N, D), (B, H, N, M)):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        if scale != 1.0:
            x = x * scale
        out.append(x.to(dtype).contiguous())
    return tuple(out)


def state(B, H, D, M, seed=0, scale=1.0):
    """A random fp32 state pair (S [B,H,D,M], z [B,H,D]) with z > 0, for carry tests.

    z is drawn as |N(0,1)| * D + 1 so that it is positive like any sum of
    feature-map values; S entries are N(0, 1) * scale * D."""
    g = torch.Generator().manual_seed(int(seed))
    S = torch.randn((B, H, D, M), generator=g, dtype=torch.float32) * (scale * D)
    z = torch.randn((B, H, D), generator=g, dtype=torch.float32).abs() * D + 1.0
    return S.contiguous(), z.contiguous()


def decode_tokens(steps, B, H, D, M, dtype=torch.bfloat16, seed=0, scale=1.0, device="cpu"):
    """Per-step decode inputs drawn as one block [steps, 3, B, H, max(D, M)] and
    split into q [steps,B,H,D], k [steps,B,H,D], v [steps,B,H,M] (q, k, v per step).
    ``device`` as in :func:`qkv`."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    W = max(D, M)
    x = torch.randn((steps, 3, B, H, W), generator=g, dtype=torch.float32, device=device)
    if scale != 1.0:
        x = x * scale
    x = x.to(dtype)
    return x[:, 0, :, :, :D].contiguous(), x[:, 1, :, :, :D].contiguous(), x[:, 2, :, :, :M].contiguous()


def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank ``rank``'s share when several processes each take an
    independent batch of a workload: rank 0 keeps ``seed``, the others are
    offset by a prime so that no two ranks draw the same stream."""
    if rank < 0:
        raise ValueError("rank must be >= 0")
    return int(seed) + 7919 * int(rank)


def workload_inputs(w: Workload, rank: int = 0):
    """Inputs of a named workload: (q, k, v) on the CPU, rank ``rank``'s batch."""
    return qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.scale, rank_seed(w.seed, rank))


def workload_betas(w: Workload, rank: int = 0):
    """Delta-rule weights of a named workload, [B, H, N], from their own seed stream."""
    return betas(w.B, w.H, w.N, w.dtype, rank_seed(w.seed, rank) + 1000000)
