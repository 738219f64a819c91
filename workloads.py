"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method: it only draws random numbers
and names the problem shapes. Recipe: a CPU ``torch.Generator`` seeded with
``seed`` draws q, k, v in that order as float32 standard normals (the
``[B, H, N, D]`` layout, D innermost), optionally scales k by an exact power of
two, then casts to the problem dtype. Decode steps draw one token per step
from the seed ``seed * 1_000_003 + step``.
"""
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                 # "causal", "noncausal", "decode" or "causal+noncausal"
    B: int
    H: int
    N: int                  # sequence length (decode: number of steps)
    D: int                  # Dk = Dv
    dtype: str              # "f32" or "bf16"
    k_scale: float = 1.0    # k is multiplied by this before the dtype cast
    note: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.N


# Shapes of the pages' workloads: a 32x32x3 pixel-channel sequence (N = 3072),
# the 2^9..2^16 sequence-length sweep, and batched autoregressive generation.
WORKLOADS = {
    "tiny": Workload("tiny causal+non-causal B=1 H=1 N=256 D=64 f32", "causal+noncausal",
                     1, 1, 256, 64, "f32"),
    "image": Workload("causal B=8 H=8 N=3072 D=64 bf16", "causal", 8, 8, 3072, 64, "bf16",
                      note="32x32x3 pixel-channel sequence"),
    "long": Workload("causal B=2 H=8 N=65536 D=64 bf16 k*1/8", "causal", 2, 8, 65536, 64,
                     "bf16", k_scale=0.125, note="long context, K scaled by 1/sqrt(D)"),
    "bidir": Workload("non-causal B=16 H=8 N=8192 D=128 bf16", "noncausal", 16, 8, 8192, 128,
                      "bf16"),
    "decode": Workload("decode 512 seq x H=8 D=64 bf16, 3072 steps", "decode", 512, 8, 3072, 64,
                       "bf16", note="fp32 state resident in device memory"),
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return TORCH_DTYPES[name]


def make_qkv(B, H, N, D, dtype="f32", seed=0, k_scale=1.0, Dv=None):
    """Returns CPU tensors q, k [B,H,N,D] and v [B,H,N,Dv] in the given dtype."""
    Dv = D if Dv is None else Dv
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, N, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, N, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, N, Dv), generator=g, dtype=torch.float32)
    if k_scale != 1.0:
        k = k * k_scale
    dt = torch_dtype(dtype)
    return q.to(dt), k.to(dt), v.to(dt)


def make_features(B, H, N, C, dtype="f32", seed=0, Dv=None):
    """Non-negative feature inputs fq, fk [B,H,N,C] (uniform on [0, 1)) and v [B,H,N,Dv]
    (standard normal) as CPU tensors, for the identity feature map."""
    Dv = C if Dv is None else Dv
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    fq = torch.rand((B, H, N, C), generator=g, dtype=torch.float32)
    fk = torch.rand((B, H, N, C), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, N, Dv), generator=g, dtype=torch.float32)
    dt = torch_dtype(dtype)
    return fq.to(dt), fk.to(dt), v.to(dt)


def make_workload(w: Workload, seed=0):
    return make_qkv(w.B, w.H, w.N, w.D, w.dtype, seed=seed, k_scale=w.k_scale)


def decode_token(B, H, D, step, dtype="bf16", seed=0):
    """q, k, v [B,H,D] for one decode step (CPU tensors)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + int(step))
    q = torch.randn((B, H, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, D), generator=g, dtype=torch.float32)
    dt = torch_dtype(dtype)
    return q.to(dt), k.to(dt), v.to(dt)


def to_f64(t: torch.Tensor):
    """Exact upcast of the values a kernel sees (bf16/f32) to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()
