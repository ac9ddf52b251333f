"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the tests, the benchmark and the oracle-side checks.
It draws random tensors and describes workload shapes; it holds none of the
attention arithmetic.

Workloads (shapes and value distributions follow the 1B-LLM prefill setting of
"Android Transformer Optimization: Attention and Mobile GPU Bottlenecks",
section "The Self-Attention Bottleneck Is Memory Traffic, Not Compute", which
discusses sequence length n=2048 in fp16, and the 32-head, D=128 setting of
"Flash Attention on Android: tiled SGEMM with RenderScript", section
"Benchmark results"):

  c1        B=1 H=1  N=256   D=64  fp16  non-causal  Q,K,V ~ N(0,1)
  c2        B=1 H=32 N=1024  D=64  fp16  causal      Q,K,V ~ N(0,1)
  c3        B=1 H=32 N=2048  D=64  fp16  non-causal  Q,K,V ~ N(0,1)
  c3c       same inputs as c3, causal
  c4        B=4 H=16 N=4096  D=128 bf16  causal      Q,K,V ~ N(0,1)
  c5        B=1 H=8  N=16384 D=128 fp16  non-causal  Q,K ~ 4*N(0,1), V ~ U(-1,1)
  p2s512    B=1 H=32 N=512   D=128 fp16  non-causal  Q,K,V ~ N(0,1)
  p2s1024   B=1 H=32 N=1024  D=128 fp16  non-causal  Q,K,V ~ N(0,1)
  lc1       B=1 H=1  N=16384 D=128 fp16  causal      Q,K,V ~ N(0,1)
  c2_f32    c2 in fp32 storage;  c3_f32   c3 in fp32 storage (same seeds, draws not rounded)

The last two are the second workload shape of "Flash Attention on Android: tiled SGEMM
with RenderScript" (section "Benchmark results": 32-head attention at head dim 128,
sequence 512 and 1024); that page measured FP32, this library computes in fp16/bf16.
``c2_f32`` and ``c3_f32`` are the first page's fp32-storage variant (section "Pitfalls I
Hit": an fp32 build beside the fp16 one) on the headline and n=2048 shapes; the fp32 draws are
used as they are. ``lc1`` is one long causal sequence with a single head: 128 query tiles, fewer than the
GPU's SMs, the longest of them 128 key tiles long. It is the case the split-KV forward
(partial results over key ranges, merged with the online-softmax update of the first
page's section "The Essence of FlashAttention: Reordering the Computation") is for.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw q, k, v in that
order as fp32 (``randn``; v of c5 as ``rand*2-1``), multiply q and k by the
workload's ``qk_mult`` (4 for c5; exact in binary), then round to the I/O
dtype with ``.to(dtype)``. The rounded tensors are the inputs of both the
CUDA path and the oracle.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import torch

__all__ = ["Workload", "WORKLOADS", "make_qkv", "attention_flops", "min_dram_bytes"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str  # "fp16" | "bf16" | "fp32"
    causal: bool
    seed: int
    qk_mult: float = 1.0
    v_uniform: bool = False
    note: str = ""

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}[self.dtype]

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 256, 64, "fp16", False, 1001,
                   note="single head, N=256, D=64, fp16, non-causal"),
    "c2": Workload("c2", 1, 32, 1024, 64, "fp16", True, 1002,
                   note="1B-class LLM prefill: 32 heads, N=1024, D=64, fp16, causal"),
    "c3": Workload("c3", 1, 32, 2048, 64, "fp16", False, 1003,
                   note="n=2048 case: 32 heads, D=64, fp16, non-causal"),
    "c3c": Workload("c3c", 1, 32, 2048, 64, "fp16", True, 1003,
                    note="n=2048 case: 32 heads, D=64, fp16, causal"),
    "c4": Workload("c4", 4, 16, 4096, 128, "bf16", True, 1004,
                   note="batched prefill: B=4, 16 heads, N=4096, D=128, bf16, causal"),
    "c5": Workload("c5", 1, 8, 16384, 128, "fp16", False, 1005, qk_mult=4.0, v_uniform=True,
                   note="long sequence: 8 heads, N=16384, D=128, fp16, Q,K x4, V~U(-1,1), non-causal"),
    "p2s512": Workload("p2s512", 1, 32, 512, 128, "fp16", False, 1006,
                       note="7B-class shape: 32 heads, N=512, D=128, fp16, non-causal"),
    "p2s1024": Workload("p2s1024", 1, 32, 1024, 128, "fp16", False, 1007,
                        note="7B-class shape: 32 heads, N=1024, D=128, fp16, non-causal"),
    "lc1": Workload("lc1", 1, 1, 16384, 128, "fp16", True, 1008,
                    note="one long causal sequence: 1 head, N=16384, D=128, fp16"),
    "c2_f32": Workload("c2_f32", 1, 32, 1024, 64, "fp32", True, 1002,
                       note="c2 with fp32 storage (tf32 tensor cores): 32 heads, N=1024, D=64, causal"),
    "c3_f32": Workload("c3_f32", 1, 32, 2048, 64, "fp32", False, 1003,
                       note="n=2048 case with fp32 storage (tf32 tensor cores): 32 heads, D=64, non-causal"),
}


def make_qkv(w: Workload):
    """Return (q, k, v) as contiguous CPU tensors [B,H,N,D] in the workload dtype."""
    g = torch.Generator(device="cpu").manual_seed(int(w.seed))
    shape = (w.B, w.H, w.N, w.D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.v_uniform:
        v = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.qk_mult != 1.0:
        q.mul_(w.qk_mult)
        k.mul_(w.qk_mult)
    dt = w.torch_dtype
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def attention_flops(B: int, H: int, N: int, D: int, causal: bool) -> float:
    """Algorithmic FLOPs: 4*N^2*D per head, half of that when causal."""
    f = 4.0 * N * N * D * B * H
    return f / 2.0 if causal else f


def min_dram_bytes(B: int, H: int, N: int, D: int, elem_bytes: int = 2, with_lse: bool = True) -> int:
    """|Q|+|K|+|V|+|O| (+|LSE| in fp32): the traffic floor of one forward pass."""
    b = 4 * B * H * N * D * elem_bytes
    if with_lse:
        b += 4 * B * H * N
    return b
