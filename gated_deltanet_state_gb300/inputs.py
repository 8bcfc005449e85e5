"""Seeded synthetic inputs shaped like the pages' GDN layers.

This module holds no arithmetic of the method: it only draws random numbers
with a torch CPU generator and shapes them.  Both the CUDA path and the CPU
oracle consume exactly these tensors (after copying to the device), so the two
see identical bits.

Value recipe (the same for every workload):
  x      ~ N(0, 1), rounded to the input dtype    pre-conv rows, [T, conv_dim]
  g      = -softplus(N(0, 1)) * 0.1               log decay (a = exp(g)), [T, Hv]
  beta   = sigmoid(N(0, 1))                       write strength, [T, Hv]
  conv_w = 0.5 * N(0, 1)                          depthwise taps, [conv_dim, 4]
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

F32, BF16 = 0, 1
_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


@dataclass(frozen=True)
class LayerShape:
    """Shape of one GDN layer plus the cache geometry it is served with."""
    num_qk_heads: int
    num_v_heads: int
    head_dim_k: int
    head_dim_v: int
    block_size: int
    chunk_size: int
    in_dtype: int = BF16
    out_dtype: int = BF16
    page_bytes: int = 0          # 0: the exact state size rounded up to 256 B
    q_scale: float = 1.0
    norm_eps: float = 1e-6

    @property
    def conv_dim(self) -> int:
        return 2 * self.num_qk_heads * self.head_dim_k + self.num_v_heads * self.head_dim_v

    @property
    def in_bytes(self) -> int:
        return 2 if self.in_dtype == BF16 else 4

    @property
    def state_bytes(self) -> int:
        return self.num_v_heads * self.head_dim_v * self.head_dim_k * 4

    @property
    def window_bytes(self) -> int:
        return 3 * self.conv_dim * self.in_bytes

    @property
    def payload_bytes(self) -> int:
        return self.state_bytes + self.window_bytes

    @property
    def page(self) -> int:
        if self.page_bytes:
            return self.page_bytes
        return (self.payload_bytes + 255) // 256 * 256

    def torch_in(self) -> torch.dtype:
        return _TORCH_DTYPE[self.in_dtype]

    def torch_out(self) -> torch.dtype:
        return _TORCH_DTYPE[self.out_dtype]


# Tiny layer: 2 qk / 2 v heads, d = 32, block 64, chunk 16, fp32 in and out.
TINY = LayerShape(2, 2, 32, 32, block_size=64, chunk_size=16, in_dtype=F32, out_dtype=F32)
# 27B-shaped layer: 16 qk heads, 48 v heads, d = 128, block 896 tokens; the
# page is one 896-token attention page of 4,096 B per token (3,670,016 B).
QWEN27B = LayerShape(16, 48, 128, 128, block_size=896, chunk_size=64, page_bytes=896 * 4096)
# 4B-shaped layer: 16 qk heads, 32 v heads, d = 128; 2.5 MiB pages.  The
# block size is not used by decode or replay; 640 = 2.5 MiB / 4 KiB.
QWEN4B = LayerShape(16, 32, 128, 128, block_size=640, chunk_size=64, page_bytes=5 * 512 * 1024)


def with_(shape: LayerShape, **kw) -> LayerShape:
    return replace(shape, **kw)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def token_inputs(shape: LayerShape, n_tokens: int, seed: int) -> dict:
    """x [T, conv_dim] (input dtype), g and beta [T, Hv] (fp32), on the CPU."""
    gen = _gen(seed)
    x = torch.randn(n_tokens, shape.conv_dim, generator=gen).to(shape.torch_in())
    g = -torch.nn.functional.softplus(torch.randn(n_tokens, shape.num_v_heads, generator=gen)) * 0.1
    beta = torch.sigmoid(torch.randn(n_tokens, shape.num_v_heads, generator=gen))
    return {"x": x.contiguous(), "g": g.float().contiguous(), "beta": beta.float().contiguous()}


def conv_weights(shape: LayerShape, seed: int) -> torch.Tensor:
    """Depthwise conv taps [conv_dim, 4], fp32."""
    gen = _gen(seed + 7919)
    return (0.5 * torch.randn(shape.conv_dim, 4, generator=gen)).float().contiguous()


def random_state(shape: LayerShape, n: int, seed: int, scale: float = 0.3) -> dict:
    """Arbitrary starting states S [n, Hv, dv, dk] fp32 and windows
    [n, 3, conv_dim] (input dtype), for tests that start from a non-zero page."""
    gen = _gen(seed + 104729)
    S = scale * torch.randn(n, shape.num_v_heads, shape.head_dim_v, shape.head_dim_k, generator=gen)
    win = torch.randn(n, 3, shape.conv_dim, generator=gen).to(shape.torch_in())
    return {"S": S.float().contiguous(), "win": win.contiguous()}


def permutation(n: int, seed: int) -> torch.Tensor:
    """A seeded random permutation of range(n), int32 (page ids)."""
    return torch.randperm(n, generator=_gen(seed + 15485863)).to(torch.int32)


def accept_lengths(n: int, hi: int, seed: int) -> torch.Tensor:
    """Accepted rows per request, uniform on [0, hi], int32."""
    return torch.randint(0, hi + 1, (n,), generator=_gen(seed + 32452843)).to(torch.int32)
