"""PyTorch layers over the fused graph-attention kernels.

"On Efficient Scaling of GNNs via IO-Aware Layers Implementations", zh/ko
technical summaries, "Methodology" (the layers are meant as drop-in
replacements) and results (GATv2: peak memory cut because no edge-wise
tensor is materialised).

``graph_attention`` is an autograd function whose forward is ``gattn_fwd``
and whose backward is ``gattn_bwd``: it saves only the node tensors (Q, K, V,
out) and the per-node lse, never an O(M*H) edge tensor.  The two modules put
the usual projections around it (plain dense GEMMs, run by torch/cuBLAS):

* ``GraphTransformerConv``: Q, K, V = x W_q, x W_k, x W_v (H heads of D),
  dot-product attention over the in-neighbours, heads concatenated, output
  projection W_o.
* ``GATv2Conv``: x_l = x W_l, x_r = x W_r; score a . LeakyReLU(x_l[i] +
  x_r[j]), the message of source j is x_r[j] (one tensor passed as both K
  and V; its gradient is dK + dV), heads concatenated.

Both run the attention in the dtype of their parameters (bf16 by default)
with fp32 arithmetic inside the kernels.
"""
from __future__ import annotations

import math

import torch
from torch import nn

from . import binding as gb


class _GraphAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, plan, kind, scale, slope, Q, K, V, a):
        score = gb.Score(kind, scale=scale, a=a, neg_slope=slope)
        out, lse = gb.gattn_fwd(plan, Q, K, V, score)
        ctx.plan, ctx.score = plan, score
        ctx.save_for_backward(Q, K, V, out, lse, a if a is not None else torch.empty(0))
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        Q, K, V, out, lse, a = ctx.saved_tensors
        dout = dout.to(Q.dtype).contiguous()
        dQ, dK, dV, da = gb.gattn_bwd(ctx.plan, Q, K, V, out, dout, lse, ctx.score)
        return None, None, None, None, dQ, dK, dV, da


def graph_attention(plan: gb.Plan, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                    kind: str = "dot", scale: float = 0.0, a: torch.Tensor | None = None,
                    neg_slope: float = 0.2):
    """Fused softmax attention over each destination's in-neighbours.

    Q, K, V: contiguous CUDA [N, H, D] (fp32 or bf16); for ``kind="gatv2"``
    ``a`` is a contiguous fp32 CUDA [H, D] parameter.  Returns (out [N, H, D],
    lse fp32 [N, H]); differentiable in Q, K, V and a.
    """
    if kind == "gatv2" and (a is None or a.dtype != torch.float32 or not a.is_contiguous()):
        raise ValueError("GATv2 needs a contiguous fp32 tensor a of shape [H, D]")
    return _GraphAttention.apply(plan, kind, float(scale), float(neg_slope), Q.contiguous(),
                                 K.contiguous(), V.contiguous(), a if kind == "gatv2" else None)


class GraphTransformerConv(nn.Module):
    """Multi-head graph-transformer attention layer (dot score)."""

    def __init__(self, in_dim: int, heads: int, head_dim: int, out_dim: int | None = None,
                 dtype=torch.bfloat16, device=None):
        super().__init__()
        self.heads, self.head_dim = heads, head_dim
        hd = heads * head_dim
        kw = {"dtype": dtype, "device": device}
        self.q = nn.Linear(in_dim, hd, bias=False, **kw)
        self.k = nn.Linear(in_dim, hd, bias=False, **kw)
        self.v = nn.Linear(in_dim, hd, bias=False, **kw)
        self.o = nn.Linear(hd, out_dim or hd, bias=False, **kw)

    def forward(self, x: torch.Tensor, plan: gb.Plan) -> torch.Tensor:
        N = x.shape[0]
        shape = (N, self.heads, self.head_dim)
        Q, K, V = (p(x).view(shape) for p in (self.q, self.k, self.v))
        out, _ = graph_attention(plan, Q, K, V, "dot", 1.0 / math.sqrt(self.head_dim))
        return self.o(out.reshape(N, self.heads * self.head_dim))


class GATv2Conv(nn.Module):
    """Multi-head GATv2 attention layer (messages x_r[j], heads concatenated)."""

    def __init__(self, in_dim: int, heads: int, head_dim: int, negative_slope: float = 0.2,
                 dtype=torch.bfloat16, device=None):
        super().__init__()
        self.heads, self.head_dim, self.slope = heads, head_dim, negative_slope
        hd = heads * head_dim
        kw = {"dtype": dtype, "device": device}
        self.lin_l = nn.Linear(in_dim, hd, bias=False, **kw)
        self.lin_r = nn.Linear(in_dim, hd, bias=False, **kw)
        self.att = nn.Parameter(torch.randn(heads, head_dim, device=device) / math.sqrt(head_dim))

    def forward(self, x: torch.Tensor, plan: gb.Plan) -> torch.Tensor:
        N = x.shape[0]
        shape = (N, self.heads, self.head_dim)
        xl = self.lin_l(x).view(shape)
        xr = self.lin_r(x).view(shape)
        out, _ = graph_attention(plan, xl, xr, xr, "gatv2", a=self.att, neg_slope=self.slope)
        return out.reshape(N, self.heads * self.head_dim)
