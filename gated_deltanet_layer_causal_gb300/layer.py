"""The whole GDN layer: input projections -> GDN core -> output projection.

The core (conv1d+SiLU, L2 norms, gates, gated delta rule, gated RMSNorm) runs in
libgdn.so through :class:`core.GDNCore`; the four projections around it are
plain dense GEMMs (torch.nn.functional.linear, i.e. cuBLAS, in the activation
dtype with fp32 accumulation).  The shape follows the layers the pages time
("[6/8] feat(models): port Qwen3.5 / Qwen3-Next GDN to the head-sharded layer",
"GB300 results": Qwen3.8-Flash, hidden 2560, 16 k-heads, 48 v-heads; prime-rl
#3860, "Summary": GatedDeltaNet declares its projections and takes the output
gate type as a keyword):

    hidden [T, D_h] --W_qkv--> x [T, C]   (q, k, v channels, flat or group-major)
                    --W_z---> z [T, H_v, d_v]
                    --W_b---> b [T, H_v],  --W_a--> a [T, H_v]
    y = GDNCore(x, conv_w, a, b, A_log, dt_bias, z, norm_w)      [T, H_v, d_v]
    out = y.reshape(T, H_v d_v) W_out^T                          [T, D_h]

The projections are separate weights so that every core input is a dense,
contiguous tensor (no copy between a GEMM and the library).
"""
from __future__ import annotations

import math

import torch
import torch.nn.functional as F

from .core import gdn_core


class GDNLayer(torch.nn.Module):
    def __init__(self, hidden: int, h_k: int, h_v: int, d: int = 128, conv_k: int = 4,
                 gate: str = "silu", layout: str = "flat", dtype=torch.bfloat16, device=None):
        super().__init__()
        if d != 128 or conv_k != 4:
            raise ValueError("the GDN library implements d = 128 and a 4-tap conv")
        if h_v % h_k:
            raise ValueError("h_v must be a multiple of h_k")
        self.hidden, self.h_k, self.h_v, self.d = hidden, h_k, h_v, d
        self.gate, self.layout = gate, layout
        C = (2 * h_k + h_v) * d
        kw = dict(dtype=dtype, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.W_qkv = torch.nn.Parameter(torch.empty(C, hidden, **kw))
        self.W_z = torch.nn.Parameter(torch.empty(h_v * d, hidden, **kw))
        self.W_b = torch.nn.Parameter(torch.empty(h_v, hidden, **kw))
        self.W_a = torch.nn.Parameter(torch.empty(h_v, hidden, **kw))
        self.W_out = torch.nn.Parameter(torch.empty(hidden, h_v * d, **kw))
        self.conv_w = torch.nn.Parameter(torch.empty(C, conv_k, **f32))
        self.A_log = torch.nn.Parameter(torch.empty(h_v, **f32))
        self.dt_bias = torch.nn.Parameter(torch.empty(h_v, **f32))
        self.norm_w = torch.nn.Parameter(torch.empty(d, **f32))
        self.reset_parameters()

    @torch.no_grad()
    def reset_parameters(self, generator=None):
        """Random init: projections ~ U(+-1/sqrt(fan_in)), conv ~ U(+-1/2),
        A_log = ln U(1, 16), dt_bias = 0, norm weight ~ N(0, 0.02) (zero-centred)."""
        for W in (self.W_qkv, self.W_z, self.W_b, self.W_a, self.W_out):
            bound = 1.0 / math.sqrt(W.shape[1])
            W.copy_(torch.empty(W.shape).uniform_(-bound, bound, generator=generator))
        self.conv_w.copy_(torch.empty(self.conv_w.shape).uniform_(-0.5, 0.5, generator=generator))
        self.A_log.copy_(torch.empty(self.h_v).uniform_(1.0, 16.0, generator=generator).log())
        self.dt_bias.zero_()
        self.norm_w.copy_(torch.empty(self.d).normal_(0.0, 0.02, generator=generator))

    def forward(self, hidden_states, cu_seqlens, cu_host=None, initial_state=None,
                output_final_state=False):
        """hidden_states [T, D_h] (packed sequences, cu_seqlens int32 [N+1])
        -> (out [T, D_h], final_state [N, H_v, d_v, d_k] or None)."""
        T = hidden_states.shape[0]
        x = F.linear(hidden_states, self.W_qkv)
        z = F.linear(hidden_states, self.W_z).view(T, self.h_v, self.d)
        b = F.linear(hidden_states, self.W_b)
        a = F.linear(hidden_states, self.W_a)
        y, fs = gdn_core(x, self.conv_w, a, b, self.A_log, self.dt_bias, z, self.norm_w,
                         cu_seqlens, self.h_k, self.h_v, initial_state=initial_state,
                         output_final_state=output_final_state, cu_host=cu_host, gate=self.gate,
                         layout=self.layout)
        return F.linear(y.reshape(T, self.h_v * self.d), self.W_out), fs
