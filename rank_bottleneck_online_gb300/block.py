"""Workloads composed from the C-ABI calls: one block, the LLaMA MLP, the full
layer without its attention core, and the SVD-style pair.

Each workload owns its device tensors (weights, saved activations, gradients
and one workspace) so that a training step is a fixed sequence of library
calls on one stream with no allocation inside it. Every arithmetic step runs
in the library's CUDA kernels; Python only sequences the calls.
"""

from __future__ import annotations

import torch

from . import binding as B
from .inputs import CONFIGS


def _dev(t, device):
    return None if t is None else t.to(device=device, non_blocking=False).contiguous()


class Block:
    """One bottleneck block: y = B_i . act(s * x @ (gamma A))_i, forward and backward."""

    def __init__(self, T, d, r, k, n, *, S=1, eps=1e-5, act="silu", has_norm=True,
                 weights=None, device="cuda", ws=None):
        self.desc = B.make_desc(T, d, r, k, n, S=S, eps=eps, act=act, has_norm=has_norm)
        self.device = torch.device(device)
        w = weights or {}
        self.gamma = _dev(w.get("gamma"), self.device) if has_norm else None
        self.A = _dev(w.get("A"), self.device)
        self.B = _dev(w.get("B"), self.device)
        need = B.workspace_bytes(self.desc)
        self.ws = ws.ensure(need) if ws is not None else B.Workspace(need, self.device)
        bf = torch.bfloat16
        self.y = torch.empty(k, T, n, dtype=bf, device=self.device)
        self.rstd = torch.empty(T, dtype=torch.float32, device=self.device) if has_norm else None
        self.dx = torch.empty(T, d, dtype=bf, device=self.device)
        self.dA = torch.empty(d, k * r, dtype=bf, device=self.device)
        self.dB = torch.empty(k, r, n, dtype=bf, device=self.device)
        self.dgamma = torch.empty(d, dtype=bf, device=self.device) if has_norm else None

    def forward(self, x, stream=None, residual=None):
        """residual [T, n] (k == 1): y = residual + block(x), added in the epilogue."""
        return B.block_fwd(self.desc, x, self.gamma, self.A, self.B, self.ws, y=self.y,
                           rstd=self.rstd, stream=stream, residual=residual)

    def backward(self, x, dy, stream=None, reuse_rstd=True, dx=None, dx_residual=None):
        """dx: where the input gradient goes (default: this block's own buffer);
        dx_residual [T, d]: added to it in the dx epilogue."""
        return B.block_bwd(self.desc, x, self.gamma, self.A, self.B, dy, self.ws,
                           rstd=self.rstd if reuse_rstd else None,
                           dx=self.dx if dx is None else dx,
                           dgamma=self.dgamma, dA=self.dA, dB=self.dB, stream=stream,
                           dx_residual=dx_residual)


class MLP:
    """LLaMA MLP of two bottlenecks: gate/up (normed, k=2) -> SwiGLU -> down (k=1)."""

    def __init__(self, T, d, r, ffn, *, S=1, eps=1e-5, act="silu", weights=None,
                 device="cuda", ws=None, fused_glu=True, checkpoint="input"):
        w = weights or {}
        self.T, self.d, self.r, self.ffn = T, d, r, ffn
        # SwiGLU forward in the gate/up up-projection's epilogue, and its backward in the
        # down block's dgrad epilogue (False: separate SwiGLU passes)
        self.fused_glu = fused_glu
        # What the backward starts from. "input": each block's input (x, and h with the
        # gate/up values it was formed from) is kept from the forward, and each block
        # regenerates its own bottleneck activation. "bottleneck": only the gate/up
        # block's r-wide bottleneck activation is kept; the backward regenerates gate,
        # up and h from it (the cut at the tensor-parallel block boundary of §2.1).
        if checkpoint not in ("input", "bottleneck"):
            raise ValueError("checkpoint is 'input' or 'bottleneck'")
        if checkpoint == "bottleneck" and not fused_glu:
            raise ValueError("the bottleneck cut regenerates gate, up and h with the fused kernel")
        self.checkpoint = checkpoint
        self.gu = Block(T, d, r, 2, ffn, S=S, eps=eps, act=act, has_norm=True,
                        weights={"gamma": w.get("gamma"), "A": w.get("A1"), "B": w.get("B1")},
                        device=device, ws=ws)
        self.dn = Block(T, ffn, r, 1, d, S=1, eps=eps, act=act, has_norm=False,
                        weights={"A": w.get("A2"), "B": w.get("B2")}, device=device,
                        ws=self.gu.ws if checkpoint == "input" else None)
        if checkpoint == "input":
            self.gu.ws = self.dn.ws   # one workspace sized for both blocks
        # (bottleneck cut: the gate/up block keeps its own workspace, whose a survives
        # the down block's forward)
        dev = self.gu.device
        self.h = torch.empty(T, ffn, dtype=torch.bfloat16, device=dev)
        self.dy1 = torch.empty(2, T, ffn, dtype=torch.bfloat16, device=dev)

    @property
    def out(self):
        return self.dn.y[0]

    def forward(self, x, stream=None, residual=None):
        """residual [T, d]: out = residual + MLP(x), added in the down block's epilogue."""
        if self.fused_glu:
            gu = self.gu
            B.block_fwd_swiglu(gu.desc, x, gu.gamma, gu.A, gu.B, gu.ws, y=gu.y, h=self.h,
                               rstd=gu.rstd, stream=stream)
        else:
            y1 = self.gu.forward(x, stream)
            B.swiglu_fwd(y1[0], y1[1], self.h, stream=stream)
        return self.dn.forward(self.h, stream, residual=residual)[0]

    def saved_bytes(self):
        """Bytes of activations the backward needs from the forward beyond the input x
        and the row scale: gate, up and h for the input cut, the gate/up block's
        bottleneck activation for the bottleneck cut."""
        if self.checkpoint == "input":
            return 3 * self.T * self.ffn * 2
        return self.T * 2 * self.r * 2

    def backward(self, x, dout, stream=None, dx_residual=None):
        """dx_residual [T, d]: added to the MLP's input gradient in the dx epilogue."""
        dy2 = dout.view(1, self.T, self.d)
        if self.checkpoint == "bottleneck":
            gu = self.gu
            a1 = B.ws_view(gu.ws, B.ws_layout(gu.desc)["a"], (self.T, 2 * self.r),
                           torch.bfloat16)
            B.block_up(gu.desc, a1, gu.B, gu.ws, y=gu.y, h=self.h, stream=stream)
        if self.fused_glu:
            B.block_bwd_swiglu(self.dn.desc, self.h, self.dn.A, self.dn.B, dy2, self.gu.y[0],
                               self.gu.y[1], self.dn.ws, dgate=self.dy1[0], dup=self.dy1[1],
                               dA=self.dn.dA, dB=self.dn.dB, stream=stream)
        else:
            dh = self.dn.backward(self.h, dy2, stream)[0]
            B.swiglu_bwd(self.gu.y[0], self.gu.y[1], dh, self.dy1[0], self.dy1[1],
                         stream=stream)
        return self.gu.backward(x, self.dy1, stream, dx_residual=dx_residual)

    def grads(self):
        return {"dx": self.gu.dx, "dgamma": self.gu.dgamma, "dA1": self.gu.dA, "dB1": self.gu.dB,
                "dA2": self.dn.dA, "dB2": self.dn.dB}


class Layer:
    """QKV (normed, k=3) -> O (k=1) on V -> residual -> MLP -> residual.

    Both residual adds run in GEMM epilogues: x1 = x + O(v) in the O block's
    up-projection, out = x1 + MLP(x1) in the MLP's down up-projection; in the backward,
    dx1 = dout + (MLP input gradient) in the MLP's dx epilogue and dx = dx1 + (QKV input
    gradient) in the QKV block's."""

    def __init__(self, T, d, r, ffn, *, S=1, eps=1e-5, act="silu", weights=None, device="cuda"):
        p = weights or {}
        self.T, self.d = T, d
        self.qkv = Block(T, d, r, 3, d, S=S, eps=eps, act=act, has_norm=True,
                         weights={"gamma": p.get("gamma1"), "A": p.get("A_qkv"),
                                  "B": p.get("B_qkv")}, device=device)
        ws = self.qkv.ws
        self.o = Block(T, d, r, 1, d, S=1, eps=eps, act=act, has_norm=False,
                       weights={"A": p.get("A_o"), "B": p.get("B_o")}, device=device, ws=ws)
        self.mlp = MLP(T, d, r, ffn, S=S, eps=eps, act=act,
                       weights={"gamma": p.get("gamma2"), "A1": p.get("A_gu"), "B1": p.get("B_gu"),
                                "A2": p.get("A_dn"), "B2": p.get("B_dn")}, device=device, ws=ws)
        ws = self.mlp.gu.ws
        for blk in (self.qkv, self.o):
            blk.ws = ws
        dev = self.qkv.device
        self.dqkv = torch.empty(3, T, d, dtype=torch.bfloat16, device=dev)

    @property
    def x1(self):
        """x + O(v): the MLP's input (the O block's output buffer)."""
        return self.o.y[0]

    @property
    def out(self):
        """x1 + MLP(x1) (the MLP's output buffer)."""
        return self.mlp.out

    @property
    def dx1(self):
        """Gradient at x1: dout + the MLP's input gradient (the MLP's dx buffer)."""
        return self.mlp.gu.dx

    @property
    def dx(self):
        """Gradient at x: dx1 + the QKV block's input gradient (its dx buffer)."""
        return self.qkv.dx

    def forward(self, x, stream=None):
        qkv = self.qkv.forward(x, stream)
        x1 = self.o.forward(qkv[2], stream, residual=x)[0]
        return self.mlp.forward(x1, stream, residual=x1)

    def backward(self, x, dout, dq, dk, stream=None):
        """dq, dk: the attention core's gradients of q and k. The QKV block's upstream
        gradient is the stacked [dq, dk, dv]; dq and dk are copied into it unless they
        are already its first two planes (`dqkv[0]`, `dqkv[1]`), and the O block writes
        dv straight into the third."""
        dx1 = self.mlp.backward(self.x1, dout, stream, dx_residual=dout)[0]
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            for i, g in enumerate((dq, dk)):
                if g.data_ptr() != self.dqkv[i].data_ptr():
                    self.dqkv[i].copy_(g)
        self.o.backward(self.qkv.y[2], dx1.view(1, self.T, self.d), stream, dx=self.dqkv[2])
        return self.qkv.backward(x, self.dqkv, stream, dx_residual=dx1)[0]


class SVDPair:
    """Two normed SVD-style bottlenecks (identity act) on one x: QKV and gate/up. The
    input gradient is the sum of the two blocks', added in the gate/up block's dx
    epilogue."""

    def __init__(self, T, d, r, ffn, *, S=1, eps=1e-5, weights=None, device="cuda"):
        p = weights or {}
        self.qkv = Block(T, d, r, 3, d, S=S, eps=eps, act="identity", has_norm=True,
                         weights={"gamma": p.get("gamma_qkv"), "A": p.get("A_qkv"),
                                  "B": p.get("B_qkv")}, device=device)
        self.gu = Block(T, d, r, 2, ffn, S=S, eps=eps, act="identity", has_norm=True,
                        weights={"gamma": p.get("gamma_gu"), "A": p.get("A_gu"),
                                 "B": p.get("B_gu")}, device=device, ws=self.qkv.ws)
        self.qkv.ws = self.gu.ws

    @property
    def dx(self):
        """Gradient at x: the QKV block's plus the gate/up block's (the latter's dx buffer)."""
        return self.gu.dx

    def forward(self, x, stream=None):
        return self.qkv.forward(x, stream), self.gu.forward(x, stream)

    def backward(self, x, dy_qkv, dy_gu, stream=None):
        dxq = self.qkv.backward(x, dy_qkv, stream)[0]
        return self.gu.backward(x, dy_gu, stream, dx_residual=dxq)[0]


def build_workload(name, tensors, device="cuda", T=None):
    """Instantiate a named workload with its (CPU) input tensors moved to ``device``."""
    c = dict(CONFIGS[name])
    if T is not None:
        c["T"] = T
    eps = 1e-5
    if c["kind"] == "block":
        return Block(c["T"], c["d"], c["r"], c["k"], c["n"], S=c["S"], eps=eps, act=c["act"],
                     weights=tensors, device=device)
    if c["kind"] == "mlp":
        return MLP(c["T"], c["d"], c["r"], c["ffn"], S=c["S"], eps=eps, act=c["act"],
                   weights=tensors, device=device)
    if c["kind"] == "layer":
        return Layer(c["T"], c["d"], c["r"], c["ffn"], S=c["S"], eps=eps, act=c["act"],
                     weights=tensors["p"], device=device)
    if c["kind"] == "svd_pair":
        return SVDPair(c["T"], c["d"], c["r"], c["ffn"], S=c["S"], eps=eps,
                       weights=tensors["p"], device=device)
    raise KeyError(name)
