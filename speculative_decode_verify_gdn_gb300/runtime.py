"""Device-resident buffers of one GDN layer and the verify -> rollback round.

Torch allocates the memory; every step of the round runs through the C ABI
(gdn_verify_step, then gdn_rollback).  Two layouts of the carried state:

* in place (default): the verify step overwrites the state and the conv
  history; accept lengths must be >= 1 (the pre-window state is gone).
* ping-pong (``keep_snapshot=True``): the verify step reads buffer ``cur`` and
  writes buffer ``1 - cur``; the rollback restores into ``1 - cur`` using
  ``cur`` as the pre-window snapshot, so an accept length of 0 is allowed and
  no copy is made to keep the snapshot.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import gdn
from .synth import Dims, Layer, Round


def _bf16(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def _f32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


@dataclass
class GdnLayerState:
    dims: gdn.GdnDims
    conv_w: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    conv_states: list          # one or two [B, W-1, C] f32 buffers
    states: list               # one or two [B, Hv, dv, dk] f32 buffers
    conv_inter: torch.Tensor   # [B, K, W-1, C]
    state_inter: torch.Tensor  # [B, K-1, Hv, dv, dk] (None when K == 1)
    x: torch.Tensor            # [B, K, C] bf16
    a: torch.Tensor            # [B, K, Hv] bf16
    b: torch.Tensor
    out: torch.Tensor          # [B, K, Hv, dv]
    accept_len: torch.Tensor   # [B] int32
    workspace: torch.Tensor    # scratch of gdn_verify_step
    cur: int = 0

    @property
    def keep_snapshot(self) -> bool:
        return len(self.states) == 2

    @property
    def state(self) -> torch.Tensor:
        return self.states[self.cur]

    @property
    def conv_state(self) -> torch.Tensor:
        return self.conv_states[self.cur]

    @classmethod
    def create(cls, d: Dims, layer: Layer, device="cuda", keep_snapshot=False, out_f32=True,
               q_scale=1.0, l2_eps=1e-6) -> "GdnLayerState":
        dims = gdn.make_dims(d.B, d.K, d.Hk, d.Hv, d.dk, d.dv, d.W, q_scale, l2_eps, int(out_f32))
        n = 2 if keep_snapshot else 1
        st = [_f32(layer.state, device) for _ in range(n)]
        cs = [_f32(layer.conv_state, device) for _ in range(n)]
        C = d.C
        return cls(
            dims=dims, conv_w=_f32(layer.conv_w, device), A_log=_f32(layer.A_log, device),
            dt_bias=_f32(layer.dt_bias, device), conv_states=cs, states=st,
            conv_inter=torch.empty((d.B, d.K, d.W - 1, C), dtype=torch.float32, device=device),
            state_inter=(torch.empty((d.B, d.K - 1, d.Hv, d.dv, d.dk), dtype=torch.float32, device=device)
                         if d.K > 1 else None),
            x=torch.empty((d.B, d.K, C), dtype=torch.bfloat16, device=device),
            a=torch.empty((d.B, d.K, d.Hv), dtype=torch.bfloat16, device=device),
            b=torch.empty((d.B, d.K, d.Hv), dtype=torch.bfloat16, device=device),
            out=torch.empty((d.B, d.K, d.Hv, d.dv), dtype=torch.float32 if out_f32 else torch.bfloat16,
                            device=device),
            accept_len=torch.full((d.B,), d.K, dtype=torch.int32, device=device),
            workspace=gdn.alloc_workspace(dims, device),
        )

    def load_round(self, rnd: Round) -> None:
        dev = self.x.device
        self.x.copy_(_bf16(rnd.x, dev))
        self.a.copy_(_bf16(rnd.a, dev))
        self.b.copy_(_bf16(rnd.b, dev))
        self.accept_len.copy_(torch.from_numpy(np.ascontiguousarray(rnd.accept_len, dtype=np.int32)).to(dev))

    def verify(self, stream=None) -> None:
        i, o = (self.cur, 1 - self.cur) if self.keep_snapshot else (0, 0)
        gdn.gdn_verify_step(self.dims, self.x, self.a, self.b, self.A_log, self.dt_bias, self.conv_w,
                            self.conv_states[i], self.conv_states[o], self.conv_inter, self.states[i],
                            self.states[o], self.state_inter, self.out, self.workspace, stream)

    def verify_tree(self, parent, stream=None) -> None:
        """Verify the loaded window as a token tree (parent [B, K] int32 on the device)."""
        i, o = (self.cur, 1 - self.cur) if self.keep_snapshot else (0, 0)
        gdn.gdn_verify_tree(self.dims, parent, self.x, self.a, self.b, self.A_log, self.dt_bias, self.conv_w,
                            self.conv_states[i], self.conv_states[o], self.conv_inter, self.states[i],
                            self.states[o], self.state_inter, self.out, self.workspace, stream)

    def verify_gated(self, z, norm_w, norm_eps=1e-6, stream=None) -> None:
        """Verify the loaded window with the gated RMS norm fused into the output
        (z [B, K, Hv, dv] bf16 and norm_w [dv] f32 on the device)."""
        i, o = (self.cur, 1 - self.cur) if self.keep_snapshot else (0, 0)
        gdn.gdn_verify_gated(self.dims, self.x, self.a, self.b, self.A_log, self.dt_bias, self.conv_w,
                             self.conv_states[i], self.conv_states[o], self.conv_inter, self.states[i],
                             self.states[o], self.state_inter, z, norm_w, norm_eps, self.out, self.workspace,
                             stream)

    def rollback(self, stream=None) -> None:
        if self.keep_snapshot:
            i, o = self.cur, 1 - self.cur
            gdn.gdn_rollback(self.dims, self.accept_len, self.states[i], self.states[o], self.state_inter,
                             self.conv_states[i], self.conv_states[o], self.conv_inter, stream)
            self.cur = o
        else:
            gdn.gdn_rollback(self.dims, self.accept_len, None, self.states[0], self.state_inter, None,
                             self.conv_states[0], self.conv_inter, stream)

    def step(self, stream=None) -> None:
        """One verify + rollback round on the loaded window and accept lengths."""
        self.verify(stream)
        self.rollback(stream)

    def verify_resume(self, accept_prev, stream=None) -> None:
        """Verify the loaded window after applying the previous window's accept lengths on read
        (gdn_verify_resume, in place, no snapshot: lengths must be >= 1).  The state buffers then
        hold this window's final state and intermediates, as after `verify`."""
        if self.keep_snapshot:
            raise ValueError("verify_resume works in place; create the state without keep_snapshot")
        S, CS = self.states[0], self.conv_states[0]
        gdn.gdn_verify_resume(self.dims, accept_prev, self.x, self.a, self.b, self.A_log, self.dt_bias, self.conv_w,
                              CS, self.conv_inter, None, CS, self.conv_inter, S, self.state_inter, None, S,
                              self.state_inter, self.out, self.workspace, stream)
