"""Device-resident synthetic layers for the workloads in ``synth.SHAPES``.

Expert weights are filled on the GPU by the counter-based generator; router
weights, biases and activations are drawn on the host (numpy) and copied.
Input generation only."""
from __future__ import annotations

import numpy as np
import torch

import synth
from synth import device as sdev


class Layer:
    """One layer's inputs on a CUDA device (IQ4_NL weights as uint8 tensors)."""

    def __init__(self, shape: synth.Shape, seed: int, layer: int, device="cuda"):
        self.shape, self.seed, self.layer = shape, seed, layer
        H, F, E = shape.H, shape.F, shape.E
        nb = F * H // 32                      # blocks of one expert matrix
        def mat(n_exp, nblk, tensor):
            t = torch.empty(n_exp * nblk * 18, dtype=torch.uint8, device=device)
            sdev.fill_iq4nl(t, n_exp, nblk, seed, layer, tensor)
            return t
        self.gate = mat(E, nb, synth.GATE)
        self.up = mat(E, nb, synth.UP)
        self.down = mat(E, nb, synth.DOWN)
        if shape.n_shared:
            nbs = shape.Fs * H // 32
            self.sh_gate = mat(1, nbs, synth.SH_GATE)
            self.sh_up = mat(1, nbs, synth.SH_UP)
            self.sh_down = mat(1, nbs, synth.SH_DOWN)
        else:
            self.sh_gate = self.sh_up = self.sh_down = None
        Wr, b = synth.router(shape, seed, layer)
        self.router_w_host, self.bias_host = Wr, b
        self.router_w = torch.from_numpy(Wr.view(np.int16)).to(device).view(torch.bfloat16)
        self.bias = torch.from_numpy(b).to(device)

    def expert_bytes_host(self, e: int):
        return synth.expert_mats(self.shape, self.seed, self.layer, e)

    def shared_bytes_host(self):
        return synth.shared_mats(self.shape, self.seed, self.layer)


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
        torch.bfloat16)


def x_sets(shape: synth.Shape, seed: int, n_sets: int, T: int, device="cuda"):
    """Activations for every layer and input set: tensor bf16 [n_sets, L, T, H]."""
    out = np.empty((n_sets, shape.L, T, shape.H), np.uint16)
    for s in range(n_sets):
        for l in range(shape.L):
            out[s, l] = synth.x_rows(seed, l, shape.H, T, input_set=s)
    return bf16_tensor(out, device)
