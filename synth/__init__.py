"""Seeded synthetic inputs for the IQ4_NL MoE layer (host side, numpy).

This module only draws random numbers and packs them into the input formats;
it holds none of the layer's arithmetic. The oracle and the CUDA library both
take their inputs from here. The large expert tensors can also be filled on
the GPU by ``synth/synth_gen.cu``, which implements the same generator from
the same definition; a test checks that the two agree byte for byte.

Generator (counter-based):
  splitmix64(z): z += 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
                 z = (z ^ z>>27) * 0x94D049BB133111EB; return z ^ z>>31
  key(seed, layer, tensor, sub) = sm(sm(sm(sm(seed) ^ layer) ^ tensor) ^ sub)
  draw i of a stream = splitmix64(key + i)
  uniform U = (draw >> 11) * 2^-53
  normal element i: Box-Muller on draws 2i (u1 = 1 - U) and 2i+1 (u2 = U)
  bf16 = round-to-nearest-even of the float32 value (itself RNE of the double)
  IQ4_NL block b: draws 3b, 3b+1, 3b+2; d = fp16(1e-4 + 3e-4 * U(draw 3b)) by
  RNE; the 16 index bytes are draws 3b+1 and 3b+2, little-endian.

Workload shapes are those of the pages' models (hidden, expert_ffn, experts,
top-k): Xing4.0-29B-A4B (PocketLLM page, Overview table), Qwen3-Next-80B-A3B
(Red Lite "What we learned", section 1) and a 384-expert top-6 DeepSeek-like
layer (Xolotl blog, "Why build an engine at all").
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids of the generator's key
GATE, UP, DOWN, SH_GATE, SH_UP, SH_DOWN, ROUTER, BIAS, X, ZIPF = range(10)

BLOCK_BYTES = 18
BLOCK_WEIGHTS = 32


def splitmix64(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def key(seed: int, layer: int, tensor: int, sub: int) -> np.uint64:
    k = splitmix64(np.array([seed], np.uint64))
    k = splitmix64(k ^ np.uint64(layer))
    k = splitmix64(k ^ np.uint64(tensor))
    k = splitmix64(k ^ np.uint64(sub))
    return k[0]


def draws(k: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return splitmix64(idx + np.uint64(k))


def uniform(bits: np.ndarray) -> np.ndarray:
    return (bits >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(k: np.uint64, n: int) -> np.ndarray:
    d = draws(k, 0, 2 * n)
    u1 = 1.0 - uniform(d[0::2])
    u2 = uniform(d[1::2])
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    f = np.asarray(v, np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return (b >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def iq4nl_blocks(seed: int, layer: int, tensor: int, expert: int, n_blocks: int,
                 start_block: int = 0) -> np.ndarray:
    """n_blocks IQ4_NL blocks of one expert's matrix, as uint8 [n_blocks, 18]."""
    k = key(seed, layer, tensor, expert)
    d = draws(k, 3 * start_block, 3 * n_blocks).reshape(n_blocks, 3)
    s = 1e-4 + 3e-4 * uniform(d[:, 0])
    scale = s.astype(np.float16).view(np.uint16)
    out = np.empty((n_blocks, BLOCK_BYTES), np.uint8)
    out[:, 0:2] = scale.reshape(-1, 1).view(np.uint8).reshape(n_blocks, 2)
    out[:, 2:10] = d[:, 1].astype("<u8").view(np.uint8).reshape(n_blocks, 8)
    out[:, 10:18] = d[:, 2].astype("<u8").view(np.uint8).reshape(n_blocks, 8)
    return out


class Shape:
    """Sizes of one MoE layer and its workload."""

    def __init__(self, name, H, F, E, k, T, L, Fs=None, n_shared=1, router_std=0.05,
                 bias_std=0.01, zipf=None):
        self.name, self.H, self.F, self.E, self.k, self.T, self.L = name, H, F, E, k, T, L
        self.Fs = F if Fs is None else Fs
        self.n_shared = n_shared
        self.router_std, self.bias_std, self.zipf = router_std, bias_std, zipf

    def expert_bytes(self, F=None) -> int:
        F = self.F if F is None else F
        return 3 * self.H * F * BLOCK_BYTES // BLOCK_WEIGHTS

    def mat_blocks(self, which: int, F=None) -> int:
        """Blocks in one expert's gate/up ([F][H/32]) or down ([H][F/32]) matrix."""
        F = self.F if F is None else F
        return F * self.H // 32


# The workloads (hidden, expert_ffn, experts, top-k, tokens, layers).
SHAPES = {
    0: Shape("tiny: hidden 256, 8 experts top-2 + shared, ffn 128, 4 tokens",
             256, 128, 8, 2, 4, 1),
    1: Shape("xing4-29b-a4b decode: hidden 3584, 64 experts top-4 + shared, ffn 1024, "
             "1 token, 38 layers", 3584, 1024, 64, 4, 1, 38),
    2: Shape("qwen3-next-80b-a3b paired decode: hidden 2048, 512 experts top-10 + shared, "
             "ffn 512, 2 tokens, 48 layers", 2048, 512, 512, 10, 2, 48),
    3: Shape("deepseek-like wide decode: hidden 4096, 384 experts top-6 + shared, ffn 2048, "
             "1/4/16 tokens, 4 layers", 4096, 2048, 384, 6, 16, 4, router_std=1.0 / 64.0),
    4: Shape("xing4-29b-a4b prefill chunk: hidden 3584, 64 experts top-4 + shared, ffn 1024, "
             "2048 tokens, 4 layers, zipf(1.1) expert bias", 3584, 1024, 64, 4, 2048, 4,
             zipf=1.1),
}


def seed_of(cfg: int) -> int:
    return 1234 + cfg


def router(shape: Shape, seed: int, layer: int):
    """Router weights (bf16 bits [E, H]) and selection bias (float32 [E])."""
    E, H = shape.E, shape.H
    w = to_bf16_bits(shape.router_std * normal(key(seed, layer, ROUTER, 0), E * H))
    b = (shape.bias_std * normal(key(seed, layer, BIAS, 0), E)).astype(np.float32)
    if shape.zipf is not None:
        # a seeded permutation gives each expert a rank r in 1..E; bias += r^-s
        u = uniform(draws(key(seed, layer, ZIPF, 0), 0, E))
        rank = np.empty(E, np.int64)
        rank[np.argsort(u, kind="stable")] = np.arange(1, E + 1)
        b = (b.astype(np.float64) + rank.astype(np.float64) ** (-shape.zipf)).astype(np.float32)
    return w.reshape(E, H), b


def x_rows(seed: int, layer: int, H: int, T: int, input_set: int = 0,
           resample=None) -> np.ndarray:
    """Activations bf16 bits [T, H] ~ N(0,1). Token t's row is drawn from
    sub-key (input_set << 32) | (t << 10) | resample[t]."""
    out = np.empty((T, H), np.uint16)
    for t in range(T):
        r = 0 if resample is None else int(resample[t])
        sub = (int(input_set) << 32) | (t << 10) | r
        out[t] = to_bf16_bits(normal(key(seed, layer, X, sub), H))
    return out


def x_row(seed: int, layer: int, H: int, t: int, input_set: int, r: int) -> np.ndarray:
    sub = (int(input_set) << 32) | (t << 10) | int(r)
    return to_bf16_bits(normal(key(seed, layer, X, sub), H))


def expert_mats(shape: Shape, seed: int, layer: int, e: int):
    """(gate, up, down) blocks of routed expert e, uint8 [n_blocks, 18] each."""
    nb = shape.F * shape.H // 32
    return (iq4nl_blocks(seed, layer, GATE, e, nb), iq4nl_blocks(seed, layer, UP, e, nb),
            iq4nl_blocks(seed, layer, DOWN, e, nb))


def shared_mats(shape: Shape, seed: int, layer: int):
    nb = shape.Fs * shape.H // 32
    return (iq4nl_blocks(seed, layer, SH_GATE, 0, nb), iq4nl_blocks(seed, layer, SH_UP, 0, nb),
            iq4nl_blocks(seed, layer, SH_DOWN, 0, nb))
