"""Seeded synthetic inputs for the CosmoFlow conv3d block.

This module is shared by the tests, the bench and the smoke check, and holds
none of the method's arithmetic: it only draws random numbers and rounds them
to the storage types the library consumes (bf16 bit patterns as uint16, fp32).

Recipe (the dark-matter histograms of the pages are not available here; these
inputs stand in for them with the same shapes and channel counts and a
positive, heavy-tailed distribution like log-scaled particle counts):

* generator: numpy ``Generator(PCG64)`` seeded from ``SeedSequence(seed)``;
  one child sequence per tensor, spawned in the order x, w1..wL, b1..bL, dY;
* activations of the CosmoFlow stack: x = log(1 + L), L ~ lognormal(0, 1);
* sweep activations: N(0, 1); the tiny single-block case: U[-1, 1];
* filters: He-normal, sigma = sqrt(2 / (27 * C_in)), mean 0, no truncation
  (the tiny case: sigma = 1/sqrt(27));
* biases: zero for the stack, N(0, 0.1^2) for the tiny case;
* upstream gradient at the top of the stack: N(0, 1);
* values are drawn in float64, rounded to float32 (round-to-nearest-even) and
  then to bf16 (round-to-nearest-even) where the consumer is bf16.
"""
from __future__ import annotations

import numpy as np

SLOPE = 0.3

STACK_CHANNELS = (4, 32, 64, 128, 256, 256)


def to_bf16_bits(a) -> np.ndarray:
    """float64/float32 array -> bf16 bit patterns (uint16), RNE via fp32."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(u16) -> np.ndarray:
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _children(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def he_normal(rng, c_out, c_in):
    sigma = np.sqrt(2.0 / (27.0 * c_in))
    return rng.normal(0.0, sigma, size=(c_out, 3, 3, 3, c_in))


def lognormal_volume(rng, n, c, d, h, w):
    return np.log1p(rng.lognormal(0.0, 1.0, size=(n, d, h, w, c)))


def stack_inputs(n: int, spatial: int = 128, channels=STACK_CHANNELS, seed: int = 20260003,
                 with_dy: bool = True):
    """The CosmoFlow-shaped stack: x [n,S,S,S,4] bf16, filters, zero biases, dY.

    Returns dict with uint16 bf16 bit arrays 'x', 'w' (list), float32 'b'
    (list) and, if asked, 'dy' at the last pooled output."""
    L = len(channels) - 1
    rngs = _children(seed, 1 + 2 * L + 1)
    x = to_bf16_bits(lognormal_volume(rngs[0], n, channels[0], spatial, spatial, spatial))
    ws = [to_bf16_bits(he_normal(rngs[1 + l], channels[l + 1], channels[l])) for l in range(L)]
    bs = [np.zeros(channels[l + 1], np.float32) for l in range(L)]
    for l in range(L):
        rngs[1 + L + l].normal(size=0)  # the bias streams exist but the biases are zero
    out = {"x": x, "w": ws, "b": bs}
    if with_dy:
        s = spatial >> L
        out["dy"] = to_bf16_bits(rngs[1 + 2 * L].normal(0.0, 1.0, size=(n, s, s, s, channels[-1])))
    return out


def tiny_block_inputs(seed: int = 20260001):
    """Single block, N=1, C_in=1, 16^3, C_out=8: x ~ U[-1,1], w ~ N(0, 1/27),
    b ~ N(0, 0.1^2).  x is drawn as fp32 and then rounded to bf16."""
    rngs = _children(seed, 4)
    x32 = rngs[0].uniform(-1.0, 1.0, size=(1, 16, 16, 16, 1)).astype(np.float32)
    w = rngs[1].normal(0.0, 1.0 / np.sqrt(27.0), size=(8, 3, 3, 3, 1))
    b = rngs[2].normal(0.0, 0.1, size=(8,)).astype(np.float32)
    return {"x32": x32, "x": to_bf16_bits(x32), "w": to_bf16_bits(w), "b": b}


def large_pair_inputs(seed: int = 20260004, spatial: int = 512):
    """Two blocks 4->32->64 on one 4 x 512^3 lognormal sample."""
    return stack_inputs(1, spatial, (4, 32, 64), seed=seed, with_dy=True)


SWEEP_SHAPES = (  # (C_in, C_out, spatial, N)
    (4, 32, 128, 8),
    (32, 64, 64, 16),
    (64, 128, 32, 32),
    (128, 256, 16, 64),
    (256, 256, 8, 128),
)


def sweep_inputs(c_in, c_out, spatial, n, seed: int = 20260005, scale_n: int | None = None):
    """Single-layer sweep shape: x, dZ ~ N(0,1) bf16, He-normal w."""
    rngs = _children(seed * 1000 + c_in * 7 + c_out, 3)
    nn = n if scale_n is None else scale_n
    x = to_bf16_bits(rngs[0].normal(0.0, 1.0, size=(nn, spatial, spatial, spatial, c_in)))
    w = to_bf16_bits(he_normal(rngs[1], c_out, c_in))
    dz = to_bf16_bits(rngs[2].normal(0.0, 1.0, size=(nn, spatial, spatial, spatial, c_out)))
    return {"x": x, "w": w, "dz": dz}


def random_case(seed, n, d, h, w, c_in, c_out, dist="normal"):
    """Small generic case for parity tests: x, w, b, dz, dy (pooled)."""
    rngs = _children(seed, 5)
    if dist == "lognormal":
        x = lognormal_volume(rngs[0], n, c_in, d, h, w)
    else:
        x = rngs[0].normal(0.0, 1.0, size=(n, d, h, w, c_in))
    wt = he_normal(rngs[1], c_out, c_in)
    b = rngs[2].normal(0.0, 0.1, size=(c_out,)).astype(np.float32)
    dz = rngs[3].normal(0.0, 1.0, size=(n, d, h, w, c_out))
    dy = rngs[4].normal(0.0, 1.0, size=(n, max(d // 2, 1), max(h // 2, 1), max(w // 2, 1), c_out))
    return {"x": to_bf16_bits(x), "w": to_bf16_bits(wt), "b": b,
            "dz": to_bf16_bits(dz), "dy": to_bf16_bits(dy)}
