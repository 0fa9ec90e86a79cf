"""FLOP accounting for conv3d layers, in the convention of the CosmoFlow
pages: 2 FLOP per multiply-add, all 3x3x3 taps counted (also those that read
zero padding), one count each for forward, backward-data and backward-weight.

This reproduces the per-sample conv FLOP rows of Table I in "The Case for
Strong Scaling in Deep Learning: Training Large 3D CNNs with Hybrid
Parallelism" (section IV) for the 128^3, 256^3 and 512^3 models.
"""
from __future__ import annotations


def conv_flops(n: int, c_in: int, c_out: int, out_voxels: int) -> int:
    """One pass (fwd, dgrad or wgrad) of a k=3 conv producing out_voxels per sample."""
    return 2 * c_out * c_in * 27 * out_voxels * n


def stack_flops(n: int, spatial: int, channels, backward: bool, skip_first_dgrad: bool = True):
    """Executed FLOPs of the pooled stride-1 stack (each block halves the width).

    Forward counts one conv per block; backward adds wgrad for every block and
    dgrad for every block but the first (its input gradient has no consumer)
    unless skip_first_dgrad is False."""
    total = 0
    s = spatial
    for l in range(len(channels) - 1):
        f = conv_flops(n, channels[l], channels[l + 1], s ** 3)
        total += f
        if backward:
            total += f  # wgrad
            if l > 0 or not skip_first_dgrad:
                total += f  # dgrad
        s //= 2
    return total


def p3_table1_forward_flops(wi: int) -> float:
    """Forward conv FLOPs per sample of the seven-conv model of Table I for
    input width wi (c4 has stride 2; pooling after every conv while the width
    allows it: p6 exists for 256 and 512, p7 only for 512)."""
    ch = [4, 16, 32, 64, 128, 256, 256, 256]
    s, tot = wi, 0
    for l in range(7):
        if l == 3:
            s //= 2  # c4 is a stride-2 convolution
        tot += conv_flops(1, ch[l], ch[l + 1], s ** 3)
        pooled = not ((wi == 128 and l >= 5) or (wi == 256 and l == 6))
        if pooled:
            s //= 2
    return float(tot)


def p3_table1_params() -> int:
    """Parameters of the Table I model: conv filters without biases plus the
    three fully connected layers (2048 inputs after the last conv/pool)."""
    ch = [4, 16, 32, 64, 128, 256, 256, 256]
    conv = sum(ch[l] * ch[l + 1] * 27 for l in range(7))
    fc = 2048 * 2048 + 2048 * 256 + 256 * 4
    return conv + fc


def op_min_bytes(kind: str, n: int, spatial: int, c_in: int, c_out: int, routed: bool = False) -> int:
    """Minimum HBM bytes of one conv op of the pooled stack (every input read
    once, every output written once, bf16 activations, uint8 argmax codes,
    fp32 weight gradients), for the roofline of the op:
      fwd   : x, w, pooled y, codes, bias
      wgrad : x, dense dZ (or, routed, the pooled gradient and the codes), dW
      dgrad : dense dZ, w, the block input (leaky-ReLU derivative), dX
    """
    v = n * spatial ** 3
    p = v // 8
    w = c_out * 27 * c_in * 2
    if kind == "fwd":
        return v * c_in * 2 + w + p * c_out * 3 + c_out * 4
    if kind == "wgrad":
        dz = p * c_out * 3 if routed else v * c_out * 2
        return v * c_in * 2 + dz + c_out * 27 * c_in * 4
    if kind == "dgrad":
        return v * c_out * 2 + w + 2 * v * c_in * 2
    raise ValueError(kind)
