"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no arithmetic of the tensor-parallel method: it only draws
random tensors.  Every tensor is drawn from ``torch.Generator`` seeded with
``seed * 1000003 + stream`` on the device it is made on, as float32 normals
scaled by ``std``, then rounded once to bf16 (round-to-nearest-even, torch's
cast).  Activations use std 1 ("activations N(0,1) after RMSNorm with gain 1"),
weights std 0.02, following the Llama-shaped workloads the pages discuss
(Megatron MLP Y = GeLU(XA)B in "Tensor Parallelism (Megatron-Style)", with
Llama's second input matrix).

The GPU path and the oracle always receive the same tensor: large cases are
drawn on the device and copied to the host for the oracle, small cases are
drawn on the host.
"""
import torch

# stream ids: one per named tensor so that adding a tensor never shifts another
STREAM_X = 1
STREAM_RESIDUAL = 2
STREAM_W_GATE = 11
STREAM_W_UP = 12
STREAM_W_DOWN = 13
STREAM_W_QKV = 14
STREAM_W_O = 15


def normal_bf16(shape, std=1.0, seed=0, stream=0, device="cpu", layer=0):
    """bf16 tensor of N(0, std^2) samples, reproducible from (seed, stream, layer, device type)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(stream) + 7919 * int(layer))
    v = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(torch.bfloat16)


def small_int_bf16(shape, lo=-4, hi=4, seed=0, stream=0, device="cpu"):
    """bf16 tensor of integers in [lo, hi]; products and sums of these stay exact in fp32."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(stream) + 104729)
    v = torch.randint(lo, hi + 1, tuple(shape), generator=g, device=device, dtype=torch.int32)
    return v.to(torch.bfloat16)


def mlp_inputs(d, ffn, M, seed=0, device="cpu", layer=0, w_std=0.02):
    """x [M,d], residual (= x), W_gate [d,ffn], W_up [d,ffn], W_down [ffn,d]; all bf16, [in,out]."""
    x = normal_bf16((M, d), 1.0, seed, STREAM_X, device, layer)
    wg = normal_bf16((d, ffn), w_std, seed, STREAM_W_GATE, device, layer)
    wu = normal_bf16((d, ffn), w_std, seed, STREAM_W_UP, device, layer)
    wd = normal_bf16((ffn, d), w_std, seed, STREAM_W_DOWN, device, layer)
    return x, wg, wu, wd


def proj_inputs(d, n_q, n_kv, hd, M, seed=0, device="cpu", layer=0, w_std=0.02):
    """x [M,d], W_qkv [d,(n_q+2 n_kv) hd], W_o [n_q hd, d]; all bf16, [in,out]."""
    x = normal_bf16((M, d), 1.0, seed, STREAM_X, device, layer)
    wqkv = normal_bf16((d, (n_q + 2 * n_kv) * hd), w_std, seed, STREAM_W_QKV, device, layer)
    wo = normal_bf16((n_q * hd, d), w_std, seed, STREAM_W_O, device, layer)
    return x, wqkv, wo
