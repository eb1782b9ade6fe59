"""Pre-norm layer stack (the pipeline-stage configuration: consecutive 405B-shaped layers'
linear parts + RMSNorm + residual, t=8) through tp_layer_forward.

Each layer is gated on its own: the oracle runs its own chain (float64 layers, activations
rounded to bf16 between layers, as they are stored), and the GPU layer L is given the
oracle chain's bf16 input to layer L.  The GPU chain's end-to-end drift from the oracle
chain is checked against a looser bar: rounding differences compound with depth."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import REL_F, bits, check_close

pytestmark = pytest.mark.gpu


def check_layer(y, y_ref, what):
    """Bar for a whole layer (two blocks composed).  The attention block's output h1 is rounded
    to bf16 and then passes through the MLP block, whose gain carries that error on: a layer
    gets the sum of two blocks' relF bars (1e-2).  Per element, y = h1 + MLP(b) holds up to two
    bf16 roundings of values the size of |y| on top of that: |err| <= 2^-7 |y_ref| + 2e-2 RMS."""
    yf, yr = O.as_f64(y), O.as_f64(y_ref)
    r = O.rel_frobenius(yf, yr)
    rms = np.sqrt(np.mean(yr * yr))
    excess = np.abs(yf - yr) - (2.0 ** -7 * np.abs(yr) + 2e-2 * rms)
    assert r <= 2 * REL_F and np.all(excess <= 0), f"{what}: relF {r:.3e}, worst excess {excess.max():.3e}"


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


class Layer:
    def __init__(self, d, ffn, n_q, n_kv, hd, t, L, dev, seed=0):
        self.sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
        _, self.wg, self.wu, self.wd = inputs.mlp_inputs(d, ffn, 1, seed=seed, device=dev, layer=L)
        _, self.wqkv, self.wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=seed, device=dev, layer=L)
        self.q_w, self.q = tpx.tp_partition_weights(self.sh, tpx.TP_W_QKV, self.wqkv)
        self.o_w, self.o = tpx.tp_partition_weights(self.sh, tpx.TP_W_O, self.wo)
        self.gu_w, self.gu = tpx.tp_partition_weights(self.sh, tpx.TP_W_GATE_UP, self.wg, self.wu)
        self.dn_w, self.dn = tpx.tp_partition_weights(self.sh, tpx.TP_W_DOWN, self.wd)
        self.heads = (n_q, n_kv, hd)

    def gpu(self, x, scratch, ws, flags=0):
        y = torch.full_like(x, float("nan"))
        tpx.tp_layer_forward(self.q, self.q_w, self.o, self.o_w, self.gu, self.gu_w, self.dn, self.dn_w,
                             x, y, scratch, ws, flags=flags)
        assert tpx.tp_sync(timeout_ms=30000) == tpx.TP_OK
        return y

    def oracle(self, xb):
        y, _ = O.layer(xb, bits(self.wqkv), bits(self.wo), bits(self.wg), bits(self.wu), bits(self.wd),
                       *self.heads)
        return y

    def check_blocks(self, xb, scratch_dev, ws, what):
        """Each block on its own, both fed from the oracle chain (its bf16 input x, and its
        attention output rounded to bf16 as stored), at the block bars (5e-3, 2e-2 RMS)."""
        dev = ws.device
        M, d = xb.shape
        to_dev = lambda b: torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(dev)
        n_q, n_kv, hd = self.heads
        x = to_dev(xb)
        a = torch.empty_like(x)
        tpx.tp_rmsnorm(x, a)
        y1 = torch.full_like(x, float("nan"))
        qkv = torch.empty((M, (n_q + 2 * n_kv) * hd), dtype=torch.bfloat16, device=dev)
        oi = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
        tpx.tp_proj_forward(self.q, self.q_w, self.o, self.o_w, a, x, y1, qkv, oi, ws)
        y1_ref, _ = O.proj(O.rmsnorm(xb), bits(self.wqkv), bits(self.wo), n_q, n_kv, hd, residual=xb)
        torch.cuda.synchronize()
        check_close(bits(y1), y1_ref, what=f"{what}: attention block")
        h1b = O.f64_to_bf16_bits(y1_ref)
        h1 = to_dev(h1b)
        b = torch.empty_like(h1)
        tpx.tp_rmsnorm(h1, b)
        y = torch.full_like(h1, float("nan"))
        h = torch.empty((M, self.wg.shape[1]), dtype=torch.bfloat16, device=dev)
        tpx.tp_mlp_forward(self.gu, self.gu_w, self.dn, self.dn_w, b, h1, y, h, ws)
        y_ref, _ = O.mlp(O.rmsnorm(h1b), bits(self.wg), bits(self.wu), bits(self.wd), residual=h1b)
        torch.cuda.synchronize()
        check_close(bits(y), y_ref, what=f"{what}: MLP block")


def test_layer_stack_per_layer_and_drift(dev):
    """Three layers with the 405B proportions scaled down (d 2048, ffn 6656 = 3.25 d,
    16 q / 8 kv heads of 128, t=8), M=16 decode tokens."""
    d, ffn, n_q, n_kv, hd, t, M, nl = 2048, 6656, 16, 8, 128, 8, 16, 3
    layers = [Layer(d, ffn, n_q, n_kv, hd, t, L, dev, seed=3) for L in range(nl)]
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(layers[0].sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(layers[0].sh, M, dev)
    x0 = inputs.normal_bf16((M, d), 1.0, 3, inputs.STREAM_X, dev)
    xo = bits(x0)                      # oracle chain (bf16 between layers)
    xg = x0                            # GPU chain
    for L, lay in enumerate(layers):
        lay.check_blocks(xo, scratch, ws, what=f"layer {L}")
        y_ref = lay.oracle(xo)
        y = lay.gpu(torch.from_numpy(xo.view(np.int16).copy()).view(torch.bfloat16).to(dev), scratch, ws)
        check_layer(bits(y), y_ref, what=f"layer {L} on the oracle chain's input")
        xg = lay.gpu(xg, scratch, ws)
        xo = O.f64_to_bf16_bits(y_ref)
    drift = O.rel_frobenius(bits(xg), O.as_f64(xo))
    assert drift <= 2e-2, f"end-to-end drift over {nl} layers: relF {drift:.3e}"


def test_405b_layer_full_size_sampled_tokens(dev):
    """One full 405B-shaped layer (d 16384, ffn 53248, 128 q / 8 kv heads, t=8) on two
    decode tokens, every output against the oracle."""
    lay = Layer(16384, 53248, 128, 8, 128, 8, 0, dev, seed=0)
    M = 2
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(lay.sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(lay.sh, M, dev)
    x = inputs.normal_bf16((M, 16384), 1.0, 0, inputs.STREAM_X, dev)
    lay.check_blocks(bits(x), scratch, ws, what="405B layer, 2 tokens")
    y = lay.gpu(x, scratch, ws)
    check_layer(bits(y), lay.oracle(bits(x)), what="405B layer, 2 tokens")


@pytest.mark.parametrize("M,wtype,fl", [(16, tpx.TP_BF16, 0), (5, tpx.TP_BF16, 0),
                                        (16, tpx.TP_FP8_E4M3, tpx.TP_F_KERNEL_TC),
                                        (16, tpx.TP_FP8_E4M3, tpx.TP_F_FP8_HILO),
                                        (40, tpx.TP_FP8_E4M3, tpx.TP_F_FP8_HILO)],
                         ids=["bf16-16", "bf16-5", "fp8-widened-16", "fp8-split-16", "fp8-split-40"])
def test_layer_norm_folded_into_blocks(dev, M, wtype, fl):
    """Decode layers run as two launches: the RMSNorms become per-token factors on the
    column-parallel accumulators (the attention block computes its input's factors, and its
    fold those of h1).  Against the oracle, against the path with separate RMSNorm launches
    (no bf16 rounding of the normalised input here, so the two differ by rounding only), and
    bit for bit from run to run."""
    # e4m3 weights stream in 128-wide k-blocks: the down projection's K per shard (ffn / t) must
    # be a multiple of 128 for the one-launch block
    d, ffn, n_q, n_kv, hd, t = 2048, 6656 if wtype == tpx.TP_BF16 else 7168, 16, 8, 128, 8
    lay = Layer(d, ffn, n_q, n_kv, hd, t, 0, dev, seed=4)
    if wtype != tpx.TP_BF16:
        lay.sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=wtype)
        lay.q_w, lay.q = tpx.tp_partition_weights(lay.sh, tpx.TP_W_QKV, lay.wqkv)
        lay.o_w, lay.o = tpx.tp_partition_weights(lay.sh, tpx.TP_W_O, lay.wo)
        lay.gu_w, lay.gu = tpx.tp_partition_weights(lay.sh, tpx.TP_W_GATE_UP, lay.wg, lay.wu)
        lay.dn_w, lay.dn = tpx.tp_partition_weights(lay.sh, tpx.TP_W_DOWN, lay.wd)
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(lay.sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(lay.sh, M, dev)
    x = inputs.normal_bf16((M, d), 1.0, 4, inputs.STREAM_X, dev)
    # e4m3 decode is fused only when asked (widened weights, or split activations)
    n0 = tpx.tp_launch_count()
    y = lay.gpu(x, scratch, ws, fl)
    assert tpx.tp_launch_count() - n0 == 2
    y_split = torch.full_like(x, float("nan"))
    tpx.tp_layer_forward(lay.q, lay.q_w, lay.o, lay.o_w, lay.gu, lay.gu_w, lay.dn, lay.dn_w, x, y_split,
                         scratch, ws, flags=tpx.TP_F_SPLIT_BLOCK)
    assert tpx.tp_sync(timeout_ms=30000) == tpx.TP_OK
    if wtype == tpx.TP_BF16:
        check_layer(bits(y), lay.oracle(bits(x)), what=f"folded-norm layer M={M}")
    else:
        deq = []
        for w in (lay.wqkv, lay.wo, lay.wg, lay.wu, lay.wd):
            q, s = O.quantize_fp8_per_channel(O.as_f64(bits(w)))
            deq.append(O.dequantize_fp8(q, s))
        y_ref, _ = O.layer(bits(x), *deq, n_q, n_kv, hd)
        check_layer(bits(y), y_ref, what=f"folded-norm fp8 layer M={M}")
    check_layer(bits(y), O.as_f64(bits(y_split)), what="folded vs separate norms")
    for _ in range(2):
        y2 = lay.gpu(x, scratch, ws, fl)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
