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
from tests.test_gpu_parity import REL_F, bits, check_close, check_h

pytestmark = pytest.mark.gpu


def check_layer(y, y_ref, h1_ref, what):
    """A whole layer against the oracle layer whose attention output h1 is rounded to bf16 as
    the GPU stores it (both start from the same bf16 input): relF <= 5e-3, the block bar.  Per
    element the layer composes two blocks: y = h1 + MLP(norm(h1)) carries the attention block's
    own error in h1 (its bf16 roundings of qkv, o_in and h1, within 2e-2 RMS(h1) per element)
    through the residual, on top of the MLP block's (within 2e-2 RMS(y)).  So the whole layer is
    held to the sum of the two block bars, |err| <= 2e-2 (RMS(y_ref) + RMS(h1_ref)); each block
    is held to its own 2e-2 RMS on its own input in Layer.check_outputs."""
    yf, yr, hr = O.as_f64(y), O.as_f64(y_ref), O.as_f64(h1_ref)
    r = O.rel_frobenius(yf, yr)
    bar = 2e-2 * (np.sqrt(np.mean(yr * yr)) + np.sqrt(np.mean(hr * hr)))
    worst = np.abs(yf - yr).max()
    assert r <= REL_F and worst <= bar, f"{what}: relF {r:.3e} (bar {REL_F}), max |err| {worst:.3e} (bar {bar:.3e})"


def _align(n):
    return (n + 255) // 256 * 256


def layer_scratch(scratch, M, d, Q, ffn):
    """The activations tp_layer_forward leaves in its scratch, at the offsets its declaration
    gives: h1 [M, d], the attention output o_in [M, d], qkv [M, Q] (shard-major) and h [M, ffn]."""
    b = _align(M * d * 2)
    view = lambda off, n, shape: scratch[off:off + n * 2].view(torch.bfloat16).view(shape)
    h1 = view(b, M * d, (M, d))
    oi = view(2 * b, M * d, (M, d))
    qk = view(4 * b, M * Q, (M, Q))
    h = view(4 * b + _align(M * Q * 2), M * ffn, (M, ffn))
    return h1, oi, qk, h


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

    def weights(self):
        return [bits(w) for w in (self.wqkv, self.wo, self.wg, self.wu, self.wd)]

    def oracle(self, xb, weights=None):
        """(y, h1) of the oracle layer, h1 rounded to bf16 between the blocks."""
        return O.layer(xb, *(weights or self.weights()), *self.heads, bf16_between_blocks=True)

    def check_outputs(self, xb, y, scratch, what, weights=None, rows=None):
        """Every output of one folded-norm layer: qkv and h1 against the oracle attention block
        on the layer's input; h and y against the oracle MLP block on the GPU's own h1 (teacher
        forcing at the block boundary); y against the whole oracle layer.  rows: check only
        these token rows (each output row depends on its own input row alone)."""
        wqkv, wo, wg, wu, wd = weights or self.weights()
        n_q, n_kv, hd = self.heads
        M, d = xb.shape
        Q, ffn, t = (n_q + 2 * n_kv) * hd, wg.shape[1], self.sh.t
        sel = slice(None) if rows is None else rows
        h1, oi, qk, h = (bits(v)[sel] for v in layer_scratch(scratch, M, d, Q, ffn))
        xb, yb = xb[sel], bits(y)[sel]
        h1_ref, qkv_ref = O.proj(O.rmsnorm(xb), wqkv, wo, n_q, n_kv, hd, residual=xb)
        cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
        check_close(O.as_f64(qk), qkv_ref[:, cols], what=f"{what}: qkv")
        check_close(O.as_f64(h1), h1_ref, what=f"{what}: h1 (attention block)")
        y_tf, h_ref = O.mlp(O.rmsnorm(h1), wg, wu, wd, residual=h1)
        check_h(h, h_ref, what=f"{what}: h")
        check_close(O.as_f64(yb), y_tf, what=f"{what}: y (MLP block on the layer's own h1)")
        check_layer(yb, *self.oracle(xb, weights), what=f"{what}: y (whole layer)")

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
        y_ref, _ = lay.oracle(xo)
        y = lay.gpu(torch.from_numpy(xo.view(np.int16).copy()).view(torch.bfloat16).to(dev), scratch, ws)
        lay.check_outputs(xo, y, scratch, what=f"layer {L} on the oracle chain's input")
        xg = lay.gpu(xg, scratch, ws)
        xo = O.f64_to_bf16_bits(y_ref)
    drift = O.rel_frobenius(bits(xg), O.as_f64(xo))
    assert drift <= 2e-2, f"end-to-end drift over {nl} layers: relF {drift:.3e}"


def test_405b_layer_full_size_decode_batch(dev):
    """One full 405B-shaped layer (d 16384, ffn 53248, 128 q / 8 kv heads, t=8) at the
    pipeline-stage stack's decode batch, M=16, through the default tp_layer_forward (the two
    folded-norm launches the stack runs): every output against the oracle, then each block on
    its own through the split path."""
    lay = Layer(16384, 53248, 128, 8, 128, 8, 0, dev, seed=0)
    M = 16
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(lay.sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(lay.sh, M, dev)
    x = inputs.normal_bf16((M, 16384), 1.0, 0, inputs.STREAM_X, dev)
    n0 = tpx.tp_launch_count()
    y = lay.gpu(x, scratch, ws)
    assert tpx.tp_launch_count() - n0 == 2
    w = lay.weights()
    lay.check_outputs(bits(x), y, scratch, what="405B layer, 16 tokens", weights=w)
    lay.check_blocks(bits(x), scratch, ws, what="405B layer, 16 tokens")


@pytest.mark.parametrize("M,wtype,fl", [(16, tpx.TP_BF16, 0), (5, tpx.TP_BF16, 0),
                                        (16, tpx.TP_FP8_E4M3, tpx.TP_F_KERNEL_TC),
                                        (16, tpx.TP_FP8_E4M3, tpx.TP_F_FP8_HILO),
                                        (40, tpx.TP_FP8_E4M3, tpx.TP_F_FP8_HILO),
                                        (40, tpx.TP_FP8_E4M3, 0)],
                         ids=["bf16-16", "bf16-5", "fp8-widened-16", "fp8-split-16", "fp8-split-40",
                              "fp8-default-40"])
def test_layer_norm_folded_into_blocks(dev, M, wtype, fl):
    """Decode layers run as two launches: the RMSNorms become per-token factors on the
    column-parallel accumulators (the attention block computes its input's factors, and its
    fold those of h1).  Every output against the oracle (e4m3 weights: on the dequantised
    weights), the path with separate RMSNorm launches as well, and bit for bit from run to run."""
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
    # two block launches; with split activations each block is preceded by the small kernel (the
    # default e4m3 block widens the weights above 32 tokens: no small kernel at M = 40)
    # that takes its input's per-token maxima
    n0 = tpx.tp_launch_count()
    y = lay.gpu(x, scratch, ws, fl)
    assert tpx.tp_launch_count() - n0 == (4 if fl == tpx.TP_F_FP8_HILO else 2)
    y_split = torch.full_like(x, float("nan"))
    tpx.tp_layer_forward(lay.q, lay.q_w, lay.o, lay.o_w, lay.gu, lay.gu_w, lay.dn, lay.dn_w, x, y_split,
                         scratch, ws, flags=tpx.TP_F_SPLIT_BLOCK)
    assert tpx.tp_sync(timeout_ms=30000) == tpx.TP_OK
    if wtype == tpx.TP_BF16:
        w = lay.weights()
    else:
        w = []
        for m in (lay.wqkv, lay.wo, lay.wg, lay.wu, lay.wd):
            q, sc = O.quantize_fp8_per_channel(O.as_f64(bits(m)))
            w.append(O.dequantize_fp8(q, sc))
    y_split_ref, h1_ref = O.layer(bits(x), *w, n_q, n_kv, hd, bf16_between_blocks=True)
    check_layer(bits(y_split), y_split_ref, h1_ref, what=f"separate-norm layer M={M}")
    y = lay.gpu(x, scratch, ws, fl)         # the scratch again holds the folded path's activations
    lay.check_outputs(bits(x), y, scratch, what=f"folded-norm layer M={M}", weights=w)
    for _ in range(2):
        y2 = lay.gpu(x, scratch, ws, fl)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def _fp8_layer(lay, d, ffn, n_q, n_kv, hd, t):
    lay.sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=tpx.TP_FP8_E4M3)
    lay.q_w, lay.q = tpx.tp_partition_weights(lay.sh, tpx.TP_W_QKV, lay.wqkv)
    lay.o_w, lay.o = tpx.tp_partition_weights(lay.sh, tpx.TP_W_O, lay.wo)
    lay.gu_w, lay.gu = tpx.tp_partition_weights(lay.sh, tpx.TP_W_GATE_UP, lay.wg, lay.wu)
    lay.dn_w, lay.dn = tpx.tp_partition_weights(lay.sh, tpx.TP_W_DOWN, lay.wd)
    w = []
    for m in (lay.wqkv, lay.wo, lay.wg, lay.wu, lay.wd):
        q, sc = O.quantize_fp8_per_channel(O.as_f64(bits(m)))
        w.append(O.dequantize_fp8(q, sc))
    return w


@pytest.mark.parametrize("M,t,wtype", [(200, 8, tpx.TP_BF16), (65, 2, tpx.TP_BF16), (300, 8, tpx.TP_FP8_E4M3)],
                         ids=["bf16-200", "bf16-65-t2", "fp8-300"])
def test_layer_prefill_norm_folded(dev, M, t, wtype):
    """Prefill layers (M > 64), with separate RMSNorm launches (the default) and with
    TP_F_FOLD_NORM, where the norms become per-token factors on the tcgen05 GEMMs' accumulators
    (the factors of x from one pass over x, those of h1 from the sums of squares the o_proj
    epilogue leaves while it writes h1) and the normalised activations are never written.
    Every output of both against the oracle, and bit for bit from run to run."""
    d, ffn, n_q, n_kv, hd = 2048, 6656 if wtype == tpx.TP_BF16 else 7168, 16, 8, 128
    lay = Layer(d, ffn, n_q, n_kv, hd, t, 0, dev, seed=5)
    w = lay.weights() if wtype == tpx.TP_BF16 else _fp8_layer(lay, d, ffn, n_q, n_kv, hd, t)
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(lay.sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(lay.sh, M, dev)
    x = inputs.normal_bf16((M, d), 1.0, 5, inputs.STREAM_X, dev)
    y_split = lay.gpu(x, scratch, ws)
    y_split_ref, h1_ref = O.layer(bits(x), *w, n_q, n_kv, hd, bf16_between_blocks=True)
    check_layer(bits(y_split), y_split_ref, h1_ref, what=f"separate-norm prefill layer M={M}")
    fold = tpx.TP_F_FOLD_NORM
    n0 = tpx.tp_launch_count()
    y = lay.gpu(x, scratch, ws, fold)
    # factors of x, QKV, attention stand-in, o_proj, factors of h1, gate/up, down
    # (e4m3 weights: each GEMM's weights widened first)
    assert tpx.tp_launch_count() - n0 == (7 if wtype == tpx.TP_BF16 else 11)
    lay.check_outputs(bits(x), y, scratch, what=f"folded-norm prefill layer M={M} t={t}", weights=w)
    y2 = lay.gpu(x, scratch, ws, fold)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_70b_layer_prefill_norm_folded_sampled_rows(dev):
    """A 70B-shaped pre-norm layer (d 8192, ffn 28672, 64 q / 8 kv heads, t = 8) at prefill,
    M = 1000, through tp_layer_forward with the norms folded (TP_F_FOLD_NORM): every output on
    sampled token rows (first, last, tile edges) against the oracle."""
    lay = Layer(8192, 28672, 64, 8, 128, 8, 0, dev, seed=6)
    M = 1000
    scratch = torch.empty(tpx.tp_layer_scratch_bytes(lay.sh, M), dtype=torch.uint8, device=dev)
    ws = tpx.new_workspace(lay.sh, M, dev)
    x = inputs.normal_bf16((M, 8192), 1.0, 6, inputs.STREAM_X, dev)
    y = lay.gpu(x, scratch, ws, tpx.TP_F_FOLD_NORM)
    rows = np.array([0, 1, 127, 128, 255, 256, 511, 512, 767, 768, 998, 999])
    w = [O.as_f64(b) for b in lay.weights()]
    lay.check_outputs(bits(x), y, scratch, what="70B prefill layer, sampled rows", weights=w, rows=rows)
    assert not torch.isnan(y).any()
