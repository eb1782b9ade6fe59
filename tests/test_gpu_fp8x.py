"""FP8 x FP8 (TP_F_FP8_ACT): e4m3 weights and per-token e4m3 activations on the tensor cores
(tcgen05 kind::f8f6f4), through the C ABI, against the float64 oracle's FP8 x FP8 reading:
the quantiser's codes and scales bit for bit; the MLP's h within the bf16 bars; its output
within the bars against the oracle fed the kernel's own h (the quantiser decides codes from
the stored bf16 h, so both sides quantise the same bits), and end to end; decode-sized
token counts (stream-K pieces) and prefill sizes; chained and unfused folds; the attention
projections."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import REL_F, REL_F_FP8, Mlp, bits, check_close

pytestmark = pytest.mark.gpu
FLAG = tpx.TP_F_FP8_ACT


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def test_quantizer_codes_and_scales_bit_exact(dev):
    M, K = 37, 1024
    x = inputs.normal_bf16((M, K), 1.0, 3, 1, dev)
    x[4] = 0.0                                    # an all-zero row: scale 1, codes 0
    x[5] *= 3.0e4                                 # a large row
    x[6] *= 1.0e-5                                # a small row (subnormal codes appear)
    x[7, 11] = -7.0e3                             # one outlier
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((M,), dtype=torch.float32, device=dev)
    tpx.tp_quantize_fp8_per_token(x, q, s)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_fp8_per_token(O.as_f64(bits(x)))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def fp8x_mlp(d, ffn, t, M, dev, seed):
    m = Mlp(d, ffn, t, M, dev, seed=seed, wtype=tpx.TP_FP8_E4M3)
    m.ws = tpx.new_workspace(m.sh, M, dev, flags=FLAG)   # with room for the quantised activations
    return m


def check_fp8x_mlp(m, flags=FLAG):
    y, h = m.run(residual=True, flags=flags)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    wg, wu, wd = m.oracle_weights()
    xb = bits(m.x)
    y_ref, h_ref = O.mlp_fp8x(xb, wg, wu, wd, residual=xb)
    what = f"FP8 x FP8 MLP d={m.d} ffn={m.ffn} t={m.t} M={m.M}"
    check_close(bits(h), h_ref, what=what + " h")
    # the row-parallel half on the kernel's own h
    hq = O.dequantize_fp8_per_token(*O.quantize_fp8_per_token(O.as_f64(bits(h))))
    check_close(bits(y), hq @ wd + O.as_f64(xb), what=what + " y (own h)")
    check_close(bits(y), y_ref, rel=REL_F_FP8, mx=1.0, what=what + " y (end to end)")
    return y, h


@pytest.mark.parametrize("t,M", [(1, 200), (8, 200), (2, 16), (8, 16), (4, 1)])
def test_fp8x_mlp(dev, t, M):
    check_fp8x_mlp(fp8x_mlp(1024, 4096, t, M, dev, seed=t * 100 + M))


def test_fp8x_chained_and_unfused_folds(dev):
    """The fused row-parallel half chains every shard's k-blocks into one accumulator; the
    unfused one writes shard partials and folds them: the same column-parallel h bit for bit,
    outputs equal up to the order of the fp32 sums, each deterministic."""
    m = fp8x_mlp(1024, 4096, 8, 48, dev, seed=9)
    y0, h0 = m.run(flags=FLAG)
    y1, h1 = m.run(flags=FLAG | tpx.TP_F_UNFUSED_REDUCE)
    y2, _ = m.run(flags=FLAG)
    assert torch.equal(h0.view(torch.int16), h1.view(torch.int16))
    assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))
    assert O.rel_frobenius(bits(y0), O.as_f64(bits(y1))) <= 1e-3


@pytest.mark.parametrize("t,M", [(2, 130), (8, 16)])
def test_fp8x_attention_projections(dev, t, M):
    d, n_q, n_kv, hd = 1024, 16, 8, 64
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=30 + t, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=tpx.TP_FP8_E4M3)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev, flags=FLAG)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y, qkv, o_in, ws, flags=FLAG)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    wq_d = O.dequantize_fp8(*O.quantize_fp8_per_channel(O.as_f64(bits(wqkv))))
    wo_d = O.dequantize_fp8(*O.quantize_fp8_per_channel(O.as_f64(bits(wo))))
    a = O.dequantize_fp8_per_token(*O.quantize_fp8_per_token(O.as_f64(bits(x))))
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    check_close(bits(qkv), (a @ wq_d)[:, cols], what=f"FP8 x FP8 qkv t={t} M={M}")
    # o_proj on the kernel's own attention output (the one-token stand-in copies v)
    oq = O.dequantize_fp8_per_token(*O.quantize_fp8_per_token(O.as_f64(bits(o_in))))
    check_close(bits(y), oq @ wo_d + O.as_f64(bits(x)), what=f"FP8 x FP8 o_proj t={t} M={M}")
