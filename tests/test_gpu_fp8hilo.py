"""Hi/lo activation codes on the e4m3-weight decode block (TP_F_FP8_HILO, the default): one persistent tcgen05
launch per block that splits each bf16 activation exactly into two e4m3 codes, x / s = hi + lo
with s a power of two per token, and multiplies e4m3 x e4m3 (kind::f8f6f4) with the weights
taken from shared memory as they landed.  The numeric reading is the default one (bf16
activations times the e4m3 weights, fp32 sums), so the checks are:
  - the oracle on the dequantised weights at the bf16 bars, t in {1, 2, 4, 8}, ragged token
    counts, with and without the residual;
  - agreement with the widening tcgen05 block (the same products, summed in another order)
    well inside those bars;
  - token rows of very different magnitudes (each token has its own scale), zero rows;
  - the Llama-3.1-70B shapes;
  - bit-for-bit repeats on one workspace shared with the other fused blocks (the maxima the
    scales come from must be back at zero after every launch)."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_fused import _fp8_proj, same_bits
from tests.test_gpu_parity import Mlp, bits, check_close, check_h

pytestmark = pytest.mark.gpu
FP8, SPL, TC = tpx.TP_FP8_E4M3, tpx.TP_F_FP8_HILO, tpx.TP_F_KERNEL_TC


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.mark.parametrize("t,M", [(1, 16), (2, 5), (4, 64), (8, 16), (8, 1), (2, 33)])
def test_hilo_blocks_vs_oracle(dev, t, M):
    m = Mlp(2048, 7168, t, M, dev, seed=23, wtype=FP8)
    for res in (True, False):
        y, h = m.run(residual=res, flags=SPL)
        y_ref, h_ref = m.oracle(residual=res)
        check_close(bits(y), y_ref, what=f"hilo MLP t={t} M={M} res={res}")
        check_h(bits(h), h_ref, what=f"hilo h t={t} M={M}")
    qkv, qkv_ref, y, y_ref = _fp8_proj(1024, 16, 8, 64, t, M, dev, seed=24, flags=SPL)
    check_close(bits(qkv), qkv_ref, what=f"hilo qkv t={t} M={M}")
    check_close(bits(y), y_ref, what=f"hilo o_proj t={t} M={M}")


def close_to(a, b, what):
    """Two GPU paths with the same products in another summation order: each stored bf16 value
    within one bf16 ulp (at most 2^-7 relative) of the other's plus 1e-3 RMS, relF far inside
    the bar."""
    af, bf = O.as_f64(bits(a)), O.as_f64(bits(b))
    r = O.rel_frobenius(af, bf)
    rms = np.sqrt(np.mean(bf * bf))
    excess = np.abs(af - bf) - (2.0 ** -7 * np.abs(bf) + 1e-3 * rms)
    assert r <= 1e-3 and np.all(excess <= 0), f"{what}: relF {r:.3e}, worst excess {excess.max():.3e}"


@pytest.mark.parametrize("t,M", [(2, 16), (8, 48)])
def test_hilo_agrees_with_widening_block(dev, t, M):
    m = Mlp(2048, 7168, t, M, dev, seed=25, wtype=FP8)
    ys, hs = m.run(flags=SPL)
    yw, hw = m.run(flags=TC)
    close_to(hs, hw, f"h hilo vs widened t={t} M={M}")
    close_to(ys, yw, f"y hilo vs widened t={t} M={M}")
    qs, _, ps, _ = _fp8_proj(1024, 16, 8, 64, t, M, dev, seed=26, flags=SPL)
    qw, _, pw, _ = _fp8_proj(1024, 16, 8, 64, t, M, dev, seed=26, flags=TC)
    close_to(qs, qw, f"qkv hilo vs widened t={t} M={M}")
    close_to(ps, pw, f"o_proj hilo vs widened t={t} M={M}")


def test_hilo_token_magnitudes(dev):
    """Every token has its own power-of-two scale: rows 2^-24 .. 2^24 apart, a zero row, a row
    with one outlier, must each meet the bar on their own."""
    t, M, d, ffn = 2, 16, 1024, 4096
    m = Mlp(d, ffn, t, M, dev, seed=27, wtype=FP8)
    x = m.x.clone()
    for i, k in enumerate(range(-24, 25, 4)):
        x[i] *= 2.0 ** k
    x[13] = 0.0
    x[14, 100] = 3.0e3
    y, h = m.run(flags=SPL, x=x)
    y_ref, h_ref = m.oracle(x=x)
    for i in range(M):
        if i == 13:
            assert torch.all(y[i] == 0) and torch.all(h[i] == 0)
            continue
        check_close(bits(y[i:i + 1]), y_ref[i:i + 1], what=f"hilo y, token {i}")
        check_h(bits(h[i:i + 1]), h_ref[i:i + 1], what=f"hilo h, token {i}")


@pytest.mark.parametrize("t,M", [(1, 16), (8, 16), (8, 4)])
def test_hilo_70b_blocks_vs_oracle(dev, t, M):
    m = Mlp(8192, 28672, t, M, dev, seed=28, wtype=FP8)
    y, h = m.run(flags=SPL)
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, what=f"hilo 70B MLP t={t} M={M}")
    check_h(bits(h), h_ref, what=f"hilo 70B h t={t} M={M}")
    qkv, qkv_ref, y, y_ref = _fp8_proj(8192, 64, 8, 128, t, M, dev, seed=29, flags=SPL)
    check_close(bits(qkv), qkv_ref, what=f"hilo 70B qkv t={t} M={M}")
    check_close(bits(y), y_ref, what=f"hilo 70B o_proj t={t} M={M}")


def test_hilo_repeats_bitwise_with_one_shared_workspace(dev):
    """Split and widening blocks of several token counts, MLP and attention, interleaved on one
    workspace with overlapping launches: every repeat gives the same bits."""
    d, ffn, n_q, n_kv, hd, t = 2048, 7168, 16, 8, 128, 8
    sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=FP8)
    _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=30, device=dev)
    _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=30, device=dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    ws = tpx.new_workspace(sh, 64, dev)
    Ms = (1, 64, 8, 32, 5)
    xs = {M: inputs.normal_bf16((M, d), 1.0 + M, 30, 40 + M, dev) for M in Ms}

    def sweep():
        outs = []
        for i, M in enumerate(Ms):
            fl = SPL if i % 2 == 0 else TC
            y1 = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
            qkv = torch.empty((M, (n_q + 2 * n_kv) * hd), dtype=torch.bfloat16, device=dev)
            oi = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
            tpx.tp_proj_forward(q, q_w, o, o_w, xs[M], xs[M], y1, qkv, oi, ws, SPL)
            y = torch.empty_like(y1)
            h = torch.empty((M, ffn), dtype=torch.bfloat16, device=dev)
            tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, y1, y1, y, h, ws, fl)
            outs.append((y1, y))
        assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
        return outs

    first = sweep()
    for _ in range(3):
        again = sweep()
        for (a1, a2), (b1, b2) in zip(first, again):
            assert same_bits(a1, b1) and same_bits(a2, b2)
    M = Ms[-1]
    deq = [O.dequantize_fp8(*O.quantize_fp8_per_channel(O.as_f64(bits(w)))) for w in (wqkv, wo)]
    y_ref, _ = O.proj(bits(xs[M]), deq[0], deq[1], n_q, n_kv, hd, residual=bits(xs[M]))
    check_close(bits(first[-1][0]), y_ref, what="shared-workspace hilo proj")
