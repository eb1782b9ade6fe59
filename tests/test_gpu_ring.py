"""The TMA-fed e4m3 decode kernel (1..32 tokens) through the C ABI, reached as the blocks' halves
in separate launches (TP_F_SPLIT_BLOCK; a whole decode block is one hi/lo launch by default),
against the float64 oracle on the dequantised weights: the MLP block (gate/up + SwiGLU, down + the shard fold) and the
attention projections (QKV, o_proj), for t in {1, 2, 4, 8} and ragged token counts; shapes
small enough that every (shard, row tile) is split across CTAs, so the pieces are merged;
the fused fold bit-equal to the unfused partials + fold path; repeat runs bit-identical."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import REL_F, REL_F_FP8, Mlp, bits, check_close

pytestmark = pytest.mark.gpu
SB = tpx.TP_F_SPLIT_BLOCK  # the halves as separate launches: the ring kernel for e4m3 decode


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def check_mlp(m, flags=SB, residual=True):
    y, h = m.run(residual=residual, flags=flags)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    y_ref, h_ref = m.oracle(residual=residual)
    what = f"e4m3 MLP d={m.d} ffn={m.ffn} t={m.t} M={m.M}"
    r, _ = check_close(bits(y), y_ref, rel=REL_F_FP8, mx=1.0, what=what)
    assert r <= REL_F, f"{what}: relF {r:.2e} above the bf16 bar"
    rh = O.rel_frobenius(bits(h), h_ref)
    assert rh <= REL_F, f"{what}: h relF {rh:.2e}"
    return y, h


@pytest.mark.parametrize("M", [1, 7, 16, 17, 32])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_ring_mlp_token_counts_and_shards(dev, t, M):
    check_mlp(Mlp(1024, 4096, t, M, dev, seed=M, wtype=tpx.TP_FP8_E4M3))


def test_ring_every_tile_split_into_pieces(dev):
    """d 256, ffn 1024, t 2: 32 gate/up units and 16 down units for 304 CTAs, so every tile is
    finished by the CTA that brings its last piece (up to four pieces a tile)."""
    for M in (1, 16, 32):
        check_mlp(Mlp(256, 1024, 2, M, dev, seed=10 + M, wtype=tpx.TP_FP8_E4M3))


def test_ring_fused_fold_bits_equal_unfused(dev):
    m = Mlp(1024, 4096, 8, 16, dev, seed=5, wtype=tpx.TP_FP8_E4M3)
    y0, h0 = m.run(flags=SB)
    y1, h1 = m.run(flags=SB | tpx.TP_F_UNFUSED_REDUCE)
    assert torch.equal(h0.view(torch.int16), h1.view(torch.int16))
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    y2, _ = m.run(flags=SB)
    assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))


def test_ring_agrees_with_the_mma_sync_kernel(dev):
    """Both e4m3 decode kernels against each other (different k orders: close, not equal)."""
    m = Mlp(2048, 7168, 8, 16, dev, seed=6, wtype=tpx.TP_FP8_E4M3)
    y0, _ = m.run(flags=SB)
    y1, _ = m.run(flags=tpx.TP_F_KERNEL_SKINNY)
    assert O.rel_frobenius(bits(y0), O.as_f64(bits(y1))) <= 2e-3


@pytest.mark.parametrize("t,M", [(1, 3), (2, 16), (8, 32)])
def test_ring_attention_projections(dev, t, M):
    d, n_q, n_kv, hd = 1024, 16, 8, 64
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=20 + t, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=tpx.TP_FP8_E4M3)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y, qkv, o_in, ws, SB)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    deq = []
    for w in (wqkv, wo):
        qc, s = O.quantize_fp8_per_channel(O.as_f64(bits(w)))
        deq.append(O.dequantize_fp8(qc, s))
    y_ref, qkv_ref = O.proj(bits(x), deq[0], deq[1], n_q, n_kv, hd, residual=bits(x))
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    check_close(bits(qkv), qkv_ref[:, cols], what=f"e4m3 qkv t={t} M={M}")
    check_close(bits(y), y_ref, what=f"e4m3 o_proj t={t} M={M}")
