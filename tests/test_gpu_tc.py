"""The tcgen05/TMA GEMM path (forced with TP_F_KERNEL_TC) against the float64 oracle:
exact-integer column- and row-parallel pieces first (a layout or descriptor mistake shows
up as a bit mismatch), then the blocks at decode and prefill token counts."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import Mlp, bits, check_close, check_h, run_proj  # noqa: F401

pytestmark = pytest.mark.gpu
TC, SK = tpx.TP_F_KERNEL_TC, tpx.TP_F_KERNEL_SKINNY


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.mark.parametrize("with_ws", [False, True])
@pytest.mark.parametrize("t,M", [(8, 19), (1, 5), (2, 64), (4, 130), (8, 300)])
def test_tc_colpar_exact_on_integers(dev, t, M, with_ws):
    """With a workspace the kernel may cut items across CTAs (stream-K); the pieces must
    still sum to the exact product."""
    d, n_q, n_kv, hd = 256, 16, 8, 32
    x = inputs.small_int_bf16((M, d), -2, 2, 1, 1, dev)
    w = inputs.small_int_bf16((d, (n_q + 2 * n_kv) * hd), -2, 2, 1, 2, dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, w)
    out = torch.full((M, (n_q + 2 * n_kv) * hd), float("nan"), dtype=torch.float32, device=dev)
    ws = tpx.new_workspace(sh, M, dev) if with_ws else None
    tpx.tp_colpar_forward(q, q_w, x, out, flags=tpx.TP_F_FP32_COLPAR_OUT | TC, ws=ws)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    full = O.as_f64(bits(x)) @ O.as_f64(bits(w))
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    assert np.array_equal(out.cpu().numpy().astype(np.float64), full[:, cols])


@pytest.mark.parametrize("t,M", [(8, 37), (2, 64), (4, 200)])
def test_tc_rowpar_partials_exact_on_integers(dev, t, M):
    d, ffn = 256, 1024
    a = inputs.small_int_bf16((M, ffn), -2, 2, 2, 1, dev)
    w = inputs.small_int_bf16((ffn, d), -2, 2, 2, 2, dev)
    sh = tpx.make_shape(d, ffn=ffn, t=t)
    w_p, desc = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, w)
    P = torch.full((t, M, d), float("nan"), dtype=torch.float32, device=dev)
    st = tpx.lib().tp_rowpar_partials(desc, tpx._ptr(w_p), tpx._ptr(a), M, tpx._ptr(P), tpx._stream(None))
    assert st == tpx.TP_OK
    # the default policy picks the tcgen05 kernel for M > 16 on this geometry
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    af, wf = O.as_f64(bits(a)), O.as_f64(bits(w))
    ks = ffn // t
    for s in range(t):
        ref = af[:, s * ks:(s + 1) * ks] @ wf[s * ks:(s + 1) * ks]
        assert np.array_equal(P[s].cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("M", [1, 8, 32, 64])
@pytest.mark.parametrize("t", [1, 8])
def test_tc_8b_mlp_decode(dev, t, M):
    m = Mlp(4096, 14336, t, M, dev)
    y, h = m.run(flags=TC)
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, what=f"tc 8B MLP t={t} M={M}")
    check_h(bits(h), h_ref, what="tc 8B h")
    y0, _ = m.run(residual=False, flags=TC)
    y0_ref, _ = m.oracle(residual=False)
    check_close(bits(y0), y0_ref, what=f"tc 8B MLP (no residual) t={t} M={M}")


def test_tc_fused_and_unfused_agree_and_are_deterministic(dev):
    """Fused: every shard's k-blocks chained in shard order into one accumulator.  Unfused:
    per-shard fp32 partials, then the left fold.  Both are fixed-order sums of the same terms,
    so they agree to rounding, and each repeats bit for bit."""
    for t, M in [(8, 64), (2, 13), (4, 40)]:
        m = Mlp(4096, 14336, t, M, dev, seed=1)
        y_ref, _ = m.oracle()
        y1, _ = m.run(flags=TC)
        y2, _ = m.run(flags=TC | tpx.TP_F_UNFUSED_REDUCE)
        check_close(bits(y1), y_ref, what=f"fused t={t} M={M}")
        check_close(bits(y2), y_ref, what=f"unfused t={t} M={M}")
        for _ in range(2):
            y3, _ = m.run(flags=TC)
            y4, _ = m.run(flags=TC | tpx.TP_F_UNFUSED_REDUCE)
            assert torch.equal(y1.view(torch.int16), y3.view(torch.int16)), (t, M)
            assert torch.equal(y2.view(torch.int16), y4.view(torch.int16)), (t, M)


@pytest.mark.parametrize("M", [65, 130, 300])
def test_tc_prefill_shaped_mlp(dev, M):
    """M > 64: one launch over all tokens; the row-parallel half chains the shards in one
    accumulator (shard order) instead of storing partials."""
    m = Mlp(1024, 4096, 8, M, dev, seed=2)
    y, h = m.run(flags=TC)
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, what=f"tc prefill-shaped MLP M={M}")
    check_h(bits(h), h_ref, what="tc prefill h")
    y0, _ = m.run(residual=False, flags=TC)
    y0_ref, _ = m.oracle(residual=False)
    check_close(bits(y0), y0_ref, what=f"tc prefill-shaped MLP (no residual) M={M}")
    y2, _ = m.run(flags=TC)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("t,M", [(8, 32), (4, 200)])
def test_tc_attention_projections(dev, t, M):
    y, qkv, y_ref, qkv_ref = run_proj(2048, 16, 8, 128, t, M, dev)
    check_close(bits(qkv), qkv_ref, what=f"tc qkv t={t} M={M}")
    check_close(bits(y), y_ref, what=f"tc o_proj t={t} M={M}")


def test_tc_and_skinny_both_within_bar(dev):
    """Both kernels at the same shape meet the bar against the oracle (they round differently,
    so they are not compared with each other)."""
    m = Mlp(4096, 14336, 8, 32, dev, seed=4)
    y_ref, _ = m.oracle()
    for f in (TC, SK):
        y, _ = m.run(flags=f)
        check_close(bits(y), y_ref, what=f"flags={f}")


@pytest.mark.parametrize("t,M", [(8, 64), (8, 16), (1, 32)])
def test_tc_streamk_rowpar_exact_on_integers(dev, t, M):
    """Row-parallel through the fused entry point (stream-K pieces, then the shard fold) on
    integers: the result is exact, so every piece and every shard must be summed once."""
    d, ffn = 1024, 8192
    a = inputs.small_int_bf16((M, ffn), -1, 1, 5, 1, dev)
    w = inputs.small_int_bf16((ffn, d), -1, 1, 5, 2, dev)
    res = inputs.small_int_bf16((M, d), -4, 4, 5, 3, dev)
    sh = tpx.make_shape(d, ffn=ffn, t=t)
    w_p, desc = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, w)
    ws = tpx.new_workspace(sh, M, dev)
    y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=dev)
    tpx.tp_rowpar_forward(desc, w_p, a, res, y, ws, flags=TC)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    exact = O.as_f64(bits(a)) @ O.as_f64(bits(w)) + O.as_f64(bits(res))
    assert np.array_equal(bits(y), O.f64_to_bf16_bits(exact))


# ---------------------------------------------------------------- full-size configurations


def _layer(dev, M, t=8, d=8192, ffn=28672, n_q=64, n_kv=8, hd=128, seed=0, wtype=tpx.TP_BF16):
    """A 70B-shaped layer's linear parts through the public entry points, as the bench runs it."""
    sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=wtype)
    x, wg, wu, wd = inputs.mlp_inputs(d, ffn, M, seed=seed, device=dev)
    _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=seed, device=dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y1 = torch.full_like(x, float("nan"))
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    h = torch.full((M, ffn), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y1, qkv, o_in, ws)
    tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, y1, y1, y, h, ws)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    return x, y1, y, (wqkv, wo, wg, wu, wd), (n_q, n_kv, hd)


def test_70b_layer_decode_full(dev):
    """70B-shaped layer at decode M=32, t=8: every output against the oracle, block by block
    (the MLP block is checked on the GPU path's own bf16 input to it)."""
    x, y1, y, (wqkv, wo, wg, wu, wd), (n_q, n_kv, hd) = _layer(dev, 32)
    y1_ref, _ = O.proj(bits(x), bits(wqkv), bits(wo), n_q, n_kv, hd, residual=bits(x))
    check_close(bits(y1), y1_ref, what="70B attention block, decode")
    y_ref, _ = O.mlp(bits(y1), bits(wg), bits(wu), bits(wd), residual=bits(y1))
    check_close(bits(y), y_ref, what="70B MLP block, decode")
    d0, _ = O.mlp(bits(y1), bits(wg), bits(wu), bits(wd))
    check_close(O.as_f64(bits(y)) - O.as_f64(bits(y1)), d0, rel=1e-2, mx=4e-2,
                what="70B MLP block without the residual (bf16 output rounding included)")


def test_70b_layer_prefill_sampled_rows(dev):
    """70B-shaped layer at prefill M=4096, t=8, in the launch configuration the bench times.
    Each output row depends only on its own input row, so the oracle checks a sample of rows
    spread over every token tile (first, last and ragged positions included)."""
    M = 4096
    x, y1, y, (wqkv, wo, wg, wu, wd), (n_q, n_kv, hd) = _layer(dev, M)
    rows = np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 2048, 3071, 4094, 4095])
    xb, y1b = bits(x)[rows], bits(y1)[rows]
    y1_ref, _ = O.proj(xb, bits(wqkv), bits(wo), n_q, n_kv, hd, residual=xb)
    check_close(y1b, y1_ref, what="70B attention block, prefill rows")
    y_ref, _ = O.mlp(y1b, bits(wg), bits(wu), bits(wd), residual=y1b)
    check_close(bits(y)[rows], y_ref, what="70B MLP block, prefill rows")
    assert not torch.isnan(y).any() and not torch.isnan(y1).any()


def test_70b_fp8_layer_prefill_sampled_rows(dev):
    """70B-shaped layer with e4m3 weights at prefill M=8192, t=8, in the launch configuration
    the bench times (each weight widened once into the workspace's bf16 scratch, 0.94 GB for
    the gate/up weight, then the tcgen05 GEMM with the per-channel scales in its epilogue).
    Sampled rows over every token tile, against the oracle on the dequantised weights."""
    M = 8192
    x, y1, y, ws_list, (n_q, n_kv, hd) = _layer(dev, M, wtype=tpx.TP_FP8_E4M3)
    deq = []
    for w in ws_list:
        q, s = O.quantize_fp8_per_channel(O.as_f64(bits(w)))
        deq.append(O.dequantize_fp8(q, s))
        del q
    wqkv, wo, wg, wu, wd = deq
    rows = np.array([0, 1, 127, 128, 255, 256, 1000, 4095, 4096, 6143, 8190, 8191])
    xb, y1b = bits(x)[rows], bits(y1)[rows]
    y1_ref, _ = O.proj(xb, wqkv, wo, n_q, n_kv, hd, residual=xb)
    check_close(y1b, y1_ref, what="70B fp8 attention block, prefill rows")
    y_ref, _ = O.mlp(y1b, wg, wu, wd, residual=y1b)
    check_close(bits(y)[rows], y_ref, what="70B fp8 MLP block, prefill rows")
    assert not torch.isnan(y).any() and not torch.isnan(y1).any()


def test_one_workspace_shared_across_token_counts(dev):
    """Back-to-back forwards with different M on one workspace (as a serving loop or the bench
    does): the work-balancing scratch sits at a fixed offset, so every call agrees on it."""
    d, ffn, t = 4096, 14336, 8
    sh = tpx.make_shape(d, ffn=ffn, t=t)
    x0, wg, wu, wd = inputs.mlp_inputs(d, ffn, 64, seed=6, device=dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    ws = tpx.new_workspace(sh, 64, dev)
    wf = [O.as_f64(bits(w)) for w in (wg, wu, wd)]
    outs = []
    for M in (32, 64, 32, 1, 64, 17):
        x = x0[:M].contiguous()
        y = torch.full_like(x, float("nan"))
        h = torch.full((M, ffn), float("nan"), dtype=torch.bfloat16, device=dev)
        tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, x, x, y, h, ws)
        outs.append((M, x, y))
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    for M, x, y in outs:
        y_ref, _ = O.mlp(bits(x), *wf, residual=bits(x))
        check_close(bits(y), y_ref, what=f"shared workspace M={M}")


# ---------------------------------------------------------------- FP8 e4m3 weights on tcgen05


@pytest.mark.parametrize("t,M", [(8, 16), (2, 1), (4, 130), (8, 300)])
def test_tc_fp8_mlp(dev, t, M):
    """e4m3 weights widened to bf16 in shared memory, scales applied per output channel in
    the epilogue: against the oracle on the dequantised weights (the 3e-2 FP8 bar, and the
    bf16 bar, which it also meets)."""
    m = Mlp(2048, 7168, t, M, dev, seed=8, wtype=tpx.TP_FP8_E4M3)
    y, h = m.run(flags=TC)
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, rel=5e-3, mx=2e-2, what=f"tc fp8 MLP t={t} M={M}")
    check_h(bits(h), h_ref, what="tc fp8 h")
    y0, _ = m.run(residual=False, flags=TC)
    y0_ref, _ = m.oracle(residual=False)
    check_close(bits(y0), y0_ref, rel=5e-3, mx=2e-2, what=f"tc fp8 MLP no residual t={t} M={M}")


def test_tc_fp8_attention_projections(dev):
    d, n_q, n_kv, hd, t, M = 1024, 8, 4, 128, 4, 48
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=5, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=tpx.TP_FP8_E4M3)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y, qkv, o_in, ws, flags=TC)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    deq = []
    for w in (wqkv, wo):
        qq, ss = O.quantize_fp8_per_channel(O.as_f64(bits(w)))
        deq.append(O.dequantize_fp8(qq, ss))
    y_ref, qkv_ref = O.proj(bits(x), deq[0], deq[1], n_q, n_kv, hd, residual=bits(x))
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    check_close(bits(qkv), qkv_ref[:, cols], what="tc fp8 qkv")
    check_close(bits(y), y_ref, what="tc fp8 o_proj")


def test_fp8_widening_is_exact_for_every_code(dev):
    """The converter's integer-plus-multiply e4m3 -> bf16 widening against the oracle's decode
    of every one of the 256 codes (NaN codes aside: quantised weights are finite)."""
    codes = torch.arange(256, dtype=torch.uint8, device=dev)
    out = torch.empty(256, dtype=torch.bfloat16, device=dev)
    tpx.tp_selftest_e4m3_decode(codes, out)
    torch.cuda.synchronize()
    want = O.e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))
    got = O.as_f64(bits(out))
    finite = ~np.isnan(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(want[finite]))   # -0 stays -0


@pytest.mark.parametrize("t,M", [(8, 300), (2, 129)])
def test_fp8_prefill_widened_once_equals_widened_per_tile(dev, t, M):
    """Prefill with e4m3 weights: widened once per call into the workspace, then a bf16 GEMM
    (workspace given), or widened tile by tile in shared memory (no workspace).  Same bf16
    values, same MMA order, same epilogue scales: the same bits, and the oracle's bar."""
    m = Mlp(2048, 7168, t, M, dev, seed=15, wtype=tpx.TP_FP8_E4M3)
    h_once = torch.full((M, m.ffn), float("nan"), dtype=torch.bfloat16, device=dev)
    h_tile = torch.full_like(h_once, float("nan"))
    ws = tpx.new_workspace(m.sh, M, dev)
    assert ws.numel() >= tpx.tp_workspace_bytes(m.sh, M) > tpx.tp_workspace_bytes(m.sh, 64)
    tpx.tp_colpar_forward(m.gu, m.gu_w, m.x, h_once, flags=TC, ws=ws)
    tpx.tp_colpar_forward(m.gu, m.gu_w, m.x, h_tile, flags=TC)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    assert torch.equal(h_once.view(torch.int16), h_tile.view(torch.int16))
    _, h_ref = m.oracle()
    check_h(bits(h_once), h_ref, what=f"fp8 prefill h t={t} M={M}")
