"""The fused decode block: one persistent tcgen05 launch per tensor-parallel block.

The column-parallel items, then the row-parallel items, run from one queue; a row-parallel
item of shard s waits only for shard s's first half, and the last of the t shard items of a
128-row output tile folds the partials in shard order.  Checked here:
  - the same bits as the split path (separate launches, per-shard partials, fold kernel)
    wherever that path also runs whole items;
  - exact products on small-integer inputs, including the attention stand-in it folds
    into the QKV epilogue;
  - the float64 oracle's bars on random inputs, t in {1, 2, 4, 8}, ragged token counts;
  - bit-for-bit repeats, and a workspace shared by blocks of different kinds and sizes
    (the scheduler words must return to zero after every launch)."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import Mlp, bits, check_close, check_h, run_proj

pytestmark = pytest.mark.gpu
UNF, SPLIT, TC = tpx.TP_F_UNFUSED_REDUCE, tpx.TP_F_SPLIT_BLOCK, tpx.TP_F_KERNEL_TC


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [1, 8, 17, 32, 64])
def test_fused_mlp_bits_equal_split_partials_path(dev, M):
    """8B MLP at t = 8: 224 gate/up and 256 down items, so the split path also runs every
    item whole; per-shard partials and the shard-order fold make the two paths identical."""
    m = Mlp(4096, 14336, 8, M, dev, seed=5)
    yf, hf = m.run()
    yu, hu = m.run(flags=UNF)
    assert same_bits(hf, hu), "h differs"
    assert same_bits(yf, yu), "y differs"
    y_ref, h_ref = m.oracle()
    check_close(bits(yf), y_ref, what=f"fused 8B MLP M={M}")
    check_h(bits(hf), h_ref, what=f"fused 8B h M={M}")
    y0f, _ = m.run(residual=False)
    y0u, _ = m.run(residual=False, flags=UNF)
    assert same_bits(y0f, y0u)


def _proj_int_case(d, n_q, n_kv, hd, t, M, dev, lo=-2, hi=2, seed=7):
    x = inputs.small_int_bf16((M, d), lo, hi, seed, 1, dev)
    wqkv = inputs.small_int_bf16((d, (n_q + 2 * n_kv) * hd), lo, hi, seed, 2, dev)
    wo = inputs.small_int_bf16((n_q * hd, d), lo, hi, seed, 3, dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y, qkv, o_in, ws)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    # expected, from the oracle's pieces: every product and sum here is an exact integer
    xf, wq, wof = O.as_f64(bits(x)), O.as_f64(bits(wqkv)), O.as_f64(bits(wo))
    qkv_b = O.f64_to_bf16_bits(xf @ wq)                       # qkv is stored in bf16
    o_ref = O.attention_one_token(qkv_b, n_q, n_kv, hd)
    y_ref = O.f64_to_bf16_bits(o_ref @ wof + xf)
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    return bits(qkv), qkv_b[:, cols], bits(o_in), O.f64_to_bf16_bits(o_ref), bits(y), y_ref


@pytest.mark.parametrize("t,M", [(1, 1), (2, 5), (4, 64), (4, 33)])
def test_fused_proj_exact_on_integers(dev, t, M):
    qkv, qkv_ref, o_in, o_ref, y, y_ref = _proj_int_case(512, 8, 4, 64, t, M, dev)
    assert np.array_equal(qkv, qkv_ref)
    assert np.array_equal(o_in, o_ref)
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("M", [1, 8, 16])
def test_fused_proj_70b_shape_exact_on_integers(dev, M):
    """The 70B attention block (80 QKV tiles, 512 o_proj tiles) at one, eight and sixteen tokens:
    qkv, the attention stand-in and y bit-exact on small integers."""
    qkv, qkv_ref, o_in, o_ref, y, y_ref = _proj_int_case(8192, 64, 8, 128, 8, M, dev, lo=-1, hi=1)
    assert np.array_equal(qkv, qkv_ref)
    assert np.array_equal(o_in, o_ref)
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_fused_70b_proj_and_mlp_vs_oracle(dev, t):
    y, qkv, y_ref, qkv_ref = run_proj(8192, 64, 8, 128, t, 16, dev, seed=8)
    check_close(bits(qkv), qkv_ref, what=f"fused 70B qkv t={t}")
    check_close(bits(y), y_ref, what=f"fused 70B proj t={t}")
    m = Mlp(8192, 28672, t, 16, dev, seed=8)
    y, h = m.run()
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, what=f"fused 70B MLP t={t}")
    check_h(bits(h), h_ref, what=f"fused 70B h t={t}")


@pytest.mark.parametrize("d,ffn,t,M", [(256, 1024, 2, 8), (256, 1024, 2, 1), (1024, 4096, 4, 3),
                                       (1024, 4096, 8, 50), (4096, 14336, 1, 64), (2048, 8192, 2, 64)])
def test_fused_mlp_small_and_ragged_vs_oracle(dev, d, ffn, t, M):
    """Small shapes make some CTAs start on row-parallel items that wait for other CTAs'
    first-half items; ragged M masks the token tile."""
    m = Mlp(d, ffn, t, M, dev, seed=9)
    for res in (True, False):
        y, h = m.run(residual=res)
        y_ref, h_ref = m.oracle(residual=res)
        check_close(bits(y), y_ref, what=f"fused MLP d={d} t={t} M={M} res={res}")
        check_h(bits(h), h_ref, what="fused h")
        y2, _ = m.run(residual=res, flags=SPLIT)
        check_close(bits(y2), y_ref, what=f"split MLP d={d} t={t} M={M} res={res}")


def test_fused_repeats_bitwise_with_one_shared_workspace(dev):
    """MLP and attention blocks of several token counts share one workspace, interleaved, with
    overlapping launches (programmatic dependent launch): every repeat gives the same bits, which
    needs the scheduler words and tile tickets back at zero after every launch."""
    d, ffn, n_q, n_kv, hd, t = 4096, 14336, 32, 8, 128, 8
    sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=11, device=dev)
    _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=11, device=dev)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    ws = tpx.new_workspace(sh, 64, dev)
    Ms = (1, 64, 8, 32, 5)
    xs = {M: inputs.normal_bf16((M, d), 1.0, 11, 40 + M, dev) for M in Ms}

    def sweep():
        outs = []
        for M in Ms:
            y1 = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
            qkv = torch.empty((M, (n_q + 2 * n_kv) * hd), dtype=torch.bfloat16, device=dev)
            oi = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
            tpx.tp_proj_forward(q, q_w, o, o_w, xs[M], xs[M], y1, qkv, oi, ws)
            y = torch.empty_like(y1)
            h = torch.empty((M, ffn), dtype=torch.bfloat16, device=dev)
            tpx.tp_mlp_forward(gu, gu_w, dn, dn_w, y1, y1, y, h, ws)
            outs.append((y1, y))
        assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
        return outs

    first = sweep()
    for _ in range(3):
        again = sweep()
        for (a1, a2), (b1, b2) in zip(first, again):
            assert same_bits(a1, b1) and same_bits(a2, b2)
    # and the last results still meet the oracle's bar
    M = Ms[-1]
    y_ref, _ = O.proj(bits(xs[M]), bits(wqkv), bits(wo), n_q, n_kv, hd, residual=bits(xs[M]))
    check_close(bits(first[-1][0]), y_ref, what="shared-workspace proj")


# ---------------------------------------------------------------- e4m3 weights

FP8 = tpx.TP_FP8_E4M3


@pytest.mark.parametrize("M", [1, 16, 64])
def test_fused_fp8_mlp_bits_equal_split_partials_path(dev, M):
    """e4m3 weights: the fused kernel widens each tile into tensor memory, the split path into
    shared memory.  Both feed the same bf16 values to the same MMA sequence and scale in the
    epilogue, so at the 8B shape (no split items on either path) the bits agree."""
    m = Mlp(4096, 14336, 8, M, dev, seed=12, wtype=FP8)
    yf, hf = m.run(flags=TC)
    yu, hu = m.run(flags=TC | UNF)
    assert same_bits(hf, hu), "h differs"
    assert same_bits(yf, yu), "y differs"
    y2, _ = m.run(flags=TC)
    assert same_bits(yf, y2)


def _fp8_proj(d, n_q, n_kv, hd, t, M, dev, seed, flags=0):
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=seed, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=FP8)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x, y, qkv, o_in, ws, flags)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    deq = []
    for w in (wqkv, wo):
        qq, ss = O.quantize_fp8_per_channel(O.as_f64(bits(w)))
        deq.append(O.dequantize_fp8(qq, ss))
    y_ref, qkv_ref = O.proj(bits(x), deq[0], deq[1], n_q, n_kv, hd, residual=bits(x))
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    return qkv, qkv_ref[:, cols], y, y_ref


@pytest.mark.parametrize("flags", [TC, 0, SPLIT], ids=["widened", "default-hilo", "halves"])
@pytest.mark.parametrize("t,M", [(1, 16), (2, 5), (4, 64), (8, 16)])
def test_fused_fp8_blocks_vs_oracle(dev, t, M, flags):
    """Against the oracle on the dequantised weights; the bf16 bar (stricter than the 3e-2 FP8
    bar) holds for both blocks: the one-launch block widening the weights (TP_F_KERNEL_TC), the
    default one-launch block on hi/lo activation codes, and the halves in separate launches
    (the mma.sync kernels)."""
    m = Mlp(2048, 7168, t, M, dev, seed=13, wtype=FP8)
    y, h = m.run(flags=flags)
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, what=f"fp8 MLP t={t} M={M} flags={flags}")
    check_h(bits(h), h_ref, what=f"fp8 h t={t} M={M}")
    y0, _ = m.run(residual=False, flags=flags)
    y0_ref, _ = m.oracle(residual=False)
    check_close(bits(y0), y0_ref, what=f"fp8 MLP no residual t={t} M={M}")
    qkv, qkv_ref, y, y_ref = _fp8_proj(1024, 16, 8, 64, t, M, dev, seed=14, flags=flags)
    check_close(bits(qkv), qkv_ref, what=f"fused fp8 qkv t={t} M={M}")
    check_close(bits(y), y_ref, what=f"fused fp8 o_proj t={t} M={M}")


@pytest.mark.parametrize("wtype,d,ffn,t,M", [(tpx.TP_BF16, 256, 1536, 8, 5), (tpx.TP_BF16, 256, 1536, 8, 16),
                                             (FP8, 384, 1536, 4, 16), (FP8, 384, 1536, 4, 33)],
                         ids=["bf16-M5", "bf16-M16", "e4m3-M16", "e4m3-M33"])
def test_fused_blocks_half_full_last_stage(dev, wtype, d, ffn, t, M):
    """A pipeline stage carries two k-blocks in one copy of weights and one of activations.
    These shapes leave an item's last stage half full: bf16 with 3 row-parallel k-blocks of 64,
    e4m3 (hi/lo, the default) with 3 k-blocks of 128 in both halves and in the attention block's
    column-parallel half.  The k-block past the item's end (zeros, or the next shard's
    activations) must not reach the products."""
    m = Mlp(d, ffn, t, M, dev, seed=31, wtype=wtype)
    for res in (True, False):
        y, h = m.run(residual=res)
        y_ref, h_ref = m.oracle(residual=res)
        check_close(bits(y), y_ref, what=f"MLP d={d} ffn={ffn} t={t} M={M} res={res}")
        check_h(bits(h), h_ref, what=f"h d={d} t={t} M={M}")
    if wtype == FP8:
        qkv, qkv_ref, y, y_ref = _fp8_proj(d, 8, 4, 64, 2, M, dev, seed=32)
        check_close(bits(qkv), qkv_ref, what=f"qkv d={d} M={M}")
        check_close(bits(y), y_ref, what=f"o_proj d={d} M={M}")
