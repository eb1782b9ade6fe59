"""Head-sharded decode attention over a KV cache through the C ABI, against the float64
oracle: the appended cache entries bit for bit, the attention output within the bf16 bars
(fp32 scores, softmax and accumulation; one bf16 rounding of the output), across chunk
boundaries, empty histories and out-of-range lengths; then the whole attention block
(QKV column-parallel, attention, o_proj row-parallel with the shard fold)."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import bits, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def unshard_qkv(q_sh, t, n_q, n_kv, hd):
    """shard-major qkv columns -> the unsharded [q | k | v] order of the oracle"""
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    out = np.empty_like(q_sh)
    out[:, cols] = q_sh
    return out


def cache_to_oracle(c, t):
    """[t, M, n_kv/t, L, hd] -> [M, n_kv, L, hd]"""
    c = np.asarray(c)
    return np.concatenate([c[s] for s in range(t)], axis=1)


def run_case(dev, t, n_q, n_kv, hd, M, L, lens, seed=0, poison=False):
    Q = (n_q + 2 * n_kv) * hd
    sh = tpx.make_shape(n_q * hd, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    qkv = inputs.normal_bf16((M, Q), 1.0, seed, 80, dev)
    kc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, seed, 81, dev)
    vc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, seed, 82, dev)
    if poison:  # the new token's slot and every slot after it hold NaN before the call
        for m, n in enumerate(lens):
            if 0 <= n < L:
                kc[:, m, :, n:] = float("nan")
                vc[:, m, :, n:] = float("nan")
    k0, v0 = bits(kc).copy(), bits(vc).copy()
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tpx.tp_attn_workspace_bytes(sh, M, L), dtype=torch.uint8, device=dev)
    tpx.tp_attn_decode(sh, qkv, kc, vc, lens_d, o_in, ws)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    qkv_u = unshard_qkv(bits(qkv), t, n_q, n_kv, hd)
    k_ref, v_ref = O.append_kv(qkv_u, cache_to_oracle(k0, t), cache_to_oracle(v0, t), lens, n_q, n_kv, hd)
    assert np.array_equal(cache_to_oracle(bits(kc), t), k_ref)
    assert np.array_equal(cache_to_oracle(bits(vc), t), v_ref)
    o_ref = O.attention_decode(qkv_u, k_ref, v_ref, lens, n_q, n_kv, hd)
    return o_in, o_ref, (sh, qkv, kc, vc, lens_d, ws)


@pytest.mark.parametrize("t,n_q,n_kv,hd", [(1, 8, 4, 64), (2, 8, 4, 128), (4, 16, 4, 256), (2, 32, 2, 64)])
def test_attention_small_shapes(dev, t, n_q, n_kv, hd):
    M, L = 7, 600                             # five 128-position chunks, the last one ragged
    lens = [0, 1, 127, 255, 256, 599, 600]    # empty history, chunk edges, the last slot, out of range
    o_in, o_ref, _ = run_case(dev, t, n_q, n_kv, hd, M, L, lens)
    got = O.as_f64(bits(o_in))
    assert not got[6].any()                   # out of range: a zero row
    check_close(got[:6], o_ref[:6], what=f"attention t={t} n_q={n_q} n_kv={n_kv} hd={hd}")


def test_attention_ignores_slots_past_the_length(dev):
    """Cache slots after the new token are never read into the result, even when they hold NaN
    (a chunk is staged whole; its rows past the end must weigh exactly zero), and the new
    token's own slot counts with the appended values even if it is staged before the append
    lands (its old content here is NaN)."""
    lens = [5, 130, 299, 127]
    o_in, o_ref, _ = run_case(dev, 2, 8, 4, 128, 4, 300, lens, seed=3, poison=True)
    got = O.as_f64(bits(o_in))
    assert np.isfinite(got).all()
    check_close(got, o_ref, what="attention with NaN past the length")


def test_attention_70b_heads_long_context_and_repeat(dev):
    """70B's heads (64 q / 8 kv of 128) at t = 8, 8 sequences of mixed lengths up to 4096."""
    t, n_q, n_kv, hd, M, L = 8, 64, 8, 128, 8, 4096
    lens = [4095, 17, 1000, 2048, 0, 3333, 256, 4000]
    o_in, o_ref, (sh, qkv, kc, vc, lens_d, ws) = run_case(dev, t, n_q, n_kv, hd, M, L, lens, seed=1)
    check_close(bits(o_in), o_ref, what="70B decode attention")
    o2 = torch.empty_like(o_in)
    tpx.tp_attn_decode(sh, qkv, kc, vc, lens_d, o2, ws)     # appends the same k, v again: same cache
    assert torch.equal(o_in.view(torch.int16), o2.view(torch.int16))


def test_attention_block_end_to_end(dev):
    """x -> QKV (column-parallel) -> attention over the cache -> o_proj (row-parallel, fold,
    residual), every step in the library, against the oracle's block with real attention."""
    d, n_q, n_kv, hd, t, M, L = 2048, 16, 8, 128, 8, 4, 1024
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=2, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    kc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 2, 83, dev)
    vc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 2, 84, dev)
    k0, v0 = bits(kc).copy(), bits(vc).copy()
    lens = [3, 700, 1023, 512]
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    Q = (n_q + 2 * n_kv) * hd
    qkv = torch.empty((M, Q), dtype=torch.bfloat16, device=dev)
    o_in = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
    y = torch.full_like(x, float("nan"))
    ws = tpx.new_workspace(sh, M, dev)
    aws = torch.empty(tpx.tp_attn_workspace_bytes(sh, M, L), dtype=torch.uint8, device=dev)
    tpx.tp_colpar_forward(q, q_w, x, qkv, ws=ws)
    tpx.tp_attn_decode(sh, qkv, kc, vc, lens_d, o_in, aws)
    tpx.tp_rowpar_forward(o, o_w, o_in, x, y, ws)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    # oracle: qkv = x Wqkv (fp64), stored as bf16; attention over the appended caches; o_proj
    qkv_ref = O.f64_to_bf16_bits(O.as_f64(bits(x)) @ O.as_f64(bits(wqkv)))
    k_ref, v_ref = O.append_kv(qkv_ref, cache_to_oracle(k0, t), cache_to_oracle(v0, t), lens, n_q, n_kv, hd)
    o_ref = O.f64_to_bf16_bits(O.attention_decode(qkv_ref, k_ref, v_ref, lens, n_q, n_kv, hd))
    y_ref = O.as_f64(o_ref) @ O.as_f64(bits(wo)) + O.as_f64(bits(x))
    check_close(bits(y), y_ref, what="attention block with a KV cache")


@pytest.mark.parametrize("wtype", [tpx.TP_BF16, tpx.TP_FP8_E4M3])
def test_attention_block_in_one_call(dev, wtype):
    """tp_attn_block_forward = QKV, the cache append + attention, o_proj with the shard fold, in one
    call: the same bits as the three calls, and the oracle's block within the bars (for e4m3
    weights, the oracle on the dequantised weights)."""
    d, n_q, n_kv, hd, t, M, L = 2048, 16, 8, 128, 8, 4, 1024
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=5, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=wtype)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    kc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 5, 85, dev)
    vc = inputs.normal_bf16((t, M, n_kv // t, L, hd), 1.0, 5, 86, dev)
    k0, v0 = bits(kc).copy(), bits(vc).copy()
    kc2, vc2 = kc.clone(), vc.clone()
    lens = [1023, 0, 300, 777]
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    Q = (n_q + 2 * n_kv) * hd
    # one call
    qkv1 = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o1 = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    y1 = torch.full_like(x, float("nan"))
    bws = tpx.new_attn_block_workspace(sh, M, L, dev)
    tpx.tp_attn_block_forward(q, q_w, o, o_w, x, x, kc, vc, lens_d, y1, qkv1, o1, bws)
    # three calls
    qkv2 = torch.empty((M, Q), dtype=torch.bfloat16, device=dev)
    o2 = torch.empty((M, n_q * hd), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty_like(x)
    ws = tpx.new_workspace(sh, M, dev)
    aws = torch.empty(tpx.tp_attn_workspace_bytes(sh, M, L), dtype=torch.uint8, device=dev)
    tpx.tp_colpar_forward(q, q_w, x, qkv2, ws=ws)
    tpx.tp_attn_decode(sh, qkv2, kc2, vc2, lens_d, o2, aws)
    tpx.tp_rowpar_forward(o, o_w, o2, x, y2, ws)
    assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
    for a_, b_ in ((qkv1, qkv2), (o1, o2), (y1, y2), (kc, kc2), (vc, vc2)):
        assert torch.equal(a_.view(torch.int16), b_.view(torch.int16))
    # oracle
    wq_ref, wo_ref = O.as_f64(bits(wqkv)), O.as_f64(bits(wo))
    if wtype == tpx.TP_FP8_E4M3:
        wq_ref = O.dequantize_fp8(*O.quantize_fp8_per_channel(wq_ref))
        wo_ref = O.dequantize_fp8(*O.quantize_fp8_per_channel(wo_ref))
    qkv_ref = O.f64_to_bf16_bits(O.as_f64(bits(x)) @ wq_ref)
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    check_close(bits(qkv1), O.as_f64(qkv_ref)[:, cols], what="block qkv")
    k_ref, v_ref = O.append_kv(qkv_ref, cache_to_oracle(k0, t), cache_to_oracle(v0, t), lens, n_q, n_kv, hd)
    o_ref = O.f64_to_bf16_bits(O.attention_decode(qkv_ref, k_ref, v_ref, lens, n_q, n_kv, hd))
    y_ref = O.as_f64(o_ref) @ wo_ref + O.as_f64(bits(x))
    check_close(bits(y1), y_ref, what=f"attention block in one call, wtype {wtype}")
