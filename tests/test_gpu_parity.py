"""GPU parity: the CUDA path through the C ABI against the float64 CPU oracle.

Bars (per the tensor-parallel split-vs-unsplit equivalence the pages ask for, checked
equal up to floating-point rounding, engineer-atlas.dev 'What must stay true after deployment'):
relative Frobenius error <= 5e-3 and max |err| <= 2e-2 * RMS(y) for bf16 weights; 3e-2
relative Frobenius for FP8 weights against the oracle on the dequantised weights.
Integer, byte and layout work (packing, quantisation codes, exact-integer products,
the shard fold order) is compared bit for bit."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O

pytestmark = pytest.mark.gpu

REL_F, MAX_RMS, REL_F_FP8 = 5e-3, 2e-2, 3e-2


@pytest.fixture(scope="module", autouse=True)
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def bits(a):
    return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def shard_view(packed, desc, s, dtype=np.uint16):
    """Shard s of a packed buffer as a [rows, K] array of raw codes."""
    buf = packed.cpu().numpy()
    st = s * desc.shard_stride_bytes
    esz = 1 if dtype == np.uint8 else 2
    raw = buf[st: st + desc.rows_per_shard * desc.k_per_shard * esz]
    return raw.view(dtype).reshape(desc.rows_per_shard, desc.k_per_shard)


def shard_scales(packed, desc, s):
    buf = packed.cpu().numpy()
    st = s * desc.shard_stride_bytes + desc.scales_offset
    return buf[st: st + desc.rows_per_shard * 4].view(np.float32)


def check_h(h, h_ref, what=""):
    """Bar for a bf16-stored activation (SwiGLU's h, RMSNorm's output).  h is stored in bf16 (one RNE rounding, relative error <= 2^-9), and SwiGLU output is
    heavy-tailed (max |h| is many times its RMS), so the per-element bar for h is relative to
    each element: |h - h_ref| <= 2^-8 |h_ref| + 1e-3 RMS(h_ref), plus the relF bar."""
    hf, hr = O.as_f64(h), O.as_f64(h_ref)
    r = O.rel_frobenius(hf, hr)
    rms = np.sqrt(np.mean(hr * hr))
    excess = np.abs(hf - hr) - (2.0 ** -8 * np.abs(hr) + 1e-3 * rms)
    assert r <= REL_F and np.all(excess <= 0), f"{what}: relF {r:.3e}, worst excess {excess.max():.3e}"


def check_close(y, y_ref, rel=REL_F, mx=MAX_RMS, what=""):
    r, m = O.rel_frobenius(y, y_ref), O.max_err_over_rms(y, y_ref)
    assert r <= rel and m <= mx, f"{what}: relF {r:.3e} (bar {rel}), max/rms {m:.3e} (bar {mx})"
    return r, m


_WCACHE = {}   # oracle weights of the last shape (they do not depend on t or M)


class Mlp:
    """Packed MLP weights + buffers for one shape."""

    def __init__(self, d, ffn, t, M, dev, seed=0, wtype=tpx.TP_BF16, ints=False):
        if ints:
            x = inputs.small_int_bf16((M, d), -2, 2, seed, 1, dev)
            wg = inputs.small_int_bf16((d, ffn), -2, 2, seed, 2, dev)
            wu = inputs.small_int_bf16((d, ffn), -2, 2, seed, 3, dev)
            wd = inputs.small_int_bf16((ffn, d), -2, 2, seed, 4, dev)
        else:
            x, wg, wu, wd = inputs.mlp_inputs(d, ffn, M, seed=seed, device=dev)
        self.x, self.wg, self.wu, self.wd = x, wg, wu, wd
        self.sh = tpx.make_shape(d, ffn=ffn, t=t, wtype=wtype)
        self.gu_w, self.gu = tpx.tp_partition_weights(self.sh, tpx.TP_W_GATE_UP, wg, wu)
        self.dn_w, self.dn = tpx.tp_partition_weights(self.sh, tpx.TP_W_DOWN, wd)
        self.ws = tpx.new_workspace(self.sh, M, dev)
        self.d, self.ffn, self.t, self.M, self.dev = d, ffn, t, M, dev
        self.seed, self.ints = seed, ints

    def run(self, residual=True, flags=0, x=None):
        x = self.x if x is None else x
        y = torch.full_like(x, float("nan"))          # poisoned: unwritten outputs show up
        h = torch.full((x.shape[0], self.ffn), float("nan"), dtype=torch.bfloat16, device=self.dev)
        tpx.tp_mlp_forward(self.gu, self.gu_w, self.dn, self.dn_w, x, x if residual else None, y, h,
                           self.ws, flags)
        torch.cuda.synchronize()
        return y, h

    def oracle_weights(self):
        key = (self.d, self.ffn, self.seed, self.sh.wtype, self.ints)
        if key not in _WCACHE:
            _WCACHE.clear()
            if self.sh.wtype == tpx.TP_BF16:
                _WCACHE[key] = [O.as_f64(bits(w)) for w in (self.wg, self.wu, self.wd)]
            else:
                deq = []
                for w in (self.wg, self.wu, self.wd):
                    q, s = O.quantize_fp8_per_channel(O.as_f64(bits(w)))
                    deq.append(O.dequantize_fp8(q, s))
                _WCACHE[key] = deq
        return _WCACHE[key]

    def oracle(self, residual=True, x=None):
        xb = bits(self.x if x is None else x)
        wg, wu, wd = self.oracle_weights()
        return O.mlp(xb, wg, wu, wd, residual=xb if residual else None)


# ---------------------------------------------------------------- partition / pack


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_pack_gate_up_and_down_bit_exact(dev, t):
    d, ffn = 64, 256
    _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=3, device=dev)
    sh = tpx.make_shape(d, ffn=ffn, t=t)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    torch.cuda.synchronize()
    ref_gu = O.pack_colpar([bits(wg), bits(wu)], "gate_up", t, ffn=ffn)
    ref_dn = O.pack_rowpar(bits(wd), t)
    for s in range(t):
        assert np.array_equal(shard_view(gu_w, gu, s), ref_gu[s])
        assert np.array_equal(shard_view(dn_w, dn, s), ref_dn[s])


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_pack_qkv_and_o_bit_exact(dev, t):
    d, n_q, n_kv, hd = 256, 16, 8, 32
    _, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, 1, seed=4, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    torch.cuda.synchronize()
    ref_q = O.pack_colpar([bits(wqkv)], "qkv", t, n_q=n_q, n_kv=n_kv, hd=hd)
    ref_o = O.pack_rowpar(bits(wo), t)
    for s in range(t):
        assert np.array_equal(shard_view(q_w, q, s), ref_q[s])
        assert np.array_equal(shard_view(o_w, o, s), ref_o[s])


@pytest.mark.parametrize("t", [1, 8])
def test_pack_fp8_codes_and_scales_bit_exact(dev, t):
    d, ffn = 128, 512
    _, wg, wu, wd = inputs.mlp_inputs(d, ffn, 1, seed=5, device=dev)
    wg[:, 7] = 0                                              # an all-zero column: scale 1, codes 0
    sh = tpx.make_shape(d, ffn=ffn, t=t, wtype=tpx.TP_FP8_E4M3)
    gu_w, gu = tpx.tp_partition_weights(sh, tpx.TP_W_GATE_UP, wg, wu)
    dn_w, dn = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    torch.cuda.synchronize()
    qg, sg = O.quantize_fp8_per_channel(O.as_f64(bits(wg)))
    qu, su = O.quantize_fp8_per_channel(O.as_f64(bits(wu)))
    qd, sd = O.quantize_fp8_per_channel(O.as_f64(bits(wd)))
    ref_gu = O.pack_colpar([qg, qu], "gate_up", t, ffn=ffn)
    ref_gu_s = O.colpar_scales([sg, su], "gate_up", t, ffn=ffn)
    ref_dn = O.pack_rowpar(qd, t)
    for s in range(t):
        assert np.array_equal(shard_view(gu_w, gu, s, np.uint8), ref_gu[s])
        assert np.array_equal(shard_scales(gu_w, gu, s), ref_gu_s[s])
        assert np.array_equal(shard_view(dn_w, dn, s, np.uint8), ref_dn[s])
        assert np.array_equal(shard_scales(dn_w, dn, s), sd)   # row-parallel: replicated


# ---------------------------------------------------------------- exact linear pieces


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_colpar_qkv_exact_on_integers_and_t_invariant(dev, t):
    """Small-integer inputs make every fp32 sum exact, so the column-parallel output must
    equal the unsharded product bit for bit, mapped through the shard layout."""
    d, n_q, n_kv, hd, M = 512, 16, 8, 32, 19
    x = inputs.small_int_bf16((M, d), -2, 2, 1, 1, dev)
    w = inputs.small_int_bf16((d, (n_q + 2 * n_kv) * hd), -2, 2, 1, 2, dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, w)
    out = torch.full((M, (n_q + 2 * n_kv) * hd), float("nan"), dtype=torch.float32, device=dev)
    tpx.tp_colpar_forward(q, q_w, x, out, flags=tpx.TP_F_FP32_COLPAR_OUT)
    torch.cuda.synchronize()
    full = O.as_f64(bits(x)) @ O.as_f64(bits(w))
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    assert np.array_equal(out.cpu().numpy().astype(np.float64), full[:, cols])


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_rowpar_partials_and_fold_exact_on_integers(dev, t):
    d, ffn, M = 256, 1024, 37
    a = inputs.small_int_bf16((M, ffn), -2, 2, 2, 1, dev)
    w = inputs.small_int_bf16((ffn, d), -2, 2, 2, 2, dev)
    res = inputs.small_int_bf16((M, d), -4, 4, 2, 3, dev)
    sh = tpx.make_shape(d, ffn=ffn, t=t)
    w_p, desc = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, w)
    P = torch.full((t, M, d), float("nan"), dtype=torch.float32, device=dev)
    tpx.tp_rowpar_partials(desc, w_p, a, P)
    y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=dev)
    tpx.tp_reduce_partials(P, t, M, d, res, y)
    torch.cuda.synchronize()
    af, wf = O.as_f64(bits(a)), O.as_f64(bits(w))
    ks = ffn // t
    for s in range(t):
        assert np.array_equal(P[s].cpu().numpy().astype(np.float64), af[:, s * ks:(s + 1) * ks] @ wf[s * ks:(s + 1) * ks])
    exact = af @ wf + O.as_f64(bits(res))
    assert np.array_equal(bits(y), O.f64_to_bf16_bits(exact))   # |sums| < 2^8: exact in bf16 range


def test_reduce_fold_order_is_left_to_right(dev):
    """Partials whose fp32 sum depends on the order: the device must equal the stated fold
    (((P0 + P1) + P2) + ...) + residual, evaluated on the host in float32."""
    t, M, d = 8, 4, 64
    rng = np.random.default_rng(11)
    vals = np.array([1e8, 1.0, -1e8, 3.0, 0.5, -7.25, 1e-3, 2e7], dtype=np.float32)
    P = np.empty((t, M, d), dtype=np.float32)
    for s in range(t):
        P[s] = vals[(s + rng.integers(0, 8, size=(M, d))) % 8] * rng.choice([1, -1], size=(M, d))
    res = inputs.normal_bf16((M, d), 1.0, 3, 9, dev)
    y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=dev)
    tpx.tp_reduce_partials(torch.from_numpy(P).to(dev), t, M, d, res, y)
    torch.cuda.synchronize()
    acc = P[0].copy()
    for s in range(1, t):
        acc = (acc + P[s]).astype(np.float32)
    acc = (acc + O.as_f64(bits(res)).astype(np.float32)).astype(np.float32)
    assert np.array_equal(bits(y), O.f64_to_bf16_bits(acc.astype(np.float64)))
    # and a different order would have given different bits for some element
    rev = P[t - 1].copy()
    for s in range(t - 2, -1, -1):
        rev = (rev + P[s]).astype(np.float32)
    assert not np.array_equal(rev, acc - O.as_f64(bits(res)).astype(np.float32))


# ---------------------------------------------------------------- the MLP block


def test_tiny_mlp_with_and_without_residual(dev):
    m = Mlp(256, 1024, 2, 8, dev)
    y, h = m.run(residual=True)
    y_ref, h_ref = m.oracle(residual=True)
    check_close(bits(y), y_ref, what="tiny MLP")
    check_h(bits(h), h_ref, what="tiny h")
    y0, _ = m.run(residual=False)
    y0_ref, _ = m.oracle(residual=False)
    check_close(bits(y0), y0_ref, what="tiny MLP, no residual")


@pytest.mark.parametrize("kernel", [0, tpx.TP_F_KERNEL_SKINNY], ids=["default", "skinny"])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_8b_mlp_decode(dev, t, M, kernel):
    m = Mlp(4096, 14336, t, M, dev)
    y, h = m.run(flags=kernel)
    y_ref, h_ref = m.oracle()
    check_close(bits(y), y_ref, what=f"8B MLP t={t} M={M} flags={kernel}")
    y0, _ = m.run(residual=False, flags=kernel)
    y0_ref, _ = m.oracle(residual=False)
    check_close(bits(y0), y0_ref, what=f"8B MLP (no residual) t={t} M={M}")
    check_h(bits(h), h_ref, what="8B h")


@pytest.mark.parametrize("M", [3, 17, 50, 100, 130])
def test_ragged_token_counts(dev, M):
    m = Mlp(512, 2048, 4, M, dev, seed=7)
    y, _ = m.run(residual=False)
    y_ref, _ = m.oracle(residual=False)
    check_close(bits(y), y_ref, what=f"ragged M={M}")


def test_skinny_fused_equals_unfused_bitwise_and_deterministic(dev):
    """The mma.sync kernel's fused fold (in the CTA, or by the last CTA of a tile) and the
    unfused partials + fold kernel compute the same per-shard partials and the same left
    fold, so they give identical bits; every path repeats bit for bit."""
    sk = tpx.TP_F_KERNEL_SKINNY
    for t, M in [(8, 64), (2, 13), (1, 5)]:
        m = Mlp(4096, 14336, t, M, dev, seed=1)
        y1, _ = m.run(flags=sk)
        y2, _ = m.run(flags=sk | tpx.TP_F_UNFUSED_REDUCE)
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), (t, M)
        for _ in range(2):
            y3, _ = m.run(flags=sk)
            assert torch.equal(y1.view(torch.int16), y3.view(torch.int16)), (t, M)
            y4, _ = m.run()
            y5, _ = m.run()
            assert torch.equal(y4.view(torch.int16), y5.view(torch.int16)), (t, M)


def test_zero_tokens_is_a_no_op(dev):
    m = Mlp(256, 1024, 2, 1, dev)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    h = torch.empty((0, 1024), dtype=torch.bfloat16, device=dev)
    tpx.tp_mlp_forward(m.gu, m.gu_w, m.dn, m.dn_w, x, x, y, h, m.ws)


def test_outputs_stay_inside_their_buffers(dev):
    """Canary bands around y and h: nothing outside the [M, d] / [M, ffn] views is written."""
    d, ffn, M = 512, 2048, 21
    m = Mlp(d, ffn, 4, M, dev)
    pad = 4096
    ybig = torch.full((M * d + 2 * pad,), -776.0, dtype=torch.bfloat16, device=dev)
    hbig = torch.full((M * ffn + 2 * pad,), -776.0, dtype=torch.bfloat16, device=dev)
    y = ybig[pad:pad + M * d].view(M, d)
    h = hbig[pad:pad + M * ffn].view(M, ffn)
    tpx.tp_mlp_forward(m.gu, m.gu_w, m.dn, m.dn_w, m.x, m.x, y, h, m.ws)
    torch.cuda.synchronize()
    for big, n in ((ybig, M * d), (hbig, M * ffn)):
        assert torch.all(big[:pad] == -776.0) and torch.all(big[pad + n:] == -776.0)
    y_ref, _ = m.oracle()
    check_close(bits(y), y_ref, what="canary run")


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_fp8_mlp_decode(dev, t):
    # 70B's d:ffn ratio at a quarter of each dim, so the CPU quantiser stays in seconds
    m = Mlp(2048, 7168, t, 16, dev, wtype=tpx.TP_FP8_E4M3)
    y, _ = m.run(residual=False)
    y_ref, _ = m.oracle(residual=False)
    r, _ = check_close(bits(y), y_ref, rel=REL_F_FP8, mx=1.0, what=f"FP8 MLP t={t}")
    assert r <= REL_F, f"FP8 MLP vs dequantised oracle relF {r:.2e} above the bf16 bar"


# ---------------------------------------------------------------- attention sub-block, RMSNorm


def run_proj(d, n_q, n_kv, hd, t, M, dev, seed=0, residual=True, flags=0):
    x, wqkv, wo = inputs.proj_inputs(d, n_q, n_kv, hd, M, seed=seed, device=dev)
    sh = tpx.make_shape(d, n_q=n_q, n_kv=n_kv, hd=hd, t=t)
    q_w, q = tpx.tp_partition_weights(sh, tpx.TP_W_QKV, wqkv)
    o_w, o = tpx.tp_partition_weights(sh, tpx.TP_W_O, wo)
    Q = (n_q + 2 * n_kv) * hd
    y = torch.full_like(x, float("nan"))
    qkv = torch.full((M, Q), float("nan"), dtype=torch.bfloat16, device=dev)
    o_in = torch.full((M, n_q * hd), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_proj_forward(q, q_w, o, o_w, x, x if residual else None, y, qkv, o_in, ws, flags)
    torch.cuda.synchronize()
    y_ref, qkv_ref = O.proj(bits(x), bits(wqkv), bits(wo), n_q, n_kv, hd,
                            residual=bits(x) if residual else None)
    cols = np.concatenate([O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0] for s in range(t)])
    return y, qkv, y_ref, qkv_ref[:, cols]


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_70b_attention_projections_decode(dev, t):
    y, qkv, y_ref, qkv_ref = run_proj(8192, 64, 8, 128, t, 32, dev)
    check_close(bits(qkv), qkv_ref, what=f"70B qkv t={t}")      # q and k columns too
    check_close(bits(y), y_ref, what=f"70B o_proj t={t}")
    y0, _, y0_ref, _ = run_proj(8192, 64, 8, 128, t, 32, dev, residual=False)
    check_close(bits(y0), y0_ref, what=f"70B o_proj no residual t={t}")


def test_proj_small_ragged(dev):
    y, qkv, y_ref, qkv_ref = run_proj(512, 8, 4, 64, 4, 5, dev, seed=3, residual=False)
    check_close(bits(qkv), qkv_ref, what="small qkv")
    check_close(bits(y), y_ref, what="small proj")


@pytest.mark.parametrize("M,d", [(16, 16384), (3, 256), (1, 8192)])
def test_rmsnorm(dev, M, d):
    x = inputs.normal_bf16((M, d), 1.5, 0, 21, dev)
    out = torch.full_like(x, float("nan"))
    tpx.tp_rmsnorm(x, out, 1e-5)
    torch.cuda.synchronize()
    ref = O.rmsnorm(bits(x), 1e-5)
    check_h(bits(out), ref, what="rmsnorm")      # bf16 output: element-relative bar
