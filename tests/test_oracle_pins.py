"""Pins for the CPU oracle: each check ties it to something other than itself
(a library's independent routine for the number formats, closed forms, printed
numbers from the pages, brute force on tiny inputs, special cases)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import tp_oracle as O


def _load(d, name):
    with open(os.path.join(d, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- formats


def test_bf16_decode_all_patterns_match_float32_upper_half():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = O.bf16_bits_to_f64(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decode_named_values():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0x3F00: 0.5, 0x4049: 3.140625,
             0x0080: 2.0 ** -126, 0x0001: 2.0 ** -133, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127}
    for b, v in cases.items():
        assert O.bf16_bits_to_f64(np.array([b], dtype=np.uint16))[0] == v


def test_bf16_encode_matches_torch_cast_on_float32_values():
    g = torch.Generator().manual_seed(5)
    v = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 20)
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16_bits(v.numpy().astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_encode_ties_to_even():
    one = 1.0
    assert O.f64_to_bf16_bits(np.array([one + 2 ** -8]))[0] == 0x3F80          # tie -> even (1.0)
    assert O.f64_to_bf16_bits(np.array([one + 3 * 2 ** -8]))[0] == 0x3F82      # tie -> even (1 + 2^-6)
    assert O.f64_to_bf16_bits(np.array([one + 2 ** -8 + 2 ** -30]))[0] == 0x3F81  # above tie


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_bits_to_f64(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin]) and np.array_equal(np.isnan(got), np.isnan(ref))
    assert O.e4m3_bits_to_f64(np.array([0x7E], dtype=np.uint8))[0] == 448.0
    assert O.e4m3_bits_to_f64(np.array([0x01], dtype=np.uint8))[0] == 2.0 ** -9
    assert O.e4m3_bits_to_f64(np.array([0x38], dtype=np.uint8))[0] == 1.0


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    g = torch.Generator().manual_seed(6)
    v = (torch.rand(200000, generator=g) * 2 - 1) * 448
    v = torch.cat([v, v * 1e-3, v * 1e-5, torch.tensor([0.0, -0.0, 448.0, -448.0])])
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.f32_to_e4m3_bits_satfinite(v.numpy())
    assert np.array_equal(got, ref)
    sat = O.f32_to_e4m3_bits_satfinite(np.array([460.0, 1000.0, -1e30, np.inf], dtype=np.float32))
    assert list(sat) == [0x7E, 0x7E, 0xFE, 0x7E]


# ---------------------------------------------------------------- SwiGLU MLP


def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(50.0) - 50.0) < 1e-15
    assert abs(O.silu(-50.0)) < 1e-18
    z = np.linspace(-20, 20, 401)
    # z*s(z) - (-z)*s(-z) = z*(s(z) + s(-z)) = z
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=0, atol=1e-13)
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16


def test_mlp_hand_example(golden_dir):
    g = _load(golden_dir, "mlp_hand_example.json")
    y, h = O.mlp(np.array(g["x"]), np.array(g["w_gate"]), np.array(g["w_up"]),
                 np.array(g["w_down"]), residual=np.array(g["x"]))
    assert np.allclose(h, g["h"], atol=g["abs_tol"], rtol=0)
    assert np.allclose(y, g["y"], atol=g["abs_tol"], rtol=0)


def _brute_mlp(x, wg, wu, wd, res):
    M, d = x.shape
    F = wg.shape[1]
    y = np.zeros((M, wd.shape[1]))
    for m in range(M):
        h = []
        for j in range(F):
            g = sum(x[m, k] * wg[k, j] for k in range(d))
            u = sum(x[m, k] * wu[k, j] for k in range(d))
            h.append(g / (1 + math.exp(-g)) * u)
        for n in range(wd.shape[1]):
            y[m, n] = res[m, n] + sum(h[j] * wd[j, n] for j in range(F))
    return y


def test_mlp_brute_force_non_square():
    rng = np.random.default_rng(1)
    M, d, F = 3, 5, 7
    x, wg, wu = rng.normal(size=(M, d)), rng.normal(size=(d, F)), rng.normal(size=(d, F))
    wd = rng.normal(size=(F, d))
    y, _ = O.mlp(x, wg, wu, wd, residual=x)
    assert np.allclose(y, _brute_mlp(x, wg, wu, wd, x), rtol=1e-12, atol=1e-12)


def test_mlp_special_cases():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(4, 16))
    wg, wu, wd = rng.normal(size=(16, 32)), rng.normal(size=(16, 32)), rng.normal(size=(32, 16))
    y, _ = O.mlp(x, wg, np.zeros_like(wu), wd, residual=x)
    assert np.array_equal(y, x)                       # up = 0 -> h = 0
    y, _ = O.mlp(x, np.zeros_like(wg), wu, wd, residual=x)
    assert np.array_equal(y, x)                       # silu(0) = 0
    y1, _ = O.mlp(x, wg, wu, wd)
    y2, _ = O.mlp(x, wg, wu, 2 * wd)
    assert np.allclose(y2, 2 * y1, rtol=1e-13, atol=1e-13)   # linear in the row-parallel matrix


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sharded_equals_unsharded(t):
    """Column split of A and row split of B, summed over shards, is the unsharded MLP."""
    rng = np.random.default_rng(3)
    x = rng.normal(size=(5, 24))
    wg, wu, wd = rng.normal(size=(24, 64)), rng.normal(size=(24, 64)), rng.normal(size=(64, 24))
    y, _ = O.mlp(x, wg, wu, wd, residual=x)
    assert np.allclose(O.sharded_mlp(x, wg, wu, wd, t, residual=x), y, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- attention sub-block


def test_attention_one_token_groups():
    # n_q 4, n_kv 2, hd 1: q heads 0,1 -> kv 0; q heads 2,3 -> kv 1
    qkv = np.array([[1, 2, 3, 4, 5, 6, 10, 20]], dtype=np.float64)
    assert list(O.attention_one_token(qkv, 4, 2, 1)[0]) == [10, 10, 20, 20]


@pytest.mark.parametrize("t", [1, 2, 4])
def test_proj_sharded_heads_equal_unsharded(t):
    """QKV column shards give each shard whole heads (its q heads and their kv heads);
    local attention then row-parallel o_proj, summed over shards, is the unsharded block."""
    rng = np.random.default_rng(4)
    d, n_q, n_kv, hd, M = 32, 8, 4, 4, 3
    x = rng.normal(size=(M, d))
    wqkv = rng.normal(size=(d, (n_q + 2 * n_kv) * hd))
    wo = rng.normal(size=(n_q * hd, d))
    y, qkv = O.proj(x, wqkv, wo, n_q, n_kv, hd, residual=x)
    qkv_sh = O.pack_colpar([wqkv], "qkv", t, n_q=n_q, n_kv=n_kv, hd=hd)
    o_sh = O.pack_rowpar(wo, t)
    z = x.copy()
    for s in range(t):
        q_s = x @ qkv_sh[s].T                          # [M, Q_s]: [q heads | k heads | v heads] of shard s
        o_in_s = O.attention_one_token(q_s, n_q // t, n_kv // t, hd)
        z = z + o_in_s @ o_sh[s].T
    assert np.allclose(z, y, rtol=1e-12, atol=1e-12)


def test_rmsnorm_closed_forms():
    x = np.array([[3.0, 4.0]])
    eps = 1e-5
    assert np.allclose(O.rmsnorm(x, eps), x / math.sqrt(12.5 + eps), rtol=1e-15)
    c = np.full((1, 64), -2.0)
    assert np.allclose(O.rmsnorm(c, eps), -2.0 / math.sqrt(4.0 + eps), rtol=1e-15)
    assert np.array_equal(O.rmsnorm(np.zeros((1, 8)), eps), np.zeros((1, 8)))


# ---------------------------------------------------------------- shard layouts


def test_gate_up_pack_layout_by_hand():
    d, ffn, t = 2, 32, 2
    wg = np.arange(d * ffn).reshape(d, ffn).astype(np.int64)
    wu = 1000 + wg
    sh = O.pack_colpar([wg, wu], "gate_up", t, ffn=ffn)
    assert [a.shape for a in sh] == [(32, 2), (32, 2)]
    # shard 0: gate 0-7, up 0-7, gate 8-15, up 8-15; shard 1 the same from column 16
    expect0 = list(range(0, 8)) + [1000 + c for c in range(0, 8)] + list(range(8, 16)) + \
        [1000 + c for c in range(8, 16)]
    assert list(sh[0][:, 0]) == expect0
    assert list(sh[1][:, 0]) == [v + 16 for v in expect0]
    assert list(sh[1][:, 1]) == [v + 16 + ffn for v in expect0]   # row k=1 of W is +ffn


def test_qkv_pack_layout_by_hand():
    d, n_q, n_kv, hd, t = 1, 4, 2, 2, 2
    w = np.arange((n_q + 2 * n_kv) * hd).reshape(1, -1)   # column index == value
    sh = O.pack_colpar([w], "qkv", t, n_q=n_q, n_kv=n_kv, hd=hd)
    # q heads {0,1} (cols 0-3), k head 0 (cols 8-9), v head 0 (cols 12-13)
    assert list(sh[0][:, 0]) == [0, 1, 2, 3, 8, 9, 12, 13]
    assert list(sh[1][:, 0]) == [4, 5, 6, 7, 10, 11, 14, 15]


def test_rowpar_pack_layout_and_bytes():
    w = np.arange(8 * 3).reshape(8, 3)                     # [in=8, out=3]
    sh = O.pack_rowpar(w, 4)
    assert sh[1].shape == (3, 2) and list(sh[1][0]) == [w[2, 0], w[3, 0]]
    assert sum(a.size for a in sh) == w.size              # per-shard bytes are 1/t of the total


def test_per_shard_bytes_are_one_over_t():
    for t in (1, 2, 4, 8):
        wg = np.zeros((64, 128), dtype=np.uint16)
        sh = O.pack_colpar([wg, wg], "gate_up", t, ffn=128)
        assert all(a.size * t == 2 * wg.size for a in sh)


# ---------------------------------------------------------------- FP8 weights


def test_fp8_quantizer_properties():
    rng = np.random.default_rng(7)
    w = (rng.normal(size=(64, 40)) * 0.02).astype(np.float32)
    w[:, 3] = 0.0
    q, s = O.quantize_fp8_per_channel(w)
    assert s[3] == 1.0 and np.all(q[:, 3] == 0)
    deq = O.dequantize_fp8(q, s)
    # each column's absmax lands on +-448 (code 0x7E / 0xFE)
    amax_rows = np.argmax(np.abs(w), axis=0)
    for n in range(40):
        if n != 3:
            assert q[amax_rows[n], n] & 0x7F == 0x7E
    # round to nearest with 3 mantissa bits: error <= 2^-4 relative, or half a subnormal step
    err = np.abs(deq - w.astype(np.float64))
    bound = np.maximum(np.abs(w) * 2.0 ** -4, s[None, :].astype(np.float64) * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)


def test_fp8_exact_values_round_trip():
    # a column whose entries are e4m3 values times a power of two scale round-trips exactly
    vals = np.array([448, 1, -0.5, 0.015625, 2 ** -9, 96, -448, 0], dtype=np.float32)
    w = np.stack([vals * 2.0 ** -10, vals], axis=1).astype(np.float32)
    q, s = O.quantize_fp8_per_channel(w)
    assert np.array_equal(O.dequantize_fp8(q, s), w.astype(np.float64))


def test_colpar_scales_layout_by_hand():
    """Packed-row scales of column-parallel FP8 shards, listed by hand.  Gate scales are
    100 + n and up scales 200 + n, so a swap of gate and up, or of two 8-feature blocks,
    changes the list.  ffn = 32, t = 2: each shard owns 16 features, packed as
    [8 gate | 8 up | 8 gate | 8 up]."""
    s_gate = np.arange(32, dtype=np.float32) + 100
    s_up = np.arange(32, dtype=np.float32) + 200
    got = O.colpar_scales([s_gate, s_up], "gate_up", 2, ffn=32)
    want0 = list(range(100, 108)) + list(range(200, 208)) + list(range(108, 116)) + list(range(208, 216))
    want1 = list(range(116, 124)) + list(range(216, 224)) + list(range(124, 132)) + list(range(224, 232))
    assert [list(map(int, g)) for g in got] == [want0, want1]
    assert all(g.dtype == np.float32 for g in got)
    # QKV: 4 q heads, 2 kv heads of 2 columns (q 0..7, k 8..11, v 12..15), t = 2, scale 10 + column:
    # shard 0 holds q heads 0,1, k head 0, v head 0; shard 1 the rest
    sq = np.arange(16, dtype=np.float32) + 10
    got = O.colpar_scales([sq], "qkv", 2, n_q=4, n_kv=2, hd=2)
    assert [list(map(int, g)) for g in got] == [[10, 11, 12, 13, 18, 19, 22, 23],
                                                [14, 15, 16, 17, 20, 21, 24, 25]]


# The FP8 quantisers divide in IEEE binary32.  A hand case where that differs from a float64
# divide: a column (or row) [a, w] with a = 43 * 2^-12 = 0.010498046875 and w = 3a/4 =
# 0.00787353515625, both bf16 values.  s = binary32(a / 448) lies just below a / 448 (43/1835008
# is not a binary32 value), so the exact quotient w / s is a little above 336 = 448 * 3/4, while
# the binary32 quotient rounds to 336.0 exactly.  336 is the midpoint between the e4m3 values
# 320 (1.010b * 2^8, code 0x7A) and 352 (1.011b * 2^8, code 0x7B): ties go to the even mantissa,
# 320, whereas the float64 quotient rounds up to 352.
_DIV_A, _DIV_W = 43 * 2.0 ** -12, 0.75 * 43 * 2.0 ** -12


def test_fp8_division_is_binary32_by_hand():
    from fractions import Fraction
    s = np.float32(np.float32(_DIV_A) / np.float32(448.0))
    assert Fraction(float(s)) < Fraction(43, 1835008)                 # s rounded down
    assert Fraction(_DIV_W) / Fraction(float(s)) > 336                 # exact quotient above the tie
    assert np.float32(_DIV_W) / s == np.float32(336.0)                 # binary32 quotient on the tie
    col = np.array([[_DIV_A], [_DIV_W]], dtype=np.float32)
    q, sc = O.quantize_fp8_per_channel(col)
    assert sc[0] == s and list(q[:, 0]) == [0x7E, 0x7A]
    q, sc = O.quantize_fp8_per_token(col.T)
    assert sc[0] == s and list(q[0, :]) == [0x7E, 0x7A]
    # the same pair with the sign flipped: codes 0xFE, 0xFA
    q, _ = O.quantize_fp8_per_channel(-col)
    assert list(q[:, 0]) == [0xFE, 0xFA]


# ---------------------------------------------------------------- accounting printed on the pages


def test_accounting_matches_printed_numbers(golden_dir):
    g = _load(golden_dir, "accounting.json")
    m70, m405 = g["models"]["llama31_70b"], g["models"]["llama31_405b"]

    def full_params(m):
        lin = O.layer_linear_params(m["d"], m["ffn"], m["n_q"], m["n_kv"], m["hd"])
        return m["n_layers"] * lin + 2 * m["vocab"] * m["d"]

    shp = {k: m70[k] for k in ("d", "ffn", "n_q", "n_kv", "hd")}
    got = {
        "decode_bytes_per_gpu_70b_tp8_bf16": O.decode_bytes_per_shard(
            **shp, n_layers=m70["n_layers"], vocab=m70["vocab"], t=8, bytes_per_param=2),
        "weights_70b_bf16_unsharded": full_params(m70) * 2,
        "allreduce_bytes_per_token_70b_bf16": O.allreduce_bytes_per_token(m70["d"], 2),
        "allreduces_per_token_70b": O.allreduces_per_token(m70["n_layers"]),
        "reduced_bytes_per_token_70b": O.allreduces_per_token(m70["n_layers"]) *
        O.allreduce_bytes_per_token(m70["d"], 2),
        "prefill_flops_70b_4096": O.forward_flops(full_params(m70), 4096),
        "weights_405b_bf16": full_params(m405) * 2,
        "weights_405b_fp8": full_params(m405) * 1,
        "weights_per_gpu_405b_fp8_tp8": full_params(m405) * 1 / 8,
    }
    for e in g["printed"]:
        v = got[e["name"]]
        assert abs(v - e["value"]) <= e["rel_tol"] * e["value"] + 1e-9, (e["name"], v, e["value"])


def test_metrics():
    y = np.array([[3.0, 4.0]])
    assert O.rel_frobenius(y, y) == 0.0
    assert abs(O.rel_frobenius(y * 1.01, y) - 0.01) < 1e-12
    assert abs(O.max_err_over_rms(y + np.array([[0.0, 0.5]]), y) - 0.5 / math.sqrt(12.5)) < 1e-12


# ---------------------------------------------------------------- the pre-norm layer


def _layer_weights(rng, d=32, ffn=64, n_q=4, n_kv=2, hd=8):
    q = (n_q + 2 * n_kv) * hd
    return (rng.normal(size=(d, q)) * 0.2, rng.normal(size=(n_q * hd, d)) * 0.2, rng.normal(size=(d, ffn)) * 0.2,
            rng.normal(size=(d, ffn)) * 0.2, rng.normal(size=(ffn, d)) * 0.2)


def test_layer_reduces_to_its_blocks():
    rng = np.random.default_rng(12)
    d = 32
    x = O.bf16_bits_to_f64(O.f64_to_bf16_bits(rng.normal(size=(3, d))))   # bf16-valued input
    wqkv, wo, wg, wu, wd = _layer_weights(rng)
    # attention output projection zero: h = x exactly, layer = x + MLP(rms(x))
    y, h = O.layer(x, wqkv, np.zeros_like(wo), wg, wu, wd, 4, 2, 8)
    assert np.array_equal(h, x)
    m, _ = O.mlp(O.rmsnorm(x), wg, wu, wd, residual=x)
    assert np.allclose(y, m, rtol=1e-13, atol=1e-13)
    # MLP down projection zero: the layer is the (bf16-stored) attention block
    y, h = O.layer(x, wqkv, wo, wg, wu, np.zeros_like(wd), 4, 2, 8, bf16_between_blocks=True)
    p, _ = O.proj(O.rmsnorm(x), wqkv, wo, 4, 2, 8, residual=x)
    assert np.array_equal(y, O.bf16_bits_to_f64(O.f64_to_bf16_bits(p)))
    # by default the layer is the two blocks composed in float64
    y, _ = O.layer(x, wqkv, wo, wg, wu, wd, 4, 2, 8)
    m, _ = O.mlp(O.rmsnorm(p), wg, wu, wd, residual=p)
    assert np.allclose(y, m, rtol=1e-13, atol=1e-13)



# ---------------------------------------------------------------- vocabulary-parallel edges

def test_vocab_padding_matches_the_shard_alignment():
    # Llama 3's 128256 ids over 8 shards: 16032 each is not a multiple of 128, so each shard
    # is padded to 16128 (126 x 128); with t = 1 the 128256 ids need 1002 x 128 = 128256
    assert O.vocab_padded(128256, 8) == 129024 and O.vocab_padded(128256, 8) // 8 == 16128
    assert O.vocab_padded(128256, 1) == 128256
    assert O.vocab_padded(1000, 4) == 1024 and O.vocab_padded(1024, 8) == 1024


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_lm_head_sharded_concatenation_equals_unsharded(t):
    rng = np.random.default_rng(t)
    d, V, M = 24, 1000, 3            # 1000 ids: the last shard carries padding
    x = rng.integers(-3, 4, size=(M, d)).astype(np.float64)
    w = rng.integers(-3, 4, size=(d, V)).astype(np.float64)
    np.testing.assert_array_equal(O.lm_head_sharded(x, w, t), O.lm_head(x, w))


def test_lm_head_brute_force_and_pack_layout():
    rng = np.random.default_rng(7)
    d, V, M, t = 5, 300, 2, 2
    x = rng.normal(size=(M, d))
    w = rng.normal(size=(d, V))
    ref = np.array([[sum(x[m, k] * w[k, v] for k in range(d)) for v in range(V)] for m in range(M)])
    np.testing.assert_allclose(O.lm_head(x, w), ref, rtol=1e-12, atol=1e-12)
    shards = O.pack_vocab(w, t)       # Vp = 512: 256 ids per shard, ids 300..511 padding
    assert [sh.shape for sh in shards] == [(256, d), (256, d)]
    np.testing.assert_array_equal(shards[0][7], w[:, 7])
    np.testing.assert_array_equal(shards[1][0], w[:, 256])
    np.testing.assert_array_equal(shards[1][43], w[:, 299])
    assert not shards[1][44:].any()


def test_embedding_lookup_by_hand_and_vocab_parallel_sum():
    V, d, t = 10, 3, 2                # Vp = 256: shard 0 owns ids 0..127, shard 1 only padding
    e = np.arange(V * d, dtype=np.float64).reshape(V, d)
    ids = [3, 0, 9, 12, -1]
    got = O.embed_lookup(ids, e)
    np.testing.assert_array_equal(got[0], [9, 10, 11])
    np.testing.assert_array_equal(got[1], [0, 1, 2])
    np.testing.assert_array_equal(got[2], [27, 28, 29])
    assert not got[3].any() and not got[4].any()          # ids no shard owns: zero rows
    for tt in (1, 2, 4, 8):
        np.testing.assert_array_equal(O.embed_lookup_sharded(ids, e, tt), got)
    shards = O.pack_embed(e, 2)
    np.testing.assert_array_equal(shards[0][:V], e)
    assert not shards[0][V:].any() and not shards[1].any()


# ---------------------------------------------------------------- decode attention over a KV cache

def _attn_case(M=3, n_q=4, n_kv=2, hd=8, L=6, seed=0):
    rng = np.random.default_rng(seed)
    qkv = rng.normal(size=(M, (n_q + 2 * n_kv) * hd))
    kc = rng.normal(size=(M, n_kv, L, hd))
    vc = rng.normal(size=(M, n_kv, L, hd))
    return qkv, kc, vc


def test_attention_with_empty_history_is_the_one_token_stand_in():
    """lens = 0: the only position is the token itself, softmax over one score is 1, so every
    q head returns its group's v: the one-token attention stand-in."""
    n_q, n_kv, hd = 4, 2, 8
    qkv, kc, vc = _attn_case(n_q=n_q, n_kv=n_kv, hd=hd)
    lens = [0, 0, 0]
    k2, v2 = O.append_kv(qkv, kc, vc, lens, n_q, n_kv, hd)
    np.testing.assert_allclose(O.attention_decode(qkv, k2, v2, lens, n_q, n_kv, hd),
                               O.attention_one_token(qkv, n_q, n_kv, hd), rtol=0, atol=1e-15)


def test_attention_equal_keys_average_the_values():
    """All keys equal: every score is the same, softmax is uniform, o is the mean of v."""
    n_q, n_kv, hd = 2, 1, 4
    qkv, kc, vc = _attn_case(M=1, n_q=n_q, n_kv=n_kv, hd=hd, L=5)
    kc[:] = 0.5
    qkv[0, n_q * hd:(n_q + 1) * hd] = 0.5          # the new token's k, equal too
    lens = [3]
    k2, v2 = O.append_kv(qkv, kc, vc, lens, n_q, n_kv, hd)
    o = O.attention_decode(qkv, k2, v2, lens, n_q, n_kv, hd)
    mean_v = v2[0, 0, :4].mean(axis=0)
    np.testing.assert_allclose(o[0, :hd], mean_v, rtol=1e-13)
    np.testing.assert_allclose(o[0, hd:], mean_v, rtol=1e-13)


def test_attention_brute_force_and_out_of_range_lengths():
    n_q, n_kv, hd, L = 4, 2, 3, 5
    qkv, kc, vc = _attn_case(M=3, n_q=n_q, n_kv=n_kv, hd=hd, L=L, seed=3)
    lens = [2, 4, 5]                                # the last is out of range: a zero row
    k2, v2 = O.append_kv(qkv, kc, vc, lens, n_q, n_kv, hd)
    o = O.attention_decode(qkv, k2, v2, lens, n_q, n_kv, hd)
    assert not o[2].any()
    np.testing.assert_array_equal(k2[2], kc[2])     # nothing appended out of range
    for m in range(2):
        for h in range(n_q):
            g = h // (n_q // n_kv)
            q = [qkv[m, h * hd + i] for i in range(hd)]
            sc = [sum(q[i] * k2[m, g, j, i] for i in range(hd)) / hd ** 0.5 for j in range(lens[m] + 1)]
            e = [np.exp(v - max(sc)) for v in sc]
            ref = [sum(e[j] * v2[m, g, j, i] for j in range(lens[m] + 1)) / sum(e) for i in range(hd)]
            np.testing.assert_allclose(o[m, h * hd:(h + 1) * hd], ref, rtol=1e-12)
    # the appended entries are the token's k and v
    np.testing.assert_array_equal(k2[1, 1, 4], qkv[1, (n_q + 1) * hd:(n_q + 2) * hd])
    np.testing.assert_array_equal(v2[0, 0, 2], qkv[0, (n_q + n_kv) * hd:(n_q + n_kv + 1) * hd])


@pytest.mark.parametrize("t", [1, 2])
def test_attention_head_sharded_equals_unsharded(t):
    """Each shard attends with its own q heads over its own kv heads (whole GQA groups): the
    per-shard outputs, placed at their heads, are the unsharded output."""
    n_q, n_kv, hd = 4, 2, 8
    qkv, kc, vc = _attn_case(n_q=n_q, n_kv=n_kv, hd=hd, seed=5)
    lens = [1, 3, 5]
    k2, v2 = O.append_kv(qkv, kc, vc, lens, n_q, n_kv, hd)
    full = O.attention_decode(qkv, k2, v2, lens, n_q, n_kv, hd)
    nqs, nkvs = n_q // t, n_kv // t
    for s in range(t):
        cols = O.colpar_columns("qkv", s, t, n_q=n_q, n_kv=n_kv, hd=hd)[0]
        qkv_s = qkv[:, cols]
        o_s = O.attention_decode(qkv_s, k2[:, s * nkvs:(s + 1) * nkvs], v2[:, s * nkvs:(s + 1) * nkvs], lens,
                                 nqs, nkvs, hd)
        np.testing.assert_allclose(o_s, full[:, s * nqs * hd:(s + 1) * nqs * hd], rtol=0, atol=0)


# ---------------------------------------------------------------- FP8 x FP8: per-token activations


def test_fp8_per_token_quantizer_properties():
    rng = np.random.default_rng(11)
    x = (rng.normal(size=(40, 64)) * 3.0).astype(np.float32)
    x[5, :] = 0.0
    q, s = O.quantize_fp8_per_token(x)
    assert s[5] == 1.0 and np.all(q[5] == 0)
    amax_cols = np.argmax(np.abs(x), axis=1)
    for m in range(40):
        if m != 5:
            assert q[m, amax_cols[m]] & 0x7F == 0x7E          # each row's absmax lands on +-448
    deq = O.dequantize_fp8_per_token(q, s)
    err = np.abs(deq - x.astype(np.float64))
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s[:, None].astype(np.float64) * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)
    # rows are independent: scaling one row leaves the others' codes alone
    x2 = x.copy()
    x2[0] *= 1000.0
    q2, _ = O.quantize_fp8_per_token(x2)
    assert np.array_equal(q2[1:], q[1:])


def test_fp8_per_token_is_the_per_channel_quantizer_of_the_transpose():
    rng = np.random.default_rng(12)
    x = (rng.normal(size=(17, 33)) * 0.7).astype(np.float32)
    q, s = O.quantize_fp8_per_token(x)
    qt, st = O.quantize_fp8_per_channel(x.T)
    assert np.array_equal(q, qt.T) and np.array_equal(s, st)


def test_fp8_per_token_exact_values_round_trip():
    vals = np.array([448, 1, -0.5, 0.015625, 2 ** -9, 96, -448, 0], dtype=np.float32)
    x = np.stack([vals * 2.0 ** -10, vals, vals * 2.0 ** 6], axis=0).astype(np.float32)
    q, s = O.quantize_fp8_per_token(x)
    assert np.array_equal(O.dequantize_fp8_per_token(q, s), x.astype(np.float64))


def _quant_row_loops(row):
    """Per-token quantisation of one row with plain loops (binary32 as numpy scalars)."""
    amax = np.float32(0.0)
    for v in row:
        amax = max(amax, abs(np.float32(v)))
    s = amax / np.float32(448.0) if amax > 0 else np.float32(1.0)
    return [O.e4m3_bits_to_f64(O.f32_to_e4m3_bits_satfinite(np.array([np.float32(v) / s], dtype=np.float32)))[0]
            * float(s) for v in row]


def test_mlp_fp8x_brute_force_and_special_cases():
    rng = np.random.default_rng(13)
    M, d, F = 3, 8, 6
    x = O.bf16_bits_to_f64(O.f64_to_bf16_bits(rng.normal(size=(M, d))))
    wg, wu, wd = (rng.normal(size=sh) * 0.5 for sh in ((d, F), (d, F), (F, d)))
    y, h = O.mlp_fp8x(x, wg, wu, wd, residual=x)
    for m in range(M):
        a = _quant_row_loops(x[m])
        hm = []
        for f in range(F):
            g = sum(a[k] * wg[k, f] for k in range(d))
            u = sum(a[k] * wu[k, f] for k in range(d))
            hm.append(float(O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.array([g / (1 + np.exp(-g)) * u])))[0]))
        assert np.allclose(h[m], hm, rtol=0, atol=0)
        hq = _quant_row_loops(np.array(hm))
        for n in range(d):
            ref = sum(hq[f] * wd[f, n] for f in range(F)) + x[m, n]
            assert abs(y[m, n] - ref) <= 1e-12 * (1 + abs(ref))
    # rows already on a power-of-two-scaled e4m3 grid quantise exactly: the column-parallel half
    # then equals the plain MLP's, rounded to bf16
    xe = np.array([[448, 1, -0.5, 96, 0, 2 ** -9, -448, 0.015625]], dtype=np.float64) * 2.0 ** -6
    _, h1 = O.mlp_fp8x(xe, wg, wu, wd)
    _, h0 = O.mlp(xe, wg, wu, wd)
    assert np.array_equal(h1, O.bf16_bits_to_f64(O.f64_to_bf16_bits(h0)))
