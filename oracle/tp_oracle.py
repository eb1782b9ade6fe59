"""CPU oracle for the Megatron tensor-parallel linear layers of a Llama-style block.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline leg may import this module.  The product path never routes through it.

What it computes, in float64, following the pages:
  * Megatron MLP, "Tensor Parallelism (Megatron-Style)" (arunshar.com, ch. 12,
    Y = GeLU(XA)B with A split by columns, B split by rows, Z = sum_k Z_k),
    in Llama's SwiGLU form (one more input matrix, split like the first,
    vidyal.ai model-parallelism, "Step 1: tensor parallelism slices every
    layer"):  y = x + (silu(x Wg) * (x Wu)) Wd.
  * The attention sub-block of "The Tensor-Parallel Shard Group"
    (scalablesystem.dev): QKV column-parallel, local attention over each
    shard's heads, o_proj row-parallel with one sum.
  * The shard layouts (column split = output dim, row split = input dim).
  * FP8 e4m3 per-output-channel weight quantization (the pages' "FP8"
    replica-density mode), per-token activation quantization for the FP8 x FP8
    path, and the bf16 / e4m3 number formats from their bit definitions.
  * The byte and flop accounting the pages print.

Everything is the plain definition: no blocking, fusion or reordering.  The
oracle is *unsharded*: the sharded form is only evaluated by
``sharded_mlp`` to pin the decomposition itself.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, special cases, brute force, printed worked numbers).
"""
import numpy as np

# --------------------------------------------------------------------------
# number formats, from their bit definitions
# --------------------------------------------------------------------------


def _bf16_value(b):
    """Value of one or more bf16 codes from the definition: the upper half of an IEEE binary32,
    1 sign, 8 exponent (bias 127), 7 mantissa bits; exponent 0 is subnormal, 255 inf/NaN."""
    b = np.asarray(b).astype(np.int64)
    sign = (b >> 15) & 1
    e = (b >> 7) & 0xFF
    m = (b & 0x7F).astype(np.float64)
    normal = np.ldexp(1.0 + m / 128.0, (e - 127).astype(np.int32))
    sub = np.ldexp(m / 128.0, -126)
    v = np.where(e == 0, sub, normal)
    v = np.where((e == 255) & (m == 0), np.inf, v)
    v = np.where((e == 255) & (m != 0), np.nan, v)
    return np.where(sign == 1, -v, v)


_BF16_TABLE = _bf16_value(np.arange(65536))   # every code evaluated once from the definition


def bf16_bits_to_f64(bits):
    """bf16 codes (uint16) -> float64 values."""
    return _BF16_TABLE[np.asarray(bits).astype(np.uint16)]


def _round_to_grid(a, mant_bits, emin):
    """Round non-negative finite float64 ``a`` to nearest-even on a binary grid with
    ``mant_bits`` fraction bits and minimum normal exponent ``emin`` (subnormals below).
    Exact: the scaling is by powers of two and np.rint rounds half to even."""
    a = np.asarray(a, dtype=np.float64)
    _, ex = np.frexp(a)              # a = f * 2**ex with f in [0.5, 1)
    e = np.maximum(ex - 1, emin)     # exponent of the leading bit, clamped at the subnormal range
    ulp = np.ldexp(1.0, (e - mant_bits).astype(np.int32))
    return np.rint(a / ulp) * ulp


def f64_to_bf16_bits(v):
    """Round float64 to bf16 (nearest, ties to even), overflow to inf."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    sign = np.signbit(v)
    a = np.abs(v)
    r = _round_to_grid(np.where(np.isfinite(a), a, 0.0), 7, -126)
    r = np.minimum(r, np.ldexp(1.0, 128))          # overflow: mapped to inf below
    big = r >= np.ldexp(1.0, 128)
    f, ex = np.frexp(r)
    e = ex - 1
    normal = r >= np.ldexp(1.0, -126)
    mant_n = np.rint((np.where(normal, r / np.ldexp(1.0, e.astype(np.int32)), 1.0) - 1.0) * 128.0)
    mant_s = np.rint(np.where(normal, 0.0, r) / np.ldexp(1.0, -133))
    bits = np.where(normal, ((e + 127).astype(np.int64) << 7) | mant_n.astype(np.int64),
                    mant_s.astype(np.int64))
    bits = np.where(r == 0, 0, bits)
    bits = np.where(big | np.isinf(a), 0x7F80, bits)
    bits = np.where(np.isnan(v), 0x7FC0, bits)
    out[...] = (bits | (sign.astype(np.int64) << 15)).astype(np.uint16)
    return out


E4M3_MAX = 448.0


def e4m3_bits_to_f64(bits):
    """OCP E4M3 (the 'fn' variant): 1 sign, 4 exponent (bias 7), 3 mantissa; no inf,
    S.1111.111 is NaN, largest finite 1.75 * 2**8 = 448."""
    b = np.asarray(bits).astype(np.uint8)
    sign = (b >> 7) & 1
    e = ((b >> 3) & 0xF).astype(np.int64)
    m = (b & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32))
    sub = np.ldexp(m / 8.0, -6)
    v = np.where(e == 0, sub, normal)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return np.where(sign == 1, -v, v)


def f32_to_e4m3_bits_satfinite(v):
    """Round (binary32) values to E4M3, nearest-even, clamping finite overflow to +-448."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    sign = np.signbit(v)
    a = np.abs(v)
    r = _round_to_grid(np.where(np.isfinite(a), a, 0.0), 3, -6)
    r = np.minimum(r, E4M3_MAX)
    r = np.where(np.isinf(a), E4M3_MAX, r)
    _, ex = np.frexp(r)
    e = ex - 1
    normal = r >= np.ldexp(1.0, -6)
    mant_n = np.rint((np.where(normal, r / np.ldexp(1.0, e.astype(np.int32)), 1.0) - 1.0) * 8.0)
    mant_s = np.rint(np.where(normal, 0.0, r) / np.ldexp(1.0, -9))
    bits = np.where(normal, ((e + 7).astype(np.int64) << 3) | mant_n.astype(np.int64),
                    mant_s.astype(np.int64))
    bits = np.where(r == 0, 0, bits)
    bits = bits | (sign.astype(np.int64) << 7)
    bits = np.where(np.isnan(v), 0x7F, bits)
    return bits.astype(np.uint8)


# --------------------------------------------------------------------------
# the block's math, unsharded, float64
# --------------------------------------------------------------------------


def as_f64(a):
    """Accept float arrays or raw bf16 bit patterns (uint16) and return float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def silu(z):
    """silu(z) = z * sigma(z) = z / (1 + exp(-z)), the Swish gate of Llama's SwiGLU MLP."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def mlp_hidden(x, w_gate, w_up):
    """h = silu(x Wg) * (x Wu): the column-parallel half of the MLP (A = [Wg|Wu] split by
    columns, the nonlinearity applied before any sum).  x [M,d]; Wg, Wu [d,F] ([in,out])."""
    x = as_f64(x)
    return silu(x @ as_f64(w_gate)) * (x @ as_f64(w_up))


def mlp(x, w_gate, w_up, w_down, residual=None):
    """y = residual + (silu(x Wg) * (x Wu)) Wd  (row-parallel half: B = Wd split by rows,
    Z = sum of the shard partials).  Returns (y, h) in float64; residual may be None."""
    h = mlp_hidden(x, w_gate, w_up)
    y = h @ as_f64(w_down)
    if residual is not None:
        y = y + as_f64(residual)
    return y, h


def attention_one_token(qkv, n_q, n_kv, hd):
    """Attention over a context of one token (the query's own k, v): softmax over a single
    score is 1, so each q head returns the v of its kv group.  q head h belongs to kv head
    floor(h / (n_q / n_kv)) (grouped-query attention, 64 q and 8 kv heads for 70B).
    qkv columns: [q heads 0..n_q-1 | k heads 0..n_kv-1 | v heads 0..n_kv-1], hd columns each.
    Returns o_in [M, n_q*hd]."""
    qkv = as_f64(qkv)
    M = qkv.shape[0]
    group = n_q // n_kv
    v0 = (n_q + n_kv) * hd
    out = np.empty((M, n_q * hd), dtype=np.float64)
    for h in range(n_q):
        g = h // group
        out[:, h * hd:(h + 1) * hd] = qkv[:, v0 + g * hd: v0 + (g + 1) * hd]
    return out


def attention_decode(qkv, k_cache, v_cache, lens, n_q, n_kv, hd):
    """Decode attention over a KV cache, one new token per sequence m (grouped-query: q head h
    reads kv head floor(h / (n_q / n_kv))).  The token's own k and v are the cache's entry at
    position lens[m]; it attends over positions 0..lens[m]:
        o[m, h] = sum_j softmax_j(q[m, h] . k[m, g, j] / sqrt(hd)) v[m, g, j].
    qkv: [M, (n_q + 2 n_kv) hd] in the unsharded column order [q | k | v]; k_cache, v_cache:
    [M, n_kv, L, hd] with the new token's k and v already at position lens[m].  Returns o_in
    [M, n_q hd].  A sequence with lens[m] outside [0, L) gets a zero row."""
    qkv = as_f64(qkv)
    k_cache, v_cache = as_f64(k_cache), as_f64(v_cache)
    M = qkv.shape[0]
    group = n_q // n_kv
    L = k_cache.shape[2]
    out = np.zeros((M, n_q * hd))
    for m in range(M):
        n = int(lens[m])
        if n < 0 or n >= L:
            continue
        for h in range(n_q):
            g = h // group
            q = qkv[m, h * hd:(h + 1) * hd]
            sc = k_cache[m, g, :n + 1] @ q / np.sqrt(hd)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            out[m, h * hd:(h + 1) * hd] = p @ v_cache[m, g, :n + 1]
    return out


def append_kv(qkv, k_cache, v_cache, lens, n_q, n_kv, hd):
    """Copies of the caches with the new token's k and v (from qkv) written at position
    lens[m] of every kv head; sequences with lens[m] outside [0, L) are left as they are."""
    qkv = np.asarray(qkv)
    k2, v2 = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    L = k2.shape[2]
    for m in range(qkv.shape[0]):
        n = int(lens[m])
        if n < 0 or n >= L:
            continue
        for g in range(n_kv):
            k2[m, g, n] = qkv[m, (n_q + g) * hd:(n_q + g + 1) * hd]
            v2[m, g, n] = qkv[m, (n_q + n_kv + g) * hd:(n_q + n_kv + g + 1) * hd]
    return k2, v2


def proj(x, w_qkv, w_o, n_q, n_kv, hd, residual=None):
    """Attention sub-block with the one-token attention stand-in:
    qkv = x Wqkv;  o_in = attention(qkv);  y = residual + o_in Wo.  Returns (y, qkv)."""
    qkv = as_f64(x) @ as_f64(w_qkv)
    o_in = attention_one_token(qkv, n_q, n_kv, hd)
    y = o_in @ as_f64(w_o)
    if residual is not None:
        y = y + as_f64(residual)
    return y, qkv


def rmsnorm(x, eps=1e-5, gain=None):
    """a = x / sqrt(mean(x^2) + eps) * g over the hidden dim (gain 1 unless given)."""
    x = as_f64(x)
    a = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    if gain is not None:
        a = a * as_f64(gain)
    return a


def layer(x, w_qkv, w_o, w_gate, w_up, w_down, n_q, n_kv, hd, eps=1e-5, bf16_between_blocks=False):
    """Pre-norm Llama layer restricted to its linear parts:
    h = x + O(attn(QKV(rms(x))));  x' = h + MLP(rms(h)).  float64 throughout; optionally the
    attention block's output h is rounded to bf16 (the activation dtype of the configs) before
    the MLP block reads it."""
    x = as_f64(x)
    hmid, _ = proj(rmsnorm(x, eps), w_qkv, w_o, n_q, n_kv, hd, residual=x)
    if bf16_between_blocks:
        hmid = bf16_bits_to_f64(f64_to_bf16_bits(hmid))
    out, _ = mlp(rmsnorm(hmid, eps), w_gate, w_up, w_down, residual=hmid)
    return out, hmid


# --------------------------------------------------------------------------
# FP8 e4m3 weights, per output channel
# --------------------------------------------------------------------------


def quantize_fp8_per_channel(w):
    """W [in,out] -> (q bits [in,out] uint8, s [out] float32) with W ~ q * s.
    s_n = absmax_k |W[k,n]| / 448 in binary32 (an all-zero column gets s_n = 1);
    q = E4M3_RNE_satfinite(W / s_n), the division in binary32.  Quantisation uses the
    whole, unsharded column, so the codes do not depend on the shard count."""
    w32 = as_f64(w).astype(np.float32)
    amax = np.max(np.abs(w32), axis=0)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = f32_to_e4m3_bits_satfinite(w32 / s[None, :])
    return q, s


def dequantize_fp8(q, s):
    """W_deq[k,n] = e4m3(q[k,n]) * s_n, in float64."""
    return e4m3_bits_to_f64(q) * np.asarray(s, dtype=np.float64)[None, :]


# --------------------------------------------------------------------------
# FP8 x FP8: activations quantised per token as well ("FP8" prefill, vidyal.ai
# model-parallelism, which credits FP8 with up to 50% higher prefill).  The pages give
# no activation scale; the reading here mirrors their weight scheme with one scale
# per token (row) over the whole, unsharded row.
# --------------------------------------------------------------------------


def quantize_fp8_per_token(x):
    """X [M,K] -> (q bits [M,K] uint8, s [M] float32) with X ~ diag(s) q.
    s_m = absmax_k |X[m,k]| / 448 in binary32 (an all-zero row gets s_m = 1);
    q = E4M3_RNE_satfinite(X / s_m), the division in binary32."""
    x32 = as_f64(x).astype(np.float32)
    amax = np.max(np.abs(x32), axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = f32_to_e4m3_bits_satfinite(x32 / s[:, None])
    return q, s


def dequantize_fp8_per_token(q, s):
    """X_deq[m,k] = e4m3(q[m,k]) * s_m, in float64."""
    return e4m3_bits_to_f64(q) * np.asarray(s, dtype=np.float64)[:, None]


def mlp_fp8x(x, w_gate, w_up, w_down, residual=None):
    """The MLP with both GEMM inputs quantised per token (weights as given, normally the
    dequantised per-channel e4m3 weights):
        a = Q(x);  h = bf16(silu(a Wg) * (a Wu));  y = residual + Q(h) Wd
    Q = quantize_fp8_per_token then dequantise.  h is rounded to bf16 first, because the
    quantiser of the row-parallel input sees the stored bf16 activations.  x holds bf16
    values.  Returns (y, h) in float64 (h on the bf16 grid)."""
    a = dequantize_fp8_per_token(*quantize_fp8_per_token(x))
    h = bf16_bits_to_f64(f64_to_bf16_bits(silu(a @ as_f64(w_gate)) * (a @ as_f64(w_up))))
    y = dequantize_fp8_per_token(*quantize_fp8_per_token(h)) @ as_f64(w_down)
    if residual is not None:
        y = y + as_f64(residual)
    return y, h


# --------------------------------------------------------------------------
# shard layouts: column split = output dim, row split = input dim
# ("ColumnParallelLinear" / "RowParallelLinear", scalablesystem.dev, "The
# Tensor-Parallel Shard Group"; A = [A_1|...|A_t], B = [B_1; ...; B_t],
# arunshar.com "Tensor Parallelism (Megatron-Style)").  Each shard is stored
# K-major: one row per output feature, the nn.Linear [out, in] orientation.
# --------------------------------------------------------------------------

GU_BLOCK = 8   # gate/up rows interleave in blocks of this many output features


def colpar_columns(kind, s, t, d=None, ffn=None, n_q=None, n_kv=None, hd=None):
    """Which output column of the unsharded [in,out] weight each packed row of shard s
    holds.  For 'gate_up' also which matrix (0 = gate, 1 = up)."""
    if kind == "gate_up":
        fs = ffn // t
        rows = np.arange(2 * fs)
        blk, j = rows // (2 * GU_BLOCK), rows % (2 * GU_BLOCK)
        col = s * fs + blk * GU_BLOCK + (j % GU_BLOCK)
        which = (j >= GU_BLOCK).astype(np.int64)
        return col, which
    if kind == "qkv":
        nqs, nkvs = n_q // t, n_kv // t
        q = s * nqs * hd + np.arange(nqs * hd)
        k = n_q * hd + s * nkvs * hd + np.arange(nkvs * hd)
        v = (n_q + n_kv) * hd + s * nkvs * hd + np.arange(nkvs * hd)
        col = np.concatenate([q, k, v])
        return col, np.zeros_like(col)
    raise ValueError(kind)


def pack_colpar(w_list, kind, t, **shape):
    """Column-parallel shards: shard s = [rows_s, in] with row r = column col(r) of the
    chosen matrix.  w_list = [Wg, Wu] for gate_up, [Wqkv] for qkv.  Works on any dtype
    (bf16 bits or fp8 codes) since it is a pure permutation."""
    out = []
    for s in range(t):
        col, which = colpar_columns(kind, s, t, **shape)
        shard = np.empty((len(col), w_list[0].shape[0]), dtype=w_list[0].dtype)
        for m, w in enumerate(w_list):
            sel = which == m
            shard[sel] = np.asarray(w)[:, col[sel]].T
        out.append(shard)
    return out


# --------------------------------------------------------------------------
# vocabulary-parallel edges of the model: the lm_head is column-parallel over the
# vocabulary (each shard's logits are a slice of the output, so the "all-gather" is a
# concatenation) and the embedding table is split by vocabulary rows (each shard holds
# the rows of its own id range; a lookup is the sum over shards of "my row, or zeros",
# scalablesystem.dev "The Tensor-Parallel Shard Group", vocab shard).  The vocabulary is
# padded with zero rows to a multiple of 128 per shard.
# --------------------------------------------------------------------------

VOCAB_ALIGN = 128


def vocab_padded(V, t):
    """V rounded up so that every one of the t shards holds a multiple of 128 ids."""
    q = VOCAB_ALIGN * t
    return (V + q - 1) // q * q


def vocab_columns(s, t, V):
    """Vocabulary ids (output columns of the lm_head) of shard s's packed rows; ids >= V are
    padding."""
    vs = vocab_padded(V, t) // t
    return s * vs + np.arange(vs)


def pack_vocab(w, t):
    """lm_head W [d, V] -> t shards [Vs, d]: row r of shard s = column s*Vs + r of W, zero for
    padding ids."""
    w = np.asarray(w)
    d, V = w.shape
    out = []
    for s in range(t):
        ids = vocab_columns(s, t, V)
        shard = np.zeros((len(ids), d), dtype=w.dtype)
        ok = ids < V
        shard[ok] = w[:, ids[ok]].T
        out.append(shard)
    return out


def pack_embed(e, t):
    """Embedding table E [V, d] -> t shards [Vs, d]: row r of shard s = E[s*Vs + r], zero for
    padding ids."""
    e = np.asarray(e)
    V, d = e.shape
    out = []
    for s in range(t):
        ids = vocab_columns(s, t, V)
        shard = np.zeros((len(ids), d), dtype=e.dtype)
        ok = ids < V
        shard[ok] = e[ids[ok]]
        out.append(shard)
    return out


def lm_head(x, w):
    """logits = x W for W [d, V]: the plain product, unsharded."""
    return as_f64(x) @ as_f64(w)


def lm_head_sharded(x, w, t):
    """The same logits evaluated shard by shard from pack_vocab's shards and concatenated in
    shard order (the column-parallel output needs no reduction), cut to the V real ids."""
    x = as_f64(x)
    V = np.asarray(w).shape[1]
    parts = [x @ as_f64(sh).T for sh in pack_vocab(w, t)]
    return np.concatenate(parts, axis=1)[:, :V]


def embed_lookup(ids, e):
    """x[m] = E[ids[m]]; an id outside [0, V) gives a zero row (no shard owns it)."""
    e = as_f64(e)
    ids = np.asarray(ids, dtype=np.int64)
    out = np.zeros((len(ids), e.shape[1]))
    ok = (ids >= 0) & (ids < e.shape[0])
    out[ok] = e[ids[ok]]
    return out


def embed_lookup_sharded(ids, e, t):
    """The vocabulary-parallel form: every shard contributes its row if the id is in its range,
    else zeros, and the contributions are summed in shard order."""
    V = np.asarray(e).shape[0]
    vs = vocab_padded(V, t) // t
    ids = np.asarray(ids, dtype=np.int64)
    acc = np.zeros((len(ids), np.asarray(e).shape[1]))
    for s, sh in enumerate(pack_embed(e, t)):
        local = ids - s * vs
        mine = (local >= 0) & (local < vs) & (ids < V)
        part = np.zeros_like(acc)
        part[mine] = as_f64(sh)[local[mine]]
        acc = acc + part
    return acc


def pack_rowpar(w, t):
    """Row-parallel shards of W [in,out]: shard s = [out, in/t], element [n,k] = W[s*in/t + k, n]."""
    w = np.asarray(w)
    ks = w.shape[0] // t
    return [np.ascontiguousarray(w[s * ks:(s + 1) * ks, :].T) for s in range(t)]


def colpar_scales(s_vec, kind, t, **shape):
    """Per packed row scale of column-parallel FP8 shards: s_{col(r)} (gate or up scale)."""
    out = []
    for s in range(t):
        col, which = colpar_columns(kind, s, t, **shape)
        sv = [np.asarray(v, dtype=np.float32) for v in s_vec]
        out.append(np.array([sv[m][c] for c, m in zip(col, which)], dtype=np.float32))
    return out


def sharded_mlp(x, w_gate, w_up, w_down, t, residual=None):
    """The MLP evaluated shard by shard as the pages decompose it: shard s computes
    Y_s = silu(x Wg_s) * (x Wu_s) from its own columns, Z_s = Y_s Wd_s from its own rows,
    and Z = sum_s Z_s (left to right).  Used only to check the decomposition."""
    x = as_f64(x)
    wg, wu, wd = as_f64(w_gate), as_f64(w_up), as_f64(w_down)
    fs = wg.shape[1] // t
    z = None
    for s in range(t):
        cols = slice(s * fs, (s + 1) * fs)
        ys = silu(x @ wg[:, cols]) * (x @ wu[:, cols])
        zs = ys @ wd[cols, :]
        z = zs if z is None else z + zs
    if residual is not None:
        z = z + as_f64(residual)
    return z


# --------------------------------------------------------------------------
# byte / flop accounting
# --------------------------------------------------------------------------


def layer_linear_params(d, ffn, n_q, n_kv, hd):
    """Parameters of one layer's linear weights: QKV, o_proj, gate, up, down."""
    q = (n_q + 2 * n_kv) * hd
    return d * q + n_q * hd * d + 3 * d * ffn


def decode_bytes_per_shard(d, ffn, n_q, n_kv, hd, n_layers, vocab, t, bytes_per_param):
    """Weight bytes one shard reads per decode step: its 1/t of every layer's linear
    weights plus its 1/t slice of the (untied) embedding and lm_head."""
    per_layer = layer_linear_params(d, ffn, n_q, n_kv, hd) * bytes_per_param / t
    vocab_shard = 2 * vocab * d * bytes_per_param / t
    return n_layers * per_layer + vocab_shard


def allreduce_bytes_per_token(d, bytes_per_elem):
    """One all-reduce sums one hidden-size vector per token."""
    return d * bytes_per_elem


def allreduces_per_token(n_layers, per_layer=2):
    """One per attention block and one per MLP block."""
    return n_layers * per_layer


def forward_flops(n_params, tokens):
    """2 flops (multiply + add) per parameter per token."""
    return 2.0 * n_params * tokens


# --------------------------------------------------------------------------
# error metrics used by the parity tests
# --------------------------------------------------------------------------


def rel_frobenius(y, y_ref):
    y, y_ref = as_f64(y), as_f64(y_ref)
    return float(np.linalg.norm(y - y_ref) / max(np.linalg.norm(y_ref), 1e-300))


def max_err_over_rms(y, y_ref):
    y, y_ref = as_f64(y), as_f64(y_ref)
    rms = np.sqrt(np.mean(y_ref * y_ref))
    return float(np.max(np.abs(y - y_ref)) / max(rms, 1e-300))
