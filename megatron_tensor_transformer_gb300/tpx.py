"""Thin ctypes binding of libtpx.so (include/tpx.h), same names as the C ABI.

Argument marshalling only: torch tensors supply device memory and streams, every
step of the computation runs in the library's CUDA kernels.  Loading fails loudly
if the library has not been built: there is no fallback path.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtpx.so")

TP_OK, TP_ERR_INVALID_ARG, TP_ERR_SHAPE, TP_ERR_ALIGN, TP_ERR_LAYOUT_MISMATCH = 0, 1, 2, 3, 4
TP_ERR_WORKSPACE, TP_ERR_CUDA, TP_ERR_TIMEOUT, TP_ERR_DEVICE_TIMEOUT, TP_ERR_UNSUPPORTED = 5, 6, 7, 8, 9
TP_BF16, TP_FP8_E4M3 = 0, 1
TP_W_GATE_UP, TP_W_DOWN, TP_W_QKV, TP_W_O, TP_W_VOCAB, TP_W_EMBED = 0, 1, 2, 3, 4, 5
TP_F_UNFUSED_REDUCE, TP_F_FP32_COLPAR_OUT = 0x1, 0x2
TP_F_KERNEL_SKINNY, TP_F_KERNEL_TC, TP_F_SERIAL, TP_F_SPLIT_BLOCK = 0x10, 0x20, 0x40, 0x80
TP_F_FP8_ACT = 0x200
TP_F_FP8_HILO = 0x400
TP_F_FOLD_NORM = 0x800

EXPORTS = ["tp_packed_bytes", "tp_describe", "tp_partition_weights", "tp_workspace_bytes",
           "tp_mlp_forward", "tp_proj_forward", "tp_reduce_partials", "tp_colpar_forward",
           "tp_rowpar_partials", "tp_rowpar_forward", "tp_rowpar_forward_noalloc",
           "tp_noalloc_scratch_capacity", "tp_rmsnorm", "tp_selftest_bounded_wait",
           "tp_layer_scratch_bytes", "tp_layer_forward", "tp_selftest_e4m3_decode", "tp_sync", "tp_status_str", "tp_launch_count",
           "tp_lm_head_forward", "tp_embed_lookup", "tp_attn_workspace_bytes", "tp_attn_decode",
           "tp_attn_block_workspace_bytes", "tp_attn_block_forward", "tp_quantize_fp8_per_token"]


class TpxError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


class Shape(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("ffn", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("t", ctypes.c_int32),
                ("wtype", ctypes.c_int32), ("vocab", ctypes.c_int32)]


class PackedDesc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("layout_version", ctypes.c_uint32),
                ("kind", ctypes.c_int32), ("wtype", ctypes.c_int32), ("shape", Shape),
                ("rows_per_shard", ctypes.c_int64), ("k_per_shard", ctypes.c_int64),
                ("shard_payload_bytes", ctypes.c_uint64), ("scales_offset", ctypes.c_uint64),
                ("shard_stride_bytes", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64)]


_lib = None


def lib():
    """Load libtpx.so once; raise if it is missing (no CPU or eager fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, V, I32, U32, SZ = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
        sig = {
            "tp_packed_bytes": (SZ, [P(Shape), I32]),
            "tp_describe": (I32, [P(Shape), I32, P(PackedDesc)]),
            "tp_partition_weights": (I32, [P(Shape), I32, V, V, V, SZ, P(PackedDesc), V]),
            "tp_workspace_bytes": (SZ, [P(Shape), I32, U32]),
            "tp_mlp_forward": (I32, [P(PackedDesc), V, P(PackedDesc), V, V, V, I32, V, V, V, SZ, U32, V]),
            "tp_proj_forward": (I32, [P(PackedDesc), V, P(PackedDesc), V, V, V, I32, V, V, V, V, SZ, U32, V]),
            "tp_reduce_partials": (I32, [V, I32, I32, I32, V, V, V]),
            "tp_colpar_forward": (I32, [P(PackedDesc), V, V, I32, V, V, SZ, U32, V]),
            "tp_rowpar_partials": (I32, [P(PackedDesc), V, V, I32, V, V]),
            "tp_rowpar_forward": (I32, [P(PackedDesc), V, V, V, I32, V, V, SZ, U32, V]),
            "tp_rowpar_forward_noalloc": (I32, [P(PackedDesc), V, V, V, I32, V, U32, V]),
            "tp_noalloc_scratch_capacity": (SZ, []),
            "tp_rmsnorm": (I32, [V, V, ctypes.c_float, I32, I32, V, V]),
            "tp_sync": (I32, [V, I32]),
            "tp_selftest_bounded_wait": (I32, [I32, V]),
            "tp_layer_scratch_bytes": (SZ, [P(Shape), I32]),
            "tp_selftest_e4m3_decode": (I32, [V, V, I32, V]),
            "tp_layer_forward": (I32, [P(PackedDesc), V, P(PackedDesc), V, P(PackedDesc), V, P(PackedDesc), V,
                                       V, I32, V, ctypes.c_float, V, SZ, V, SZ, U32, V]),
            "tp_status_str": (ctypes.c_char_p, [I32]),
            "tp_lm_head_forward": (I32, [P(PackedDesc), V, V, I32, V, V, SZ, U32, V]),
            "tp_embed_lookup": (I32, [P(PackedDesc), V, V, I32, V, V]),
            "tp_attn_workspace_bytes": (SZ, [P(Shape), I32, I32]),
            "tp_attn_decode": (I32, [P(Shape), V, V, V, I32, V, I32, V, V, SZ, V]),
            "tp_attn_block_workspace_bytes": (SZ, [P(Shape), I32, I32, U32]),
            "tp_quantize_fp8_per_token": (I32, [V, I32, I32, V, V, V]),
            "tp_attn_block_forward": (I32, [P(PackedDesc), V, P(PackedDesc), V, V, V, I32, V, V, I32, V, V, V, V,
                                            V, SZ, U32, V]),
            "tp_launch_count": (ctypes.c_uint64, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def status_str(s):
    return lib().tp_status_str(int(s)).decode()


def _check(st, where):
    if st != TP_OK:
        raise TpxError(st, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        if not torch.cuda.is_available():
            return ctypes.c_void_p(None)
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_shape(d, ffn=0, n_q=0, n_kv=0, hd=0, t=1, wtype=TP_BF16, vocab=0):
    return Shape(d, ffn, n_q, n_kv, hd, t, wtype, vocab)


def tp_packed_bytes(shape, kind):
    return lib().tp_packed_bytes(ctypes.byref(shape), kind)


def tp_describe(shape, kind):
    d = PackedDesc()
    _check(lib().tp_describe(ctypes.byref(shape), kind, ctypes.byref(d)), "tp_describe")
    return d


def tp_workspace_bytes(shape, M, flags=0):
    return lib().tp_workspace_bytes(ctypes.byref(shape), M, flags)


def tp_partition_weights(shape, kind, W0, W1=None, stream=None, packed=None):
    """Returns (packed uint8 device tensor, PackedDesc)."""
    n = tp_packed_bytes(shape, kind)
    if n == 0:
        tp_describe(shape, kind)  # raises with the precise status
    if packed is None:
        packed = torch.empty(n, dtype=torch.uint8, device=W0.device)
    d = PackedDesc()
    _check(lib().tp_partition_weights(ctypes.byref(shape), kind, _ptr(W0), _ptr(W1), _ptr(packed),
                                      packed.numel(), ctypes.byref(d), _stream(stream)),
           "tp_partition_weights")
    return packed, d


def new_workspace(shape, M, device, flags=0):
    """Zero-filled workspace (the ticket counters must start at zero)."""
    return torch.zeros(max(1, tp_workspace_bytes(shape, M, flags)), dtype=torch.uint8, device=device)


def tp_mlp_forward(gu, gu_w, dn, dn_w, x, residual, y, h, ws, flags=0, stream=None):
    M = x.shape[0]
    _check(lib().tp_mlp_forward(ctypes.byref(gu), _ptr(gu_w), ctypes.byref(dn), _ptr(dn_w), _ptr(x),
                                _ptr(residual), M, _ptr(y), _ptr(h), _ptr(ws),
                                0 if ws is None else ws.numel(), flags, _stream(stream)),
           "tp_mlp_forward")
    return y


def tp_proj_forward(qkv, qkv_w, o, o_w, x, residual, y, qkv_out, o_in, ws, flags=0, stream=None):
    M = x.shape[0]
    _check(lib().tp_proj_forward(ctypes.byref(qkv), _ptr(qkv_w), ctypes.byref(o), _ptr(o_w), _ptr(x),
                                 _ptr(residual), M, _ptr(y), _ptr(qkv_out), _ptr(o_in), _ptr(ws),
                                 0 if ws is None else ws.numel(), flags, _stream(stream)),
           "tp_proj_forward")
    return y


def tp_reduce_partials(partials, t, M, d, residual, y, stream=None):
    _check(lib().tp_reduce_partials(_ptr(partials), t, M, d, _ptr(residual), _ptr(y), _stream(stream)),
           "tp_reduce_partials")
    return y


def tp_colpar_forward(desc, w, x, out, flags=0, stream=None, ws=None):
    _check(lib().tp_colpar_forward(ctypes.byref(desc), _ptr(w), _ptr(x), x.shape[0], _ptr(out), _ptr(ws),
                                   0 if ws is None else ws.numel(), flags, _stream(stream)), "tp_colpar_forward")
    return out


def tp_rowpar_partials(desc, w, a, partials, stream=None):
    _check(lib().tp_rowpar_partials(ctypes.byref(desc), _ptr(w), _ptr(a), a.shape[0], _ptr(partials),
                                    _stream(stream)), "tp_rowpar_partials")
    return partials


def tp_rowpar_forward(desc, w, a, residual, y, ws, flags=0, stream=None):
    _check(lib().tp_rowpar_forward(ctypes.byref(desc), _ptr(w), _ptr(a), _ptr(residual), a.shape[0], _ptr(y),
                                   _ptr(ws), 0 if ws is None else ws.numel(), flags, _stream(stream)),
           "tp_rowpar_forward")
    return y


def tp_rowpar_forward_noalloc(desc, w, a, residual, y, flags=0, stream=None):
    """tp_rowpar_forward without a workspace argument: for callers that cannot allocate
    device memory (the library's own static scratch array is used)."""
    _check(lib().tp_rowpar_forward_noalloc(ctypes.byref(desc), _ptr(w), _ptr(a), _ptr(residual), a.shape[0],
                                           _ptr(y), flags, _stream(stream)), "tp_rowpar_forward_noalloc")
    return y


def tp_noalloc_scratch_capacity():
    return lib().tp_noalloc_scratch_capacity()


def tp_rmsnorm(x, out, eps=1e-5, gain=None, stream=None):
    _check(lib().tp_rmsnorm(_ptr(x), _ptr(gain), eps, x.shape[0], x.shape[1], _ptr(out), _stream(stream)),
           "tp_rmsnorm")
    return out


def tp_sync(stream=None, timeout_ms=2000):
    return lib().tp_sync(_stream(stream), timeout_ms)


def tp_selftest_bounded_wait(timeout_us, stream=None):
    _check(lib().tp_selftest_bounded_wait(timeout_us, _stream(stream)), "tp_selftest_bounded_wait")


def tp_layer_scratch_bytes(shape, M):
    return lib().tp_layer_scratch_bytes(ctypes.byref(shape), M)


def tp_layer_forward(qkv, qkv_w, o, o_w, gu, gu_w, dn, dn_w, x, y, scratch, ws, eps=1e-5, flags=0, stream=None):
    _check(lib().tp_layer_forward(ctypes.byref(qkv), _ptr(qkv_w), ctypes.byref(o), _ptr(o_w), ctypes.byref(gu),
                                  _ptr(gu_w), ctypes.byref(dn), _ptr(dn_w), _ptr(x), x.shape[0], _ptr(y), eps,
                                  _ptr(scratch), scratch.numel(), _ptr(ws), ws.numel(), flags, _stream(stream)),
           "tp_layer_forward")
    return y


def tp_selftest_e4m3_decode(codes, out, stream=None):
    _check(lib().tp_selftest_e4m3_decode(_ptr(codes), _ptr(out), codes.numel(), _stream(stream)),
           "tp_selftest_e4m3_decode")
    return out


def tp_launch_count():
    return lib().tp_launch_count()


def tp_lm_head_forward(desc, w, x, logits, ws=None, flags=0, stream=None):
    _check(lib().tp_lm_head_forward(ctypes.byref(desc), _ptr(w), _ptr(x), x.shape[0], _ptr(logits), _ptr(ws),
                                    0 if ws is None else ws.numel(), flags, _stream(stream)), "tp_lm_head_forward")
    return logits


def tp_embed_lookup(desc, w, ids, x, stream=None):
    _check(lib().tp_embed_lookup(ctypes.byref(desc), _ptr(w), _ptr(ids), ids.shape[0], _ptr(x), _stream(stream)),
           "tp_embed_lookup")
    return x


def tp_attn_block_workspace_bytes(shape, M, L, flags=0):
    return lib().tp_attn_block_workspace_bytes(ctypes.byref(shape), M, L, flags)


def new_attn_block_workspace(shape, M, L, device, flags=0):
    """Zero-filled workspace of tp_attn_block_forward (its projection counters start at zero)."""
    return torch.zeros(max(1, tp_attn_block_workspace_bytes(shape, M, L, flags)), dtype=torch.uint8, device=device)


def tp_attn_block_forward(qkv, qkv_w, o, o_w, x, residual, k_cache, v_cache, lens, y, qkv_out, o_in, ws, flags=0,
                          stream=None):
    """k_cache, v_cache: [t, M, n_kv/t, L, hd] bf16; lens: [M] int32 on the device."""
    L = k_cache.shape[3]
    _check(lib().tp_attn_block_forward(ctypes.byref(qkv), _ptr(qkv_w), ctypes.byref(o), _ptr(o_w), _ptr(x),
                                       _ptr(residual), x.shape[0], _ptr(k_cache), _ptr(v_cache), L, _ptr(lens),
                                       _ptr(y), _ptr(qkv_out), _ptr(o_in), _ptr(ws), ws.numel(), flags,
                                       _stream(stream)), "tp_attn_block_forward")
    return y


def tp_quantize_fp8_per_token(x, q, s, stream=None):
    """x: [M, K] bf16; q: [M, K] uint8 codes; s: [M] fp32 (all on the device)."""
    _check(lib().tp_quantize_fp8_per_token(_ptr(x), x.shape[0], x.shape[1], _ptr(q), _ptr(s), _stream(stream)),
           "tp_quantize_fp8_per_token")
    return q, s


def tp_attn_workspace_bytes(shape, M, L):
    return lib().tp_attn_workspace_bytes(ctypes.byref(shape), M, L)


def tp_attn_decode(shape, qkv, k_cache, v_cache, lens, o_in, ws, stream=None):
    """k_cache, v_cache: [t, M, n_kv/t, L, hd] bf16; lens: [M] int32 on the device."""
    L = k_cache.shape[3]
    _check(lib().tp_attn_decode(ctypes.byref(shape), _ptr(qkv), _ptr(k_cache), _ptr(v_cache), L, _ptr(lens),
                                qkv.shape[0], _ptr(o_in), _ptr(ws), ws.numel(), _stream(stream)), "tp_attn_decode")
    return o_in

