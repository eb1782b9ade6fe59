"""Host-side checks of the C ABI: the library loads, exports every declared entry point,
describes packed layouts, and rejects bad arguments before touching the device.  None of
these calls launches a kernel, so they run without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from megatron_tensor_transformer_gb300 import tpx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tpx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", tpx.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(tpx.lib(), n)
    assert sorted(tpx.EXPORTS) == names


def test_describe_8b_gate_up_and_down():
    sh = tpx.make_shape(4096, ffn=14336, t=8)
    gu = tpx.tp_describe(sh, tpx.TP_W_GATE_UP)
    assert (gu.rows_per_shard, gu.k_per_shard) == (2 * 1792, 4096)
    assert gu.shard_payload_bytes == 2 * 1792 * 4096 * 2
    assert gu.shard_payload_bytes * 8 == 2 * 4096 * 14336 * 2      # 1/t of the gate+up bytes
    dn = tpx.tp_describe(sh, tpx.TP_W_DOWN)
    assert (dn.rows_per_shard, dn.k_per_shard) == (4096, 1792)
    assert tpx.tp_packed_bytes(sh, tpx.TP_W_DOWN) == dn.total_bytes == 8 * dn.shard_stride_bytes


def test_describe_70b_qkv_o_and_fp8_scales():
    sh = tpx.make_shape(8192, n_q=64, n_kv=8, hd=128, t=8, wtype=tpx.TP_FP8_E4M3)
    q = tpx.tp_describe(sh, tpx.TP_W_QKV)
    assert (q.rows_per_shard, q.k_per_shard) == (1280, 8192)         # 8 q + 1 k + 1 v heads
    assert q.shard_payload_bytes == 1280 * 8192
    assert q.scales_offset % 256 == 0 and q.shard_stride_bytes >= q.scales_offset + 1280 * 4
    o = tpx.tp_describe(sh, tpx.TP_W_O)
    assert (o.rows_per_shard, o.k_per_shard) == (8192, 1024)


@pytest.mark.parametrize("kw,status", [
    (dict(d=4096, ffn=14336, t=3), tpx.TP_ERR_SHAPE),
    (dict(d=4096, ffn=14337, t=1), tpx.TP_ERR_ALIGN),               # F_s odd
    (dict(d=4096, ffn=14336 + 4, t=8), tpx.TP_ERR_SHAPE),           # t does not divide ffn
    (dict(d=4100, ffn=14336, t=8), tpx.TP_ERR_ALIGN),
    (dict(d=4096, ffn=8 * 12, t=8), tpx.TP_ERR_ALIGN),               # F_s = 12, not a multiple of 8
])
def test_bad_mlp_shapes(kw, status):
    sh = tpx.make_shape(**kw)
    with pytest.raises(tpx.TpxError) as e:
        tpx.tp_describe(sh, tpx.TP_W_GATE_UP)
    assert e.value.status == status
    assert tpx.tp_packed_bytes(sh, tpx.TP_W_GATE_UP) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(d=8192, n_q=64, n_kv=8, hd=128, t=16), tpx.TP_ERR_SHAPE),  # t must be 1,2,4,8
    (dict(d=8192, n_q=64, n_kv=2, hd=128, t=4), tpx.TP_ERR_SHAPE),   # t > n_kv: replication unsupported
    (dict(d=8192, n_q=60, n_kv=8, hd=128, t=8), tpx.TP_ERR_SHAPE),   # n_kv does not divide n_q
    (dict(d=8192, n_q=64, n_kv=8, hd=100, t=8), tpx.TP_ERR_ALIGN),
])
def test_bad_head_splits(kw, status):
    with pytest.raises(tpx.TpxError) as e:
        tpx.tp_describe(tpx.make_shape(**kw), tpx.TP_W_QKV)
    assert e.value.status == status


FAKE = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: every call below fails its checks first


def _call_mlp(gu, dn, M=8, flags=0, ws=FAKE, ws_bytes=1 << 30):
    L = tpx.lib()
    return L.tp_mlp_forward(ctypes.byref(gu), FAKE, ctypes.byref(dn), FAKE, FAKE, None, M, FAKE, FAKE,
                            ws, ws_bytes, flags, None)


def test_wrong_shard_layout_is_rejected():
    """A packed buffer for another t (the believable but wrong output of loading the
    wrong shard, scalablesystem.dev 'The Checkpoint Loader') must not run."""
    gu = tpx.tp_describe(tpx.make_shape(4096, ffn=14336, t=8), tpx.TP_W_GATE_UP)
    dn4 = tpx.tp_describe(tpx.make_shape(4096, ffn=14336, t=4), tpx.TP_W_DOWN)
    assert _call_mlp(gu, dn4) == tpx.TP_ERR_LAYOUT_MISMATCH
    dn8 = tpx.tp_describe(tpx.make_shape(4096, ffn=14336, t=8), tpx.TP_W_DOWN)
    assert _call_mlp(dn8, dn8) == tpx.TP_ERR_LAYOUT_MISMATCH          # kind swapped
    bad = tpx.tp_describe(tpx.make_shape(4096, ffn=14336, t=8), tpx.TP_W_GATE_UP)
    bad.shard_stride_bytes += 256                                       # tampered geometry
    assert _call_mlp(bad, dn8) == tpx.TP_ERR_LAYOUT_MISMATCH
    bad = tpx.tp_describe(tpx.make_shape(4096, ffn=14336, t=8), tpx.TP_W_GATE_UP)
    bad.magic = 0
    assert _call_mlp(bad, dn8) == tpx.TP_ERR_LAYOUT_MISMATCH


def test_argument_errors_before_launch():
    sh = tpx.make_shape(4096, ffn=14336, t=8)
    gu, dn = tpx.tp_describe(sh, tpx.TP_W_GATE_UP), tpx.tp_describe(sh, tpx.TP_W_DOWN)
    assert _call_mlp(gu, dn, M=-1) == tpx.TP_ERR_INVALID_ARG
    assert _call_mlp(gu, dn, flags=0x100) == tpx.TP_ERR_INVALID_ARG              # unknown flag bit
    assert _call_mlp(gu, dn, flags=0x1000) == tpx.TP_ERR_INVALID_ARG
    # the hi/lo e4m3 block flag is a block flag: accepted (the call goes on to the workspace
    # check), alone or with the widening flag
    for fl in (tpx.TP_F_FP8_HILO, tpx.TP_F_FP8_HILO | tpx.TP_F_KERNEL_TC):
        assert _call_mlp(gu, dn, flags=fl, ws=None, ws_bytes=0) == tpx.TP_ERR_WORKSPACE
    assert _call_mlp(gu, dn, ws=None, ws_bytes=0) == tpx.TP_ERR_WORKSPACE
    need = tpx.tp_workspace_bytes(sh, 8)
    assert _call_mlp(gu, dn, ws_bytes=need - 1) == tpx.TP_ERR_WORKSPACE
    L = tpx.lib()
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert L.tp_mlp_forward(ctypes.byref(gu), FAKE, ctypes.byref(dn), FAKE, odd, None, 8, FAKE, FAKE,
                            FAKE, 1 << 30, 0, None) == tpx.TP_ERR_ALIGN
    assert L.tp_reduce_partials(FAKE, 3, 4, 64, None, FAKE, None) == tpx.TP_ERR_SHAPE
    assert L.tp_reduce_partials(FAKE, 2, 4, 60, None, FAKE, None) == tpx.TP_ERR_ALIGN
    assert L.tp_rmsnorm(FAKE, None, ctypes.c_float(1e-5), -1, 64, FAKE, None) == tpx.TP_ERR_INVALID_ARG
    # M == 0 is a valid empty call that enqueues nothing
    assert _call_mlp(gu, dn, M=0) == tpx.TP_OK


def test_status_strings():
    for s in range(10):
        assert tpx.status_str(s).startswith("TP_")


def test_attention_arguments_before_launch():
    """Decode attention: workspace size from its definition (fp32 partials per 128-position chunk
    and one counter per sequence and kv head), and the refusals that need no device."""
    L_ = tpx.lib()
    sh = tpx.make_shape(8192, n_q=64, n_kv=8, hd=128, t=8)
    M, L, G = 32, 4096, 8
    assert tpx.tp_attn_workspace_bytes(sh, M, L) == M * 8 * (L // 128) * G * (128 + 2) * 4 + M * 8 * 4
    assert tpx.tp_attn_workspace_bytes(sh, 3, 130) == 3 * 8 * 2 * G * 130 * 4 + 3 * 8 * 4   # ragged chunk

    def call(shape, M=4, L=256, ws_bytes=1 << 30, p=FAKE):
        return L_.tp_attn_decode(ctypes.byref(shape), p, p, p, L, p, M, p, p, ws_bytes, None)

    assert call(sh, M=-1) == tpx.TP_ERR_INVALID_ARG
    assert call(sh, L=0) == tpx.TP_ERR_INVALID_ARG
    assert call(tpx.make_shape(2176, n_q=34, n_kv=2, hd=64, t=2)) == tpx.TP_ERR_UNSUPPORTED   # 17 q per kv
    assert call(tpx.make_shape(1536, n_q=16, n_kv=4, hd=96, t=2)) == tpx.TP_ERR_UNSUPPORTED   # head dim 96
    assert call(sh, M=1 << 16, L=1 << 12) == tpx.TP_ERR_UNSUPPORTED                           # 2^31 cache rows
    assert call(sh, ws_bytes=tpx.tp_attn_workspace_bytes(sh, 4, 256) - 1) == tpx.TP_ERR_WORKSPACE
    assert call(sh, p=ctypes.c_void_p((1 << 20) + 8)) == tpx.TP_ERR_ALIGN
    assert call(sh, M=0) == tpx.TP_OK


def test_attention_block_arguments_before_launch():
    """The one-call attention block: its workspace is the projections' (aligned) then the
    attention's; shape, workspace and flag refusals need no device."""
    L_ = tpx.lib()
    sh = tpx.make_shape(8192, n_q=64, n_kv=8, hd=128, t=8)
    M, L = 32, 4096
    proj = tpx.tp_workspace_bytes(sh, M)
    need = -(-proj // 256) * 256 + tpx.tp_attn_workspace_bytes(sh, M, L)
    assert tpx.tp_attn_block_workspace_bytes(sh, M, L) == need
    q, o = tpx.tp_describe(sh, tpx.TP_W_QKV), tpx.tp_describe(sh, tpx.TP_W_O)

    def call(qd=q, od=o, M=4, L=256, ws_bytes=1 << 32, flags=0, p=FAKE):
        return L_.tp_attn_block_forward(ctypes.byref(qd), FAKE, ctypes.byref(od), FAKE, p, None, M, p, p, L, p,
                                        p, p, p, p, ws_bytes, flags, None)

    assert call(M=-1) == tpx.TP_ERR_INVALID_ARG
    assert call(L=0) == tpx.TP_ERR_INVALID_ARG
    assert call(flags=0x100) == tpx.TP_ERR_INVALID_ARG
    assert call(ws_bytes=tpx.tp_attn_block_workspace_bytes(sh, 4, 256) - 1) == tpx.TP_ERR_WORKSPACE
    assert call(p=ctypes.c_void_p((1 << 20) + 8)) == tpx.TP_ERR_ALIGN
    assert call(od=q) == tpx.TP_ERR_LAYOUT_MISMATCH                       # O slot given a QKV descriptor
    o4 = tpx.tp_describe(tpx.make_shape(8192, n_q=64, n_kv=8, hd=128, t=4), tpx.TP_W_O)
    assert call(od=o4) == tpx.TP_ERR_LAYOUT_MISMATCH                      # the two halves of different blocks
    sh17 = tpx.make_shape(2176, n_q=34, n_kv=2, hd=64, t=2)
    assert call(qd=tpx.tp_describe(sh17, tpx.TP_W_QKV), od=tpx.tp_describe(sh17, tpx.TP_W_O)) == \
        tpx.TP_ERR_UNSUPPORTED                                            # 17 q heads per kv head
    assert call(M=0) == tpx.TP_OK
