"""The allocation-free row-parallel entry point (tp_rowpar_forward_noalloc).

It is for callers that cannot allocate device memory, such as a plugin inside a
framework whose allocator owns the device, or a latency-critical path that cannot take
cudaMalloc's implicit synchronisation.  Its scratch is a static device array inside the
library.  This file is collected last, so a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from megatron_tensor_transformer_gb300 import build
    build.build_library()
    tpx.lib()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _bits(a):
    return a.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("d,ffn,t,M,flags", [
    (4096, 14336, 8, 8, 0),                            # tickets: shards split across CTAs
    (4096, 14336, 8, 64, 0),
    (4096, 14336, 8, 33, tpx.TP_F_UNFUSED_REDUCE),     # partials, then the separate fold
    (256, 1024, 2, 8, 0),
])
def test_noalloc_matches_workspace_entry_point_twice(dev, d, ffn, t, M, flags):
    sh = tpx.make_shape(d, ffn=ffn, t=t)
    wd = inputs.normal_bf16((ffn, d), 0.02, 0, inputs.STREAM_W_DOWN, dev)
    w, desc = tpx.tp_partition_weights(sh, tpx.TP_W_DOWN, wd)
    ws = tpx.new_workspace(sh, M, dev)
    for call in range(2):                               # two calls in a row on the shared array
        a = inputs.normal_bf16((M, ffn), 1.0, call, 31, dev)
        res = inputs.normal_bf16((M, d), 1.0, call, 32, dev)
        y_ref = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
        tpx.tp_rowpar_forward(desc, w, a, res, y_ref, ws, flags)
        y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=dev)
        tpx.tp_rowpar_forward_noalloc(desc, w, a, res, y, flags)
        torch.cuda.synchronize()
        assert O.rel_frobenius(_bits(y), _bits(y_ref)) <= 5e-3
        assert O.max_err_over_rms(_bits(y), _bits(y_ref)) <= 2e-2
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))   # same kernels, same bits


@pytest.mark.parametrize("kind,M", [(tpx.TP_W_O, 16), (tpx.TP_W_DOWN, 16), (tpx.TP_W_DOWN, 5)])
def test_noalloc_e4m3_weights_match_workspace_entry_point_twice(dev, kind, M):
    """e4m3 weights at decode token counts run the TMA-fed kernel, which keeps its work pieces
    in the balancing scratch and its counters in the ticket words of the static array: two calls
    in a row, each bit-equal to the workspace entry point."""
    d, ffn, n_q, n_kv, hd, t = 8192, 28672, 64, 8, 128, 8
    sh = tpx.make_shape(d, ffn=ffn, n_q=n_q, n_kv=n_kv, hd=hd, t=t, wtype=tpx.TP_FP8_E4M3)
    K = ffn if kind == tpx.TP_W_DOWN else n_q * hd
    wt = inputs.normal_bf16((K, d), 0.02, 0, inputs.STREAM_W_DOWN, dev)
    w, desc = tpx.tp_partition_weights(sh, kind, wt)
    del wt
    ws = tpx.new_workspace(sh, M, dev)
    for call in range(2):
        a = inputs.normal_bf16((M, K), 1.0, call, 33, dev)
        res = inputs.normal_bf16((M, d), 1.0, call, 34, dev)
        y_ref = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
        tpx.tp_rowpar_forward(desc, w, a, res, y_ref, ws)
        y = torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=dev)
        tpx.tp_rowpar_forward_noalloc(desc, w, a, res, y)
        assert tpx.tp_sync(timeout_ms=20000) == tpx.TP_OK
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_noalloc_rejects_requests_beyond_its_scratch(dev):
    cap = tpx.tp_noalloc_scratch_capacity()
    assert cap == 32 << 20
    # 405B-shaped o_proj at 64 tokens needs 8 * 64 * 16384 * 4 bytes of partials: 32 MiB + more.
    # Real (small) device buffers stand in for the operands: the call must return before it
    # touches them, and if it ever did not, it would still touch only memory of this process.
    sh = tpx.make_shape(16384, n_q=128, n_kv=8, hd=128, t=8)
    desc = tpx.tp_describe(sh, tpx.TP_W_O)
    buf = torch.zeros(4096, dtype=torch.uint8, device=dev)
    p = ctypes.c_void_p(buf.data_ptr())
    st = tpx.lib().tp_rowpar_forward_noalloc(ctypes.byref(desc), p, p, None, 64, p, 0, None)
    assert st == tpx.TP_ERR_WORKSPACE
    # the quantised-activation path needs scratch this entry point does not hold: refused up front
    sh8 = tpx.make_shape(256, ffn=1024, t=2, wtype=tpx.TP_FP8_E4M3)
    desc8 = tpx.tp_describe(sh8, tpx.TP_W_DOWN)
    st = tpx.lib().tp_rowpar_forward_noalloc(ctypes.byref(desc8), p, p, None, 8, p, tpx.TP_F_FP8_ACT, None)
    assert st == tpx.TP_ERR_UNSUPPORTED
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    assert int(buf.count_nonzero()) == 0
