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


def test_noalloc_rejects_requests_beyond_its_scratch(dev):
    cap = tpx.tp_noalloc_scratch_capacity()
    assert cap == 32 << 20
    # 405B-shaped o_proj at 64 tokens needs 8 * 64 * 16384 * 4 bytes of partials: 32 MiB + more
    sh = tpx.make_shape(16384, n_q=128, n_kv=8, hd=128, t=8)
    desc = tpx.tp_describe(sh, tpx.TP_W_O)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check fails first
    st = tpx.lib().tp_rowpar_forward_noalloc(ctypes.byref(desc), fake, fake, None, 64, fake, 0, None)
    assert st == tpx.TP_ERR_WORKSPACE
