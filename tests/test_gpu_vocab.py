"""The vocabulary-parallel edges through the C ABI: the lm_head (column-parallel over the
vocabulary, padded to 128 ids per shard, the shards' logits concatenated) and the embedding
lookup (table split by vocabulary rows), against the float64 oracle."""
import numpy as np
import pytest
import torch

from megatron_tensor_transformer_gb300 import inputs, tpx
from oracle import tp_oracle as O
from tests.test_gpu_parity import REL_F, bits, check_close

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


def shard_rows(packed, desc, s):
    buf = packed.cpu().numpy()
    st = s * desc.shard_stride_bytes
    return buf[st: st + desc.rows_per_shard * desc.k_per_shard * 2].view(np.uint16).reshape(
        desc.rows_per_shard, desc.k_per_shard)


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_pack_vocab_and_embed_bit_exact(dev, t):
    d, V = 256, 1000
    w = inputs.normal_bf16((d, V), 0.02, 1, 60, dev)
    e = inputs.normal_bf16((V, d), 1.0, 1, 61, dev)
    sh = tpx.make_shape(d, t=t, vocab=V)
    w_p, wd = tpx.tp_partition_weights(sh, tpx.TP_W_VOCAB, w)
    e_p, ed = tpx.tp_partition_weights(sh, tpx.TP_W_EMBED, e)
    assert wd.rows_per_shard == O.vocab_padded(V, t) // t
    ref_w, ref_e = O.pack_vocab(bits(w), t), O.pack_embed(bits(e), t)
    for s in range(t):
        assert np.array_equal(shard_rows(w_p, wd, s), ref_w[s])
        assert np.array_equal(shard_rows(e_p, ed, s), ref_e[s])


@pytest.mark.parametrize("t,M", [(1, 1), (2, 5), (8, 16), (8, 130)])
def test_lm_head_exact_on_integers(dev, t, M):
    """Small-integer inputs: every product and sum is exact in fp32, so the logits equal the
    oracle bit for bit; nothing is written past the real vocabulary."""
    d, V = 512, 3000
    x = inputs.small_int_bf16((M, d), -2, 2, 2, 62, dev)
    w = inputs.small_int_bf16((d, V), -2, 2, 2, 63, dev)
    sh = tpx.make_shape(d, t=t, vocab=V)
    w_p, wd = tpx.tp_partition_weights(sh, tpx.TP_W_VOCAB, w)
    buf = torch.full((M * V + 512,), float("nan"), dtype=torch.float32, device=dev)
    logits = buf[: M * V].view(M, V)
    ws = tpx.new_workspace(sh, M, dev)
    tpx.tp_lm_head_forward(wd, w_p, x, logits, ws=ws)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    ref = O.lm_head(bits(x), bits(w))
    assert np.array_equal(logits.cpu().numpy().astype(np.float64), ref)
    assert torch.isnan(buf[M * V:]).all()                  # canary past the output


def test_lm_head_llama70b_vocab_sampled_columns(dev):
    """Llama-3 70B's output layer: d 8192, 128256 ids over 8 shards (16128 per shard after
    padding), 32 decode tokens; bf16 inputs, fp32 logits, against the oracle on 4096 sampled
    ids (the oracle's product restricted to those columns is the same definition)."""
    d, V, t, M = 8192, 128256, 8, 32
    x = inputs.normal_bf16((M, d), 1.0, 3, 64, dev)
    w = inputs.normal_bf16((d, V), 0.02, 3, 65, dev)
    sh = tpx.make_shape(d, t=t, vocab=V)
    w_p, wd = tpx.tp_partition_weights(sh, tpx.TP_W_VOCAB, w)
    logits = torch.full((M, V), float("nan"), dtype=torch.float32, device=dev)
    tpx.tp_lm_head_forward(wd, w_p, x, logits, ws=tpx.new_workspace(sh, M, dev))
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    assert not torch.isnan(logits).any()
    cols = np.sort(np.random.default_rng(0).choice(V, 4096, replace=False))
    cols[-1] = V - 1                                        # the last real id, next to the padding
    ref = O.lm_head(bits(x), bits(w)[:, cols])
    got = logits[:, torch.from_numpy(cols).to(dev)].cpu().numpy().astype(np.float64)
    assert O.rel_frobenius(got, ref) <= 1e-5                # fp32 accumulate, fp32 output
    # the same logits again, bit for bit
    l2 = torch.empty_like(logits)
    tpx.tp_lm_head_forward(wd, w_p, x, l2)
    assert torch.equal(logits, l2)


@pytest.mark.parametrize("t", [1, 8])
def test_embed_lookup_exact_with_out_of_range_ids(dev, t):
    d, V = 1024, 5000
    e = inputs.normal_bf16((V, d), 1.0, 4, 66, dev)
    sh = tpx.make_shape(d, t=t, vocab=V)
    e_p, ed = tpx.tp_partition_weights(sh, tpx.TP_W_EMBED, e)
    ids_np = np.array([0, 1, 4999, 2500, 637, -1, 5000, 5123, 4096, 127, 128], dtype=np.int32)
    ids = torch.from_numpy(ids_np).to(dev)
    x = torch.full((len(ids_np), d), float("nan"), dtype=torch.bfloat16, device=dev)
    tpx.tp_embed_lookup(ed, e_p, ids, x)
    assert tpx.tp_sync(timeout_ms=10000) == tpx.TP_OK
    ref = O.embed_lookup(ids_np, bits(e))
    assert np.array_equal(O.as_f64(bits(x)), ref)
