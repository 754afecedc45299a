"""GPU parity: a many-layer decode step captured as a CUDA graph (attn_decode_graph_*)
against per-call attn_decode and the oracle, including replays after the sequences grow."""
import math

import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs
from tests.gpu_util import check_attention
from tests.test_decode_gpu import oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    eta.build()
    eta.load_library()


def to_cuda(x: inputs.DecodeStepInputs):
    return ([t.cuda() for t in x.q], [t.cuda() for t in x.k_cache], [t.cuda() for t in x.v_cache],
            x.block_table.cuda(), x.seq_lens.cuda())


def eager(qs, ks, vs, bt, sl, scale):
    outs = [eta.attn_decode(qs[l], ks[l], vs[l], bt, sl, scale=scale) for l in range(len(qs))]
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return outs


def check_layers(oracle, x, g, scale, what):
    for l in range(len(x.q)):
        o_ref, lse_ref = oracle_decode(oracle, x.layer(l), scale)
        check_attention(g.out[l], g.lse[l], o_ref, lse_ref, f"{what} layer {l}")


def test_graph_equals_eager_and_oracle(oracle):
    x = inputs.decode_step_inputs(3, 5, 8, 2, 128, 16, len_lo=1, len_hi=1500, seed=11, extra_blocks=3, poison=True)
    scale = 1.0 / math.sqrt(128)
    qs, ks, vs, bt, sl = to_cuda(x)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale)
    assert g.layers == 3
    g.launch()
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    ref = eager(qs, ks, vs, bt, sl, scale)
    for l in range(3):
        assert torch.equal(g.out[l], ref[l][0]), f"layer {l}: graph O differs from attn_decode"
        assert torch.equal(g.lse[l], ref[l][1]), f"layer {l}: graph lse differs from attn_decode"
    check_layers(oracle, x, g, scale, "graph")
    g.close()


@pytest.mark.parametrize("d,Hq,Hkv,bs", [(64, 16, 1, 16), (128, 32, 8, 64), (128, 12, 4, 256)])
def test_graph_shapes(oracle, d, Hq, Hkv, bs):
    x = inputs.decode_step_inputs(2, 4, Hq, Hkv, d, bs, len_lo=1, len_hi=2100, seed=d + Hq + bs, extra_blocks=2,
                                  poison=True)
    scale = 1.0 / math.sqrt(d)
    qs, ks, vs, bt, sl = to_cuda(x)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale)
    g.launch()
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    check_layers(oracle, x, g, scale, f"d={d} G={Hq // Hkv} bs={bs}")
    g.close()


def test_graph_replay_after_sequences_grow(oracle):
    """Capture once; between replays write new queries, grow the lengths (across block
    boundaries, up to the table's capacity) in place: each replay matches the oracle at
    the lengths of that moment."""
    final = [1, 16, 17, 500, 1023, 2048]
    x = inputs.decode_step_inputs(2, len(final), 8, 2, 128, 16, seq_lens=final, seed=12, extra_blocks=1)
    scale = 1.0 / math.sqrt(128)
    qs, ks, vs, bt, sl = to_cuda(x)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale)
    gen = torch.Generator().manual_seed(99)
    for step, delta in enumerate([1, 0]):
        lens = torch.tensor([max(L - delta * (L // 2 + 1), 0) for L in final], dtype=torch.int32)
        if step == 0:
            lens[0] = 0  # an empty sequence on the first step
        qn = [torch.randn(t.shape, generator=gen).to(torch.bfloat16) for t in x.q]
        for l in range(2):
            qs[l].copy_(qn[l])
        sl.copy_(lens)
        g.launch()
        torch.cuda.synchronize()
        assert eta.attn_get_device_error() == 0
        xs = inputs.DecodeStepInputs(q=qn, k_cache=x.k_cache, v_cache=x.v_cache, block_table=x.block_table,
                                     seq_lens=lens, block_size=16)
        check_layers(oracle, xs, g, scale, f"replay {step}")
        if step == 0:
            assert torch.isneginf(g.lse[0][0]).all() and (g.out[0][0] == 0).all()
    g.close()


def test_many_layers_many_replays_are_deterministic():
    x = inputs.decode_step_inputs(12, 3, 8, 2, 128, 16, len_lo=100, len_hi=3000, seed=13)
    qs, ks, vs, bt, sl = to_cuda(x)
    scale = 1.0 / math.sqrt(128)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale)
    ref = eager(qs, ks, vs, bt, sl, scale)
    for _ in range(4):
        g.launch()
    torch.cuda.synchronize()
    for l in range(12):
        assert torch.equal(g.out[l], ref[l][0]) and torch.equal(g.lse[l], ref[l][1])
    g.close()


def test_graph_on_a_side_stream_and_shared_workspace():
    x = inputs.decode_step_inputs(2, 4, 8, 2, 128, 16, len_lo=1, len_hi=900, seed=14)
    qs, ks, vs, bt, sl = to_cuda(x)
    scale = 1.0 / math.sqrt(128)
    ws = torch.empty(eta.attn_decode_workspace_size(4, 8, 2, 128, 16, bt.shape[1]), dtype=torch.uint8, device="cuda")
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale, workspace=ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.launch()
    s.synchronize()
    ref = eager(qs, ks, vs, bt, sl, scale)
    for l in range(2):
        assert torch.equal(g.out[l], ref[l][0])
    g.close()
    with pytest.raises(RuntimeError):
        g.launch()


def test_graph_reports_bad_block_id():
    x = inputs.decode_step_inputs(2, 2, 8, 2, 128, 16, seq_lens=[100, 50], seed=15)
    qs, ks, vs, bt, sl = to_cuda(x)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl)
    bt[0, 2] = ks[0].shape[0] + 5  # inside sequence 0's length; written after capture
    g.launch()
    assert eta.attn_get_device_error() == -7
    assert eta.attn_get_device_error() == 0
    g.close()


def test_full_c8_step_every_layer(oracle):
    """The decode-step workload the bench replays: every layer's output against attn_decode
    bitwise, and every sequence of every layer against the oracle."""
    c = inputs.C8
    x = inputs.decode_step_config_inputs(c)
    qs, ks, vs, bt, sl = to_cuda(x)
    scale = 1.0 / math.sqrt(c.d)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale)
    g.launch()
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    ref = eager(qs, ks, vs, bt, sl, scale)
    for l in range(c.n_layers):
        assert torch.equal(g.out[l], ref[l][0]) and torch.equal(g.lse[l], ref[l][1])
    for l in range(c.n_layers):
        o_ref, lse_ref = oracle_decode(oracle, x.layer(l), scale)
        check_attention(g.out[l], g.lse[l], o_ref, lse_ref, f"C8 layer {l}")
    g.close()


def test_graph_and_per_call_decode_share_a_workspace():
    x = inputs.decode_step_inputs(3, 4, 8, 2, 128, 16, len_lo=1, len_hi=2500, seed=16)
    qs, ks, vs, bt, sl = to_cuda(x)
    scale = 1.0 / math.sqrt(128)
    ws = torch.empty(eta.attn_decode_workspace_size(4, 8, 2, 128, 16, bt.shape[1]), dtype=torch.uint8, device="cuda")
    ref = eager(qs, ks, vs, bt, sl, scale)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=scale, workspace=ws)
    for _ in range(2):
        g.launch()
        o1, lse1 = eta.attn_decode(qs[1], ks[1], vs[1], bt, sl, scale=scale, workspace=ws)
        torch.cuda.synchronize()
        for l in range(3):
            assert torch.equal(g.out[l], ref[l][0]) and torch.equal(g.lse[l], ref[l][1])
        assert torch.equal(o1, ref[1][0])
    g.close()


def test_graph_over_more_sequences_than_one_launch_holds(oracle):
    """2100 sequences: each layer is two chained launches inside the graph."""
    gen = torch.Generator().manual_seed(17)
    lens = torch.randint(0, 70, (2100,), generator=gen).tolist()
    x = inputs.decode_step_inputs(2, 2100, 8, 2, 64, 16, seq_lens=lens, seed=17, extra_blocks=2, poison=True)
    qs, ks, vs, bt, sl = to_cuda(x)
    g = eta.attn_decode_graph_create(qs, ks, vs, bt, sl, scale=0.125)
    g.launch()
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    seqs = [0, 5, 2047, 2048, 2099]
    for l in range(2):
        o_ref, lse_ref = oracle_decode(oracle, x.layer(l), 0.125, seqs=seqs)
        check_attention(g.out[l][seqs], g.lse[l][seqs], o_ref, lse_ref, f"2100 sequences layer {l}")
    g.close()
