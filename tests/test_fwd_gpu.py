"""GPU parity: attn_fwd (prefill) through the C ABI against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs
from tests.gpu_util import check_attention, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    eta.build()
    eta.load_library()


def run_fwd(q, k, v, causal, window, scale=None):
    o, lse = eta.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return o, lse


def case(oracle, B, Hq, Hkv, Nq, Nk, d, causal, window, seed=0, boost=0.0, what=""):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed, k_boost_frac=boost)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, causal, window)
    o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), scale, causal, window)
    return check_attention(o, lse, o_ref, lse_ref, what)


def test_c1_single_head_noncausal(oracle):
    c = inputs.C1
    case(oracle, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.causal, c.window, what=c.name)


SWEEP_N = [1, 63, 64, 65, 127, 128, 129, 255, 257, 1000]
SWEEP_MASKS = [(False, -1), (True, -1), (True, 0), (True, 1), (True, 127), (True, 128), (True, 129), (False, 129)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", SWEEP_N)
@pytest.mark.parametrize("causal,window", SWEEP_MASKS)
def test_boundary_sweep(oracle, N, d, causal, window):
    case(oracle, 1, 2, 1, N, N, d, causal, window, seed=N + d, what=f"N={N} d={d} c={causal} w={window}")


# Grids of at most half the SMs run one query tile per block; with 160 heads the same
# ragged shapes keep two tiles per block (row tiles 2r, 2r + 1 of a head, or two heads of a
# kv head), so both launch forms see every boundary case.
@pytest.mark.parametrize("N", [1, 65, 129, 257, 1000])
@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 129), (False, 129)])
def test_boundary_sweep_paired_blocks(oracle, N, causal, window):
    case(oracle, 1, 160, 160, N, N, 128, causal, window, seed=N + 7, what=f"160 heads N={N} c={causal} w={window}")


@pytest.mark.parametrize("Nq,Nk", [(300, 100), (1000, 300), (300, 1000)])
def test_rectangular_many_heads(oracle, Nq, Nk):
    """Bottom-right causal alignment over many blocks: with Nq > Nk the leading rows see no
    key and must come out as O = 0, lse = -inf."""
    case(oracle, 1, 160, 160, Nq, Nk, 128, True, -1, seed=Nq + 3 * Nk, what=f"160 heads {Nq}x{Nk}")


@pytest.mark.parametrize("Hq,Hkv", [(96, 32), (128, 32), (256, 64), (192, 64)])
def test_gqa_paired_blocks(oracle, Hq, Hkv):
    case(oracle, 1, Hq, Hkv, 300, 300, 128, True, -1, seed=Hq + Hkv, what=f"GQA {Hq}/{Hkv} paired blocks")


@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 100), (1, 1000), (129, 1), (200, 257)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular(oracle, Nq, Nk, causal):
    case(oracle, 2, 2, 2, Nq, Nk, 128, causal, -1, seed=Nq * 7 + Nk, what=f"{Nq}x{Nk} c={causal}")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 2), (8, 2), (8, 1), (3, 1)])
def test_gqa_mapping(oracle, Hq, Hkv):
    case(oracle, 2, Hq, Hkv, 300, 300, 128, True, -1, seed=Hq * 10 + Hkv, what=f"GQA {Hq}/{Hkv}")
    case(oracle, 1, Hq, Hkv, 200, 200, 64, False, 50, seed=Hq * 11 + Hkv, what=f"GQA window {Hq}/{Hkv}")


def test_reduced_workload_shapes(oracle):
    # the shapes of the four prefill workloads at sizes the oracle finishes quickly
    case(oracle, 2, 4, 4, 640, 640, 128, True, -1, seed=2, what="C2-like")
    case(oracle, 1, 4, 4, 1000, 1000, 128, True, -1, seed=3, boost=0.01, what="C3-like (boosted keys)")
    case(oracle, 2, 8, 2, 777, 777, 128, True, 200, seed=4, what="C4-like (GQA + window)")


def test_late_maximum_every_tile(oracle):
    """Scores rise along the keys so the running max moves on every key tile."""
    B, H, N, d = 1, 2, 1024, 128
    q = torch.zeros(B, H, N, d)
    q[..., 0] = 1.0
    k = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(5)) * 0.1
    k[..., 0] = torch.linspace(0.0, 60.0 * math.sqrt(d), N)  # scaled score grows to 60
    v = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(6))
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, causal, -1)
        o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), 1 / math.sqrt(d), causal, -1)
        check_attention(o, lse, o_ref, lse_ref, f"late max causal={causal}")


def test_large_logit_range(oracle):
    """Logits near +-200: exp overflows unless the running max is subtracted."""
    B, H, N, d = 1, 2, 384, 64
    g = torch.Generator().manual_seed(7)
    q = (torch.randn(B, H, N, d, generator=g) * 6).bfloat16()
    k = (torch.randn(B, H, N, d, generator=g) * 6).bfloat16()
    v = torch.randn(B, H, N, d, generator=g).bfloat16()
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, causal, -1)
        o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), 1 / math.sqrt(d), causal, -1)
        assert np.abs(lse_ref).max() > 100
        check_attention(o, lse, o_ref, lse_ref, f"large logits causal={causal}")


def test_rows_without_keys(oracle):
    # Nq > Nk with bottom-right causal alignment: the first Nq - Nk rows see nothing
    case(oracle, 1, 2, 2, 300, 100, 128, True, -1, seed=8, what="Nq>Nk causal")
    q, k, v = inputs.prefill_inputs(1, 2, 2, 70, 0, 64, seed=9)
    o, lse = eta.attn_fwd(q.cuda(), torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda"),
                          torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_no_reads_past_inputs_no_writes_past_outputs(oracle):
    """K/V are followed by NaN in memory and outputs are framed by canaries: the
    ragged tail tile must neither read the NaNs nor touch the canaries."""
    B, Hq, Hkv, N, d = 1, 4, 2, 333, 128
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, N, N, d, seed=10)
    pad = 4096

    def framed(t):
        flat = torch.full((t.numel() + 2 * pad,), float("nan"), dtype=t.dtype, device="cuda")
        flat[pad:pad + t.numel()] = t.reshape(-1).cuda()
        return flat, flat[pad:pad + t.numel()].view(t.shape)

    _, qd = framed(q)
    _, kd = framed(k)
    _, vd = framed(v)
    canary_o = torch.full((q.numel() + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    canary_l = torch.full((B * Hq * N + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = canary_o[pad:pad + q.numel()].view(q.shape)
    lse = canary_l[pad:pad + B * Hq * N].view(B, Hq, N)
    for causal in (False, True):
        eta.attn_fwd(qd, kd, vd, causal=causal, out=o, lse=lse)
        torch.cuda.synchronize()
        assert eta.attn_get_device_error() == 0
        assert torch.all(canary_o[:pad] == 7) and torch.all(canary_o[-pad:] == 7)
        assert torch.all(canary_l[:pad] == 7) and torch.all(canary_l[-pad:] == 7)
        o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), 1 / math.sqrt(d), causal, -1)
        check_attention(o, lse, o_ref, lse_ref, f"framed causal={causal}")


def test_deterministic_and_stream_aware():
    q, k, v = inputs.prefill_inputs(1, 4, 4, 700, 700, 128, seed=11)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = eta.attn_fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = eta.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("cfg", [inputs.C2, inputs.C3, inputs.C4], ids=lambda c: c.name)
def test_full_size_every_row(oracle, cfg):
    """Full workload in the bench's launch configuration: every output element and every
    lse of every head against the oracle ("Modern attention kernels", "Numerical
    validation": long rows with large logit ranges, GQA mapping; C3 also moves the running
    max late in many rows through its doubled K rows)."""
    q, k, v = inputs.prefill_config_inputs(cfg)
    o, lse = run_fwd(q, k, v, cfg.causal, cfg.window)
    o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), cfg.scale, cfg.causal, cfg.window)
    check_attention(o, lse, o_ref, lse_ref, cfg.name)
