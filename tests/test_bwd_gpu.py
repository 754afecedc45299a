"""GPU parity: attn_bwd (dQ, dK, dV) through the C ABI against the fp64 oracle's
gradients, on the same bf16 inputs; o and lse come from attn_fwd as a caller would
pass them.

Tolerances (each gradient tensor against the oracle, relative to the reference's own
scale, since gradients have no fixed magnitude):
  max |err|  <= GRAD_MAX_REL  * max |ref|  (+ ABS_FLOOR)
  mean |err| <= GRAD_MEAN_REL * mean |ref| (+ ABS_FLOOR)
The kernel rounds P and dS to bf16 before the tensor-core products (relative error
2^-9 per term, fp32 accumulation), takes D_i from the bf16 O of the forward and rounds
each gradient to bf16 on output (relative 2^-9), so single elements can be off by a few
2^-9 of the largest entry and the mean error stays near the output rounding.
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs
from tests.gpu_util import f64

pytestmark = pytest.mark.gpu

GRAD_MAX_REL = 2e-2
GRAD_MEAN_REL = 5e-3
ABS_FLOOR = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    eta.build()
    eta.load_library()


def run_bwd(q, k, v, do, causal, window, scale, poison=True):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = eta.attn_fwd(qd, kd, vd, causal=causal, window=window, scale=scale)
    dq = dk = dv = None
    if poison:  # every element must be written
        dq = torch.full_like(qd, float("nan"))
        dk = torch.full_like(kd, float("nan"))
        dv = torch.full_like(vd, float("nan"))
    dq, dk, dv = eta.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal, window=window, scale=scale, dq=dq, dk=dk,
                              dv=dv)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return dq, dk, dv


def check_grad(got, ref, name):
    g = f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite entries"
    err = np.abs(g - ref)
    if ref.size == 0:
        return 0.0, 0.0
    # An absolute floor covers gradients that vanish exactly (one visible key: P = 1 and
    # dS = dP - D = 0), where fp32 rounding of lse leaves residues near 1e-7.
    scale_max = max(np.abs(ref).max(), ABS_FLOOR / GRAD_MAX_REL)
    scale_mean = max(np.abs(ref).mean(), ABS_FLOOR / GRAD_MEAN_REL)
    rmax = err.max() / scale_max
    rmean = err.mean() / scale_mean
    assert rmax <= GRAD_MAX_REL, f"{name}: max |err| / max |ref| = {rmax:.3e}"
    assert rmean <= GRAD_MEAN_REL, f"{name}: mean |err| / mean |ref| = {rmean:.3e}"
    return float(rmax), float(rmean)


def case(oracle, B, Hq, Hkv, Nq, Nk, d, causal, window, seed=0, boost=0.0, what=""):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed, k_boost_frac=boost)
    do = inputs.grad_output(B, Hq, Nq, d, seed=seed)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = run_bwd(q, k, v, do, causal, window, scale)
    rq, rk, rv = oracle.attn_bwd(f64(q), f64(k), f64(v), f64(do), scale, causal, window)
    out = {}
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        out[name] = check_grad(got, ref, f"{what} {name}")
    return out


SWEEP_N = [1, 64, 127, 128, 129, 257, 500]
SWEEP_MASKS = [(False, -1), (True, -1), (True, 0), (True, 127), (True, 129), (False, 200)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", SWEEP_N)
@pytest.mark.parametrize("causal,window", SWEEP_MASKS)
def test_bwd_boundary_sweep(oracle, N, d, causal, window):
    case(oracle, 1, 2, 1, N, N, d, causal, window, seed=N + d, what=f"N={N} d={d} c={causal} w={window}")


@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 100), (1, 700), (129, 1), (200, 257), (384, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_rectangular(oracle, Nq, Nk, causal):
    """Bottom-right causal alignment; Nq > Nk leaves the first Nq - Nk rows without keys."""
    case(oracle, 2, 2, 2, Nq, Nk, 128, causal, -1, seed=Nq * 7 + Nk, what=f"{Nq}x{Nk} c={causal}")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (6, 2), (8, 1), (3, 1)])
def test_bwd_gqa_sums_over_group(oracle, Hq, Hkv):
    """dK, dV of a kv head sum the contributions of every query head that reads it."""
    case(oracle, 2, Hq, Hkv, 300, 300, 128, True, -1, seed=Hq * 10 + Hkv, what=f"GQA {Hq}/{Hkv}")


def test_bwd_large_logits(oracle):
    """1% of keys scaled by 2 (the long-causal workload's outliers): peaked rows."""
    case(oracle, 1, 4, 2, 640, 640, 128, True, -1, seed=5, boost=0.01, what="boosted keys")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_multi_tile_window(oracle, d):
    """Window narrower than a tile over several key tiles: most tiles see two query tiles."""
    case(oracle, 1, 2, 2, 1100, 1100, d, True, 200, seed=d, what=f"window 200 d={d}")


def test_bwd_no_queries():
    """Nq = 0: nothing flows back, dK = dV = 0 (every element written)."""
    d = 128
    k = torch.randn(1, 2, 300, d).to(torch.bfloat16).cuda()
    v = torch.randn(1, 2, 300, d).to(torch.bfloat16).cuda()
    q = torch.empty(1, 2, 0, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, 0, dtype=torch.float32, device="cuda")
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    dq, dk, dv = eta.attn_bwd(q, k, v, q, q, lse, causal=True, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    assert dq.numel() == 0
    assert torch.all(dk == 0) and torch.all(dv == 0)


def test_bwd_no_keys():
    """Nk = 0: every row is empty (O = 0, lse = -inf), so dQ = 0."""
    d = 64
    q = torch.randn(2, 2, 100, d).to(torch.bfloat16).cuda()
    k = torch.empty(2, 1, 0, d, dtype=torch.bfloat16, device="cuda")
    o, lse = eta.attn_fwd(q, k, k)
    do = torch.randn_like(q.float()).to(torch.bfloat16)
    dq = torch.full_like(q, float("nan"))
    dq, dk, dv = eta.attn_bwd(q, k, k, o, do, lse, dq=dq)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    assert torch.all(dq == 0) and dk.numel() == 0


def test_bwd_deterministic_dk_dv():
    """dK and dV accumulate in one block's tensor memory in a fixed order: repeated calls
    give identical bits (dQ sums partials with atomics, so only its value is stable)."""
    q, k, v = inputs.prefill_inputs(1, 4, 2, 700, 700, 128, seed=3)
    do = inputs.grad_output(1, 4, 700, 128, seed=3)
    a = run_bwd(q, k, v, do, True, -1, 0.1, poison=False)
    b = run_bwd(q, k, v, do, True, -1, 0.1, poison=False)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2e-2 * a[0].float().abs().max().item()


def test_bwd_full_size_whole_heads_and_invariants(oracle):
    """At the long-causal size (B=1, H=32, N=8192, d=128), as the bench runs it:
    - four whole heads (each its own kv head: first, last and two inside) element by
      element against the oracle's dQ, dK and dV at the stated gradient tolerances;
    - every head: sum_j dK_j = 0 (each row of dS sums to zero) and sum_j dV_j = sum_i dO_i
      (each row of P sums to one)."""
    c = inputs.C3
    q, k, v = inputs.prefill_config_inputs(c)
    do = inputs.grad_output(c.B, c.Hq, c.Nq, c.d, seed=c.seed)
    scale = 1.0 / math.sqrt(c.d)
    dq, dk, dv = run_bwd(q, k, v, do, c.causal, c.window, scale)
    dk64, dv64 = dk.double(), dv.double()
    sum_dk = dk64.sum(dim=2)
    assert (sum_dk.abs() <= 1e-2 * dk64.abs().sum(dim=2) + 1e-3).all()
    sum_dv = dv64.sum(dim=2)
    sum_do = do.cuda().double().sum(dim=2)
    assert ((sum_dv - sum_do).abs() <= 1e-2 * dv64.abs().sum(dim=2) + 1e-2).all()
    assert torch.isfinite(dq.float()).all()
    assert c.Hq == c.Hkv  # one query head per kv head: a head is a whole kv-head group
    heads = [0, 11, 22, c.Hq - 1]
    rq, rk, rv = oracle.attn_bwd(f64(q[:, heads]), f64(k[:, heads]), f64(v[:, heads]), f64(do[:, heads]), scale,
                                 c.causal, c.window)
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    for i, h in enumerate(heads):
        for name, got, ref in (("dq", dq[:, h], rq[:, i]), ("dk", dk[:, h], rk[:, i]), ("dv", dv[:, h], rv[:, i])):
            check_grad(got, ref, f"C3 head {h} {name}")
