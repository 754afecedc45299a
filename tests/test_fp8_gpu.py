"""GPU parity: attn_fwd_fp8 (E4M3 Q, K, transposed V, per-tensor scales) through the C ABI
against the fp64 oracle on the same codes.

Tolerance, from the one rounding the kernel adds to the definition: each unnormalised
probability, held as p_j = 2^6 * 2^(s_j - m) with m lagging the row maximum by less than
4x (so p_j <= 2^8), is rounded to E4M3 for the P V product: relative error <= 2^-4 for
p_j >= 2^-6 (probabilities down to 2^-12 of the maximum's weight), absolute <= 2^-10 in
p_j below (<= 2^-16 of the maximum's weight); the row sum keeps the unrounded values. So
for an output element |O - O_ref| <= 2^-4 * sum_j P_j |v_j| + (absolute part), with P
the exact probabilities: the bound term A = sum_j P_j |v_j| is the oracle's own
attention over |V| (the V codes with the sign bit cleared). The absolute part is at most
2^-16 |v_j| per key of negligible weight, with random signs: ~sqrt(n) 2^-16 |v| <= 1.5e-3
for n <= 8192 keys. On top come the bf16 rounding of O (2^-9 relative) and the fp32
accumulation. Checked: per element |err| <= 2^-4 A + 2^-8 |O_ref| + 2e-3, and mean |err|
<= 2^-6 mean(A) (the per-probability errors have random signs and average out). lse
does not see the rounding: |err| / max(|lse|, 1) <= 1e-3 as for bf16.
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs
from tests.gpu_util import LSE_REL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    eta.build()
    eta.load_library()


def run(x: inputs.Fp8PrefillInputs, causal, window=-1, scale=None):
    o, lse = eta.attn_fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.vt8.cuda(), x.q_descale, x.k_descale, x.v_descale,
                              causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return o, lse


def check_fp8(oracle, x, o, lse, causal, window=-1, scale=None, what=""):
    d = x.q8.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    args = (x.q8.numpy(), x.k8.numpy())
    o_ref, lse_ref = oracle.attn_fwd_fp8(*args, x.vt8.numpy(), scale, x.q_descale, x.k_descale, x.v_descale,
                                         causal, window)
    bound, _ = oracle.attn_fwd_fp8(*args, (x.vt8 & 0x7F).numpy(), scale, x.q_descale, x.k_descale, x.v_descale,
                                   causal, window)
    og, lg = f64(o), f64(lse)
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    err = np.abs(og - o_ref)
    tol = 2.0 ** -4 * bound + 2.0 ** -8 * np.abs(o_ref) + 2e-3
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), f"{what}: O err {err[worst]:.3e} > {tol[worst]:.3e} at {worst}"
    assert err.mean() <= 2.0 ** -6 * bound.mean() + 1e-6, f"{what}: mean err {err.mean():.3e}"
    ref_inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), ref_inf), f"{what}: -inf lse pattern"
    fin = ~ref_inf
    if fin.any():
        rel = np.abs(lg[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)
        assert rel.max() <= LSE_REL, f"{what}: lse rel err {rel.max():.3e}"
    return float(err.max()), float(err.mean())


@pytest.mark.parametrize("Nq,Nk,causal,window", [
    (128, 128, False, -1),
    (256, 256, True, -1),
    (300, 304, True, -1),       # ragged tiles, Nk a multiple of 16
    (200, 512, True, -1),       # bottom-right causal alignment
    (500, 128, True, -1),       # leading rows see no key
    (384, 384, True, 100),      # sliding window
    (320, 400, False, 50),      # left limit only
    (1000, 1008, True, -1),     # several tiles in both directions
])
def test_fp8_shapes(oracle, Nq, Nk, causal, window):
    x = inputs.fp8_prefill_inputs(1, 2, 2, Nq, Nk, 128, seed=Nq + Nk)
    o, lse = run(x, causal, window)
    check_fp8(oracle, x, o, lse, causal, window, what=f"Nq={Nq} Nk={Nk} causal={causal} w={window}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 3), (4, 4), (8, 1)])
def test_fp8_gqa(oracle, Hq, Hkv):
    x = inputs.fp8_prefill_inputs(2, Hq, Hkv, 192, 256, 128, seed=Hq * 10 + Hkv)
    o, lse = run(x, True)
    check_fp8(oracle, x, o, lse, True, what=f"GQA {Hq}/{Hkv}")


def test_fp8_large_logits_peaked_rows(oracle):
    """A scale that makes rows nearly one-hot: the probabilities near 1 carry the largest
    absolute rounding, and the lazy rescale may leave them up to 2^8 before rounding."""
    x = inputs.fp8_prefill_inputs(1, 2, 1, 256, 256, 128, seed=31)
    o, lse = run(x, True, scale=0.6)
    check_fp8(oracle, x, o, lse, True, scale=0.6, what="peaked")


def test_fp8_late_maximum(oracle):
    """The largest score of each row sits in the last key tile: every earlier P was rounded
    against a stale maximum and must be rescaled."""
    x = inputs.fp8_prefill_inputs(1, 1, 1, 128, 512, 128, seed=32)
    k = x.k8.view(torch.float8_e4m3fn).float()
    q = x.q8.view(torch.float8_e4m3fn).float()
    k[0, 0, 500] = q[0, 0].mean(dim=0).sign() * 240.0  # aligned with every query row
    x.k8 = k.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    o, lse = run(x, False)
    check_fp8(oracle, x, o, lse, False, what="late maximum")


def test_fp8_no_keys_and_no_queries():
    x = inputs.fp8_prefill_inputs(1, 2, 1, 64, 16, 128, seed=33)
    q8 = x.q8.cuda()
    k0 = torch.empty((1, 1, 0, 128), dtype=torch.uint8, device="cuda")
    v0 = torch.empty((1, 1, 128, 0), dtype=torch.uint8, device="cuda")
    o, lse = eta.attn_fwd_fp8(q8, k0, v0, 1.0, 1.0, 1.0, causal=False)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()
    q0 = torch.empty((1, 2, 0, 128), dtype=torch.uint8, device="cuda")
    o, lse = eta.attn_fwd_fp8(q0, x.k8.cuda(), x.vt8.cuda(), 1.0, 1.0, 1.0)
    assert o.numel() == 0


def test_fp8_deterministic_and_scale_linear(oracle):
    x = inputs.fp8_prefill_inputs(1, 4, 2, 256, 256, 128, seed=34)
    o1, l1 = run(x, True)
    o2, l2 = run(x, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # V's scale only multiplies O (power of two: exact in bf16)
    o3, l3 = eta.attn_fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.vt8.cuda(), x.q_descale, x.k_descale, 4 * x.v_descale,
                              causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o3.float(), 4 * o1.float()) and torch.equal(l3, l1)


def test_fp8_float8_dtype_accepted():
    x = inputs.fp8_prefill_inputs(1, 2, 1, 128, 128, 128, seed=35)
    o1, _ = run(x, True)
    o2, _ = eta.attn_fwd_fp8(x.q8.cuda().view(torch.float8_e4m3fn), x.k8.cuda().view(torch.float8_e4m3fn),
                             x.vt8.cuda().view(torch.float8_e4m3fn), x.q_descale, x.k_descale, x.v_descale,
                             causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_fp8_paired_blocks(oracle):
    """160 heads keep two query tiles per block (small grids run one per block)."""
    x = inputs.fp8_prefill_inputs(1, 160, 160, 300, 304, 128, seed=160)
    o, lse = run(x, True)
    check_fp8(oracle, x, o, lse, True, what="160 heads")


def test_fp8_full_long_causal_every_row(oracle):
    """The long causal workload (B1 H32 N8192 d128, 1 % of K rows doubled) in E4M3, as the
    bench times it: every row of every head against the oracle on the decoded values, with
    the derived E4M3 bound per element."""
    c = inputs.C3
    x = inputs.fp8_prefill_inputs(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, seed=c.seed, k_boost_frac=c.k_boost_frac)
    o, lse = run(x, True)
    check_fp8(oracle, x, o, lse, True, what="C3 in E4M3, every row")
