"""GPU: attn_decode_noalloc, the decode entry point for callers that cannot allocate
device memory where they run decode (a serving runtime that reserved HBM for its own
pools and forbids further cudaMalloc, a plugin inside another framework's execution plan
where allocation calls are not allowed). Its split partials live in a static array inside
the library instead of a caller-supplied workspace.

Called through the C ABI twice in a row (the shared array keeps the first call's
contents), its output must match both the fp64 oracle and attn_decode with a caller-
supplied workspace, within the tolerances of the other parity tests, and the device's
free memory must not change between the two calls.

This file is collected last on purpose, and it passes both alone and after the rest.
"""
import math

import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs
from tests.gpu_util import check_attention, f64

pytestmark = pytest.mark.gpu

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def _compare(o, lse, o_ref, lse_ref):
    err = (o.float() - o_ref.float()).abs()
    assert torch.isfinite(o.float()).all()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
    fin = ~torch.isneginf(lse_ref)
    rel = (lse[fin] - lse_ref[fin]).abs() / lse_ref[fin].abs().clamp_min(1.0)
    assert rel.max().item() <= LSE_REL


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_decode_matches_oracle_and_workspace_decode(oracle, d):
    eta.build()
    lib = eta.load_library()
    S, Hq, Hkv, bs = 12, 32, 8, 16
    x = inputs.decode_inputs(S, Hq, Hkv, d, bs, len_lo=1, len_hi=6000, seed=21 + d, extra_blocks=4, poison=True)
    x.seq_lens[0] = 0  # an empty sequence too
    dev = torch.device("cuda")
    q, kc, vc = x.q.to(dev), x.k_cache.to(dev), x.v_cache.to(dev)
    bt, sl = x.block_table.to(dev), x.seq_lens.to(dev)
    mb = bt.shape[1]
    scale = 1.0 / math.sqrt(d)
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb) <= 64 << 20

    o_ws, lse_ws = eta.attn_decode(q, kc, vc, bt, sl, scale=scale)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    kc64 = torch.nan_to_num(x.k_cache.double()).numpy()
    vc64 = torch.nan_to_num(x.v_cache.double()).numpy()
    o_ref, lse_ref = oracle.attn_decode(f64(x.q), kc64, vc64, x.block_table.numpy(), x.seq_lens.numpy(), scale)

    # outputs for both calls exist before the first one, so nothing in between allocates
    outs = [(torch.full_like(q, float("nan")), torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev))
            for _ in range(2)]
    stream = torch.cuda.current_stream().cuda_stream or None
    free = []
    for o, lse in outs:  # two calls in a row: the shared array keeps the previous call's contents
        rc = lib.attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), sl.data_ptr(),
                                     o.data_ptr(), lse.data_ptr(), S, Hq, Hkv, d, bs, mb, kc.shape[0], scale,
                                     stream)
        assert rc == 0, eta.attn_status_string(rc)
        torch.cuda.synchronize()
        assert eta.attn_get_device_error() == 0
        free.append(torch.cuda.mem_get_info()[0])
        _compare(o, lse, o_ws, lse_ws)
        check_attention(o, lse, o_ref, lse_ref, f"noalloc d={d}")
    assert free[0] == free[1], f"device free memory changed between calls: {free[0]} -> {free[1]}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    eta.build()
    lib = eta.load_library()
    # 64 sequences x 32 query heads x 64 splits (32k context) needs ~65 MiB of partials.
    # Real (small) device buffers: the size check must reject the call before any launch,
    # and nothing here would let a kernel read past them if it did not.
    S, Hq, Hkv, d, bs, mb, nblk = 64, 32, 8, 128, 16, 2048, 4
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb) > 64 << 20
    dev = torch.device("cuda")
    q = torch.zeros((S, Hq, d), dtype=torch.bfloat16, device=dev)
    o = torch.zeros_like(q)
    lse = torch.zeros((S, Hq), dtype=torch.float32, device=dev)
    kc = torch.zeros((nblk, Hkv, bs, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    bt = torch.zeros((S, mb), dtype=torch.int32, device=dev)
    sl = torch.ones((S,), dtype=torch.int32, device=dev)
    rc = lib.attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), sl.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), S, Hq, Hkv, d, bs, mb, nblk, 0.1, None)
    assert rc == -4, eta.attn_status_string(rc)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    assert torch.all(o == 0) and torch.all(lse == 0)  # nothing was written
