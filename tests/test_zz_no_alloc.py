"""GPU: attn_decode_noalloc, the decode entry point for callers that cannot allocate
device memory (a runtime that reserved HBM for its own pools, a plugin inside another
framework's execution plan). Its split partials live in a static array inside the
library. Called through the C ABI twice in a row, its output must match attn_decode
(with a caller-supplied workspace) within the parity tolerances of the other tests.

This file is collected last on purpose, and it passes both alone and after the rest.
"""
import math

import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs

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


def test_noalloc_decode_matches_workspace_decode():
    eta.build()
    lib = eta.load_library()
    S, Hq, Hkv, d, bs = 12, 32, 8, 128, 16
    x = inputs.decode_inputs(S, Hq, Hkv, d, bs, len_lo=1, len_hi=6000, seed=21, extra_blocks=4, poison=True)
    x.seq_lens[0] = 0  # an empty sequence too
    dev = torch.device("cuda")
    q, kc, vc = x.q.to(dev), x.k_cache.to(dev), x.v_cache.to(dev)
    bt, sl = x.block_table.to(dev), x.seq_lens.to(dev)
    mb = bt.shape[1]
    scale = 1.0 / math.sqrt(d)
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb) <= 64 << 20

    o_ref, lse_ref = eta.attn_decode(q, kc, vc, bt, sl, scale=scale)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0

    stream = torch.cuda.current_stream().cuda_stream or None
    for _ in range(2):  # two calls in a row: the shared array keeps the previous call's contents
        o = torch.full_like(q, float("nan"))
        lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev)
        rc = lib.attn_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), sl.data_ptr(),
                                     o.data_ptr(), lse.data_ptr(), S, Hq, Hkv, d, bs, mb, kc.shape[0], scale,
                                     stream)
        assert rc == 0, eta.attn_status_string(rc)
        torch.cuda.synchronize()
        assert eta.attn_get_device_error() == 0
        _compare(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    eta.build()
    lib = eta.load_library()
    # 64 sequences x 32 query heads x 64 splits (32k context) needs ~65 MiB of partials
    S, Hq, Hkv, d, bs, mb = 64, 32, 8, 128, 16, 2048
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb) > 64 << 20
    fake = 0x7F0000000000
    rc = lib.attn_decode_noalloc(fake, fake, fake, fake, fake, fake, fake, S, Hq, Hkv, d, bs, mb, 1000, 0.1, None)
    assert rc == -4, eta.attn_status_string(rc)
