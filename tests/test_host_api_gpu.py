"""GPU: the host-buffer entry points (attn_fwd_host, attn_decode_host) give bitwise the
results of attn_fwd / attn_decode, for pinned and pageable host memory, every chunking,
GQA, several batch entries, and on a side stream."""

import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    eta.build()
    eta.load_library()


def fwd_host_case(B, Hq, Hkv, Nq, Nk, d, causal, window, chunk, pinned, seed):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pinned)
    l_h = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=pinned)
    q_d, k_d, v_d = torch.empty_like(q, device="cuda"), torch.empty_like(k, device="cuda"), torch.empty_like(v, device="cuda")
    o_d = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    l_d = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    eta.attn_fwd_host(q, k, v, o_h, l_h, q_d, k_d, v_d, o_d, l_d, causal=causal, window=window, chunk_kv_heads=chunk)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    o_ref, l_ref = eta.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_ref.cpu()), "attn_fwd_host O differs from attn_fwd"
    assert torch.equal(l_h, l_ref.cpu()), "attn_fwd_host lse differs from attn_fwd"


@pytest.mark.parametrize("chunk", [0, 1, 3, 8])
def test_fwd_host_chunkings(chunk):
    fwd_host_case(2, 16, 8, 300, 300, 128, True, -1, chunk, True, 41 + chunk)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal,window", [
    (1, 4, 4, 128, 128, 64, False, -1),
    (3, 8, 2, 200, 333, 128, True, -1),
    (1, 6, 3, 257, 257, 128, True, 64),
])
def test_fwd_host_shapes(B, Hq, Hkv, Nq, Nk, d, causal, window):
    fwd_host_case(B, Hq, Hkv, Nq, Nk, d, causal, window, 0, True, B * 7 + Hq)


def test_fwd_host_pageable_memory():
    fwd_host_case(1, 8, 2, 256, 256, 128, True, -1, 1, False, 49)


def test_fwd_host_on_a_side_stream():
    q, k, v = [t.pin_memory() for t in inputs.prefill_inputs(1, 8, 4, 256, 256, 128, seed=50)]
    o_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    l_h = torch.empty((1, 8, 256), dtype=torch.float32, pin_memory=True)
    dev = [torch.empty_like(t, device="cuda") for t in (q, k, v)]
    o_d = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    l_d = torch.empty((1, 8, 256), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eta.attn_fwd_host(q, k, v, o_h, l_h, *dev, o_d, l_d, causal=True)
    s.synchronize()
    o_ref, _ = eta.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_ref.cpu())


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_host_equals_decode(pinned):
    x = inputs.decode_inputs(5, 8, 2, 128, 16, len_lo=1, len_hi=2000, seed=51, extra_blocks=2)
    hs = [x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens]
    if pinned:
        hs = [t.pin_memory() for t in hs]
    o_h = torch.empty(x.q.shape, dtype=torch.bfloat16, pin_memory=pinned)
    l_h = torch.empty(x.q.shape[:2], dtype=torch.float32, pin_memory=pinned)
    ds = [torch.empty_like(t, device="cuda") for t in hs]
    o_d = torch.empty(x.q.shape, dtype=torch.bfloat16, device="cuda")
    l_d = torch.empty(x.q.shape[:2], dtype=torch.float32, device="cuda")
    eta.attn_decode_host(*hs, o_h, l_h, *ds, o_d, l_d)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    o_ref, l_ref = eta.attn_decode(*[t.cuda() for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)])
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_ref.cpu()) and torch.equal(l_h, l_ref.cpu())
