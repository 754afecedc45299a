"""GPU parity: attn_prefill_paged (chunked prefill over a paged cache) through the C ABI
against the fp64 oracle on the same bf16 inputs, with NaN in every cache slot no sequence
owns and in the query rows past each q_len; bitwise agreement with attn_fwd when the cache
is contiguous; full-size sampled rows of the chunked-prefill workload."""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import inputs
from tests.gpu_util import check_attention, f64

pytestmark = pytest.mark.gpu

SENTINEL = 3.0  # written into o / lse before the call: rows past q_len must keep it


@pytest.fixture(scope="module", autouse=True)
def built():
    eta.build()
    eta.load_library()


def run(x, causal, window, scale):
    dev = torch.device("cuda")
    q = x.q.to(dev)
    out = torch.full_like(q, SENTINEL)
    lse = torch.full(q.shape[:3], SENTINEL, dtype=torch.float32, device=dev)
    o, l = eta.attn_prefill_paged(q, x.k_cache.to(dev), x.v_cache.to(dev), x.block_table.to(dev), x.q_lens.to(dev),
                                  x.kv_lens.to(dev), causal=causal, window=window, scale=scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return o, l


def check(oracle, x, causal, window, what, scale=None):
    d = x.q.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = run(x, causal, window, scale)
    kc = torch.nan_to_num(x.k_cache.double()).numpy()
    vc = torch.nan_to_num(x.v_cache.double()).numpy()
    qd = torch.nan_to_num(x.q.double()).numpy()
    o_ref, lse_ref = oracle.attn_prefill_paged(qd, kc, vc, x.block_table.numpy(), x.q_lens.numpy(),
                                               x.kv_lens.numpy(), scale, causal, window)
    o_h, lse_h = f64(o), f64(lse)
    for s in range(x.q.shape[0]):
        n = int(x.q_lens[s])
        if n > 0:
            check_attention(o_h[s, :, :n], lse_h[s, :, :n], o_ref[s, :, :n], lse_ref[s, :, :n], f"{what} seq{s}")
        assert np.all(o_h[s, :, n:] == SENTINEL) and np.all(lse_h[s, :, n:] == SENTINEL), f"{what} seq{s}: rows past q_len written"


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("d", [64, 128])
def test_block_sizes(oracle, bs, d):
    q_lens = [130, 1, 0, 200, 64]
    kv_lens = [300, 129, 17, 200, 1000]
    x = inputs.paged_prefill_inputs(5, 8, 2, d, bs, q_lens, kv_lens, seed=bs + d, extra_blocks=3, poison=True)
    check(oracle, x, True, -1, f"bs={bs} d={d}")


@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 0), (True, 100), (True, 128), (False, 70)])
def test_masks(oracle, causal, window):
    q_lens = [257, 128, 33]
    kv_lens = [700, 128, 401]
    x = inputs.paged_prefill_inputs(3, 4, 4, 128, 16, q_lens, kv_lens, seed=7, extra_blocks=2, poison=True)
    check(oracle, x, causal, window, f"c={causal} w={window}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (6, 2), (3, 1)])
def test_gqa(oracle, Hq, Hkv):
    x = inputs.paged_prefill_inputs(2, Hq, Hkv, 128, 32, [300, 77], [900, 77], seed=Hq * 10 + Hkv, poison=True)
    check(oracle, x, True, -1, f"GQA {Hq}/{Hkv}")


def test_full_prefill_and_single_query_edges(oracle):
    """q_len = kv_len (a whole prompt), q_len = 1 (decode-like), q_len = 0 (nothing to do)."""
    x = inputs.paged_prefill_inputs(4, 4, 2, 128, 16, [513, 1, 0, 1], [513, 1, 5, 2000], seed=3, extra_blocks=4,
                                    poison=True)
    check(oracle, x, True, -1, "edges")


def test_contiguous_cache_matches_dense_prefill_bitwise():
    """With an identity block table the cache rows of a sequence are contiguous per kv
    head; the paged kernel then feeds the tensor cores the same tiles as attn_fwd."""
    B, Hq, Hkv, N, d, bs = 1, 8, 2, 1000, 128, 16
    x = inputs.paged_prefill_inputs(1, Hq, Hkv, d, bs, [N], [N], seed=11, identity_table=True)
    nblk = (N + bs - 1) // bs
    # [num_blocks][Hkv][bs][d] -> [1][Hkv][N][d]
    k = x.k_cache[:nblk].permute(1, 0, 2, 3).reshape(Hkv, nblk * bs, d)[:, :N][None].contiguous()
    v = x.v_cache[:nblk].permute(1, 0, 2, 3).reshape(Hkv, nblk * bs, d)[:, :N][None].contiguous()
    dev = torch.device("cuda")
    o_d, l_d = eta.attn_fwd(x.q.to(dev), k.to(dev), v.to(dev), causal=True)
    o_p, l_p = run(x, True, -1, 1.0 / math.sqrt(d))
    assert torch.equal(o_d, o_p) and torch.equal(l_d, l_p)


def test_bad_block_table_entry_sets_error():
    """An entry outside [0, num_blocks) is reported in the device error word, and the call
    stays in bounds (the kernel clamps the block it reads)."""
    x = inputs.paged_prefill_inputs(2, 4, 2, 128, 16, [10, 20], [40, 60], seed=5)
    bt = x.block_table.clone()
    bt[1, 2] = 10_000
    dev = torch.device("cuda")
    eta.attn_prefill_paged(x.q.to(dev), x.k_cache.to(dev), x.v_cache.to(dev), bt.to(dev), x.q_lens.to(dev),
                           x.kv_lens.to(dev))
    torch.cuda.synchronize()
    assert eta.binding.STATUS_NAMES[eta.attn_get_device_error()] == "ATTN_ERR_DEVICE_BOUNDS"
    assert eta.attn_get_device_error() == 0  # read-and-clear


def test_chunked_prefill_workload_every_row(oracle):
    """The benchmark's chunked-prefill workload at full size: every new row of every
    sequence and query head against the oracle ("Modern attention kernels", "Numerical
    validation": GQA mapping, paged blocks that cross sequence tails)."""
    c = inputs.C6
    x = inputs.paged_prefill_config_inputs(c)
    o, lse = run(x, c.causal, -1, c.scale)
    o_ref, l_ref = oracle.attn_prefill_paged(x.q.double().numpy(), x.k_cache.double().numpy(),
                                             x.v_cache.double().numpy(), x.block_table.numpy(), x.q_lens.numpy(),
                                             x.kv_lens.numpy(), c.scale, c.causal)
    ql = x.q_lens.tolist()
    assert min(ql) == max(ql) == o.shape[2]  # every padded row is a real row in this workload
    check_attention(o, lse, o_ref, l_ref, "C6 every row")
