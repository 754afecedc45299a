"""GPU parity: attn_fwd_blocksparse through the C ABI against the fp64 oracle on the same
bf16 inputs and block index; bitwise agreement with attn_fwd when every block is listed
(the kernel then visits the same tiles in the same order); empty block rows; invalid
indices reported in the device error word."""
import math

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


def run(q, k, v, pat, causal, window, scale=None):
    rp, ci = inputs.block_csr(pat)
    dev = torch.device("cuda")
    o, lse = eta.attn_fwd_blocksparse(q.to(dev), k.to(dev), v.to(dev), rp.to(dev), ci.to(dev), causal=causal,
                                      window=window, scale=scale)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return o, lse


def case(oracle, B, Hq, Hkv, Nq, Nk, d, causal, window, pat, seed, what):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = run(q, k, v, pat, causal, window)
    rp, ci = inputs.block_csr(pat)
    o_ref, lse_ref = oracle.attn_fwd_blocksparse(f64(q), f64(k), f64(v), rp.numpy(), ci.numpy(), scale, causal,
                                                 window)
    check_attention(o, lse, o_ref, lse_ref, what)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 200), (False, 300)])
def test_random_patterns(oracle, d, causal, window):
    Nq = Nk = 900  # 8 blocks, ragged last block
    pat = inputs.random_pattern(8, 8, 0.5, seed=d + (3 if causal else 0), empty_rows=(2,))
    case(oracle, 1, 4, 2, Nq, Nk, d, causal, window, pat, seed=d, what=f"d={d} c={causal} w={window}")


@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (1000, 300), (129, 129), (1, 700)])
def test_rectangular(oracle, Nq, Nk):
    nq, nk = -(-Nq // 128), -(-Nk // 128)
    pat = inputs.random_pattern(nq, nk, 0.6, seed=Nq + Nk)
    case(oracle, 2, 2, 2, Nq, Nk, 128, True, -1, pat, seed=Nq, what=f"{Nq}x{Nk}")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 2), (3, 1)])
def test_gqa_and_pairing(oracle, Hq, Hkv):
    """Even groups pair two query heads per block (one list); odd groups pair two row
    tiles (two lists merged into one walk)."""
    pat = inputs.global_local_pattern(6, 6, 1, 2)
    pat[3] = inputs.random_pattern(1, 6, 0.5, seed=Hq)[0]
    case(oracle, 1, Hq, Hkv, 700, 700, 128, True, -1, pat, seed=Hq * 10 + Hkv, what=f"GQA {Hq}/{Hkv}")


def test_global_local_pattern(oracle):
    pat = inputs.global_local_pattern(16, 16, 1, 4)
    case(oracle, 1, 4, 4, 2000, 2000, 128, True, -1, pat, seed=4, what="global+local")


def test_empty_pattern_gives_empty_rows():
    q, k, v = inputs.prefill_inputs(1, 2, 2, 300, 300, 64, seed=1)
    pat = torch.zeros((3, 3), dtype=torch.bool)
    o, lse = run(q, k, v, pat, True, -1)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("shape", [(1, 4, 2, 1000, 1000, 128, True, -1), (2, 3, 3, 700, 900, 64, False, 300),
                                   (1, 32, 32, 8192, 8192, 128, True, -1)])
def test_full_pattern_equals_dense_bitwise(shape):
    B, Hq, Hkv, Nq, Nk, d, causal, window = shape
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq)
    pat = torch.ones((-(-Nq // 128), -(-Nk // 128)), dtype=torch.bool)
    o, lse = run(q, k, v, pat, causal, window)
    dev = torch.device("cuda")
    od, ld = eta.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=window)
    assert torch.equal(o, od) and torch.equal(lse, ld)


def test_invalid_index_sets_error():
    """A key block past the end and an out-of-order entry are reported and skipped."""
    q, k, v = inputs.prefill_inputs(1, 2, 2, 256, 256, 64, seed=2)
    dev = torch.device("cuda")
    rp = torch.tensor([0, 2, 4], dtype=torch.int32, device=dev)
    ci = torch.tensor([0, 7, 1, 0], dtype=torch.int32, device=dev)  # 7 >= 2 blocks; row 1 descending
    eta.attn_fwd_blocksparse(q.to(dev), k.to(dev), v.to(dev), rp, ci, causal=False)
    torch.cuda.synchronize()
    assert eta.binding.STATUS_NAMES[eta.attn_get_device_error()] == "ATTN_ERR_DEVICE_BOUNDS"
    assert eta.attn_get_device_error() == 0


def test_c7_workload_every_row(oracle):
    """The benchmark's block-sparse workload at full size (32 heads of 32768 tokens, key
    block 0 plus the 8 blocks ending at the diagonal, causal): every output element and lse
    against the oracle."""
    c = inputs.C7
    q, k, v, pat = inputs.sparse_config_inputs(c)
    o, lse = run(q, k, v, pat, c.causal, -1, c.scale)
    rp, ci = inputs.block_csr(pat)
    o_ref, lse_ref = oracle.attn_fwd_blocksparse(f64(q), f64(k), f64(v), rp.numpy(), ci.numpy(), c.scale, c.causal,
                                                 -1)
    check_attention(o, lse, o_ref, lse_ref, c.name)


def test_random_pattern_paired_blocks(oracle):
    """160 heads keep two query tiles per block (small grids run one per block)."""
    pat = inputs.random_pattern(8, 8, 0.5, seed=160, empty_rows=(3,))
    case(oracle, 1, 160, 160, 900, 900, 128, True, -1, pat, seed=160, what="160 heads")
