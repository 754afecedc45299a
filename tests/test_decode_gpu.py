"""GPU parity: attn_decode (paged GQA split-KV decode) through the C ABI against the oracle."""
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


def run_decode(x: inputs.PagedDecodeInputs, scale, workspace=None):
    o, lse = eta.attn_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), x.block_table.cuda(),
                             x.seq_lens.cuda(), scale=scale, workspace=workspace)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
    return o, lse


def oracle_decode(oracle, x: inputs.PagedDecodeInputs, scale, seqs=None):
    """Oracle on the given sequences, with a compact copy of just their blocks
    (the oracle then walks its own block table)."""
    S = x.q.shape[0]
    seqs = list(range(S)) if seqs is None else list(seqs)
    bs = x.block_size
    table = x.block_table.numpy()
    lens = x.seq_lens.numpy()
    used = []
    for s in seqs:
        n = (int(lens[s]) + bs - 1) // bs
        used.extend(int(b) for b in table[s, :n])
    used = sorted(set(used)) or [0]
    remap = {b: i for i, b in enumerate(used)}
    kc = f64(x.k_cache[used])
    vc = f64(x.v_cache[used])
    t2 = np.full((len(seqs), table.shape[1]), -1, dtype=np.int32)
    for r, s in enumerate(seqs):
        n = (int(lens[s]) + bs - 1) // bs
        t2[r, :n] = [remap[int(b)] for b in table[s, :n]]
    return oracle.attn_decode(f64(x.q[seqs]), kc, vc, t2, lens[seqs].astype(np.int32), scale)


def case(oracle, S, Hq, Hkv, d, bs, lens=None, lo=1, hi=1, seed=0, poison=True, what=""):
    x = inputs.decode_inputs(S, Hq, Hkv, d, bs, seq_lens=lens, len_lo=lo, len_hi=hi, seed=seed,
                             extra_blocks=3, poison=poison)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_decode(x, scale)
    o_ref, lse_ref = oracle_decode(oracle, x, scale)
    check_attention(o, lse, o_ref, lse_ref, what)
    return x, o, lse


def test_c5_shape_reduced(oracle):
    c = inputs.C5
    case(oracle, 8, c.Hq, c.Hkv, c.d, c.block_size, lo=1, hi=3000, seed=1, what="C5-like")


LENS = [0, 1, 15, 16, 17, 511, 512, 513, 1023, 1024, 1025, 2049]


@pytest.mark.parametrize("d", [64, 128])
def test_length_boundaries(oracle, d):
    case(oracle, len(LENS), 8, 2, d, 16, lens=LENS, seed=2, what=f"lengths d={d}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (32, 8), (16, 2), (16, 1), (32, 1), (12, 4), (12, 1), (48, 2)])
def test_group_sizes(oracle, Hq, Hkv):
    case(oracle, 5, Hq, Hkv, 128, 16, lo=1, hi=1500, seed=Hq + Hkv, what=f"G={Hq // Hkv}")


@pytest.mark.parametrize("bs", [16, 32, 64, 256])
def test_block_sizes(oracle, bs):
    case(oracle, 6, 8, 2, 128, bs, lo=1, hi=1800, seed=bs, what=f"block_size={bs}")


def test_nan_in_unowned_slots_is_never_used(oracle):
    x, o, lse = case(oracle, 6, 8, 2, 128, 16, lens=[3, 17, 40, 100, 515, 1001], seed=3, poison=True,
                     what="poisoned")
    assert torch.isnan(x.k_cache.float()).any()  # the poison is really there
    assert torch.all(torch.isfinite(o))


def test_identity_table_matches_prefill_last_row():
    """With an identity block table the cache is contiguous per sequence: decode of
    one sequence equals the last row of causal prefill over the same keys."""
    L, Hq, Hkv, d, bs = 777, 8, 2, 128, 16
    x = inputs.decode_inputs(1, Hq, Hkv, d, bs, seq_lens=[L], seed=4, identity_table=True)
    o_dec, lse_dec = run_decode(x, 1 / math.sqrt(d))
    nblk = (L + bs - 1) // bs
    k = x.k_cache[:nblk].permute(1, 0, 2, 3).reshape(Hkv, nblk * bs, d)[:, :L][None]
    v = x.v_cache[:nblk].permute(1, 0, 2, 3).reshape(Hkv, nblk * bs, d)[:, :L][None]
    q = torch.zeros(1, Hq, L, d, dtype=torch.bfloat16)
    q[0, :, L - 1] = x.q[0]
    o_pre, lse_pre = eta.attn_fwd(q.cuda(), k.contiguous().cuda(), v.contiguous().cuda(), causal=True)
    torch.cuda.synchronize()
    assert (o_dec[0].float() - o_pre[0, :, L - 1].float()).abs().max().item() <= 2e-2
    assert (lse_dec[0] - lse_pre[0, :, L - 1]).abs().max().item() <= 1e-3 * max(1.0, lse_pre.abs().max().item())


def test_workspace_reuse_is_deterministic():
    x = inputs.decode_inputs(4, 8, 2, 128, 16, len_lo=100, len_hi=3000, seed=5)
    ws = torch.empty(eta.attn_decode_workspace_size(4, 8, 2, 128, 16, x.block_table.shape[1]), dtype=torch.uint8,
                     device="cuda")
    o1, l1 = run_decode(x, 0.1, workspace=ws)
    o2, l2 = run_decode(x, 0.1, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_block_id_sets_device_error():
    x = inputs.decode_inputs(2, 8, 2, 128, 16, seq_lens=[100, 50], seed=6)
    bt = x.block_table.clone()
    nb = x.k_cache.shape[0]
    bt[0, 2] = nb + 5  # inside sequence 0's length
    eta.attn_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), bt.cuda(), x.seq_lens.cuda())
    assert eta.attn_get_device_error() == -7
    assert eta.attn_get_device_error() == 0  # read clears it
    bt = x.block_table.clone()
    bt[1, 0] = -1
    eta.attn_decode(x.q.cuda(), x.k_cache.cuda(), x.v_cache.cuda(), bt.cuda(), x.seq_lens.cuda())
    assert eta.attn_get_device_error() == -7


def test_full_c5_every_sequence(oracle):
    """The full decode workload as the bench runs it: all 64 sequences (every query head)
    against the oracle, eight sequences per oracle call so that its fp64 copies of the
    cache stay near 2 GB ("Modern attention kernels", "Numerical validation": GQA mapping,
    paged blocks that cross sequence tails)."""
    c = inputs.C5
    x = inputs.decode_config_inputs(c)
    o, lse = run_decode(x, c.scale)
    o, lse = o.cpu(), lse.cpu()
    for s0 in range(0, c.num_seqs, 8):
        seqs = list(range(s0, min(s0 + 8, c.num_seqs)))
        o_ref, lse_ref = oracle_decode(oracle, x, c.scale, seqs)
        check_attention(o[seqs], lse[seqs], o_ref, lse_ref, f"C5 sequences {seqs[0]}-{seqs[-1]}")


def test_more_sequences_than_one_launch_holds(oracle):
    """2500 sequences run as two launches (2048 + 452): sequences on both sides of the cut
    against the oracle, with empty and one-token sequences among them."""
    gen = torch.Generator().manual_seed(21)
    lens = torch.randint(0, 41, (2500,), generator=gen).tolist()
    lens[2047], lens[2048], lens[2499] = 0, 1, 40
    x = inputs.decode_inputs(2500, 8, 2, 64, 16, seq_lens=lens, seed=21, extra_blocks=4, poison=True)
    o, lse = run_decode(x, 0.125)
    seqs = [0, 1, 2, 1000, 2046, 2047, 2048, 2049, 2300, 2499]
    o_ref, lse_ref = oracle_decode(oracle, x, 0.125, seqs=seqs)
    check_attention(o[seqs], lse[seqs], o_ref, lse_ref, "2500 sequences")


def test_counters_left_at_zero_for_the_next_call():
    """A launch puts its completion counters back to zero and zeroes the claim counter the
    next launch of a chain uses: a workspace reused by back-to-back calls of different
    batches gives the same results as fresh workspaces."""
    xa = inputs.decode_inputs(6, 8, 2, 128, 16, len_lo=1, len_hi=3000, seed=22)
    xb = inputs.decode_inputs(3, 8, 2, 128, 16, len_lo=1, len_hi=700, seed=23, max_blocks_per_seq=190)
    ws = torch.zeros(max(eta.attn_decode_workspace_size(6, 8, 2, 128, 16, xa.block_table.shape[1]),
                         eta.attn_decode_workspace_size(3, 8, 2, 128, 16, xb.block_table.shape[1])),
                     dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(128)
    ref_a, ref_b = run_decode(xa, scale), run_decode(xb, scale)
    for _ in range(3):
        for x, ref in ((xa, ref_a), (xb, ref_b)):
            o, lse = run_decode(x, scale, workspace=ws)
            assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])
    # claim counters: the one the next launch would use is zero; completion counters: four
    # per (sequence, kv head), all zero
    torch.cuda.synchronize()
    assert int(ws[8:16].count_nonzero()) == 0
    assert int(ws[16:16 + 4 * 6 * 2 * 4].count_nonzero()) == 0


def test_bounded_wait_reports_timeout_and_context_survives():
    """A barrier wait that nothing completes gives up after its time limit: the host reads
    ATTN_ERR_DEVICE_TIMEOUT, the read clears it, and the next calls run normally."""
    from exact_tiled_attention_06_gb300 import binding
    binding.attn_selftest_wait_timeout()
    assert eta.attn_get_device_error() == -6
    assert eta.attn_get_device_error() == 0
    x = inputs.decode_inputs(3, 8, 2, 128, 16, len_lo=1, len_hi=500, seed=60)
    run_decode(x, 1.0 / math.sqrt(128))
    q, k, v = [t.cuda() for t in inputs.prefill_inputs(1, 2, 1, 130, 130, 64, seed=61)]
    eta.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0


def team_size(S, Hq, Hkv, d, bs, lens):
    """The warps per item the kernel picks: the largest power of two up to d/32 with items x T
    <= worker warps (152 x 8 on a full GB300), counted from the true lengths."""
    mb = max(1, -(-max(lens) // bs))  # the generator's table width
    chunk = eta.attn_decode_chunk_tokens(S, Hq, Hkv, bs, mb)
    HG = Hkv * -(-(Hq // Hkv) // 16)
    items = sum(max(1, -(-L // chunk)) for L in lens) * HG
    n_split_max = -(-(mb * bs) // chunk)
    kmax = d // 32
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    warps = min(sms, -(-(n_split_max * S * HG * kmax) // 8)) * 8
    T = 1
    while T * 2 <= kmax and items * T * 2 <= warps:
        T *= 2
    return T, chunk, items


@pytest.mark.parametrize("S,Hq,Hkv,d,lens,want_T", [
    (3, 8, 2, 128, [1500, 700, 2000], 4),                  # few items: four warps per item
    (8, 64, 8, 128, [600, 610, 590, 620, 605, 598, 615, 601], 2),
    (8, 64, 8, 128, [1500, 1490, 1510, 1480, 1520, 1500, 1470, 1530], 1),
    (3, 8, 2, 64, [1500, 700, 2000], 2),                    # d = 64: two warps at most
    (16, 16, 8, 64, [3000 + 37 * i for i in range(16)], 1),
    (1, 8, 2, 128, [9000], 4),                              # 71 chunks: the merge's long path
    (5, 8, 2, 128, [0, 1, 5, 17, 33], 4),                   # fewer sub-pages than warps per item
    (3, 64, 2, 128, [700, 1300, 90], 4),                    # 32 query heads per kv head: 2 groups
    (2, 32, 8, 128, [4000, 3000], 2),                       # 32 chunks: a slice's merge in two load groups
    (4, 4, 1, 128, [36000, 37000, 39000, 40000], 1),        # 313 chunks: a whole row's merge, long path
])
def test_warp_teams(oracle, S, Hq, Hkv, d, lens, want_T):
    """Items shared by T warps of a block (sub-pages dealt round-robin, partials combined in
    shared memory, the merge split into T column slices) against the oracle, for each T the
    kernel can pick."""
    T, chunk, items = team_size(S, Hq, Hkv, d, 16, lens)
    assert T == want_T, (T, chunk, items)
    case(oracle, S, Hq, Hkv, d, 16, lens=lens, seed=S + Hq + d, what=f"T={T} chunk={chunk} items={items}")


@pytest.mark.parametrize("S", [255, 256, 257])
def test_plan_order_paths(oracle, S):
    """Up to 256 sequences the block orders them by counting, above by a bitonic sort: both
    give the same work plan, so the results agree with the oracle on either side."""
    r = np.random.default_rng(S)
    lens = [int(v) for v in r.integers(0, 300, S)]
    case(oracle, S, 8, 2, 128, 16, lens=lens, seed=S, what=f"S={S}")


@pytest.mark.parametrize("S,Hq,Hkv,d,lo,hi", [
    (3, 8, 2, 128, 1, 2500),      # four warps per item
    (8, 64, 8, 128, 590, 620),    # two warps per item
    (3, 8, 2, 64, 1, 2500),       # d = 64, two warps per item
    (16, 16, 8, 64, 2900, 3500),  # one warp per item
    (300, 8, 2, 128, 0, 300),     # the bitonic-sort plan, empty sequences among them
])
def test_repeated_launches_are_bitwise_identical(S, Hq, Hkv, d, lo, hi):
    """Claims, team combines and per-slice merges race for nothing: thirty launches on one
    workspace give the same bits."""
    x = inputs.decode_inputs(S, Hq, Hkv, d, 16, len_lo=lo, len_hi=hi, seed=S + d)
    args = [t.cuda() for t in (x.q, x.k_cache, x.v_cache, x.block_table, x.seq_lens)]
    ws = torch.empty(eta.attn_decode_workspace_size(S, Hq, Hkv, d, 16, x.block_table.shape[1]), dtype=torch.uint8,
                     device="cuda")
    o0, l0 = eta.attn_decode(*args, workspace=ws)
    for _ in range(30):
        o, lse = eta.attn_decode(*args, workspace=ws)
        assert torch.equal(o, o0) and torch.equal(lse, l0)
    torch.cuda.synchronize()
    assert eta.attn_get_device_error() == 0
