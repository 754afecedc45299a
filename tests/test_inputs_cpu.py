"""CPU: the seeded input generators -- determinism, shapes, and the structure each workload
promises (shared tables, owned slots, NaN only where no sequence reads)."""
import torch

from exact_tiled_attention_06_gb300 import inputs


def test_decode_step_layers_share_table_and_differ_in_data():
    x = inputs.decode_step_inputs(4, 3, 8, 2, 64, 16, len_lo=1, len_hi=200, seed=5, extra_blocks=2, poison=True)
    base = inputs.decode_inputs(3, 8, 2, 64, 16, len_lo=1, len_hi=200, seed=5, extra_blocks=2, poison=True)
    assert torch.equal(x.block_table, base.block_table) and torch.equal(x.seq_lens, base.seq_lens)
    assert torch.equal(x.q[0], base.q)
    assert torch.equal(torch.nan_to_num(x.k_cache[0]), torch.nan_to_num(base.k_cache))
    nan0 = torch.isnan(x.k_cache[0])
    for l in range(1, 4):
        assert torch.equal(torch.isnan(x.k_cache[l]), nan0) and torch.equal(torch.isnan(x.v_cache[l]), nan0)
        assert not torch.equal(x.q[l], x.q[0])
        assert not torch.equal(torch.nan_to_num(x.k_cache[l]), torch.nan_to_num(x.k_cache[0]))
    # 4 layers x sum L tokens x Hkv (2) x d (64) x 2 bytes x (K and V)
    assert x.kv_bytes == 4 * int(x.seq_lens.sum()) * 2 * 64 * 2 * 2


def test_decode_step_is_deterministic_and_owned_slots_are_finite():
    a = inputs.decode_step_inputs(3, 4, 8, 2, 128, 16, len_lo=1, len_hi=100, seed=7, poison=True)
    b = inputs.decode_step_inputs(3, 4, 8, 2, 128, 16, len_lo=1, len_hi=100, seed=7, poison=True)
    for l in range(3):
        assert torch.equal(a.q[l], b.q[l])
        assert torch.equal(torch.nan_to_num(a.v_cache[l]), torch.nan_to_num(b.v_cache[l]))
        for s in range(4):
            L = int(a.seq_lens[s])
            for t in range(L):
                blk = int(a.block_table[s, t // 16])
                assert torch.isfinite(a.k_cache[l][blk, :, t % 16]).all()


def test_c8_workload_shape():
    c = inputs.C8
    assert (c.n_layers, c.num_seqs, c.Hq, c.Hkv, c.d, c.block_size) == (32, 8, 32, 8, 128, 16)
    assert c.name in inputs.DECODE_STEP_CONFIGS
