"""CPU: the benchmark's FLOP and byte accounting against the figures the pages print."""
import json
import os

import numpy as np

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_figures.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_score_matrix_sizes_match_memory_table():
    g = golden()["score_matrix_mib_bf16"]
    for n, mib in g["values"].items():
        assert round(bench.score_matrix_bytes(int(n)) / 2 ** 20, 1) == mib


def test_score_matrix_mb_per_head():
    g = golden()
    assert bench.score_matrix_bytes(4096) / 2 ** 20 == g["score_matrix_mb_4096"]["value"]
    assert round(bench.score_matrix_bytes(8192) / 1e6) == g["score_matrix_mb_8192"]["value"]


def test_naive_traffic_and_time_estimate():
    g = golden()["naive_prefill_traffic"]
    b = bench.naive_score_traffic_bytes(g["N"], g["heads"], g["layers"])
    assert int(b / 1e9) == g["gb"]
    assert round(b / (g["hbm_tbs"] * 1e12) * 1e3) == g["ms"]


def test_flops_per_head():
    # 4 N^2 d per head without a mask; causal keeps N (N + 1) / 2 pairs
    N, d = 8192, 128
    assert bench.attention_flops(1, 1, N, N, d) == 4 * N * N * d
    assert bench.attention_flops(1, 1, N, N, d, causal=True) == 4 * d * N * (N + 1) // 2
    # window w (with causal): row i keeps min(i, w) + 1 keys
    w = 1024
    want = sum(min(i, w) + 1 for i in range(4096))
    assert bench.allowed_pairs(4096, 4096, True, w) == want


def test_decode_bytes():
    assert bench.decode_kv_bytes([1024, 2048], 8, 128) == (1024 + 2048) * 8 * 128 * 2 * 2


def test_backward_flops_are_five_matmuls():
    """Backward: 5 matmuls of 2 d FLOPs per allowed pair, 2.5 x the forward's 2."""
    for args in ((1, 32, 8192, 8192, 128, True, -1), (2, 32, 4096, 4096, 128, True, 1024), (1, 1, 7, 13, 64, False, -1)):
        assert bench.backward_flops(*args) * 2 == bench.attention_flops(*args) * 5
    # one head, no mask: 10 N^2 d
    assert bench.backward_flops(1, 1, 64, 64, 128) == 10 * 64 * 64 * 128


def test_paged_prefill_flops():
    """Per sequence, the prefill count with Nq = q_len and Nk = kv_len."""
    q, kv = [2048, 5, 0, 1], [4096, 5, 7, 9000]
    want = sum(bench.attention_flops(1, 32, a, b, 128, True) for a, b in zip(q, kv))
    assert bench.paged_prefill_flops(q, kv, 32, 128, True) == want
    # a whole prompt (q_len = kv_len) equals causal prefill; one query sees every key
    assert bench.paged_prefill_flops([300], [300], 4, 64, True) == bench.attention_flops(1, 4, 300, 300, 64, True)
    assert bench.paged_prefill_flops([1], [77], 1, 64, True) == 4 * 64 * 77


def test_blocksparse_pairs():
    """A full pattern counts the dense mask's pairs; a block-diagonal one counts the blocks."""
    for Nq, Nk, causal, window in ((300, 300, True, -1), (200, 450, True, 100), (257, 129, False, -1)):
        nq, nk = -(-Nq // 128), -(-Nk // 128)
        full = np.ones((nq, nk), dtype=bool)
        assert bench.blocksparse_pairs(full, Nq, Nk, causal, window) == bench.allowed_pairs(Nq, Nk, causal, window)
    eye = np.eye(3, dtype=bool)
    assert bench.blocksparse_pairs(eye, 384, 384, False, -1) == 3 * 128 * 128
    assert bench.blocksparse_pairs(eye, 384, 384, True, -1) == 3 * 128 * 129 // 2


def test_traffic_records_are_well_formed(monkeypatch):
    """Every DRAM-traffic record names a kernel whose sources the bench hashes, and the bench
    reports a record's bytes only while those sources are the ones it was captured on."""
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                        "dram_traffic.json")
    with open(path) as f:
        records = {k: v for k, v in json.load(f).items() if not k.startswith("_")}
    assert records
    for name, rec in records.items():
        assert name in bench.KERNEL_SOURCES, name
        assert isinstance(rec["bytes_per_launch"], int) and rec["bytes_per_launch"] > 0, name
        assert len(rec["source_hash"]) == 16 and int(rec["source_hash"], 16) >= 0, name
        assert rec["case"], name
        monkeypatch.setattr(bench, "kernel_source_hash", lambda k, h=rec["source_hash"]: h)
        assert bench.load_traffic(name) == float(rec["bytes_per_launch"])
        monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
        assert bench.load_traffic(name) is None
    # decode: within a few percent of the algorithmic bytes it was captured against
    assert 1.0 < records["attn_decode_sm103"]["bytes_per_launch"] / 3884961792 < 1.05
    assert 1.0 < records["attn_decode_sm103_c8_step"]["bytes_per_launch"] / 1071251456 < 1.05
