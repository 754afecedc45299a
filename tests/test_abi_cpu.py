"""CPU: the C-ABI library builds for sm_103a, loads without a GPU, exports every
symbol include/attn.h declares, and rejects bad arguments before any launch."""
import ctypes
import json
import os
import re

import pytest

import exact_tiled_attention_06_gb300 as eta
from exact_tiled_attention_06_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    eta.build()
    return eta.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_layout_version_and_status_strings(lib):
    assert eta.attn_kv_layout_version() == 1
    for code, name in binding.STATUS_NAMES.items():
        assert eta.attn_status_string(code) == name


FAKE = 0x7F0000000000  # never dereferenced: every call below fails validation first


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=64, scale=0.125,
        causal=0, window=-1):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, window, None)


def test_fwd_argument_validation(lib):
    assert fwd(lib, q=None) == -1
    assert fwd(lib, lse=None) == -1
    assert fwd(lib, B=0) == -1
    assert fwd(lib, Hq=3, Hkv=2) == -1       # Hq % Hkv != 0
    assert fwd(lib, Nq=-1) == -1
    assert fwd(lib, scale=0.0) == -1
    assert fwd(lib, scale=float("nan")) == -1
    assert fwd(lib, d=96) == -2
    assert fwd(lib, d=256) == -2
    assert fwd(lib, q=FAKE + 8) == -3        # not 16-byte aligned
    assert fwd(lib, lse=FAKE + 2) == -3
    assert fwd(lib, Nq=0) == 0               # nothing to do: no launch


def bwd(lib, ws_bytes=None, q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, Hq=4,
        Hkv=2, Nq=200, Nk=300, d=128, scale=0.1, causal=1, window=-1, ws=FAKE):
    if ws_bytes is None:
        ws_bytes = lib.attn_bwd_workspace_size(B, Hq, Nq, d)
    return lib.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, window, ws, ws_bytes,
                        None)


def test_bwd_argument_validation(lib):
    assert bwd(lib, q=None) == -1
    assert bwd(lib, do=None) == -1
    assert bwd(lib, dk=None) == -1
    assert bwd(lib, Hq=3, Hkv=2) == -1
    assert bwd(lib, Nk=-1) == -1
    assert bwd(lib, scale=float("inf")) == -1
    assert bwd(lib, d=96) == -2
    assert bwd(lib, dq=FAKE + 2) == -3
    assert bwd(lib, lse=FAKE + 1) == -3
    assert bwd(lib, ws_bytes=64) == -4
    assert bwd(lib, ws=None) == -4
    assert bwd(lib, ws=FAKE + 8) == -3
    # no queries: q, o, dout, lse, dq may be null (k, v, dk, dv are still needed)
    assert bwd(lib, Nq=0, q=None, o=None, do=None, lse=None, dq=None, k=None) == -1
    # no queries and no keys: nothing to do
    assert bwd(lib, Nq=0, Nk=0, q=None, o=None, do=None, lse=None, dq=None, k=None, v=None, dk=None,
               dv=None) == 0


def test_bwd_workspace_size(lib):
    """D_i rows (fp32, padded to 256 bytes), then the fp32 dQ accumulator."""
    up = lambda x: -(-x // 256) * 256
    for B, Hq, Nq, d in ((1, 4, 200, 128), (2, 3, 77, 64), (1, 1, 1, 64)):
        rows = B * Hq * Nq
        assert eta.attn_bwd_workspace_size(B, Hq, Nq, d) == up(rows * 4) + rows * d * 4
    assert eta.attn_bwd_workspace_size(1, 4, 200, 96) == 0
    assert eta.attn_bwd_workspace_size(0, 4, 200, 64) == 0


def bsp(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, Nq=300, Nk=300, d=64, scale=0.125, causal=1,
        window=-1, rp=FAKE, ci=FAKE):
    return lib.attn_fwd_blocksparse(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, window, rp, ci, None)


def test_fwd_blocksparse_argument_validation(lib):
    assert bsp(lib, rp=None) == -1
    assert bsp(lib, ci=None) == -1
    assert bsp(lib, q=None) == -1
    assert bsp(lib, Hq=3, Hkv=2) == -1
    assert bsp(lib, scale=-0.5) == -1
    assert bsp(lib, d=80) == -2
    assert bsp(lib, Nk=262145) == -2          # the merged walk holds 2048 key blocks per tile
    assert bsp(lib, rp=FAKE + 2) == -3
    assert bsp(lib, o=FAKE + 4) == -3
    assert bsp(lib, Nq=0) == 0


def ppf(lib, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, ql=FAKE, kl=FAKE, o=FAKE, lse=FAKE, S=4, Hq=8, Hkv=2, d=128, bs=16,
        mb=64, nb=256, max_q=300, scale=0.1, causal=1, window=-1):
    return lib.attn_prefill_paged(q, kc, vc, bt, ql, kl, o, lse, S, Hq, Hkv, d, bs, mb, nb, max_q, scale, causal,
                                  window, None)


def test_prefill_paged_argument_validation(lib):
    assert ppf(lib, q=None) == -1
    assert ppf(lib, kl=None) == -1
    assert ppf(lib, Hq=6, Hkv=4) == -1
    assert ppf(lib, nb=0) == -1
    assert ppf(lib, max_q=-1) == -1
    assert ppf(lib, scale=0.0) == -1
    assert ppf(lib, d=32) == -2
    assert ppf(lib, bs=8) == -2              # below 16
    assert ppf(lib, bs=48) == -2             # not a power of two
    assert ppf(lib, bs=512) == -2            # above 256
    assert ppf(lib, nb=1 << 26) == -2        # cache rows past 2^31
    assert ppf(lib, o=FAKE + 8) == -3
    assert ppf(lib, ql=FAKE + 2) == -3
    assert ppf(lib, S=0) == 0                # nothing to do: no launch
    assert ppf(lib, max_q=0) == 0


def dec(lib, ws_bytes=None, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, o=FAKE, lse=FAKE, S=4, Hq=8, Hkv=2, d=128,
        bs=16, mb=64, nb=256, scale=0.1, ws=FAKE):
    if ws_bytes is None:
        ws_bytes = lib.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb)
    return lib.attn_decode(q, kc, vc, bt, sl, o, lse, S, Hq, Hkv, d, bs, mb, nb, scale, ws, ws_bytes, None)


def fp8(lib, q=FAKE, k=FAKE, vt=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, Nq=8, Nk=16, d=128, scale=0.1, qs=0.01,
        ks=0.01, vs=0.01, causal=0, window=-1):
    return lib.attn_fwd_fp8(q, k, vt, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, qs, ks, vs, causal, window, None)


def test_fp8_argument_validation(lib):
    assert fp8(lib, q=None) == -1
    assert fp8(lib, vt=None) == -1
    assert fp8(lib, vt=None, k=None, Nk=0, Nq=0) == 0   # no keys: k and vt are never read
    assert fp8(lib, Hq=3, Hkv=2) == -1
    assert fp8(lib, qs=0.0) == -1
    assert fp8(lib, ks=float("inf")) == -1
    assert fp8(lib, vs=-1.0) == -1
    assert fp8(lib, d=64) == -2                        # d = 128 only
    assert fp8(lib, Nk=100) == -2                      # V^T rows must stay 16-byte aligned
    assert fp8(lib, vt=FAKE + 8) == -3
    assert fp8(lib, Nq=0) == 0                         # nothing to compute: no launch


def test_host_entry_points_validation(lib):
    F = FAKE
    fh = lambda **kw: lib.attn_fwd_host(*(kw.get(n, F) for n in ("qh", "kh", "vh", "oh", "lh", "qd", "kd", "vd", "od",
                                                                  "ld")), 1, 2, 1, kw.get("Nq", 8), 16,
                                        kw.get("d", 128), 0.1, 0, -1, 0, None)
    assert fh(qh=None) == -1
    assert fh(kd=None) == -1
    assert fh(d=80) == -2
    assert fh(od=F + 8) == -3
    assert fh(Nq=0, qh=None, oh=None, lh=None, qd=None, od=None, ld=None) == 0
    ws = lib.attn_decode_workspace_size(4, 8, 2, 128, 16, 64)
    dh = lambda **kw: lib.attn_decode_host(*(kw.get(n, F) for n in ("qh", "kh", "vh", "bh", "sh", "oh", "lh", "qd",
                                                                     "kd", "vd", "bd", "sd", "od", "ld")), 4, 8, 2,
                                           kw.get("d", 128), kw.get("bs", 16), 64, 256, 0.1, F, kw.get("wsb", ws), None)
    assert dh(sh=None) == -1
    assert dh(vd=None) == -1
    assert dh(bs=24) == -2
    assert dh(ld=F + 2) == -3
    assert dh(wsb=16) == -4


def test_decode_argument_validation(lib):
    assert dec(lib, q=None) == -1
    assert dec(lib, bt=None) == -1
    assert dec(lib, Hq=6, Hkv=4) == -1
    assert dec(lib, nb=0) == -1
    assert dec(lib, scale=-1.0) == -1
    assert dec(lib, d=80) == -2
    assert dec(lib, bs=8) == -2               # block size must be a multiple of 16
    assert dec(lib, bs=24) == -2
    assert dec(lib, bs=512) == -2
    assert dec(lib, nb=1 << 26) == -2         # cache rows past 2^31
    assert dec(lib, kc=FAKE + 4) == -3
    assert dec(lib, ws_bytes=16) == -4        # workspace too small
    assert dec(lib, ws=None) == -4
    assert dec(lib, S=0) == 0                 # empty batch: no launch


def test_noalloc_decode_validates_like_decode(lib):
    """attn_decode_noalloc shares attn_decode's argument checks: the same bad arguments give
    the same status, before any CUDA call (no GPU here)."""
    cases = [dict(q=None), dict(bt=None), dict(Hq=6, Hkv=4), dict(nb=0), dict(scale=-1.0), dict(d=80), dict(bs=8),
             dict(bs=24), dict(bs=512), dict(nb=1 << 26), dict(kc=FAKE + 4), dict(lse=FAKE + 2), dict(S=-1),
             dict(S=70000), dict(mb=-1), dict(S=0)]
    for kw in cases:
        a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, o=FAKE, lse=FAKE, S=4, Hq=8, Hkv=2, d=128, bs=16, mb=64,
                 nb=256, scale=0.1)
        a.update(kw)
        want = dec(lib, **kw)
        got = lib.attn_decode_noalloc(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["o"], a["lse"], a["S"], a["Hq"],
                                      a["Hkv"], a["d"], a["bs"], a["mb"], a["nb"], a["scale"], None)
        assert got == want, (kw, got, want)
    # partials beyond the 64 MiB static scratch: rejected before any CUDA call
    assert lib.attn_decode_workspace_size(64, 32, 8, 128, 16, 2048) > 64 << 20
    assert lib.attn_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 32, 8, 128, 16, 2048, 1000, 0.1,
                                   None) == -4


def graph_create(lib, n=2, bad_layer=None, field=None, value=None, S=4, Hq=8, Hkv=2, d=128, bs=16, mb=64, nb=256,
                 scale=0.1, ws=FAKE, ws_bytes=None, out_ptr=True):
    """attn_decode_graph_create with fake pointers; (field, value) replaces one pointer of
    layer ``bad_layer`` (q, kc, vc, o, lse)."""
    if ws_bytes is None:
        ws_bytes = lib.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb)
    arrs = {}
    for name in ("q", "kc", "vc", "o", "lse"):
        vals = [FAKE] * max(n, 1)
        if name == field and bad_layer is not None:
            vals[bad_layer] = value
        arrs[name] = (ctypes.c_void_p * len(vals))(*vals)
    h = ctypes.c_void_p(0x1234)
    rc = lib.attn_decode_graph_create(n, arrs["q"], arrs["kc"], arrs["vc"], arrs["o"], arrs["lse"], FAKE, FAKE, S, Hq,
                                      Hkv, d, bs, mb, nb, scale, ws, ws_bytes, ctypes.byref(h) if out_ptr else None)
    return rc, h.value


def test_decode_graph_argument_validation(lib):
    """Every layer's pointers are checked before any CUDA call; the handle is NULL on failure."""
    assert graph_create(lib, n=0) == (-1, None)
    assert graph_create(lib, n=5000) == (-1, None)
    assert graph_create(lib, out_ptr=False)[0] == -1
    assert graph_create(lib, n=3, bad_layer=2, field="vc", value=None) == (-1, None)
    assert graph_create(lib, n=3, bad_layer=1, field="kc", value=FAKE + 4) == (-3, None)
    assert graph_create(lib, n=3, bad_layer=2, field="lse", value=FAKE + 2) == (-3, None)
    assert graph_create(lib, d=80) == (-2, None)
    assert graph_create(lib, bs=24) == (-2, None)
    assert graph_create(lib, Hq=6, Hkv=4) == (-1, None)
    assert graph_create(lib, ws_bytes=16) == (-4, None)
    assert graph_create(lib, ws=FAKE + 8) == (-3, None)
    assert lib.attn_decode_graph_launch(None, None) == -1
    assert lib.attn_decode_graph_layers(None) == 0
    assert lib.attn_decode_graph_destroy(None) == 0


def test_workspace_size_matches_split_plan(lib):
    """Counters (two 8-byte claim counters, four ints per (sequence, kv head): one per
    column slice a team of up to four warps merges), then the fp32 partial log-sums and partial outputs of
    every possible split, 256-byte aligned."""
    S, Hq, Hkv, d, bs, mb = 64, 32, 8, 128, 16, 2048
    chunk = eta.attn_decode_chunk_tokens(S, Hq, Hkv, bs, mb)
    n_split = -(-mb * bs // chunk)
    rows = n_split * S * Hq
    up = lambda x: -(-x // 256) * 256
    want = up(16 + 4 * S * Hkv * 4) + up(rows * 4) + rows * d * 4
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb) == want
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, 96, bs, mb) == 0
    assert chunk % bs == 0 and chunk % 16 == 0


def test_split_plan_halves_chunk_for_small_batches(lib):
    """Fewer items than worker warps (1216): the chunk halves, down to 128 keys, staying a
    multiple of the block size; large batches keep 512."""
    def items(S, Hq, Hkv, bs, mb):
        chunk = eta.attn_decode_chunk_tokens(S, Hq, Hkv, bs, mb)
        return chunk, -(-mb * bs // chunk) * S * Hkv * -(-(Hq // Hkv) // 16)
    assert items(64, 32, 8, 16, 2048)[0] == 512           # the long decode workload
    chunk, n = items(8, 32, 8, 16, 125)                    # 8 sequences of <= 2000 tokens
    assert chunk == 128 and n == 16 * 8 * 8                # the floor: 1024 items
    chunk, n = items(8, 32, 8, 16, 250)                    # <= 4000 tokens
    assert chunk == 128 and n == 32 * 8 * 8                # 256 would give 16 x 64 = 1024 items
    assert items(1, 8, 1, 16, 4)[0] == 128                 # tiny: floor of 128 keys
    assert items(1, 8, 1, 128, 4)[0] == 128                # stays a multiple of a 128-token block
    assert items(1, 8, 1, 256, 4)[0] == 256
    assert items(2, 64, 2, 16, 64)[0] == 128               # 32 query heads per kv head: 2 groups
    assert items(80, 64, 2, 16, 64)[0] == 256              # 80 seqs x 2 kv x 2 groups x 4 splits = 1280
    # the workspace follows the plan
    S, Hq, Hkv, d, bs, mb = 8, 32, 8, 128, 16, 125
    rows = (mb * bs // 128 + (mb * bs % 128 > 0)) * S * Hq
    up = lambda x: -(-x // 256) * 256
    assert eta.attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb) == up(16 + 4 * S * Hkv * 4) + up(rows * 4) + rows * d * 4


def test_split_plan_reproduces_flashdecoding_example(lib):
    with open(os.path.join(GOLDEN, "flashdecoding_split_example.json")) as f:
        g = json.load(f)
    mb = g["kv_len"] // g["block_size"]
    chunk = eta.attn_decode_chunk_tokens(g["batch"], g["heads"], g["heads"], g["block_size"], mb)
    assert chunk == g["chunk"]
    n_split = g["kv_len"] // chunk
    assert n_split == g["chunks"]
    assert g["batch"] * g["heads"] == g["units_without_split"]
    assert (g["batch"] * g["heads"] * n_split) // g["units_without_split"] == g["parallelism_gain"]


def test_product_path_has_no_oracle_import():
    """The CUDA path never touches the CPU oracle (no fallback, no shared code)."""
    pkg = os.path.dirname(eta.__file__)
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), fn
                assert "liboracle" not in text and "attn_oracle" not in text, fn
