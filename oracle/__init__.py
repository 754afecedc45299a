"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``exact_tiled_attention_06_gb300``) never imports
it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over independent rows). This module only compiles it with gcc and marshals
numpy arrays through ctypes. Every function takes and returns float64 arrays.

What each function follows (pages by title and section):

* ``attn_fwd`` / ``attn_fwd_rows`` -- the plain definition, with the score and
  probability rows materialised: "Modern attention kernels",
  "Standard attention materializes quadratic state"; safe softmax from
  "Attention kernels" (the safe-softmax derivation).
* ``attn_fwd_blocked`` -- the query-outer blocked online-softmax loop of
  "Flash attention and IO-aware attention" (its code listing) with the
  unnormalised accumulator and one final divide of "Modern attention kernels",
  "Online softmax makes tiling exact".
* ``attn_fwd_split`` -- per-chunk partials merged with the two-partial
  rescaling of "Attention kernels" (FlashDecoding).
* ``attn_bwd`` -- gradients of attention by the chain rule with the probability rows
  recomputed ("Modern attention kernels", "Backward pass recomputes scores").
* ``attn_decode`` -- one query per sequence over a paged cache, addressed with
  the block-table formula of "Modern attention kernels",
  "Paged attention changes addressing".
* ``attn_fwd_blocksparse`` -- prefill restricted to the score blocks a CSR block index
  lists ("Modern attention kernels", "Kernel structure" and the table of variants),
  materialised per row with the block membership added to the mask.
* ``attn_prefill_paged`` -- several new queries per sequence over a paged cache
  (chunked prefill): the keys are gathered with the same formula and each new row
  goes through the materialised row routine, bottom-right causal.

Pins: every function is checked in ``tests/test_oracle_pins.py`` against
closed forms, invariants, brute force on tiny inputs and a hand-derived golden
example; ``tests/test_oracle_mutants.py`` plants mistakes in a copy of the C
source and checks that the pins catch them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.POINTER(ctypes.c_int64)


def compile_source(src: str, out: str) -> None:
    """Compile one oracle C source into a shared library with gcc + OpenMP."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-Wall", "-shared", "-fPIC", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` (once) and return the library path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    c_int, c_double = ctypes.c_int, ctypes.c_double
    lib.oracle_attn_fwd.argtypes = [_D, _D, _D, _D, _D] + [c_int] * 6 + [c_double, c_int, c_int]
    lib.oracle_attn_fwd_rows.argtypes = [_D, _D, _D] + [c_int] * 6 + [c_double, c_int, c_int, _I64,
                                                                        ctypes.c_int64, _D, _D]
    lib.oracle_attn_fwd_blocked.argtypes = [_D, _D, _D, _D, _D] + [c_int] * 6 + [c_double, c_int, c_int,
                                                                                 c_int, c_int]
    lib.oracle_attn_fwd_split.argtypes = [_D, _D, _D, _D, _D] + [c_int] * 6 + [c_double, c_int, c_int, c_int]
    lib.oracle_attn_decode.argtypes = [_D, _D, _D, _I32, _I32, _D, _D] + [c_int] * 7 + [c_double]
    lib.oracle_attn_bwd.argtypes = [_D] * 7 + [c_int] * 6 + [c_double, c_int, c_int]
    lib.oracle_attn_fwd_blocksparse.argtypes = [_D] * 5 + [c_int] * 6 + [c_double, c_int, c_int, _I32, _I32, c_int,
                                                                             c_int]
    lib.oracle_attn_prefill_paged.argtypes = [_D, _D, _D, _I32, _I32, _I32, _D, _D] + [c_int] * 8 + [c_double, c_int,
                                                                                                   c_int]
    _U8 = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = c_double
    lib.oracle_e4m3_decode.argtypes = [_U8, _D, ctypes.c_int64]
    lib.oracle_attn_fwd_fp8.argtypes = [_U8, _U8, _U8, _D, _D] + [c_int] * 6 + [c_double] * 4 + [c_int, c_int]
    lib.oracle_num_threads.argtypes = []
    for f in (lib.oracle_attn_fwd, lib.oracle_attn_fwd_rows, lib.oracle_attn_fwd_blocked,
              lib.oracle_attn_fwd_split, lib.oracle_attn_decode, lib.oracle_attn_bwd, lib.oracle_attn_prefill_paged,
              lib.oracle_attn_fwd_blocksparse, lib.oracle_num_threads):
        f.restype = c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed).

    ``path`` lets a test load a separately compiled copy of the source."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _pu8(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (status {rc})")


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B][H][N][d]")
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, dk) != (B, d) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k, v")
    return B, Hq, Hkv, Nq, Nk, d


class Oracle:
    """Thin marshalling layer over one loaded oracle library."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def attn_fwd(self, q, k, v, scale, causal=False, window=-1):
        """Materialised attention. Returns (o [B][Hq][Nq][d], lse [B][Hq][Nq])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Nq, Nk, d = _shapes(q, k, v)
        o = np.zeros((B, Hq, Nq, d))
        lse = np.zeros((B, Hq, Nq))
        _check(self.lib.oracle_attn_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Nq, Nk, d,
                                        float(scale), int(bool(causal)), int(window)), "oracle_attn_fwd")
        return o, lse

    def attn_fwd_rows(self, q, k, v, rows, scale, causal=False, window=-1):
        """Materialised attention for selected rows ``rows`` = int [n][3] of (b, hq, i)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Nq, Nk, d = _shapes(q, k, v)
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        n = rows.shape[0]
        o = np.zeros((n, d))
        lse = np.zeros((n,))
        _check(self.lib.oracle_attn_fwd_rows(_p(q), _p(k), _p(v), B, Hq, Hkv, Nq, Nk, d, float(scale),
                                             int(bool(causal)), int(window), rows.ctypes.data_as(_I64),
                                             n, _p(o), _p(lse)), "oracle_attn_fwd_rows")
        return o, lse

    def attn_fwd_blocked(self, q, k, v, scale, causal=False, window=-1, block_r=128, block_c=128):
        """Blocked online-softmax attention (query blocks outer, key/value blocks inner)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Nq, Nk, d = _shapes(q, k, v)
        o = np.zeros((B, Hq, Nq, d))
        lse = np.zeros((B, Hq, Nq))
        _check(self.lib.oracle_attn_fwd_blocked(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Nq, Nk, d,
                                                float(scale), int(bool(causal)), int(window),
                                                int(block_r), int(block_c)), "oracle_attn_fwd_blocked")
        return o, lse

    def attn_fwd_split(self, q, k, v, scale, causal=False, window=-1, chunk=512):
        """Split-KV attention: per-chunk partials merged by the two-partial rescaling."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Nq, Nk, d = _shapes(q, k, v)
        o = np.zeros((B, Hq, Nq, d))
        lse = np.zeros((B, Hq, Nq))
        _check(self.lib.oracle_attn_fwd_split(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Nq, Nk, d,
                                              float(scale), int(bool(causal)), int(window), int(chunk)),
               "oracle_attn_fwd_split")
        return o, lse

    def e4m3_decode(self, codes):
        """Real values of 8-bit E4M3 codes (uint8 array, any shape)."""
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.zeros(c.shape, dtype=np.float64)
        _check(self.lib.oracle_e4m3_decode(_pu8(c), _p(out), c.size), "oracle_e4m3_decode")
        return out

    def attn_fwd_fp8(self, q8, k8, vt8, scale, q_descale, k_descale, v_descale, causal=False, window=-1):
        """Attention over E4M3 codes: q8 [B][Hq][Nq][d], k8 [B][Hkv][Nk][d], vt8 [B][Hkv][d][Nk]
        (uint8), real values = code value x the tensor's descale. Returns (o, lse) in fp64."""
        q8 = np.ascontiguousarray(q8, dtype=np.uint8)
        k8 = np.ascontiguousarray(k8, dtype=np.uint8)
        vt8 = np.ascontiguousarray(vt8, dtype=np.uint8)
        B, Hq, Nq, d = q8.shape
        Bk, Hkv, Nk, dk = k8.shape
        if Bk != B or dk != d or vt8.shape != (B, Hkv, d, Nk):
            raise ValueError("fp8 shapes disagree")
        o = np.zeros((B, Hq, Nq, d))
        lse = np.zeros((B, Hq, Nq))
        _check(self.lib.oracle_attn_fwd_fp8(_pu8(q8), _pu8(k8), _pu8(vt8), _p(o), _p(lse), B, Hq,
                                            Hkv, Nq, Nk, d, float(scale), float(q_descale), float(k_descale),
                                            float(v_descale), int(bool(causal)), int(window)), "oracle_attn_fwd_fp8")
        return o, lse

    def attn_bwd(self, q, k, v, dout, scale, causal=False, window=-1):
        """Gradients (dq, dk, dv) of sum(dout * O) for O = attention(q, k, v), materialised."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, Hq, Hkv, Nq, Nk, d = _shapes(q, k, v)
        if dout.shape != q.shape:
            raise ValueError("dout must have the shape of q")
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        _check(self.lib.oracle_attn_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), B, Hq, Hkv, Nq,
                                        Nk, d, float(scale), int(bool(causal)), int(window)), "oracle_attn_bwd")
        return dq, dk, dv

    def attn_fwd_blocksparse(self, q, k, v, row_ptr, col_idx, scale, causal=False, window=-1, block_q=128,
                             block_k=128):
        """Block-sparse attention: (row_ptr, col_idx) list the key blocks of each query block."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Nq, Nk, d = _shapes(q, k, v)
        rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
        ci = np.ascontiguousarray(col_idx, dtype=np.int32)
        if rp.shape != ((Nq + block_q - 1) // block_q + 1,):
            raise ValueError("row_ptr must have one entry per query block plus one")
        if ci.size == 0:
            ci = np.zeros(1, dtype=np.int32)
        o = np.zeros((B, Hq, Nq, d))
        lse = np.zeros((B, Hq, Nq))
        _check(self.lib.oracle_attn_fwd_blocksparse(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Nq, Nk, d,
                                                    float(scale), int(bool(causal)), int(window),
                                                    rp.ctypes.data_as(_I32), ci.ctypes.data_as(_I32), int(block_q),
                                                    int(block_k)), "oracle_attn_fwd_blocksparse")
        return o, lse

    def attn_prefill_paged(self, q, k_cache, v_cache, block_table, q_lens, kv_lens, scale, causal=True, window=-1):
        """Paged prefill. q [S][Hq][max_q][d]; caches [num_blocks][Hkv][bs][d]; block_table int32
        [S][max_blocks]; q_lens, kv_lens int32 [S]. Returns (o, lse) shaped like q and [S][Hq][max_q];
        rows i >= q_lens[s] are zero in o and NaN in lse (not computed)."""
        q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        ql = np.ascontiguousarray(q_lens, dtype=np.int32)
        kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
        S, Hq, max_q, d = q.shape
        nb, Hkv, bs, dk = kc.shape
        if dk != d or vc.shape != kc.shape or bt.ndim != 2 or bt.shape[0] != S or ql.shape != (S,) or kl.shape != (S,):
            raise ValueError("paged prefill shape mismatch")
        o = np.zeros(q.shape)
        lse = np.full((S, Hq, max_q), np.nan)
        _check(self.lib.oracle_attn_prefill_paged(_p(q), _p(kc), _p(vc), bt.ctypes.data_as(_I32),
                                                  ql.ctypes.data_as(_I32), kl.ctypes.data_as(_I32), _p(o), _p(lse),
                                                  S, Hq, Hkv, d, bs, bt.shape[1], nb, max_q, float(scale),
                                                  int(bool(causal)), int(window)), "oracle_attn_prefill_paged")
        return o, lse

    def attn_decode(self, q, k_cache, v_cache, block_table, seq_lens, scale):
        """Paged one-query decode. q [S][Hq][d]; caches [num_blocks][Hkv][bs][d];
        block_table int32 [S][max_blocks]; seq_lens int32 [S]. Returns (o [S][Hq][d], lse [S][Hq])."""
        q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        S, Hq, d = q.shape
        nb, Hkv, bs, dk = kc.shape
        if dk != d or vc.shape != kc.shape or bt.ndim != 2 or bt.shape[0] != S or sl.shape != (S,):
            raise ValueError("decode shape mismatch")
        o = np.zeros((S, Hq, d))
        lse = np.zeros((S, Hq))
        _check(self.lib.oracle_attn_decode(_p(q), _p(kc), _p(vc), bt.ctypes.data_as(_I32),
                                           sl.ctypes.data_as(_I32), _p(o), _p(lse), S, Hq, Hkv, d, bs,
                                           bt.shape[1], nb, float(scale)), "oracle_attn_decode")
        return o, lse


_default = None


def default() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def attn_fwd(*a, **kw):
    return default().attn_fwd(*a, **kw)


def attn_fwd_rows(*a, **kw):
    return default().attn_fwd_rows(*a, **kw)


def attn_fwd_blocked(*a, **kw):
    return default().attn_fwd_blocked(*a, **kw)


def attn_fwd_split(*a, **kw):
    return default().attn_fwd_split(*a, **kw)


def attn_decode(*a, **kw):
    return default().attn_decode(*a, **kw)


def attn_bwd(*a, **kw):
    return default().attn_bwd(*a, **kw)


def attn_prefill_paged(*a, **kw):
    return default().attn_prefill_paged(*a, **kw)


def attn_fwd_blocksparse(*a, **kw):
    return default().attn_fwd_blocksparse(*a, **kw)


def e4m3_decode(*a, **kw):
    return default().e4m3_decode(*a, **kw)


def attn_fwd_fp8(*a, **kw):
    return default().attn_fwd_fp8(*a, **kw)


def num_threads() -> int:
    return default().num_threads()
