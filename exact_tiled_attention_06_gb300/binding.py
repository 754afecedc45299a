"""Thin ctypes binding over libattn.so (include/attn.h), same names as the C ABI.

Only argument marshalling happens here: torch tensors provide device memory and
the current CUDA stream; every step of the computation runs in the library's
kernels. There is no fallback: if the library is missing or returns an error,
these functions raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import buildlib as _build

ATTN_OK = 0
STATUS_NAMES = {
    0: "ATTN_OK", -1: "ATTN_ERR_INVALID_ARG", -2: "ATTN_ERR_UNSUPPORTED", -3: "ATTN_ERR_MISALIGNED",
    -4: "ATTN_ERR_WORKSPACE", -5: "ATTN_ERR_LAUNCH", -6: "ATTN_ERR_DEVICE_TIMEOUT", -7: "ATTN_ERR_DEVICE_BOUNDS",
    -8: "ATTN_ERR_CUDA",
}

# Every symbol include/attn.h declares.
EXPORTED = ("attn_fwd", "attn_fwd_fp8", "attn_fwd_blocksparse", "attn_prefill_paged", "attn_bwd_workspace_size", "attn_bwd", "attn_decode_workspace_size", "attn_decode",
            "attn_decode_chunk_tokens", "attn_get_device_error", "attn_kv_layout_version", "attn_status_string",
            "attn_decode_noalloc", "attn_decode_graph_create", "attn_decode_graph_launch", "attn_decode_graph_layers",
            "attn_decode_graph_destroy", "attn_fwd_host", "attn_decode_host",
            "attn_selftest_wait_timeout")


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {STATUS_NAMES.get(status, status)} ({status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libattn.so (it must have been built with ``build()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"libattn.so is not built ({p}); run exact_tiled_attention_06_gb300.build()")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, f, f, i, i, vp]
        lib.attn_fwd_fp8.restype = i
        lib.attn_fwd_blocksparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, vp]
        lib.attn_fwd_blocksparse.restype = i
        lib.attn_prefill_paged.argtypes = [vp] * 8 + [i] * 8 + [f, i, i, vp]
        lib.attn_prefill_paged.restype = i
        lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.attn_bwd_workspace_size.restype = sz
        lib.attn_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, i, vp, sz, vp]
        lib.attn_bwd.restype = i
        lib.attn_decode_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.attn_decode_workspace_size.restype = sz
        lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.attn_decode.restype = i
        lib.attn_decode_chunk_tokens.argtypes = [i, i, i, i, i]
        lib.attn_decode_chunk_tokens.restype = i
        lib.attn_get_device_error.argtypes = [vp]
        lib.attn_get_device_error.restype = i
        lib.attn_kv_layout_version.argtypes = []
        lib.attn_kv_layout_version.restype = i
        lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
        lib.attn_decode_noalloc.restype = i
        lib.attn_decode_graph_create.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz,
                                                 ctypes.POINTER(vp)]
        lib.attn_decode_graph_create.restype = i
        lib.attn_decode_graph_launch.argtypes = [vp, vp]
        lib.attn_decode_graph_launch.restype = i
        lib.attn_decode_graph_layers.argtypes = [vp]
        lib.attn_decode_graph_layers.restype = i
        lib.attn_decode_graph_destroy.argtypes = [vp]
        lib.attn_decode_graph_destroy.restype = i
        lib.attn_fwd_host.argtypes = [vp] * 10 + [i, i, i, i, i, i, f, i, i, i, vp]
        lib.attn_fwd_host.restype = i
        lib.attn_decode_host.argtypes = [vp] * 14 + [i, i, i, i, i, i, i, f, vp, sz, vp]
        lib.attn_decode_host.restype = i
        lib.attn_selftest_wait_timeout.argtypes = [vp]
        lib.attn_selftest_wait_timeout.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_kv_layout_version() -> int:
    return int(load_library().attn_kv_layout_version())


def attn_get_device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the device error word."""
    return int(load_library().attn_get_device_error(_stream_handle(stream)))


def attn_fwd(q, k, v, causal=False, window=-1, scale=None, out=None, lse=None, stream=None):
    """Prefill attention. q [B][Hq][Nq][d], k/v [B][Hkv][Nk][d] bf16 (CUDA, contiguous).
    Returns (o bf16 [B][Hq][Nq][d], lse fp32 [B][Hq][Nq])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if Bk != B or dk != d or v.shape != k.shape:
        raise ValueError("q/k/v shapes disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    rc = load_library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                 float(scale), int(bool(causal)), int(window), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def _need_u8(t, name: str, ndim: int):
    """An E4M3 tensor: uint8 or torch.float8_e4m3fn, CUDA, contiguous; returned as uint8."""
    if isinstance(t, torch.Tensor) and t.dtype == getattr(torch, "float8_e4m3fn", None):
        t = t.view(torch.uint8)
    _need(t, name, torch.uint8, ndim)
    return t


def attn_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, causal=False, window=-1, scale=None, out=None,
                 lse=None, stream=None):
    """FP8 prefill. q8 [B][Hq][Nq][128], k8 [B][Hkv][Nk][128], vt8 [B][Hkv][128][Nk] E4M3 (uint8 or
    float8_e4m3fn, CUDA); real inputs = codes x the per-tensor descales. ``scale`` defaults to
    1/sqrt(d). Returns (o bf16 [B][Hq][Nq][128], lse fp32 [B][Hq][Nq])."""
    q8 = _need_u8(q8, "q8", 4)
    k8 = _need_u8(k8, "k8", 4)
    vt8 = _need_u8(vt8, "vt8", 4)
    B, Hq, Nq, d = q8.shape
    Bk, Hkv, Nk, dk = k8.shape
    if Bk != B or dk != d or tuple(vt8.shape) != (B, Hkv, d, Nk):
        raise ValueError("q8/k8/vt8 shapes disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, Nq, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q8.device)
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    rc = load_library().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                     float(scale), float(q_descale), float(k_descale), float(v_descale),
                                     int(bool(causal)), int(window), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return out, lse


def attn_fwd_blocksparse(q, k, v, row_ptr, col_idx, causal=False, window=-1, scale=None, out=None, lse=None,
                         stream=None):
    """Block-sparse prefill. q [B][Hq][Nq][d], k/v [B][Hkv][Nk][d] bf16; row_ptr int32
    [ceil(Nq / 128) + 1] and col_idx int32 list the 128 x 128 blocks to visit (device)."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    _need(row_ptr, "row_ptr", torch.int32, 1)
    _need(col_idx, "col_idx", torch.int32, 1)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if Bk != B or dk != d or v.shape != k.shape:
        raise ValueError("q/k/v shapes disagree")
    if row_ptr.shape[0] != (Nq + 127) // 128 + 1:
        raise ValueError("row_ptr must have ceil(Nq / 128) + 1 entries")
    if col_idx.numel() == 0:
        col_idx = torch.zeros(1, dtype=torch.int32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    rc = load_library().attn_fwd_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                             float(scale), int(bool(causal)), int(window), _ptr(row_ptr),
                                             _ptr(col_idx), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_blocksparse")
    return out, lse


def attn_prefill_paged(q, k_cache, v_cache, block_table, q_lens, kv_lens, causal=True, window=-1, scale=None,
                       out=None, lse=None, stream=None):
    """Paged (chunked) prefill. q [S][Hq][max_q][d] bf16; caches [num_blocks][Hkv][bs][d] bf16;
    block_table int32 [S][max_blocks]; q_lens, kv_lens int32 [S] (device). Returns (o, lse);
    rows past q_lens[s] are left as they were in ``out`` / ``lse`` (uninitialised if allocated here)."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(q_lens, "q_lens", torch.int32, 1)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    S, Hq, max_q, d = q.shape
    nb, Hkv, bs, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape or block_table.shape[0] != S or q_lens.shape[0] != S \
            or kv_lens.shape[0] != S:
        raise ValueError("paged prefill shapes disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((S, Hq, max_q), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    rc = load_library().attn_prefill_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(q_lens),
                                           _ptr(kv_lens), _ptr(out), _ptr(lse), S, Hq, Hkv, d, bs,
                                           block_table.shape[1], nb, max_q, float(scale), int(bool(causal)),
                                           int(window), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_prefill_paged")
    return out, lse


def attn_bwd_workspace_size(B, Hq, Nq, d) -> int:
    return int(load_library().attn_bwd_workspace_size(B, Hq, Nq, d))


def attn_bwd(q, k, v, o, dout, lse, causal=False, window=-1, scale=None, workspace=None, dq=None, dk=None,
             dv=None, stream=None):
    """Attention backward. q, o, dout [B][Hq][Nq][d] bf16; k, v [B][Hkv][Nk][d] bf16;
    lse fp32 [B][Hq][Nq] (o and lse from attn_fwd). Returns (dq, dk, dv) in bf16."""
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, name, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk_ = k.shape
    if Bk != B or dk_ != d or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("backward shapes disagree")
    if lse.shape != (B, Hq, Nq):
        raise ValueError("lse must be [B][Hq][Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_bwd_workspace_size(B, Hq, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", torch.bfloat16, 4)
    _need(dk, "dk", torch.bfloat16, 4)
    _need(dv, "dv", torch.bfloat16, 4)
    rc = load_library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)), int(window),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_decode_workspace_size(num_seqs, Hq, Hkv, d, block_size, max_blocks_per_seq) -> int:
    return int(load_library().attn_decode_workspace_size(num_seqs, Hq, Hkv, d, block_size, max_blocks_per_seq))


def attn_decode_chunk_tokens(num_seqs, Hq, Hkv, block_size, max_blocks_per_seq) -> int:
    return int(load_library().attn_decode_chunk_tokens(num_seqs, Hq, Hkv, block_size, max_blocks_per_seq))


def attn_decode(q, k_cache, v_cache, block_table, seq_lens, scale=None, workspace=None, out=None, lse=None,
                stream=None):
    """Paged one-query decode. q [S][Hq][d] bf16; caches [num_blocks][Hkv][bs][d] bf16;
    block_table int32 [S][max_blocks]; seq_lens int32 [S]. Returns (o [S][Hq][d], lse [S][Hq])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, Hq, d = q.shape
    nb, Hkv, bs, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape or block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("decode shapes disagree")
    mb = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((S, Hq), dtype=torch.float32, device=q.device)
    rc = load_library().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                                    _ptr(out), _ptr(lse), S, Hq, Hkv, d, bs, mb, nb, float(scale),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode")
    return out, lse


def attn_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, scale=None, out=None, lse=None, stream=None):
    """attn_decode for callers that cannot allocate device scratch: the split partials
    live in a 64 MiB static array inside the library (calls must not overlap on the
    GPU). Inputs and outputs as for attn_decode; ``out``/``lse`` are allocated here
    only when not given."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, Hq, d = q.shape
    nb, Hkv, bs, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape or block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("decode shapes disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((S, Hq), dtype=torch.float32, device=q.device)
    rc = load_library().attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                            _ptr(seq_lens), _ptr(out), _ptr(lse), S, Hq, Hkv, d, bs,
                                            block_table.shape[1], nb, float(scale), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_noalloc")
    return out, lse


class DecodeGraph:
    """A decode step over several layers captured once by ``attn_decode_graph_create`` and
    replayed by ``launch()`` (one graph launch per step). The object keeps references to
    every tensor the graph points at, so they stay alive and in place; rewrite their
    contents (queries, cache rows, block table, lengths) between launches."""

    def __init__(self, handle: int, tensors, outs, lses):
        self._handle = handle
        self._tensors = tensors
        self.out = outs
        self.lse = lses

    @property
    def layers(self) -> int:
        return int(load_library().attn_decode_graph_layers(self._handle)) if self._handle else 0

    def launch(self, stream=None):
        if not self._handle:
            raise RuntimeError("DecodeGraph is closed")
        rc = load_library().attn_decode_graph_launch(self._handle, _stream_handle(stream))
        if rc != ATTN_OK:
            raise AttnError(rc, "attn_decode_graph_launch")
        return self.out, self.lse

    def close(self):
        """Release the graph (synchronise any stream it was launched on first)."""
        if self._handle:
            h, self._handle = self._handle, None
            rc = load_library().attn_decode_graph_destroy(h)
            if rc != ATTN_OK:
                raise AttnError(rc, "attn_decode_graph_destroy")

    def __del__(self):
        try:
            if self._handle:
                torch.cuda.synchronize()
                self.close()
        except Exception:
            pass


def attn_decode_graph_create(qs, k_caches, v_caches, block_table, seq_lens, scale=None, workspace=None,
                             outs=None, lses=None) -> DecodeGraph:
    """Capture one decode call per layer (attn_decode's shapes; per-layer q, caches and
    outputs, one shared block table and seq_lens) into a CUDA graph. Returns a
    ``DecodeGraph`` whose ``launch()`` replays the step; ``out``/``lse`` hold the
    per-layer outputs it writes."""
    n = len(qs)
    if n == 0 or len(k_caches) != n or len(v_caches) != n:
        raise ValueError("one q, k_cache and v_cache per layer")
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, Hq, d = qs[0].shape
    nb, Hkv, bs, _ = k_caches[0].shape
    for l in range(n):
        _need(qs[l], f"q[{l}]", torch.bfloat16, 3)
        _need(k_caches[l], f"k_cache[{l}]", torch.bfloat16, 4)
        _need(v_caches[l], f"v_cache[{l}]", torch.bfloat16, 4)
        if qs[l].shape != (S, Hq, d) or k_caches[l].shape != (nb, Hkv, bs, d) or v_caches[l].shape != (nb, Hkv, bs, d):
            raise ValueError(f"layer {l}: shapes differ from layer 0")
    if block_table.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("decode shapes disagree")
    mb = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qs[0].device)
    if outs is None:
        outs = [torch.empty_like(qs[0]) for _ in range(n)]
    if lses is None:
        lses = [torch.empty((S, Hq), dtype=torch.float32, device=qs[0].device) for _ in range(n)]
    arr = ctypes.c_void_p * n
    h = ctypes.c_void_p()
    rc = load_library().attn_decode_graph_create(
        n, arr(*[t.data_ptr() for t in qs]), arr(*[t.data_ptr() for t in k_caches]),
        arr(*[t.data_ptr() for t in v_caches]), arr(*[t.data_ptr() for t in outs]), arr(*[t.data_ptr() for t in lses]),
        _ptr(block_table), _ptr(seq_lens), S, Hq, Hkv, d, bs, mb, nb, float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), ctypes.byref(h))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_graph_create")
    return DecodeGraph(h.value, (list(qs), list(k_caches), list(v_caches), block_table, seq_lens, workspace),
                       outs, lses)


def _need_host(t, name: str, dtype: torch.dtype, ndim: int):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor with {ndim} dimensions")


def attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, causal=False, window=-1, scale=None,
                  chunk_kv_heads=0, stream=None):
    """attn_fwd from host tensors (pinned for overlap): the inputs are copied into the device
    tensors *_d chunk by chunk while earlier chunks compute and copy back into o_h / lse_h.
    Returns (o_h, lse_h); complete when ``stream`` is."""
    for n, t, nd in (("q_h", q_h, 4), ("k_h", k_h, 4), ("v_h", v_h, 4), ("o_h", o_h, 4)):
        _need_host(t, n, torch.bfloat16, nd)
    _need_host(lse_h, "lse_h", torch.float32, 3)
    for n, t in (("q_d", q_d), ("k_d", k_d), ("v_d", v_d), ("o_d", o_d)):
        _need(t, n, torch.bfloat16, 4)
    _need(lse_d, "lse_d", torch.float32, 3)
    B, Hq, Nq, d = q_h.shape
    Bk, Hkv, Nk, dk = k_h.shape
    if (Bk != B or dk != d or v_h.shape != k_h.shape or q_d.shape != q_h.shape or k_d.shape != k_h.shape
            or v_d.shape != v_h.shape or o_h.shape != q_h.shape or o_d.shape != q_h.shape
            or tuple(lse_h.shape) != (B, Hq, Nq) or lse_d.shape != lse_h.shape):
        raise ValueError("host / device shapes disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load_library().attn_fwd_host(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(lse_h), _ptr(q_d), _ptr(k_d),
                                      _ptr(v_d), _ptr(o_d), _ptr(lse_d), B, Hq, Hkv, Nq, Nk, d, float(scale),
                                      int(bool(causal)), int(window), int(chunk_kv_heads), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return o_h, lse_h


def attn_decode_host(q_h, k_cache_h, v_cache_h, block_table_h, seq_lens_h, o_h, lse_h, q_d, k_cache_d, v_cache_d,
                     block_table_d, seq_lens_d, o_d, lse_d, scale=None, workspace=None, stream=None):
    """attn_decode from host tensors: everything is copied in, decoded and copied back in
    order on ``stream``. Returns (o_h, lse_h); complete when ``stream`` is."""
    _need_host(q_h, "q_h", torch.bfloat16, 3)
    _need_host(k_cache_h, "k_cache_h", torch.bfloat16, 4)
    _need_host(v_cache_h, "v_cache_h", torch.bfloat16, 4)
    _need_host(block_table_h, "block_table_h", torch.int32, 2)
    _need_host(seq_lens_h, "seq_lens_h", torch.int32, 1)
    _need_host(o_h, "o_h", torch.bfloat16, 3)
    _need_host(lse_h, "lse_h", torch.float32, 2)
    S, Hq, d = q_h.shape
    nb, Hkv, bs, _ = k_cache_h.shape
    mb = block_table_h.shape[1]
    for n, t, ref in (("q_d", q_d, q_h), ("k_cache_d", k_cache_d, k_cache_h), ("v_cache_d", v_cache_d, v_cache_h),
                      ("block_table_d", block_table_d, block_table_h), ("seq_lens_d", seq_lens_d, seq_lens_h),
                      ("o_d", o_d, o_h), ("lse_d", lse_d, lse_h)):
        _need(t, n, ref.dtype, ref.dim())
        if t.shape != ref.shape:
            raise ValueError(f"{n} shape differs from its host tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_size(S, Hq, Hkv, d, bs, mb)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_d.device)
    rc = load_library().attn_decode_host(_ptr(q_h), _ptr(k_cache_h), _ptr(v_cache_h), _ptr(block_table_h),
                                         _ptr(seq_lens_h), _ptr(o_h), _ptr(lse_h), _ptr(q_d), _ptr(k_cache_d),
                                         _ptr(v_cache_d), _ptr(block_table_d), _ptr(seq_lens_d), _ptr(o_d),
                                         _ptr(lse_d), S, Hq, Hkv, d, bs, mb, nb, float(scale), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_host")
    return o_h, lse_h


def attn_selftest_wait_timeout(stream=None) -> None:
    """Launch a block whose barrier wait runs out (about 2 s); the device error word then
    reads ATTN_ERR_DEVICE_TIMEOUT. For failure-detection tests."""
    rc = load_library().attn_selftest_wait_timeout(_stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_selftest_wait_timeout")
