"""GB300-native exact tiled attention (sm_103a): prefill (dense, block-sparse, or over a paged
cache), its backward, and paged GQA decode (per call, or a many-layer step replayed as a CUDA
graph).

The compute lives in ``libattn.so`` (CUDA, built in-tree by ``build()``); its C ABI is
``include/attn.h``. ``binding`` exposes the same entry points to Python with torch
tensors as device memory. ``inputs`` holds the seeded synthetic workloads.
"""
from .buildlib import build
from .binding import (AttnError, DecodeGraph, attn_bwd, attn_bwd_workspace_size, attn_decode,
                      attn_decode_chunk_tokens, attn_decode_graph_create, attn_decode_noalloc,
                      attn_decode_workspace_size, attn_fwd, attn_fwd_blocksparse, attn_fwd_fp8,
                      attn_fwd_host, attn_decode_host, attn_get_device_error,
                      attn_kv_layout_version, attn_prefill_paged, attn_status_string, load_library)

__all__ = ["build", "AttnError", "attn_fwd", "attn_fwd_fp8", "attn_fwd_host", "attn_decode_host", "attn_fwd_blocksparse", "attn_prefill_paged", "attn_bwd",
           "attn_bwd_workspace_size", "attn_decode", "attn_decode_noalloc", "attn_decode_workspace_size",
           "attn_decode_graph_create", "DecodeGraph", "attn_decode_chunk_tokens", "attn_get_device_error",
           "attn_kv_layout_version", "attn_status_string", "load_library"]
