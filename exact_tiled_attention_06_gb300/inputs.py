"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws random numbers, rounds
them to bf16 and lays out paged caches and block tables. Both the CUDA path and
the CPU oracle are fed from here; neither is imported by it.

Recipe (one ``torch.Generator`` on the CPU per call, seeded explicitly):

* prefill: q, k, v drawn in that order, iid N(0, 1) in fp32, rounded to bf16
  (round-to-nearest-even). Optional "boosted" keys: per (b, kv head) slice, a
  seeded choice of ``floor(frac * Nk)`` distinct token rows of K is multiplied
  by ``boost`` (2.0 is exact in bf16). This forces late running-max rises.
* decode: sequence lengths uniform integers in [len_lo, len_hi], then a random
  permutation of the ``sum(ceil(L / block_size))`` physical blocks (plus
  ``extra_blocks`` unused ones), then q, then the K cache, then the V cache,
  iid N(0, 1) rounded to bf16. The block table lists each sequence's physical
  blocks in logical order; unused entries are -1. ``poison`` fills every cache
  slot that no sequence owns (tail slots of a last block, unused blocks) with NaN.
* block-sparse prefill: the prefill recipe for q, k, v; the block index is either
  a global + local pattern (every query block lists the first ``n_global`` key
  blocks and the ``n_local`` blocks ending at its diagonal block) or a seeded
  random pattern, stored as CSR (row_ptr, col_idx).
* paged prefill: the cache and table of the decode recipe for the sequences'
  kv lengths (query lengths drawn first when not given), then q [S][Hq][max_q][d]
  from a generator seeded apart; ``poison`` also fills q rows past each q_len with NaN.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# Head dimension and tile sizes every path supports.
SUPPORTED_HEAD_DIMS = (64, 128)


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    window: int = -1          # keys allowed left of the diagonal; -1 = unlimited
    k_boost_frac: float = 0.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int
    Hq: int
    Hkv: int
    d: int
    block_size: int
    len_lo: int
    len_hi: int
    seed: int = 0
    extra_blocks: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class PagedPrefillConfig:
    name: str
    num_seqs: int
    Hq: int
    Hkv: int
    d: int
    block_size: int
    q_len: int              # new queries per sequence (a prefill chunk)
    ctx_lo: int             # cached tokens before the chunk, uniform integers in [ctx_lo, ctx_hi]
    ctx_hi: int
    causal: bool = True
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads (shapes of the pages' examples: N=512/d=64 single head;
# 2k and 8k causal prefill with d=128; GQA with 4 query heads per kv head and a
# sliding window; paged GQA decode with 16-token pages and up to 32k context).
C1 = PrefillConfig("C1_single_head_noncausal_N512_d64", 1, 1, 1, 512, 512, 64, False)
C2 = PrefillConfig("C2_causal_B4_H16_N2048_d128", 4, 16, 16, 2048, 2048, 128, True)
C3 = PrefillConfig("C3_long_causal_B1_H32_N8192_d128_boost1pct", 1, 32, 32, 8192, 8192, 128, True,
                   k_boost_frac=0.01)
C4 = PrefillConfig("C4_gqa_causal_window1024_B2_Hq32_Hkv8_N4096_d128", 2, 32, 8, 4096, 4096, 128, True,
                   window=1024)
C5 = DecodeConfig("C5_paged_gqa_decode_S64_Hq32_Hkv8_d128_bs16_L1k_32k", 64, 32, 8, 128, 16, 1024, 32768)

# Chunked prefill over a paged cache (the pages give no numbers for it): 16 sequences,
# each appending a 2048-token chunk to 0..14336 earlier tokens, GQA 32/8, 16-token blocks.
C6 = PagedPrefillConfig("C6_chunked_prefill_paged_S16_q2048_ctx0_14k_Hq32_Hkv8_d128_bs16", 16, 32, 8, 128, 16,
                        2048, 0, 14336)

@dataclass(frozen=True)
class SparsePrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    n_global: int   # key blocks every query block lists (from the start)
    n_local: int    # key blocks ending at the query block's diagonal block
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Long-context block-sparse prefill with a global + local pattern (the pages name the
# pattern, not a size): 32k tokens, one global key block and an 8-block local band.
C7 = SparsePrefillConfig("C7_blocksparse_global1_local8_B1_H32_N32768_d128_causal", 1, 32, 32, 32768, 128, True, 1, 8)

PREFILL_CONFIGS = {c.name: c for c in (C1, C2, C3, C4)}
SPARSE_CONFIGS = {C7.name: C7}
PAGED_PREFILL_CONFIGS = {C6.name: C6}
DECODE_CONFIGS = {C5.name: C5}


def _bf16_normal(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=0, k_boost_frac=0.0, k_boost=2.0):
    """Return host bf16 tensors q [B][Hq][Nq][d], k, v [B][Hkv][Nk][d]."""
    gen = torch.Generator().manual_seed(int(seed))
    q = _bf16_normal(gen, (B, Hq, Nq, d))
    k = _bf16_normal(gen, (B, Hkv, Nk, d))
    v = _bf16_normal(gen, (B, Hkv, Nk, d))
    n_boost = int(math.floor(k_boost_frac * Nk))
    if n_boost > 0:
        for b in range(B):
            for h in range(Hkv):
                rows = torch.randperm(Nk, generator=gen)[:n_boost]
                k[b, h, rows] = (k[b, h, rows].float() * k_boost).to(torch.bfloat16)
    return q, k, v


def grad_output(B, Hq, Nq, d, seed=0):
    """Return a host bf16 upstream gradient dO [B][Hq][Nq][d] (standard normal entries,
    drawn from a generator seeded apart from q, k, v)."""
    gen = torch.Generator().manual_seed(int(seed) * 7919 + 104729)
    return _bf16_normal(gen, (B, Hq, Nq, d))


def prefill_config_inputs(cfg: PrefillConfig, seed=None):
    return prefill_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.Nq, cfg.Nk, cfg.d,
                          seed=cfg.seed if seed is None else seed, k_boost_frac=cfg.k_boost_frac)


@dataclass
class PagedDecodeInputs:
    q: torch.Tensor            # [S][Hq][d] bf16
    k_cache: torch.Tensor      # [num_blocks][Hkv][bs][d] bf16
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [S][max_blocks] int32, -1 = unused
    seq_lens: torch.Tensor     # [S] int32
    block_size: int
    extra: dict = field(default_factory=dict)

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V that the sequences own (every token, both caches)."""
        Hkv, d = self.k_cache.shape[1], self.k_cache.shape[3]
        return int(self.seq_lens.to(torch.int64).sum()) * Hkv * d * 2 * 2


def decode_inputs(num_seqs, Hq, Hkv, d, block_size, seq_lens=None, len_lo=1, len_hi=1, seed=0,
                  extra_blocks=0, max_blocks_per_seq=None, poison=False, identity_table=False,
                  chunk_blocks=4096):
    """Paged decode inputs. ``seq_lens`` (list) overrides the drawn lengths."""
    gen = torch.Generator().manual_seed(int(seed))
    if seq_lens is None:
        lens = torch.randint(len_lo, len_hi + 1, (num_seqs,), generator=gen, dtype=torch.int64)
    else:
        lens = torch.as_tensor(list(seq_lens), dtype=torch.int64)
        assert lens.numel() == num_seqs
    nblk = [(int(L) + block_size - 1) // block_size for L in lens]
    used = sum(nblk)
    num_blocks = max(used + int(extra_blocks), 1)
    if identity_table:
        perm = torch.arange(num_blocks, dtype=torch.int64)
    else:
        perm = torch.randperm(num_blocks, generator=gen)
    mb = max(nblk) if nblk else 0
    if max_blocks_per_seq is not None:
        assert max_blocks_per_seq >= mb
        mb = max_blocks_per_seq
    mb = max(mb, 1)
    table = torch.full((num_seqs, mb), -1, dtype=torch.int32)
    pos = 0
    for s, n in enumerate(nblk):
        table[s, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    q = _bf16_normal(gen, (num_seqs, Hq, d))
    caches = []
    for _ in range(2):
        c = torch.empty((num_blocks, Hkv, block_size, d), dtype=torch.bfloat16)
        for b0 in range(0, num_blocks, chunk_blocks):
            b1 = min(num_blocks, b0 + chunk_blocks)
            c[b0:b1] = _bf16_normal(gen, (b1 - b0, Hkv, block_size, d))
        caches.append(c)
    k_cache, v_cache = caches
    if poison:
        owned = torch.zeros((num_blocks, block_size), dtype=torch.bool)
        for s in range(num_seqs):
            L = int(lens[s])
            for lb in range(nblk[s]):
                phys = int(table[s, lb])
                n_tok = min(block_size, L - lb * block_size)
                owned[phys, :n_tok] = True
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        mask = ~owned  # [num_blocks][bs]
        for c in (k_cache, v_cache):
            c.masked_fill_(mask[:, None, :, None], nan)
    return PagedDecodeInputs(q=q, k_cache=k_cache, v_cache=v_cache, block_table=table,
                             seq_lens=lens.to(torch.int32), block_size=block_size)


def decode_config_inputs(cfg: DecodeConfig, seed=None, poison=False):
    return decode_inputs(cfg.num_seqs, cfg.Hq, cfg.Hkv, cfg.d, cfg.block_size, len_lo=cfg.len_lo,
                         len_hi=cfg.len_hi, seed=cfg.seed if seed is None else seed,
                         extra_blocks=cfg.extra_blocks, poison=poison)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor E4M3 quantisation: scale = max|x| / 448 (1 for an all-zero tensor), codes =
    x / scale cast to torch's float8_e4m3fn (round to nearest even). Returns (uint8 codes,
    scale) with x ~ codes * scale."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    scale = amax / 448.0 if amax > 0 else 1.0
    codes = (x.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale


@dataclass
class Fp8PrefillInputs:
    q8: torch.Tensor    # E4M3 codes [B][Hq][Nq][d]
    k8: torch.Tensor    # E4M3 codes [B][Hkv][Nk][d]
    vt8: torch.Tensor   # E4M3 codes [B][Hkv][d][Nk] (V transposed)
    q_descale: float
    k_descale: float
    v_descale: float


def fp8_prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=0, k_boost_frac=0.0):
    """The prefill recipe (N(0,1) -> bf16, optional K boost) quantised per tensor to E4M3;
    V is handed over transposed."""
    q, k, v = prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=seed, k_boost_frac=k_boost_frac)
    q8, qs = quantize_e4m3(q)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    return Fp8PrefillInputs(q8=q8, k8=k8, vt8=v8.transpose(-1, -2).contiguous(), q_descale=qs, k_descale=ks,
                            v_descale=vs)


@dataclass(frozen=True)
class DecodeStepConfig:
    """One decode step of an n-layer model: every layer has its own cache and queries; the
    block table and lengths belong to the sequences and are shared by the layers."""
    name: str
    n_layers: int
    num_seqs: int
    Hq: int
    Hkv: int
    d: int
    block_size: int
    len_lo: int
    len_hi: int
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# A small-batch decode step of a 32-layer model (the pages' launch-overhead example counts
# a 32-layer decode step; they give no batch or lengths): 8 sequences of 512..2048 tokens.
C8 = DecodeStepConfig("C8_decode_step_L32_S8_Hq32_Hkv8_d128_bs16_L512_2k", 32, 8, 32, 8, 128, 16, 512, 2048)
DECODE_STEP_CONFIGS = {C8.name: C8}


@dataclass
class DecodeStepInputs:
    q: list                    # per layer [S][Hq][d] bf16
    k_cache: list              # per layer [num_blocks][Hkv][bs][d] bf16
    v_cache: list
    block_table: torch.Tensor  # [S][max_blocks] int32, shared by the layers
    seq_lens: torch.Tensor     # [S] int32, shared by the layers
    block_size: int

    def layer(self, l: int) -> PagedDecodeInputs:
        return PagedDecodeInputs(q=self.q[l], k_cache=self.k_cache[l], v_cache=self.v_cache[l],
                                 block_table=self.block_table, seq_lens=self.seq_lens, block_size=self.block_size)

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V the sequences own, summed over the layers."""
        return len(self.q) * self.layer(0).kv_bytes


def decode_step_inputs(n_layers, num_seqs, Hq, Hkv, d, block_size, seq_lens=None, len_lo=1, len_hi=1, seed=0,
                       extra_blocks=0, max_blocks_per_seq=None, poison=False):
    """Layer 0 is ``decode_inputs(..., seed)``; layer l > 0 draws its q and caches from a
    generator seeded with (seed, l) and shares layer 0's table, lengths and (with
    ``poison``) NaN pattern in the slots no sequence owns."""
    base = decode_inputs(num_seqs, Hq, Hkv, d, block_size, seq_lens=seq_lens, len_lo=len_lo, len_hi=len_hi,
                         seed=seed, extra_blocks=extra_blocks, max_blocks_per_seq=max_blocks_per_seq, poison=poison)
    qs, ks, vs = [base.q], [base.k_cache], [base.v_cache]
    unowned = torch.isnan(base.k_cache) if poison else None
    for l in range(1, n_layers):
        gen = torch.Generator().manual_seed(int(seed) * 1_000_003 + l)
        qs.append(_bf16_normal(gen, tuple(base.q.shape)))
        for lst in (ks, vs):
            c = _bf16_normal(gen, tuple(base.k_cache.shape))
            if unowned is not None:
                c.masked_fill_(unowned, float("nan"))
            lst.append(c)
    return DecodeStepInputs(q=qs, k_cache=ks, v_cache=vs, block_table=base.block_table, seq_lens=base.seq_lens,
                            block_size=block_size)


def decode_step_config_inputs(cfg: DecodeStepConfig, seed=None, poison=False):
    return decode_step_inputs(cfg.n_layers, cfg.num_seqs, cfg.Hq, cfg.Hkv, cfg.d, cfg.block_size, len_lo=cfg.len_lo,
                              len_hi=cfg.len_hi, seed=cfg.seed if seed is None else seed, poison=poison)


@dataclass
class PagedPrefillInputs:
    q: torch.Tensor            # [S][Hq][max_q][d] bf16
    k_cache: torch.Tensor      # [num_blocks][Hkv][bs][d] bf16
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [S][max_blocks] int32, -1 = unused
    q_lens: torch.Tensor       # [S] int32
    kv_lens: torch.Tensor      # [S] int32
    block_size: int


def paged_prefill_inputs(num_seqs, Hq, Hkv, d, block_size, q_lens, kv_lens, max_q=None, seed=0, extra_blocks=0,
                         poison=False, identity_table=False, max_blocks_per_seq=None):
    """Paged prefill inputs for given per-sequence query and cache lengths."""
    assert len(q_lens) == num_seqs and len(kv_lens) == num_seqs
    assert all(0 <= a <= b for a, b in zip(q_lens, kv_lens))
    x = decode_inputs(num_seqs, Hq, Hkv, d, block_size, seq_lens=list(kv_lens), seed=seed, extra_blocks=extra_blocks,
                      poison=poison, identity_table=identity_table, max_blocks_per_seq=max_blocks_per_seq)
    max_q = max(q_lens) if max_q is None else max_q
    gen = torch.Generator().manual_seed(int(seed) * 7919 + 31337)
    q = _bf16_normal(gen, (num_seqs, Hq, max_q, d))
    if poison:
        for s, n in enumerate(q_lens):
            q[s, :, n:, :] = float("nan")
    return PagedPrefillInputs(q=q, k_cache=x.k_cache, v_cache=x.v_cache, block_table=x.block_table,
                              q_lens=torch.as_tensor(list(q_lens), dtype=torch.int32),
                              kv_lens=torch.as_tensor(list(kv_lens), dtype=torch.int32), block_size=block_size)


def paged_prefill_config_inputs(cfg: PagedPrefillConfig, seed=None):
    """The chunked-prefill workload: context lengths drawn first, then the cache and q."""
    sd = cfg.seed if seed is None else seed
    gen = torch.Generator().manual_seed(int(sd) * 104729 + 7)
    ctx = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (cfg.num_seqs,), generator=gen, dtype=torch.int64)
    q_lens = [cfg.q_len] * cfg.num_seqs
    kv_lens = [int(c) + cfg.q_len for c in ctx]
    return paged_prefill_inputs(cfg.num_seqs, cfg.Hq, cfg.Hkv, cfg.d, cfg.block_size, q_lens, kv_lens, seed=sd)


def block_csr(pattern):
    """Boolean block pattern [n_qblk][n_kblk] -> CSR (row_ptr, col_idx) as int32 tensors."""
    pat = torch.as_tensor(pattern, dtype=torch.bool)
    counts = pat.sum(dim=1).to(torch.int64)
    row_ptr = torch.zeros(pat.shape[0] + 1, dtype=torch.int64)
    row_ptr[1:] = torch.cumsum(counts, dim=0)
    col_idx = torch.nonzero(pat, as_tuple=False)[:, 1]
    return row_ptr.to(torch.int32), col_idx.to(torch.int32)


def global_local_pattern(n_qblk, n_kblk, n_global, n_local):
    """Every query block r lists key blocks [0, n_global) and the n_local blocks ending at its
    diagonal block r + (n_kblk - n_qblk) (bottom-right alignment), clipped to the key range."""
    pat = torch.zeros((n_qblk, n_kblk), dtype=torch.bool)
    for r in range(n_qblk):
        diag = r + (n_kblk - n_qblk)
        pat[r, :max(0, min(n_global, n_kblk))] = True
        lo, hi = max(0, diag - n_local + 1), min(n_kblk, diag + 1)
        if hi > lo:
            pat[r, lo:hi] = True
    return pat


def random_pattern(n_qblk, n_kblk, density, seed=0, empty_rows=()):
    """Seeded random block pattern; rows in ``empty_rows`` list nothing."""
    gen = torch.Generator().manual_seed(int(seed))
    pat = torch.rand((n_qblk, n_kblk), generator=gen) < density
    for r in empty_rows:
        pat[r] = False
    return pat


def sparse_config_inputs(cfg: SparsePrefillConfig, seed=None):
    """q, k, v of the block-sparse workload and its global + local pattern."""
    q, k, v = prefill_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d, seed=cfg.seed if seed is None else seed)
    nb = (cfg.N + 127) // 128
    pat = global_local_pattern(nb, nb, cfg.n_global, cfg.n_local)
    return q, k, v, pat
