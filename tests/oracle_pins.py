"""Checks that pin the fp64 oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch. ``test_oracle_pins.py`` runs them against the committed oracle;
``test_oracle_mutants.py`` runs them against copies with planted mistakes and
expects at least one to fail for each mistake.

What each pin rests on (pages by title and section):

* blocked == materialised, split == unsplit: the tiling rule is exact
  ("Modern attention kernels", "Online softmax makes tiling exact"; "Attention
  kernels", safe/online softmax derivation and FlashDecoding) -- in fp64 the
  difference is rounding only, bounded here by 1e-12.
* probabilities sum to one (safe softmax definition) -> V = 1 gives O = 1.
* equal scores give the mean of V; one dominant key returns its V row; the
  first causal row sees only key 0 (closed forms).
* translation invariance ("Flash attention and IO-aware attention", the online
  softmax paragraph): adding a constant to a row's scores leaves O unchanged
  and shifts lse by the constant.
* permutation invariance of the key/value set (non-causal).
* a window at least as long as the context equals plain causal.
* GQA equals MHA with the kv heads duplicated ("Attention kernels", GQA).
* paged decode equals contiguous attention for any block table ("Modern
  attention kernels", "Paged attention changes addressing").
* an independent numpy brute force on tiny inputs.
* the hand-derived three-key example in ``tests/golden/three_keys.json``.
* backward ("Modern attention kernels", "Backward pass recomputes scores"): central
  finite differences of sum(dO * O) through the forward oracle; torch autograd of a
  plain softmax attention on tiny inputs; the exact invariants sum_j dK_j = 0 (softmax
  is shift invariant per row) and sum_j dV_j = sum over non-empty rows of dO_i; GQA
  gradients equal the summed gradients of duplicated heads.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, B, Hq, Hkv, Nq, Nk, d):
    r = _rng(seed)
    return (r.standard_normal((B, Hq, Nq, d)), r.standard_normal((B, Hkv, Nk, d)),
            r.standard_normal((B, Hkv, Nk, d)))


def _allowed_range(i, Nq, Nk, causal, window):
    """Allowed keys of row i as a half-open range [lo, hi) (slice form)."""
    diag = i + (Nk - Nq)
    hi = min(Nk, diag + 1) if causal else Nk
    lo = max(0, diag - window) if window >= 0 else 0
    return lo, max(lo, hi)


def _close(a, b, tol, what):
    a, b = np.asarray(a), np.asarray(b)
    fin_a, fin_b = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fin_a, fin_b), f"{what}: finite pattern differs"
    assert np.array_equal(a[~fin_a], b[~fin_b]), f"{what}: non-finite values differ"
    if fin_a.any():
        err = np.max(np.abs(a[fin_a] - b[fin_b]))
        assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


MASKS = [
    # (Nq, Nk, causal, window)
    (37, 37, False, -1),
    (37, 37, True, -1),
    (29, 41, True, -1),     # Nq < Nk: bottom-right causal alignment
    (41, 29, True, -1),     # Nq > Nk: leading rows see no key
    (40, 40, True, 5),
    (33, 47, False, 9),     # left limit only
    (40, 40, True, 0),      # diagonal only
]


def pin_blocked_equals_materialised(orc):
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, v = _qkv(100 + mi, 2, 4, 2, Nq, Nk, 8)
        o_ref, l_ref = orc.attn_fwd(q, k, v, 0.35, causal, window)
        for br, bc in [(1, 1), (7, 7), (16, 5), (64, 64), (Nq, Nk)]:
            o, l = orc.attn_fwd_blocked(q, k, v, 0.35, causal, window, br, bc)
            _close(o, o_ref, TOL, f"blocked O mask{mi} ({br},{bc})")
            _close(l, l_ref, TOL, f"blocked lse mask{mi} ({br},{bc})")


def pin_split_equals_unsplit(orc):
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, v = _qkv(200 + mi, 1, 4, 4, Nq, Nk, 8)
        o_ref, l_ref = orc.attn_fwd(q, k, v, 0.4, causal, window)
        for chunk in (1, 5, 16, Nk):
            o, l = orc.attn_fwd_split(q, k, v, 0.4, causal, window, chunk)
            _close(o, o_ref, TOL, f"split O mask{mi} chunk{chunk}")
            _close(l, l_ref, TOL, f"split lse mask{mi} chunk{chunk}")


def pin_probabilities_sum_to_one(orc):
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, _ = _qkv(300 + mi, 1, 2, 1, Nq, Nk, 6)
        q *= 3.0
        v = np.ones((1, 1, Nk, 6))
        for name, (o, lse) in (("materialised", orc.attn_fwd(q, k, v, 0.5, causal, window)),
                               ("blocked", orc.attn_fwd_blocked(q, k, v, 0.5, causal, window, 8, 8)),
                               ("split", orc.attn_fwd_split(q, k, v, 0.5, causal, window, 7))):
            for i in range(Nq):
                lo, hi = _allowed_range(i, Nq, Nk, causal, window)
                want = 1.0 if hi > lo else 0.0
                assert np.max(np.abs(o[0, :, i, :] - want)) <= 1e-13, f"{name} row {i} mask{mi}"


def pin_equal_scores_give_mean(orc):
    """q = 0 makes every score 0: O is the mean of V over the allowed keys and
    lse = ln(count). All keys equal makes every score s: lse = s + ln(count)."""
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        _, k, v = _qkv(400 + mi, 1, 2, 2, Nq, Nk, 5)
        q0 = np.zeros((1, 2, Nq, 5))
        o, lse = orc.attn_fwd(q0, k, v, 0.7, causal, window)
        qr, _, _ = _qkv(450 + mi, 1, 2, 2, Nq, Nk, 5)
        kc = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
        o2, lse2 = orc.attn_fwd(qr, kc, v, 0.7, causal, window)
        for h in range(2):
            for i in range(Nq):
                lo, hi = _allowed_range(i, Nq, Nk, causal, window)
                if hi == lo:
                    assert np.all(o[0, h, i] == 0) and lse[0, h, i] == -np.inf
                    continue
                mean = v[0, h, lo:hi].mean(axis=0)
                assert np.max(np.abs(o[0, h, i] - mean)) <= 1e-13
                assert abs(lse[0, h, i] - math.log(hi - lo)) <= 1e-13
                s = 0.7 * float(qr[0, h, i] @ k[0, h, 0])
                assert np.max(np.abs(o2[0, h, i] - mean)) <= 1e-13
                assert abs(lse2[0, h, i] - (s + math.log(hi - lo))) <= 1e-12


def pin_dominant_key(orc):
    """k_j* = c q with a >= 60-nat margin: O = V[j*], lse = s* to rounding."""
    r = _rng(500)
    d, Nk = 16, 50
    q = r.standard_normal((1, 1, 1, d))
    k = r.standard_normal((1, 1, Nk, d))
    v = r.standard_normal((1, 1, Nk, d))
    jstar = 31
    scale = 0.25
    others = scale * (k[0, 0] @ q[0, 0, 0])
    c = (np.max(others) + 60.0) / (scale * float(q[0, 0, 0] @ q[0, 0, 0])) + 1.0
    k[0, 0, jstar] = c * q[0, 0, 0]
    sstar = scale * float(q[0, 0, 0] @ k[0, 0, jstar])
    for fn in (lambda: orc.attn_fwd(q, k, v, scale),
               lambda: orc.attn_fwd_blocked(q, k, v, scale, block_r=1, block_c=8),
               lambda: orc.attn_fwd_split(q, k, v, scale, chunk=9)):
        o, lse = fn()
        assert np.max(np.abs(o[0, 0, 0] - v[0, 0, jstar])) <= 1e-13 * np.max(np.abs(v))
        assert abs(lse[0, 0, 0] - sstar) <= 1e-13 * abs(sstar)


def pin_first_causal_row(orc):
    """With Nq == Nk and causal masking, row 0 sees key 0 only."""
    q, k, v = _qkv(600, 2, 4, 2, 23, 23, 8)
    o, lse = orc.attn_fwd(q, k, v, 0.3, causal=True)
    for b in range(2):
        for h in range(4):
            hk = h // 2
            assert np.max(np.abs(o[b, h, 0] - v[b, hk, 0])) <= 1e-15
            assert abs(lse[b, h, 0] - 0.3 * float(q[b, h, 0] @ k[b, hk, 0])) <= 1e-14


def pin_translation_invariance(orc):
    """An extra dimension with q = 1 and k = c adds scale*c to every score."""
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, v = _qkv(700 + mi, 1, 2, 1, Nq, Nk, 6)
        c = 3.75
        qa = np.concatenate([q, np.ones(q.shape[:-1] + (1,))], axis=-1)
        ka = np.concatenate([k, np.full(k.shape[:-1] + (1,), c)], axis=-1)
        va = np.concatenate([v, np.zeros(v.shape[:-1] + (1,))], axis=-1)
        o, lse = orc.attn_fwd(q, k, v, 0.5, causal, window)
        oa, lsea = orc.attn_fwd(qa, ka, va, 0.5, causal, window)
        _close(oa[..., :6], o, 1e-13, f"translated O mask{mi}")
        fin = np.isfinite(lse)
        assert np.array_equal(fin, np.isfinite(lsea))
        assert np.max(np.abs(lsea[fin] - (lse[fin] + 0.5 * c))) <= 1e-12


def pin_permutation_invariance(orc):
    q, k, v = _qkv(800, 1, 3, 3, 19, 31, 8)
    perm = _rng(801).permutation(31)
    o, lse = orc.attn_fwd(q, k, v, 0.3)
    o2, lse2 = orc.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.3)
    _close(o2, o, 1e-13, "permuted O")
    _close(lse2, lse, 1e-13, "permuted lse")


def pin_long_window_is_plain_mask(orc):
    q, k, v = _qkv(900, 1, 2, 2, 30, 30, 8)
    oc, lc = orc.attn_fwd(q, k, v, 0.3, causal=True)
    ow, lw = orc.attn_fwd(q, k, v, 0.3, causal=True, window=30)
    _close(ow, oc, 0.0, "window>=Nk O")
    _close(lw, lc, 0.0, "window>=Nk lse")
    on, ln_ = orc.attn_fwd(q, k, v, 0.3, causal=False)
    ow2, lw2 = orc.attn_fwd(q, k, v, 0.3, causal=False, window=60)
    _close(ow2, on, 0.0, "noncausal long window O")
    _close(lw2, ln_, 0.0, "noncausal long window lse")


def pin_gqa_equals_duplicated_heads(orc):
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS[:5]):
        q, k, v = _qkv(1000 + mi, 2, 8, 2, Nq, Nk, 8)
        o, lse = orc.attn_fwd(q, k, v, 0.3, causal, window)
        kd, vd = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
        o2, lse2 = orc.attn_fwd(q, kd, vd, 0.3, causal, window)
        _close(o, o2, 0.0, f"GQA O mask{mi}")
        _close(lse, lse2, 0.0, f"GQA lse mask{mi}")


def _gather_contiguous(kc, vc, table, lens, s, bs):
    L = int(lens[s])
    tok = np.arange(L)
    phys = table[s, tok // bs]
    off = tok % bs
    return kc[phys, :, off, :].transpose(1, 0, 2), vc[phys, :, off, :].transpose(1, 0, 2)


def pin_paged_decode_equals_contiguous(orc):
    r = _rng(1100)
    S, Hq, Hkv, d, bs = 5, 8, 2, 8, 4
    lens = np.array([1, 4, 5, 13, 0], dtype=np.int32)
    nblk = (lens + bs - 1) // bs
    nb = int(nblk.sum()) + 3
    for identity in (True, False):
        perm = np.arange(nb) if identity else r.permutation(nb)
        table = np.full((S, 5), -1, dtype=np.int32)
        pos = 0
        for s in range(S):
            table[s, :nblk[s]] = perm[pos:pos + nblk[s]]
            pos += nblk[s]
        kc = r.standard_normal((nb, Hkv, bs, d))
        vc = r.standard_normal((nb, Hkv, bs, d))
        q = r.standard_normal((S, Hq, d))
        o, lse = orc.attn_decode(q, kc, vc, table, lens, 0.4)
        for s in range(S):
            ks, vs = _gather_contiguous(kc, vc, table, lens, s, bs)
            if lens[s] == 0:
                assert np.all(o[s] == 0) and np.all(lse[s] == -np.inf)
                continue
            of, lf = orc.attn_fwd(q[s][None, :, None, :], ks[None], vs[None], 0.4)
            _close(o[s], of[0, :, 0, :], 1e-14, f"decode O seq{s}")
            _close(lse[s], lf[0, :, 0], 1e-14, f"decode lse seq{s}")


def pin_numpy_bruteforce(orc):
    """Independent vectorised restatement on tiny inputs."""
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, v = _qkv(1200 + mi, 2, 4, 2, Nq, Nk, 3)
        o, lse = orc.attn_fwd(q, k, v, 0.6, causal, window)
        kk = np.repeat(k, 2, axis=1)
        vv = np.repeat(v, 2, axis=1)
        s = 0.6 * np.einsum("bhid,bhjd->bhij", q, kk)
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        diag = i + (Nk - Nq)
        keep = np.ones((Nq, Nk), dtype=bool)
        if causal:
            keep &= j <= diag
        if window >= 0:
            keep &= j >= diag - window
        s = np.where(keep, s, -np.inf)
        with np.errstate(invalid="ignore", divide="ignore"):
            lse_np = np.log(np.sum(np.exp(s), axis=-1))
            p = np.exp(s - lse_np[..., None])
        p = np.nan_to_num(p, nan=0.0)
        o_np = np.einsum("bhij,bhjd->bhid", p, vv)
        _close(o, o_np, 1e-12, f"numpy O mask{mi}")
        _close(lse, lse_np, 1e-12, f"numpy lse mask{mi}")


def pin_golden_three_keys(orc):
    with open(os.path.join(GOLDEN, "three_keys.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], dtype=np.float64)[None, None, None, :]
    k = np.array(g["k"], dtype=np.float64)[None, None]
    v = np.array(g["v"], dtype=np.float64)[None, None]
    for fn in (lambda: orc.attn_fwd(q, k, v, g["scale"]),
               lambda: orc.attn_fwd_blocked(q, k, v, g["scale"], block_r=1, block_c=2),
               lambda: orc.attn_fwd_split(q, k, v, g["scale"], chunk=2)):
        o, lse = fn()
        assert np.max(np.abs(o[0, 0, 0] - np.array(g["o"]))) <= 1e-14
        assert abs(lse[0, 0, 0] - g["lse"]) <= 1e-14


def pin_large_logits_and_late_maximum(orc):
    """Scores rising along the keys (largest last) and logits near 700, where a
    softmax without the max subtraction overflows."""
    d, Nk = 4, 64
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, 1, Nk, d))
    k[0, 0, :, 0] = np.linspace(0.0, 700.0, Nk)  # strictly increasing scores
    v = _rng(1300).standard_normal((1, 1, Nk, d))
    o, lse = orc.attn_fwd(q, k, v, 1.0)
    assert np.all(np.isfinite(o)) and np.isfinite(lse).all()
    gap = 700.0 / (Nk - 1)
    w = np.exp(-gap * np.arange(Nk)[::-1])        # relative weights to the last key
    want = (w[:, None] * v[0, 0]).sum(0) / w.sum()
    assert np.max(np.abs(o[0, 0, 0] - want)) <= 1e-13
    assert abs(lse[0, 0, 0] - (700.0 + math.log(w.sum()))) <= 1e-12
    for bc in (1, 3, 16):
        ob, lb = orc.attn_fwd_blocked(q, k, v, 1.0, block_r=1, block_c=bc)
        _close(ob, o, 1e-13, f"late-max blocked bc={bc}")
        _close(lb, lse, 1e-12, f"late-max blocked lse bc={bc}")


BWD_MASKS = [(6, 6, False, -1), (6, 6, True, -1), (4, 7, True, -1), (7, 4, True, -1), (6, 6, True, 2)]


def pin_bwd_finite_differences(orc):
    h = 1e-6
    for mi, (Nq, Nk, causal, window) in enumerate(BWD_MASKS):
        q, k, v = _qkv(1400 + mi, 1, 2, 1, Nq, Nk, 3)
        do = _rng(1450 + mi).standard_normal(q.shape)
        dq, dk, dv = orc.attn_bwd(q, k, v, do, 0.7, causal, window)

        def loss(q_, k_, v_):
            o, _ = orc.attn_fwd(q_, k_, v_, 0.7, causal, window)
            return float((o * do).sum())

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy(); xp[idx] += h
                xm = x.copy(); xm[idx] -= h
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.max(np.abs(num - g))
            assert err <= 1e-7 * max(1.0, np.max(np.abs(g))), f"d{name} finite differences mask{mi}: {err:.2e}"


def pin_bwd_torch_autograd(orc):
    import torch
    for mi, (Nq, Nk, causal, window) in enumerate(BWD_MASKS):
        q, k, v = _qkv(1500 + mi, 2, 4, 2, Nq, Nk, 5)
        do = _rng(1550 + mi).standard_normal(q.shape)
        dq, dk, dv = orc.attn_bwd(q, k, v, do, 0.45, causal, window)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        kk = tk.repeat_interleave(2, dim=1)
        vv = tv.repeat_interleave(2, dim=1)
        sc = 0.45 * tq @ kk.transpose(-1, -2)
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        diag = i + (Nk - Nq)
        keep = torch.ones(Nq, Nk, dtype=torch.bool)
        if causal:
            keep &= j <= diag
        if window >= 0:
            keep &= j >= diag - window
        sc = sc.masked_fill(~keep, float("-inf"))
        p = torch.softmax(sc, dim=-1)
        p = torch.nan_to_num(p, nan=0.0)  # rows with no key
        o = p @ vv
        (o * torch.tensor(do)).sum().backward()
        for name, mine, ref in (("q", dq, tq.grad), ("k", dk, tk.grad), ("v", dv, tv.grad)):
            assert np.max(np.abs(mine - ref.numpy())) <= 1e-12 * max(1.0, float(ref.abs().max())), \
                f"d{name} autograd mask{mi}"


def pin_bwd_invariants(orc):
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, v = _qkv(1600 + mi, 1, 4, 2, Nq, Nk, 8)
        do = _rng(1650 + mi).standard_normal(q.shape)
        dq, dk, dv = orc.attn_bwd(q, k, v, do, 0.3, causal, window)
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-11 * max(1.0, np.max(np.abs(dk))), f"sum dK mask{mi}"
        nonempty = np.array([_allowed_range(i, Nq, Nk, causal, window)[1] >
                             _allowed_range(i, Nq, Nk, causal, window)[0] for i in range(Nq)])
        for hk in range(2):
            want = do[0, 2 * hk:2 * hk + 2][:, nonempty].sum(axis=(0, 1))
            assert np.max(np.abs(dv[0, hk].sum(axis=0) - want)) <= 1e-11, f"sum dV mask{mi}"


def pin_bwd_gqa_equals_duplicated_heads(orc):
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS[:5]):
        q, k, v = _qkv(1700 + mi, 1, 6, 2, Nq, Nk, 4)
        do = _rng(1750 + mi).standard_normal(q.shape)
        dq, dk, dv = orc.attn_bwd(q, k, v, do, 0.3, causal, window)
        kd, vd = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
        dq2, dk2, dv2 = orc.attn_bwd(q, kd, vd, do, 0.3, causal, window)
        _close(dq, dq2, 1e-12, f"GQA dq mask{mi}")
        _close(dk, dk2.reshape(1, 2, 3, Nk, 4).sum(axis=2), 1e-12, f"GQA dk mask{mi}")
        _close(dv, dv2.reshape(1, 2, 3, Nk, 4).sum(axis=2), 1e-12, f"GQA dv mask{mi}")


def _paged_case(seed, S, Hq, Hkv, d, bs, q_lens, kv_lens, max_q, identity=False, extra=2):
    r = _rng(seed)
    kv = np.asarray(kv_lens, dtype=np.int32)
    nblk = (kv + bs - 1) // bs
    mb = int(max(1, nblk.max()))
    nb = int(nblk.sum()) + extra
    perm = np.arange(nb) if identity else r.permutation(nb)
    table = np.full((S, mb), -1, dtype=np.int32)
    pos = 0
    for s in range(S):
        table[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += nblk[s]
    kc = r.standard_normal((nb, Hkv, bs, d))
    vc = r.standard_normal((nb, Hkv, bs, d))
    q = r.standard_normal((S, Hq, max_q, d))
    return q, kc, vc, table, np.asarray(q_lens, dtype=np.int32), kv


def pin_paged_prefill_single_query_is_decode(orc):
    """One new query per sequence: the last position sees every key, as in decode."""
    S, Hq, Hkv, d, bs = 4, 6, 2, 8, 4
    kv = [1, 5, 9, 13]
    q, kc, vc, table, ql, kl = _paged_case(1800, S, Hq, Hkv, d, bs, [1] * S, kv, 3)
    o, lse = orc.attn_prefill_paged(q, kc, vc, table, ql, kl, 0.5, causal=True)
    od, ld = orc.attn_decode(q[:, :, 0, :], kc, vc, table, kl, 0.5)
    _close(o[:, :, 0, :], od, 1e-14, "paged prefill q_len=1 O")
    _close(lse[:, :, 0], ld, 1e-14, "paged prefill q_len=1 lse")
    assert np.all(o[:, :, 1:, :] == 0) and np.all(np.isnan(lse[:, :, 1:])), "rows past q_len must stay untouched"


def pin_paged_prefill_equals_gathered_prefill(orc):
    """Keys and values gathered with numpy fancy indexing (a second implementation of
    the address formula), then the pinned prefill with Nq = q_len, Nk = kv_len."""
    S, Hq, Hkv, d = 3, 4, 2, 8
    for bs, identity in ((4, True), (4, False), (8, False), (16, False)):
        for causal, window in ((True, -1), (False, -1), (True, 3)):
            ql, kv = [5, 1, 7], [9, 1, 23]
            q, kc, vc, table, ql, kl = _paged_case(1850 + bs + (7 if identity else 0), S, Hq, Hkv, d, bs, ql, kv, 8,
                                                   identity=identity)
            o, lse = orc.attn_prefill_paged(q, kc, vc, table, ql, kl, 0.3, causal=causal, window=window)
            for s in range(S):
                t = np.arange(kl[s])
                phys = table[s, t // bs]
                ks = kc[phys, :, t % bs, :].transpose(1, 0, 2)  # [Hkv][kv_len][d]
                vs = vc[phys, :, t % bs, :].transpose(1, 0, 2)
                of, lf = orc.attn_fwd(q[s:s + 1, :, :ql[s], :], ks[None], vs[None], 0.3, causal, window)
                _close(o[s, :, :ql[s], :], of[0], 1e-14, f"paged prefill bs={bs} seq{s} O")
                _close(lse[s, :, :ql[s]], lf[0], 1e-14, f"paged prefill bs={bs} seq{s} lse")


def _csr(pattern):
    """Dense boolean block pattern [n_qblk][n_kblk] -> (row_ptr, col_idx)."""
    rows = [np.flatnonzero(r).astype(np.int32) for r in np.asarray(pattern, dtype=bool)]
    row_ptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    col_idx = np.concatenate(rows).astype(np.int32) if sum(len(r) for r in rows) else np.zeros(0, np.int32)
    return row_ptr, col_idx


def pin_blocksparse_full_pattern_is_dense(orc):
    """Every block listed: exactly the dense masks."""
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        q, k, v = _qkv(1900 + mi, 1, 4, 2, Nq, Nk, 4)
        for bq, bk in ((3, 5), (4, 4), (Nq, Nk)):
            nqb, nkb = -(-Nq // bq), -(-Nk // bk)
            rp, ci = _csr(np.ones((nqb, nkb)))
            o, lse = orc.attn_fwd_blocksparse(q, k, v, rp, ci, 0.5, causal, window, bq, bk)
            od, ld = orc.attn_fwd(q, k, v, 0.5, causal, window)
            _close(o, od, 1e-14, f"full pattern O {mi} ({bq},{bk})")
            _close(lse, ld, 1e-14, f"full pattern lse {mi} ({bq},{bk})")


def pin_blocksparse_numpy_bruteforce(orc):
    """Random block patterns (empty block rows included), unequal block sizes: the element
    mask is the block pattern expanded with numpy, intersected with the dense mask."""
    r = _rng(1950)
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS):
        bq, bk = 2, 3
        nqb, nkb = -(-Nq // bq), -(-Nk // bk)
        pat = r.random((nqb, nkb)) < 0.5
        pat[0, :] = False  # an empty block row
        rp, ci = _csr(pat)
        q, k, v = _qkv(1960 + mi, 1, 2, 1, Nq, Nk, 3)
        o, lse = orc.attn_fwd_blocksparse(q, k, v, rp, ci, 0.7, causal, window, bq, bk)
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        diag = i + (Nk - Nq)
        keep = pat[i // bq, j // bk]
        if causal:
            keep = keep & (j <= diag)
        if window >= 0:
            keep = keep & (j >= diag - window)
        s = 0.7 * np.einsum("bhid,bhjd->bhij", q, np.repeat(k, 2, axis=1))
        s = np.where(keep, s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        e = np.where(keep, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
        l = e.sum(axis=-1, keepdims=True)
        pr = np.divide(e, l, out=np.zeros_like(e), where=l > 0)
        ref_o = np.einsum("bhij,bhjd->bhid", pr, np.repeat(v, 2, axis=1))
        ref_lse = np.where(l[..., 0] > 0, m[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
        _close(o, ref_o, 1e-13, f"blocksparse numpy O {mi}")
        assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), "blocksparse empty-row pattern"
        fin = np.isfinite(ref_lse)
        _close(lse[fin], ref_lse[fin], 1e-13, f"blocksparse numpy lse {mi}")


def pin_blocksparse_block_diagonal_is_segments(orc):
    """A block-diagonal pattern (equal block sizes, no other mask) splits the sequence into
    independent segments: each equals plain attention on its slice."""
    N, b = 12, 4
    q, k, v = _qkv(1990, 1, 2, 2, N, N, 5)
    rp, ci = _csr(np.eye(N // b, dtype=bool))
    o, lse = orc.attn_fwd_blocksparse(q, k, v, rp, ci, 0.4, False, -1, b, b)
    for t in range(N // b):
        sl = slice(t * b, (t + 1) * b)
        os_, ls_ = orc.attn_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.4)
        _close(o[:, :, sl], os_, 1e-14, f"segment {t} O")
        _close(lse[:, :, sl], ls_, 1e-14, f"segment {t} lse")


def pin_e4m3_decode(orc):
    """E4M3 codes: closed forms from the format definition, strict order of the positive
    codes, and all 256 codes against torch's float8_e4m3fn conversion."""
    closed = {0x38: 1.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x07: 7.0 / 8 * 2.0 ** -6, 0x08: 2.0 ** -6, 0xB8: -1.0,
              0x40: 2.0, 0x30: 0.5, 0x3C: 1.5, 0x77: 240.0, 0x00: 0.0}
    codes = np.array(list(closed), dtype=np.uint8)
    _close(orc.e4m3_decode(codes), np.array(list(closed.values())), 0.0, "e4m3 closed forms")
    z = orc.e4m3_decode(np.array([0x80, 0x7F, 0xFF], dtype=np.uint8))
    assert z[0] == 0.0 and np.signbit(z[0]) and np.isnan(z[1]) and np.isnan(z[2]), "e4m3 -0 / NaN codes"
    pos = orc.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0), "positive E4M3 codes must increase strictly"
    try:
        import torch
    except ImportError:
        return
    allc = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allc.copy()).view(torch.float8_e4m3fn).float().double().numpy()
    got = orc.e4m3_decode(allc)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "e4m3 NaN codes differ from torch"
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "e4m3 values differ from torch float8_e4m3fn"


def _fp8_case(seed, B, Hq, Hkv, Nq, Nk, d):
    r = _rng(seed)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    q8 = r.choice(finite, (B, Hq, Nq, d))
    k8 = r.choice(finite, (B, Hkv, Nk, d))
    vt8 = r.choice(finite, (B, Hkv, d, Nk))
    return q8, k8, vt8


def pin_fp8_numpy_bruteforce(orc):
    """FP8 attention = numpy softmax attention over the decoded values (decoded by torch's
    float8_e4m3fn, V transposed back with numpy) times the per-tensor scales."""
    try:
        import torch
    except ImportError:
        return
    dec = lambda c: torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).double().numpy()
    for mi, (Nq, Nk, causal, window) in enumerate(MASKS[:5]):
        q8, k8, vt8 = _fp8_case(2100 + mi, 1, 2, 1, Nq, Nk, 4)
        qs, ks, vs, sc = 0.003, 0.0021, 0.013, 0.5
        o, lse = orc.attn_fwd_fp8(q8, k8, vt8, sc, qs, ks, vs, causal, window)
        q = dec(q8) * qs
        k = np.repeat(dec(k8) * ks, 2, axis=1)
        v = np.repeat(np.swapaxes(dec(vt8), 2, 3) * vs, 2, axis=1)
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        diag = i + (Nk - Nq)
        keep = np.ones((Nq, Nk), dtype=bool)
        if causal:
            keep &= j <= diag
        if window >= 0:
            keep &= j >= diag - window
        s_ = sc * np.einsum("bhid,bhjd->bhij", q, k)
        s_ = np.where(keep, s_, -np.inf)
        m = s_.max(axis=-1, keepdims=True)
        e = np.where(keep, np.exp(s_ - np.where(np.isfinite(m), m, 0.0)), 0.0)
        l = e.sum(axis=-1, keepdims=True)
        pr = np.divide(e, l, out=np.zeros_like(e), where=l > 0)
        _close(o, np.einsum("bhij,bhjd->bhid", pr, v), 1e-13, f"fp8 numpy O {mi}")
        ref_lse = np.where(l[..., 0] > 0, m[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
        _close(lse, ref_lse, 1e-12, f"fp8 numpy lse {mi}")


def pin_fp8_scale_folding(orc):
    """The scales enter as the definition says: doubling q's scale equals doubling the
    softmax scale; V's scale multiplies O and leaves lse unchanged."""
    q8, k8, vt8 = _fp8_case(2200, 1, 2, 2, 9, 11, 8)
    o1, l1 = orc.attn_fwd_fp8(q8, k8, vt8, 0.3, 0.02, 0.01, 0.05, True, -1)
    o2, l2 = orc.attn_fwd_fp8(q8, k8, vt8, 0.6, 0.01, 0.01, 0.05, True, -1)
    _close(o1, o2, 1e-14, "fp8 q scale vs softmax scale (O)")
    _close(l1, l2, 1e-12, "fp8 q scale vs softmax scale (lse)")
    o3, l3 = orc.attn_fwd_fp8(q8, k8, vt8, 0.3, 0.02, 0.01, 0.1, True, -1)
    _close(o3, 2.0 * o1, 1e-14, "fp8 v scale multiplies O")
    _close(l3, l1, 0.0, "fp8 v scale leaves lse")


ALL_PINS = [
    pin_blocked_equals_materialised,
    pin_split_equals_unsplit,
    pin_probabilities_sum_to_one,
    pin_equal_scores_give_mean,
    pin_dominant_key,
    pin_first_causal_row,
    pin_translation_invariance,
    pin_permutation_invariance,
    pin_long_window_is_plain_mask,
    pin_gqa_equals_duplicated_heads,
    pin_paged_decode_equals_contiguous,
    pin_numpy_bruteforce,
    pin_golden_three_keys,
    pin_large_logits_and_late_maximum,
    pin_bwd_finite_differences,
    pin_bwd_torch_autograd,
    pin_bwd_invariants,
    pin_bwd_gqa_equals_duplicated_heads,
    pin_paged_prefill_single_query_is_decode,
    pin_paged_prefill_equals_gathered_prefill,
    pin_blocksparse_full_pattern_is_dense,
    pin_blocksparse_numpy_bruteforce,
    pin_blocksparse_block_diagonal_is_segments,
    pin_e4m3_decode,
    pin_fp8_numpy_bruteforce,
    pin_fp8_scale_folding,
]
