"""Pins for the fp64 oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` takes an oracle build (``lib=None`` means the real one) and
raises ``AssertionError`` on a mismatch.  The same pins run against the real
oracle (they must all pass) and against copies of the oracle with a planted
mistake (at least one must fail), see ``test_oracle.py``.

What pins what:
  * hand-computed closed forms in ``tests/golden/*.json`` (scale, causal mask,
    bottom-right alignment, GQA head map, split rule, split + merge);
  * exact brute force on tiny inputs: scores in rational arithmetic, exp/ln
    in 50-digit decimal arithmetic, textbook softmax without max subtraction;
  * a library routine: torch's float64 scaled_dot_product_attention, with
    torch's own lower-right causal bias for Sq != Skv;
  * invariants: rows of P sum to one, permutation invariance (non-causal),
    linearity in V, split-then-merge == unsplit, merge of one split ==
    identity, decode == prefill with one query;
  * closed forms: equal keys, causal row 0, Q = 0, one dominant key, and a
    constant score shift.
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-12


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    both_ninf = np.isneginf(a) & np.isneginf(b)
    assert np.array_equal(np.isneginf(a), np.isneginf(b)), f"{what}: -inf pattern differs"
    assert not np.isnan(a).any(), f"{what}: NaN"
    d = np.where(both_ninf, 0.0, np.abs(np.where(both_ninf, 0.0, a) - np.where(both_ninf, 0.0, b)))
    err = float(d.max()) if d.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def _bf16(shape, rng, scale=1.0):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
    return x.to(torch.bfloat16).to(torch.float64).numpy()


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)

    def arr(x):
        return np.array([float(t) for t in x], np.float64)

    return g, arr


# ---------------------------------------------------------------- fixtures
def _pin_golden_prefill(name, lib):
    g, arr = _golden(name)
    B, Hq, Hkv, Sq, Skv, d = g["B"], g["Hq"], g["Hkv"], g["Sq"], g["Skv"], g["d"]
    q = arr(g["q"]).reshape(B, Sq, Hq, d)
    k = arr(g["k"]).reshape(B, Skv, Hkv, d)
    v = arr(g["v"]).reshape(B, Skv, Hkv, d)
    o, lse = oracle.sdpa(q, k, v, g["causal"], g["scale"], lib=lib)
    _close(o.reshape(-1), arr(g["expect_o"]), g["tol"], name + " O")
    _close(lse.reshape(-1), arr(g["expect_lse"]), g["tol"], name + " LSE")


def pin_golden_two_key(lib=None):
    _pin_golden_prefill("two_key_ln2.json", lib)


def pin_golden_causal_prefix(lib=None):
    _pin_golden_prefill("causal_prefix_mean.json", lib)


def pin_golden_bottom_right(lib=None):
    _pin_golden_prefill("causal_bottom_right.json", lib)


def pin_golden_gqa_map(lib=None):
    _pin_golden_prefill("gqa_head_map.json", lib)


def pin_golden_split_merge(lib=None):
    g, arr = _golden("split_merge_uniform.json")
    B, Hq, Hkv, d, Lmax = g["B"], g["Hq"], g["Hkv"], g["d"], g["Lmax"]
    q = arr(g["q"]).reshape(B, Hq, d)
    k = arr(g["k"]).reshape(B, Lmax, Hkv, d)
    v = arr(g["v"]).reshape(B, Lmax, Hkv, d)
    lens = np.array(g["kv_lens"], np.int32)
    po, pl = oracle.decode_split(q, k, v, lens, g["scale"], g["n_splits"], g["min_rows"], lib=lib)
    _close(po.reshape(-1), arr(g["expect_part_o"]), g["tol"], "split part_o")
    _close(pl.reshape(-1), arr(g["expect_part_lse"]), g["tol"], "split part_lse")
    o, lse = oracle.merge(po, pl, lib=lib)
    _close(o.reshape(-1), arr(g["expect_o"]), g["tol"], "merge O")
    _close(lse.reshape(-1), arr(g["expect_lse"]), g["tol"], "merge LSE")
    o2, lse2 = oracle.decode(q, k, v, lens, g["scale"], lib=lib)
    _close(o2.reshape(-1), arr(g["expect_o"]), g["tol"], "decode O")
    _close(lse2.reshape(-1), arr(g["expect_lse"]), g["tol"], "decode LSE")


def pin_golden_split_rule(lib=None):
    g, _ = _golden("split_rule.json")
    for c in g["cases"]:
        got = [list(oracle.split_bounds(c["L"], c["n_splits"], c["min_rows"], s, lib=lib))
               for s in range(c["n_splits"])]
        assert got == c["bounds"], f"split rule {c['L'], c['n_splits'], c['min_rows']}: {got}"


# ---------------------------------------------------------------- brute force
def _exact_attention(q, k, v, causal, scale):
    """Textbook softmax in exact / 50-digit arithmetic: exp(s)/sum exp(s), no max."""
    getcontext().prec = 50
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    group = Hq // Hkv
    sc = Fraction(scale)
    o = np.zeros((B, Sq, Hq, d))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            kvh = h // group
            for i in range(Sq):
                pos = i + (Skv - Sq)  # key position of query i
                allowed = [j for j in range(Skv) if (not causal) or j <= pos]
                if not allowed:
                    lse[b, h, i] = -math.inf
                    continue
                ex = []
                for j in allowed:
                    s = sc * sum(Fraction(float(q[b, i, h, t])) * Fraction(float(k[b, j, kvh, t]))
                                 for t in range(d))
                    ex.append((Decimal(s.numerator) / Decimal(s.denominator)).exp())
                Z = sum(ex)
                for t in range(d):
                    num = sum(e * Decimal(float(v[b, j, kvh, t])) for e, j in zip(ex, allowed))
                    o[b, i, h, t] = float(num / Z)
                lse[b, h, i] = float(Z.ln())
    return o, lse


def pin_brute_force_exact(lib=None):
    rng = np.random.default_rng(12345)
    cases = [
        (1, 1, 1, 1, 1, 1, False, 0.5),
        (1, 2, 2, 4, 4, 3, True, 0.125),
        (2, 4, 2, 3, 5, 4, True, 0.25),    # Sq < Skv, bottom-right causal, GQA
        (1, 4, 2, 5, 3, 3, True, 0.5),     # Sq > Skv: first rows fully masked
        (2, 6, 3, 4, 6, 2, False, 0.5),
        (1, 4, 1, 3, 7, 5, False, 1.0 / 8),
    ]
    for B, Hq, Hkv, Sq, Skv, d, causal, scale in cases:
        q = _bf16((B, Sq, Hq, d), rng)
        k = _bf16((B, Skv, Hkv, d), rng)
        v = _bf16((B, Skv, Hkv, d), rng)
        o, lse = oracle.sdpa(q, k, v, causal, scale, lib=lib)
        eo, el = _exact_attention(q, k, v, causal, scale)
        tag = f"brute {B, Hq, Hkv, Sq, Skv, d, causal}"
        _close(o, eo, 1e-12, tag + " O")
        _close(lse, el, 1e-12, tag + " LSE")
        # the selected-rows entry point computes the same rows
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(Sq)]
        ro, rl = oracle.sdpa_rows(q, k, v, causal, scale, rows, lib=lib)
        _close(ro, np.stack([eo[b, i, h] for b, h, i in rows]), 1e-12, tag + " rows O")
        _close(rl, np.array([el[b, h, i] for b, h, i in rows]), 1e-12, tag + " rows LSE")


def pin_varlen_brute_force(lib=None):
    """Packed variable-length prefill: every sequence against an independent brute
    force of its own rows and keys (offsets, key ranges, bottom-right causal bound
    of the new rows after a history, the [Hq, total_q] LSE layout)."""
    rng = np.random.default_rng(2468)
    Hq, Hkv, d, max_kv = 4, 2, 3, 7
    seqs = [(2, 5), (0, 3), (3, 3), (1, 7), (2, 0)]  # (new query rows Sq_b, keys L_b)
    B = len(seqs)
    cu = np.cumsum([0] + [sq for sq, _ in seqs]).astype(np.int32)
    lens = np.array([L for _, L in seqs], np.int32)
    q = _bf16((int(cu[-1]), Hq, d), rng)
    kc = _bf16((B, max_kv, Hkv, d), rng)
    vc = _bf16((B, max_kv, Hkv, d), rng)
    for causal in (True, False):
        o, lse = oracle.sdpa_varlen(q, kc, vc, cu, lens, causal, 0.5, lib=lib)
        assert o.shape == (cu[-1], Hq, d) and lse.shape == (Hq, cu[-1])
        for b, (sq, L) in enumerate(seqs):
            if sq == 0:
                continue
            eo, el = _exact_attention(q[None, cu[b]:cu[b + 1]], kc[b:b + 1, :L], vc[b:b + 1, :L], causal, 0.5)
            _close(o[cu[b]:cu[b + 1]], eo[0], 1e-12, f"varlen b={b} causal={causal} O")
            _close(lse[:, cu[b]:cu[b + 1]], el[0], 1e-12, f"varlen b={b} causal={causal} LSE")


def _exact_window(q, k, v, window, n_sink, scale):
    """Brute force of causal attention over a window plus sinks, with the mask as
    an explicit key set per query (independent of the oracle's predicate)."""
    getcontext().prec = 50
    B, Sq, Hq, d = q.shape
    _, Skv, Hkv, _ = k.shape
    group = Hq // Hkv
    o = np.zeros((B, Sq, Hq, d))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            kvh = h // group
            for i in range(Sq):
                p = i + (Skv - Sq)
                keys = set(range(max(0, p - window + 1), min(p, Skv - 1) + 1)) | set(range(min(n_sink, p + 1, Skv)))
                allowed = sorted(keys)
                if not allowed:
                    lse[b, h, i] = -math.inf
                    continue
                ex = []
                for j in allowed:
                    s_ = Fraction(scale) * sum(Fraction(float(q[b, i, h, t])) * Fraction(float(k[b, j, kvh, t]))
                                               for t in range(d))
                    ex.append((Decimal(s_.numerator) / Decimal(s_.denominator)).exp())
                Z = sum(ex)
                for t in range(d):
                    o[b, i, h, t] = float(sum(e * Decimal(float(v[b, j, kvh, t])) for e, j in zip(ex, allowed)) / Z)
                lse[b, h, i] = float(Z.ln())
    return o, lse


def pin_window_brute_force(lib=None):
    """Sliding window plus sinks against the exact brute force, including windows of
    one position, sinks overlapping the window, Sq < Skv and Sq > Skv."""
    rng = np.random.default_rng(97531)
    cases = [  # B, Hq, Hkv, Sq, Skv, d, window, n_sink
        (1, 2, 1, 9, 9, 3, 3, 2),
        (1, 2, 2, 7, 7, 2, 1, 0),
        (2, 4, 2, 4, 10, 3, 4, 3),   # new rows after a history
        (1, 2, 1, 6, 4, 2, 2, 1),    # more rows than keys: early rows see nothing
        (1, 1, 1, 8, 8, 4, 5, 8),    # sinks cover everything: plain causal
    ]
    for B, Hq, Hkv, Sq, Skv, d, W_, ns in cases:
        q, k, v = _bf16((B, Sq, Hq, d), rng), _bf16((B, Skv, Hkv, d), rng), _bf16((B, Skv, Hkv, d), rng)
        o, lse = oracle.sdpa_window(q, k, v, W_, ns, 0.5, lib=lib)
        eo, el = _exact_window(q, k, v, W_, ns, 0.5)
        tag = f"window {B, Hq, Hkv, Sq, Skv, d, W_, ns}"
        _close(o, eo, 1e-12, tag + " O")
        _close(lse, el, 1e-12, tag + " LSE")
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(Sq)]
        ro, rl = oracle.sdpa_window_rows(q, k, v, W_, ns, 0.5, rows, lib=lib)
        _close(ro, np.stack([eo[b, i, h] for b, h, i in rows]), 1e-12, tag + " rows O")
        _close(rl, np.array([el[b, h, i] for b, h, i in rows]), 1e-12, tag + " rows LSE")


def pin_varlen_window_brute_force(lib=None):
    """Packed sequences with a sliding window and sinks: every sequence against the
    explicit-key-set brute force of its own rows and keys (offsets, per-sequence key
    counts, the window measured from each sequence's own bottom-right position)."""
    rng = np.random.default_rng(1357)
    Hq, Hkv, d, max_kv = 4, 2, 3, 12
    seqs = [(3, 9), (0, 4), (5, 5), (2, 12), (4, 2), (1, 0)]  # (new query rows, keys)
    B = len(seqs)
    cu = np.cumsum([0] + [sq for sq, _ in seqs]).astype(np.int32)
    lens = np.array([L for _, L in seqs], np.int32)
    q = _bf16((int(cu[-1]), Hq, d), rng)
    kc = _bf16((B, max_kv, Hkv, d), rng)
    vc = _bf16((B, max_kv, Hkv, d), rng)
    for W_, ns in ((3, 2), (1, 0), (4, 5)):
        o, lse = oracle.sdpa_varlen_window(q, kc, vc, cu, lens, W_, ns, 0.5, lib=lib)
        assert o.shape == (cu[-1], Hq, d) and lse.shape == (Hq, cu[-1])
        for b, (sq, L) in enumerate(seqs):
            if sq == 0:
                continue
            eo, el = _exact_window(q[None, cu[b]:cu[b + 1]], kc[b:b + 1, :L], vc[b:b + 1, :L], W_, ns, 0.5)
            _close(o[cu[b]:cu[b + 1]], eo[0], 1e-12, f"varlen window b={b} W={W_} sinks={ns} O")
            _close(lse[:, cu[b]:cu[b + 1]], el[0], 1e-12, f"varlen window b={b} W={W_} sinks={ns} LSE")


def pin_window_closed_forms(lib=None):
    """A window of one position returns the query's own value row (LSE = its own
    score); a window or sink set covering every key is plain causal attention; and
    the union of a window and disjoint sinks is the LSE merge of the two branches
    computed separately (the FMHA page's two-pass form)."""
    rng = np.random.default_rng(8642)
    B, Hq, Hkv, S, d = 1, 4, 2, 40, 8
    q, k, v = _bf16((B, S, Hq, d), rng), _bf16((B, S, Hkv, d), rng), _bf16((B, S, Hkv, d), rng)
    o, lse = oracle.sdpa_window(q, k, v, 1, 0, 0.3, lib=lib)
    hk = [h // (Hq // Hkv) for h in range(Hq)]
    _close(o[0], np.stack([v[0, :, hk[h]] for h in range(Hq)], 1), 1e-12, "window 1 O")
    own = np.stack([[0.3 * float(np.dot(q[0, i, h].astype(np.float64), k[0, i, hk[h]].astype(np.float64)))
                     for i in range(S)] for h in range(Hq)])
    _close(lse[0], own, 1e-12, "window 1 LSE")
    oc, lc = oracle.sdpa(q, k, v, True, 0.3, lib=lib)
    for W_, ns in ((S, 0), (10 * S, 3), (2, S)):
        ow, lw = oracle.sdpa_window(q, k, v, W_, ns, 0.3, lib=lib)
        _close(ow, oc, 1e-12, f"cover W={W_} sinks={ns} O")
        _close(lw, lc, 1e-12, f"cover W={W_} sinks={ns} LSE")
    # two branches: rows i >= W_ + ns have disjoint window [i-W_+1, i] and sinks [0, ns)
    W_, ns = 6, 4
    ow, lw = oracle.sdpa_window(q, k, v, W_, ns, 0.3, lib=lib)
    for i in range(W_ + ns, S):
        for h in range(Hq):
            lo = i - W_ + 1
            win = oracle.sdpa(q[:, i:i + 1], k[:, lo:i + 1], v[:, lo:i + 1], False, 0.3, lib=lib)
            snk = oracle.sdpa(q[:, i:i + 1], k[:, :ns], v[:, :ns], False, 0.3, lib=lib)
            lw_, ls_ = win[1][0, h, 0], snk[1][0, h, 0]
            M = max(lw_, ls_)
            a, b_ = math.exp(lw_ - M), math.exp(ls_ - M)
            om = (a * win[0][0, 0, h] + b_ * snk[0][0, 0, h]) / (a + b_)
            _close(ow[0, i, h], om, 1e-12, f"two-branch merge row {i} O")
            _close(lw[0, h, i], M + math.log(a + b_), 1e-12, f"two-branch merge row {i} LSE")


# ---------------------------------------------------------------- library routine
def pin_torch_sdpa(lib=None):
    from torch.nn.attention.bias import causal_lower_right
    rng = np.random.default_rng(7)
    for B, Hq, Hkv, Sq, Skv, d, causal in [(2, 4, 2, 33, 33, 16, True), (1, 6, 2, 17, 40, 8, True),
                                           (2, 4, 4, 20, 31, 32, False), (1, 2, 1, 9, 9, 64, True)]:
        scale = 1.0 / math.sqrt(d)
        q = _bf16((B, Sq, Hq, d), rng)
        k = _bf16((B, Skv, Hkv, d), rng)
        v = _bf16((B, Skv, Hkv, d), rng)
        o, lse = oracle.sdpa(q, k, v, causal, scale, lib=lib)
        G = Hq // Hkv
        tq = torch.from_numpy(q).permute(0, 2, 1, 3)  # B,H,S,d
        tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
        tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
        mask = causal_lower_right(Sq, Skv) if causal else None
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
        _close(o, ref.permute(0, 2, 1, 3).numpy(), 1e-12, "torch sdpa O")
        # LSE through torch.logsumexp of torch.matmul scores, lower-right mask
        s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
        if causal:
            i = torch.arange(Sq).view(-1, 1)
            j = torch.arange(Skv).view(1, -1)
            s = s.masked_fill(j > i + (Skv - Sq), float("-inf"))
        _close(lse, torch.logsumexp(s, dim=-1).numpy(), 1e-12, "torch logsumexp LSE")


def pin_head_dim_512(lib=None):
    """Head dimension 512 (the prefill's widest head): exact brute force on a tiny
    causal GQA case with Sq < Skv, and torch's float64 SDPA on a larger one with
    Sq > Skv (fully masked leading rows)."""
    from torch.nn.attention.bias import causal_lower_right
    rng = np.random.default_rng(512)
    B, Hq, Hkv, Sq, Skv, d = 1, 2, 1, 3, 5, 512
    scale = 1.0 / math.sqrt(d)
    q, k, v = _bf16((B, Sq, Hq, d), rng), _bf16((B, Skv, Hkv, d), rng), _bf16((B, Skv, Hkv, d), rng)
    o, lse = oracle.sdpa(q, k, v, True, scale, lib=lib)
    eo, el = _exact_attention(q, k, v, True, scale)
    _close(o, eo, 1e-12, "d512 brute O")
    _close(lse, el, 1e-12, "d512 brute LSE")
    B, Hq, Hkv, Sq, Skv = 2, 4, 2, 37, 29
    q, k, v = _bf16((B, Sq, Hq, d), rng), _bf16((B, Skv, Hkv, d), rng), _bf16((B, Skv, Hkv, d), rng)
    o, lse = oracle.sdpa(q, k, v, True, scale, lib=lib)
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    live = Sq - Skv  # rows before this one admit no key (bottom-right alignment)
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq[:, :, live:], tk, tv, attn_mask=causal_lower_right(Sq - live, Skv), scale=scale)
    _close(o[:, live:], ref.permute(0, 2, 1, 3).numpy(), 1e-12, "d512 torch sdpa O")
    assert np.all(o[:, :live] == 0) and np.all(np.isneginf(lse[:, :, :live])), "d512 masked rows"
    s_ = torch.matmul(tq, tk.transpose(-1, -2)) * scale
    i = torch.arange(Sq).view(-1, 1)
    j = torch.arange(Skv).view(1, -1)
    s_ = s_.masked_fill(j > i + (Skv - Sq), float("-inf"))
    _close(lse[:, :, live:], torch.logsumexp(s_, dim=-1)[:, :, live:].numpy(), 1e-12, "d512 LSE")


# ---------------------------------------------------------------- invariants
def pin_rows_sum_to_one(lib=None):
    """V = a constant per KV head -> O = that constant iff every row of P sums to 1."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, Sq, Skv, d = 2, 4, 2, 13, 13, 8
    q = _bf16((B, Sq, Hq, d), rng, 2.0)
    k = _bf16((B, Skv, Hkv, d), rng, 2.0)
    c = np.array([1.5, -2.25])
    v = np.broadcast_to(c.reshape(1, 1, Hkv, 1), (B, Skv, Hkv, d)).copy()
    for causal in (False, True):
        o, _ = oracle.sdpa(q, k, v, causal, 0.3, lib=lib)
        expect = np.broadcast_to(np.repeat(c, Hq // Hkv).reshape(1, 1, Hq, 1), o.shape)
        _close(o, expect, 1e-12, f"P rows sum to one (causal={causal})")


def pin_permutation_invariance(lib=None):
    rng = np.random.default_rng(4)
    B, Hq, Hkv, Sq, Skv, d = 1, 4, 2, 9, 21, 16
    q, k, v = _bf16((B, Sq, Hq, d), rng), _bf16((B, Skv, Hkv, d), rng), _bf16((B, Skv, Hkv, d), rng)
    perm = rng.permutation(Skv)
    o1, l1 = oracle.sdpa(q, k, v, False, 0.25, lib=lib)
    o2, l2 = oracle.sdpa(q, k[:, perm], v[:, perm], False, 0.25, lib=lib)
    _close(o1, o2, 1e-12, "permutation O")
    _close(l1, l2, 1e-12, "permutation LSE")


def pin_linearity_in_v(lib=None):
    rng = np.random.default_rng(5)
    B, Hq, Hkv, Sq, Skv, d = 1, 2, 2, 11, 11, 8
    q, k = _bf16((B, Sq, Hq, d), rng), _bf16((B, Skv, Hkv, d), rng)
    v1, v2 = _bf16((B, Skv, Hkv, d), rng), _bf16((B, Skv, Hkv, d), rng)
    oa, _ = oracle.sdpa(q, k, v1, True, 0.5, lib=lib)
    ob, _ = oracle.sdpa(q, k, v2, True, 0.5, lib=lib)
    oc, _ = oracle.sdpa(q, k, v1 + 2.0 * v2, True, 0.5, lib=lib)
    _close(oc, oa + 2.0 * ob, 1e-12, "linearity in V")


def _decode_case(rng, B=5, Hq=6, Hkv=2, d=16, lens=(1, 29, 52, 0, 77)):
    Lmax = max(lens) if lens else 0
    q = _bf16((B, Hq, d), rng)
    kc = _bf16((B, Lmax, Hkv, d), rng)
    vc = _bf16((B, Lmax, Hkv, d), rng)
    return q, kc, vc, np.array(lens, np.int32)


def pin_split_merge_equals_unsplit(lib=None):
    rng = np.random.default_rng(6)
    q, kc, vc, lens = _decode_case(rng)
    o_ref, l_ref = oracle.decode(q, kc, vc, lens, 0.25, lib=lib)
    for n_splits, min_rows in [(1, 1), (3, 1), (8, 1), (16, 5), (4, 100), (7, 0)]:
        po, pl = oracle.decode_split(q, kc, vc, lens, 0.25, n_splits, min_rows, lib=lib)
        o, lse = oracle.merge(po, pl, lib=lib)
        _close(o, o_ref, 1e-12, f"split+merge O ({n_splits},{min_rows})")
        _close(lse, l_ref, 1e-12, f"split+merge LSE ({n_splits},{min_rows})")
        # empty splits carry o = 0, lse = -inf
        for b, L in enumerate(lens):
            for s in range(n_splits):
                lo, hi = oracle.split_bounds(int(L), n_splits, min_rows, s, lib=lib)
                if lo == hi:
                    assert np.all(np.isneginf(pl[b, :, s])) and np.all(po[b, :, s] == 0.0)


def pin_merge_identity(lib=None):
    rng = np.random.default_rng(8)
    po = rng.standard_normal((3, 4, 1, 8))
    pl = rng.standard_normal((3, 4, 1)) * 3
    pl[1, 2, 0] = -math.inf
    po[1, 2, 0] = 0.0
    o, lse = oracle.merge(po, pl, lib=lib)
    _close(o, po[:, :, 0], 1e-15, "merge identity O")
    _close(lse, pl[:, :, 0], 1e-15, "merge identity LSE")


def pin_decode_equals_prefill(lib=None):
    rng = np.random.default_rng(9)
    q, kc, vc, lens = _decode_case(rng)
    o, lse = oracle.decode(q, kc, vc, lens, 0.3, lib=lib)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(np.isneginf(lse[b])) and np.all(o[b] == 0.0)
            continue
        po, pl = oracle.sdpa(q[b:b + 1, None], kc[b:b + 1, :L], vc[b:b + 1, :L], False, 0.3, lib=lib)
        _close(o[b], po[0, 0], 1e-12, "decode vs prefill O")
        _close(lse[b], pl[0, :, 0], 1e-12, "decode vs prefill LSE")


# ---------------------------------------------------------------- closed forms
def pin_closed_forms(lib=None):
    rng = np.random.default_rng(10)
    B, Hq, Hkv, S, d = 1, 2, 1, 12, 8
    # (a) all keys equal -> uniform P over admissible keys
    q = _bf16((B, S, Hq, d), rng)
    k1 = _bf16((1, 1, 1, d), rng)
    k = np.broadcast_to(k1, (B, S, Hkv, d)).copy()
    v = _bf16((B, S, Hkv, d), rng)
    o, lse = oracle.sdpa(q, k, v, True, 0.5, lib=lib)
    for i in range(S):
        for h in range(Hq):
            s = 0.5 * float(np.dot(q[0, i, h], k1[0, 0, 0]))
            _close(o[0, i, h], v[0, :i + 1, 0].mean(axis=0), 1e-12, "equal keys O")
            _close(lse[0, h, i], s + math.log(i + 1), 1e-12, "equal keys LSE")
    # (b) causal row 0 sees only key 0: O = v_0, LSE = S_00
    k = _bf16((B, S, Hkv, d), rng)
    o, lse = oracle.sdpa(q, k, v, True, 0.5, lib=lib)
    for h in range(Hq):
        _close(o[0, 0, h], v[0, 0, 0], 1e-15, "row 0 O")
        _close(lse[0, h, 0], 0.5 * float(np.dot(q[0, 0, h], k[0, 0, 0])), 1e-12, "row 0 LSE")
    # (c) Q = 0: prefix mean, LSE = ln(#admissible)
    o, lse = oracle.sdpa(np.zeros_like(q), k, v, True, 0.5, lib=lib)
    for i in range(S):
        _close(o[0, i, 0], v[0, :i + 1, 0].mean(axis=0), 1e-12, "Q=0 O")
        _close(lse[0, 0, i], math.log(i + 1), 1e-12, "Q=0 LSE")
    # (d) one key 60 above the rest: O = its value row to ~e^-60
    qd = np.zeros((1, 1, 1, 2))
    qd[0, 0, 0] = [1.0, 0.0]
    kd = np.zeros((1, 5, 1, 2))
    kd[0, 3, 0] = [60.0, 0.0]
    vd = _bf16((1, 5, 1, 2), rng)
    o, lse = oracle.sdpa(qd, kd, vd, False, 1.0, lib=lib)
    _close(o[0, 0, 0], vd[0, 3, 0], 1e-20, "dominant key O")
    _close(lse[0, 0, 0], 60.0 + math.log1p(4 * math.exp(-60)), 1e-12, "dominant key LSE")
    # (e) a constant added to every score shifts LSE, leaves O unchanged
    a, bcoef = 2.0, 1.5
    q2 = np.concatenate([q, np.full((B, S, Hq, 1), a)], axis=-1)
    k2 = np.concatenate([k, np.full((B, S, Hkv, 1), bcoef)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, S, Hkv, 1))], axis=-1)
    o1, l1 = oracle.sdpa(q, k, v, True, 0.5, lib=lib)
    o2, l2 = oracle.sdpa(q2, k2, v2, True, 0.5, lib=lib)
    _close(o2[..., :d], o1, 1e-12, "score shift O")
    _close(l2, l1 + 0.5 * a * bcoef, 1e-12, "score shift LSE")


ALL_PINS = [
    pin_golden_two_key, pin_golden_causal_prefix, pin_golden_bottom_right, pin_golden_gqa_map,
    pin_golden_split_merge, pin_golden_split_rule, pin_brute_force_exact, pin_torch_sdpa,
    pin_rows_sum_to_one, pin_permutation_invariance, pin_linearity_in_v,
    pin_split_merge_equals_unsplit, pin_merge_identity, pin_decode_equals_prefill, pin_closed_forms,
    pin_varlen_brute_force, pin_window_brute_force, pin_window_closed_forms,
    pin_varlen_window_brute_force, pin_head_dim_512,
]
