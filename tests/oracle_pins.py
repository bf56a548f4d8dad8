"""Pins for the FP64 oracle: facts fixed by the mathematics, not by the oracle.

Each pin takes an oracle instance (the real one, or a planted mutant) and raises
AssertionError when the instance disagrees with the fact.  The list follows the
cases the pages test (decode, 8-token verify, full vs SWA with sinks, ragged page
boundaries; sglang PR #41886, "Accuracy Tests") and the NaN-tail contract
(sammysun0711/sglang PR #35, "Modifications").
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from asymmetric_kv_paged_gb300.workloads import (BF16_NAN, DQK, DV, E4M3_NAN, bf16_bits,
                                                 bf16_values, make_workload)
from brute import brute_attention

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"


def _small_cases():
    """Tiny problems spanning the feature matrix (ragged n, GQA, windows, sinks,
    page sizes 1/3/16, bf16 and fp8)."""
    return [
        make_workload(11, [37], [1], hq=4, hkv=1, page_size=16),
        make_workload(12, [50, 9, 23], [8, 1, 3], hq=4, hkv=2, page_size=3),
        make_workload(13, [64, 40], [8, 8], hq=8, hkv=2, page_size=16, window=7, sinks=True),
        make_workload(14, [19, 33], [5, 1], hq=2, hkv=2, page_size=1, window=4, sinks=True),
        make_workload(15, [45, 30], [6, 2], hq=4, hkv=1, page_size=16, kv_dtype="fp8",
                      sinks=True),
        make_workload(16, [26], [26], hq=6, hkv=3, page_size=4, window=5, kv_dtype="fp8"),
    ]


def pin_e4m3_table(o):
    """All 256 E4M3 codes equal torch's float8_e4m3fn -> float32 cast (NaN at 0x7F/0xFF)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([o.e4m3_to_double(int(c)) for c in codes])
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref)
    assert set(np.nonzero(nan_ref)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan_ref], ref[~nan_ref].astype(np.float64))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def pin_bf16_widening(o):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 0x7F80, size=200).astype(np.uint16)   # finite, both signs below
    bits[::2] |= 0x8000
    got = np.array([o.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(got, bf16_values(bits).astype(np.float64))


def pin_brute_force(o):
    """Agreement with independent long-double brute force on tiny inputs."""
    for w in _small_cases():
        pb = w.host_arrays()
        out, lse = o.attn_paged(pb)
        bout, blse = brute_attention(pb)
        _close(out, bout, what=f"brute out {w.name}")
        _close(lse, blse, what=f"brute lse {w.name}")


def pin_uniform_logits(o):
    """q = 0 gives equal logits: out is the mean of the visible V rows, and with a
    sink sigma the denominator gains e^sigma: out = sum_j v_j / (|V| + e^sigma)."""
    for sinks in (False, True):
        w = make_workload(21, [70, 33], [1, 1], hq=4, hkv=2, page_size=16, q_std=0.0,
                          sinks=sinks)
        out, lse = o.attn_paged(w.host_arrays())
        G = w.hq // w.hkv
        for b in range(w.batch):
            L = int(w.seq_lens[b])
            rows = []
            for p in range((L + 15) // 16):          # walk the request's pages in order
                page = int(w.page_table[b, p])
                rows.extend(bf16_values(w.v_cache[page, :min(16, L - 16 * p)]).astype(np.float64))
            Vb = np.stack(rows)                      # [L, hkv, 128]
            for h in range(w.hq):
                extra = math.exp(float(w.sinks[h])) if sinks else 0.0
                expect = Vb[:, h // G, :].sum(axis=0) / (L + extra)
                _close(out[w.qo_indptr[b], h], expect, what="uniform out")
                _close(lse[w.qo_indptr[b], h], math.log(L + extra), what="uniform lse")


def pin_single_key(o):
    """One visible key returns its V row: L = 1, and window 1 for every row of a
    prefill (n = L).  With a sink and q = 0: v / (1 + e^sigma)."""
    w = make_workload(31, [1], [1], hq=2, hkv=1, page_size=4)
    out, _ = o.attn_paged(w.host_arrays())
    v0 = bf16_values(w.v_cache[w.page_table[0, 0], 0, 0]).astype(np.float64)
    assert np.array_equal(out[0, 0], v0) and np.array_equal(out[0, 1], v0)

    w = make_workload(32, [29], [29], hq=2, hkv=1, page_size=4, window=1, q_std=0.0,
                      sinks=True)
    out, _ = o.attn_paged(w.host_arrays())
    for t in range(29):
        v = bf16_values(w.v_cache[w.page_table[0, t // 4], t % 4, 0]).astype(np.float64)
        for h in range(2):
            _close(out[t, h], v / (1.0 + math.exp(float(w.sinks[h]))), what="single key + sink")


def pin_sink_minus_inf(o):
    """A sink of -inf is the same as no sink at all."""
    w = make_workload(41, [40, 17], [3, 1], hq=4, hkv=2, page_size=8, window=9)
    pb = w.host_arrays()
    out0, lse0 = o.attn_paged(pb)
    pb["sinks"] = np.full(w.hq, -np.inf, np.float32)
    out1, lse1 = o.attn_paged(pb)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_window_ge_len(o):
    """A window at least as long as the context is full attention."""
    w = make_workload(42, [40, 17], [8, 2], hq=4, hkv=2, page_size=8)
    pb = w.host_arrays()
    out0, lse0 = o.attn_paged(pb)
    pb["window"] = 40
    out1, lse1 = o.attn_paged(pb)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_split_merge(o):
    """Partials over any split of the keys, combined by the LSE merge, equal the
    unsplit row (with the sink folded in at the merge); empty splits are harmless."""
    rng = np.random.default_rng(7)
    for w in (make_workload(51, [97], [8], hq=4, hkv=2, page_size=16, sinks=True),
              make_workload(52, [60, 12], [3, 1], hq=2, hkv=1, page_size=5, window=11,
                            sinks=True)):
        pb = w.host_arrays()
        full, full_lse = o.attn_paged(pb)
        Lmax = int(w.seq_lens.max())
        cuts = np.sort(rng.choice(np.arange(1, Lmax), size=5, replace=False))
        bounds = [0, *cuts.tolist(), Lmax, Lmax + 10]    # the last split sees no key
        parts = [o.attn_partial(pb, lo, hi) for lo, hi in zip(bounds[:-1], bounds[1:])]
        assert any(np.isneginf(p[1]).any() for p in parts), "expected an empty split"
        for r in range(w.total_q * w.hq):
            h = r % w.hq
            o_parts = np.stack([p[0][r] for p in parts])
            l_parts = np.array([p[1][r] for p in parts])
            m, ml = o.merge(o_parts, l_parts, float(w.sinks[h]))
            _close(m, full.reshape(-1, DV)[r], what="merge out")
            _close(ml, full_lse.reshape(-1)[r], what="merge lse")


def pin_page_permutation(o):
    """Moving pages in the pool (and the table with them) changes nothing."""
    w = make_workload(61, [50, 31], [4, 1], hq=4, hkv=2, page_size=8, window=13, sinks=True)
    pb = w.host_arrays()
    out0, lse0 = o.attn_paged(pb)
    perm = np.random.default_rng(3).permutation(w.num_pages)    # new home of page p: perm[p]
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    pb.update(k_cache=k2, v_cache=v2, page_table=perm[w.page_table].astype(np.int32))
    out1, lse1 = o.attn_paged(pb)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_head_duplication(o):
    """GQA with G q heads per KV head equals G = 1 on replicated K/V heads."""
    w = make_workload(71, [33, 20], [8, 1], hq=8, hkv=2, page_size=4, window=6, sinks=True)
    pb = w.host_arrays()
    out0, lse0 = o.attn_paged(pb)
    G = w.hq // w.hkv
    rep = np.arange(w.hq) // G
    pb.update(k_cache=np.ascontiguousarray(w.k_cache[:, :, rep]),
              v_cache=np.ascontiguousarray(w.v_cache[:, :, rep]))
    out1, lse1 = o.attn_paged(pb)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_mode_consistency(o):
    """Verify row t of a request with n new tokens equals a decode call whose
    context ends at that token (L' = L - n + t + 1)."""
    for window, sinks in ((0, False), (5, True)):
        w = make_workload(81, [41], [8], hq=4, hkv=2, page_size=6, window=window, sinks=sinks)
        pb = w.host_arrays()
        out, lse = o.attn_paged(pb)
        for t in range(8):
            d = dict(pb)
            d.update(q=w.q[t:t + 1], qo_indptr=np.array([0, 1], np.int32),
                     seq_lens=np.array([41 - 8 + t + 1], np.int32))
            o1, l1 = o.attn_paged(d)
            assert np.array_equal(o1[0], out[t]) and np.array_equal(l1[0], lse[t])


def pin_scale_invariance(o):
    """(2q, scale/2) gives the same scores, so the same output."""
    w = make_workload(91, [30], [4], hq=2, hkv=1, page_size=8, sinks=True)
    pb = w.host_arrays()
    out0, lse0 = o.attn_paged(pb)
    q2 = w.q.copy()
    nz = (q2 & 0x7FFF) != 0
    q2[nz] += np.uint16(0x0080)                       # exponent + 1: exact doubling
    assert np.array_equal(bf16_values(q2), 2 * bf16_values(w.q))
    pb.update(q=q2, softmax_scale=w.softmax_scale / 2)
    out1, lse1 = o.attn_paged(pb)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_kv_scales(o):
    """fp8 scales: doubling k_scale equals doubling the softmax scale; doubling
    v_scale doubles the output and leaves lse alone."""
    w = make_workload(92, [40], [3], hq=2, hkv=1, page_size=8, kv_dtype="fp8", sinks=True)
    pb = w.host_arrays()
    out0, lse0 = o.attn_paged(pb)
    a = dict(pb, k_scale=2 * w.k_scale)
    b = dict(pb, softmax_scale=2 * w.softmax_scale)
    oa, la = o.attn_paged(a)
    ob, lb = o.attn_paged(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)
    assert not np.allclose(oa, out0)
    c = dict(pb, v_scale=2 * w.v_scale)
    oc, lc = o.attn_paged(c)
    assert np.array_equal(oc, 2 * out0) and np.array_equal(lc, lse0)


def pin_nan_independence(o):
    """Unused slots (NaN-poisoned) never reach the result: refill them with finite
    junk and nothing changes."""
    for kv in ("bf16", "fp8"):
        w = make_workload(93, [45, 20], [8, 1], hq=4, hkv=2, page_size=16, window=10,
                          sinks=True, kv_dtype=kv)
        pb = w.host_arrays()
        out0, lse0 = o.attn_paged(pb)
        nan_code = BF16_NAN if kv == "bf16" else E4M3_NAN
        assert (w.k_cache == nan_code).any()
        k2, v2 = w.k_cache.copy(), w.v_cache.copy()
        junk = 0x4100 if kv == "bf16" else 0x50
        k2[k2 == nan_code] = junk
        v2[v2 == nan_code] = junk
        out1, lse1 = o.attn_paged(dict(pb, k_cache=k2, v_cache=v2))
        assert np.all(np.isfinite(out0))
        assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def drop_unseen_pages(w):
    """The table with every page that holds no key the request's queries can see
    (wholly below the window, or past the last key) replaced by -1, as a cache
    that evicts such pages would leave it; also the number of pages dropped below
    the window."""
    pt = w.page_table.copy()
    P = w.page_size
    below = 0
    for b in range(w.batch):
        lo, L = w.visible_range(b)
        pt[b, :lo // P] = -1
        pt[b, -(-L // P):] = -1
        below += lo // P
    return pt, below


def pin_evicted_pages_unread(o):
    """Pages that no query of a request can see are never looked up: dropping them
    from the table (-1, outside the pool) changes nothing.  With page size 1 the
    page just below the window is dropped too, so one key too many is caught."""
    for seed, P, win, kv in ((95, 4, 5, "bf16"), (96, 1, 3, "fp8"), (97, 8, 16, "bf16")):
        w = make_workload(seed, [60, 33, 17], [1, 8, 3], hq=4, hkv=2, page_size=P,
                          window=win, sinks=True, kv_dtype=kv)
        pb = w.host_arrays()
        out0, lse0 = o.attn_paged(pb)
        pt, below = drop_unseen_pages(w)
        assert below > 0
        out1, lse1 = o.attn_paged(dict(pb, page_table=pt))
        assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_hand_golden(o):
    """The hand-derived two-key case in tests/golden/hand_two_keys.json."""
    with open(os.path.join(GOLDEN, "hand_two_keys.json")) as f:
        g = json.load(f)
    e = math.e
    ev = lambda s: eval(s, {"__builtins__": {}}, {"e": e, "log": math.log})  # noqa: E731
    q = np.zeros((1, 1, DQK), np.uint16)
    q[0, 0, 0] = int(bf16_bits(np.array([1.0], np.float32))[0])
    k = np.full((3, 1, 1, DQK), BF16_NAN, np.uint16)
    v = np.full((3, 1, 1, DV), BF16_NAN, np.uint16)
    k[0, 0, 0, :] = 0
    k[1, 0, 0, :] = 0
    k[1, 0, 0, 0] = int(bf16_bits(np.array([2.0], np.float32))[0])
    v[0, 0, 0, :] = 0
    v[1, 0, 0, :] = 0
    v[0, 0, 0, 0] = int(bf16_bits(np.array([1.0], np.float32))[0])
    v[1, 0, 0, 1] = int(bf16_bits(np.array([1.0], np.float32))[0])
    base = dict(q=q, k_cache=k, v_cache=v, qo_indptr=np.array([0, 1], np.int32),
                seq_lens=np.array([2], np.int32), page_table=np.array([[0, 1]], np.int32),
                sinks=None, window=0, softmax_scale=0.5)
    for key, upd in (("no_sink", {}), ("sink_1", {"sinks": np.array([1.0], np.float32)}),
                     ("window_1", {"window": 1})):
        out, lse = o.attn_paged(dict(base, **upd))
        exp_out = np.zeros(DV)
        exp_out[0] = ev(g[key]["out0"])
        exp_out[1] = ev(g[key]["out1"])
        _close(out[0, 0], exp_out, rtol=1e-15, atol=1e-15, what=key)
        _close(lse[0, 0], ev(g[key]["lse"]), rtol=1e-15, atol=1e-15, what=key)


ALL_PINS = [pin_e4m3_table, pin_bf16_widening, pin_brute_force, pin_uniform_logits,
            pin_single_key, pin_sink_minus_inf, pin_window_ge_len, pin_split_merge,
            pin_page_permutation, pin_head_duplication, pin_mode_consistency,
            pin_scale_invariance, pin_kv_scales, pin_nan_independence, pin_evicted_pages_unread,
            pin_hand_golden]
