"""C-ABI library checks that need no GPU: it loads, exports what the header
declares, validates problems, and its schedule covers every visible key once."""
import os
import re

import numpy as np
import pytest

from asymmetric_kv_paged_gb300 import binding as B
from asymmetric_kv_paged_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = B.load()
    declared = header_functions()
    assert "attn_plan" in declared and "attn_run_paged" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(B.EXPORTED)


def test_stamps_are_only_in_the_profiling_build():
    # the default build records no timestamps: the entry point exists and says so
    with pytest.raises(B.AttnError) as e:
        B.attn_debug_stamps(clear=False)
    assert e.value.status == B.ATTN_ERR_UNSUPPORTED


def test_status_strings():
    assert B.attn_status_string(0) == "ok"
    assert "workspace" in B.attn_status_string(B.ATTN_ERR_WORKSPACE)


def _problem(**kw):
    base = dict(batch=2, num_q_heads=16, num_kv_heads=2, page_size=16, num_pages=100,
                page_table_stride=8, kv_dtype=B.ATTN_KV_BF16, window=0, has_sinks=False,
                qo_indptr=[0, 1, 9], seq_lens=[100, 120])
    base.update(kw)
    return B.make_problem(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim_qk=64), B.ATTN_ERR_UNSUPPORTED),
    (dict(head_dim_qk=256), B.ATTN_ERR_UNSUPPORTED),
    (dict(head_dim_v=192), B.ATTN_ERR_UNSUPPORTED),
    (dict(head_dim_qk=128, head_dim_v=64), B.ATTN_ERR_UNSUPPORTED),
    (dict(num_q_heads=15), B.ATTN_ERR_UNSUPPORTED),
    (dict(seq_lens=[100, 5]), B.ATTN_ERR_INVALID_ARG),          # L < n
    (dict(qo_indptr=[0, 3, 2]), B.ATTN_ERR_INVALID_ARG),        # non-monotone
    (dict(qo_indptr=[1, 2, 9]), B.ATTN_ERR_INVALID_ARG),        # must start at 0
    (dict(seq_lens=[100, 129]), B.ATTN_ERR_INVALID_ARG),        # needs 9 pages > stride 8
    (dict(page_size=0), B.ATTN_ERR_INVALID_ARG),
    (dict(num_kv_heads=0), B.ATTN_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_problems(kw, status):
    prob, keep = _problem(**kw)
    with pytest.raises(B.AttnError) as e:
        B.attn_plan_host(prob, 152, keep)
    assert e.value.status == status


def _problem_of(w, seq_lens=None):
    return B.make_problem(
        batch=w.batch, num_q_heads=w.hq, num_kv_heads=w.hkv, page_size=w.page_size,
        num_pages=w.num_pages, page_table_stride=w.page_table.shape[1],
        kv_dtype=B.ATTN_KV_BF16, window=w.window, has_sinks=False, qo_indptr=w.qo_indptr,
        seq_lens=w.seq_lens if seq_lens is None else seq_lens)


def test_plan_rejects_bad_problems_beyond_shapes():
    # element type outside the enum
    prob, keep = _problem(kv_dtype=7)
    with pytest.raises(B.AttnError) as e:
        B.attn_plan_host(prob, 152, keep)
    assert e.value.status == B.ATTN_ERR_UNSUPPORTED
    # an empty pool, a negative batch, and host arrays missing for a batch
    for kw in (dict(num_pages=0), dict(batch=-1)):
        prob, keep = _problem(**kw)
        with pytest.raises(B.AttnError) as e:
            B.attn_plan_host(prob, 152, keep)
        assert e.value.status == B.ATTN_ERR_INVALID_ARG
    for field in ("qo_indptr_host", "seq_lens_host"):
        prob, keep = _problem()
        setattr(prob, field, None)
        with pytest.raises(B.AttnError) as e:
            B.attn_plan_host(prob, 152, keep)
        assert e.value.status == B.ATTN_ERR_INVALID_ARG
    # flat query rows x heads must stay within the kernels' int32 arithmetic
    n = 2_000_000
    prob, keep = _problem(batch=1, num_q_heads=64, num_kv_heads=4, page_table_stride=n // 16 + 1,
                          num_pages=n // 16 + 2, qo_indptr=[0, n], seq_lens=[n])
    with pytest.raises(B.AttnError) as e:
        B.attn_plan_host(prob, 152, keep)
    assert e.value.status == B.ATTN_ERR_UNSUPPORTED
    # no SM count
    prob, keep = _problem()
    with pytest.raises(B.AttnError) as e:
        B.attn_plan_host(prob, 0, keep)
    assert e.value.status == B.ATTN_ERR_INVALID_ARG


def test_replayable_plan_validates_and_sizes_for_the_bounds():
    prob, keep = _problem(seq_lens=[100, 5])          # a bound below n
    with pytest.raises(B.AttnError) as e:
        B.attn_plan_replayable_host(prob, 152, keep)
    assert e.value.status == B.ATTN_ERR_INVALID_ARG
    # a batch with no query row plans to nothing and needs no workspace
    prob, keep = _problem(qo_indptr=[0, 0, 0])
    plan = B.attn_plan_replayable_host(prob, 152, keep)
    info = B.attn_plan_info(plan)
    assert info["blocks"] == info["segments"] == info["ctas"] == 0
    assert info["workspace_bytes"] == 0
    # the workspace covers the worst split of any lengths within the bounds:
    # (largest block rows) x (blocks + CTAs) partial rows of 128 floats + one lse
    prob, keep = _problem()
    plan = B.attn_plan_replayable_host(prob, 152, keep)
    info = B.attn_plan_info(plan)
    rows = int(B.attn_plan_blocks(plan)[:, 3].max()) * (info["blocks"] + info["ctas"])
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert info["workspace_bytes"] == align(rows * 128 * 4) + align(rows * 4)
    # a static plan never needs replanning
    sprob, skeep = _problem()
    with pytest.raises(B.AttnError) as e:
        B.attn_plan_replan_host(B.attn_plan_host(sprob, 152, skeep), [100, 120])
    assert e.value.status == B.ATTN_ERR_INVALID_ARG


def _coverage_check(w, num_sms):
    prob, keep = _problem_of(w)
    return _check_plan(B.attn_plan_host(prob, num_sms, keep), w, num_sms)


def _check_plan(plan, w, num_sms, replayable=False):
    """The plan's work list covers every (request, KV head, row) once, with the
    key range its rows see, each block's tiles once in split order, and CTA
    loads balanced; a static prefill plan stages each (request, KV head)'s keys
    once; returns the plan's info."""
    info = B.attn_plan_info(plan)
    blocks = B.attn_plan_blocks(plan)
    segs = B.attn_plan_segments(plan)
    tile = info["key_tile"]
    R = info["rows_per_block"]
    G = w.hq // w.hkv
    assert info["ctas"] <= num_sms
    # every (b, g, row) lives in exactly one block; block key range = union of its rows' keys
    seen = set()
    for (b, g, row0, nrows, klo, khi, nsplit, prb) in blocks:
        n = int(w.qo_indptr[b + 1] - w.qo_indptr[b])
        L = int(w.seq_lens[b])
        assert 0 < nrows <= R
        for r in range(row0, row0 + nrows):
            assert (b, g, r) not in seen
            seen.add((b, g, r))
        i_first = L - n + row0 // G
        i_last = L - n + (row0 + nrows - 1) // G
        assert khi == i_last + 1
        assert klo == (max(0, i_first - w.window + 1) if w.window > 0 else 0)
    expect = {(b, g, r) for b in range(w.batch) for g in range(w.hkv)
              for r in range(int(w.qo_indptr[b + 1] - w.qo_indptr[b]) * G)}
    assert seen == expect
    # segments of each block tile its key range exactly once, in split order
    by_block = {}
    for cta, blk, t0, t1, split in segs:
        by_block.setdefault(blk, []).append((split, t0, t1, cta))
    for bi, (b, g, row0, nrows, klo, khi, nsplit, prb) in enumerate(blocks):
        parts = sorted(by_block[bi])
        assert [p[0] for p in parts] == list(range(nsplit))
        assert parts[0][1] == klo // tile and parts[-1][2] == (khi - 1) // tile + 1
        for (s0, a0, b0, _), (s1, a1, b1, _) in zip(parts, parts[1:]):
            assert b0 == a1
        assert (prb >= 0) == (nsplit > 1)
    # CTA loads are balanced (stream-K dealing): max <= mean + slack (the
    # replayable deal balances tiles plus switch charges: checked by its test)
    loads = np.zeros(info["ctas"], np.int64)
    for cta, blk, t0, t1, split in segs:
        loads[cta] += t1 - t0
    if not replayable:
        assert loads.max() <= int(np.ceil(loads.sum() / info["ctas"])) * 1.25 + 2
    # each CTA's head record (what the kernels read first): its segment range,
    # its tile count, its first segment and that segment's block
    heads = B.attn_plan_cta_heads(plan)
    assert heads.shape == (info["ctas"], 20)
    for c in range(info["ctas"]):
        mine = np.nonzero(segs[:, 0] == c)[0]
        h = heads[c]
        if len(mine) == 0:
            assert h[0] == h[1] and h[2] == 0
            continue
        assert h[0] == mine[0] and h[1] == mine[-1] + 1
        assert h[2] == int((segs[mine, 3] - segs[mine, 2]).sum())
        assert list(h[4:8]) == list(segs[mine[0], 1:5])
        bi = segs[mine[0], 1]
        assert list(h[8:12]) == list(blocks[bi, :4]) and list(h[15:19]) == list(blocks[bi, 4:8])
    # Staging units (static prefill plans only): one per (request, KV head)
    # with blocks, over whole 128-key tiles from the tile of the smallest key_lo
    # to that of the largest key_hi, rows and tiles laid out back to back in
    # unit order; a block's head record places its keys at row srow + j.
    units = B.attn_plan_stage_units(plan)
    if R != 256 or replayable:
        assert len(units) == 0
        assert all(heads[c][19] == 0 for c in range(info["ctas"]))
        return info
    expect_units = {}
    for (b, g, row0, nrows, klo, khi, nsplit, prb) in blocks:
        lo, hi = expect_units.get((b, g), (klo, khi))
        expect_units[(b, g)] = (min(lo, klo), max(hi, khi))
    assert len(units) == len(expect_units)
    row = tiles = 0
    srow = {}
    for (b, g, j0, klo, khi, ntiles, row_base, tile_off) in units:
        assert expect_units[(b, g)] == (klo, khi)
        assert j0 == klo // 128 * 128 and j0 + 128 * ntiles >= khi > j0 + 128 * (ntiles - 1)
        assert row_base == row and tile_off == tiles
        row += 128 * ntiles
        tiles += ntiles
        srow[(b, g)] = row_base - j0
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    part = int(blocks[:, 6][blocks[:, 6] > 1].dot(blocks[:, 3][blocks[:, 6] > 1]))
    partial = align(part * 128 * 4) + align(part * 4) if part else 0
    assert info["workspace_bytes"] == partial + align(row * w.dqk * 2) + align(row * 128 * 2)
    for c in range(info["ctas"]):
        if heads[c][1] > heads[c][0]:
            b, g = heads[c][8], heads[c][9]
            assert heads[c][19] == srow[(b, g)]
    return info


@pytest.mark.parametrize("case", [
    dict(seq=[37], n=[1], hq=8, hkv=1, P=16, W=0),
    dict(seq=[500, 9, 2300], n=[8, 1, 3], hq=16, hkv=2, P=128, W=0),
    dict(seq=[640, 400], n=[8, 8], hq=8, hkv=2, P=16, W=70),
    dict(seq=[190, 333], n=[5, 1], hq=2, hkv=2, P=1, W=4),
    dict(seq=[3000], n=[300], hq=64, hkv=4, P=128, W=0),
    dict(seq=[1000, 1000, 1000], n=[1, 8, 1], hq=16, hkv=2, P=128, W=128),
    dict(seq=[5000, 700, 260], n=[40, 1, 20], hq=16, hkv=2, P=16, W=300),   # windowed prefill
])
@pytest.mark.parametrize("num_sms", [1, 7, 152])
def test_schedule_covers_every_key_once(case, num_sms):
    w = W.make_workload(0, case["seq"], case["n"], hq=case["hq"], hkv=case["hkv"],
                        page_size=case["P"], window=case["W"])
    _coverage_check(w, num_sms)


def test_named_configs_schedule_shape():
    # shapes of the named workloads, without drawing their values
    for name, seq, n, hq, hkv, P, Wn, rows in [
        ("decode", [1024 + 37 * i for i in range(32)], [1] * 32, 16, 2, 128, 0, 64),
        ("verify", [46008] * 4, [8] * 4, 16, 2, 128, 0, 64),
        ("swa", [8192] * 64, [1, 8] * 32, 16, 2, 128, 128, 64),
        ("prefill", [30096], [4096], 64, 4, 128, 0, 256),
    ]:
        prob, keep = B.make_problem(batch=len(seq), num_q_heads=hq, num_kv_heads=hkv,
                                    page_size=P, num_pages=9375,
                                    page_table_stride=max((s + P - 1) // P for s in seq),
                                    kv_dtype=0, window=Wn, has_sinks=False,
                                    qo_indptr=np.concatenate([[0], np.cumsum(n)]), seq_lens=seq)
        plan = B.attn_plan_host(prob, 152, keep)
        info = B.attn_plan_info(plan)
        assert info["rows_per_block"] == rows, name
        assert 0 < info["ctas"] <= 152


def test_symmetric_head_dim_pair_is_planned_without_the_prefill_kernel():
    # 128/128 (a layer with a symmetric pair of its own) is accepted; its large
    # blocks stay at 128 rows, since the 256-row prefill kernel is built for
    # 192/128 only
    for seq, n, hq, hkv, rows in [([46008] * 4, [8] * 4, 16, 2, 64),
                                  ([30096], [4096], 64, 4, 128)]:
        for dqk, want in [(128, rows), (192, 256 if n[0] > 8 else rows)]:
            prob, keep = B.make_problem(batch=len(seq), num_q_heads=hq, num_kv_heads=hkv,
                                        page_size=128, num_pages=9375,
                                        page_table_stride=max((s + 127) // 128 for s in seq),
                                        kv_dtype=0, window=0, has_sinks=False,
                                        qo_indptr=np.concatenate([[0], np.cumsum(n)]),
                                        seq_lens=seq, head_dim_qk=dqk, head_dim_v=128)
            info = B.attn_plan_info(B.attn_plan_host(prob, 152, keep))
            assert info["rows_per_block"] == want, (dqk, seq)


def test_small_blocks_are_not_split_when_ctas_suffice():
    # 64 requests of a windowed mix (2-3 key tiles per block, 128 blocks) on 152
    # SMs: every block fits a CTA of its own, so none is cut and no merge runs
    seq = [8192] * 64
    n = [1, 8] * 32
    prob, keep = B.make_problem(batch=64, num_q_heads=16, num_kv_heads=2, page_size=128,
                                num_pages=9375, page_table_stride=64, kv_dtype=0, window=128,
                                has_sinks=False, qo_indptr=np.concatenate([[0], np.cumsum(n)]),
                                seq_lens=seq)
    plan = B.attn_plan_host(prob, 152, keep)
    info = B.attn_plan_info(plan)
    assert info["multi_split_blocks"] == 0 and info["workspace_bytes"] == 0
    assert info["segments"] == info["blocks"] == 128
    # with fewer SMs than blocks the same blocks are dealt (and cut) as usual
    plan = B.attn_plan_host(prob, 100, keep)
    info = B.attn_plan_info(plan)
    assert info["ctas"] <= 100 and info["segments"] >= info["blocks"]


@pytest.mark.parametrize("seed", range(12))
def test_schedule_invariants_on_random_problems(seed):
    # seeded random shapes: ragged lengths, empty requests, every page size
    # class (gather, divisor, multiple), windows, GQA ratios and SM counts
    rng = np.random.default_rng(1000 + seed)
    batch = int(rng.integers(1, 24))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 8, 16]))
    P = int(rng.choice([1, 3, 16, 64, 128]))
    n = rng.integers(0, 40, batch)
    n[rng.random(batch) < 0.5] = 1
    seq = n + rng.integers(0, 3000, batch)
    seq = np.maximum(seq, 1)
    win = int(rng.choice([0, 0, 1, 17, 128]))
    num_sms = int(rng.choice([1, 7, 64, 152]))
    w = W.make_workload(seed, seq.tolist(), n.tolist(), hq=hq, hkv=hkv, page_size=P, window=win)
    _coverage_check(w, num_sms)


def test_headers_compile_as_plain_c(tmp_path):
    # the boundary is a C ABI: both headers must stand alone in C99, with no
    # CUDA or C++ header behind them
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi.c"
    src.write_text('#include "attn_paged.h"\n#include "attn_paged_debug.h"\n'
                   "int main(void) { attn_plan_t p = 0; attn_problem_t q; (void)p; (void)q;\n"
                   "  return ATTN_OK; }\n")
    inc = os.path.join(ROOT, "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{inc}",
                    "-fsyntax-only", str(src)], check=True)


# ---- replayable plans: the work list is rebuilt from each run's lengths ----

def _random_bounds(seed):
    rng = np.random.default_rng(2000 + seed)
    batch = int(rng.integers(1, 20))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 8, 16]))
    P = int(rng.choice([1, 3, 16, 64, 128]))
    n = rng.integers(0, 40, batch)
    n[rng.random(batch) < 0.5] = 1
    bound = n + rng.integers(0, 3000, batch)
    bound = np.maximum(bound, 1)
    win = int(rng.choice([0, 0, 1, 17, 128]))
    num_sms = int(rng.choice([1, 7, 64, 152]))
    w = W.make_workload(seed, bound.tolist(), n.tolist(), hq=hq, hkv=hkv, page_size=P, window=win)
    return w, n, bound, num_sms, rng


def _with_lens(w, lens):
    import copy
    w2 = copy.copy(w)
    w2.seq_lens = np.asarray(lens, np.int32)
    return w2


@pytest.mark.parametrize("seed", range(12))
def test_replayable_replan_keeps_schedule_invariants(seed):
    """For lengths anywhere within the bounds, the host mirror of the device
    planner gives a valid work list: every row once, the key range of the run's
    lengths, equal CTA shares, and the capacities the plan was sized for."""
    w, n, bound, num_sms, rng = _random_bounds(seed)
    prob, keep = _problem_of(w)
    plan = B.attn_plan_replayable_host(prob, num_sms, keep)
    info0 = B.attn_plan_info(plan)
    assert info0["ctas"] <= num_sms
    max_rows = max(int(nrows) for nrows in B.attn_plan_blocks(plan)[:, 3]) if info0["blocks"] else 0
    cap_rows = max_rows * (info0["blocks"] + info0["ctas"])
    for trial in range(6):
        lens = n + (rng.random(w.batch) * (bound - n + 1)).astype(np.int64)
        lens = np.minimum(lens, bound)
        if trial == 0:
            lens = bound.copy()
        elif trial == 1:
            lens = n.copy()                              # only the new tokens
        assert B.attn_plan_replan_host(plan, lens) == 0
        info = _check_plan(plan, _with_lens(w, lens), num_sms, replayable=True)
        assert info["ctas"] == info0["ctas"] and info["blocks"] == info0["blocks"]
        assert info["segments"] <= info["blocks"] + info["ctas"]
        segs = B.attn_plan_segments(plan)
        loads = np.bincount(segs[:, 0], weights=segs[:, 3] - segs[:, 2],
                            minlength=info["ctas"]) if len(segs) else np.zeros(1)
        busy = loads[loads > 0]
        if len(busy):
            # equal shares of tile positions, rounded down; on shares of 32
            # tiles or more each block adds 4 positions without a tile, paid by
            # the CTA whose share reaches into it
            nseg = np.bincount(segs[:, 0], minlength=info["ctas"])
            charge = 4 if loads.sum() >= 32 * len(busy) else 0
            cost = loads + charge * nseg
            assert cost[:len(busy)].max() - cost[:len(busy)].min() <= 1 + charge * 2
            assert busy.max() - busy.min() <= 1 + charge * nseg.max()
            assert np.all(loads[:len(busy)] > 0)         # the working CTAs come first
        blocks = B.attn_plan_blocks(plan)
        multi = blocks[blocks[:, 6] > 1]
        used = int((multi[:, 6] * multi[:, 3]).sum())
        assert used <= cap_rows
        if len(multi):
            # partial rows packed in block order
            ends = multi[:, 7] + multi[:, 6] * multi[:, 3]
            assert multi[0, 7] == 0 and np.array_equal(multi[1:, 7], ends[:-1])


def test_replayable_replan_clamps_lengths_and_matches_static_ranges():
    w = W.make_workload(3, [500, 90, 1300], [8, 1, 3], hq=16, hkv=2, page_size=16, window=100)
    prob, keep = _problem_of(w)
    plan = B.attn_plan_replayable_host(prob, 152, keep)
    first = B.attn_plan_blocks(plan).copy()
    # lengths outside [n_b, bound_b] are clamped, and flagged like the device does
    assert B.attn_plan_replan_host(plan, [4, 91, 2000]) == 4
    clamped = B.attn_plan_blocks(plan).copy()
    assert B.attn_plan_replan_host(plan, [8, 90, 1300]) == 0
    assert np.array_equal(B.attn_plan_blocks(plan), clamped)
    # the bounds themselves give back the plan as built
    assert B.attn_plan_replan_host(plan, [500, 90, 1300]) == 0
    assert np.array_equal(B.attn_plan_blocks(plan), first)
    # key ranges are those of a static plan for the same lengths
    for lens in ([200, 90, 1000], [8, 1, 3], [499, 77, 1299]):
        assert B.attn_plan_replan_host(plan, lens) == 0
        sprob, skeep = _problem_of(w, lens)
        static = B.attn_plan_blocks(B.attn_plan_host(sprob, 152, skeep))
        assert np.array_equal(B.attn_plan_blocks(plan)[:, :6], static[:, :6])
