"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Tolerances (max-abs / mean-abs on outputs): 2e-2 / 2e-3 with bf16 K/V, 6e-2 /
6e-3 with fp8 K/V; page-table indexing bit-exact.  The case matrix follows the
pages' attention tests (decode, 8-token verify, full vs SWA with sinks, ragged
page boundaries, CUDA graph replay; sglang PR #41886, "Accuracy Tests") and the
NaN-tail contract (sammysun0711/sglang PR #35).
"""
import zlib

import numpy as np
import pytest

from asymmetric_kv_paged_gb300 import workloads as W
from oracle import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-3), "fp8": (6e-2, 6e-3)}
LSE_TOL = {"bf16": 2e-3, "fp8": 1e-2}


def _runner():
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    return DeviceWorkload


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_rows(w, got_out, got_lse, ref_out, ref_lse, what=""):
    mx, mean = TOL[w.kv_dtype]
    assert np.all(np.isfinite(got_out)), f"{what}: non-finite output"
    err = np.abs(got_out - ref_out)
    assert err.max() <= mx, f"{what}: max abs err {err.max():.4g} > {mx}"
    assert err.mean() <= mean, f"{what}: mean abs err {err.mean():.4g} > {mean}"
    if got_lse is not None:
        lerr = np.abs(got_lse - ref_lse)
        assert lerr.max() <= LSE_TOL[w.kv_dtype] * max(1.0, np.abs(ref_lse).max()), \
            f"{what}: lse err {lerr.max():.4g}"


def run_and_check(w, rows=None):
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    out = bf16_to_f64(dw.out).reshape(-1, W.DV)
    lse = dw.lse.cpu().numpy().astype(np.float64).reshape(-1)
    if rows is None:
        ref_out, ref_lse = oracle.attn_paged(w.host_arrays())
        ref_out = ref_out.reshape(-1, W.DV)
        ref_lse = ref_lse.reshape(-1)
        check_rows(w, out, lse, ref_out, ref_lse, w.name)
    else:
        ref_out, ref_lse = oracle.attn_paged(w.host_arrays(), rows=rows)
        check_rows(w, out[rows], lse[rows], ref_out, ref_lse, w.name)
    assert B_err(dw) == 0
    return dw


def B_err(dw):
    from asymmetric_kv_paged_gb300 import binding as B
    return B.attn_get_device_error(dw.plan)


SMALL = [
    # name, seq_lens, n, hq, hkv, P, window, sinks, kv
    ("decode_g8_p16", [512], [1], 8, 1, 16, 0, False, "bf16"),
    ("decode_ragged_p128", [1000, 129, 3000, 64, 700], [1] * 5, 16, 2, 128, 0, False, "bf16"),
    ("decode_ragged_p3", [50, 333, 1], [1, 1, 1], 8, 2, 3, 0, False, "bf16"),
    ("decode_g1", [300, 77], [1, 1], 4, 4, 16, 0, False, "bf16"),
    ("decode_g16", [900], [1], 16, 1, 128, 0, True, "bf16"),
    ("verify_p1", [1000, 555], [8, 8], 16, 2, 1, 0, False, "bf16"),
    ("verify_p128", [2000, 130], [8, 3], 16, 2, 128, 0, False, "bf16"),
    ("swa_sinks_mixed", [700, 700, 260, 900], [1, 8, 8, 1], 16, 2, 128, 128, True, "bf16"),
    ("swa_small_window", [400, 90], [8, 2], 8, 2, 16, 5, True, "bf16"),
    ("window_one", [300], [8], 8, 1, 16, 1, True, "bf16"),
    ("prefill_g16", [700], [300], 32, 2, 128, 0, False, "bf16"),
    ("prefill_from_empty", [257], [257], 8, 1, 16, 0, False, "bf16"),
    ("prefill_swa", [900], [200], 16, 2, 64, 100, True, "bf16"),
    ("empty_requests", [100, 50, 20], [3, 0, 1], 8, 2, 16, 0, False, "bf16"),
    ("fp8_decode", [2000, 333], [1, 1], 16, 2, 128, 0, False, "fp8"),
    ("fp8_verify_sinks", [1500, 700], [8, 8], 16, 2, 16, 0, True, "fp8"),
    ("fp8_prefill", [900], [256], 64, 4, 128, 0, False, "fp8"),
    ("fp8_swa", [800, 300], [8, 1], 16, 2, 128, 128, True, "fp8"),
    # gathered (page sizes TMA cannot tile) with blocks of more than 64 rows: M = 128
    ("prefill_p1_gather", [600], [100], 8, 1, 1, 0, True, "bf16"),
    ("fp8_prefill_p3_gather", [500, 90], [80, 3], 16, 2, 3, 0, False, "fp8"),
    # every block of 33-64 rows: M = 64 with two threads per row; partly filled
    # blocks, a window with sinks, and one block cut over many CTAs
    ("verify_half_40rows", [900, 700], [5, 5], 16, 2, 16, 0, True, "bf16"),
    ("verify_half_swa_fp8", [3000, 2500], [8, 6], 16, 2, 128, 100, True, "fp8"),
    ("verify_half_split", [20000], [8], 16, 2, 128, 0, False, "bf16"),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_parity_small(case):
    name, seq, n, hq, hkv, P, win, sinks, kv = case
    w = W.make_workload(zlib.crc32(name.encode()) % 1000, seq, n, hq=hq, hkv=hkv, page_size=P, window=win,
                        sinks=sinks, kv_dtype=kv, name=name)
    run_and_check(w)


# Layers with the symmetric pair 128/128 (a model whose SWA layers carry a
# head-dim pair of their own: sglang PR #32818, "Three changes", item 1).
# Blocks of more than 128 rows run on the split-KV kernel at M = 128.
SYM = ["decode_ragged_p128", "decode_ragged_p3", "verify_p1", "verify_p128", "verify_half_split",
       "swa_sinks_mixed",
       "swa_small_window", "prefill_g16", "empty_requests", "fp8_decode", "fp8_verify_sinks",
       "fp8_prefill", "fp8_swa", "fp8_prefill_p3_gather"]


@pytest.mark.parametrize("name", SYM)
def test_parity_symmetric_head_dims(name):
    _, seq, n, hq, hkv, P, win, sinks, kv = next(c for c in SMALL if c[0] == name)
    w = W.make_workload(zlib.crc32(name.encode()) % 1000 + 7, seq, n, hq=hq, hkv=hkv, page_size=P,
                        window=win, sinks=sinks, kv_dtype=kv, name="sym_" + name, dqk=128)
    assert w.q.shape[2] == 128 and w.k_cache.shape[3] == 128
    run_and_check(w)


@pytest.mark.parametrize("P", [1, 16, 128])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_v_path_bit_exact(P, kv):
    """window 1 with n = L: every row sees only its own key, p = 2^0 = 1 exactly,
    so the output is that key's V row converted to bf16 without rounding (the
    sign of a zero aside)."""
    L = 300
    w = W.make_workload(7, [L], [L], hq=4, hkv=2, page_size=P, window=1, kv_dtype=kv)
    w.v_scale = 1.0
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    got = dw.out.view(torch.int16).cpu().numpy().view(np.uint16)      # [L, hq, 128]
    t = np.arange(L)
    slots = w.page_table[0, t // P].astype(np.int64) * P + t % P
    vc = w.v_cache.reshape(-1, w.hkv, W.DV)[slots]                      # [L, hkv, 128]
    if kv == "bf16":
        expect = vc
    else:
        f = torch.from_numpy(vc.copy()).view(torch.float8_e4m3fn).to(torch.bfloat16)
        expect = f.view(torch.int16).numpy().view(np.uint16)
    G = w.hq // w.hkv
    # -0 may come out as +0: the accumulator adds the zero products of masked keys
    plus0 = lambda bits: np.where(bits == 0x8000, 0, bits)  # noqa: E731
    for h in range(w.hq):
        bad = np.argwhere(plus0(got[:, h]) != plus0(expect[:, h // G]))
        assert len(bad) == 0, (f"head {h}: {len(bad)} elements differ, first (token, column, got, "
                               f"expected): {[(int(t_), int(c), hex(got[t_, h, c]), hex(expect[t_, h // G, c])) for t_, c in bad[:6]]}")


@pytest.mark.parametrize("P", [1, 16, 128])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_k_path_index_exact(P, kv):
    """window 1 with n = L and one-hot queries: row t's only score is
    scale * k_t[d], so lse / scale recovers column d of the K row the kernel
    read.  Columns 0-2 of every key row hold base-16 digits of its position
    (integers 1..16, exact in bf16 and E4M3) and column 3 its KV head, so
    each (token, head) must name exactly its own key and head."""
    L, hq, hkv = 300, 8, 2
    G = hq // hkv
    w = W.make_workload(21, [L], [L], hq=hq, hkv=hkv, page_size=P, window=1, kv_dtype=kv)
    w.k_scale = 1.0
    t = np.arange(L)
    code = np.stack([t % 16 + 1, (t // 16) % 16 + 1, t // 256 + 1], axis=1)     # [L, 3]
    slots = w.page_table[0, t // P].astype(np.int64) * P + t % P
    kc = w.k_cache.reshape(-1, hkv, W.DQK).copy()
    for g in range(hkv):
        vals = np.concatenate([code, np.full((L, 1), g + 1)], axis=1).astype(np.float32)
        if kv == "bf16":
            kc[slots, g, :4] = W.bf16_bits(vals)
        else:
            kc[slots, g, :4] = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    w.k_cache = kc.reshape(w.k_cache.shape)
    q = np.zeros((L, hq, W.DQK), np.float32)
    for h in range(hq):
        q[:, h, h % G] = 1.0
    w.q = W.bf16_bits(q)
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    got = dw.lse.cpu().numpy().astype(np.float64) / w.softmax_scale          # [L, hq]
    assert B_err(dw) == 0
    for h in range(hq):
        u, g = h % G, h // G
        expect = code[:, u] if u < 3 else np.full(L, g + 1)
        assert np.all(np.abs(got[:, h] - expect) < 1e-3), f"head {h}"


@pytest.mark.parametrize("q_std", [1e5, 1e-6], ids=["q_1e5", "q_1e-6"])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_fp8_keeps_q_exact(q_std, mode):
    """With FP8 caches Q stays bf16: queries far outside fp16's range (|q| ~ 1e5)
    or deep in its subnormals (|q| ~ 1e-6), with the softmax scale set so the
    scores stay of order one, still match the oracle (the pages keep Q.K in
    16-bit: model card "Things that were measured and did not help")."""
    seq, n, hq, hkv = ([1500, 333], [8, 1], 16, 2) if mode == "decode" else ([700], [200], 32, 2)
    w = W.make_workload(31 if mode == "decode" else 32, seq, n, hq=hq, hkv=hkv, page_size=16,
                        kv_dtype="fp8", q_std=q_std,
                        softmax_scale=1.0 / (q_std * np.sqrt(W.DQK)), name=f"fp8_q{q_std:g}")
    run_and_check(w)


@pytest.mark.parametrize("P", [1, 128])
def test_fp8_every_code_exact(P):
    """Every finite E4M3 code through both load paths.  V: window 1 with n = L, so
    row t returns V row t bit for bit (the code's exact bf16 value, a zero's sign
    aside).  K: one-hot
    queries read one K column each, and lse / scale recovers that element."""
    L, hq, hkv = 300, 8, 2
    G = hq // hkv
    w = W.make_workload(41, [L], [L], hq=hq, hkv=hkv, page_size=P, window=1, kv_dtype="fp8")
    w.k_scale = w.v_scale = 1.0
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    t = np.arange(L)
    slots = w.page_table[0, t // P].astype(np.int64) * P + t % P
    vc = w.v_cache.reshape(-1, hkv, W.DV).copy()
    kc = w.k_cache.reshape(-1, hkv, W.DQK).copy()
    for g in range(hkv):
        vc[slots, g] = finite[(t[:, None] * W.DV + np.arange(W.DV) + 97 * g) % finite.size]
        kc[slots, g, :G] = finite[(t[:, None] * G + np.arange(G) + 31 * g) % finite.size]
    w.v_cache = vc.reshape(w.v_cache.shape)
    w.k_cache = kc.reshape(w.k_cache.shape)
    q = np.zeros((L, hq, W.DQK), np.float32)
    for h in range(hq):
        q[:, h, h % G] = 1.0
    w.q = W.bf16_bits(q)
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    assert B_err(dw) == 0
    got_v = dw.out.view(torch.int16).cpu().numpy().view(np.uint16)
    as_bf16 = lambda codes: torch.from_numpy(np.ascontiguousarray(codes)).view(
        torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_k = dw.lse.cpu().numpy().astype(np.float64) / w.softmax_scale
    # -0 comes out as +0: the accumulator adds the zero products of the tile's
    # other (masked) keys, so only the sign of a zero may differ
    plus0 = lambda bits: np.where(bits == 0x8000, 0, bits)  # noqa: E731
    for h in range(hq):
        g = h // G
        assert np.array_equal(plus0(got_v[:, h]), plus0(as_bf16(vc[slots, g]))), f"V, head {h}"
        expect = torch.from_numpy(kc[slots, g, h % G].copy()).view(torch.float8_e4m3fn).double().numpy()
        assert np.all(np.abs(got_k[:, h] - expect) <= 1e-5 * np.maximum(1.0, np.abs(expect))), \
            f"K, head {h}"


def test_repeat_runs_bit_identical():
    w = W.make_workload(8, [3000, 1200], [8, 1], hq=16, hkv=2, page_size=128, sinks=True)
    dw = _runner()(w)
    dw.run()
    a = dw.out.clone()
    dw.run()
    torch.cuda.synchronize()
    assert torch.equal(a, dw.out)


def test_graph_replay_bit_identical():
    """attn_run_paged allocates and synchronises nothing, so it can be captured."""
    w = W.make_workload(9, [2500, 700, 64], [8, 1, 8], hq=16, hkv=2, page_size=128, window=128,
                        sinks=True)
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    eager = dw.out.clone()
    eager_lse = dw.lse.clone()
    dw.out.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.run(stream=s)
    for _ in range(3):
        dw.out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, dw.out) and torch.equal(eager_lse, dw.lse)


def test_run_argument_errors():
    from asymmetric_kv_paged_gb300 import binding as B
    w = W.make_workload(10, [500, 300], [8, 1], hq=16, hkv=2, page_size=16, window=64,
                        sinks=True)
    dw = _runner()(w)
    base = dict(plan=dw.plan, q=dw.q, k_cache=dw.k_cache, v_cache=dw.v_cache,
                page_table=dw.page_table, seq_lens=dw.seq_lens, qo_indptr=dw.qo_indptr,
                sinks=dw.sinks, window=64, softmax_scale=w.softmax_scale, k_scale=1.0,
                v_scale=1.0, out=dw.out, lse_out=dw.lse, workspace=dw.workspace)
    for upd, status in [(dict(window=65), B.ATTN_ERR_INVALID_ARG),
                        (dict(sinks=None), B.ATTN_ERR_INVALID_ARG),
                        (dict(q=None), B.ATTN_ERR_INVALID_ARG),
                        (dict(softmax_scale=float("nan")), B.ATTN_ERR_INVALID_ARG),
                        (dict(softmax_scale=-w.softmax_scale), B.ATTN_ERR_INVALID_ARG),
                        (dict(softmax_scale=0.0), B.ATTN_ERR_INVALID_ARG)]:
        with pytest.raises(B.AttnError) as e:
            B.attn_run_paged(**dict(base, **upd))
        assert e.value.status == status
    if dw.plan.workspace_bytes > 0:
        small = torch.empty(dw.plan.workspace_bytes - 1, dtype=torch.uint8, device="cuda")
        with pytest.raises(B.AttnError) as e:
            B.attn_run_paged(**dict(base, workspace=small))
        assert e.value.status == B.ATTN_ERR_WORKSPACE
    B.attn_run_paged(**base)
    torch.cuda.synchronize()


@pytest.mark.parametrize("n", [1, 40], ids=["decode", "prefill_staged"])
def test_bad_page_id_sets_error_word(n):
    """A page id outside the pool is never dereferenced: its rows read as zero and
    the plan's device error word records it (the split-KV kernel, and the
    staging pass of a prefill plan)."""
    from asymmetric_kv_paged_gb300 import binding as B
    w = W.make_workload(12, [200], [n], hq=8, hkv=1, page_size=16)
    w.page_table = w.page_table.copy()
    w.page_table[0, 3] = w.num_pages + 5
    dw = _runner()(w)
    if n > 1:
        assert len(B.attn_plan_stage_units(dw.plan)) == 1
    dw.run()
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) & 1
    assert B.attn_get_device_error(dw.plan) == 0     # read-and-clear
    assert torch.isfinite(dw.out.float()).all()


# Per-rank shapes under 8-way tensor parallelism.  The pages test "TP8 per-rank
# shapes for hidden sizes 4096 and 6144" (sglang PR #41886, "Accuracy Tests")
# without giving head counts; 64 to 128 q heads over 8 ranks, with the KV heads
# split or replicated, gives 8 to 16 q heads and 1 or 2 KV heads per rank.
TP8_SHAPES = [(8, 1), (12, 1), (16, 1), (16, 2)]
TP8_MODES = [
    # name, seq_lens, n, P, window, sinks
    ("decode", [1000, 129, 2900, 64, 700], [1] * 5, 128, 0, False),
    ("verify", [1500, 300, 77], [8, 8, 8], 16, 0, False),
    ("swa_sinks", [700, 700, 260, 900], [1, 8, 8, 1], 128, 128, True),
]


@pytest.mark.parametrize("mode", TP8_MODES, ids=[m[0] for m in TP8_MODES])
@pytest.mark.parametrize("shape", TP8_SHAPES, ids=lambda s: f"hq{s[0]}_hkv{s[1]}")
def test_parity_tp8_rank_shapes(shape, mode):
    hq, hkv = shape
    name, seq, n, P, win, sinks = mode
    w = W.make_workload(zlib.crc32(f"tp8_{hq}_{hkv}_{name}".encode()) % 1000, seq, n, hq=hq,
                        hkv=hkv, page_size=P, window=win, sinks=sinks,
                        name=f"tp8_{name}_hq{hq}_hkv{hkv}")
    run_and_check(w)


@pytest.mark.parametrize("P,kv", [(1, "bf16"), (3, "fp8"), (16, "bf16"), (16, "fp8"),
                                  (128, "bf16"), (128, "fp8")])
def test_evicted_pages_are_never_read(P, kv):
    """A sliding-window cache may drop the pages that no query of a request can
    see: entries of -1 there are never looked up, so the output keeps its bits
    and the device error word stays clear."""
    from oracle_pins import drop_unseen_pages
    w = W.make_workload(14 + P, [1500, 700, 3000, 129], [1, 8, 3, 8], hq=16, hkv=2,
                        page_size=P, window=200, sinks=True, kv_dtype=kv)
    full = run_and_check(w)
    w.page_table, below = drop_unseen_pages(w)
    assert below > 0
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    assert torch.equal(full.out, dw.out) and torch.equal(full.lse, dw.lse)
    assert B_err(dw) == 0


# ---- full-size workloads, in the benchmark's launch configuration ----

def block_rows(w, blk):
    """Flat output rows (token * Hq + head) of one plan block
    {b, g, row0, nrows, ...}: block row r is token tok0 + r / G, head g*G + r % G."""
    G = w.hq // w.hkv
    b, g, row0, nrows = (int(x) for x in blk[:4])
    r = row0 + np.arange(nrows)
    tok = int(w.qo_indptr[b]) + r // G
    return tok * w.hq + g * G + r % G


def whole_blocks_to_check(w, plan, count=16):
    """Indices of at least `count` whole row blocks: the first and last block of
    every KV head, then blocks cut over several CTAs (their partials go through
    the merge), the blocks just before and after each such cut first."""
    from asymmetric_kv_paged_gb300 import binding as B
    blocks = B.attn_plan_blocks(plan)
    segs = B.attn_plan_segments(plan)
    pick = []
    for g in range(w.hkv):
        idx = np.nonzero(blocks[:, 1] == g)[0]
        if len(idx):
            pick += [int(idx[0]), int(idx[-1])]
    split = [int(i) for i in np.nonzero(blocks[:, 6] > 1)[0]]
    # blocks whose first segment starts a CTA's share, i.e. sit right after a cut
    starts = {int(segs[i, 1]) for i in range(len(segs))
              if i == 0 or segs[i, 0] != segs[i - 1, 0]}
    for i in split + sorted(starts):
        if len(set(pick)) >= count:
            break
        pick.append(i)
    rng = np.random.default_rng(5)
    while len(set(pick)) < min(count, len(blocks)):
        pick.append(int(rng.integers(len(blocks))))
    return sorted(set(pick)), blocks


@pytest.mark.slow
@pytest.mark.parametrize("name", list(W.CONFIG_NAMES) + list(W.EXTRA_NAMES))
def test_parity_named_config(name):
    """Every output row of the decode, verify and SWA workloads (the 128/128 SWA
    shape included) at full size, and
    at least 16 whole row blocks of the prefill chunk (first and last block of
    every KV head and blocks split over several CTAs), each against the oracle."""
    w = W.named(name)
    if name != "c5_chunked_prefill":
        run_and_check(w)
        return
    dw = _runner()(w)
    dw.run()
    torch.cuda.synchronize()
    assert B_err(dw) == 0
    picked, blocks = whole_blocks_to_check(w, dw.plan)
    assert len(picked) >= 16
    assert any(blocks[i, 6] > 1 for i in picked), "no split block among the checked ones"
    rows = np.unique(np.concatenate([block_rows(w, blocks[i]) for i in picked]))
    out = bf16_to_f64(dw.out).reshape(-1, W.DV)
    lse = dw.lse.cpu().numpy().astype(np.float64).reshape(-1)
    ref_out, ref_lse = oracle.attn_paged(w.host_arrays(), rows=rows)
    check_rows(w, out[rows], lse[rows], ref_out, ref_lse, w.name)


def test_batch_without_query_rows():
    """Every request has zero new tokens: planning and running succeed and launch
    nothing that touches the (empty) outputs."""
    from asymmetric_kv_paged_gb300 import binding as B
    w = W.make_workload(13, [40, 70], [0, 0], hq=8, hkv=2, page_size=16)
    dw = _runner()(w)
    assert dw.plan.workspace_bytes == 0
    dw.run()
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 0


@pytest.mark.parametrize("seed", range(96))
def test_parity_random_shapes(seed):
    """Seeded random problems, every output row against the oracle: ragged
    lengths and query counts (decode, verify, short and long prefill blocks, so
    M = 64 with and without two threads per row, M = 128 and the 256-row
    prefill kernel), page sizes 1 / 3 / 16 / 64 / 128, windows, sinks, GQA
    ratios, BF16 and FP8 caches, and both head-dim pairs."""
    rng = np.random.default_rng(5000 + seed)
    batch = int(rng.integers(1, 6))
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 4, 8, 16]))
    P = int(rng.choice([1, 3, 16, 64, 128]))
    kind = rng.choice(["decode", "verify", "verify_wide", "prefill"])
    if kind == "decode":
        n = np.ones(batch, np.int64)
    elif kind == "verify":
        n = rng.integers(1, 9, batch)
    elif kind == "verify_wide":          # blocks of 40-64 rows: two threads per row
        hq = 8 * hkv
        n = rng.integers(5, 9, batch)
    else:
        n = rng.integers(1, 300, batch)
    n[rng.random(batch) < 0.2] = 0
    seq = n + rng.integers(0, 1500, batch)
    seq = np.maximum(seq, 1)
    win = int(rng.choice([0, 0, 0, 7, 100]))
    kv = str(rng.choice(["bf16", "fp8"]))
    dqk = int(rng.choice([192, 192, 128]))
    w = W.make_workload(seed, seq.tolist(), n.tolist(), hq=hq, hkv=hkv, page_size=P, window=win,
                        sinks=bool(rng.random() < 0.5), kv_dtype=kv, dqk=dqk,
                        name=f"random{seed}_{kind}_{kv}_p{P}_d{dqk}")
    if w.total_q == 0:
        pytest.skip("no query rows drawn")
    run_and_check(w)
