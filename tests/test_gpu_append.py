"""attn_append_kv against the append oracle, through the C ABI: the whole K
and V caches after the append, bit for bit (bf16 rows unchanged; E4M3 codes
of value / scale; every other slot, NaN fillers included, untouched)."""
import numpy as np
import pytest

from asymmetric_kv_paged_gb300 import workloads as W
from oracle import append as A

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    # name, seq_lens, n, hq, hkv, P, kv, query/key head dim
    ("decode_p128", [1000, 129, 3000], [1, 1, 1], 16, 2, 128, "bf16", 192),
    ("verify_p16", [700, 40], [8, 8], 16, 2, 16, "bf16", 192),
    ("prefill_p1", [300], [120], 8, 1, 1, "bf16", 192),
    ("ragged_empty", [90, 50, 20], [5, 0, 3], 8, 2, 3, "bf16", 192),
    ("fp8_verify_p128", [900, 300], [8, 3], 16, 2, 128, "fp8", 192),
    ("fp8_prefill_p3", [260], [200], 16, 4, 3, "fp8", 192),
    # a layer with the symmetric pair 128/128
    ("sym_verify_p16", [700, 40], [8, 8], 16, 2, 16, "bf16", 128),
    ("sym_fp8_prefill_p3", [260], [200], 16, 4, 3, "fp8", 128),
]


def _new_rows(seed, total_q, hkv, dqk=192):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((total_q, hkv, dqk)) * 2).astype(np.float32)
    v = (rng.standard_normal((total_q, hkv, 128)) * 2).astype(np.float32)
    return W.bf16_bits(k), W.bf16_bits(v)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_append_bit_exact(case):
    from asymmetric_kv_paged_gb300 import binding as B
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    name, seq, n, hq, hkv, P, kv, dqk = case
    w = W.make_workload(17, seq, n, hq=hq, hkv=hkv, page_size=P, kv_dtype=kv, name=name, dqk=dqk)
    dw = DeviceWorkload(w)
    kn, vn = _new_rows(23, w.total_q, hkv, dqk)
    ks, vs = (w.k_scale, w.v_scale) if kv == "fp8" else (1.0, 1.0)
    ref_k, ref_v, skipped = A.append_kv(kn, vn, w.k_cache, w.v_cache, w.page_table, w.seq_lens,
                                        w.qo_indptr, kv, ks, vs)
    assert skipped == 0
    d_kn = torch.from_numpy(kn).view(torch.bfloat16).cuda()
    d_vn = torch.from_numpy(vn).view(torch.bfloat16).cuda()
    B.attn_append_kv(dw.plan, d_kn, d_vn, dw.k_cache, dw.v_cache, dw.page_table, dw.seq_lens,
                     dw.qo_indptr, ks, vs)
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 0
    vt = np.uint16 if kv == "bf16" else np.uint8
    got_k = dw.k_cache.view(torch.int16 if kv == "bf16" else torch.uint8).cpu().numpy().view(vt)
    got_v = dw.v_cache.view(torch.int16 if kv == "bf16" else torch.uint8).cpu().numpy().view(vt)
    assert np.array_equal(got_k.reshape(ref_k.shape), ref_k)
    assert np.array_equal(got_v.reshape(ref_v.shape), ref_v)


def test_append_then_attend_matches_oracle():
    """Append the new tokens' K/V, then run attention over the updated cache:
    the output matches the attention oracle on the oracle-appended cache."""
    from asymmetric_kv_paged_gb300 import binding as B
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    from oracle import oracle
    w = W.make_workload(29, [600, 257], [8, 1], hq=16, hkv=2, page_size=16, kv_dtype="fp8",
                        sinks=True, name="append_attend")
    dw = DeviceWorkload(w)
    kn, vn = _new_rows(31, w.total_q, w.hkv)
    ref_k, ref_v, _ = A.append_kv(kn, vn, w.k_cache, w.v_cache, w.page_table, w.seq_lens,
                                  w.qo_indptr, "fp8", w.k_scale, w.v_scale)
    B.attn_append_kv(dw.plan, torch.from_numpy(kn).view(torch.bfloat16).cuda(),
                     torch.from_numpy(vn).view(torch.bfloat16).cuda(), dw.k_cache, dw.v_cache,
                     dw.page_table, dw.seq_lens, dw.qo_indptr, w.k_scale, w.v_scale)
    dw.run()
    torch.cuda.synchronize()
    pb = w.host_arrays()
    pb["k_cache"], pb["v_cache"] = ref_k, ref_v
    ref, _ = oracle.attn_paged(pb)
    err = np.abs(dw.out.float().cpu().numpy() - ref)
    assert err.max() <= 6e-2 and err.mean() <= 6e-3


def test_append_out_of_pool_page_sets_error_word():
    from asymmetric_kv_paged_gb300 import binding as B
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    w = W.make_workload(37, [200], [4], hq=8, hkv=1, page_size=16)
    dw = DeviceWorkload(w)
    before_k = dw.k_cache.clone()
    pt = dw.page_table.clone()
    pt[0, (200 - 1) // 16] = w.num_pages + 5            # the page of the new tokens
    kn, vn = _new_rows(41, w.total_q, 1)
    B.attn_append_kv(dw.plan, torch.from_numpy(kn).view(torch.bfloat16).cuda(),
                     torch.from_numpy(vn).view(torch.bfloat16).cuda(), dw.k_cache, dw.v_cache,
                     pt, dw.seq_lens, dw.qo_indptr, 1.0, 1.0)
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) & 1
    assert torch.equal(dw.k_cache.view(torch.int16), before_k.view(torch.int16))


def test_serving_steps_append_then_replayed_attention():
    """Three decode serving steps on one replayable plan, back to back on one
    stream: each appends the new token's K/V rows (lengths grown by one) and
    runs attention (device planner, attention kernel, merge, launched as
    programmatic dependents).  Every step's output matches the attention oracle
    on the oracle-appended cache."""
    import bench
    from asymmetric_kv_paged_gb300 import binding as B
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    from oracle import oracle
    w = W.make_workload(43, [700, 300, 1000, 65], [1, 1, 1, 1], hq=16, hkv=2, page_size=16,
                        kv_dtype="bf16", sinks=True, name="serving_steps")
    steps = 3
    g = bench.grown_workload(w, steps)
    dw = DeviceWorkload(g, replayable=True)
    L0 = w.seq_lens.astype(np.int32)
    kc, vc = g.k_cache, g.v_cache
    outs, refs = [], []
    for s in range(steps):
        lens = L0 + 1 + s                       # the new token sits at position L0 + s
        kn, vn = _new_rows(50 + s, w.total_q, w.hkv)
        kc, vc, skipped = A.append_kv(kn, vn, kc, vc, g.page_table, lens, w.qo_indptr, "bf16")
        assert skipped == 0
        dw.seq_lens.copy_(torch.from_numpy(lens))
        B.attn_append_kv(dw.plan, torch.from_numpy(kn).view(torch.bfloat16).cuda(),
                         torch.from_numpy(vn).view(torch.bfloat16).cuda(), dw.k_cache, dw.v_cache,
                         dw.page_table, dw.seq_lens, dw.qo_indptr, 1.0, 1.0)
        dw.run()
        outs.append(dw.out.float().clone())
        pb = g.host_arrays()
        pb["k_cache"], pb["v_cache"], pb["seq_lens"] = kc, vc, lens
        refs.append(oracle.attn_paged(pb)[0])
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 0
    for s in range(steps):
        err = np.abs(outs[s].cpu().numpy() - refs[s])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (s, err.max(), err.mean())
