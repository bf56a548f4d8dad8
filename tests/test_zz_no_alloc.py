"""attn_run_paged_no_workspace: attention for callers that cannot allocate.

Plugins that a host framework hands tensors but no allocator, and serving loops
that forbid cudaMalloc on the hot path, cannot provide the workspace that
attn_run_paged asks for.  This entry point runs the same kernels on a scratch
array the library owns.  Here its output, on two calls in a row, is compared
with attn_run_paged's output on a problem whose blocks are split over several
CTAs (so the scratch really carries split-KV partials): the same kernels on the
same plan must give the same bits, which also keeps it inside the parity
tolerance of the other GPU tests.  This file is collected last so that a run
stopping at its first failure has already run every other test; it also passes
on its own in a fresh process.
"""
import numpy as np
import pytest

from asymmetric_kv_paged_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3      # bf16 K/V parity tolerance


def _device_workload():
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    w = W.make_workload(4242, [20000, 9000, 300], [8, 1, 3], hq=16, hkv=2, page_size=128,
                        window=0, sinks=True, name="no_alloc")
    return w, DeviceWorkload(w)


def test_no_workspace_matches_workspace_path_twice():
    from asymmetric_kv_paged_gb300 import binding as B
    w, dw = _device_workload()
    assert dw.plan.workspace_bytes > 0, "the case must use split-KV partials"
    assert dw.plan.workspace_bytes <= B.NO_WORKSPACE_MAX_BYTES
    dw.run()
    torch.cuda.synchronize()
    ref = dw.out.float().clone()
    ref_lse = dw.lse.clone()
    for _ in range(2):
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        B.attn_run_paged_no_workspace(dw.plan, dw.q, dw.k_cache, dw.v_cache, dw.page_table,
                                      dw.seq_lens, dw.qo_indptr, dw.sinks, w.window,
                                      w.softmax_scale, w.k_scale, w.v_scale, out, lse)
        torch.cuda.synchronize()
        got = out.float()
        assert torch.isfinite(got).all()
        err = (got - ref).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
        assert (lse - ref_lse).abs().max().item() <= 2e-3 * max(1.0, ref_lse.abs().max().item())
        # same kernels, same plan, same inputs: bit for bit the workspace path's result
        assert torch.equal(got, ref) and torch.equal(lse, ref_lse)
    assert B.attn_get_device_error(dw.plan) == 0


def test_no_workspace_under_graph_capture():
    """The entry point is meant for callers that capture the step in a CUDA
    graph: after one eager call (which looks the scratch address up), a
    captured call replays with the workspace path's bits and no device error."""
    from asymmetric_kv_paged_gb300 import binding as B
    w, dw = _device_workload()
    dw.run()
    torch.cuda.synchronize()
    ref = dw.out.float().clone()
    ref_lse = dw.lse.clone()
    out = torch.empty_like(dw.out)
    lse = torch.empty_like(dw.lse)

    def call(stream):
        B.attn_run_paged_no_workspace(dw.plan, dw.q, dw.k_cache, dw.v_cache, dw.page_table,
                                      dw.seq_lens, dw.qo_indptr, dw.sinks, w.window,
                                      w.softmax_scale, w.k_scale, w.v_scale, out, lse, stream)

    call(torch.cuda.current_stream())          # eager first: the scratch address lookup
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.float(), ref) and torch.equal(lse, ref_lse)
    assert B.attn_get_device_error(dw.plan) == 0


@pytest.mark.parametrize("case", [
    # name, seq_lens, new tokens, hq, hkv, page size, window, sinks, kv dtype
    ("fp8_p128", [1500, 700], [40, 1], 16, 2, 128, 0, False, "fp8"),
    ("bf16_p16_window_sinks", [2600, 90], [200, 40], 16, 2, 16, 300, True, "bf16"),
    ("fp8_p1_window", [1500], [160], 8, 1, 1, 700, False, "fp8"),
])
def test_prefill_staged_equals_direct_cache_reads(case):
    """A prefill plan run with a workspace stages its keys into 16-bit scratch
    rows that the prefill kernel loads by TMA; without one (this entry point)
    the prefill kernel reads the paged caches itself.  The operand tiles hold
    the same values for every key a row can see, and keys it cannot see are
    masked to exact zeros of P either way, so the two give the same output."""
    from asymmetric_kv_paged_gb300 import binding as B
    from asymmetric_kv_paged_gb300.runner import DeviceWorkload
    name, seq, n, hq, hkv, P, win, sinks, kv = case
    w = W.make_workload(77, seq, n, hq=hq, hkv=hkv, page_size=P, window=win, sinks=sinks,
                        kv_dtype=kv, name=name)
    dw = DeviceWorkload(w)
    info = B.attn_plan_info(dw.plan)
    assert info["rows_per_block"] == 256 and len(B.attn_plan_stage_units(dw.plan)) > 0
    dw.run()
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 0
    ref = dw.out.float().clone()
    ref_lse = dw.lse.clone()
    out = torch.full_like(dw.out, float("nan"))
    lse = torch.full_like(dw.lse, float("nan"))
    B.attn_run_paged_no_workspace(dw.plan, dw.q, dw.k_cache, dw.v_cache, dw.page_table,
                                  dw.seq_lens, dw.qo_indptr, dw.sinks, w.window,
                                  w.softmax_scale, w.k_scale, w.v_scale, out, lse)
    torch.cuda.synchronize()
    assert B.attn_get_device_error(dw.plan) == 0
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out.float(), ref) and torch.equal(lse, ref_lse)


def test_no_workspace_rejects_plans_above_the_limit():
    from asymmetric_kv_paged_gb300 import binding as B
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    for batch, L in ((64, 9000), (96, 9000), (128, 12000)):
        seq = [L] * batch
        prob, keep = B.make_problem(batch=batch, num_q_heads=32, num_kv_heads=2, page_size=128,
                                    num_pages=20000, page_table_stride=(L + 127) // 128,
                                    kv_dtype=0, window=0, has_sinks=False,
                                    qo_indptr=np.arange(0, 8 * batch + 1, 8), seq_lens=seq)
        plan = B.attn_plan(prob, torch.cuda.current_device(), keep)
        if plan.workspace_bytes > B.NO_WORKSPACE_MAX_BYTES:
            break
    else:
        pytest.skip("no test problem needs more scratch than the limit on this device")
    with pytest.raises(B.AttnError) as e:
        B.attn_run_paged_no_workspace(plan, t, t, t, t, t, t, None, 0, 0.1, 1.0, 1.0, t, None)
    assert e.value.status == B.ATTN_ERR_WORKSPACE
