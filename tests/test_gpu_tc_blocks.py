"""tcgen05 building blocks in isolation: 128-byte swizzled K-major / MN-major
shared-memory operands, instruction descriptors, tensor-memory accumulators.
Compared with a plain fp32 PyTorch product of the same operands."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run(mode, variant, ab_type, n, a, b):
    from asymmetric_kv_paged_gb300 import binding as B
    rows, cols = 128, (n if mode == 0 else 128)
    d = torch.full((rows, cols), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attn_debug_tc_gemm(mode, variant, ab_type, n, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "tensor-core completion wait timed out"
    return d


@pytest.mark.parametrize("ab_type", [0, 1], ids=["fp16", "bf16"])
@pytest.mark.parametrize("n", [64, 128])
def test_qk_shape_kmajor(ab_type, n):
    g = torch.Generator(device="cuda").manual_seed(1)
    dt = torch.float16 if ab_type == 0 else torch.bfloat16
    a = torch.randn(128, 192, device="cuda", generator=g).to(dt)
    b = torch.randn(n, 192, device="cuda", generator=g).to(dt)
    d = _run(0, 0, ab_type, n, a, b)
    ref = a.float() @ b.float().T
    err = (d - ref).abs().max().item()
    assert err < 1e-3 * ref.abs().max().item(), err


@pytest.mark.parametrize("ab_type", [0, 1], ids=["fp16", "bf16"])
def test_pv_shape_mnmajor(ab_type):
    g = torch.Generator(device="cuda").manual_seed(2)
    dt = torch.float16 if ab_type == 0 else torch.bfloat16
    a = torch.rand(128, 64, device="cuda", generator=g).to(dt)
    b = torch.randn(64, 128, device="cuda", generator=g).to(dt)
    ref = a.float() @ b.float()
    errs = []
    for variant in (0, 1):
        d = _run(1, variant, ab_type, 64, a, b)
        errs.append((d - ref).abs().max().item())
    tol = 1e-3 * ref.abs().max().item()
    assert errs[0] < tol, f"leading-offset variant err {errs[0]:.3g}, stride variant {errs[1]:.3g}"


def test_m64_accumulator_lanes():
    """An M=64 product lands in TMEM lanes 0-15 of each 32-lane subpartition:
    row r in lane 32*(r//16) + r%16 (the layout the attention kernel reads)."""
    import numpy as np
    g = torch.Generator(device="cuda").manual_seed(3)
    a = torch.randn(64, 192, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(64, 192, device="cuda", generator=g).to(torch.bfloat16)
    from asymmetric_kv_paged_gb300 import binding as B
    d = torch.zeros((128, 64), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attn_debug_tc_gemm(2, 0, 1, 64, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = (a.float() @ b.float().T).cpu().numpy()
    got = d.cpu().numpy()
    tol = 1e-3 * np.abs(ref).max()
    found = {}
    for lane in range(128):
        for r in range(64):
            if np.all(np.isfinite(got[lane])) and np.abs(got[lane] - ref[r]).max() < tol:
                found[r] = lane
    expect = {r: 32 * (r // 16) + r % 16 for r in range(64)}
    assert found == expect, f"row -> lane map: {sorted(found.items())}"


@pytest.mark.parametrize("mode,rows", [(3, 128), (4, 64)])
def test_pv_with_p_in_tmem(mode, rows):
    """P.V with the A operand (P) read from tensor memory: each row written by
    the thread that owns its accumulator lane, two bf16 values per column."""
    import numpy as np
    g = torch.Generator(device="cuda").manual_seed(5 + mode)
    a = torch.rand(rows, 64, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(64, 128, device="cuda", generator=g).to(torch.bfloat16)
    from asymmetric_kv_paged_gb300 import binding as B
    d = torch.zeros((128, 128), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attn_debug_tc_gemm(mode, 0, 1, 64, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = (a.float() @ b.float()).cpu().numpy()
    got = d.cpu().numpy()
    lanes = [r if rows == 128 else 32 * (r // 16) + r % 16 for r in range(rows)]
    err = np.abs(got[lanes] - ref).max()
    assert err < 1e-3 * np.abs(ref).max(), f"max err {err:.3g}"


def test_sixteen_lane_tmem_shapes():
    """The 16x256b / 16x128b TMEM access shapes on an M=64 accumulator: thread
    t of warp w sees rows 16w + t/4 and 16w + t/4 + 8, column pairs
    8i + 2(t%4) + {0,1} (loads) and columns 4i + t%4 (stores)."""
    import numpy as np
    g = torch.Generator(device="cuda").manual_seed(11)
    a = torch.randn(64, 192, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(64, 192, device="cuda", generator=g).to(torch.bfloat16)
    from asymmetric_kv_paged_gb300 import binding as B
    d = torch.zeros(6144, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attn_debug_tc_gemm(5, 0, 1, 64, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = (a.float() @ b.float().T).cpu().numpy()
    got = d.cpu().numpy()
    ld = got[:4096].reshape(4, 32, 32)
    tol = 1e-3 * np.abs(ref).max()
    for w in range(4):
        for t in range(32):
            for i in range(8):
                for h in range(2):
                    row = 16 * w + t // 4 + 8 * h
                    for e in range(2):
                        col = 8 * i + 2 * (t % 4) + e
                        assert abs(ld[w, t, 4 * i + 2 * h + e] - ref[row, col]) < tol, (w, t, i, h, e)
    stv = got[4096:].reshape(4, 32, 16)
    for w in range(4):
        for lane in range(16):
            for col in range(16):
                i, tq = divmod(col, 4)
                h, tr = divmod(lane, 8)
                t = 4 * tr + tq
                assert stv[w, lane, col] == float(w * 100000 + t * 100 + 2 * i + h), (w, lane, col)


def test_two_half_sixteen_lane_tmem_shapes():
    """The 16x32bx2 TMEM access shapes on an M=64 accumulator: threads t < 16
    of warp w see row 16w + t at columns [0, 32), threads t >= 16 the same row
    16w + t - 16 at the split offset (columns [32, 64)); the store puts thread
    t's registers in row 16w + t % 16 at columns 64 + 16 (t // 16) + j."""
    import numpy as np
    g = torch.Generator(device="cuda").manual_seed(12)
    a = torch.randn(64, 192, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(64, 192, device="cuda", generator=g).to(torch.bfloat16)
    from asymmetric_kv_paged_gb300 import binding as B
    d = torch.zeros(8192, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attn_debug_tc_gemm(6, 0, 1, 64, a, b, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = (a.float() @ b.float().T).cpu().numpy()
    got = d.cpu().numpy()
    ld = got[:4096].reshape(4, 32, 32)
    tol = 1e-3 * np.abs(ref).max()
    for w in range(4):
        for t in range(32):
            row, c0 = 16 * w + t % 16, 32 * (t // 16)
            assert np.all(np.abs(ld[w, t] - ref[row, c0:c0 + 32]) < tol), (w, t)
    stv = got[4096:].reshape(4, 32, 32)
    for w in range(4):
        for lane in range(16):
            for col in range(32):
                t = lane + 16 * (col // 16)
                assert stv[w, lane, col] == float(w * 100000 + t * 100 + col % 16), (w, lane, col)
