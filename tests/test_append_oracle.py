"""Pins of the KV-append oracle (oracle/append.py) on CPU: the E4M3 encoder
against the format (every finite code round-trips, ties go to the even
mantissa, magnitudes past 448 saturate) and against torch's float8_e4m3fn
cast (a library routine) on in-range values; the append itself against the
placement rule (position i = seq_lens[b] - n_b + t -> page_table[b][i // P],
offset i % P) and its FP8 codes against the decoded values."""
import numpy as np
import pytest

from oracle import append as A

torch = pytest.importorskip("torch")


def test_every_finite_code_round_trips():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue                       # NaN codes
        assert A.e4m3_encode(A.e4m3_decode(c)) == c, hex(c)


def test_ties_go_to_the_even_mantissa_and_large_values_saturate():
    vals = sorted({A.e4m3_decode(c) for c in range(0x7F)})
    for lo, hi in zip(vals, vals[1:]):
        mid = (lo + hi) / 2
        c = A.e4m3_encode(mid)
        assert A.e4m3_decode(c) in (lo, hi) and (c & 1) == 0, (lo, hi, hex(c))
    for x, code in ((448.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (-0.0, 0x80)):
        assert A.e4m3_encode(x) == code


def test_encoder_matches_torch_cast_in_range():
    x = np.random.default_rng(7).standard_normal(50000).astype(np.float32)
    x = np.concatenate([x * 100, x * 1e-2, x * 1e-3])
    x = x[np.abs(x) < 448]
    ours = np.array([A.e4m3_encode(v) for v in x], np.uint8)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_append_places_rows_and_changes_nothing_else():
    rng = np.random.default_rng(3)
    P, hkv, pages = 4, 2, 12
    seq = np.array([7, 3, 9])
    n = np.array([2, 0, 3])
    qo = np.concatenate([[0], np.cumsum(n)])
    pt = rng.permutation(pages)[:9].reshape(3, 3).astype(np.int32)
    kc = rng.integers(0, 2 ** 16, (pages, P, hkv, 192), dtype=np.uint16)
    vc = rng.integers(0, 2 ** 16, (pages, P, hkv, 128), dtype=np.uint16)
    kn = rng.integers(0, 2 ** 16, (int(qo[-1]), hkv, 192), dtype=np.uint16)
    vn = rng.integers(0, 2 ** 16, (int(qo[-1]), hkv, 128), dtype=np.uint16)
    k2, v2, skipped = A.append_kv(kn, vn, kc, vc, pt, seq, qo, "bf16")
    assert skipped == 0
    touched = set()
    for b in range(3):
        for t in range(int(n[b])):
            i = int(seq[b]) - int(n[b]) + t
            page, off = int(pt[b][i // P]), i % P
            touched.add((page, off))
            assert np.array_equal(k2[page, off], kn[qo[b] + t])
            assert np.array_equal(v2[page, off], vn[qo[b] + t])
    for page in range(pages):
        for off in range(P):
            if (page, off) not in touched:
                assert np.array_equal(k2[page, off], kc[page, off])
                assert np.array_equal(v2[page, off], vc[page, off])


def test_fp8_append_codes_decode_near_the_scaled_values():
    rng = np.random.default_rng(5)
    P, hkv, pages = 16, 1, 4
    seq, n = np.array([20]), np.array([5])
    qo = np.array([0, 5])
    pt = np.array([[2, 0]], np.int32)
    x = (rng.standard_normal((5, hkv, 192)) * 3).astype(np.float32)
    kn = (x.view(np.uint32) >> 16).astype(np.uint16)            # bf16 bits (truncated)
    vn = kn[:, :, :128].copy()
    kc = np.zeros((pages, P, hkv, 192), np.uint8)
    vc = np.zeros((pages, P, hkv, 128), np.uint8)
    k2, v2, _ = A.append_kv(kn, vn, kc, vc, pt, seq, qo, "fp8", k_scale=0.5, v_scale=2.0)
    for t in range(5):
        i = 15 + t
        page, off = int(pt[0][i // P]), i % P
        want = A.bf16_to_f32(kn[t]) / np.float32(0.5)
        got = np.vectorize(A.e4m3_decode)(k2[page, off]).astype(np.float64)
        assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -4 + 2.0 ** -10)


def test_out_of_pool_page_is_skipped():
    kc = np.zeros((2, 4, 1, 192), np.uint16)
    vc = np.zeros((2, 4, 1, 128), np.uint16)
    kn = np.ones((1, 1, 192), np.uint16)
    vn = np.ones((1, 1, 128), np.uint16)
    k2, v2, skipped = A.append_kv(kn, vn, kc, vc, np.array([[5]]), np.array([1]), np.array([0, 1]),
                                  "bf16")
    assert skipped == 1 and not k2.any() and not v2.any()
