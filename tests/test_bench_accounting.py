"""The benchmark's roofline numerators against closed forms (CPU only).

bench.py counts algorithmic bytes (each visible key's K and V row once per KV
head, Q in, bf16 out, touched page-table entries, sinks) and FLOPs (2 x (192 +
128) per visible (query row, key) pair) by looping over requests.  Here the
same quantities are written out by hand for each named workload's shape; the
workloads are built without their caches, since only the shapes matter.
"""
import numpy as np

import bench
from asymmetric_kv_paged_gb300 import workloads as W

ROW = 192 + 128


def shape(name, seq, n, hq, hkv, P, window=0, kv="bf16", sinks=False, dqk=192):
    seq = np.asarray(seq, np.int32)
    n = np.asarray(n, np.int64)
    qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    empty = np.zeros(0, np.uint16)
    return W.Workload(name=name, hq=hq, hkv=hkv, page_size=P, num_pages=1, window=window,
                      kv_dtype=kv, qo_indptr=qo, seq_lens=seq,
                      page_table=np.zeros((len(seq), 1), np.int32), q=empty, k_cache=empty,
                      v_cache=empty, sinks=np.zeros(hq, np.float32) if sinks else None,
                      softmax_scale=1.0, dqk=dqk)


def test_tiny_decode():
    w = shape("c1", [512], [1], 8, 1, 16)
    kv = 512 * 1 * ROW * 2
    q_out = 1 * 8 * ROW * 2
    table = (512 // 16) * 4
    assert bench.algorithmic_bytes(w) == kv + q_out + table == 332_928
    assert bench.algorithmic_flops(w) == 2 * ROW * 512 * 8


def test_verify_both_page_sizes():
    L = 46_000 + 8
    q_out = 4 * 8 * 16 * ROW * 2
    kv = 4 * L * 2 * ROW * 2
    w = shape("c3a", [L] * 4, [8] * 4, 16, 2, 128)
    assert bench.algorithmic_bytes(w) == kv + q_out + 4 * (-(-L // 128)) * 4 == 235_894_400
    w = shape("c3b", [L] * 4, [8] * 4, 16, 2, 1)
    assert bench.algorithmic_bytes(w) == kv + q_out + 4 * L * 4 == 236_624_768
    # row t of a request sees 46,000 + t + 1 keys
    pairs = 4 * 16 * sum(46_000 + t + 1 for t in range(8))
    assert pairs == 23_554_304
    assert bench.algorithmic_flops(w) == 2 * ROW * pairs


def test_swa_with_sinks():
    n = [1, 8] * 32
    w = shape("c4", [8192] * 64, n, 16, 2, 128, window=128, sinks=True)
    # a decode row sees the last 128 keys; an 8-token block's rows together see 135,
    # which cross one page boundary (8192 - 135 = 8057 < 63 * 128 = 8064)
    keys = 32 * 128 + 32 * 135
    kv = keys * 2 * ROW * 2
    q_out = (32 * 1 + 32 * 8) * 16 * ROW * 2
    table = (32 * 1 + 32 * 2) * 4
    assert bench.algorithmic_bytes(w) == kv + q_out + table + 16 * 4 == 13_722_048
    # every row sees exactly 128 keys (all positions are past the window)
    assert bench.algorithmic_flops(w) == 2 * ROW * (32 + 256) * 16 * 128


def test_swa_with_sinks_symmetric_head_dims():
    # the same batch on a layer whose pair is 128/128: 256 bytes per K row
    n = [1, 8] * 32
    w = shape("c4s", [8192] * 64, n, 16, 2, 128, window=128, sinks=True, dqk=128)
    row = 128 + 128
    keys = 32 * 128 + 32 * 135
    kv = keys * 2 * row * 2
    q_out = (32 * 1 + 32 * 8) * 16 * row * 2
    table = (32 * 1 + 32 * 2) * 4
    assert bench.algorithmic_bytes(w) == kv + q_out + table + 16 * 4 == 10_977_728
    assert bench.algorithmic_flops(w) == 2 * row * (32 + 256) * 16 * 128


def test_chunked_prefill():
    L, n = 30_096, 4096
    w = shape("c5", [L], [n], 64, 4, 128, kv="fp8")
    kv = L * 4 * ROW * 1
    q_out = n * 64 * ROW * 2
    table = (-(-L // 128)) * 4
    assert bench.algorithmic_bytes(w) == kv + q_out + table
    # row t sees 26,000 + t + 1 keys: n * 26,001 + n (n - 1) / 2 per head
    pairs = 64 * (n * 26_001 + n * (n - 1) // 2)
    assert pairs == 7_352_745_984
    assert bench.algorithmic_flops(w) == 2 * ROW * pairs
