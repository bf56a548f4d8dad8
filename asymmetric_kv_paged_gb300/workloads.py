"""Seeded synthetic workloads for paged asymmetric-KV attention.

This module only draws inputs: request lengths, page tables, Q/K/V bit patterns
and sink logits.  It holds none of the attention arithmetic, so the GPU tests,
the benchmark and the CPU oracle can all consume the very same host bytes.

Recipe (numpy PCG64, ``default_rng(seed)``), draw order fixed:
  seq_lens -> per-request query counts -> page permutation -> q -> kv_seed -> sinks.
  * K and V values are float32 N(0, std^2), drawn row-chunk by row-chunk from
    child generators of SeedSequence((kv_seed, 0)) and ((kv_seed, 1)), kv_seed
    being the next draw of the main generator after q.
  * bf16 values are round-to-nearest-even of the float32 draws.
  * fp8 K/V: float32 N(0,1) draws, per-tensor scale = amax / 448, codes are
    RNE(x / scale) in OCP E4M3 (torch's float8_e4m3fn cast; no overflow because
    |x / scale| <= 448).
  * Only slots that some query can see get values.  Every other slot (the tail
    of a last page, keys left of a sliding window, pages nobody references) holds
    NaN: bf16 0x7FC0, fp8 0x7F.  Unused page-table columns point at a page no
    request owns (all NaN), so a kernel that reads past a request's pages
    produces NaN instead of touching memory outside the pool.
The five named workloads mirror the pages' shapes: the 1.2M-slot pools and page
sizes 1/128 of the FA4 A/B (sglang PR #41886, "Speed Tests"), the ~46K-token
verify of the RTX PRO 6000 model card ("Benchmarks"), and its 4096-token prefill
chunk after 26K cached tokens ("What the kernels do").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DQK = 192
DV = 128
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
POOL_SLOTS = 1_200_000


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (torch's CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


_CHUNK = 32768


def _draw_rows(seed: int, stream: int, rows: int, width: int, std: float) -> np.ndarray:
    """float32 N(0, std^2) values [rows, width], drawn in chunks of 32768 rows from
    child generators of SeedSequence((seed, stream)); chunks run on threads, the
    values depend only on the seed."""
    import concurrent.futures as cf
    out = np.empty((rows, width), dtype=np.float32)
    nchunks = (rows + _CHUNK - 1) // _CHUNK
    children = np.random.SeedSequence((seed, stream)).spawn(max(nchunks, 1))

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(rows, (c + 1) * _CHUNK)
        g = np.random.default_rng(children[c])
        out[lo:hi] = g.standard_normal((hi - lo, width), dtype=np.float32)
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    with cf.ThreadPoolExecutor(max_workers=min(16, max(1, nchunks))) as ex:
        list(ex.map(fill, range(nchunks)))
    return out


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 -> OCP E4M3 codes, round to nearest even (torch's CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


@dataclass
class Workload:
    name: str
    hq: int
    hkv: int
    page_size: int
    num_pages: int
    window: int
    kv_dtype: str                    # "bf16" | "fp8"
    qo_indptr: np.ndarray            # int32 [B+1]
    seq_lens: np.ndarray             # int32 [B]
    page_table: np.ndarray           # int32 [B, stride]
    q: np.ndarray                    # uint16 (bf16 bits) [total_q, Hq, Dqk] (Dqk 192 or 128)
    k_cache: np.ndarray              # uint16 | uint8 [num_pages, P, Hkv, Dqk]
    v_cache: np.ndarray              # uint16 | uint8 [num_pages, P, Hkv, 128]
    sinks: np.ndarray | None         # float32 [Hq] or None
    softmax_scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    meta: dict = field(default_factory=dict)
    dqk: int = DQK                   # query/key head dim (the value head dim is 128)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    def host_arrays(self) -> dict:
        return dict(q=self.q, k_cache=self.k_cache, v_cache=self.v_cache,
                    qo_indptr=self.qo_indptr, seq_lens=self.seq_lens,
                    page_table=self.page_table, sinks=self.sinks, window=self.window,
                    softmax_scale=self.softmax_scale, k_scale=self.k_scale,
                    v_scale=self.v_scale)

    def visible_range(self, b: int) -> tuple[int, int]:
        """Slots of request b that hold values (all others are NaN): [lo, L)."""
        L = int(self.seq_lens[b])
        n = int(self.qo_indptr[b + 1] - self.qo_indptr[b])
        lo = 0
        if self.window > 0:
            lo = max(0, L - n - self.window + 1)
        return (lo, L) if n > 0 else (L, L)


def make_workload(seed: int, seq_lens, n_per_req, hq: int, hkv: int, page_size: int,
                  num_pages: int | None = None, window: int = 0, sinks: bool = False,
                  kv_dtype: str = "bf16", k_std: float = 1.0, v_std: float = 1.0,
                  q_std: float = 1.0, softmax_scale: float | None = None,
                  name: str = "custom", rng: np.random.Generator | None = None,
                  pages_in_order: bool = False, dqk: int = DQK) -> Workload:
    """Build one workload.  `seq_lens` and `n_per_req` are per request (n <= L);
    `dqk` is the query/key head dim (the value head dim is 128)."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    seq = np.asarray(seq_lens, dtype=np.int64)
    n = np.asarray(n_per_req, dtype=np.int64)
    B = seq.shape[0]
    assert n.shape == (B,) and np.all(n >= 0) and np.all(n <= seq)
    pages_per = (seq + page_size - 1) // page_size
    need = int(pages_per.sum())
    if num_pages is None:
        num_pages = need + 2
    assert num_pages > need, "pool must keep at least one unreferenced page"
    stride = max(1, int(pages_per.max()) if B else 1)

    perm = np.arange(num_pages) if pages_in_order else rng.permutation(num_pages)
    spare = int(perm[need])                   # a page nobody owns: stays NaN
    page_table = np.full((B, stride), spare, dtype=np.int32)
    off = 0
    for b in range(B):
        page_table[b, :pages_per[b]] = perm[off:off + pages_per[b]]
        off += int(pages_per[b])

    qo_indptr = np.zeros(B + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(n)
    total_q = int(qo_indptr[-1])
    q = bf16_bits(rng.standard_normal((total_q, hq, dqk), dtype=np.float32) * np.float32(q_std))

    # slots that some query can see
    slot_lists = []
    for b in range(B):
        L, nb = int(seq[b]), int(n[b])
        lo = max(0, L - nb - window + 1) if window > 0 else 0
        if nb == 0:
            lo = L
        keys = np.arange(lo, L, dtype=np.int64)
        slot_lists.append(page_table[b, keys // page_size].astype(np.int64) * page_size + keys % page_size)
    slots = np.concatenate(slot_lists) if slot_lists else np.zeros(0, np.int64)

    nslot = num_pages * page_size
    kv_seed = int(rng.integers(0, 2**63 - 1))
    k_vals = _draw_rows(kv_seed, 0, slots.size, hkv * dqk, k_std)
    v_vals = _draw_rows(kv_seed, 1, slots.size, hkv * DV, v_std)
    if kv_dtype == "bf16":
        k_cache = np.full((nslot, hkv * dqk), BF16_NAN, dtype=np.uint16)
        v_cache = np.full((nslot, hkv * DV), BF16_NAN, dtype=np.uint16)
        k_cache[slots] = bf16_bits(k_vals)
        v_cache[slots] = bf16_bits(v_vals)
        k_scale = v_scale = 1.0
    elif kv_dtype == "fp8":
        k_cache = np.full((nslot, hkv * dqk), E4M3_NAN, dtype=np.uint8)
        v_cache = np.full((nslot, hkv * DV), E4M3_NAN, dtype=np.uint8)
        k_amax = float(np.abs(k_vals).max()) if k_vals.size else 1.0
        v_amax = float(np.abs(v_vals).max()) if v_vals.size else 1.0
        k_scale = float(np.float32(k_amax / 448.0)) or 1.0
        v_scale = float(np.float32(v_amax / 448.0)) or 1.0
        k_cache[slots] = e4m3_codes(k_vals / np.float32(k_scale))
        v_cache[slots] = e4m3_codes(v_vals / np.float32(v_scale))
    else:
        raise ValueError(kv_dtype)
    del k_vals, v_vals

    sink_arr = rng.standard_normal(hq, dtype=np.float32) if sinks else None
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(dqk)
    return Workload(name=name, hq=hq, hkv=hkv, page_size=page_size, num_pages=num_pages,
                    window=window, kv_dtype=kv_dtype, qo_indptr=qo_indptr,
                    seq_lens=seq.astype(np.int32), page_table=page_table, q=q,
                    k_cache=k_cache.reshape(num_pages, page_size, hkv, dqk),
                    v_cache=v_cache.reshape(num_pages, page_size, hkv, DV),
                    sinks=sink_arr, softmax_scale=float(softmax_scale),
                    k_scale=k_scale, v_scale=v_scale, dqk=dqk)


# ---------------------------------------------------------------------------
# The named workloads.  C3 comes in two page sizes (a: 128, b: 1).

# Further measured shapes (not among the configs above): an SWA layer with a
# symmetric head-dim pair of its own.
EXTRA_NAMES = ("c4s_swa_sinks_d128",)
CONFIG_NAMES = ("c1_tiny_decode", "c2_batched_decode", "c3a_verify_p128", "c3b_verify_p1",
                "c4_swa_sinks", "c5_chunked_prefill")


def tiny_decode() -> Workload:
    """1 request, 1 token, 8 q heads / 1 KV head, 512 keys, page 16, 32 of 64 pages."""
    rng = np.random.default_rng(1001)
    return make_workload(0, [512], [1], hq=8, hkv=1, page_size=16, num_pages=64,
                         name="c1_tiny_decode", rng=rng)


def batched_decode() -> Workload:
    """32 requests x 1 token, 16/2 heads, L ~ U[1024, 32768] not page aligned, page 128,
    1.2M-slot pool, K ~ 0.5 N(0,1), V ~ N(0,1)."""
    rng = np.random.default_rng(1002)
    seq = rng.integers(1024, 32768, size=32, endpoint=True)
    for i in range(seq.size):
        while seq[i] % 128 == 0:
            seq[i] = rng.integers(1024, 32768, endpoint=True)
    return make_workload(0, seq, np.ones(32, np.int64), hq=16, hkv=2, page_size=128,
                         num_pages=POOL_SLOTS // 128, k_std=0.5, name="c2_batched_decode",
                         rng=rng)


def batched_decode_small() -> Workload:
    """The batched decode shape at a profiler-friendly size: 32 requests, L ~
    U[1024, 8192] not page aligned, 16/2 heads, page 128, 2,000-page pool
    (~190 MB of K/V per step, still larger than L2)."""
    rng = np.random.default_rng(1012)
    seq = rng.integers(1024, 8192, size=32, endpoint=True)
    for i in range(seq.size):
        while seq[i] % 128 == 0:
            seq[i] = rng.integers(1024, 8192, endpoint=True)
    return make_workload(0, seq, np.ones(32, np.int64), hq=16, hkv=2, page_size=128,
                         num_pages=2000, k_std=0.5, name="c2_batched_decode_small", rng=rng)


def verify(page_size: int) -> Workload:
    """4 requests x 8 causal draft tokens over a 46,000-token prefix, 16/2 heads."""
    rng = np.random.default_rng(1003)
    name = "c3a_verify_p128" if page_size == 128 else f"c3b_verify_p{page_size}"
    return make_workload(0, [46008] * 4, [8] * 4, hq=16, hkv=2, page_size=page_size,
                         num_pages=POOL_SLOTS // page_size, name=name, rng=rng)


def swa_sinks(dqk: int = DQK) -> Workload:
    """64 requests (32 decode + 32 eight-token verify rows, seeded shuffle), L = 8192,
    window 128, per-head sinks N(0,1), 16/2 heads, page 128.  With dqk = 128: the
    same batch on a sliding-window layer whose own head-dim pair is 128/128."""
    rng = np.random.default_rng(1004)
    seq = np.full(64, 8192, np.int64)
    n = np.array([1] * 32 + [8] * 32, np.int64)
    rng.shuffle(n)
    name = "c4_swa_sinks" if dqk == DQK else f"c4s_swa_sinks_d{dqk}"
    return make_workload(0, seq, n, hq=16, hkv=2, page_size=128, num_pages=POOL_SLOTS // 128,
                         window=128, sinks=True, name=name, rng=rng, dqk=dqk)


def chunked_prefill() -> Workload:
    """1 request: a 4096-token causal chunk after 26,000 cached tokens, 64/4 heads,
    page 128, fp8 E4M3 K/V with per-tensor scales."""
    rng = np.random.default_rng(1005)
    return make_workload(0, [30096], [4096], hq=64, hkv=4, page_size=128,
                         num_pages=POOL_SLOTS // 128, kv_dtype="fp8",
                         name="c5_chunked_prefill", rng=rng)


def named(name: str) -> Workload:
    return {
        "c1_tiny_decode": tiny_decode,
        "c2_batched_decode": batched_decode,
        "c2_batched_decode_small": batched_decode_small,
        "c3a_verify_p128": lambda: verify(128),
        "c3b_verify_p1": lambda: verify(1),
        "c4_swa_sinks": swa_sinks,
        "c4s_swa_sinks_d128": lambda: swa_sinks(128),
        "c5_chunked_prefill": chunked_prefill,
    }[name]()
