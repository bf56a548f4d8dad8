"""FP64/CPU oracle for the KV-append step (numpy), test infrastructure only.

The tests and the benchmark's CPU leg are its only callers; the product path
never imports it, and it imports nothing from the product package.

Definition (the step before attention, model card
MiMo-V2.6-Flash-RL-FP8KV-W4A8-2x-RTX-PRO-6000, "What the kernels do": an FP8
E4M3 KV cache with per-tensor scales): request b's new token t sits at
position i = seq_lens[b] - n_b + t; its K and V rows go to page
page_table[b][i // P], offset i % P, every KV head.  BF16 caches take the
bf16 bits unchanged.  FP8 caches take the E4M3 code nearest to x / scale,
where x is the bf16 value and the quotient is the fp32 IEEE quotient (the
precision the kernel decides in); ties go to the code with an even mantissa,
magnitudes beyond the largest finite E4M3 value (448) saturate to it.

The encoder is the definition read literally: it looks for the nearest value
among all finite E4M3 codes, decoded from the format (sign, 4-bit exponent
with bias 7, 3-bit mantissa, subnormals below 2^-6; 0x7F/0xFF are NaN).
Parity pins: tests/test_oracle_pins.py (append section).
"""
from __future__ import annotations

import numpy as np


def e4m3_decode(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# the 127 non-negative finite codes 0x00..0x7E, in increasing value order
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = np.array([e4m3_decode(int(c)) for c in _POS_CODES], dtype=np.float64)


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code to x, ties to even mantissa, saturating at 448."""
    if np.isnan(x):
        return 0x7F
    sign = 0x80 if np.signbit(x) else 0
    a = abs(float(x))
    if a >= _POS_VALUES[-1]:
        return sign | 0x7E
    d = np.abs(_POS_VALUES - a)
    best = np.flatnonzero(d == d.min())
    if best.size > 1:                      # a tie between two neighbours
        best = best[(_POS_CODES[best] & 1) == 0]
    return sign | int(_POS_CODES[best[0]])


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def append_kv(k_new, v_new, k_cache, v_cache, page_table, seq_lens, qo_indptr,
              kv_dtype: str, k_scale: float = 1.0, v_scale: float = 1.0):
    """Returns (k_cache, v_cache) after the append, as new arrays, and the number
    of tokens skipped for an out-of-pool page id.  k_new/v_new: uint16 (bf16 bits)
    [total_q, Hkv, D]; caches: uint16 (bf16) or uint8 (E4M3) [pages, P, Hkv, D]."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    num_pages, P = kc.shape[0], kc.shape[1]
    skipped = 0
    for b in range(len(seq_lens)):
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        n = q1 - q0
        for t in range(n):
            i = int(seq_lens[b]) - n + t
            page = int(page_table[b][i // P])
            if page < 0 or page >= num_pages:
                skipped += 1
                continue
            for cache, new, scale in ((kc, k_new, k_scale), (vc, v_new, v_scale)):
                row = np.asarray(new[q0 + t])
                if kv_dtype == "bf16":
                    cache[page, i % P] = row
                else:
                    q = bf16_to_f32(row) / np.float32(scale)      # fp32 IEEE quotient
                    cache[page, i % P] = np.vectorize(e4m3_encode, otypes=[np.uint8])(q)
    return kc, vc, skipped
