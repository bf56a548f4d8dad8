"""Independent brute-force attention for tiny inputs (numpy long double).

Written separately from the oracle and sharing nothing with it: it gathers each
request's keys into dense K/V arrays through the page table, builds the whole
masked score matrix for the request, appends the sink as one more logit column,
and takes a vectorised softmax in extended precision.  Decoding of FP8 codes goes
through torch's float8_e4m3fn cast (a library routine), bf16 through a bit view.
"""
from __future__ import annotations

import numpy as np
import torch


def decode_kv(cache: np.ndarray) -> np.ndarray:
    if cache.dtype == np.uint16:
        return (cache.astype(np.uint32) << 16).view(np.float32).astype(np.longdouble)
    t = torch.from_numpy(np.ascontiguousarray(cache)).view(torch.float8_e4m3fn).to(torch.float32)
    return t.numpy().astype(np.longdouble)


def brute_attention(pb: dict):
    q = (np.asarray(pb["q"], np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.longdouble)
    K = decode_kv(pb["k_cache"]) * np.longdouble(pb.get("k_scale", 1.0))
    V = decode_kv(pb["v_cache"]) * np.longdouble(pb.get("v_scale", 1.0))
    qo = np.asarray(pb["qo_indptr"])
    seq = np.asarray(pb["seq_lens"])
    pt = np.asarray(pb["page_table"])
    W = int(pb.get("window", 0))
    scale = np.longdouble(pb["softmax_scale"])
    sinks = pb.get("sinks")
    _, P, hkv, _ = K.shape
    total_q, hq, _ = q.shape
    G = hq // hkv
    dv = V.shape[-1]
    out = np.zeros((total_q, hq, dv), np.longdouble)
    lse = np.zeros((total_q, hq), np.longdouble)
    for b in range(seq.shape[0]):
        L = int(seq[b])
        n = int(qo[b + 1] - qo[b])
        if n == 0:
            continue
        j = np.arange(L)
        Kb = K[pt[b, j // P], j % P]          # [L, hkv, 192]
        Vb = V[pt[b, j // P], j % P]          # [L, hkv, 128]
        pos = L - n + np.arange(n)             # absolute position of each new token
        vis = j[None, :] <= pos[:, None]
        if W > 0:
            vis &= j[None, :] > (pos[:, None] - W)
        for h in range(hq):
            g = h // G
            qb = q[qo[b]:qo[b + 1], h, :]      # [n, 192]
            s = np.full((n, L + 1), -np.inf, dtype=np.longdouble)
            for r in range(n):
                cols = np.nonzero(vis[r])[0]
                s[r, cols] = scale * (Kb[cols, g, :] @ qb[r])
            s[:, L] = np.longdouble(sinks[h]) if sinks is not None else -np.inf
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            Z = e.sum(axis=1)
            for r in range(n):
                cols = np.nonzero(vis[r])[0]
                out[qo[b] + r, h] = (e[r, cols] @ Vb[cols, g, :]) / Z[r]
            lse[qo[b]:qo[b + 1], h] = m[:, 0] + np.log(Z)
    return out, lse
