"""Contiguous-cache brute force used to pin the oracle.

It never looks at a pool: every sequence's K/V comes straight from the drawn
values in logical position order (the "Contiguous" column of weft's
"Cache layouts" table), and attention is the textbook softmax(scale q K^T) V
with a matmul as the only library step.
"""
import numpy as np

from paged_kv_cache_wf_gb300 import workloads as W


def brute_attention(layout, vals, scale):
    """fp64 outputs [T_total, H_q, D] for every new query row (decode or prefill)."""
    g = layout.geom
    G = g.G
    q_all = W.storage_to_f64(vals.q, g.dtype)
    out = np.zeros((layout.T_total, g.H_q, g.D))
    cq = layout.cu_q_lens
    for b in range(layout.B):
        K = W.storage_to_f64(W.dense_sequence(layout, vals, b, "k"), g.dtype)  # [L, H_kv, D]
        V = W.storage_to_f64(W.dense_sequence(layout, vals, b, "v"), g.dtype)
        L = int(layout.seq_lens[b])
        n = int(layout.q_lens[b])
        assert K.shape[0] == L
        c = L - n
        for i in range(n):
            visible = c + i + 1  # causal: positions 0 .. c+i (a decode row sees all L)
            for hq in range(g.H_q):
                h = hq // G
                s = scale * (K[:visible, h, :] @ q_all[cq[b] + i, hq])
                w = np.exp(s - s.max())
                out[cq[b] + i, hq] = (w @ V[:visible, h, :]) / w.sum()
    return out
