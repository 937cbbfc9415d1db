"""Brute-force dense attention with an explicit n x n mask (numpy, float64).

A second, independent statement of the Longformer pattern used only to pin
the loop oracle: it builds the whole boolean mask from index grids and runs
ordinary dense softmax attention, where the oracle walks each row's window.
Pattern (velog.io/@lainshower/Longformer, section 3-1): band |j - i| <= w/2
with dilation gaps, look-back only when causal (section 4.1), global tokens
as full rows (scored with qg, kg, vg) and full columns, padding masked.
w is one window for every head or a sequence with one per head (section 4.1).
rel_bias: optional [H, w + 1] table added to the band keys' scores of
ordinary rows at window step t (entry t + w/2), the T5-style position bias of
the Memorizing Transformer notes.
"""
import numpy as np


def masks(n, w, delta, causal, global_idx, L):
    """(mask for ordinary rows, mask for global rows), each [n, n] bool."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    off = j - i
    half = w // 2
    band = (off % delta == 0) & (off >= -delta * half)
    band &= (off <= 0) if causal else (off <= delta * half)
    is_g = np.zeros(n, dtype=bool)
    is_g[list(global_idx)] = True
    key_ok = j < L
    order_ok = (j <= i) if causal else np.ones_like(band)
    local = (band | (is_g[None, :] & order_ok)) & key_ok & (i < L)
    glob = key_ok & order_ok & (i < L)
    return local, glob


def bias_matrix(n, w, delta, causal, table):
    """[n, n] additive bias: table[t + w/2] on the band at window step t, 0 elsewhere."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    off = j - i
    half = w // 2
    band = (off % delta == 0) & (off >= -delta * half) & (off <= (0 if causal else delta * half))
    t = np.clip(off // delta + half, 0, w)
    return np.where(band, np.asarray(table, dtype=np.float64)[t], 0.0)


def attention(q, k, v, w, dilation, causal=False, pad_len=None, qg=None, kg=None, vg=None,
              global_idx=(), rel_bias=None):
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, n, d = q.shape
    out = np.zeros_like(q)
    rank = {g: r for r, g in enumerate(global_idx)}
    for b in range(B):
        L = n - (pad_len[b] if pad_len is not None else 0)
        for h in range(H):
            local, glob = masks(n, w[h] if np.ndim(w) else w, dilation[h], causal, global_idx, L)
            qq = q[b, h].copy()
            kk = np.repeat(k[b, h][None], n, axis=0)  # per-row key matrix [n, n, d]
            vv = np.repeat(v[b, h][None], n, axis=0)
            m = local.copy()
            for g, r in rank.items():
                qq[g] = np.asarray(qg, dtype=np.float64)[b, h, r]
                kk[g] = np.asarray(kg, dtype=np.float64)[b, h]
                vv[g] = np.asarray(vg, dtype=np.float64)[b, h]
                m[g] = glob[g]
            s = np.einsum("id,ijd->ij", qq, kk) / np.sqrt(d)
            if rel_bias is not None:  # band keys of ordinary rows only
                bm = bias_matrix(n, w, dilation[h], causal, rel_bias[h])
                bm[list(global_idx)] = 0.0
                s = s + bm
            s = np.where(m, s, -np.inf)
            rowmax = np.max(s, axis=1, keepdims=True)
            rowmax = np.where(np.isfinite(rowmax), rowmax, 0.0)
            p = np.where(m, np.exp(s - rowmax), 0.0)
            tot = p.sum(axis=1, keepdims=True)
            o = np.einsum("ij,ijd->id", p, vv)
            out[b, h] = np.where(tot > 0, o / np.where(tot > 0, tot, 1.0), 0.0)
    return out
