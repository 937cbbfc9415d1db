"""Pins for the fp64 oracle's backward (oracle.bwd), each against something
other than the backward itself:

- central finite differences of the forward oracle (a directional derivative
  per input tensor, fp64, on small patterns that cover dilation, causality,
  padding, global rows and global columns inside and outside the band);
- torch autograd through a dense attention with an explicit n x n mask (the
  mask grids of tests/dense_ref.py);
- the full-attention limit against autograd through torch's
  scaled_dot_product_attention;
- closed forms and invariants: w = 0 (out = v), constant values (no score
  gradient), sum over keys of dk = 0 and of dv = sum of dout over the rows;
- the relative position bias's gradient against central differences on
  exactly representable float32 tables and against dense autograd.
"""
import itertools
import zlib

import numpy as np
import pytest
import torch

import oracle
from dense_ref import masks as dense_masks
from dense_ref import bias_matrix


def _problem(rng, B, H, n, d, G):
    x = {name: rng.standard_normal((B, H, n, d)) for name in ("q", "k", "v", "kg", "vg", "dout")}
    x["qg"] = rng.standard_normal((B, H, G, d))
    return x


def _fwd(x, pat):
    return oracle.fwd(x["q"], x["k"], x["v"], qg=x["qg"], kg=x["kg"], vg=x["vg"], **pat)


def _bwd(x, pat):
    return oracle.bwd(x["q"], x["k"], x["v"], x["dout"], qg=x["qg"], kg=x["kg"], vg=x["vg"], **pat)


PATTERNS = [
    dict(w=6, dilation=[1, 2], causal=False, pad_len=[0, 5], global_idx=[0, 9]),
    dict(w=4, dilation=[3, 1], causal=True, pad_len=[2, 0], global_idx=[4, 17]),
    dict(w=8, dilation=[1, 1], causal=False, pad_len=None, global_idx=[]),
    dict(w=0, dilation=[2, 1], causal=True, pad_len=[0, 11], global_idx=[1]),
    dict(w=40, dilation=[1, 4], causal=False, pad_len=[3, 0], global_idx=[0, 5, 19]),
    # a window per head (section 4.1 "Attention Pattern")
    dict(w=[2, 10], dilation=[1, 2], causal=False, pad_len=[0, 4], global_idx=[3, 20]),
    dict(w=[8, 0], dilation=[2, 1], causal=True, pad_len=None, global_idx=[6]),
]


@pytest.mark.parametrize("pi", range(len(PATTERNS)))
@pytest.mark.parametrize("name", ["q", "k", "v", "qg", "kg", "vg"])
def test_gradient_matches_central_differences(pi, name):
    pat = dict(PATTERNS[pi])
    G = len(pat["global_idx"])
    if name in ("qg", "kg", "vg") and G == 0:
        pytest.skip("no global tokens in this pattern")
    rng = np.random.default_rng(zlib.crc32(repr((pi, name)).encode()))
    B, H, n, d = 2, 2, 21, 5
    x = _problem(rng, B, H, n, d, G)
    grads = _bwd(x, pat)
    u = rng.standard_normal(x[name].shape)
    eps = 1e-5

    def loss(sign):
        y = dict(x)
        y[name] = x[name] + sign * eps * u
        return float(np.sum(x["dout"] * _fwd(y, pat)))

    fd = (loss(1) - loss(-1)) / (2 * eps)
    an = float(np.sum(grads["d" + name] * u))
    assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (fd, an)


def _dense_torch(x, pat):
    """Dense masked attention in torch fp64 (autograd-able), from the mask grids."""
    q, k, v, qg, kg, vg = (x[t] for t in ("q", "k", "v", "qg", "kg", "vg"))
    B, H, n, d = q.shape
    gidx = pat["global_idx"]
    rank = {g: r for r, g in enumerate(gidx)}
    rows = []
    for b in range(B):
        L = n - (pat["pad_len"][b] if pat["pad_len"] else 0)
        heads = []
        for h in range(H):
            wh = pat["w"][h] if np.ndim(pat["w"]) else pat["w"]
            local, glob = dense_masks(n, wh, pat["dilation"][h], pat["causal"], gidx, L)
            outs = []
            for i in range(n):
                if i in rank:
                    qi, kk, vv, m = qg[b, h, rank[i]], kg[b, h], vg[b, h], glob[i]
                else:
                    qi, kk, vv, m = q[b, h, i], k[b, h], v[b, h], local[i]
                m = torch.as_tensor(m)
                if not bool(m.any()):
                    outs.append(torch.zeros(d, dtype=torch.float64))
                    continue
                s = (kk @ qi) / np.sqrt(d)
                s = torch.where(m, s, torch.tensor(float("-inf"), dtype=torch.float64))
                outs.append(torch.softmax(s, dim=0) @ vv)
            heads.append(torch.stack(outs))
        rows.append(torch.stack(heads))
    return torch.stack(rows)


@pytest.mark.parametrize("pi", range(len(PATTERNS)))
def test_gradient_matches_dense_mask_autograd(pi):
    pat = dict(PATTERNS[pi])
    G = len(pat["global_idx"])
    rng = np.random.default_rng(100 + pi)
    B, H, n, d = 2, 2, 23, 4
    x = _problem(rng, B, H, n, d, G)
    grads = _bwd(x, pat)
    tx = {t: torch.tensor(a, requires_grad=(t != "dout")) for t, a in x.items()}
    out = _dense_torch(tx, pat)
    (out * tx["dout"]).sum().backward()
    for t in ("q", "k", "v") + (("qg", "kg", "vg") if G else ()):
        np.testing.assert_allclose(grads["d" + t], tx[t].grad.numpy(), atol=1e-12, rtol=0, err_msg=t)


@pytest.mark.parametrize("causal", [False, True])
def test_full_attention_limit_matches_sdpa_autograd(causal):
    g = torch.Generator().manual_seed(5 + causal)
    q, k, v, dout = (torch.randn(2, 3, 33, 16, generator=g, dtype=torch.float64) for _ in range(4))
    for t in (q, k, v):
        t.requires_grad_(True)
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
    (out * dout).sum().backward()
    grads = oracle.bwd(q.detach(), k.detach(), v.detach(), dout, w=70, dilation=[1, 1, 1], causal=causal)
    for name, t in (("dq", q), ("dk", k), ("dv", v)):
        np.testing.assert_allclose(grads[name], t.grad.numpy(), atol=1e-12, rtol=0, err_msg=name)


def test_w0_gradient_is_identity_on_values():
    """w = 0 and no globals: out = v, so dv = dout and dq = dk = 0."""
    rng = np.random.default_rng(7)
    x = _problem(rng, 2, 2, 30, 8, 0)
    pat = dict(w=0, dilation=[1, 3], causal=False, pad_len=[0, 4], global_idx=[])
    g = _bwd(x, pat)
    want_dv = x["dout"].copy()
    want_dv[1, :, 26:] = 0.0  # padding rows are never attended
    np.testing.assert_array_equal(g["dv"], want_dv)
    assert np.all(g["dq"] == 0) and np.all(g["dk"] == 0)


def test_constant_values_give_no_score_gradient():
    """Every value row equal: out is that row whatever the weights, so the
    score gradient vanishes (dq = dk = 0 up to rounding)."""
    rng = np.random.default_rng(8)
    x = _problem(rng, 1, 2, 40, 6, 2)
    row = rng.standard_normal(6)
    x["v"][:] = row
    x["vg"][:] = row
    pat = dict(w=10, dilation=[1, 2], causal=True, pad_len=None, global_idx=[3, 30])
    g = _bwd(x, pat)
    for t in ("dq", "dk", "dqg", "dkg"):
        assert np.abs(g[t]).max() <= 1e-12, t


@pytest.mark.parametrize("pi", range(len(PATTERNS)))
def test_key_gradient_sums_vanish_and_value_gradient_sums_dout(pi):
    """Per row the score gradients sum to zero (softmax is shift-invariant), so
    the key gradients of each (b, h) sum to zero; the weights sum to one, so
    the value gradients sum to the dout of the rows that attend anything."""
    pat = dict(PATTERNS[pi])
    G = len(pat["global_idx"])
    rng = np.random.default_rng(200 + pi)
    B, H, n, d = 2, 2, 25, 3
    x = _problem(rng, B, H, n, d, G)
    g = _bwd(x, pat)
    dk_sum = g["dk"].sum(axis=2) + (g["dkg"].sum(axis=2) if G else 0.0)
    assert np.abs(dk_sum).max() <= 1e-12
    want = np.zeros((B, H, d))
    for b in range(B):
        L = n - (pat["pad_len"][b] if pat["pad_len"] else 0)
        want[b] = x["dout"][b, :, :L].sum(axis=1)
    dv_sum = g["dv"].sum(axis=2) + (g["dvg"].sum(axis=2) if G else 0.0)
    np.testing.assert_allclose(dv_sum, want, atol=1e-12, rtol=0)


def test_bf16_inputs_decode_exactly():
    """bf16 inputs (and dout) give the gradient of the same values in float64."""
    g = torch.Generator().manual_seed(9)
    t = {n: torch.randn(1, 2, 19, 8, generator=g).to(torch.bfloat16) for n in ("q", "k", "v", "dout")}
    pat = dict(w=6, dilation=[1, 2], causal=False, global_idx=[])
    a = oracle.bwd(t["q"], t["k"], t["v"], t["dout"], **pat)
    b = oracle.bwd(*(t[n].double() for n in ("q", "k", "v", "dout")), **pat)
    for name in a:
        np.testing.assert_array_equal(a[name], b[name])


# ---------------------------------------------------------------- relative position bias
BIAS_PATTERNS = [
    dict(w=6, dilation=[1, 2], causal=False, pad_len=[0, 5], global_idx=[0, 9]),
    dict(w=4, dilation=[3, 1], causal=True, pad_len=None, global_idx=[]),
    dict(w=40, dilation=[1, 2], causal=False, pad_len=[2, 0], global_idx=[11]),
]


def _table(rng, H, w):
    """A bias table on a 2^-10 grid, so that +- 2^-12 steps stay exact in float32."""
    return np.round(rng.standard_normal((H, w + 1)) * 1024) / 1024


@pytest.mark.parametrize("pi", range(len(BIAS_PATTERNS)))
def test_bias_gradient_matches_central_differences(pi):
    pat = BIAS_PATTERNS[pi]
    rng = np.random.default_rng(300 + pi)
    B, H, n, d = 2, 2, 23, 4
    x = _problem(rng, B, H, n, d, len(pat["global_idx"]))
    rb = _table(rng, H, pat["w"])
    grads = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], qg=x["qg"], kg=x["kg"], vg=x["vg"],
                       rel_bias=rb.astype(np.float32), **pat)
    u = rng.choice([-1.0, 1.0], size=rb.shape)
    eps = 2.0 ** -12

    def loss(sign):
        t = (rb + sign * eps * u).astype(np.float32)
        assert np.array_equal(t.astype(np.float64), rb + sign * eps * u)
        out = oracle.fwd(x["q"], x["k"], x["v"], qg=x["qg"], kg=x["kg"], vg=x["vg"], rel_bias=t, **pat)
        return float(np.sum(x["dout"] * out))

    fd = (loss(1) - loss(-1)) / (2 * eps)
    an = float(np.sum(grads["drel_bias"] * u))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


@pytest.mark.parametrize("pi", range(len(BIAS_PATTERNS)))
def test_bias_gradient_matches_dense_autograd(pi):
    """Every gradient, the bias's included, against autograd through dense
    masked attention with the bias matrix gathered from a leaf table."""
    pat = BIAS_PATTERNS[pi]
    gidx = pat["global_idx"]
    rng = np.random.default_rng(400 + pi)
    B, H, n, d = 2, 2, 23, 4
    x = _problem(rng, B, H, n, d, len(gidx))
    rb = _table(rng, H, pat["w"]).astype(np.float32)
    grads = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], qg=x["qg"], kg=x["kg"], vg=x["vg"], rel_bias=rb, **pat)
    tx = {t: torch.tensor(a, requires_grad=(t != "dout")) for t, a in x.items()}
    table = torch.tensor(rb.astype(np.float64), requires_grad=True)
    rank = {g: r for r, g in enumerate(gidx)}
    w, causal = pat["w"], pat["causal"]
    rows = []
    for b in range(B):
        L = n - (pat["pad_len"][b] if pat["pad_len"] else 0)
        heads = []
        for h in range(H):
            dl = pat["dilation"][h]
            local, glob = dense_masks(n, w, dl, causal, gidx, L)
            # the bias matrix as a gather from the leaf table (indices from the grids)
            onehot = np.stack([bias_matrix(n, w, dl, causal, np.eye(w + 1)[t]) for t in range(w + 1)], -1)
            bm = torch.tensor(onehot) @ table[h]
            outs = []
            for i in range(n):
                if i in rank:
                    qi, kk, vv, m, bi = tx["qg"][b, h, rank[i]], tx["kg"][b, h], tx["vg"][b, h], glob[i], 0.0
                else:
                    qi, kk, vv, m, bi = tx["q"][b, h, i], tx["k"][b, h], tx["v"][b, h], local[i], bm[i]
                m = torch.as_tensor(m)
                if not bool(m.any()):
                    outs.append(torch.zeros(d, dtype=torch.float64))
                    continue
                s = (kk @ qi) / np.sqrt(d) + bi
                s = torch.where(m, s, torch.tensor(float("-inf"), dtype=torch.float64))
                outs.append(torch.softmax(s, dim=0) @ vv)
            heads.append(torch.stack(outs))
        rows.append(torch.stack(heads))
    out = torch.stack(rows)
    (out * tx["dout"]).sum().backward()
    np.testing.assert_allclose(grads["drel_bias"], table.grad.numpy(), atol=1e-12, rtol=0)
    for t in ("q", "k", "v") + (("qg", "kg", "vg") if gidx else ()):
        np.testing.assert_allclose(grads["d" + t], tx[t].grad.numpy(), atol=1e-12, rtol=0, err_msg=t)
