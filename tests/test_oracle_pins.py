"""Pins for the fp64 oracle: it is checked against things other than itself.

- hand-written attended sets and hand-computed softmax outputs (tests/golden/)
- a brute-force dense implementation with an explicit n x n mask
- the full-attention limit against torch's scaled_dot_product_attention
- closed forms (constant values, w = 0, uniform weights) and invariants
  (dilation residue identity, causal and padding NaN poison, global symmetry)
"""
import itertools
import json
import math
import os
import zlib

import numpy as np
import pytest
import torch

import oracle
from dense_ref import attention as dense_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_sets():
    cases = []
    cur = None
    for line in open(os.path.join(GOLDEN, "attended_sets.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case "):
            parts = line.split()
            kv = dict(p.split("=") for p in parts[2:])
            cur = {
                "name": parts[1],
                "n": int(kv["n"]),
                "w": int(kv["w"]),
                "dilation": [int(x) for x in kv["dilation"].split(",")],
                "causal": bool(int(kv["causal"])),
                "global_idx": [] if kv["global"] == "-" else [int(x) for x in kv["global"].split(",")],
                "pad": int(kv["pad"]),
                "rows": {},
            }
            cases.append(cur)
            continue
        head, rest = line.split(":", 1)
        hs = head.split()
        h, i = int(hs[0]), int(hs[1])
        is_g = len(hs) > 2 and hs[2] == "G"
        cur["rows"][(h, i)] = (sorted(int(x) for x in rest.split()), is_g)
    return cases


SET_CASES = _parse_sets()


@pytest.mark.parametrize("case", SET_CASES, ids=[c["name"] for c in SET_CASES])
def test_golden_attended_sets(case):
    H = len(case["dilation"])
    assert len(case["rows"]) == H * case["n"]
    for (h, i), (keys, is_g) in case["rows"].items():
        got, got_g = oracle.attended(n=case["n"], w=case["w"], dilation=case["dilation"],
                                     causal=case["causal"], global_idx=case["global_idx"],
                                     pad_len=[case["pad"]], h=h, i=i)
        assert got == keys, (h, i)
        assert got_g == (is_g and keys != [])


@pytest.mark.parametrize("case", SET_CASES, ids=[c["name"] for c in SET_CASES])
def test_golden_sets_through_outputs(case):
    """With all scores equal (q = 0, qg = 0) the output is the uniform average of
    the attended values; with v = identity rows it is indicator(set) / |set|."""
    n, H = case["n"], len(case["dilation"])
    G = len(case["global_idx"])
    d = n
    z = np.zeros((1, H, n, d))
    eye = np.broadcast_to(np.eye(n), (1, H, n, d)).copy()
    k = np.random.default_rng(0).standard_normal((1, H, n, d))
    out = oracle.fwd(z, k, eye, w=case["w"], dilation=case["dilation"], causal=case["causal"],
                     pad_len=[case["pad"]], qg=np.zeros((1, H, G, d)), kg=k.copy(), vg=eye.copy(),
                     global_idx=case["global_idx"])
    for (h, i), (keys, _) in case["rows"].items():
        want = np.zeros(n)
        if keys:
            want[keys] = 1.0 / len(keys)
        np.testing.assert_allclose(out[0, h, i], want, atol=1e-15, rtol=0)


def _val(x):
    if isinstance(x, str):
        assert x.startswith("ln(") and x.endswith(")")
        return math.log(float(x[3:-1]))
    return float(x)


def _arr(rows, H=1):
    return np.array([[[[_val(x) for x in r] for r in rows]]], dtype=np.float64)


SOFTMAX_CASES = json.load(open(os.path.join(GOLDEN, "softmax_by_hand.json")))["cases"]


@pytest.mark.parametrize("case", SOFTMAX_CASES, ids=[c["name"] for c in SOFTMAX_CASES])
def test_golden_softmax_by_hand(case):
    G = len(case["global_idx"])
    kw = {}
    if G:
        kw = dict(qg=_arr(case["qg"]), kg=_arr(case["kg"]), vg=_arr(case["vg"]))
    out = oracle.fwd(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]), w=case["w"],
                     dilation=case["dilation"], causal=bool(case["causal"]),
                     global_idx=case["global_idx"], **kw)
    np.testing.assert_allclose(out[0, 0], np.array(case["out"]), rtol=1e-13, atol=1e-13)


def _rand_problem(rng, B, H, n, d, G):
    q, k, v = (rng.standard_normal((B, H, n, d)) for _ in range(3))
    qg = rng.standard_normal((B, H, G, d))
    kg, vg = rng.standard_normal((B, H, n, d)), rng.standard_normal((B, H, n, d))
    return q, k, v, qg, kg, vg


GRID = []
for n, d, w, dl, causal, gsel, pad in itertools.product(
        [1, 2, 7, 64, 130], [1, 8, 64], [0, 2, 6, 64, 600], [1, 2, 3, 4], [False, True],
        ["none", "one", "few", "all"], [False, True]):
    GRID.append((n, d, w, dl, causal, gsel, pad))
# a deterministic subsample keeps the CPU suite quick while touching every value
GRID = [g for t, g in enumerate(GRID) if t % 7 == 0]


@pytest.mark.parametrize("n,d,w,dl,causal,gsel,pad", GRID)
def test_oracle_matches_dense_mask(n, d, w, dl, causal, gsel, pad):
    rng = np.random.default_rng(zlib.crc32(repr((n, d, w, dl, causal, gsel, pad)).encode()))
    gidx = {"none": [], "one": [0], "few": sorted(set([0, n // 3, n - 1])), "all": list(range(n))}[gsel]
    B, H = 2, 2
    dil = [1, dl]
    pads = [0, (n // 3) if pad else 0]
    q, k, v, qg, kg, vg = _rand_problem(rng, B, H, n, d, len(gidx))
    got = oracle.fwd(q, k, v, w=w, dilation=dil, causal=causal, pad_len=pads, qg=qg, kg=kg, vg=vg,
                     global_idx=gidx)
    want = dense_attention(q, k, v, w, dil, causal, pads, qg, kg, vg, gidx)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("wh,dil", [([0, 6, 64], [1, 1, 1]), ([10, 2, 30], [1, 3, 2]), ([4, 4, 600], [2, 1, 1])])
def test_per_head_windows_match_dense_mask(wh, dil, causal):
    """A window per head (section 4.1 "Attention Pattern") against the dense
    mask built head by head; one head's window reaches past the sequence."""
    n, d, B = 130, 8, 2
    gidx = [0, 64, 129]
    pads = [0, 40]
    rng = np.random.default_rng(sum(wh) + 7 * causal)
    q, k, v, qg, kg, vg = _rand_problem(rng, B, len(wh), n, d, len(gidx))
    got = oracle.fwd(q, k, v, w=wh, dilation=dil, causal=causal, pad_len=pads, qg=qg, kg=kg, vg=vg,
                     global_idx=gidx)
    want = dense_attention(q, k, v, wh, dil, causal, pads, qg, kg, vg, gidx)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)
    # and a head's rows do not depend on the other heads' windows
    for h, w in enumerate(wh):
        one = oracle.fwd(q, k, v, w=w, dilation=dil, causal=causal, pad_len=pads, qg=qg, kg=kg, vg=vg,
                         global_idx=gidx)
        np.testing.assert_array_equal(got[:, h], one[:, h])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(5, 3), (64, 16), (200, 64)])
def test_full_attention_limit_matches_sdpa(n, d, causal):
    """w >= 2n, dilation 1, no globals, no padding is ordinary (causal) attention."""
    g = torch.Generator().manual_seed(n * 7 + d)
    q, k, v = (torch.randn(2, 3, n, d, generator=g, dtype=torch.float64) for _ in range(3))
    want = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
    got = oracle.fwd(q, k, v, w=2 * n + 2, dilation=[1, 1, 1], causal=causal)
    np.testing.assert_allclose(got, want.numpy(), atol=1e-12, rtol=0)


def test_constant_values_rows_sum_to_one():
    rng = np.random.default_rng(3)
    B, H, n, d = 2, 3, 97, 16
    q, k, _, qg, kg, _ = _rand_problem(rng, B, H, n, d, 2)
    c = rng.standard_normal(d)
    v = np.broadcast_to(c, (B, H, n, d)).copy()
    out = oracle.fwd(q * 4, k, v, w=10, dilation=[1, 2, 5], causal=False, pad_len=[0, 7], qg=qg,
                     kg=kg, vg=v.copy(), global_idx=[3, 50])
    np.testing.assert_allclose(out[0], np.broadcast_to(c, (H, n, d)), atol=1e-13)
    np.testing.assert_allclose(out[1, :, : n - 7], np.broadcast_to(c, (H, n - 7, d)), atol=1e-13)
    assert np.all(out[1, :, n - 7:] == 0.0)


def test_w0_is_identity():
    rng = np.random.default_rng(4)
    q, k, v, *_ = _rand_problem(rng, 1, 2, 33, 8, 0)
    out = oracle.fwd(q, k, v, w=0, dilation=[1, 3])
    assert np.array_equal(out, v)


def test_causal_first_row_is_its_value():
    rng = np.random.default_rng(5)
    q, k, v, *_ = _rand_problem(rng, 1, 2, 20, 8, 0)
    out = oracle.fwd(q, k, v, w=8, dilation=[1, 3], causal=True)
    assert np.array_equal(out[0, 0, 0], v[0, 0, 0])
    for i in range(3):  # rows below the dilation see only themselves
        assert np.array_equal(out[0, 1, i], v[0, 1, i])


@pytest.mark.parametrize("causal", [False, True])
def test_dilation_residue_identity(causal):
    """A delta-dilated window on row r + delta*m equals the undilated window on
    the subsequence r, r + delta, r + 2*delta, ..."""
    rng = np.random.default_rng(6)
    n, d, w = 61, 8, 6
    q, k, v, *_ = _rand_problem(rng, 1, 1, n, d, 0)
    for delta in (2, 3, 4):
        dil = oracle.fwd(q, k, v, w=w, dilation=[delta], causal=causal)
        for r in range(delta):
            sub = oracle.fwd(q[:, :, r::delta], k[:, :, r::delta], v[:, :, r::delta], w=w,
                             dilation=[1], causal=causal)
            np.testing.assert_allclose(dil[:, :, r::delta], sub, atol=1e-14, rtol=0)


@pytest.mark.parametrize("delta,causal", [(1, False), (3, False), (1, True), (4, True)])
def test_interior_window_count(delta, causal):
    n, w = 300, 16
    for i in range(delta * w, n - delta * w):
        keys, _ = oracle.attended(n=n, w=w, dilation=[delta], causal=causal, i=i)
        assert len(keys) == (w // 2 + 1 if causal else w + 1)
        assert all((j - i) % delta == 0 for j in keys)
        assert max(abs(j - i) for j in keys) == delta * w // 2


def test_causal_never_reads_the_future():
    rng = np.random.default_rng(7)
    n, d = 90, 8
    q, k, v, qg, kg, vg = _rand_problem(rng, 1, 2, n, d, 2)
    gidx = [10, 40]
    base = oracle.fwd(q, k, v, w=12, dilation=[1, 2], causal=True, qg=qg, kg=kg, vg=vg, global_idx=gidx)
    for i0 in (0, 9, 10, 41, 89):
        kp, vp, kgp, vgp = k.copy(), v.copy(), kg.copy(), vg.copy()
        for a in (kp, vp, kgp, vgp):
            a[:, :, i0 + 1:] = np.nan
        got = oracle.fwd(q, kp, vp, w=12, dilation=[1, 2], causal=True, qg=qg, kg=kgp, vg=vgp,
                         global_idx=gidx)
        assert np.array_equal(got[:, :, : i0 + 1], base[:, :, : i0 + 1])


def test_padding_poison_and_zero_rows():
    rng = np.random.default_rng(8)
    n, d = 70, 8
    q, k, v, qg, kg, vg = _rand_problem(rng, 2, 2, n, d, 3)
    gidx = [0, 30, 65]
    pads = [0, 20]
    base = oracle.fwd(q, k, v, w=10, dilation=[1, 2], pad_len=pads, qg=qg, kg=kg, vg=vg, global_idx=gidx)
    poisoned = [a.copy() for a in (q, k, v, kg, vg)]
    for a in poisoned:
        a[1, :, n - 20:] = np.nan
    got = oracle.fwd(poisoned[0], poisoned[1], poisoned[2], w=10, dilation=[1, 2], pad_len=pads, qg=qg,
                     kg=poisoned[3], vg=poisoned[4], global_idx=gidx)
    assert np.array_equal(got, base)
    assert np.all(got[1, :, n - 20:] == 0.0)


def test_global_tokens_see_and_are_seen_by_all():
    rng = np.random.default_rng(9)
    n, d = 80, 8
    q, k, v, qg, kg, vg = _rand_problem(rng, 1, 1, n, d, 2)
    gidx = [5, 60]
    kw = dict(w=4, dilation=[1], qg=qg, kg=kg, vg=vg, global_idx=gidx)
    base = oracle.fwd(q, k, v, **kw)
    # perturbing the key of a global token changes every ordinary row
    k2 = k.copy()
    k2[0, 0, 60] += 1.0
    changed = np.any(oracle.fwd(q, k2, v, **kw) != base, axis=-1)[0, 0]
    assert all(changed[i] for i in range(n) if i not in gidx)
    # perturbing any global-projection key changes every global row
    for j in (0, 33, 79):
        kg2 = kg.copy()
        kg2[0, 0, j] += 1.0
        out = oracle.fwd(q, k, v, **{**kw, "kg": kg2})
        assert all(np.any(out[0, 0, g] != base[0, 0, g]) for g in gidx)
    # a global row is dense attention of qg over all keys with kg, vg
    for r, g in enumerate(gidx):
        s = kg[0, 0] @ qg[0, 0, r] / math.sqrt(d)
        p = np.exp(s - s.max())
        np.testing.assert_allclose(base[0, 0, g], p @ vg[0, 0] / p.sum(), atol=1e-13)


def test_bf16_and_f32_inputs_decode_exactly():
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(1, 2, 40, 8, generator=g) for _ in range(3))
    for dt in (torch.bfloat16, torch.float32):
        qq, kk, vv = (x.to(dt) for x in (q, k, v))
        a = oracle.fwd(qq, kk, vv, w=6, dilation=[1, 2])
        b = oracle.fwd(qq.double(), kk.double(), vv.double(), w=6, dilation=[1, 2])
        assert np.array_equal(a, b)


def test_sampled_rows_equal_full_rows():
    rng = np.random.default_rng(12)
    B, H, n, d = 2, 2, 50, 8
    q, k, v, qg, kg, vg = _rand_problem(rng, B, H, n, d, 1)
    kw = dict(w=6, dilation=[1, 3], causal=False, pad_len=[0, 5], qg=qg, kg=kg, vg=vg, global_idx=[7])
    full = oracle.fwd(q, k, v, **kw)
    rows = [0, 7, 49, 50 + 7, 2 * n + 3, 4 * n - 1]
    part = oracle.fwd(q, k, v, rows=rows, **kw)
    assert np.array_equal(part, full.reshape(-1, d)[rows])


def test_rejects_invalid_patterns():
    z = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=3, dilation=[1])  # odd window
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=[5], dilation=[1])  # odd window of a head
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=[2, 2], dilation=[1])  # one window per head
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=2, dilation=[0])
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=2, dilation=[1], qg=np.zeros((1, 1, 2, 2)), kg=z, vg=z, global_idx=[2, 1])


# ---------------------------------------------------------------- relative position bias
BIAS_CASES = [  # n, d, w, dilation, causal, global_idx, pad_len
    (40, 8, 6, [1, 2], False, [], None),
    (64, 4, 10, [1, 3], True, [0, 33], [0, 9]),
    (50, 8, 8, [2, 1], False, [5, 6, 49], [7, 0]),
    (30, 2, 100, [1, 1], False, [0], None),      # the window reaches past both ends
    (33, 5, 0, [1, 2], True, [2], [0, 3]),
]


@pytest.mark.parametrize("case", BIAS_CASES, ids=str)
def test_relative_bias_matches_dense_mask(case):
    """The T5-style bias (Memorizing Transformer notes, "Position bias"),
    read as one scalar per head and window step added to the band keys'
    scores, against the dense mask with the bias matrix built from index
    grids; global columns outside the band and global rows get none."""
    n, d, w, dil, causal, gidx, pads = case
    rng = np.random.default_rng(n + 10 * w + causal)
    B, H = 2, len(dil)
    q, k, v, qg, kg, vg = _rand_problem(rng, B, H, n, d, len(gidx))
    rb = rng.standard_normal((H, w + 1)).astype(np.float32) * 2
    got = oracle.fwd(q, k, v, w=w, dilation=dil, causal=causal, pad_len=pads, qg=qg, kg=kg, vg=vg,
                     global_idx=gidx, rel_bias=rb)
    want = dense_attention(q, k, v, w, dil, causal, pads, qg, kg, vg, gidx, rel_bias=rb)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)


def test_relative_bias_zero_table_is_no_bias():
    rng = np.random.default_rng(3)
    q, k, v, qg, kg, vg = _rand_problem(rng, 1, 2, 70, 8, 2)
    kw = dict(w=12, dilation=[1, 2], causal=False, qg=qg, kg=kg, vg=vg, global_idx=[0, 40])
    np.testing.assert_array_equal(oracle.fwd(q, k, v, **kw),
                                  oracle.fwd(q, k, v, rel_bias=np.zeros((2, 13), np.float32), **kw))


@pytest.mark.parametrize("causal", [False, True])
def test_relative_bias_constant_shift_cancels_without_globals(causal):
    """Softmax is invariant to a constant added to every score of a row: a
    table holding one value changes nothing when every key is a band key."""
    rng = np.random.default_rng(4 + causal)
    q, k, v = (rng.standard_normal((2, 3, 80, 8)) for _ in range(3))
    kw = dict(w=16, dilation=[1, 2, 5], causal=causal, pad_len=[0, 13])
    base = oracle.fwd(q, k, v, **kw)
    shifted = oracle.fwd(q, k, v, rel_bias=np.full((3, 17), 3.25, np.float32), **kw)
    np.testing.assert_allclose(shifted, base, atol=1e-12, rtol=0)


def test_relative_bias_peaked_at_the_token_returns_its_value():
    """A bias of +80 at step 0 and 0 elsewhere: each row's weight on itself is
    1 - O(w e^-80), so the output is the row's own value."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((1, 2, 60, 8)) * 0.1 for _ in range(3))
    rb = np.zeros((2, 9), np.float32)
    rb[:, 4] = 80.0
    out = oracle.fwd(q, k, v, w=8, dilation=[1, 3], rel_bias=rb)
    np.testing.assert_allclose(out, v, atol=1e-30 + 1e-12, rtol=0)


def test_relative_bias_steps_index_the_table():
    """One row by hand: with q = 0 every score is its bias, so the weights are
    softmax(bias over the row's window steps) and the output their average of
    v.  Row 10 of a dilation-2 head with w = 4 reads keys 6, 8, 10, 12, 14 at
    steps -2..2, i.e. table entries 0..4."""
    n, d = 20, 3
    q = np.zeros((1, 1, n, d))
    k = np.ones((1, 1, n, d))
    v = np.arange(n * d, dtype=np.float64).reshape(1, 1, n, d)
    table = np.array([[0.5, -1.0, 2.0, 0.25, 1.5]], np.float32)
    out = oracle.fwd(q, k, v, w=4, dilation=[2], rel_bias=table)
    wts = np.exp(table[0].astype(np.float64))
    wts /= wts.sum()
    want = sum(wt * v[0, 0, j] for wt, j in zip(wts, [6, 8, 10, 12, 14]))
    np.testing.assert_allclose(out[0, 0, 10], want, rtol=1e-14, atol=0)


def test_relative_bias_rejected_shapes():
    z = np.zeros((1, 2, 8, 2))
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=4, dilation=[1, 1], rel_bias=np.zeros((2, 4), np.float32))
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, w=[4, 4], dilation=[1, 1], rel_bias=np.zeros((2, 5), np.float32))


@pytest.mark.parametrize("causal", [False, True])
def test_per_head_window_pair_count_matches_dense_masks(causal):
    """The oracle's pair count with a window per head equals the number of
    attended entries in the dense masks built head by head."""
    from dense_ref import masks
    n, wh, dil, gidx, pads = 70, [0, 6, 40, 200], [1, 2, 1, 3], [0, 35], [0, 11]
    pairs, gpairs = oracle.count_pairs(B=2, H=4, n=n, w=wh, dilation=dil, causal=causal, global_idx=gidx,
                                       pad_len=pads)
    want = wantg = 0
    for b in range(2):
        L = n - pads[b]
        for h in range(4):
            local, glob = masks(n, wh[h], dil[h], causal, gidx, L)
            for i in range(n):
                if i in gidx:
                    want += int(glob[i].sum())
                    wantg += int(glob[i].sum())
                else:
                    want += int(local[i].sum())
    assert (pairs, gpairs) == (want, wantg)
