"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs, plus properties that must hold at any size.

Tolerances: bf16 I/O with fp32 accumulation, max |err| <= 2e-2 and
mean |err| <= 2e-3; fp32, max |err| <= 1e-4.
"""
import itertools
import zlib

import numpy as np
import pytest
import torch

import long_sequence_sliding_longformer_b300 as lf
import oracle
import workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_MAX = 2e-2, 2e-3, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_sequence_sliding_longformer_b300 import _build
    _build.build()
    lf.load()
    assert lf.device_error(clear=True) == 0


def run(wl, inp, **kw):
    out = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                  pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, **kw)
    torch.cuda.synchronize()
    return out


def check(wl, got, want, rows=None):
    g = got.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g.reshape(-1, wl.d)[rows]
    assert np.all(np.isfinite(g))
    err = np.abs(g - want)
    if wl.dtype == "f32":
        assert err.max() <= F32_MAX, err.max()
    else:
        assert err.max() <= BF16_MAX, err.max()
        assert err.mean() <= BF16_MEAN, err.mean()
    return err


def sample_rows(wl, rng, extra=4096):
    """Row ids covering the first/last two tiles of every head, all global rows
    and a random spread (flat ids (b*H + h)*n + i)."""
    rows = set()
    n = wl.n
    for b in range(wl.B):
        for h in range(wl.H):
            base = (b * wl.H + h) * n
            for i in list(range(0, min(n, 256))) + list(range(max(0, n - 256), n)):
                rows.add(base + i)
            for g in wl.global_idx:
                rows.add(base + g)
    total = wl.B * wl.H * n
    rows.update(rng.integers(0, total, size=extra).tolist())
    return np.array(sorted(rows), dtype=np.int64)


# ---------------------------------------------------------------- named workloads
def test_fp32_window64_full():
    wl = workloads.fp32_window64()
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


def test_bf16_encoder_full():
    wl = workloads.bf16_encoder()
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


def test_bf16_charlm_causal_dilated_full():
    wl = workloads.bf16_charlm()
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


def test_bf16_qa_padded_full():
    wl = workloads.bf16_qa_padded()
    inp = workloads.make_inputs(wl, "cuda")
    out = run(wl, inp)
    check(wl, out, oracle.wl_fwd(wl, inp))
    for b, p in enumerate(wl.pad_len):
        if p:
            assert torch.all(out[b, :, wl.n - p:] == 0)


@pytest.mark.parametrize("n", workloads.LED_LENGTHS)
def test_bf16_led_sampled(n):
    wl = workloads.bf16_led(n)
    inp = workloads.make_inputs(wl, "cuda")
    out = run(wl, inp)
    rows = sample_rows(wl, np.random.default_rng(n), extra=2048 if n > 32768 else 4096)
    check(wl, out, oracle.wl_fwd(wl, inp, rows=rows), rows=rows)
    del inp, out
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- random small patterns
SMALL = []
for n, d, w, dil, causal, G, pad in itertools.product(
        [1, 7, 127, 128, 129, 300, 1000], [64, 128], [0, 2, 6, 64, 256, 2000], [(1,), (1, 3)],
        [False, True], [0, 1, 5, 130], [False, True]):
    SMALL.append((n, d, w, dil, causal, G, pad))
SMALL = [c for t, c in enumerate(SMALL) if t % 23 == 0]


def _small_wl(n, d, w, dil, causal, G, pad, dtype):
    rng = np.random.default_rng(zlib.crc32(repr((n, d, w, dil, causal, G, pad, dtype)).encode()))
    G = min(G, n)
    gidx = sorted(rng.choice(n, size=G, replace=False).tolist()) if G else []
    B = 2
    pads = [0, int(rng.integers(0, n + 1))] if pad else None
    return workloads.custom("small", dtype, B, len(dil), n, d, w, dil, causal, gidx, pads,
                            seed=int(rng.integers(0, 2**31)))


@pytest.mark.parametrize("n,d,w,dil,causal,G,pad", SMALL)
def test_bf16_small_patterns(n, d, w, dil, causal, G, pad):
    wl = _small_wl(n, d, w, dil, causal, G, pad, "bf16")
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


@pytest.mark.parametrize("n,d,w,dil,causal,G,pad",
                         [(n, dd, w, dil, c, G, p) for (n, _, w, dil, c, G, p), dd in
                          zip(SMALL, itertools.cycle([1, 17, 64, 128]))])
def test_f32_small_patterns(n, d, w, dil, causal, G, pad):
    wl = _small_wl(n, d, w, dil, causal, G, pad, "f32")
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


@pytest.mark.parametrize("dil", [(2,), (4,), (7,), (1, 2, 3, 4, 5, 6, 7, 8, 9)])
def test_bf16_many_residue_classes(dil):
    """More (dilation, residue) classes than one launch holds are split across launches."""
    wl = workloads.custom("dil", "bf16", 1, len(dil), 777, 64, 16, dil, False, (5, 400), None, seed=3)
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_global_rows_on_band_kernel(causal):
    """d = 64 with many global tokens: their rows run through the band kernel's
    global-row mode (queries from qg, keys kg/vg over the row's valid length).
    Two query tiles of global tokens, some of them in a padded region."""
    gidx = tuple(sorted(set(range(0, 600, 4)) | {599}))  # 151 tokens
    wl = workloads.custom("gband", "bf16", 2, 3, 600, 64, 64, (1, 2, 3), causal, gidx, (0, 170), seed=21)
    inp = workloads.make_inputs(wl, "cuda")
    out = run(wl, inp)
    check(wl, out, oracle.wl_fwd(wl, inp))
    assert torch.all(out[1, :, 600 - 170:] == 0)


def test_bf16_more_globals_than_shared_memory_holds():
    """1100 global tokens: the band kernels keep the first 1024 positions in
    shared memory and read the rest from the kernel parameters; both the
    global key columns of the band rows and the global rows (global-row mode
    at d = 64) cross that boundary."""
    gidx = tuple(range(0, 2200, 2))
    wl = workloads.custom("g1100", "bf16", 1, 1, 2200, 64, 64, (1,), False, gidx, None, seed=23)
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("G,w", [(1, 64), (2, 64), (4, 64), (5, 64), (4, 2000), (3, 6)])
def test_bf16_few_globals_on_ring(G, w, causal):
    """d = 64 with one to five global tokens (the ring kernel's gathered key
    entry holding a few columns).  The tokens sit at the start, inside, near
    the end and in batch row 1's padding; dilated heads put some of them
    outside a row's residue class, w = 2000 puts every one inside every band,
    and causal rows before a token must not see it."""
    gidx = (0, 301, 702, 850, 999)[:G]
    wl = workloads.custom("fold", "bf16", 2, 3, 1000, 64, w, (1, 2, 3), causal, gidx, (0, 230), seed=40 + G)
    inp = workloads.make_inputs(wl, "cuda")
    out = run(wl, inp)
    assert lf.last_band_kernel() == "band_ring"
    check(wl, out, oracle.wl_fwd(wl, inp))


@pytest.mark.parametrize("d,G,causal", [(64, 0, False), (64, 1, True), (64, 20, False), (128, 1, False),
                                         (128, 0, True)])
def test_bf16_per_head_windows(d, G, causal):
    """A window per head (section 4.1 "Attention Pattern"): one launch, each
    tile reading its head's reach from its segment.  d = 64 runs the ring
    kernel even with G = 20 (the duo kernel keeps one window per launch),
    d = 128 the pair kernel."""
    wh = [512, 64, 0, 64, 2000, 512]
    dil = [1, 1, 2, 3, 1, 2]
    gidx = tuple(range(0, 900, 45))[:G]
    wl = workloads.custom("hw", "bf16", 2, 6, 900, d, wh, dil, causal, gidx, (0, 250), seed=50 + d + G)
    inp = workloads.make_inputs(wl, "cuda")
    out = run(wl, inp)
    assert lf.last_band_kernel() == ("band_pair" if d == 128 else "band_ring")
    check(wl, out, oracle.wl_fwd(wl, inp))


@pytest.mark.parametrize("causal", [False, True])
def test_f32_per_head_windows(causal):
    wl = workloads.custom("hw32", "f32", 2, 4, 500, 40, [6, 100, 0, 1200], (1, 2, 1, 3), causal, (0, 250),
                          (0, 90), seed=60)
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


def test_bf16_many_globals():
    wl = workloads.custom("glob", "bf16", 1, 2, 1500, 64, 32, (1, 2), False, tuple(range(0, 1500, 5)),
                          (0,), seed=4)
    inp = workloads.make_inputs(wl, "cuda")
    check(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


# ---------------------------------------------------------------- properties
def test_w0_returns_values_exactly():
    wl = workloads.custom("w0", "bf16", 2, 3, 700, 64, 0, (1, 2, 3), False, (), None, seed=5)
    inp = workloads.make_inputs(wl, "cuda")
    assert torch.equal(run(wl, inp), inp.v)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_constant_values_give_constant_rows(dtype):
    wl = workloads.custom("c", dtype, 1, 2, 900, 64, 64, (1, 3), True, (0, 450), (0,), seed=6)
    inp = workloads.make_inputs(wl, "cuda")
    c = torch.randn(wl.d, device="cuda").to(wl.torch_dtype)
    inp.v = c.expand_as(inp.v).contiguous()
    inp.vg = c.expand_as(inp.vg).contiguous()
    out = run(wl, inp).float()
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert torch.allclose(out, c.float().expand_as(out), atol=tol, rtol=0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_every_output_element_is_written(dtype):
    wl = workloads.custom("nan", dtype, 2, 2, 600, 64, 40, (1, 2), False, (3, 300), (0, 150), seed=7)
    inp = workloads.make_inputs(wl, "cuda")
    out = torch.full_like(inp.q, float("nan"))
    run(wl, inp, out=out)
    assert not torch.isnan(out).any()


def test_run_to_run_bitwise_determinism():
    wl = workloads.bf16_qa_padded()
    inp = workloads.make_inputs(wl, "cuda")
    a = run(wl, inp).clone()
    b = run(wl, inp)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_padding_poison_leaves_valid_rows_unchanged(dtype):
    n = 1024
    wl = workloads.custom("pad", dtype, 2, 2, n, 64, 64, (1, 2), False, (0, 700, 900), (0, 300), seed=8)
    inp = workloads.make_inputs(wl, "cuda")
    base = run(wl, inp).clone()
    for t in (inp.q, inp.k, inp.v, inp.kg, inp.vg):
        t[1, :, n - 300:] = float("nan")
    out = run(wl, inp)
    assert torch.equal(out, base)
    assert torch.all(out[1, :, n - 300:] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_causal_rows_ignore_later_tiles(dtype):
    """Causal rows before a tile boundary P0 (a multiple of 128 times every
    dilation) read no key at or after P0: NaN there changes nothing before it."""
    n, P0 = 2048, 1536
    wl = workloads.custom("causal", dtype, 1, 3, n, 64, 128, (1, 2, 4), True, (10, 1000, 1700), None,
                          seed=9)
    inp = workloads.make_inputs(wl, "cuda")
    base = run(wl, inp).clone()
    for t in (inp.q, inp.k, inp.v, inp.kg, inp.vg):
        t[:, :, P0:] = float("nan")
    out = run(wl, inp)
    assert torch.equal(out[:, :, :P0], base[:, :, :P0])


def test_keys_outside_every_window_of_a_tile_cannot_reach_it():
    """The band kernel computes 128 query rows at a time; a key outside the
    union of that tile's windows (and not global) must not affect those rows,
    whatever it holds."""
    n, w, t = 2048, 128, 6
    wl = workloads.custom("oow", "bf16", 1, 2, n, 64, w, (1, 1), False, (5,), None, seed=11)
    inp = workloads.make_inputs(wl, "cuda")
    base = run(wl, inp).clone()
    lo, hi = 128 * t - w // 2, 128 * t + 127 + w // 2
    outside = torch.ones(n, dtype=torch.bool, device="cuda")
    outside[lo:hi + 1] = False
    outside[5] = False
    for x in (inp.q, inp.k, inp.v):
        x[:, :, outside] = float("nan")
    out = run(wl, inp)
    assert torch.equal(out[:, :, 128 * t:128 * t + 128], base[:, :, 128 * t:128 * t + 128])


def test_full_window_equals_dense_attention():
    """w >= 2n, one head, no globals: ordinary attention (checked against
    torch's fp32 SDPA on the same bf16 values)."""
    wl = workloads.custom("full", "bf16", 1, 4, 640, 128, 2000, (1, 1, 1, 1), False, (), None, seed=10)
    inp = workloads.make_inputs(wl, "cuda")
    out = run(wl, inp).float()
    want = torch.nn.functional.scaled_dot_product_attention(inp.q.float(), inp.k.float(), inp.v.float())
    err = (out - want).abs()
    assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN


def test_invalid_call_leaves_out_untouched():
    q = torch.randn(1, 1, 256, 64, device="cuda", dtype=torch.bfloat16)
    out = torch.full_like(q, 7.0)
    with pytest.raises(lf.LfError) as e:
        lf.attn(q, q.clone(), q.clone(), w=3, out=out)  # odd window
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_runs_on_a_side_stream():
    wl = workloads.bf16_encoder()
    inp = workloads.make_inputs(wl, "cuda")
    ref = run(wl, inp).clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, qg=inp.qg, kg=inp.kg,
                      vg=inp.vg, global_idx=wl.global_idx)
    s.synchronize()
    assert torch.equal(out, ref)


def test_no_device_error_after_suite():
    assert lf.device_error() == 0
