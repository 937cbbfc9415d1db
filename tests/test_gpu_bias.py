"""GPU parity of the relative position bias (Memorizing Transformer notes,
"Position bias"): lf_attn_fwd_bias / lf_attn_bwd_bias and their fp32 forms
through the C ABI against the fp64 oracle on the same seeded inputs and the
same fp32 table.

Tolerances as for the plain calls: forward bf16 max |err| <= 2e-2 and mean
<= 2e-3, fp32 max <= 1e-4; backward (fp32 arithmetic throughout, the bias
gradient included) max |err| <= 2e-4 * max(1, max |grad|) per tensor.
"""
import numpy as np
import pytest
import torch

import long_sequence_sliding_longformer_b300 as lf
import oracle
import workloads

pytestmark = pytest.mark.gpu
REL = 2e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_sequence_sliding_longformer_b300 import _build
    _build.build()
    lf.load()
    assert lf.device_error(clear=True) == 0


CASES = [
    # name, dtype, B, H, n, d, w, dilation, causal, global_idx, pad_len, band kernel
    ("bf16_d64", "bf16", 2, 3, 700, 64, 64, (1, 2, 1), False, (0, 350), (0, 120), "band_ring"),
    ("bf16_d64_g20", "bf16", 1, 2, 900, 64, 128, (1, 1), False, tuple(range(0, 900, 45)), None, "band_ring"),
    ("bf16_d64_causal", "bf16", 2, 2, 600, 64, 512, (1, 3), True, (5,), (40, 0), "band_ring"),
    ("bf16_d128", "bf16", 1, 2, 800, 128, 256, (1, 2), False, (0,), None, "band_pair"),
    ("bf16_d128_causal", "bf16", 2, 1, 500, 128, 1024, (1,), True, (), (0, 77), "band_pair"),
    ("f32_d40", "f32", 2, 2, 300, 40, 30, (1, 2), False, (0, 150), (0, 50), "band_simt_f32"),
    ("f32_d64_causal", "f32", 1, 3, 257, 64, 100, (1, 1, 4), True, (3,), None, "band_simt_f32"),
]


def setup(case, seed=7):
    name, dtype, B, H, n, d, w, dil, causal, gidx, pad, kernel = case
    wl = workloads.custom(name, dtype, B, H, n, d, w, dil, causal, gidx, pad, seed=seed)
    inp = workloads.make_inputs(wl, "cuda")
    g = torch.Generator(device="cpu").manual_seed(seed + 100)
    table = (torch.randn(H, w + 1, generator=g) * 2).cuda()
    return wl, inp, table, kernel


def fwd(wl, inp, table):
    out = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal, pad_len=wl.pad_len,
                  qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, rel_bias=table)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forward_with_bias_matches_oracle(case):
    wl, inp, table, kernel = setup(case)
    out = fwd(wl, inp, table)
    assert lf.last_band_kernel() == kernel
    want = oracle.wl_fwd(wl, inp, rel_bias=table.cpu().numpy())
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - want)
    if wl.dtype == "f32":
        assert err.max() <= 1e-4, err.max()
    else:
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    # the bias matters: the same call without it is far from this output
    plain = oracle.wl_fwd(wl, inp)
    assert np.abs(plain - want).max() > 0.1


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_with_bias_matches_oracle(case):
    wl, inp, table, _ = setup(case, seed=8)
    g = torch.Generator(device="cpu").manual_seed(9)
    dout = torch.randn(wl.B, wl.H, wl.n, wl.d, generator=g).to(wl.torch_dtype).cuda()
    got = lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                      pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx,
                      rel_bias=table)
    torch.cuda.synchronize()
    want = oracle.wl_bwd(wl, inp, dout, rel_bias=table.cpu().numpy())
    assert set(got) == set(want)
    for name, wv in want.items():
        gv = got[name].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(gv)), name
        err = np.abs(gv - wv).max()
        assert err <= REL * max(1.0, np.abs(wv).max()), (name, err, np.abs(wv).max())


def test_bias_gradient_is_bitwise_reproducible():
    wl, inp, table, _ = setup(CASES[0], seed=10)
    dout = torch.randn(wl.B, wl.H, wl.n, wl.d, generator=torch.Generator().manual_seed(3)).to(wl.torch_dtype).cuda()
    kw = dict(w=wl.w, dilation=wl.dilation, causal=wl.causal, pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg,
              vg=inp.vg, global_idx=wl.global_idx, rel_bias=table)
    a = lf.attn_bwd(inp.q, inp.k, inp.v, dout, **kw)
    a = {k: v.clone() for k, v in a.items()}
    b = lf.attn_bwd(inp.q, inp.k, inp.v, dout, **kw)
    for name in a:
        assert torch.equal(a[name], b[name]), name


def test_zero_table_equals_the_plain_call():
    """A zero table changes no score: the bias kernels give the plain
    kernels' result (same tiles, same order of operations up to the scale
    folding, so equal within the bf16 rounding of P)."""
    wl, inp, _, _ = setup(CASES[3])
    zero = torch.zeros(wl.H, wl.w + 1, device="cuda")
    a = fwd(wl, inp, zero).float()
    b = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal, pad_len=wl.pad_len,
                qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx).float()
    torch.cuda.synchronize()
    assert (a - b).abs().max().item() <= 8e-3


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 32)])
def test_bias_across_the_batch_launch_split(dtype, d):
    """260 batch rows: the forward and backward run in blocks of 256 batch
    rows, and the bias gradient is summed over the blocks' launches."""
    B, H, n, w = 260, 2, 80, 16
    wl = workloads.custom("bias_b260", dtype, B, H, n, d, w, (1, 2), False, (3,), None, seed=12)
    inp = workloads.make_inputs(wl, "cuda")
    table = (torch.randn(H, w + 1, generator=torch.Generator().manual_seed(13)) * 2).cuda()
    out = fwd(wl, inp, table)
    want = oracle.wl_fwd(wl, inp, rel_bias=table.cpu().numpy())
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - want)
    assert err.max() <= (1e-4 if dtype == "f32" else 2e-2), err.max()
    dout = torch.randn(B, H, n, d, generator=torch.Generator().manual_seed(14)).to(wl.torch_dtype).cuda()
    got = lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=w, dilation=wl.dilation, qg=inp.qg, kg=inp.kg, vg=inp.vg,
                      global_idx=wl.global_idx, rel_bias=table)
    torch.cuda.synchronize()
    wg = oracle.wl_bwd(wl, inp, dout, rel_bias=table.cpu().numpy())
    for name, wv in wg.items():
        e = np.abs(got[name].cpu().numpy().astype(np.float64) - wv).max()
        assert e <= REL * max(1.0, np.abs(wv).max()), (name, e)


def test_many_distinct_head_windows():
    """Twelve heads, nine distinct windows in one launch, dilations mixed."""
    wh = [0, 2, 6, 64, 130, 64, 512, 2, 1000, 6, 40, 512]
    dil = [1, 2, 1, 3, 1, 1, 2, 1, 1, 4, 1, 1]
    wl = workloads.custom("hw12", "bf16", 2, 12, 600, 64, wh, dil, False, (0, 300), (0, 70), seed=15)
    inp = workloads.make_inputs(wl, "cuda")
    out = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg,
                  vg=inp.vg, global_idx=wl.global_idx)
    torch.cuda.synchronize()
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - oracle.wl_fwd(wl, inp))
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
