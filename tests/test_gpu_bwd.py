"""GPU parity of the backward (lf_attn_bwd / lf_attn_bwd_f32 through the C
ABI) against the fp64 oracle gradient on the same seeded inputs.

Tolerance: the kernels compute in fp32 from the same input values as the
oracle (no bf16 rounding inside, unlike the forward's P), so the error is
fp32 accumulation only: max |err| <= 2e-4 * max(1, max |grad|) per tensor.
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


def dout_for(wl, seed=1):
    g = torch.Generator(device="cpu").manual_seed(1000 + seed)
    return torch.randn((wl.B, wl.H, wl.n, wl.d), generator=g).to(wl.torch_dtype).cuda()


def run_bwd(wl, inp, dout):
    g = lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                    pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx)
    torch.cuda.synchronize()
    return g


def check_grads(got, want):
    assert set(got) == set(want)
    for name, w in want.items():
        gv = got[name].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(gv)), name
        err = np.abs(gv - w).max()
        assert err <= REL * max(1.0, np.abs(w).max()), (name, err, np.abs(w).max())


CASES = [
    # name, dtype, B, H, n, d, w, dilation, causal, global_idx, pad_len
    ("bf16_d64_plain", "bf16", 1, 2, 300, 64, 32, (1, 1), False, (), None),
    ("bf16_d64_dil_pad_g", "bf16", 2, 3, 513, 64, 64, (1, 2, 5), False, (0, 77, 400), (0, 100)),
    ("bf16_d64_causal_g", "bf16", 2, 2, 700, 64, 128, (1, 3), True, (5, 300, 650), (30, 0)),
    ("bf16_d128_g", "bf16", 1, 2, 640, 128, 256, (1, 2), False, (0,), None),
    ("bf16_d128_causal", "bf16", 2, 1, 400, 128, 64, (2,), True, (), (0, 57)),
    ("bf16_d64_many_g", "bf16", 1, 2, 512, 64, 64, (1, 1), False, tuple(range(0, 512, 8)), None),
    ("bf16_d64_w0", "bf16", 1, 2, 200, 64, 0, (1, 2), False, (3,), None),
    ("f32_d64", "f32", 1, 2, 512, 64, 64, (1, 2), False, (0, 200), (0,)),
    ("f32_d40_causal", "f32", 2, 2, 333, 40, 30, (1, 4), True, (11,), (7, 0)),
    ("f32_d128_g", "f32", 1, 1, 300, 128, 100, (3,), False, (0, 1, 2), None),
    ("f32_d7", "f32", 1, 3, 97, 7, 10, (1, 2, 3), True, (), None),
    # a window per head (section 4.1 "Attention Pattern")
    ("bf16_d64_heads_w", "bf16", 2, 3, 400, 64, [16, 128, 0], (1, 2, 1), False, (0, 150), (0, 60)),
    ("bf16_d128_heads_w", "bf16", 1, 2, 500, 128, [64, 256], (1, 1), True, (3,), None),
    ("f32_d48_heads_w", "f32", 1, 3, 300, 48, [64, 8, 200], (2, 1, 1), True, (7,), None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(case):
    name, dtype, B, H, n, d, w, dil, causal, gidx, pad = case
    wl = workloads.custom(name, dtype, B, H, n, d, w, dil, causal, gidx, pad, seed=31)
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl)
    check_grads(run_bwd(wl, inp, dout), oracle.wl_bwd(wl, inp, dout))


@pytest.mark.parametrize("wl", [workloads.fp32_window64(), workloads.bf16_encoder(),
                                workloads.bf16_charlm(), workloads.bf16_qa_padded(),
                                workloads.bf16_led(8192)], ids=lambda wl: wl.name)
def test_backward_named_workloads_full(wl):
    """Every gradient element of the benchmark patterns (LED at n = 8192)."""
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl, 2)
    check_grads(run_bwd(wl, inp, dout), oracle.wl_bwd(wl, inp, dout))


def test_backward_is_bitwise_deterministic():
    wl = workloads.bf16_qa_padded()
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl, 3)
    a = {k: t.clone() for k, t in run_bwd(wl, inp, dout).items()}
    for _ in range(2):
        b = run_bwd(wl, inp, dout)
        for k in a:
            assert torch.equal(a[k], b[k]), k


def test_backward_batch_beyond_one_launch():
    """B = 258 and H = 260 split into blocks of 256 batch rows and 256 heads."""
    wl = workloads.custom("split", "bf16", 258, 1, 128, 64, 16, (1,), False, (0,), None, seed=32)
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl, 4)
    check_grads(run_bwd(wl, inp, dout), oracle.wl_bwd(wl, inp, dout))
    wl = workloads.custom("splith", "f32", 1, 260, 64, 32, 8, tuple(1 + h % 3 for h in range(260)), True,
                          (), None, seed=33)
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl, 5)
    check_grads(run_bwd(wl, inp, dout), oracle.wl_bwd(wl, inp, dout))


def test_backward_padding_poison_leaves_valid_gradients_unchanged():
    """NaN in the padded tail of every input and of dout changes no gradient of
    a valid position, and the padded positions' gradients are zero."""
    n = 512
    wl = workloads.custom("pad", "bf16", 2, 2, n, 64, 64, (1, 2), False, (0, 300, 480), (0, 200), seed=34)
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl, 6)
    base = {k: t.clone() for k, t in run_bwd(wl, inp, dout).items()}
    for t in (inp.q, inp.k, inp.v, inp.kg, inp.vg, dout):
        t[1, :, n - 200:] = float("nan")
    got = run_bwd(wl, inp, dout)
    for k in ("dq", "dk", "dv", "dkg", "dvg"):
        assert torch.equal(got[k][1, :, : n - 200], base[k][1, :, : n - 200]), k
        assert torch.equal(got[k][0], base[k][0]), k
        assert torch.all(got[k][1, :, n - 200:] == 0), k
    # the global token at 480 lies in batch row 1's padding: its dqg row is zero there
    assert torch.all(got["dqg"][1, :, 2] == 0)
    assert torch.equal(got["dqg"][:, :, :2], base["dqg"][:, :, :2])


def test_backward_rejects_bad_arguments():
    wl = workloads.custom("bad", "bf16", 1, 1, 64, 64, 8, (1,), False, (), None, seed=35)
    inp = workloads.make_inputs(wl, "cuda")
    dout = dout_for(wl)
    with pytest.raises(lf.LfError):
        lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=7)  # odd window
    wl96 = workloads.custom("bad96", "bf16", 1, 1, 64, 96, 8, (1,), False, (), None, seed=36)
    inp96 = workloads.make_inputs(wl96, "cuda")
    with pytest.raises(lf.LfError):
        lf.attn_bwd(inp96.q, inp96.k, inp96.v, dout_for(wl96), w=8)  # bf16 d = 96
