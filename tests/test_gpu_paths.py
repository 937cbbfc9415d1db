"""GPU tests of paths the product takes besides the plain forward: run-to-run
bitwise determinism where the global rows go through the split-key partials
and their fixed-order merge, a batch larger than one launch takes, the
bounded-wait timeout path, and host-side fault injection.

Every failure here is made on the host or by a wait limit: no kernel is made
to fault, trap or hang.
"""
import numpy as np
import pytest
import torch

import long_sequence_sliding_longformer_b300 as lf
import oracle
import workloads

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
LF_ERR_TIMEOUT = 5
LF_ERR_NO_MEMORY = 4
LF_ERR_CUDA = 3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_sequence_sliding_longformer_b300 import _build
    _build.build()
    lf.load()
    assert lf.device_error(clear=True) == 0
    yield
    lf.set_wait_limit_ns(0)
    lf.device_error(clear=True)


def run(wl, inp, **kw):
    out = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                  pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, **kw)
    torch.cuda.synchronize()
    return out


def check_bf16(wl, got, want):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    err = np.abs(g - want)
    assert err.max() <= BF16_MAX, err.max()
    assert err.mean() <= BF16_MEAN, err.mean()


# ---------------------------------------------------------------- determinism
@pytest.mark.parametrize("wl", [workloads.bf16_encoder(), workloads.bf16_led(8192),
                                workloads.bf16_led(32768)], ids=lambda wl: wl.name)
def test_split_key_merge_is_bitwise_deterministic(wl):
    """The encoder and LED patterns (one global token) take the streaming
    global-row pass: per key chunk partial states, merged in a fixed order by
    the last CTA of each row.  Repeated calls give the same bits."""
    inp = workloads.make_inputs(wl, "cuda")
    a = run(wl, inp).clone()
    for _ in range(3):
        assert torch.equal(run(wl, inp), a)


# ---------------------------------------------------------------- batch split
def test_batch_beyond_one_launch_matches_oracle():
    """B = 260 exceeds the 256 batch rows one launch carries: the call is split
    on the host into launches of 256 and 4 rows."""
    wl = workloads.custom("b260", "bf16", 260, 1, 256, 64, 32, (1,), False, (0, 100), None, seed=21)
    inp = workloads.make_inputs(wl, "cuda")
    check_bf16(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


def test_batch_beyond_one_launch_padded_causal():
    pad = tuple((7 * b) % 200 for b in range(258))
    wl = workloads.custom("b258", "bf16", 258, 2, 256, 64, 64, (1, 2), True, (3,), pad, seed=22)
    inp = workloads.make_inputs(wl, "cuda")
    check_bf16(wl, run(wl, inp), oracle.wl_fwd(wl, inp))


# ---------------------------------------------------------------- timeout path
@pytest.mark.parametrize("wl,kernel", [
    (workloads.custom("to_ring", "bf16", 1, 4, 2048, 64, 128, (1, 1, 2, 4), False, (), None, seed=23),
     "band_ring"),
    (workloads.custom("to_duo", "bf16", 1, 4, 2048, 64, 128, (1,) * 4, False, tuple(range(0, 1600, 100)), None,
                      seed=24),
     "band_duo"),
    (workloads.custom("to_pair", "bf16", 1, 2, 2048, 128, 256, (1, 1), False, (), None, seed=25),
     "band_pair"),
], ids=lambda x: getattr(x, "name", x))
def test_wait_limit_reports_timeout_then_recovers(wl, kernel):
    """With a pipeline-wait limit of 1 ns every wait that is not satisfied at
    once gives up: the kernel records LF_ERR_TIMEOUT in the device error word,
    drains its copies and MMAs (drain waits keep their own limit) and returns.
    The context stays usable: with the default limit restored and the word
    cleared, the same call matches the oracle."""
    inp = workloads.make_inputs(wl, "cuda")
    assert lf.device_error(clear=True) == 0
    lf.set_wait_limit_ns(1)
    try:
        run(wl, inp)
        code = lf.device_error()
    finally:
        lf.set_wait_limit_ns(0)
    assert lf.last_band_kernel() == kernel
    assert code & 0xFF == LF_ERR_TIMEOUT, hex(code)
    assert lf.device_error(clear=True) == code
    assert lf.device_error() == 0
    out = run(wl, inp)
    assert lf.device_error() == 0
    check_bf16(wl, out, oracle.wl_fwd(wl, inp))


# ---------------------------------------------------------------- fault injection
@pytest.mark.parametrize("fault,status", [("alloc", LF_ERR_NO_MEMORY), ("launch", LF_ERR_CUDA)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_injected_host_fault_leaves_out_untouched(monkeypatch, fault, status, dtype):
    """LF_FAULT=alloc|launch makes the call fail at its scratch allocation or
    its first launch; the status says which, and `out` keeps its contents."""
    wl = workloads.custom("fault", dtype, 1, 2, 512, 64, 64, (1, 2), False, (0,), None, seed=26)
    inp = workloads.make_inputs(wl, "cuda")
    out = torch.full_like(inp.q, 7.0)
    monkeypatch.setenv("LF_FAULT", fault)
    with pytest.raises(lf.LfError) as ei:
        run(wl, inp, out=out)
    assert ei.value.status == status
    assert torch.all(out == 7.0)
    monkeypatch.delenv("LF_FAULT")
    run(wl, inp, out=out)
    want = oracle.wl_fwd(wl, inp)
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.abs(g - want).max() <= (BF16_MAX if dtype == "bf16" else 1e-4)
    assert lf.device_error() == 0
