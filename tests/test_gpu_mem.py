"""GPU parity of the memory combine (lf_mem_combine through the C ABI)
against the fp64 oracle (oracle.mem_combine) on the same seeded inputs.

Tolerance: bf16 inputs and output, fp32 arithmetic: |err| <= 8e-3 * |want|
+ 2e-3 (the output's rounding is at most 2^-9 relative).
"""
import numpy as np
import pytest
import torch

import long_sequence_sliding_longformer_b300 as lf
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_sequence_sliding_longformer_b300 import _build
    _build.build()
    lf.load()
    assert lf.device_error(clear=True) == 0


def draw(B, H, n, d, M, km, seed, empty=0.1):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(B, H, n, d, generator=g).to(torch.bfloat16)
    local = torch.randn(B, H, n, d, generator=g).to(torch.bfloat16)
    mk = torch.randn(B, H, M, d, generator=g).to(torch.bfloat16)
    mv = torch.randn(B, H, M, d, generator=g).to(torch.bfloat16)
    idx = torch.randint(0, max(M, 1), (B, H, n, km), generator=g, dtype=torch.int32)
    idx[torch.rand(B, H, n, km, generator=g) < empty] = -1
    if M == 0:
        idx[:] = -1
    gate = torch.rand(H, generator=g)
    return [t.cuda() for t in (q, local, mk, mv, idx, gate)]


def check(got, want):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    err = np.abs(g - want)
    assert np.all(err <= 8e-3 * np.abs(want) + 2e-3), err.max()


@pytest.mark.parametrize("case", [(2, 3, 200, 64, 500, 32), (1, 2, 333, 128, 1000, 7), (3, 1, 64, 64, 40, 1),
                                  (1, 4, 100, 128, 3000, 32)], ids=str)
def test_memory_combine_matches_oracle(case):
    B, H, n, d, M, km = case
    q, local, mk, mv, idx, gate = draw(B, H, n, d, M, km, seed=sum(case))
    out = lf.mem_combine(q, local, mk, mv, idx, gate)
    torch.cuda.synchronize()
    check(out, oracle.mem_combine(q, local, mk, mv, idx, gate))
    assert lf.device_error() == 0


def test_memory_combine_in_place_and_empty_rows():
    q, local, mk, mv, idx, gate = draw(1, 2, 150, 64, 300, 32, seed=21)
    idx[0, 1, 7] = -1  # a query with no retrieved pair
    want = oracle.mem_combine(q, local, mk, mv, idx, gate)
    out = lf.mem_combine(q, local, mk, mv, idx, gate, out=local)
    torch.cuda.synchronize()
    assert out.data_ptr() == local.data_ptr()
    check(out, want)


def test_memory_combine_without_memory():
    q, local, _, _, idx, gate = draw(1, 2, 50, 64, 0, 4, seed=22)
    mk = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    out = lf.mem_combine(q, local, mk, mk.clone(), idx, gate)
    torch.cuda.synchronize()
    want = (1.0 - gate.double().cpu().numpy())[None, :, None, None] * local.double().cpu().numpy()
    check(out, want)


def test_memory_index_out_of_range_is_reported_and_skipped():
    """The kernel checks each index before reading: an out-of-range one is an
    empty slot and sets the device error word (no access outside the memory)."""
    q, local, mk, mv, idx, gate = draw(1, 1, 64, 64, 100, 8, seed=23, empty=0.0)
    idx[0, 0, 5, 3] = 100
    idx[0, 0, 9, 0] = -7
    out = lf.mem_combine(q, local, mk, mv, idx, gate)
    code = lf.device_error(clear=True)
    assert code == 1 | (7 << 8)
    fixed = idx.clone()
    fixed[0, 0, 5, 3] = -1
    fixed[0, 0, 9, 0] = -1
    check(out, oracle.mem_combine(q, local, mk, mv, fixed, gate))
    assert lf.device_error() == 0


def test_memory_combine_char_lm_shape_sampled():
    """The char-LM pattern's shape (B1 H8 n23040 d64) with 32 retrieved pairs
    from a 65536-entry memory per head, checked on every row."""
    q, local, mk, mv, idx, gate = draw(1, 8, 23040, 64, 65536, 32, seed=24, empty=0.0)
    out = lf.mem_combine(q, local, mk, mv, idx, gate)
    torch.cuda.synchronize()
    check(out, oracle.mem_combine(q, local, mk, mv, idx, gate))


def test_memory_combine_is_bitwise_deterministic():
    q, local, mk, mv, idx, gate = draw(2, 4, 500, 128, 2000, 32, seed=25)
    a = lf.mem_combine(q, local, mk, mv, idx, gate).clone()
    assert torch.equal(lf.mem_combine(q, local, mk, mv, idx, gate), a)
