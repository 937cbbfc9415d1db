"""GPU parity of the per-head projections (lf_proj_heads through the C ABI)
against the fp64 oracle (oracle.proj) on the same seeded inputs.

Tolerance: bf16 operands with fp32 accumulation and a bf16 output (round to
nearest even, relative error <= 2^-9): |err| <= 4e-3 * |y| + 1e-3.
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


def draw(B, n, K, N, seed, bias=False):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(B, n, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16)
    b = torch.randn(N, generator=g).float() if bias else None
    return x.cuda(), w.cuda(), (b.cuda() if b is not None else None)


def check(got, want):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    err = np.abs(g - want)
    bound = 4e-3 * np.abs(want) + 1e-3
    assert np.all(err <= bound), (err.max(), np.unravel_index(np.argmax(err - bound), err.shape))


CASES = [
    # B, n, K, n_out, H, d, bias
    (1, 200, 64, 3, 2, 64, False),     # N = 384: 128-wide column tiles, a ragged row tile
    (2, 300, 768, 3, 12, 64, True),    # the encoder's hidden size, ragged rows, bias
    (1, 129, 128, 1, 1, 128, False),   # one 128-column tile, 129 rows
    (1, 256, 2048, 5, 16, 128, True),  # the LED hidden size, q k v kg vg
    (3, 64, 192, 2, 3, 64, False),     # K = 3 x 64
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_n%d_K%d_o%d_H%d_d%d%s" % (c[:6] + ("_bias" if c[6] else "",)))
def test_projection_matches_oracle(case):
    B, n, K, n_out, H, d, bias = case
    x, w, b = draw(B, n, K, n_out * H * d, seed=sum(case[:6]), bias=bias)
    y = lf.proj_heads(x, w, H=H, d=d, bias=b)
    torch.cuda.synchronize()
    check(y, oracle.proj(x, w, H=H, d=d, bias=b))


def test_projection_full_size_sampled_rows():
    """The encoder's projection (B2 n4096, hidden 768, q k v) against the
    oracle on sampled tokens (first and last rows of each batch row and a
    random spread)."""
    B, n, H, d = 2, 4096, 12, 64
    K = H * d
    x, w, b = draw(B, n, K, 3 * K, seed=7, bias=True)
    y = lf.proj_heads(x, w, H=H, d=d, bias=b)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    sel = np.unique(np.concatenate([np.arange(64), np.arange(n - 64, n), rng.integers(0, n, 256)]))
    want = oracle.proj(x[:, sel], w, H=H, d=d, bias=b)
    check(y[:, :, :, sel], want)


def test_identity_weights_split_heads_exactly():
    B, n, H, d = 2, 333, 4, 64
    K = H * d
    g = torch.Generator(device="cpu").manual_seed(9)
    x = torch.randn(B, n, K, generator=g).to(torch.bfloat16).cuda()
    w = torch.cat([torch.eye(K), -torch.eye(K)]).to(torch.bfloat16).cuda()
    y = lf.proj_heads(x, w, H=H, d=d)
    torch.cuda.synchronize()
    heads = x.view(B, n, H, d).permute(0, 2, 1, 3)
    assert torch.equal(y[0], heads)
    assert torch.equal(y[1], -heads)


def test_projection_is_bitwise_deterministic():
    x, w, b = draw(2, 1000, 512, 3 * 8 * 64, seed=10, bias=True)
    a = lf.proj_heads(x, w, H=8, d=64, bias=b).clone()
    for _ in range(2):
        assert torch.equal(lf.proj_heads(x, w, H=8, d=64, bias=b), a)


def test_projection_feeds_the_band_kernel():
    """q, k, v, kg, vg from one call and qg from the global tokens' hidden
    states in a second, then the forward: the same as the forward on the
    oracle's projections rounded to bf16."""
    import workloads
    B, n, H, d, w_ = 1, 1024, 4, 64, 128
    K = H * d
    gidx = (0, 500)
    x, wq, _ = draw(B, n, K, 5 * K, seed=11)
    _, wg, _ = draw(1, 1, K, K, seed=12)
    y = lf.proj_heads(x, wq, H=H, d=d)
    xg = x[:, list(gidx)].contiguous()
    qg = lf.proj_heads(xg, wg, H=H, d=d)[0]
    q, k, v, kg, vg = (y[t].contiguous() for t in range(5))
    out = lf.attn(q, k, v, w=w_, qg=qg, kg=kg, vg=vg, global_idx=gidx)
    torch.cuda.synchronize()
    wl = workloads.custom("proj_fwd", "bf16", B, H, n, d, w_, (1,) * H, False, gidx, None, 0)
    inp = workloads.Inputs(q, k, v, qg, kg, vg)
    want = oracle.wl_fwd(wl, inp)
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - want)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_projection_rejects_unsupported_sizes():
    x, w, _ = draw(1, 10, 96, 128, seed=13)  # K not a multiple of 64
    with pytest.raises(lf.LfError):
        lf.proj_heads(x, w, H=2, d=64)
    x, w, _ = draw(1, 10, 64, 96, seed=14)  # d = 48
    with pytest.raises(lf.LfError):
        lf.proj_heads(x, w, H=2, d=48)
