"""GPU parity of global tokens that differ between batch rows
(lf_attn_fwd_varglobal / lf_attn_bwd_varglobal through the C ABI): each batch
row against the fp64 oracle run on that row alone with its own list."""
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


def draw(B, H, n, d, lists, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).cuda()
    total = sum(len(x) for x in lists)
    return t(B, H, n, d), t(B, H, n, d), t(B, H, n, d), t(total * H, d), t(B, H, n, d), t(B, H, n, d)


@pytest.mark.parametrize("d,causal", [(64, False), (64, True), (128, False)])
def test_per_row_global_lists_match_oracle(d, causal):
    B, H, n, w = 4, 3, 700, 64
    lists = [[0, 1, 2, 3, 4], [], [10, 400], list(range(0, 700, 20))]  # QA-like spans of different lengths
    pad = [0, 50, 100, 0]
    q, k, v, qg, kg, vg = draw(B, H, n, d, lists, seed=31 + d + causal)
    dil = [1, 2, 1]
    out = lf.attn_varglobal(q, k, v, w=w, global_idx=lists, qg=qg, kg=kg, vg=vg, dilation=dil, causal=causal,
                            pad_len=pad)
    dout = torch.randn(B, H, n, d, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    grads = lf.attn_bwd_varglobal(q, k, v, dout, w=w, global_idx=lists, qg=qg, kg=kg, vg=vg, dilation=dil,
                                  causal=causal, pad_len=pad)
    torch.cuda.synchronize()
    off = 0
    for b, lst in enumerate(lists):
        G = len(lst)
        qgb = qg[off * H:(off + G) * H].view(1, H, G, d) if G else None
        kw = dict(w=w, dilation=dil, causal=causal, pad_len=[pad[b]], global_idx=lst,
                  qg=qgb, kg=kg[b:b + 1] if G else None, vg=vg[b:b + 1] if G else None)
        want = oracle.fwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], **kw)
        err = np.abs(out[b:b + 1].float().cpu().numpy().astype(np.float64) - want)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (b, err.max())
        wg = oracle.bwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], dout[b:b + 1], **kw)
        got = {"dq": grads["dq"][b:b + 1], "dk": grads["dk"][b:b + 1], "dv": grads["dv"][b:b + 1]}
        if G:
            got.update(dqg=grads["dqg"][off * H:(off + G) * H].view(1, H, G, d), dkg=grads["dkg"][b:b + 1],
                       dvg=grads["dvg"][b:b + 1])
        else:
            assert torch.all(grads["dkg"][b] == 0) and torch.all(grads["dvg"][b] == 0)
        for name, wv in wg.items():
            e = np.abs(got[name].cpu().numpy().astype(np.float64) - wv).max()
            assert e <= 2e-4 * max(1.0, np.abs(wv).max()), (b, name, e)
        off += G


def test_per_row_lists_are_all_validated_first():
    """A bad list in the last row fails the call before anything runs."""
    B, H, n, d = 3, 2, 128, 64
    lists = [[0], [5, 6], [9, 9]]  # not strictly increasing
    q, k, v, qg, kg, vg = draw(B, H, n, d, lists, seed=40)
    out = torch.full_like(q, 7.0)
    with pytest.raises(lf.LfError):
        lf.attn_varglobal(q, k, v, w=16, global_idx=lists, qg=qg, kg=kg, vg=vg, out=out)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
