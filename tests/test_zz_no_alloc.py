"""lf_attn_fwd_noalloc: the bf16 forward for callers that cannot allocate
device memory while they run (a memory budget fixed at start-up, no room for
an allocator failure mid-step, or a host that owns the allocator).  Its
global-row scratch is a fixed array inside the library instead of a
per-call allocation.  Called here through the C ABI and compared with
lf_attn_fwd, which allocates.  Kept in its own file, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import long_sequence_sliding_longformer_b300 as lf
import workloads

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


def _fn():
    lib = lf.load()
    f = lib.lf_attn_fwd_noalloc
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [P, P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P]
    f.restype = ctypes.c_int
    return lib, f


def _i32(xs):
    return None if xs is None else (ctypes.c_int32 * max(len(xs), 1))(*xs)


def _call(f, wl, inp, out, stream):
    G = wl.G
    return f(inp.q.data_ptr(), inp.k.data_ptr(), inp.v.data_ptr(),
             inp.qg.data_ptr() if G else None, inp.kg.data_ptr() if G else None,
             inp.vg.data_ptr() if G else None, _i32(wl.global_idx) if G else None, G,
             out.data_ptr(), wl.B, wl.H, wl.n, wl.d, wl.w, _i32(wl.dilation), int(wl.causal),
             _i32(wl.pad_len), stream)


@pytest.mark.gpu
def test_no_alloc_matches_allocating_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib, f = _fn()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [workloads.bf16_qa_padded(), workloads.bf16_encoder()]
    for wl in cases:
        inp = workloads.make_inputs(wl, "cuda")
        ref = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                      pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx)
        torch.cuda.synchronize()
        for call in range(2):
            out = torch.full_like(inp.q, float("nan"))
            st = _call(f, wl, inp, out, stream)
            assert st == 0, lib.lf_last_error_message().decode()
            torch.cuda.synchronize()
            err = (out.float() - ref.float()).abs()
            assert torch.isfinite(out.float()).all(), (wl.name, call)
            assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN, (wl.name, call)
    assert lf.device_error() == 0


def test_no_alloc_rejects_scratch_beyond_its_array():
    """B*H*n_global*(d+2) fp32 values beyond 16 MiB are refused before any GPU work."""
    lib, f = _fn()
    wl = workloads.custom("big", "bf16", 16, 16, 8192, 128, 64, (1,) * 16, False, tuple(range(200)))
    fake = [0x100000 * (t + 1) << 12 for t in range(7)]  # aligned, never dereferenced
    st = f(fake[0], fake[1], fake[2], fake[3], fake[4], fake[5], _i32(wl.global_idx), wl.G, fake[6],
           wl.B, wl.H, wl.n, wl.d, wl.w, _i32(wl.dilation), 0, None, None)
    assert st == 2
    assert "static scratch" in lib.lf_last_error_message().decode()


@pytest.mark.gpu
def test_no_alloc_grows_key_chunks_to_fit_on_the_d128_streaming_path():
    """d = 128 takes the CUDA-core streaming pass for the global rows.  With
    n = 200 the occupancy rule leaves 128-key chunks (two per row); 1500
    (b, h) planes x 15 global tokens then need 23.4 MB of partial states, more
    than the 16 MiB array, and the chunk grows to the whole row (11.7 MB)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib, f = _fn()
    stream = torch.cuda.current_stream().cuda_stream
    wl = workloads.custom("grow", "bf16", 6, 250, 200, 128, 32, (1,) * 250, False,
                          tuple(range(0, 200, 14))[:15], None, seed=41)
    assert wl.G == 15
    inp = workloads.make_inputs(wl, "cuda")
    ref = lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                  pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx)
    out = torch.full_like(inp.q, float("nan"))
    st = _call(f, wl, inp, out, stream)
    assert st == 0, lib.lf_last_error_message().decode()
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    err = (out.float() - ref.float()).abs()
    assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN
    # the global tokens' rows against the oracle, row by row
    import oracle
    rows = np.array([(b * wl.H + h) * wl.n + g for b in (0, 5) for h in (0, 123, 249) for g in wl.global_idx])
    want = oracle.wl_fwd(wl, inp, rows=rows)
    got = out.float().cpu().numpy().reshape(-1, wl.d)[rows].astype(np.float64)
    assert np.abs(got - want).max() <= BF16_MAX
    assert lf.device_error() == 0
