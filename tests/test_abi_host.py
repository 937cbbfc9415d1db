"""The C-ABI library on the host (no GPU): it builds, loads, exports every
symbol include/lf_attn.h declares, rejects invalid arguments before touching
the device, and counts the pattern's useful work exactly."""
import ctypes
import os
import re

import numpy as np
import pytest

import long_sequence_sliding_longformer_b300 as lf
from long_sequence_sliding_longformer_b300 import _build
import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lf_attn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return lf.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lf_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("lf_attn_fwd", "lf_attn_fwd_f32", "lf_status_string", "lf_last_error_message"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["LF_OK", "LF_ERR_INVALID_ARG", "LF_ERR_UNSUPPORTED", "LF_ERR_CUDA",
                                 "LF_ERR_NO_MEMORY", "LF_ERR_TIMEOUT"]):
        assert lib.lf_status_string(code).decode() == name
    assert lib.lf_status_string(99).decode() == "LF_ERR_UNKNOWN"


def _arr(xs):
    return (ctypes.c_int32 * max(len(xs), 1))(*xs)


FAKE = 0x10000  # an aligned address that is never dereferenced: validation rejects first


def _call(lib, fn="lf_attn_fwd", *, q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, qg=None, kg=None,
          vg=None, gidx=None, G=0, out=FAKE + 0x300000, B=1, H=1, n=64, d=64, w=8, dil=(1,),
          causal=0, pad=None):
    f = getattr(lib, fn)
    return f(q, k, v, qg, kg, vg, _arr(gidx) if gidx is not None else None, G, out, B, H, n, d, w,
             _arr(dil) if dil is not None else None, causal, _arr(pad) if pad is not None else None, None)


INVALID = [
    dict(w=7),                       # odd window
    dict(w=-2),
    dict(B=-1),
    dict(n=-5),
    dict(d=0),
    dict(causal=2),
    dict(dil=(0,)),
    dict(dil=None),
    dict(q=None),
    dict(out=None),
    dict(q=FAKE + 8),                # misaligned
    dict(out=FAKE),                  # aliases q
    dict(pad=(65,)),                 # pad > n
    dict(pad=(-1,)),
    dict(G=2, gidx=None, qg=FAKE + 0x400000, kg=FAKE + 0x500000, vg=FAKE + 0x600000),
    dict(G=2, gidx=(3, 3), qg=FAKE + 0x400000, kg=FAKE + 0x500000, vg=FAKE + 0x600000),
    dict(G=2, gidx=(5, 2), qg=FAKE + 0x400000, kg=FAKE + 0x500000, vg=FAKE + 0x600000),
    dict(G=1, gidx=(64,), qg=FAKE + 0x400000, kg=FAKE + 0x500000, vg=FAKE + 0x600000),
    dict(G=1, gidx=(0,), qg=None, kg=FAKE + 0x500000, vg=FAKE + 0x600000),
    dict(G=-1),
]


@pytest.mark.parametrize("kw", INVALID, ids=[str(k) for k in INVALID])
@pytest.mark.parametrize("fn", ["lf_attn_fwd", "lf_attn_fwd_f32"])
def test_invalid_arguments_are_rejected_on_the_host(lib, fn, kw):
    assert _call(lib, fn, **kw) == 1
    assert lib.lf_last_error_message().decode() != ""


@pytest.mark.parametrize("kw", [dict(d=32), dict(d=96), dict(d=256)])
def test_bf16_head_dims_outside_64_128_are_unsupported(lib, kw):
    assert _call(lib, "lf_attn_fwd", **kw) == 2


def test_fp32_head_dim_limit(lib):
    assert _call(lib, "lf_attn_fwd_f32", d=129) == 2


def test_too_many_globals_unsupported(lib):
    g = list(range(4097))
    assert _call(lib, n=5000, G=4097, gidx=g, qg=FAKE + 0x4000000, kg=FAKE + 0x8000000,
                 vg=FAKE + 0xC000000, q=FAKE, k=FAKE + 0x1000000, v=FAKE + 0x2000000,
                 out=FAKE + 0x3000000) == 2


def test_empty_problems_are_no_ops(lib):
    for kw in (dict(B=0), dict(H=0, dil=()), dict(n=0)):
        assert _call(lib, **kw) == 0


def _oracle_pairs(B, H, n, w, dil, causal, pad, gidx):
    tot = 0
    for b in range(B):
        for h in range(H):
            for i in range(n):
                keys, _ = oracle.attended(n=n, w=w, dilation=dil, causal=causal, global_idx=gidx,
                                          pad_len=pad, b=b, h=h, i=i, B=B)
                tot += len(keys)
    return tot


@pytest.mark.parametrize("B,H,n,w,dil,causal,pad,gidx", [
    (1, 1, 64, 8, [1], False, None, []),
    (2, 2, 100, 10, [1, 3], True, [0, 17], [0, 50]),
    (1, 3, 37, 0, [1, 2, 5], False, [4], [1, 2, 36]),
    (2, 1, 50, 200, [2], False, [0, 49], [7]),
    (1, 2, 90, 12, [4, 1], True, None, list(range(0, 90, 9))),
])
def test_pair_count_matches_oracle_sets(lib, B, H, n, w, dil, causal, pad, gidx):
    pairs, flops = lf.count_pairs(B=B, H=H, n=n, d=8, w=w, dilation=dil, causal=causal, pad_len=pad,
                                  global_idx=gidx)
    assert pairs == _oracle_pairs(B, H, n, w, dil, causal, pad, gidx)
    assert flops == 4 * 8 * pairs


def test_pair_count_of_named_workloads(lib):
    # the fp32 window-64 workload: 512 rows, interior rows attend 65 keys
    wl = workloads.fp32_window64()
    pairs, _ = lf.count_pairs(B=wl.B, H=wl.H, n=wl.n, d=wl.d, w=wl.w, dilation=wl.dilation)
    assert pairs == 512 * 65 - 2 * sum(32 - t for t in range(32))
    # the causal char-LM workload: look-back 256 on every residue class
    wl = workloads.bf16_charlm()
    pairs, _ = lf.count_pairs(B=wl.B, H=wl.H, n=wl.n, d=wl.d, w=wl.w, dilation=wl.dilation,
                              causal=True)
    want = 0
    for delta in wl.dilation:
        for r in range(delta):
            n_r = len(range(r, wl.n, delta))
            want += sum(min(m, 256) + 1 for m in range(n_r))
    assert pairs == want


@pytest.mark.parametrize("B,H,n,w,dil,causal,pad,gidx", [
    (2, 2, 100, 10, [1, 3], True, [0, 17], [0, 50]),
    (1, 3, 37, 0, [1, 2, 5], False, [4], [1, 2, 36]),
    (1, 2, 90, 12, [4, 1], True, None, list(range(0, 90, 9))),
])
def test_oracle_pattern_count_matches_row_sets(B, H, n, w, dil, causal, pad, gidx):
    # the oracle's whole-pattern count (the benchmark's reference arm counts
    # FLOPs with it) against the sum of its per-row attended sets
    pairs, gpairs = oracle.count_pairs(B=B, H=H, n=n, w=w, dilation=dil, causal=causal,
                                       global_idx=gidx, pad_len=pad)
    assert pairs == _oracle_pairs(B, H, n, w, dil, causal, pad, gidx)
    want_g = 0
    for b in range(B):
        L = n - (pad[b] if pad else 0)
        want_g += H * sum((g + 1 if causal else L) for g in gidx if g < L)
    assert gpairs == want_g


@pytest.mark.parametrize("wl", workloads.all_workloads(), ids=lambda wl: wl.name)
def test_pair_count_of_named_workloads_oracle_vs_library(lib, wl):
    # both benchmark arms count the same useful work, each without the other's code
    pairs, _ = oracle.wl_count_pairs(wl)
    lpairs, _ = lf.count_pairs(B=wl.B, H=wl.H, n=wl.n, d=wl.d, w=wl.w, dilation=wl.dilation,
                               causal=wl.causal, pad_len=wl.pad_len, global_idx=wl.global_idx)
    assert pairs == lpairs


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import importlib
    monkeypatch.setattr(lf, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(lf, "_lib", None)
    with pytest.raises(RuntimeError):
        lf.load()


# ---------------------------------------------------------------- new entry points: refused on the host
# (fake, 16-byte aligned pointers that are never dereferenced: each call must
# fail its validation before it touches the device)
_FAKE = [(0x100000 * (t + 1)) << 12 for t in range(16)]


def _i32p(xs):
    import ctypes
    return (ctypes.c_int32 * max(len(xs), 1))(*xs)


@pytest.mark.parametrize("K,n_out,H,d,status", [
    (96, 3, 2, 64, 2),    # K not a multiple of 64
    (128, 3, 2, 48, 2),   # d not a multiple of 32
    (128, 1, 1, 96, 2),   # n_out*H*d = 96, not a multiple of 128
    (128, 0, 2, 64, 1),   # no output
    (0, 3, 2, 64, 1),     # K < 1
])
def test_projection_sizes_refused_on_host(lib, K, n_out, H, d, status):
    st = lib.lf_proj_heads(_FAKE[0], _FAKE[1], None, _FAKE[2], 2, 100, K, n_out, H, d, None)
    assert st == status, lib.lf_last_error_message().decode()


def test_projection_misaligned_pointer_refused(lib):
    assert lib.lf_proj_heads(_FAKE[0] + 8, _FAKE[1], None, _FAKE[2], 2, 100, 128, 3, 2, 64, None) == 1
    assert "aligned" in lib.lf_last_error_message().decode()


@pytest.mark.parametrize("d,km,status", [(96, 32, 2), (64, 33, 2), (64, 0, 2)])
def test_memory_combine_sizes_refused_on_host(lib, d, km, status):
    st = lib.lf_mem_combine(_FAKE[0], _FAKE[1], _FAKE[2], _FAKE[3], _FAKE[4], _FAKE[5], _FAKE[6],
                            1, 2, 100, d, 1000, km, None)
    assert st == status, lib.lf_last_error_message().decode()


def test_memory_combine_out_overlapping_an_input_refused(lib):
    # out == local is allowed (in place); out overlapping q is not
    st = lib.lf_mem_combine(_FAKE[0], _FAKE[1], _FAKE[2], _FAKE[3], _FAKE[4], _FAKE[5], _FAKE[0] + 16,
                            1, 2, 100, 64, 1000, 32, None)
    assert st == 1
    assert "overlaps" in lib.lf_last_error_message().decode()


def _bwd_args(lib, d=64, w=8, G=0, gidx=None):
    import ctypes
    f = _FAKE
    return [f[0], f[1], f[2], f[3] if G else None, f[4] if G else None, f[5] if G else None,
            _i32p(gidx) if G else None, G, f[6], f[7], f[8], f[9], f[10] if G else None,
            f[11] if G else None, f[12] if G else None, 1, 2, 64, d, w, _i32p([1, 2]), 0, None, None]


def test_backward_refuses_bad_patterns_on_host(lib):
    assert lib.lf_attn_bwd(*_bwd_args(lib, w=7)) == 1            # odd window
    assert lib.lf_attn_bwd(*_bwd_args(lib, d=96)) == 2           # bf16 d = 96
    assert lib.lf_attn_bwd(*_bwd_args(lib, G=2, gidx=[5, 5])) == 1  # global list not increasing
    args = _bwd_args(lib)
    args[9] = _FAKE[0]  # dk overlapping q
    assert lib.lf_attn_bwd(*args) == 1
    assert "overlaps" in lib.lf_last_error_message().decode()


def test_varglobal_refuses_bad_offsets_on_host(lib):
    f = _FAKE
    # offsets must start at 0 and not decrease; a bad list in the last row is found first
    for offs, gidx in (([1, 1, 2], [3, 4]), ([0, 2, 1], [3, 4]), ([0, 1, 3], [3, 9, 9])):
        st = lib.lf_attn_fwd_varglobal(f[0], f[1], f[2], f[3], f[4], f[5], _i32p(offs), _i32p(gidx), f[6],
                                       2, 2, 64, 64, 8, _i32p([1, 1]), 0, None, None)
        assert st == 1, (offs, gidx)


@pytest.mark.parametrize("fn", ["lf_attn_fwd_hw", "lf_attn_fwd_hw_f32"])
def test_per_head_windows_refused_on_host(lib, fn):
    """A window per head: the list is required, and each entry must be even
    and >= 0 (the bad entry is named in the message)."""
    f = _FAKE
    call = lambda wh, H=2: getattr(lib, fn)(f[0], f[1], f[2], None, None, None, None, 0, f[6], 1, H, 64, 64,
                                           _i32p(wh) if wh is not None else None, _i32p([1] * H), 0, None,
                                           None)
    assert call(None) == 1
    assert "w_heads" in lib.lf_last_error_message().decode()
    assert call([8, 7]) == 1
    assert "w_heads[1]" in lib.lf_last_error_message().decode()
    assert call([8, -2]) == 1
    assert call(None, H=0) == 0  # no heads: nothing to do


def test_per_head_window_backward_refused_on_host(lib):
    args = _bwd_args(lib)
    args[19] = _i32p([4, 3])  # odd window of head 1
    assert lib.lf_attn_bwd_hw(*args) == 1
    assert "w_heads[1]" in lib.lf_last_error_message().decode()
    args[19] = None
    assert lib.lf_attn_bwd_hw(*args) == 1


def test_bias_entries_refused_on_host(lib):
    """The bias table is required; its gradient needs w <= 4096 and must not
    overlap the other gradients."""
    f = _FAKE
    fwd = lambda rb: lib.lf_attn_fwd_bias(f[0], f[1], f[2], None, None, None, None, 0, f[6], 1, 2, 64, 64, 8,
                                          _i32p([1, 1]), 0, None, rb, None)
    assert fwd(None) == 1
    assert "rel_bias" in lib.lf_last_error_message().decode()
    assert fwd(f[13] + 2) == 1  # misaligned table
    args = _bwd_args(lib)
    bwd = lambda rb, drb, w=8: lib.lf_attn_bwd_bias(*(args[:19] + [w] + args[20:-1] + [rb, drb, None]))
    assert bwd(None, None) == 1
    assert bwd(f[13], f[14], w=4098) == 2  # the bias gradient's window limit
    assert bwd(f[13], f[7]) == 1  # d_rel_bias overlaps dq
    assert "overlaps" in lib.lf_last_error_message().decode()
