"""fp64 CPU oracle for Longformer-style attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it, and it loads nothing of theirs.

The arithmetic lives in ``lf_oracle.c`` (plain C, double precision, one loop
per output row); this module only builds it with gcc and marshals arrays.
See that file's header for the pattern definitions and the readings taken
where the pages (velog.io/@lainshower/Longformer, sections 3-1 and 4.1) are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lf_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblf_oracle.so")
_lib = None

_F64, _F32, _BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile lf_oracle.c into liblf_oracle.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.lf_oracle_fwd.argtypes = [ctypes.c_int, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P,
                                      P, i32, P, P, P, ctypes.c_int64, P, i32]
        lib.lf_oracle_fwd.restype = ctypes.c_int
        lib.lf_oracle_attended.argtypes = [P, i32, i32, i32, i32, i32, P, P, i32, P, i32, i32, i32, P, P]
        lib.lf_oracle_attended.restype = i32
        lib.lf_oracle_bwd.argtypes = [ctypes.c_int, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P,
                                      P, i32, P, P, P, P, P, P, P, P, P, i32]
        lib.lf_oracle_bwd.restype = ctypes.c_int
        lib.lf_oracle_proj.argtypes = [ctypes.c_int, P, P, P, i32, i32, i32, i32, i32, i32, P, i32]
        lib.lf_oracle_proj.restype = ctypes.c_int
        lib.lf_oracle_mem_combine.argtypes = [ctypes.c_int, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, i32]
        lib.lf_oracle_mem_combine.restype = ctypes.c_int
        lib.lf_oracle_count_pairs.argtypes = [P, i32, i32, i32, i32, i32, P, P, i32, P, P, P]
        lib.lf_oracle_count_pairs.restype = i32
        lib.lf_oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def _as_array(x):
    """-> (contiguous numpy array, dtype code).  bf16 torch tensors keep their bits."""
    if x is None:
        return None, None
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), _BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, _F64
    if x.dtype == np.float32:
        return x, _F32
    if x.dtype == np.uint16:
        return x, _BF16
    raise TypeError("oracle inputs must be float64, float32 or bf16, got %s" % x.dtype)


def _i32(seq) -> Optional[np.ndarray]:
    if seq is None:
        return None
    return np.ascontiguousarray(np.asarray(list(seq), dtype=np.int32))


def _ptr(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


def _bias_table(rel_bias, H: int, w0: int, wh) -> Optional[np.ndarray]:
    """The relative bias table as contiguous float32 [H, w + 1], or None."""
    if rel_bias is None:
        return None
    if wh is not None:
        raise ValueError("a relative bias takes one window for every head")
    try:
        import torch

        if isinstance(rel_bias, torch.Tensor):
            rel_bias = rel_bias.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    rb = np.ascontiguousarray(np.asarray(rel_bias, dtype=np.float32))
    if rb.shape != (H, w0 + 1):
        raise ValueError("rel_bias must be [H, w + 1] = [%d, %d], got %s" % (H, w0 + 1, rb.shape))
    return rb


def _window(w, H: int):
    """w: one window for every head, or one per head -> (scalar, per-head
    int32 array or None)."""
    if np.ndim(w) == 0:
        return int(w), None
    wh = _i32(w)
    if len(wh) != H:
        raise ValueError("w needs one entry per head (or a single int)")
    return 0, wh


def max_threads() -> int:
    return int(_load().lf_oracle_max_threads())


def fwd(q, k, v, *, w, dilation: Optional[Sequence[int]] = None, causal: bool = False,
        pad_len: Optional[Sequence[int]] = None, qg=None, kg=None, vg=None,
        global_idx: Sequence[int] = (), rows: Optional[Sequence[int]] = None,
        rel_bias=None, threads: int = 0) -> np.ndarray:
    """Attention output in float64.

    q, k, v, kg, vg: [B, H, n, d]; qg: [B, H, G, d] (row r belongs to
    global_idx[r]).  All inputs share one dtype (float64, float32 or bf16).
    rows: optional flat row ids ((b*H + h)*n + i); then the result is
    [len(rows), d] instead of [B, H, n, d].  w: the window of every head, or
    a sequence with the window of each head.  rel_bias: optional [H, w + 1]
    float32 table added to the band keys' scores (entry t + w/2 for window
    step t).
    """
    lib = _load()
    qa, code = _as_array(q)
    ka, kc = _as_array(k)
    va, vc = _as_array(v)
    if not (code == kc == vc):
        raise TypeError("q, k, v must share a dtype")
    B, H, n, d = qa.shape
    G = len(global_idx)
    qga = kga = vga = None
    if G:
        qga, c1 = _as_array(qg)
        kga, c2 = _as_array(kg)
        vga, c3 = _as_array(vg)
        if not (c1 == c2 == c3 == code):
            raise TypeError("qg, kg, vg must share q's dtype")
        if qga.shape != (B, H, G, d) or kga.shape != qa.shape or vga.shape != qa.shape:
            raise ValueError("global tensor shapes do not match")
    if ka.shape != qa.shape or va.shape != qa.shape:
        raise ValueError("q, k, v shapes differ")
    dil = _i32(dilation if dilation is not None else [1] * H)
    w0, wh = _window(w, H)
    if len(dil) != H:
        raise ValueError("dilation needs one entry per head")
    gidx = _i32(global_idx) if G else None
    pads = _i32(pad_len)
    rb = _bias_table(rel_bias, H, w0, wh)
    rws = None
    if rows is not None:
        rws = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.zeros((len(rws), d), dtype=np.float64)
    else:
        out = np.zeros((B, H, n, d), dtype=np.float64)
    rc = lib.lf_oracle_fwd(code, _ptr(qa), _ptr(ka), _ptr(va), _ptr(qga), _ptr(kga), _ptr(vga),
                           _ptr(gidx), G, B, H, n, d, w0, _ptr(wh), _ptr(dil), int(bool(causal)),
                           _ptr(pads), _ptr(rb), _ptr(rws), 0 if rws is None else len(rws), _ptr(out),
                           int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the problem (code %d)" % rc)
    return out


def bwd(q, k, v, dout, *, w, dilation: Optional[Sequence[int]] = None, causal: bool = False,
        pad_len: Optional[Sequence[int]] = None, qg=None, kg=None, vg=None,
        global_idx: Sequence[int] = (), rel_bias=None, threads: int = 0) -> dict:
    """Gradients of sum(dout * out) in float64: a dict with dq, dk, dv and,
    when there are global tokens, dqg, dkg, dvg (each the shape of its input),
    and with rel_bias its gradient drel_bias [H, w + 1].  dout has out's shape
    and the inputs' dtype."""
    lib = _load()
    qa, code = _as_array(q)
    ka, kc = _as_array(k)
    va, vc = _as_array(v)
    da, dc = _as_array(dout)
    if not (code == kc == vc == dc):
        raise TypeError("q, k, v, dout must share a dtype")
    B, H, n, d = qa.shape
    if ka.shape != qa.shape or va.shape != qa.shape or da.shape != qa.shape:
        raise ValueError("q, k, v, dout shapes differ")
    G = len(global_idx)
    qga = kga = vga = None
    if G:
        qga, c1 = _as_array(qg)
        kga, c2 = _as_array(kg)
        vga, c3 = _as_array(vg)
        if not (c1 == c2 == c3 == code):
            raise TypeError("qg, kg, vg must share q's dtype")
        if qga.shape != (B, H, G, d) or kga.shape != qa.shape or vga.shape != qa.shape:
            raise ValueError("global tensor shapes do not match")
    dil = _i32(dilation if dilation is not None else [1] * H)
    w0, wh = _window(w, H)
    if len(dil) != H:
        raise ValueError("dilation needs one entry per head")
    gidx = _i32(global_idx) if G else None
    pads = _i32(pad_len)
    g = {name: np.zeros((B, H, n, d), dtype=np.float64) for name in ("dq", "dk", "dv")}
    if G:
        g["dqg"] = np.zeros((B, H, G, d), dtype=np.float64)
        g["dkg"] = np.zeros((B, H, n, d), dtype=np.float64)
        g["dvg"] = np.zeros((B, H, n, d), dtype=np.float64)
    rb = _bias_table(rel_bias, H, w0, wh)
    if rb is not None:
        g["drel_bias"] = np.zeros(rb.shape, dtype=np.float64)
    rc = lib.lf_oracle_bwd(code, _ptr(qa), _ptr(ka), _ptr(va), _ptr(qga), _ptr(kga), _ptr(vga), _ptr(da),
                           _ptr(gidx), G, B, H, n, d, w0, _ptr(wh), _ptr(dil), int(bool(causal)), _ptr(pads),
                           _ptr(rb), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g.get("dqg")),
                           _ptr(g.get("dkg")), _ptr(g.get("dvg")), _ptr(g.get("drel_bias")), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the problem (code %d)" % rc)
    return g


def proj(x, w, *, H: int, d: int, bias=None, threads: int = 0) -> np.ndarray:
    """Per-head linear projections in float64: x [B, n, K] hidden states,
    w [n_out*H*d, K] stacked weights, bias [n_out*H*d] (float32) or None ->
    [n_out, B, H, n, d], y[t, b, h, i, c] = x[b, i] . w[t*H*d + h*d + c] + bias."""
    lib = _load()
    xa, code = _as_array(x)
    wa, wc = _as_array(w)
    if code != wc:
        raise TypeError("x and w must share a dtype")
    B, n, K = xa.shape
    N = wa.shape[0]
    if wa.shape[1] != K or N % (H * d) != 0:
        raise ValueError("w must be [n_out*H*d, K]")
    n_out = N // (H * d)
    ba = None
    if bias is not None:
        ba = np.ascontiguousarray(np.asarray(bias.cpu() if hasattr(bias, "cpu") else bias, dtype=np.float32))
        if ba.shape != (N,):
            raise ValueError("bias must be [n_out*H*d]")
    y = np.zeros((n_out, B, H, n, d), dtype=np.float64)
    rc = lib.lf_oracle_proj(code, _ptr(xa), _ptr(wa), _ptr(ba), B, n, K, n_out, H, d, _ptr(y), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the projection sizes")
    return y


def mem_combine(q, local, mem_k, mem_v, idx, gate, threads: int = 0) -> np.ndarray:
    """Memory attention over retrieved (key, value) pairs mixed with the local
    output, in float64: q, local [B, H, n, d]; mem_k, mem_v [B, H, M, d];
    idx [B, H, n, km] int32 (-1: empty slot); gate [H] in [0, 1]."""
    lib = _load()
    qa, code = _as_array(q)
    la, lc = _as_array(local)
    ka, kc = _as_array(mem_k)
    va, vc = _as_array(mem_v)
    if not (code == lc == kc == vc):
        raise TypeError("q, local, mem_k, mem_v must share a dtype")
    B, H, n, d = qa.shape
    M = ka.shape[2]
    ia = np.ascontiguousarray(np.asarray(idx.cpu() if hasattr(idx, "cpu") else idx, dtype=np.int32))
    km = ia.shape[3]
    if la.shape != qa.shape or ka.shape != (B, H, M, d) or va.shape != ka.shape or ia.shape != (B, H, n, km):
        raise ValueError("shapes do not match")
    ga = np.ascontiguousarray(np.asarray(gate.cpu() if hasattr(gate, "cpu") else gate, dtype=np.float64))
    if ga.shape != (H,):
        raise ValueError("gate needs one weight per head")
    out = np.zeros((B, H, n, d), dtype=np.float64)
    rc = lib.lf_oracle_mem_combine(code, _ptr(qa), _ptr(la), _ptr(ka), _ptr(va), _ptr(ia), _ptr(ga), B, H, n, d,
                                   M, km, _ptr(out), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the memory combine (sizes or an index out of range)")
    return out


def attended(*, n: int, w, dilation: Sequence[int], causal: bool = False,
             global_idx: Sequence[int] = (), pad_len: Optional[Sequence[int]] = None,
             b: int = 0, h: int = 0, i: int = 0, B: int = 1):
    """(sorted list of attended keys, is_global_row) for one row."""
    lib = _load()
    H = len(dilation)
    dil = _i32(dilation)
    gidx = _i32(global_idx) if len(global_idx) else None
    pads = _i32(pad_len)
    keys = np.zeros(max(n, 1), dtype=np.int32)
    isg = np.zeros(1, dtype=np.int32)
    w0, wh = _window(w, H)
    cnt = lib.lf_oracle_attended(_ptr(gidx), len(global_idx), B, H, n, w0, _ptr(wh), _ptr(dil),
                                 int(bool(causal)), _ptr(pads), b, h, i, _ptr(keys), _ptr(isg))
    if cnt < 0:
        raise ValueError("oracle rejected the pattern")
    return sorted(int(x) for x in keys[:cnt]), bool(isg[0])


def count_pairs(*, B: int, H: int, n: int, w, dilation: Sequence[int], causal: bool = False,
                global_idx: Sequence[int] = (), pad_len: Optional[Sequence[int]] = None):
    """(attended pairs over every row, pairs on the global tokens' own rows),
    by enumerating each row's attended set."""
    lib = _load()
    dil = _i32(dilation)
    gidx = _i32(global_idx) if len(global_idx) else None
    pads = _i32(pad_len)
    pairs = np.zeros(1, dtype=np.int64)
    gpairs = np.zeros(1, dtype=np.int64)
    w0, wh = _window(w, H)
    rc = lib.lf_oracle_count_pairs(_ptr(gidx), len(global_idx), B, H, n, w0, _ptr(wh), _ptr(dil),
                                   int(bool(causal)), _ptr(pads), _ptr(pairs), _ptr(gpairs))
    if rc != 0:
        raise ValueError("oracle rejected the pattern")
    return int(pairs[0]), int(gpairs[0])


def wl_count_pairs(wl):
    """count_pairs() for a workloads.Workload."""
    return count_pairs(B=wl.B, H=wl.H, n=wl.n, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                       global_idx=wl.global_idx, pad_len=wl.pad_len)


def wl_bwd(wl, inputs, dout, threads: int = 0, rel_bias=None) -> dict:
    """bwd() for a workloads.Workload, its Inputs and an upstream gradient."""
    return bwd(inputs.q, inputs.k, inputs.v, dout, w=wl.w, dilation=wl.dilation, causal=wl.causal,
               pad_len=wl.pad_len, qg=inputs.qg, kg=inputs.kg, vg=inputs.vg,
               global_idx=wl.global_idx, rel_bias=rel_bias, threads=threads)


def wl_fwd(wl, inputs, rows=None, threads: int = 0, rel_bias=None) -> np.ndarray:
    """fwd() for a workloads.Workload and its Inputs."""
    return fwd(inputs.q, inputs.k, inputs.v, w=wl.w, dilation=wl.dilation, causal=wl.causal,
               pad_len=wl.pad_len, qg=inputs.qg, kg=inputs.kg, vg=inputs.vg,
               global_idx=wl.global_idx, rows=rows, rel_bias=rel_bias, threads=threads)
