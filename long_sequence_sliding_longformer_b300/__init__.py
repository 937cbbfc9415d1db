"""Longformer-style band attention on one B300 -- Python binding of liblf_attn.

Argument marshalling only: every step of the computation runs in the CUDA
library's kernels (see include/lf_attn.h for the operation and its ABI).
There is no fallback: if the library is missing or a call fails, an error is
raised.

    out = attn(q, k, v, w=512, dilation=[1]*H, causal=False,
               qg=qg, kg=kg, vg=vg, global_idx=[0], pad_len=None)

q, k, v, kg, vg: [B, H, n, d] CUDA tensors (bf16 with d in {64, 128}, or
fp32 with d <= 128); qg: [B, H, G, d].  The call is asynchronous on the
current CUDA stream (or `stream`).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

__all__ = ["attn", "attn_bwd", "proj_heads", "mem_combine", "attn_varglobal", "attn_bwd_varglobal", "count_pairs", "set_band_events", "launch_count", "last_band_kernel", "set_wait_limit_ns", "device_error", "LfError",
           "load", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblf_attn.so")
_lib = None

_STATUS = {0: "LF_OK", 1: "LF_ERR_INVALID_ARG", 2: "LF_ERR_UNSUPPORTED", 3: "LF_ERR_CUDA",
           4: "LF_ERR_NO_MEMORY", 5: "LF_ERR_TIMEOUT"}


class LfError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS.get(status, status), message))
        self.status = status


def load():
    """Load liblf_attn.so (built by _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("liblf_attn.so is not built; run long_sequence_sliding_longformer_b300._build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fwd_args = [P, P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P]
    for name in ("lf_attn_fwd", "lf_attn_fwd_f32"):
        fn = getattr(lib, name)
        fn.argtypes = fwd_args
        fn.restype = ctypes.c_int
    bwd_args = [P, P, P, P, P, P, P, i32, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, P, i32, P, P]
    for name in ("lf_attn_bwd", "lf_attn_bwd_f32"):
        fn = getattr(lib, name)
        fn.argtypes = bwd_args
        fn.restype = ctypes.c_int
    for name in ("lf_attn_fwd_bias", "lf_attn_fwd_bias_f32"):
        fn = getattr(lib, name)
        fn.argtypes = fwd_args[:-1] + [P, P]
        fn.restype = ctypes.c_int
    for name in ("lf_attn_bwd_bias", "lf_attn_bwd_bias_f32"):
        fn = getattr(lib, name)
        fn.argtypes = bwd_args[:-1] + [P, P, P]
        fn.restype = ctypes.c_int
    # per-head windows: the w argument becomes a host array
    for name, args, at in (("lf_attn_fwd_hw", fwd_args, 13), ("lf_attn_fwd_hw_f32", fwd_args, 13),
                           ("lf_attn_bwd_hw", bwd_args, 19), ("lf_attn_bwd_hw_f32", bwd_args, 19)):
        fn = getattr(lib, name)
        fn.argtypes = args[:at] + [P] + args[at + 1:]
        fn.restype = ctypes.c_int
    lib.lf_proj_heads.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P]
    lib.lf_proj_heads.restype = ctypes.c_int
    lib.lf_mem_combine.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
    lib.lf_mem_combine.restype = ctypes.c_int
    lib.lf_attn_fwd_varglobal.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, P, i32, P, P]
    lib.lf_attn_fwd_varglobal.restype = ctypes.c_int
    lib.lf_attn_bwd_varglobal.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                          i32, i32, i32, i32, i32, P, i32, P, P]
    lib.lf_attn_bwd_varglobal.restype = ctypes.c_int
    lib.lf_attn_count_pairs.argtypes = [i32, i32, i32, i32, i32, P, i32, P, P, i32,
                                        ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)]
    lib.lf_attn_count_pairs.restype = ctypes.c_int
    lib.lf_status_string.argtypes = [ctypes.c_int]
    lib.lf_status_string.restype = ctypes.c_char_p
    lib.lf_last_error_message.restype = ctypes.c_char_p
    lib.lf_attn_set_band_events.argtypes = [P, P]
    lib.lf_attn_set_band_events.restype = ctypes.c_int
    lib.lf_attn_launch_count.restype = ctypes.c_uint64
    lib.lf_attn_last_band_kernel.restype = ctypes.c_char_p
    lib.lf_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.lf_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.lf_device_error.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise LfError(status, load().lf_last_error_message().decode())


def _i32_array(seq) -> Optional[ctypes.Array]:
    if seq is None:
        return None
    seq = [int(x) for x in seq]
    return (ctypes.c_int32 * max(len(seq), 1))(*seq)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_table(t: torch.Tensor, H: int, w: int, name: str):
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (H, w + 1):
        raise ValueError("%s must be a contiguous fp32 CUDA tensor of shape (%d, %d)" % (name, H, w + 1))


def _window(w, H: int):
    """w as one int (every head) or one int per head: (the call's w
    argument, whether it is the per-head array)."""
    if isinstance(w, int) or (torch.is_tensor(w) and w.dim() == 0) or hasattr(w, "__index__"):
        return int(w), False
    ws = [int(x) for x in w]
    if len(ws) != H:
        raise ValueError("w needs one entry per head (or a single int)")
    return _i32_array(ws), True


def attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, w,
         dilation: Optional[Sequence[int]] = None, causal: bool = False,
         pad_len: Optional[Sequence[int]] = None, qg: Optional[torch.Tensor] = None,
         kg: Optional[torch.Tensor] = None, vg: Optional[torch.Tensor] = None,
         global_idx: Sequence[int] = (), out: Optional[torch.Tensor] = None,
         rel_bias: Optional[torch.Tensor] = None,
         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Sliding / dilated / causal window attention with global tokens.  w is
    the window of every head, or a sequence of one window per head.
    rel_bias: optional fp32 CUDA tensor [H, w + 1], added to the band keys'
    scores at window step t (entry t + w/2); needs one w for every head."""
    lib = load()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, n, d]")
    B, H, n, d = q.shape
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bf16 or fp32, got %s" % q.dtype)
    tensors = [("q", q), ("k", k), ("v", v)]
    G = len(global_idx)
    if G:
        tensors += [("qg", qg), ("kg", kg), ("vg", vg)]
    for name, t in tensors:
        if t is None:
            raise ValueError("%s is required" % name)
        if not t.is_cuda or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor of dtype %s" % (name, q.dtype))
        want = (B, H, G, d) if name == "qg" else (B, H, n, d)
        if tuple(t.shape) != want:
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), want))
    if out is None:
        out = torch.empty_like(q)
    elif tuple(out.shape) != (B, H, n, d) or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, H, n, d] tensor of q's dtype")
    dil = _i32_array(dilation if dilation is not None else [1] * H)
    if len(dilation if dilation is not None else [1] * H) != H:
        raise ValueError("dilation needs one entry per head")
    gidx = _i32_array(global_idx) if G else None
    pads = _i32_array(pad_len)
    if pad_len is not None and len(pad_len) != B:
        raise ValueError("pad_len needs one entry per batch row")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    warg, per_head = _window(w, H)
    bf = q.dtype == torch.bfloat16
    extra = []
    if rel_bias is not None:
        if per_head:
            raise ValueError("a relative bias takes one window for every head")
        _check_table(rel_bias, H, warg, "rel_bias")
        fn = lib.lf_attn_fwd_bias if bf else lib.lf_attn_fwd_bias_f32
        extra = [rel_bias.data_ptr()]
    elif per_head:
        fn = lib.lf_attn_fwd_hw if bf else lib.lf_attn_fwd_hw_f32
    else:
        fn = lib.lf_attn_fwd if bf else lib.lf_attn_fwd_f32
    with torch.cuda.device(q.device):
        _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(qg) if G else None,
                  _ptr(kg) if G else None, _ptr(vg) if G else None, gidx, G, out.data_ptr(),
                  B, H, n, d, warg, dil, int(bool(causal)), pads, *extra, s.cuda_stream))
    return out


def count_pairs(*, B: int, H: int, n: int, d: int, w: int, dilation: Sequence[int],
                causal: bool = False, pad_len: Optional[Sequence[int]] = None,
                global_idx: Sequence[int] = ()):
    """(attended pairs, useful FLOPs = 4*d*pairs) of a pattern; host only."""
    lib = load()
    pairs = ctypes.c_int64(0)
    flops = ctypes.c_double(0.0)
    _check(lib.lf_attn_count_pairs(B, H, n, d, int(w), _i32_array(dilation), int(bool(causal)),
                                   _i32_array(pad_len), _i32_array(global_idx) if len(global_idx) else None,
                                   len(global_idx), ctypes.byref(pairs), ctypes.byref(flops)))
    return int(pairs.value), float(flops.value)


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor, *, w,
             dilation: Optional[Sequence[int]] = None, causal: bool = False,
             pad_len: Optional[Sequence[int]] = None, qg: Optional[torch.Tensor] = None,
             kg: Optional[torch.Tensor] = None, vg: Optional[torch.Tensor] = None,
             global_idx: Sequence[int] = (), grads: Optional[dict] = None,
             rel_bias: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Gradients of sum(dout * attn(...)): a dict of fp32 tensors dq, dk, dv
    and, with global tokens, dqg, dkg, dvg, and with rel_bias its gradient
    drel_bias [H, w + 1] (preallocated ones may be passed in `grads`)."""
    lib = load()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, n, d]")
    B, H, n, d = q.shape
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q must be bf16 or fp32, got %s" % q.dtype)
    G = len(global_idx)
    tensors = [("q", q), ("k", k), ("v", v), ("dout", dout)]
    if G:
        tensors += [("qg", qg), ("kg", kg), ("vg", vg)]
    for name, t in tensors:
        if t is None:
            raise ValueError("%s is required" % name)
        if not t.is_cuda or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor of dtype %s" % (name, q.dtype))
        want = (B, H, G, d) if name == "qg" else (B, H, n, d)
        if tuple(t.shape) != want:
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), want))
    names = ["dq", "dk", "dv"] + (["dqg", "dkg", "dvg"] if G else [])
    if rel_bias is not None:
        names.append("drel_bias")
    g = dict(grads) if grads else {}
    for name in names:
        want = (B, H, G, d) if name == "dqg" else (H, int(w) + 1) if name == "drel_bias" else (B, H, n, d)
        if name not in g:
            g[name] = torch.empty(want, dtype=torch.float32, device=q.device)
        t = g[name]
        if tuple(t.shape) != want or t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("%s must be a contiguous fp32 CUDA tensor of shape %s" % (name, want))
    dil = _i32_array(dilation if dilation is not None else [1] * H)
    if len(dilation if dilation is not None else [1] * H) != H:
        raise ValueError("dilation needs one entry per head")
    gidx = _i32_array(global_idx) if G else None
    pads = _i32_array(pad_len)
    if pad_len is not None and len(pad_len) != B:
        raise ValueError("pad_len needs one entry per batch row")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    warg, per_head = _window(w, H)
    bf = q.dtype == torch.bfloat16
    gp = lambda name: _ptr(g[name]) if name in g else None
    extra = []
    if rel_bias is not None:
        if per_head:
            raise ValueError("a relative bias takes one window for every head")
        _check_table(rel_bias, H, warg, "rel_bias")
        fn = lib.lf_attn_bwd_bias if bf else lib.lf_attn_bwd_bias_f32
        extra = [rel_bias.data_ptr(), gp("drel_bias")]
    elif per_head:
        fn = lib.lf_attn_bwd_hw if bf else lib.lf_attn_bwd_hw_f32
    else:
        fn = lib.lf_attn_bwd if bf else lib.lf_attn_bwd_f32
    with torch.cuda.device(q.device):
        _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(qg) if G else None,
                  _ptr(kg) if G else None, _ptr(vg) if G else None, gidx, G, dout.data_ptr(),
                  gp("dq"), gp("dk"), gp("dv"), gp("dqg"), gp("dkg"), gp("dvg"),
                  B, H, n, d, warg, dil, int(bool(causal)), pads, *extra, s.cuda_stream))
    return {name: g[name] for name in names}


def proj_heads(x: torch.Tensor, w: torch.Tensor, *, H: int, d: int, bias: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Per-head projections: x [B, n, K] bf16, w [n_out*H*d, K] bf16, bias
    [n_out*H*d] fp32 or None -> [n_out, B, H, n, d] bf16."""
    lib = load()
    if x.dim() != 3 or w.dim() != 2:
        raise ValueError("x must be [B, n, K] and w [n_out*H*d, K]")
    B, n, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or N % (H * d) != 0:
        raise ValueError("w must be [n_out*H*d, K]")
    for name, t in (("x", x), ("w", w)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bf16 CUDA tensor" % name)
    if bias is not None and (not bias.is_cuda or bias.dtype != torch.float32 or tuple(bias.shape) != (N,)
                             or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous fp32 CUDA tensor of shape [%d]" % N)
    n_out = N // (H * d)
    if out is None:
        out = torch.empty((n_out, B, H, n, d), dtype=torch.bfloat16, device=x.device)
    elif tuple(out.shape) != (n_out, B, H, n, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of shape %s" % ((n_out, B, H, n, d),))
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        _check(lib.lf_proj_heads(x.data_ptr(), w.data_ptr(), _ptr(bias) if bias is not None else None,
                                 out.data_ptr(), B, n, K, n_out, H, d, s.cuda_stream))
    return out


def mem_combine(q: torch.Tensor, local: torch.Tensor, mem_k: torch.Tensor, mem_v: torch.Tensor,
                idx: torch.Tensor, gate: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """gate[h] * attention(q, retrieved memory pairs) + (1 - gate[h]) * local.
    q, local [B, H, n, d] bf16; mem_k, mem_v [B, H, M, d] bf16; idx [B, H, n, km]
    int32 (-1: empty slot); gate [H] fp32.  out may be local (in place)."""
    lib = load()
    B, H, n, d = q.shape
    M, km = mem_k.shape[2], idx.shape[3]
    checks = [("q", q, torch.bfloat16, (B, H, n, d)), ("local", local, torch.bfloat16, (B, H, n, d)),
              ("mem_k", mem_k, torch.bfloat16, (B, H, M, d)), ("mem_v", mem_v, torch.bfloat16, (B, H, M, d)),
              ("idx", idx, torch.int32, (B, H, n, km)), ("gate", gate, torch.float32, (H,))]
    for name, t, dt, shape in checks:
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError("%s must be a contiguous %s CUDA tensor of shape %s" % (name, dt, shape))
    if out is None:
        out = torch.empty_like(q)
    elif tuple(out.shape) != (B, H, n, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor of q's shape")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _check(lib.lf_mem_combine(q.data_ptr(), local.data_ptr(), mem_k.data_ptr(), mem_v.data_ptr(),
                                  idx.data_ptr(), gate.data_ptr(), out.data_ptr(), B, H, n, d, M, km,
                                  s.cuda_stream))
    return out


def attn_varglobal(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, w: int,
                   global_idx: Sequence[Sequence[int]], qg: Optional[torch.Tensor] = None,
                   kg: Optional[torch.Tensor] = None, vg: Optional[torch.Tensor] = None,
                   dilation: Optional[Sequence[int]] = None, causal: bool = False,
                   pad_len: Optional[Sequence[int]] = None, out: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """attn() with one global list per batch row: global_idx[b] lists batch row
    b's global positions; qg packs the rows' [H, G_b, d] blocks one after the
    other ([sum_b H * G_b, d] or any shape with that many elements)."""
    lib = load()
    B, H, n, d = q.shape
    if len(global_idx) != B:
        raise ValueError("global_idx needs one list per batch row")
    offs = [0]
    for lst in global_idx:
        offs.append(offs[-1] + len(lst))
    total = offs[-1]
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("kg", kg), ("vg", vg)) if total else ()):
        if t is None or not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != (B, H, n, d):
            raise ValueError("%s must be a contiguous bf16 CUDA tensor of shape %s" % (name, (B, H, n, d)))
    if total and (qg is None or not qg.is_cuda or qg.dtype != torch.bfloat16 or not qg.is_contiguous()
                  or qg.numel() != total * H * d):
        raise ValueError("qg must be a contiguous bf16 CUDA tensor of %d elements" % (total * H * d))
    if out is None:
        out = torch.empty_like(q)
    flat = [int(x) for lst in global_idx for x in lst]
    dil = _i32_array(dilation if dilation is not None else [1] * H)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _check(lib.lf_attn_fwd_varglobal(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         _ptr(qg) if total else None, _ptr(kg) if total else None,
                                         _ptr(vg) if total else None, _i32_array(offs),
                                         _i32_array(flat) if total else None, out.data_ptr(), B, H, n, d,
                                         int(w), dil, int(bool(causal)), _i32_array(pad_len), s.cuda_stream))
    return out


def attn_bwd_varglobal(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor, *, w: int,
                       global_idx: Sequence[Sequence[int]], qg: Optional[torch.Tensor] = None,
                       kg: Optional[torch.Tensor] = None, vg: Optional[torch.Tensor] = None,
                       dilation: Optional[Sequence[int]] = None, causal: bool = False,
                       pad_len: Optional[Sequence[int]] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> dict:
    """attn_bwd() for attn_varglobal(): fp32 dq, dk, dv and, with any global
    token, dqg (packed like qg), dkg, dvg."""
    lib = load()
    B, H, n, d = q.shape
    offs = [0]
    for lst in global_idx:
        offs.append(offs[-1] + len(lst))
    total = offs[-1]
    if dout.shape != q.shape or dout.dtype != q.dtype or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous tensor like q")
    f32 = lambda shape: torch.empty(shape, dtype=torch.float32, device=q.device)
    g = {"dq": f32((B, H, n, d)), "dk": f32((B, H, n, d)), "dv": f32((B, H, n, d))}
    if total:
        g.update(dqg=f32((total * H, d)), dkg=f32((B, H, n, d)), dvg=f32((B, H, n, d)))
    flat = [int(x) for lst in global_idx for x in lst]
    dil = _i32_array(dilation if dilation is not None else [1] * H)
    gp = lambda name: _ptr(g[name]) if name in g else None
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _check(lib.lf_attn_bwd_varglobal(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         _ptr(qg) if total else None, _ptr(kg) if total else None,
                                         _ptr(vg) if total else None, _i32_array(offs),
                                         _i32_array(flat) if total else None, dout.data_ptr(),
                                         gp("dq"), gp("dk"), gp("dv"), gp("dqg"), gp("dkg"), gp("dvg"),
                                         B, H, n, d, int(w), dil, int(bool(causal)), _i32_array(pad_len),
                                         s.cuda_stream))
    return g


def set_band_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]):
    """Record `start`/`stop` around the band kernel of every later call (None, None clears)."""
    for e in (start, stop):
        if e is not None and not e.cuda_event:
            raise ValueError("record the event once before passing it (torch creates it lazily)")
    sp = None if start is None else ctypes.c_void_p(start.cuda_event)
    ep = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check(load().lf_attn_set_band_events(sp, ep))


def launch_count() -> int:
    return int(load().lf_attn_launch_count())


def last_band_kernel() -> str:
    """Name of the band kernel the last call on this thread launched ("" before any)."""
    return load().lf_attn_last_band_kernel().decode()


def set_wait_limit_ns(ns: int):
    """Limit of the kernels' pipeline waits on the current device (0: the 2 s default); for tests."""
    _check(load().lf_set_wait_limit_ns(int(ns)))


def device_error(clear: bool = False) -> int:
    code = ctypes.c_uint32(0)
    _check(load().lf_device_error(ctypes.byref(code), int(bool(clear))))
    return int(code.value)
