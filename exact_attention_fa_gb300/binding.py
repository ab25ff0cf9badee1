"""Thin ctypes binding of libfa_gb300.so: argument marshalling only.

Each function takes torch tensors, checks dtype/shape/device/contiguity, and passes raw device
pointers and the current CUDA stream to the C entry point of the same name (include/fa.h). Every
step of the computation runs in the library's kernels; there is no fallback: if the library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

FA_OK = 0
_STATUS = {
    1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED", 4: "FA_ERR_CUDA",
    5: "FA_ERR_DEVICE_TIMEOUT", 6: "FA_ERR_NO_DEVICE", 7: "FA_ERR_TOO_LARGE",
    8: "FA_ERR_SCRATCH_LIMIT",
}
FA_NOALLOC_SCRATCH_BYTES = 4 << 20

# (name, restype, argtypes) of every symbol declared in include/fa.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = [
    ("fa_fwd", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    ("fa_fwd_fp32", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    ("fa_fwd_fp32_fa1", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    ("fa_fwd_blocksparse", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    ("fa_fwd_fp8", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _I, _P]),
    ("fa_bwd_workspace_bytes", ctypes.c_size_t, [_I, _I, _I, _I]),
    ("fa_bwd", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    ("fa_bwd_noalloc", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    ("fa_bwd_blocksparse", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P,
                                _P]),
    ("fa_decode", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P]),
    ("fa_decode_ctas", _I, [_I, _I, _I, _I, _I]),
    ("fa_decode_workspace_bytes", ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    ("fa_set_exp2_emulation", _I, [_I]),
    ("fa_get_exp2_emulation", _I, []),
    ("fa_selftest_wait_timeout", _I, [ctypes.c_uint, _P]),
    ("fa_check_device_error", _I, [_P]),
    ("fa_status_string", ctypes.c_char_p, [_I]),
    ("fa_abi_version", _I, []),
]


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({text})")
        self.status = status


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads (building first if needed) the library and declares every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.build_library()
    if not os.path.exists(path):
        raise FAError("load", -1, f"{path} is missing")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != FA_OK:
        raise FAError(fn, status, load().fa_status_string(status).decode())


def _call(fn: str, device: torch.device, *args):
    """Calls entry point `fn` with `device` current: the library works on the current CUDA device
    (its per-device state, the stream's device), which must be the tensors' own."""
    with torch.cuda.device(device):
        status = getattr(load(), fn)(*args)
    _check(fn, status)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _bhnd(q: torch.Tensor, *others: torch.Tensor, dtype=torch.bfloat16):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    tensors = (q,) + others
    for t in tensors:
        if t.shape != q.shape:
            raise ValueError(f"shape mismatch: {tuple(t.shape)} vs {tuple(q.shape)}")
        if t.dtype != dtype:
            raise TypeError(f"expected {dtype}, got {t.dtype}")
    for t in tensors:
        if not t.is_cuda or t.device != q.device:
            raise ValueError("all tensors must be on the same CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")
    return q.shape


def _rows(t: torch.Tensor, shape, dtype=torch.float32):
    if tuple(t.shape) != tuple(shape[:3]) or t.dtype != dtype or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"expected a contiguous {dtype} CUDA tensor of shape {tuple(shape[:3])}")


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool = False):
    """bf16 forward into preallocated o [B,H,N,d] bf16 and lse [B,H,N] fp32."""
    B, H, N, d = _bhnd(q, k, v, o)
    _rows(lse, q.shape)
    _call("fa_fwd", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
          float(scale), int(bool(causal)), _stream(q))


def fa_fwd_fp32(q, k, v, o, lse, scale: float, causal: bool = False):
    """fp32 forward (FMA pipes) into preallocated o [B,H,N,d] fp32 and lse [B,H,N] fp32."""
    B, H, N, d = _bhnd(q, k, v, o, dtype=torch.float32)
    _rows(lse, q.shape)
    _call("fa_fwd_fp32", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
          float(scale), int(bool(causal)), _stream(q))


def fa_fwd_fp32_fa1(q, k, v, o, lse, scale: float, causal: bool = False):
    """fa_fwd_fp32 with the FlashAttention-1 per-block normalised update (same result)."""
    B, H, N, d = _bhnd(q, k, v, o, dtype=torch.float32)
    _rows(lse, q.shape)
    _call("fa_fwd_fp32_fa1", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
          float(scale), int(bool(causal)), _stream(q))


def fa_fwd_blocksparse(q, k, v, o, lse, scale: float, block_mask, causal: bool = False):
    """Block-sparse bf16 forward; block_mask is a uint8 CUDA tensor [ceil(N/128)] * 2; causal
    additionally applies the causal mask."""
    B, H, N, d = _bhnd(q, k, v, o)
    _rows(lse, q.shape)
    nt = (N + 127) // 128
    if (block_mask.dtype != torch.uint8 or tuple(block_mask.shape) != (nt, nt)
            or not block_mask.is_cuda or not block_mask.is_contiguous()):
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor [{nt}, {nt}]")
    _call("fa_fwd_blocksparse", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N,
          d, float(scale), int(bool(causal)), _ptr(block_mask), _stream(q))


def fa_fwd_fp8(q, k, v, o, lse, scale: float, v_scale: float = 1.0, causal: bool = False):
    """e4m3 forward: q, k, v torch.float8_e4m3fn [B,H,N,d] (d = 128); o bf16 and lse fp32
    preallocated; o = v_scale * softmax(scale * q k^T) v."""
    B, H, N, d = _bhnd(q, k, v, dtype=torch.float8_e4m3fn)
    _bhnd(o)
    if tuple(o.shape) != tuple(q.shape) or o.device != q.device:
        raise ValueError("o must be a bf16 tensor of q's shape on q's device")
    _rows(lse, q.shape)
    _call("fa_fwd_fp8", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
          float(scale), float(v_scale), int(bool(causal)), _stream(q))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool, workspace):
    """Backward: dq fp32, dk/dv bf16 (preallocated); workspace from fa_bwd_workspace_bytes."""
    B, H, N, d = _bhnd(q, k, v, o, do, dk, dv)
    _bhnd(dq, dtype=torch.float32)
    if tuple(dq.shape) != tuple(q.shape):
        raise ValueError("dq must have the shape of q")
    _rows(lse, q.shape)
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace.numel() * workspace.element_size() < need or not workspace.is_cuda:
        raise ValueError(f"workspace must hold at least {need} bytes on the device")
    _call("fa_bwd", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
          _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)), _ptr(workspace),
          _stream(q))


def fa_bwd_blocksparse(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool, block_mask,
                       workspace):
    """Block-sparse backward: fa_bwd with the forward's uint8 tile mask [ceil(N/128)] * 2."""
    B, H, N, d = _bhnd(q, k, v, o, do, dk, dv)
    _bhnd(dq, dtype=torch.float32)
    if tuple(dq.shape) != tuple(q.shape):
        raise ValueError("dq must have the shape of q")
    _rows(lse, q.shape)
    nt = (N + 127) // 128
    if (block_mask.dtype != torch.uint8 or tuple(block_mask.shape) != (nt, nt)
            or not block_mask.is_cuda or not block_mask.is_contiguous()):
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor [{nt}, {nt}]")
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace.numel() * workspace.element_size() < need or not workspace.is_cuda:
        raise ValueError(f"workspace must hold at least {need} bytes on the device")
    _call("fa_bwd_blocksparse", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
          _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
          _ptr(block_mask), _ptr(workspace), _stream(q))


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool):
    """fa_bwd for callers that cannot allocate: the library's static scratch replaces the
    workspace (see include/fa.h for its size limit and sharing rules)."""
    B, H, N, d = _bhnd(q, k, v, o, do, dk, dv)
    _bhnd(dq, dtype=torch.float32)
    if tuple(dq.shape) != tuple(q.shape):
        raise ValueError("dq must have the shape of q")
    _rows(lse, q.shape)
    _call("fa_bwd_noalloc", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
          _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)), _stream(q))


def fa_decode_ctas(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().fa_decode_ctas(B, H, Nq, Nk, d))


def fa_decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().fa_decode_workspace_bytes(B, H, Nq, Nk, d))


def fa_decode(q, k, v, o, lse, scale: float, n_ctas: int = 0, workspace=None):
    """Decoding forward: q, o bf16 [B,H,Nq,d] (Nq <= 8), k, v bf16 [B,H,Nk,d], lse fp32 [B,H,Nq];
    workspace: fa_decode_workspace_bytes(...) bytes on the device."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _bhnd(q, o)
    _bhnd(k, v)
    if k.shape[:2] != q.shape[:2] or k.shape[3] != d or q.device != k.device:
        raise ValueError("q and k/v must share B, H, d and the device")
    _rows(lse, q.shape)
    need = fa_decode_workspace_bytes(B, H, Nq, Nk, d)
    if (workspace is None or not workspace.is_cuda or not workspace.is_contiguous()
            or workspace.numel() * workspace.element_size() < need):
        raise ValueError(f"workspace must be a contiguous CUDA tensor of at least {need} bytes")
    _call("fa_decode", q.device, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
          float(scale), int(n_ctas), _ptr(workspace), _stream(q))


def fa_set_exp2_emulation(per32: int):
    """Exponentials out of every 32 per row that the bf16 forward computes on the FMA pipes
    (0, the default, or 4); process-wide, for the forward calls enqueued afterwards."""
    _check("fa_set_exp2_emulation", load().fa_set_exp2_emulation(int(per32)))


def fa_get_exp2_emulation() -> int:
    return int(load().fa_get_exp2_emulation())


def fa_selftest_wait_timeout(timeout_us: int = 20000, device=None):
    """Runs the library's bounded-wait self-test kernel (a wait that can only time out)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    _call("fa_selftest_wait_timeout", dev, int(timeout_us), s)


def fa_check_device_error(device=None):
    """Synchronises the current stream and raises if a kernel recorded a device-side error."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    _call("fa_check_device_error", dev, s)


# ------------------------------------------------------------------------------- conveniences

def attention_forward(q, k, v, scale: float | None = None, causal: bool = False, block_mask=None):
    """Allocates O and lse with torch and runs the matching entry point (bf16, fp32 or e4m3;
    e4m3 inputs give a bf16 O)."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if q.dtype == torch.float8_e4m3fn:
        if block_mask is not None:
            raise ValueError("the e4m3 forward takes no block mask")
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
        fa_fwd_fp8(q, k, v, o, lse, scale, 1.0, causal)
        return o, lse
    o = torch.empty_like(q)
    if q.dtype == torch.float32:
        if block_mask is not None:
            raise ValueError("block-sparse attention is bf16 only")
        fa_fwd_fp32(q, k, v, o, lse, scale, causal)
    elif block_mask is not None:
        fa_fwd_blocksparse(q, k, v, o, lse, scale, block_mask, causal)
    else:
        fa_fwd(q, k, v, o, lse, scale, causal)
    return o, lse


def attention_decode(q, k, v, scale: float | None = None, n_ctas: int = 0):
    """Allocates O, lse and the workspace and runs fa_decode (n_ctas = 0: the library's choice)."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    B, H, Nq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    ws = torch.empty(max(16, fa_decode_workspace_bytes(B, H, Nq, k.shape[2], d)),
                     dtype=torch.uint8, device=q.device)
    fa_decode(q, k, v, o, lse, scale, n_ctas, ws)
    return o, lse


def attention_backward(q, k, v, o, lse, do, scale: float | None = None, causal: bool = False,
                       block_mask=None):
    """Allocates dq (fp32), dk, dv (bf16) and the workspace, and runs fa_bwd (with a tile mask:
    fa_bwd_blocksparse)."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    B, H, N, d = q.shape
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = torch.empty(max(16, fa_bwd_workspace_bytes(B, H, N, d)), dtype=torch.uint8,
                     device=q.device)
    if block_mask is not None:
        fa_bwd_blocksparse(q, k, v, o, do, lse, dq, dk, dv, scale, causal, block_mask, ws)
    else:
        fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal, ws)
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    """Forward and backward through the library, for use inside autograd graphs: the forward
    saves Q, K, V, O and lse, the backward runs fa_bwd (fa_bwd_blocksparse with a tile mask) on
    them."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal, block_mask):
        o, lse = attention_forward(q, k, v, scale, causal=causal, block_mask=block_mask)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale, ctx.causal, ctx.block_mask = scale, causal, block_mask
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = attention_backward(q, k, v, o, lse, do.contiguous(), ctx.scale,
                                        causal=ctx.causal, block_mask=ctx.block_mask)
        return dq.to(q.dtype), dk, dv, None, None, None


def attention(q, k, v, scale: float | None = None, causal: bool = False, block_mask=None):
    """O (and lse) of bf16 [B, H, N, d] inputs, differentiable with respect to Q, K and V: the
    gradients come from the library's backward (dQ, computed in fp32, is returned in Q's dtype;
    call attention_backward directly to keep it in fp32)."""
    if q.dtype != torch.bfloat16:
        raise ValueError("attention() differentiates the bf16 path; use attention_forward for "
                         "fp32 or e4m3 inputs")
    scale = q.shape[-1] ** -0.5 if scale is None else float(scale)
    return _Attention.apply(q, k, v, scale, bool(causal), block_mask)
