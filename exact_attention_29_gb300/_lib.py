"""ctypes binding of libfa.so: argument marshalling only.

Every function here checks tensor shapes/dtypes/devices, turns tensors into
raw device pointers and the current torch stream into a cudaStream_t, calls
the C ABI of the same name, and raises ``FaError`` on a non-OK status. All
arithmetic runs in the CUDA kernels; there is no fallback of any kind. If
``libfa.so`` is missing the first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# FA_LIBRARY may name another build of the library (libfa_debug.so: FA_DEBUG protocol checks)
LIB_PATH = os.environ.get("FA_LIBRARY") or os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_CHECK = 5

_lib = None
_lock = threading.Lock()

_VP = ctypes.c_void_p
_I = ctypes.c_int
_SIGNATURES = {
    "fa_fwd": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, ctypes.c_float, _VP], _I),
    "fa_fwd_host": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, ctypes.c_float, _VP], _I),
    "fa_decode": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP], _I),
    "fa_bwd": ([_VP] * 9 + [_I] * 5 + [ctypes.c_float, _VP], _I),
    "fa_decode_gqa": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP], _I),
    "fa_fwd_sparse": ([_VP, _VP, _VP, _VP, _I, _VP, _VP] + [_I] * 5 + [ctypes.c_float, _VP], _I),
    "fa_fwd_sparse_plan": ([_VP] + [_I] * 5 + [ctypes.POINTER(ctypes.c_longlong)] * 2, _I),
    "fa_quantize_fp8": ([_VP, _VP, _VP, _VP] + [_I] * 7 + [_VP], _I),
    "fa_fwd_fp8": ([_VP] * 8 + [_I] * 5 + [ctypes.c_float, _I, _VP], _I),
    "fa_bwd_plan": ([_I, _I, _I, _I, ctypes.POINTER(ctypes.c_longlong)], _I),
    "fa_decode_noalloc": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP], _I),
    "fa_status_string": ([_I], ctypes.c_char_p),
    "fa_last_error_string": ([], ctypes.c_char_p),
    "fa_check_device_error": ([_VP], _I),
    "fa_last_error_site": ([], _I),
    "fa_fwd_plan": ([_I, _I, _I, ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong)], _I),
    "fa_selftest_mma": ([_I, _VP, _VP, _VP, _I, _I, _VP], _I),
    "fa_selftest_wait_timeout": ([ctypes.c_uint, _VP], _I),
}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _lib
        text = lib.fa_status_string(status).decode() if lib else str(status)
        detail = lib.fa_last_error_string().decode() if (lib and status != FA_OK) else ""
        super().__init__(f"{where}: {text}" + (f" [{detail}]" if detail else ""))


def load_library() -> ctypes.CDLL:
    """Load libfa.so (once). Raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m exact_attention_29_gb300.build` "
                                   "(the CUDA library is required; there is no fallback)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (argtypes, restype) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = lib
    return _lib


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FaError(status, where)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _require(t: torch.Tensor, name: str, dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _require_shape(t: torch.Tensor, name: str, dtype, shape, device) -> None:
    """t must be a contiguous CUDA tensor of `dtype` and exactly `shape` on `device`
    (the library is given raw pointers, so a wrong extent would be written past)."""
    _require(t, name, dtype, len(shape))
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _same_device(device, **tensors) -> None:
    """Every tensor the library is handed must live on `device` (the call's device)."""
    for name, t in tensors.items():
        if t.device != device:
            raise ValueError(f"{name} must be on {device}, got {t.device}")


def _on(device, stream):
    """The library launches on the CUDA device that is current when it is called:
    make the tensors' device current for the call, and refuse a stream of
    another device."""
    if stream is not None and getattr(stream, "device", device) != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return torch.cuda.device(device)


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False, scale: float | None = None,
           o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Fused prefill attention. q, k, v: bf16 [B, H, N, d] on the GPU.

    Returns (o bf16 [B, H, N, d], lse fp32 [B, H, N]); enqueued on ``stream``
    (default: the current torch stream).
    """
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape [B, H, N, d]")
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    for t, n in ((k, "k"), (v, "v"), (o, "o")):
        _require_shape(t, n, torch.bfloat16, q.shape, q.device)
    _require_shape(lse, "lse", torch.float32, (B, H, N), q.device)
    with _on(q.device, stream):
        st = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                        1 if causal else 0, float(scale), _stream_handle(stream))
    _check(st, "fa_fwd")
    return o, lse


def fa_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False, scale: float | None = None,
                o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """fa_fwd on HOST tensors: q, k, v bf16 [B, H, N, d] in CPU memory (pinned
    for asynchronous copies). The library uploads them, runs the forward and
    downloads o and lse, all enqueued on ``stream``; the results are valid once
    the stream has passed the call. Returns (o, lse) as CPU tensors (pinned when
    allocated here)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
            raise ValueError(f"{n} must be a CPU tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 tensor [B, H, N, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same shape [B, H, N, d]")
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    for t, n, dt, shp in ((o, "o", torch.bfloat16, q.shape), (lse, "lse", torch.float32, (B, H, N))):
        if t.device.type != "cpu" or t.dtype != dt or tuple(t.shape) != tuple(shp) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU {dt} tensor of shape {tuple(shp)}")
    lib = load_library()
    st = lib.fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                         1 if causal else 0, float(scale), _stream_handle(stream))
    _check(st, "fa_fwd_host")
    return o, lse


def fa_fwd_sparse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor, causal: bool = False,
                  scale: float | None = None, o=None, lse=None, stream=None):
    """Block-sparse forward. q, k, v bf16 [B, H, N, d]; mask uint8 (or bool) on
    the GPU, [T, T] or [H, T, T] with T = ceil(N / 128).

    Returns (o bf16 [B, H, N, d], lse fp32 [B, H, N]).
    """
    lib = load_library()
    _require(q, "q", torch.bfloat16, 4)
    B, H, N, d = q.shape
    for t, n in ((k, "k"), (v, "v")):
        _require_shape(t, n, torch.bfloat16, q.shape, q.device)
    T = (N + 127) // 128
    mask = mask.to(torch.uint8).contiguous()
    if mask.dim() == 2:
        mask = mask.unsqueeze(0)
    if mask.shape[1:] != (T, T) or mask.shape[0] not in (1, H) or mask.device != q.device:
        raise ValueError("mask must be [T, T] or [H, T, T] on the device of q, T = ceil(N/128)")
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _require_shape(o, "o", torch.bfloat16, q.shape, q.device)
    _require_shape(lse, "lse", torch.float32, (B, H, N), q.device)
    with _on(q.device, stream):
        st = lib.fa_fwd_sparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), mask.data_ptr(), mask.shape[0], o.data_ptr(),
                               lse.data_ptr(), B, H, N, d, 1 if causal else 0, float(scale), _stream_handle(stream))
    _check(st, "fa_fwd_sparse")
    return o, lse


def fa_fwd_sparse_plan(mask, B: int, H: int, N: int, causal: bool = False):
    """(pairs_allowed, pairs_computed) of fa_fwd_sparse for a host mask [T, T] or [H, T, T]."""
    import numpy as np

    lib = load_library()
    m = np.ascontiguousarray(np.asarray(mask.cpu() if hasattr(mask, "cpu") else mask) != 0, dtype=np.uint8)
    if m.ndim == 2:
        m = m[None]
    a, c = ctypes.c_longlong(0), ctypes.c_longlong(0)
    _check(lib.fa_fwd_sparse_plan(m.ctypes.data, m.shape[0], B, H, N, 1 if causal else 0, ctypes.byref(a),
                                  ctypes.byref(c)), "fa_fwd_sparse_plan")
    return a.value, c.value


def _pitch16(n: int) -> int:
    return (n + 15) // 16 * 16


def fa_quantize_fp8(x: torch.Tensor, signs: torch.Tensor | None = None, per_head: bool = False,
                    transpose: bool = False, stream=None):
    """Block-quantize bf16 x [B, H, N, 128] to e4m3 codes (uint8).

    signs: fp32 [128] of +-1 for the incoherent rotation (None: no rotation).
    Returns (codes, scales): codes [B, H, N, 128] or, transposed, [B, H, 128,
    pitch] with pitch = N rounded up to 16; scales [B, H, ceil(N/128)] or
    [B, H] (per_head).
    """
    lib = load_library()
    _require(x, "x", torch.bfloat16, 4)
    B, H, N, d = x.shape
    pitch = _pitch16(N)
    if transpose:
        codes = torch.zeros((B, H, d, pitch), dtype=torch.uint8, device=x.device)
    else:
        codes = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    tiles = (N + 127) // 128
    scales = torch.empty((B, H) if per_head else (B, H, tiles), dtype=torch.float32, device=x.device)
    sp = 0
    if signs is not None:
        _require(signs, "signs", torch.float32, 1)
        _same_device(x.device, signs=signs)
        sp = signs.data_ptr()
    with _on(x.device, stream):
        st = lib.fa_quantize_fp8(x.data_ptr(), sp, codes.data_ptr(), scales.data_ptr(), B, H, N, d, int(per_head),
                                 int(transpose), pitch if transpose else 0, _stream_handle(stream))
    _check(st, "fa_quantize_fp8")
    return codes, scales


def fa_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, vt8: torch.Tensor, q_scale: torch.Tensor, k_scale: torch.Tensor,
               v_scale: torch.Tensor, causal: bool = False, scale: float | None = None, o=None, lse=None,
               stream=None):
    """FP8 forward. q8, k8 uint8 [B, H, N, 128]; vt8 uint8 [B, H, 128, pitch];
    scales from fa_quantize_fp8. Returns (o bf16 [B, H, N, 128], lse fp32 [B, H, N])."""
    lib = load_library()
    for t, n in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")):
        _require(t, n, torch.uint8, 4)
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or vt8.shape[:3] != (B, H, d) or vt8.shape[3] < N:
        raise ValueError("shapes must be q8, k8 [B,H,N,d] and vt8 [B,H,d,pitch >= N]")
    if k8.device != q8.device or vt8.device != q8.device:
        raise ValueError("q8, k8 and vt8 must be on the same device")
    tiles = (N + 127) // 128
    _require_shape(q_scale, "q_scale", torch.float32, (B, H, tiles), q8.device)
    _require_shape(k_scale, "k_scale", torch.float32, (B, H, tiles), q8.device)
    _require_shape(v_scale, "v_scale", torch.float32, (B, H), q8.device)
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _require_shape(o, "o", torch.bfloat16, (B, H, N, d), q8.device)
    _require_shape(lse, "lse", torch.float32, (B, H, N), q8.device)
    with _on(q8.device, stream):
        st = lib.fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), q_scale.data_ptr(), k_scale.data_ptr(),
                            v_scale.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 1 if causal else 0,
                            float(scale), vt8.shape[3], _stream_handle(stream))
    _check(st, "fa_fwd_fp8")
    return o, lse


def fa_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
           dout: torch.Tensor, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
           stream=None):
    """Gradients of fa_fwd. q, k, v, o, dout bf16 [B,H,N,d]; lse fp32 [B,H,N] (from fa_fwd).

    Returns (dq, dk, dv), bf16 [B,H,N,d].
    """
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _require(t, n, torch.bfloat16, 4)
    _require(lse, "lse", torch.float32, 3)
    if not (k.shape == v.shape == o.shape == dout.shape == q.shape):
        raise ValueError("q, k, v, o and dout must have the same shape [B, H, N, d]")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N):
        raise ValueError("lse must be [B, H, N]")
    _same_device(q.device, k=k, v=v, o=o, lse=lse, dout=dout)
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _require(t, n, torch.bfloat16, 4)
        if t.shape != q.shape:
            raise ValueError(f"{n} must match q")
    _same_device(q.device, dq=dq, dk=dk, dv=dv)
    with _on(q.device, stream):
        st = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, 1 if causal else 0, float(scale),
                        _stream_handle(stream))
    _check(st, "fa_bwd")
    return dq, dk, dv


def fa_bwd_plan(N: int, d: int, block: int = 128, causal: bool = False) -> int:
    """Number of fp32 additions into dQ that fa_bwd makes (host only)."""
    lib = load_library()
    adds = ctypes.c_longlong(0)
    _check(lib.fa_bwd_plan(N, d, block, 1 if causal else 0, ctypes.byref(adds)), "fa_bwd_plan")
    return adds.value


def fa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seqlens: torch.Tensor,
              num_splits: int, o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Flash-Decoding. q bf16 [B, H, d]; caches bf16 [B, H, L, d]; seqlens int32 [B] on the GPU.

    Returns (o bf16 [B, H, d], lse fp32 [B, H]).
    """
    lib = load_library()
    _require(q, "q", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(seqlens, "seqlens", torch.int32, 1)
    B, H, L, d = k_cache.shape
    if v_cache.shape != k_cache.shape or q.shape != (B, H, d) or seqlens.shape != (B,):
        raise ValueError("shapes must be q [B,H,d], caches [B,H,L,d], seqlens [B]")
    _same_device(q.device, k_cache=k_cache, v_cache=v_cache, seqlens=seqlens)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _require_shape(o, "o", torch.bfloat16, (B, H, d), q.device)
    _require_shape(lse, "lse", torch.float32, (B, H), q.device)
    with _on(q.device, stream):
        st = lib.fa_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seqlens.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, L, d, int(num_splits), _stream_handle(stream))
    _check(st, "fa_decode")
    return o, lse


def fa_decode_gqa(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seqlens: torch.Tensor,
                  num_splits: int, o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Flash-Decoding with grouped K/V heads. q bf16 [B, Hq, d]; caches bf16
    [B, Hkv, L, d] with Hq a multiple of Hkv (query head h uses K/V head
    h // (Hq // Hkv)); seqlens int32 [B] on the GPU.

    Returns (o bf16 [B, Hq, d], lse fp32 [B, Hq]).
    """
    lib = load_library()
    _require(q, "q", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(seqlens, "seqlens", torch.int32, 1)
    B, Hkv, L, d = k_cache.shape
    Hq = q.shape[1]
    if v_cache.shape != k_cache.shape or q.shape != (B, Hq, d) or seqlens.shape != (B,):
        raise ValueError("shapes must be q [B,Hq,d], caches [B,Hkv,L,d], seqlens [B]")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    _same_device(q.device, k_cache=k_cache, v_cache=v_cache, seqlens=seqlens)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _require_shape(o, "o", torch.bfloat16, (B, Hq, d), q.device)
    _require_shape(lse, "lse", torch.float32, (B, Hq), q.device)
    with _on(q.device, stream):
        st = lib.fa_decode_gqa(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seqlens.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, Hq, Hkv, L, d, int(num_splits), _stream_handle(stream))
    _check(st, "fa_decode_gqa")
    return o, lse


NOALLOC_WORKSPACE_FLOATS = 1 << 22


def fa_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seqlens: torch.Tensor,
                      num_splits: int, o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Flash-Decoding that allocates no device memory inside the call.

    Same arguments and results as ``fa_decode``; the split partials go to a
    fixed 16 MiB array owned by libfa.so instead of a per-call allocation, for
    callers that cannot allocate while decoding (a serving engine whose KV-cache
    pool owns nearly all device memory, or a latency-critical loop). Requires
    B * H * num_splits * (d + 1) <= 4,194,304; all calls share the array, so
    calls must not overlap on the GPU. Pass ``o`` and ``lse`` to avoid torch
    allocating the outputs.
    """
    lib = load_library()
    _require(q, "q", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(seqlens, "seqlens", torch.int32, 1)
    B, H, L, d = k_cache.shape
    if v_cache.shape != k_cache.shape or q.shape != (B, H, d) or seqlens.shape != (B,):
        raise ValueError("shapes must be q [B,H,d], caches [B,H,L,d], seqlens [B]")
    _same_device(q.device, k_cache=k_cache, v_cache=v_cache, seqlens=seqlens)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _require_shape(o, "o", torch.bfloat16, (B, H, d), q.device)
    _require_shape(lse, "lse", torch.float32, (B, H), q.device)
    with _on(q.device, stream):
        st = lib.fa_decode_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seqlens.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), B, H, L, d, int(num_splits), _stream_handle(stream))
    _check(st, "fa_decode_noalloc")
    return o, lse


def fa_check_device_error(stream=None) -> int:
    """Synchronise the stream and return the site code of a kernel wait that ran out
    (0 if none); raises FaError(FA_ERR_TIMEOUT) when one did."""
    lib = load_library()
    with torch.cuda.device(stream.device if stream is not None else torch.cuda.current_device()):
        st = lib.fa_check_device_error(_stream_handle(stream))
    site = lib.fa_last_error_site()
    if st in (FA_ERR_TIMEOUT, FA_ERR_CHECK):
        err = FaError(st, f"fa_check_device_error (site {site})")
        err.site = site
        raise err
    _check(st, "fa_check_device_error")
    return site


def fa_last_error_site() -> int:
    """Site code read by the calling thread's most recent fa_check_device_error (0 if none)."""
    return load_library().fa_last_error_site()


def fa_fwd_plan(N: int, block: int = 128, causal: bool = False):
    """(pairs_total, pairs_computed) of the prefill tile plan; host only."""
    lib = load_library()
    tot, done = ctypes.c_longlong(0), ctypes.c_longlong(0)
    _check(lib.fa_fwd_plan(N, block, 1 if causal else 0, ctypes.byref(tot), ctypes.byref(done)), "fa_fwd_plan")
    return tot.value, done.value


def fa_selftest_mma(mode: int, a: torch.Tensor, b: torch.Tensor, n: int, k: int, stream=None) -> torch.Tensor:
    lib = load_library()
    if mode in (4, 5):  # a CTA pair: 256 rows of D, then the two CTAs' TMEM base addresses
        d = torch.empty((256 * n + 2,), dtype=torch.float32, device=a.device)
    else:
        d = torch.empty((128, n), dtype=torch.float32, device=a.device)
    _same_device(a.device, b=b)
    _check(lib.fa_selftest_mma(mode, a.data_ptr(), b.data_ptr(), d.data_ptr(), n, k, _stream_handle(stream)),
           "fa_selftest_mma")
    return d


def fa_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    lib = load_library()
    _check(lib.fa_selftest_wait_timeout(int(timeout_us), _stream_handle(stream)), "fa_selftest_wait_timeout")
