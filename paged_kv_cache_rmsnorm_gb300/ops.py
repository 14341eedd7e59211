"""Thin ctypes binding of libpkv.so (include/pkv.h), with torch tensors as arguments.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  torch provides device memory and the current
stream.  If the library has not been built, every call raises — there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB_PATH

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 128
BLOCK_SIZE = 256
MAX_POSITION = 40960

EFLAG_NAMES = {
    0x1: "position",
    0x2: "slot",
    0x4: "block_id",
    0x8: "context",
    0x10: "timeout",
    0x20: "seqlen",
}

# every symbol include/pkv.h declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
SIGNATURES = {
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_version": (ctypes.c_int, []),
    "pkv_init": (ctypes.c_int, [ctypes.c_int]),
    "pkv_shutdown": (ctypes.c_int, []),
    "pkv_check_errors": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "pkv_qknorm_rope_store": (ctypes.c_int, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "pkv_attn_decode_workspace_size": (ctypes.c_size_t, [_I32, _I32]),
    "pkv_attn_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, ctypes.c_float, _P, _P,
                                       ctypes.c_size_t, _P]),
    "pkv_attn_prefill": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _I32, _I32, ctypes.c_float,
                                        _P, _P]),
    "pkv_attn_decode_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, ctypes.c_float, _P, _P,
                                               _P]),
    "pkv_add_rmsnorm": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I32, ctypes.c_float, _P]),
    "pkv_qkv_rope_store": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "pkv_bm_create": (ctypes.c_void_p, [_I32]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_num_free_blocks": (_I64, [_P]),
    "pkv_bm_ref_count": (_I32, [_P, _I32]),
    "pkv_bm_allocate": (ctypes.c_int, [_P, _I64, _P, _I32, _P]),
    "pkv_bm_append": (ctypes.c_int, [_P, _I64, _I32, _P]),
    "pkv_bm_free": (ctypes.c_int, [_P, _I64]),
    "pkv_bm_seq_info": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
    "pkv_bm_block_table": (ctypes.c_int, [_P, _P, _I32, _P, _I32]),
    "pkv_bm_slot_mapping": (ctypes.c_int, [_P, _I64, _I32, _I32, _P]),
}

_lib = None
_lock = threading.Lock()


class PkvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"pkv error {code}: {message}")
        self.code = code


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libpkv.so (built by ``_build.build``) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:  # the common case, without taking the lock
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'); "
                "there is no fallback path")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _check(rc: int) -> None:
    if rc != 0:
        raise PkvError(rc, load_library().pkv_last_error().decode())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device: int | None = None) -> int:
    """The cudaStream_t handle of ``stream`` (default: the current stream of ``device``, else of the
    current device, where the library launches).  The raw-handle query costs well under a
    microsecond; building the current torch.cuda.Stream object costs several, a large part of a
    small call."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device() if device is None else device)
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


def init(device: int | None = None) -> None:
    """Eager per-device set-up (RoPE table upload); call before CUDA-graph capture."""
    dev = torch.cuda.current_device() if device is None else int(device)
    _check(load_library().pkv_init(dev))


def check_errors(stream=None) -> list[str]:
    """Synchronise ``stream`` and return (and clear) the kernels' out-of-range flags."""
    flags = ctypes.c_uint32(0)
    rc = load_library().pkv_check_errors(ctypes.c_void_p(_stream(stream)), ctypes.byref(flags))
    if rc not in (0, -4):
        _check(rc)
    return [n for b, n in EFLAG_NAMES.items() if flags.value & b]


def qknorm_rope_store(q, k, v, positions, slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache, stream=None):
    """pkv_qknorm_rope_store: q/k RMSNorm + RoPE + slot scatter; q is rewritten in place."""
    strides = []
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 3)
        st = t.stride()
        if st[2] != 1 or st[1] != HEAD_DIM:
            raise ValueError(f"{n} needs contiguous heads of {HEAD_DIM} (strides (*, 128, 1))")
        strides.append(st[0])
    if q.shape[1:] != (NUM_Q_HEADS, HEAD_DIM) or k.shape[1:] != (NUM_KV_HEADS, HEAD_DIM) or v.shape != k.shape:
        raise ValueError("q must be [T, 32, 128] and k, v [T, 8, 128]")
    T = q.shape[0]
    if k.shape[0] != T:
        raise ValueError("q, k, v disagree on the token count")
    for t, n in ((positions, "positions"), (slot_mapping, "slot_mapping")):
        _need(t, n, torch.int32, 1)
        if t.shape[0] != T or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 [T]")
    for t, n in ((q_norm_w, "q_norm_w"), (k_norm_w, "k_norm_w")):
        _need(t, n, torch.bfloat16, 1)
        if t.shape[0] != HEAD_DIM or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 [128]")
    nb = _cache_blocks(k_cache, v_cache)
    _check(load_library().pkv_qknorm_rope_store(
        q.data_ptr(), strides[0], k.data_ptr(), strides[1], v.data_ptr(), strides[2], positions.data_ptr(),
        slot_mapping.data_ptr(), q_norm_w.data_ptr(), k_norm_w.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        T, nb, _stream(stream)))


def _cache_blocks(k_cache, v_cache) -> int:
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
        if t.shape[1:] != (BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous bf16 [num_blocks, 256, 8, 128]")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    return k_cache.shape[0]


# (device index, stream handle) -> zero-initialised workspace used only by calls on that stream
_workspaces: dict[tuple[int, int], torch.Tensor] = {}


def decode_workspace_size(batch: int, max_context: int) -> int:
    return int(load_library().pkv_attn_decode_workspace_size(int(batch), int(max_context)))


def _stream_object(stream, dev: torch.device) -> torch.cuda.Stream:
    if stream is None:
        return torch.cuda.current_stream(dev)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=dev)


def decode_workspace(batch: int, max_context: int, device=None, stream=None) -> torch.Tensor | None:
    """A zero-initialised workspace for pkv_attn_decode on ``stream`` (default: the current one).

    One workspace is kept per (device, stream) and grown on demand, so decode calls on different
    streams never share split tickets or partials.  It is allocated and zeroed on that stream, so
    the caching allocator only hands a replaced buffer out again after the stream's earlier
    kernels, the only ones that used it, are done with it.
    """
    need = decode_workspace_size(batch, max_context)
    if need == 0:
        return None
    index = torch.cuda.current_device() if device is None else torch.device(device).index
    key = (index, _stream(stream, index))
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        dev = torch.device("cuda", index)
        with torch.cuda.stream(_stream_object(stream, dev)):
            ws = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def attn_decode(q, k_cache, v_cache, context_lens, block_table, max_context: int, scale: float, out=None,
                workspace=None, stream=None):
    """pkv_attn_decode: one query token per sequence over its paged context."""
    _need(q, "q", torch.bfloat16, 3)
    if q.shape[1:] != (NUM_Q_HEADS, HEAD_DIM) or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 [B, 32, 128]")
    B = q.shape[0]
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    if context_lens.shape[0] != B or block_table.shape[0] != B or not block_table.is_contiguous():
        raise ValueError("context_lens [B] and a contiguous block_table [B, max_blocks] are required")
    nb = _cache_blocks(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, max_context, q.device, stream)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().pkv_attn_decode(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), context_lens.data_ptr(), block_table.data_ptr(), B,
        block_table.shape[1], nb, int(max_context), float(scale), out.data_ptr(), ws_ptr, ws_bytes, _stream(stream)))
    return out


def attn_decode_noalloc(q, k_cache, v_cache, context_lens, block_table, max_context: int, scale: float, out,
                        error_flags=None, stream=None):
    """pkv_attn_decode_noalloc: decode without any device allocation (static scratch inside the library).

    ``out`` must be supplied by the caller; ``error_flags`` is an optional int32 [1] CUDA tensor the kernel
    ORs its out-of-range bits into.
    """
    _need(q, "q", torch.bfloat16, 3)
    if q.shape[1:] != (NUM_Q_HEADS, HEAD_DIM) or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 [B, 32, 128]")
    B = q.shape[0]
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    if context_lens.shape[0] != B or block_table.shape[0] != B or not block_table.is_contiguous():
        raise ValueError("context_lens [B] and a contiguous block_table [B, max_blocks] are required")
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    nb = _cache_blocks(k_cache, v_cache)
    flags_ptr = None
    if error_flags is not None:
        _need(error_flags, "error_flags", torch.int32, 1)
        flags_ptr = error_flags.data_ptr()
    _check(load_library().pkv_attn_decode_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), context_lens.data_ptr(), block_table.data_ptr(), B,
        block_table.shape[1], nb, int(max_context), float(scale), out.data_ptr(), flags_ptr, _stream(stream)))
    return out


def attn_prefill(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q: int,
                 max_seqlen_k: int, scale: float, out=None, stream=None):
    """pkv_attn_prefill: causal varlen attention of a flat batch over the paged cache."""
    _need(q, "q", torch.bfloat16, 3)
    if q.shape[1:] != (NUM_Q_HEADS, HEAD_DIM) or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 [total_q, 32, 128]")
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, n, torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 2)
    S = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != S + 1 or block_table.shape[0] != S or not block_table.is_contiguous():
        raise ValueError("cu_seqlens_q/k [S+1] and a contiguous block_table [S, max_blocks] are required")
    nb = _cache_blocks(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    _check(load_library().pkv_attn_prefill(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
        block_table.data_ptr(), S, block_table.shape[1], nb, q.shape[0], int(max_seqlen_q), int(max_seqlen_k),
        float(scale), out.data_ptr(), _stream(stream)))
    return out


HIDDEN = 4096


def add_rmsnorm(x, residual, weight, out=None, eps: float = 1e-6, stream=None):
    """pkv_add_rmsnorm: the decoder layer's RMSNorm with the pending residual add folded in.

    ``residual`` (bf16 [T, 4096], or None for the first layer) is overwritten with the bf16 sum
    x + residual; returns ``out`` = RMSNorm of the fp32 sum (a new tensor unless given).
    """
    _need(x, "x", torch.bfloat16, 2)
    if x.shape[1] != HIDDEN or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 [T, 4096]")
    _need(weight, "weight", torch.bfloat16, 1)
    if weight.shape[0] != HIDDEN or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous bf16 [4096]")
    res_ptr = None
    if residual is not None:
        _need(residual, "residual", torch.bfloat16, 2)
        if residual.shape != x.shape or not residual.is_contiguous():
            raise ValueError("residual must be a contiguous bf16 tensor shaped like x")
        res_ptr = residual.data_ptr()
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, 2)
    if out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like x")
    _check(load_library().pkv_add_rmsnorm(x.data_ptr(), res_ptr, weight.data_ptr(), out.data_ptr(), x.shape[0],
                                          HIDDEN, float(eps), _stream(stream)))
    return out


QKV_OUT = 6144


def qkv_rope_store(x, w_qkv, positions, slot_mapping, q_norm_w, k_norm_w, k_cache, v_cache, q_out=None, stream=None):
    """pkv_qkv_rope_store: y = x w_qkv^T, then q/k RMSNorm + RoPE and the K/V scatter; returns q [T, 32, 128]."""
    _need(x, "x", torch.bfloat16, 2)
    if x.shape[1] != HIDDEN or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 [T, 4096]")
    _need(w_qkv, "w_qkv", torch.bfloat16, 2)
    if tuple(w_qkv.shape) != (QKV_OUT, HIDDEN) or not w_qkv.is_contiguous():
        raise ValueError("w_qkv must be a contiguous bf16 [6144, 4096]")
    T = x.shape[0]
    for t, n in ((positions, "positions"), (slot_mapping, "slot_mapping")):
        _need(t, n, torch.int32, 1)
        if t.shape[0] != T or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 [T]")
    for t, n in ((q_norm_w, "q_norm_w"), (k_norm_w, "k_norm_w")):
        _need(t, n, torch.bfloat16, 1)
        if t.shape[0] != HEAD_DIM:
            raise ValueError(f"{n} must be bf16 [128]")
    nb = _cache_blocks(k_cache, v_cache)
    if q_out is None:
        q_out = torch.empty(T, NUM_Q_HEADS, HEAD_DIM, dtype=torch.bfloat16, device=x.device)
    _need(q_out, "q_out", torch.bfloat16, 3)
    if q_out.shape != (T, NUM_Q_HEADS, HEAD_DIM) or not q_out.is_contiguous():
        raise ValueError("q_out must be a contiguous bf16 [T, 32, 128]")
    _check(load_library().pkv_qkv_rope_store(
        x.data_ptr(), w_qkv.data_ptr(), positions.data_ptr(), slot_mapping.data_ptr(), q_norm_w.data_ptr(),
        k_norm_w.data_ptr(), q_out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), T, nb, _stream(stream)))
    return q_out
