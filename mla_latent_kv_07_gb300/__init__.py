"""Python binding of libmla (absorbed MLA decode over a latent KV cache, GB300).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  There is no
fallback: if ``_build/libmla.so`` is missing the first call raises.

Functions mirror the C ABI in ``include/mla.h``:
    cache_append, workspace_size, decode, decode_sparse, workspace_status
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import layout  # noqa: F401  (byte/flop accounting)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmla.so")

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3_B128 = 1
MLA_KV_FP8_E4M3_B128_POW2 = 2
DEV_END_POS_CLAMPED = 0x1
DEV_APPEND_SKIPPED = 0x2
DEV_PIPELINE_TIMEOUT = 0x4

STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_OUT_OF_RANGE",
          3: "MLA_ERR_UNSUPPORTED", 4: "MLA_ERR_WORKSPACE", 5: "MLA_ERR_CUDA"}


class MLAError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}" + (f" ({detail})" if detail else ""))


class _CCache(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("kv", ctypes.c_void_p),
                ("kv_scale", ctypes.c_void_p), ("pe", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmla.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run `python -m mla_latent_kv_07_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
            L.mla_cache_append.argtypes = [P, P, P, P, I32, P]
            L.mla_cache_append.restype = I32
            L.mla_workspace_size.argtypes = [I32, I32, I32, I32]
            L.mla_workspace_size.restype = SZ
            L.mla_decode.argtypes = [P, P, P, P, I32, I32, I32, F, P, P, P, SZ, P]
            L.mla_decode.restype = I32
            L.mla_decode_append.argtypes = [P, P, P, P, P, P, I32, I32, I32, F, P, P, P, SZ, P]
            L.mla_decode_append.restype = I32
            L.mla_topk_select.argtypes = [P, P, I32, I32, I32, P, P]
            L.mla_topk_select.restype = I32
            L.mla_selftest_decode_timeout.argtypes = [P, P, P, P, I32, I32, I32, F, P, P, P, SZ, P]
            L.mla_selftest_decode_timeout.restype = I32
            L.mla_decode_mtp.argtypes = [P, P, P, P, I32, I32, I32, I32, F, P, P, P, SZ, P]
            L.mla_decode_mtp.restype = I32
            L.mla_decode_sparse.argtypes = [P, P, P, P, I32, I32, I32, F, P, I32, P, P, P, P, P,
                                            P, P, SZ, P]
            L.mla_decode_sparse.restype = I32
            L.mla_workspace_status.argtypes = [P, P, P]
            L.mla_workspace_status.restype = I32
            L.mla_status_string.argtypes = [I32]
            L.mla_status_string.restype = ctypes.c_char_p
            L.mla_last_error.restype = ctypes.c_char_p
            L.mla_decode_noalloc.argtypes = [P, P, P, P, I32, I32, I32, F, P, P, P]
            L.mla_decode_noalloc.restype = I32
            L.mla_absorb_q.argtypes = [P, P, I32, I32, P, P, P]
            L.mla_absorb_q.restype = I32
            L.mla_project_out.argtypes = [P, P, I32, I32, P, P, P]
            L.mla_project_out.restype = I32
            L.mla_read_ceiling.argtypes = [P, SZ, P, P]
            L.mla_read_ceiling.restype = I32
            L.mla_trace_begin.argtypes = [I32]
            L.mla_trace_begin.restype = I32
            L.mla_trace_end.argtypes = [P, P, P]
            L.mla_trace_end.restype = I32
            _lib = L
    return _lib


def _check(code: int, what: str):
    if code != 0:
        raise MLAError(code, what, lib().mla_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: want contiguous cuda {dtype} {tuple(shape)}, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}")


class Cache:
    """Caller-owned latent cache: kv [Bmax, S, 512] (bf16 or e4m3 bytes),
    kv_scale fp32 [Bmax, S, 4] (FP8 formats only), pe bf16 [Bmax, S, 64].
    fmt: MLA_KV_BF16, MLA_KV_FP8_E4M3_B128, or MLA_KV_FP8_E4M3_B128_POW2
    (FP8 whose appends round every block scale up to a power of two)."""

    def __init__(self, max_batch: int, max_seq_len: int, fmt: int = MLA_KV_BF16,
                 device="cuda", kv=None, kv_scale=None, pe=None):
        self.fmt, self.max_batch, self.max_seq_len = fmt, max_batch, max_seq_len
        shape = (max_batch, max_seq_len)
        if kv is None:
            kv = torch.zeros(shape + (512,), dtype=torch.bfloat16 if fmt == 0 else torch.uint8,
                             device=device)
        if fmt != MLA_KV_BF16 and kv_scale is None:
            kv_scale = torch.zeros(shape + (4,), dtype=torch.float32, device=device)
        if pe is None:
            pe = torch.zeros(shape + (64,), dtype=torch.bfloat16, device=device)
        _need(kv, torch.bfloat16 if fmt == 0 else torch.uint8, shape + (512,), "kv")
        _need(pe, torch.bfloat16, shape + (64,), "pe")
        if fmt != MLA_KV_BF16:
            _need(kv_scale, torch.float32, shape + (4,), "kv_scale")
        self.kv, self.kv_scale, self.pe = kv, kv_scale, pe
        self._c = _CCache(fmt, max_batch, max_seq_len, kv.data_ptr(),
                          kv_scale.data_ptr() if kv_scale is not None else None, pe.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self._c)


def cache_append(cache: Cache, kv_new, pe_new, start_pos, stream=None) -> None:
    """Write kv_new[b] / pe_new[b] (bf16 [B,512] / [B,64]) at row start_pos[b]."""
    B = kv_new.shape[0]
    _need(kv_new, torch.bfloat16, (B, 512), "kv_new")
    _need(pe_new, torch.bfloat16, (B, 64), "pe_new")
    pos = (ctypes.c_int32 * B)(*[int(x) for x in start_pos])
    _check(lib().mla_cache_append(cache.ref, _ptr(kv_new), _ptr(pe_new), pos, B,
                                  _stream(stream)), "mla_cache_append")


def workspace_size(B: int, H: int, max_end_pos: int, topk: int = 0) -> int:
    n = lib().mla_workspace_size(B, H, max_end_pos, topk)
    if n == 0:
        raise MLAError(3, "mla_workspace_size")
    return int(n)


def alloc_workspace(B: int, H: int, max_end_pos: int, topk: int = 0, device="cuda"):
    return torch.empty(workspace_size(B, H, max_end_pos, topk), dtype=torch.uint8, device=device)


def _outputs(B, H, device, out, lse, want_lse):
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=device)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=device)
    return out, lse


def decode(cache: Cache, q_latent, q_pe, end_pos, max_end_pos: int, softmax_scale: float,
           out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """Absorbed decode; returns (out bf16 [B,H,512], lse fp32 [B,H] or None)."""
    B, H, _ = q_latent.shape
    _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
    _need(q_pe, torch.bfloat16, (B, H, 64), "q_pe")
    _need(end_pos, torch.int32, (B,), "end_pos")
    out, lse = _outputs(B, H, q_latent.device, out, lse, want_lse)
    if workspace is None:
        workspace = alloc_workspace(B, H, max_end_pos, 0, q_latent.device)
    _check(lib().mla_decode(cache.ref, _ptr(q_latent), _ptr(q_pe), _ptr(end_pos), int(max_end_pos),
                            B, H, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                            workspace.numel(), _stream(stream)), "mla_decode")
    return out, lse


def decode_append(cache: Cache, kv_new, pe_new, q_latent, q_pe, end_pos, max_end_pos: int,
                  softmax_scale: float, out=None, lse=None, workspace=None, want_lse: bool = True,
                  stream=None):
    """Append row end_pos[b]-1 of every sequence (kv_new bf16 [B,512], pe_new
    bf16 [B,64]) and decode over it, in one call (see mla_decode_append);
    returns (out, lse) as decode."""
    B, H, _ = q_latent.shape
    _need(kv_new, torch.bfloat16, (B, 512), "kv_new")
    _need(pe_new, torch.bfloat16, (B, 64), "pe_new")
    _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
    _need(q_pe, torch.bfloat16, (B, H, 64), "q_pe")
    _need(end_pos, torch.int32, (B,), "end_pos")
    out, lse = _outputs(B, H, q_latent.device, out, lse, want_lse)
    if workspace is None:
        workspace = alloc_workspace(B, H, max_end_pos, 0, q_latent.device)
    _check(lib().mla_decode_append(cache.ref, _ptr(kv_new), _ptr(pe_new), _ptr(q_latent), _ptr(q_pe),
                                   _ptr(end_pos), int(max_end_pos), B, H, float(softmax_scale), _ptr(out),
                                   _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mla_decode_append")
    return out, lse


def topk_select(scores, end_pos, K: int, out=None, stream=None):
    """Top-k positions per sequence from fp32 scores [B, max_end_pos]:
    int32 [B, K], increasing, -1 padded (the index lists decode_sparse takes)."""
    B, S = scores.shape
    if scores.dtype != torch.float32 or not scores.is_contiguous() or not scores.is_cuda:
        raise ValueError(f"scores: want contiguous cuda float32 [B, S], got {scores.dtype} on {scores.device}")
    _need(end_pos, torch.int32, (B,), "end_pos")
    if out is None:
        out = torch.empty((B, K), dtype=torch.int32, device=scores.device)
    _need(out, torch.int32, (B, K), "out")
    _check(lib().mla_topk_select(_ptr(scores), _ptr(end_pos), B, S, int(K), _ptr(out), _stream(stream)),
           "mla_topk_select")
    return out


def selftest_decode_timeout(cache: Cache, q_latent, q_pe, end_pos, max_end_pos: int,
                            softmax_scale: float, workspace, stream=None) -> int:
    """mla_decode with the first unit's first tile withheld and short waits:
    returns the workspace status word (MLA_DEV_PIPELINE_TIMEOUT expected)."""
    B, H, _ = q_latent.shape
    _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
    _need(q_pe, torch.bfloat16, (B, H, 64), "q_pe")
    _need(end_pos, torch.int32, (B,), "end_pos")
    out, lse = _outputs(B, H, q_latent.device, None, None, True)
    _check(lib().mla_selftest_decode_timeout(cache.ref, _ptr(q_latent), _ptr(q_pe), _ptr(end_pos),
                                             int(max_end_pos), B, H, float(softmax_scale), _ptr(out),
                                             _ptr(lse), _ptr(workspace), workspace.numel(),
                                             _stream(stream)), "mla_selftest_decode_timeout")
    return workspace_status(workspace, stream)


def decode_mtp(cache: Cache, q_latent, q_pe, end_pos, max_end_pos: int, softmax_scale: float,
               out=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """Multi-token decode of s new tokens per sequence (token j of sequence b
    attends to positions 0 .. end_pos[b]-s+j); q_latent [B,s,H,512], q_pe
    [B,s,H,64].  Returns (out bf16 [B,s,H,512], lse fp32 [B,s,H] or None)."""
    B, s, H, _ = q_latent.shape
    _need(q_latent, torch.bfloat16, (B, s, H, 512), "q_latent")
    _need(q_pe, torch.bfloat16, (B, s, H, 64), "q_pe")
    _need(end_pos, torch.int32, (B,), "end_pos")
    out, lse = _outputs(B * s, H, q_latent.device, None if out is None else out.view(B * s, H, 512),
                        None if lse is None else lse.view(B * s, H), want_lse)
    if workspace is None:
        workspace = alloc_workspace(B * s, H, max_end_pos, 0, q_latent.device)
    _check(lib().mla_decode_mtp(cache.ref, _ptr(q_latent), _ptr(q_pe), _ptr(end_pos),
                                int(max_end_pos), B, s, H, float(softmax_scale), _ptr(out), _ptr(lse),
                                _ptr(workspace), workspace.numel(), _stream(stream)), "mla_decode_mtp")
    return out.view(B, s, H, 512), None if lse is None else lse.view(B, s, H)


def decode_noalloc(cache: Cache, q_latent, q_pe, end_pos, max_end_pos: int, softmax_scale: float,
                   out=None, lse=None, want_lse: bool = True, stream=None):
    """Dense decode through mla_decode_noalloc: no workspace is passed; the
    library uses its own static device scratch (for callers that cannot
    allocate).  Returns (out, lse)."""
    B, H, _ = q_latent.shape
    _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
    _need(q_pe, torch.bfloat16, (B, H, 64), "q_pe")
    _need(end_pos, torch.int32, (B,), "end_pos")
    out, lse = _outputs(B, H, q_latent.device, out, lse, want_lse)
    _check(lib().mla_decode_noalloc(cache.ref, _ptr(q_latent), _ptr(q_pe), _ptr(end_pos),
                                    int(max_end_pos), B, H, float(softmax_scale), _ptr(out),
                                    _ptr(lse), _stream(stream)), "mla_decode_noalloc")
    return out, lse


def decode_sparse(cache: Cache, q_latent, q_pe, end_pos, max_end_pos: int, softmax_scale: float,
                  topk, kv_new=None, pe_new=None, out=None, lse=None, gidx=None, gcount=None,
                  workspace=None, want_lse: bool = True, stream=None):
    """Top-k sparse decode (optionally appending kv_new/pe_new at end_pos-1 first).
    Returns (out, lse)."""
    B, H, _ = q_latent.shape
    K = topk.shape[1]
    _need(q_latent, torch.bfloat16, (B, H, 512), "q_latent")
    _need(q_pe, torch.bfloat16, (B, H, 64), "q_pe")
    _need(end_pos, torch.int32, (B,), "end_pos")
    _need(topk, torch.int32, (B, K), "topk")
    if kv_new is not None:
        _need(kv_new, torch.bfloat16, (B, 512), "kv_new")
        _need(pe_new, torch.bfloat16, (B, 64), "pe_new")
    out, lse = _outputs(B, H, q_latent.device, out, lse, want_lse)
    if workspace is None:
        workspace = alloc_workspace(B, H, max_end_pos, K, q_latent.device)
    _check(lib().mla_decode_sparse(cache.ref, _ptr(q_latent), _ptr(q_pe), _ptr(end_pos),
                                   int(max_end_pos), B, H, float(softmax_scale), _ptr(topk), K,
                                   _ptr(kv_new), _ptr(pe_new), _ptr(out), _ptr(lse), _ptr(gidx),
                                   _ptr(gcount), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "mla_decode_sparse")
    return out, lse


def workspace_status(workspace, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib().mla_workspace_status(_ptr(workspace), ctypes.byref(flags), _stream(stream)),
           "mla_workspace_status")
    return int(flags.value)


def absorb_q(q_nope, wkv_b, out=None, status=None, stream=None):
    """q_latent [B,H,512] bf16 = q_nope [B,H,128] . W_UK (rows 0..127 of each
    head of wkv_b [H,256,512] bf16)."""
    B, H, _ = q_nope.shape
    _need(q_nope, torch.bfloat16, (B, H, 128), "q_nope")
    _need(wkv_b, torch.bfloat16, (H, 256, 512), "wkv_b")
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    _need(out, torch.bfloat16, (B, H, 512), "out")
    _check(lib().mla_absorb_q(_ptr(q_nope), _ptr(wkv_b), B, H, _ptr(out), _ptr(status), _stream(stream)),
           "mla_absorb_q")
    return out


def project_out(x, wkv_b, out=None, status=None, stream=None):
    """o [B,H,128] bf16 = W_UV . x for x [B,H,512] bf16 (W_UV: rows 128..255
    of each head of wkv_b)."""
    B, H, _ = x.shape
    _need(x, torch.bfloat16, (B, H, 512), "x")
    _need(wkv_b, torch.bfloat16, (H, 256, 512), "wkv_b")
    if out is None:
        out = torch.empty((B, H, 128), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (B, H, 128), "out")
    _check(lib().mla_project_out(_ptr(x), _ptr(wkv_b), B, H, _ptr(out), _ptr(status), _stream(stream)),
           "mla_project_out")
    return out


def read_ceiling(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Stream all bytes of the contiguous CUDA tensor `buf` (a measurement of
    the achievable HBM read rate); XOR-folds them into the int32 `sink`."""
    if not (buf.is_cuda and buf.is_contiguous()):
        raise ValueError("buf must be a contiguous CUDA tensor")
    if sink.dtype != torch.int32 or not sink.is_cuda or sink.numel() < 1:
        raise ValueError("sink must be a CUDA int32 tensor")
    nbytes = buf.numel() * buf.element_size()
    _check(lib().mla_read_ceiling(buf.data_ptr(), nbytes, sink.data_ptr(), _stream(stream)),
           "mla_read_ceiling")


def trace_begin(max_records: int) -> None:
    """Start timing the main decode kernel of every call on this thread."""
    _check(lib().mla_trace_begin(int(max_records)), "mla_trace_begin")


def trace_end():
    """Stop tracing; returns (summed main-kernel ms, timed launches, kernel launches)."""
    ms = ctypes.c_float(0)
    n = ctypes.c_int32(0)
    k = ctypes.c_int32(0)
    _check(lib().mla_trace_end(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(k)), "mla_trace_end")
    return float(ms.value), int(n.value), int(k.value)
