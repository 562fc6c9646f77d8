"""CPU oracle for absorbed MLA decode over a latent KV cache -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  The library (``mla_latent_kv_07_gb300``) never does,
and the two share no code: this file wraps ``mla_oracle.c`` (plain C, fp64
attention, fp32 where the cache-write step fixes it) through ctypes.

Array conventions: bf16 values travel as ``np.uint16`` bit patterns, FP8 codes
as ``np.uint8``, scales as ``np.float32``; results are ``np.float64``.

Sources: "DeepSeek-V3.2-Exp . KV cache" (cache-write and MQA-decode excerpts),
"DeepSeek MLA architecture: how Multi-Head Latent Attention cuts KV cache by
93%" sections 3-4 (decoupled rotary term, matrix absorption).  The readings
taken where the pages are silent are listed at the top of ``mla_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

DC, DR, BLK = 512, 64, 128
NBLK = DC // BLK


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C, no FMA contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.orc_e4m3_encode_array.argtypes = [P, I64, P]
            lib.orc_e4m3_value_array.argtypes = [P, I64, P]
            lib.orc_f32_to_bf16_array.argtypes = [P, I64, P]
            lib.orc_quantize_rows.argtypes = [P, I64, P, P, I32]
            lib.orc_dequant_rows.argtypes = [P, P, I64, P]
            lib.orc_sparse_gather_lists.argtypes = [P, I32, I32, P, P, P]
            lib.orc_decode_absorbed.argtypes = [I32, I64, P, P, P, P, P, I32, P, P, I32, D,
                                                P, I32, P, P, P, I64]
            lib.orc_decode_absorbed.restype = I32
            lib.orc_decode_naive.argtypes = [I32, I64, P, P, P, P, P, P, I32, I32, P, D, P, P]
            lib.orc_decode_naive.restype = I32
            lib.orc_num_threads.restype = I32
            lib.orc_set_num_threads.argtypes = [I32]
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats

def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's OpenMP loops from here on (timing only)."""
    _load().orc_set_num_threads(int(n))


def e4m3_encode(y) -> np.ndarray:
    """fp32 -> E4M3 code, nearest-even, saturating to +-448."""
    y = _c(y, np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().orc_e4m3_encode_array(_p(y), y.size, _p(out))
    return out


def e4m3_value(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_e4m3_value_array(_p(codes), codes.size, _p(out))
    return out


def bf16_round(f) -> np.ndarray:
    """fp32 -> bf16 bit pattern, nearest-even."""
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().orc_f32_to_bf16_array(_p(f), f.size, _p(out))
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------ cache-write step

def quantize_rows(x_bits, pow2: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Latent rows [..., 512] (bf16 bits) -> (codes [..., 512] u8, scales [..., 4] f32).

    ``pow2`` selects the power-of-two scale format: each block's scale is the
    smallest power of two >= fp32(amax / 448) (the cache-write excerpt of
    "DeepSeek-V3.2-Exp . KV cache" passes a scale format to act_quant without
    defining it; this is the exponent-only reading)."""
    x = _c(x_bits, np.uint16)
    assert x.shape[-1] == DC
    n = x.size // DC
    q = np.empty(x.shape, np.uint8)
    s = np.empty(x.shape[:-1] + (NBLK,), np.float32)
    _load().orc_quantize_rows(_p(x), n, _p(q), _p(s), 1 if pow2 else 0)
    return q, s


def dequant_rows(q, scales) -> np.ndarray:
    """(codes, scales) -> the bf16 latent the decode attends to (bits)."""
    q = _c(q, np.uint8)
    s = _c(scales, np.float32)
    n = q.size // DC
    assert s.size == n * NBLK
    out = np.empty(q.shape, np.uint16)
    _load().orc_dequant_rows(_p(q), _p(s), n, _p(out))
    return out


def cache_append(cache: dict, kv_new_bits, pe_new_bits, start_pos) -> None:
    """Write row start_pos[b] of every sequence b < B, in place.

    ``cache`` holds numpy arrays: 'fmt' (0 bf16, 1 fp8, 2 fp8 with
    power-of-two scales), 'kv', 'pe' and, for fmt 1 and 2, 'kv_scale'.  bf16
    rows are copied; FP8 rows are block-quantised.
    A start_pos outside [0, max_seq_len) raises (the library refuses it too).
    """
    kv_new = _c(kv_new_bits, np.uint16).reshape(-1, DC)
    pe_new = _c(pe_new_bits, np.uint16).reshape(-1, DR)
    S = cache["kv"].shape[1]
    for b, t in enumerate(np.asarray(start_pos).reshape(-1)):
        if not 0 <= t < S:
            raise IndexError(f"start_pos {t} outside [0, {S})")
        if cache["fmt"] == 0:
            cache["kv"][b, t] = kv_new[b]
        else:
            q, s = quantize_rows(kv_new[b:b + 1], pow2=cache["fmt"] == 2)
            cache["kv"][b, t] = q[0]
            cache["kv_scale"][b, t] = s[0]
        cache["pe"][b, t] = pe_new[b]


# ------------------------------------------------------ gather indices

def sparse_gather_lists(topk, end_pos) -> tuple[np.ndarray, np.ndarray]:
    """Per sequence: sorted unique top-k entries in [0, end_pos); -1 padded."""
    topk = _c(topk, np.int32)
    B, K = topk.shape
    ep = _c(end_pos, np.int32)
    gidx = np.empty((B, K), np.int32)
    gcount = np.empty((B,), np.int32)
    _load().orc_sparse_gather_lists(_p(topk), B, K, _p(ep), _p(gidx), _p(gcount))
    return gidx, gcount


def topk_select(scores, end_pos, K: int) -> np.ndarray:
    """Top-k position selection per sequence (the ``topk_indices`` the V3.2
    sparse decode consumes, "DeepSeek-V3.2-Exp . KV cache", MQA-decode
    excerpt: an index list per sequence that the mask keeps).  The pages show
    only the call, not the scoring; the selection taken here is its plainest
    reading: among positions 0 .. end_pos[b]-1 of row b of ``scores`` [B, S]
    (fp32), the K with the largest score; equal scores go to the lower
    position; -0 equals +0; NaN ranks below -inf.  Returns int32 [B, K]: the
    selected positions in increasing order, then -1 (fewer than K valid)."""
    s = np.asarray(scores, np.float32)
    B, S = s.shape
    ep = np.asarray(end_pos).reshape(-1)
    out = np.full((B, K), -1, np.int32)
    for b in range(B):
        T = int(min(max(int(ep[b]), 0), S))
        row = s[b, :T].astype(np.float64)
        nan = np.isnan(row)
        neg = np.where(nan, 0.0, -row)            # score descending; -0 == +0
        order = np.lexsort((np.arange(T), neg, nan))   # last key first: non-NaN, score, position
        sel = np.sort(order[:K])
        out[b, :sel.size] = sel
    return out


# ------------------------------------------------------ absorbed decode

def decode_absorbed(cache: dict, q_latent, q_pe, end_pos, softmax_scale: float,
                    pairs=None, topk=None, weights_upto: int = 0):
    """fp64 absorbed decode.

    q_latent [B, H, 512] and q_pe [B, H, 64] are bf16 bits (uint16) or exact
    floats; ``pairs`` is an [n, 2] array of (b, h) to evaluate (default all).
    Returns (out [n, 512] f64, lse [n] f64) and, if ``weights_upto`` > 0, the
    attention weights [n, weights_upto] of positions 0..weights_upto-1.
    """
    ql = np.asarray(q_latent)
    qp = np.asarray(q_pe)
    if ql.dtype == np.uint16:
        ql = bf16_bits_to_f64(ql)
    if qp.dtype == np.uint16:
        qp = bf16_bits_to_f64(qp)
    ql = _c(ql, np.float64)
    qp = _c(qp, np.float64)
    B, H, dc = ql.shape
    assert dc == DC and qp.shape == (B, H, DR)
    if pairs is None:
        pairs = np.array([(b, h) for b in range(B) for h in range(H)], np.int32)
    pairs = _c(pairs, np.int32).reshape(-1, 2)
    n = pairs.shape[0]
    kv = np.ascontiguousarray(cache["kv"])
    pe = _c(cache["pe"], np.uint16)
    S = kv.shape[1]
    scale = None
    if cache["fmt"] in (1, 2):
        scale = _c(cache["kv_scale"], np.float32)
    ep = _c(end_pos, np.int32)
    K = 0
    if topk is not None:
        topk = _c(topk, np.int32)
        K = topk.shape[1]
    out = np.empty((n, DC), np.float64)
    lse = np.empty((n,), np.float64)
    w = np.empty((n, weights_upto), np.float64) if weights_upto > 0 else None
    err = _load().orc_decode_absorbed(int(cache["fmt"]), S, _p(kv), _p(scale), _p(pe),
                                      _p(ql), _p(qp), H, _p(ep), _p(topk), K,
                                      float(softmax_scale), _p(pairs), n, _p(out), _p(lse),
                                      _p(w), weights_upto)
    if err:
        raise MemoryError("oracle allocation failed")
    return (out, lse, w) if w is not None else (out, lse)


def decode_absorbed_mtp(cache: dict, q_latent, q_pe, end_pos, softmax_scale: float,
                        token=None, pairs=None):
    """fp64 absorbed decode of s new tokens per sequence (multi-token decode).

    q_latent [B, s, H, 512], q_pe [B, s, H, 64].  The s new tokens of sequence
    b sit at positions end_pos[b]-s .. end_pos[b]-1; token j attends to the
    cache positions up to and including its own: 0 .. end_pos[b]-s+j.  This
    causal reading is not printed on the pages: the MQA-decode excerpt of
    "DeepSeek-V3.2-Exp . KV cache" scores every token of the step against all
    of kv_cache[:bsz, :end_pos] and adds only the top-k index mask; the reading
    follows from decoding token by token (a token never sees later ones) and
    from the `mask` argument that excerpt hands to its indexer.  That is the single-token
    decode with end_pos[b] - (s-1-j) (a token with no position attends to
    nothing: out 0, lse -inf).  Returns (out [B, s, H, 512], lse [B, s, H]);
    with ``token`` = j, only token j, for the (b, h) ``pairs`` (default all):
    (out [n, 512], lse [n]).
    """
    ql = np.asarray(q_latent)
    qp = np.asarray(q_pe)
    B, s, H = ql.shape[:3]
    ep = np.asarray(end_pos, np.int64)
    if token is not None:
        e = np.maximum(ep - (s - 1 - token), 0).astype(np.int32)
        return decode_absorbed(cache, np.ascontiguousarray(ql[:, token]), np.ascontiguousarray(qp[:, token]),
                               e, softmax_scale, pairs=pairs)
    out = np.empty((B, s, H, DC), np.float64)
    lse = np.empty((B, s, H), np.float64)
    for j in range(s):
        e = np.maximum(ep - (s - 1 - j), 0).astype(np.int32)
        o, l = decode_absorbed(cache, np.ascontiguousarray(ql[:, j]), np.ascontiguousarray(qp[:, j]), e,
                               softmax_scale)
        out[:, j] = o.reshape(B, H, DC)
        lse[:, j] = l.reshape(B, H)
    return out, lse


def _f64(x):
    x = np.asarray(x)
    return bf16_bits_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def absorb_q(q_nope, wkv_b):
    """fp64 q_latent[b, h, c] = sum_n q_nope[b, h, n] * W_UK[h, n, c], with
    W_UK[h] = wkv_b[h, 0:128, :] ("DeepSeek MLA architecture ...", section 4:
    the key up-projection folded into the query).  Inputs: bf16 bits or floats."""
    q = _f64(q_nope)
    w = _f64(wkv_b)
    return np.einsum("bhn,hnc->bhc", q, w[:, :128, :])


def project_out(x, wkv_b):
    """fp64 o[b, h, v] = sum_c W_UV[h, v, c] * x[b, h, c], with W_UV[h] =
    wkv_b[h, 128:256, :] (the value up-projection applied after the latent
    attention).  Inputs: bf16 bits or floats."""
    xx = _f64(x)
    w = _f64(wkv_b)
    return np.einsum("bhc,hvc->bhv", xx, w[:, 128:, :])


def decode_naive(cache: dict, wkv_b, q_nope, q_pe, end_pos, softmax_scale: float):
    """fp64 non-absorbed MHA: keys/values expanded through wkv_b [H, 256, 512].

    Returns (o [B, H, 128], lse [B, H]).  Tiny inputs only.
    """
    w = _c(wkv_b, np.float64)
    qn = _c(q_nope, np.float64)
    qp = np.asarray(q_pe)
    if qp.dtype == np.uint16:
        qp = bf16_bits_to_f64(qp)
    qp = _c(qp, np.float64)
    B, H, _ = qn.shape
    kv = np.ascontiguousarray(cache["kv"])
    pe = _c(cache["pe"], np.uint16)
    scale = _c(cache["kv_scale"], np.float32) if cache["fmt"] in (1, 2) else None
    ep = _c(end_pos, np.int32)
    o = np.empty((B, H, 128), np.float64)
    lse = np.empty((B, H), np.float64)
    err = _load().orc_decode_naive(int(cache["fmt"]), kv.shape[1], _p(kv), _p(scale), _p(pe),
                                   _p(w), _p(qn), _p(qp), B, H, _p(ep), float(softmax_scale),
                                   _p(o), _p(lse))
    if err:
        raise MemoryError("oracle allocation failed")
    return o, lse
