"""Shared helpers of the GPU parity tests: seeded caches in oracle form and on
the device, and the acceptance check.

Acceptance (floats): max |gpu - ref| <= 1e-2 * max |ref| and
||gpu - ref||_2 <= 5e-3 * ||ref||_2, applied to the outputs and, separately,
to the log-sum-exps (finite entries; -inf must match exactly).  Integer and
byte results (FP8 codes, scales, gather lists) must match bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import mla_latent_kv_07_gb300 as mla
from mla_latent_kv_07_gb300 import inputs
from oracle import oracle as orc

MAX_REL = 1e-2
L2_REL = 5e-3


def bits(t):
    return inputs.bf16_bits(t)


def oracle_cache(kv_bf16: torch.Tensor, pe_bf16: torch.Tensor, fmt: int) -> dict:
    kv = bits(kv_bf16)
    pe = bits(pe_bf16)
    if fmt == 0:
        return {"fmt": 0, "kv": kv, "pe": pe}
    q, s = orc.quantize_rows(kv, pow2=fmt == 2)
    return {"fmt": fmt, "kv": q, "kv_scale": s, "pe": pe}


def device_cache(oc: dict) -> mla.Cache:
    B, S = oc["kv"].shape[:2]
    if oc["fmt"] == 0:
        kv = torch.from_numpy(oc["kv"].view(np.int16)).view(torch.bfloat16).cuda()
        return mla.Cache(B, S, 0, kv=kv, pe=_pe(oc))
    kv = torch.from_numpy(oc["kv"]).cuda()
    sc = torch.from_numpy(oc["kv_scale"]).cuda()
    return mla.Cache(B, S, oc["fmt"], kv=kv, kv_scale=sc, pe=_pe(oc))


def _pe(oc):
    return torch.from_numpy(oc["pe"].view(np.int16)).view(torch.bfloat16).cuda()


def workload_cache(w: inputs.Workload):
    """Seeded bf16 rows of a workload -> (oracle cache, device cache)."""
    oc = oracle_cache(inputs.latent_rows(w), inputs.rotary_rows(w), w.fmt)
    return oc, device_cache(oc)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_close(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern differs"
    g, r = got[~ninf], ref[~ninf]
    if r.size == 0:
        return
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    scale = np.abs(r).max()
    err = np.abs(g - r)
    max_rel = err.max() / scale if scale > 0 else err.max()
    l2 = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    assert max_rel <= MAX_REL and l2 <= L2_REL, f"{what}: max_rel={max_rel:.3e} l2_rel={l2:.3e}"
    return max_rel, l2


def sample_pairs(B: int, H: int, per_seq: int, seed: int) -> np.ndarray:
    """(b, h) output pairs to check at full size: for every sequence the first
    and last heads (0 and H - 1) plus `per_seq` further heads drawn uniformly
    without replacement from 1 .. H - 2 (all of them when fewer remain)."""
    rng = np.random.default_rng(seed)
    pairs = []
    inner = np.arange(1, H - 1)
    for b in range(B):
        pick = rng.choice(inner, size=min(per_seq, inner.size), replace=False) if inner.size else []
        hs = sorted({0, H - 1} | {int(h) for h in pick})
        pairs += [(b, h) for h in hs]
    return np.array(pairs, np.int32)
