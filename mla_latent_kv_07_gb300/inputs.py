"""Seeded synthetic inputs and the named workloads.

This module holds no arithmetic of the method: it only draws random tensors
(bf16 N(0,1) latents, rotary keys and queries; sequence lengths; top-k index
lists) with fixed seeds, and describes the five workloads by their sizes.  The
tests feed the same tensors to the CPU oracle and to the CUDA library; the
benchmark draws them on the device.

Seeding: every tensor of workload ``w`` (1-based) uses its own generator seed
``1000 * w + tensor_id`` with the ids below, so any tensor can be redrawn
alone.  Values are float32 N(0,1) rounded to bf16 by torch's cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DC, DR, BLK = 512, 64, 128

T_KV, T_PE, T_QL, T_QP, T_LEN, T_TOPK, T_KVNEW, T_PENEW = range(1, 9)
T_QNOPE, T_WKVB = 10, 11   # q_nope and wkv_b (workloads with the absorption products)

# 1/sqrt(qk_nope_head_dim + qk_rope_head_dim) = 1/sqrt(128 + 64), and the YaRN
# attention-scale correction (0.1 * mscale * ln(rope_factor) + 1)^2 with the
# page defaults rope_factor = 40, mscale = 1.
SCALE_BASE = 192.0 ** -0.5
SCALE_YARN = SCALE_BASE * (0.1 * 1.0 * math.log(40.0) + 1.0) ** 2


@dataclass(frozen=True)
class Workload:
    index: int            # 1-based workload number; drives the seeds
    name: str
    B: int
    H: int
    S: int                # max_seq_len of the cache buffers
    fmt: int              # 0 = bf16 latent, 1 = FP8 e4m3 + per-128 fp32 scales
    softmax_scale: float
    T: int = 0            # fixed end_pos for every sequence (0: drawn)
    T_lo: int = 0         # drawn end_pos range (inclusive) when T == 0
    T_hi: int = 0
    topk: int = 0         # 0: dense decode
    append: bool = False  # a new row is appended at end_pos - 1 before decoding
    mtp: int = 1          # new tokens per sequence decoded at once (multi-token decode)
    absorb: bool = False  # the step also runs the query absorption and value projection
    notes: dict = field(default_factory=dict)


WORKLOADS = {
    1: Workload(1, "tiny_b1_h16_t256_bf16", B=1, H=16, S=256, fmt=0, softmax_scale=SCALE_BASE,
                T=256, notes={"append": "one FP8 row appended at start_pos 255 of a 1x256 FP8 cache"}),
    2: Workload(2, "v3_b8_h128_t4096_bf16", B=8, H=128, S=4096, fmt=0, softmax_scale=SCALE_YARN,
                T=4096),
    3: Workload(3, "serving_b32_h128_t1k-16k_fp8", B=32, H=128, S=16384, fmt=1,
                softmax_scale=SCALE_YARN, T_lo=1024, T_hi=16384),
    4: Workload(4, "longctx_b4_h128_t131072_fp8", B=4, H=128, S=131072, fmt=1,
                softmax_scale=SCALE_YARN, T=131072),
    5: Workload(5, "sparse_b16_h128_t32768_k2048_fp8", B=16, H=128, S=32768, fmt=1,
                softmax_scale=SCALE_YARN, T=32768, topk=2048, append=True),
    # beyond the headline table: workload 2 with two new tokens per sequence
    6: Workload(6, "mtp2_b8_h128_t4096_bf16", B=8, H=128, S=4096, fmt=0, softmax_scale=SCALE_YARN,
                T=4096, mtp=2),
    # a prefill chunk: 512 new tokens of one sequence over its 4096-position
    # prefix (causal among the chunk's tokens; the chunk's rows are in the cache)
    8: Workload(8, "prefill_chunk_b1_s512_h128_t4096_bf16", B=1, H=128, S=4096, fmt=0,
                softmax_scale=SCALE_YARN, T=4096, mtp=512),
    # workload 2 as a whole attention step: q_nope -> q_latent -> decode -> o
    7: Workload(7, "attn_b8_h128_t4096_bf16", B=8, H=128, S=4096, fmt=0, softmax_scale=SCALE_YARN,
                T=4096, absorb=True),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """float32 N(0,1) draws cast to bf16."""
    g = _gen(seed, device)
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def end_positions(w: Workload, device="cpu") -> torch.Tensor:
    if w.T:
        return torch.full((w.B,), w.T, dtype=torch.int32, device=device)
    g = _gen(1000 * w.index + T_LEN)
    return torch.randint(w.T_lo, w.T_hi + 1, (w.B,), generator=g, dtype=torch.int32).to(device)


def topk_indices(B: int, K: int, end_pos, seed: int) -> torch.Tensor:
    """Per sequence: K-1 distinct positions drawn from 0..T-2, plus T-1 (the
    newest position), in draw order.  Sequences shorter than K keep all of
    0..T-1 and pad with -1.  Returns int32 [B, K] on the CPU."""
    g = _gen(seed)
    out = torch.full((B, K), -1, dtype=torch.int32)
    for b in range(B):
        T = int(end_pos[b])
        if T <= 0:
            continue
        n = min(K - 1, T - 1)
        perm = torch.randperm(T - 1, generator=g)[:n].to(torch.int32)
        row = torch.cat([perm, torch.tensor([T - 1], dtype=torch.int32)])
        out[b, :row.numel()] = row
    return out


def queries(w: Workload, device="cpu", H: int | None = None):
    """q_latent, q_pe: [B, H, .] (or [B, mtp, H, .] for a multi-token workload)."""
    H = H or w.H
    lead = (w.B, H) if w.mtp == 1 else (w.B, w.mtp, H)
    ql = randn_bf16(lead + (DC,), 1000 * w.index + T_QL, device)
    qp = randn_bf16(lead + (DR,), 1000 * w.index + T_QP, device)
    return ql, qp


def latent_rows(w: Workload, device="cpu", S: int | None = None) -> torch.Tensor:
    """bf16 latent rows [B, S, 512]; the FP8 cache is made from these."""
    return randn_bf16((w.B, S or w.S, DC), 1000 * w.index + T_KV, device)


def rotary_rows(w: Workload, device="cpu", S: int | None = None) -> torch.Tensor:
    return randn_bf16((w.B, S or w.S, DR), 1000 * w.index + T_PE, device)


def new_rows(w: Workload, device="cpu"):
    """The rows appended by the cache-write step: kv_new [B, 512], pe_new [B, 64]."""
    return (randn_bf16((w.B, DC), 1000 * w.index + T_KVNEW, device),
            randn_bf16((w.B, DR), 1000 * w.index + T_PENEW, device))


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def absorb_inputs(w: Workload, device="cpu"):
    """q_nope [B, H, 128] (N(0,1)) and wkv_b [H, 256, 512] (N(0,1) * 0.05, as bf16)."""
    qn = randn_bf16((w.B, w.H, 128), 1000 * w.index + T_QNOPE, device)
    wkv = (randn_bf16((w.H, 256, DC), 1000 * w.index + T_WKVB, device).float() * 0.05).to(torch.bfloat16)
    return qn, wkv
