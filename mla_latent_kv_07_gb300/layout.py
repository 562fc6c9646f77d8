"""Cache layout constants and the algorithmic byte / flop accounting.

Layouts (row-major, caller-owned, one slot per sequence):
  bf16 cache: kv [Bmax, S, 512] bf16, pe [Bmax, S, 64] bf16
  FP8  cache: kv [Bmax, S, 512] e4m3 bytes, kv_scale [Bmax, S, 4] fp32
              (one scale per 128-wide block of the latent), pe [Bmax, S, 64] bf16

The latent width 512 (kv_lora_rank) and rotary width 64 (qk_rope_head_dim)
are the DeepSeek-V3 values ("How Multi-Head Latent Attention (MLA) Reduces KV
Cache Memory in DeepSeek-V3", "Memory Savings Analysis": 512 + 64 = 576
values per position).
"""
DC = 512     # latent width
DR = 64      # rotary key width
BLK = 128    # FP8 block width
NBLK = DC // BLK


def latent_bytes(tokens: int, fmt: int) -> int:
    """Bytes of the latent part alone (no rotary key, no scales)."""
    return tokens * DC * (2 if fmt == 0 else 1)


def cache_bytes_per_token(fmt: int) -> int:
    """Bytes the decode reads per attended position: latent + rotary (+ scales).
    bf16: 1024 + 128 = 1152; FP8: 512 + 128 + 16 = 656."""
    return DC * 2 + DR * 2 if fmt == 0 else DC + DR * 2 + NBLK * 4


def flops_per_token(H: int) -> int:
    """Score (576-wide dot) and value sum (512-wide axpy) per head and position."""
    return 2 * H * (DC + DR) + 2 * H * DC


def step_bytes(tokens_total: int, B: int, H: int, fmt: int) -> int:
    """Algorithmic HBM bytes of one decode call: every attended cache position
    once, plus the queries in and the bf16 outputs out."""
    return (tokens_total * cache_bytes_per_token(fmt)
            + B * H * (DC + DR) * 2 + B * H * DC * 2)


def step_flops(tokens_total: int, H: int) -> int:
    return tokens_total * flops_per_token(H)
