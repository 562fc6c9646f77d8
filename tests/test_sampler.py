"""The full-size parity tests check sampled (sequence, head) outputs; this pins
the sampler itself (CPU only): every sequence includes the first and the last
head, the other heads are distinct and spread over the whole range."""
import numpy as np

from mla_cases import sample_pairs


def test_every_sequence_has_first_and_last_head():
    for B, H, per_seq, seed in [(8, 128, 6, 2), (32, 128, 8, 3), (4, 128, 4, 4), (1, 16, 20, 1)]:
        pairs = sample_pairs(B, H, per_seq, seed)
        for b in range(B):
            hs = pairs[pairs[:, 0] == b, 1]
            assert 0 in hs and H - 1 in hs
            assert len(set(hs.tolist())) == len(hs)
            assert len(hs) == min(H, per_seq + 2)
            assert hs.min() >= 0 and hs.max() <= H - 1


def test_heads_spread_over_the_range():
    # uniform draws: across the workload-3 sample the upper half of the heads
    # is hit about as often as the lower half
    pairs = sample_pairs(32, 128, 8, 3)
    inner = pairs[(pairs[:, 1] > 0) & (pairs[:, 1] < 127), 1]
    upper = np.count_nonzero(inner >= 64)
    assert 0.35 * inner.size <= upper <= 0.65 * inner.size
    assert inner.max() >= 120 and inner.min() <= 7
