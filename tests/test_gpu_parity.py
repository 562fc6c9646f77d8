"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs, called through the C ABI (ctypes binding).  Small cases compare every
output and span several tiles with ragged tails; every benchmark workload
runs at its full size in the launch configuration the benchmark times and
compares sampled (sequence, token, head) outputs the oracle computes one by
one.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_07_gb300 as mla
from mla_latent_kv_07_gb300 import inputs
from oracle import oracle as orc

from mla_cases import (bits, check_close, device_cache, f64, oracle_cache, sample_pairs,
                       workload_cache)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_latent_kv_07_gb300 import build
    build.build()
    mla.lib()


def _rand_bf16(shape, seed):
    return inputs.randn_bf16(shape, seed)


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_append_bit_exact(fmt):
    B, S = 64, 300
    g = torch.Generator().manual_seed(7)
    kv_new = (torch.randn(B, 512, generator=g) * torch.exp(torch.randn(B, 1, generator=g) * 4)).to(torch.bfloat16)
    kv_new[0, :128] = 0.0                         # an all-zero block
    kv_new[1, 128:256] = 448.0                    # scale exactly 1
    kv_new[2, 256:384] = torch.tensor([2.0 ** -9, -2.0 ** -10] * 64)
    kv_new[4, 384:512] = torch.tensor([2.0 ** -132, -(2.0 ** -133)] * 64)   # subnormal fp32 scale
    kv_new[5, :128] = 450.0                       # power-of-two scale 2 (format 2)
    pe_new = _rand_bf16((B, 64), 8)
    start = np.random.default_rng(9).integers(0, S, B).astype(np.int32)
    start[3] = S - 1
    oc = oracle_cache(_rand_bf16((B, S, 512), 10), _rand_bf16((B, S, 64), 11), fmt)
    dc = device_cache(oc)
    mla.cache_append(dc, kv_new.cuda(), pe_new.cuda(), start)
    orc.cache_append(oc, bits(kv_new), bits(pe_new), start)
    torch.cuda.synchronize()
    if fmt == 0:
        assert np.array_equal(bits(dc.kv.cpu()), oc["kv"])
    else:
        assert np.array_equal(dc.kv.cpu().numpy(), oc["kv"])
        assert np.array_equal(dc.kv_scale.cpu().numpy().view(np.uint32), oc["kv_scale"].view(np.uint32))
    assert np.array_equal(bits(dc.pe.cpu()), oc["pe"])


def test_append_refuses_positions_past_the_cache():
    oc = oracle_cache(_rand_bf16((2, 8, 512), 1), _rand_bf16((2, 8, 64), 2), 1)
    dc = device_cache(oc)
    before = dc.kv.clone()
    with pytest.raises(mla.MLAError) as e:
        mla.cache_append(dc, _rand_bf16((2, 512), 3).cuda(), _rand_bf16((2, 64), 4).cuda(), [1, 8])
    assert e.value.code == 2
    torch.cuda.synchronize()
    assert torch.equal(before, dc.kv)


# ------------------------------------------------------------ small dense

SMALL = [  # (fmt, H, end_pos per sequence, S)
    (0, 16, [1, 31, 32, 33], 64),
    (1, 16, [100, 257, 5], 300),
    (0, 32, [64, 1, 200], 256),
    (1, 64, [129, 77], 160),
    (0, 128, [300, 33, 1], 320),
    (1, 128, [1000, 513, 2, 64], 1024),
    (2, 64, [129, 77], 160),                    # power-of-two scales: read like format 1
    (2, 128, [1000, 513, 2, 64], 1024),
]


@pytest.mark.parametrize("fmt,H,ends,S", SMALL)
def test_decode_small_all_outputs(fmt, H, ends, S):
    B = len(ends)
    seed = 100 * H + S + fmt
    oc = oracle_cache(_rand_bf16((B, S, 512), seed), _rand_bf16((B, S, 64), seed + 1), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), seed + 2), _rand_bf16((B, H, 64), seed + 3)
    end_pos = np.array(ends, np.int32)
    sm = 0.1352
    out, lse = mla.decode(dc, ql.cuda(), qp.cuda(), torch.from_numpy(end_pos).cuda(), S, sm)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), end_pos, sm)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


def test_rows_past_end_pos_are_never_used():
    # NaN codes, infinite scales and NaN rotary keys beyond end_pos
    B, S, H = 2, 200, 128
    oc = oracle_cache(_rand_bf16((B, S, 512), 21), _rand_bf16((B, S, 64), 22), 1)
    ends = np.array([77, 130], np.int32)
    for b, T in enumerate(ends):
        oc["kv"][b, T:] = 0x7F
        oc["kv_scale"][b, T:] = np.inf
        oc["pe"][b, T:] = 0x7FC0
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 23), _rand_bf16((B, H, 64), 24)
    out, lse = mla.decode(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.2)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.2)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


@pytest.mark.parametrize("fmt", [0, 1])
def test_rising_scores_rescale_mid_unit(fmt):
    # the latent rows drift along a fixed direction u, 100 units per 48
    # positions: a head whose query has q.u ~ 1 sees its maximum score rise by
    # ~19 (log2 units) every tile -- past the lazy-rescale threshold, so its
    # running reference and its rows of O are rescaled inside a unit (units
    # here span about four tiles), while heads with q.u < 0 keep their first
    # reference.  Each CTA of a pair owns half the heads and scales the other
    # half's rows of its own output half on the owner's request.
    B, S, H = 2, 8192, 128
    rng = np.random.default_rng(77 + fmt)
    u = rng.standard_normal(512)
    u /= np.linalg.norm(u)
    t = np.arange(S, dtype=np.float64)[None, :, None]
    kv = torch.from_numpy(rng.standard_normal((B, S, 512)) + 100.0 * (t / 48.0) * u[None, None, :]).float()
    kv_bf16 = kv.to(torch.bfloat16)
    oc = oracle_cache(kv_bf16, _rand_bf16((B, S, 64), 79), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 80), _rand_bf16((B, H, 64), 81)
    ends = np.array([8192, 6000], np.int32)
    out, lse = mla.decode(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.1352)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.1352)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


@pytest.mark.parametrize("fmt", [0, 1])
def test_single_unit_sequences_write_directly(fmt):
    # sequences of one or two tiles get a single unit, which writes the final
    # output (and lse, when asked) itself; the long one is split and combined
    B, S, H = 3, 512, 128
    oc = oracle_cache(_rand_bf16((B, S, 512), 91), _rand_bf16((B, S, 64), 92), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 93), _rand_bf16((B, H, 64), 94)
    ends = np.array([30, 96, 500], np.int32)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.16)
    for want_lse in (True, False):
        out, lse = mla.decode(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.16,
                              want_lse=want_lse)
        check_close(f64(out).reshape(-1, 512), ref, f"out (lse={want_lse})")
        if want_lse:
            check_close(f64(lse).reshape(-1), ref_lse, "lse")


def test_empty_and_clamped_sequences():
    B, S, H = 3, 64, 16
    oc = oracle_cache(_rand_bf16((B, S, 512), 31), _rand_bf16((B, S, 64), 32), 0)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 33), _rand_bf16((B, H, 64), 34)
    ends = torch.tensor([0, 40, 50], dtype=torch.int32).cuda()
    ws = mla.alloc_workspace(B, H, 48)
    out, lse = mla.decode(dc, ql.cuda(), qp.cuda(), ends, 48, 0.3, workspace=ws)
    flags = mla.workspace_status(ws)
    assert flags == mla.DEV_END_POS_CLAMPED           # 50 > max_end_pos 48
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), np.array([0, 40, 48], np.int32), 0.3)
    o = f64(out).reshape(-1, 512)
    assert (o[:H] == 0).all() and np.isneginf(f64(lse)[0]).all()
    check_close(o, ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")
    ends_ok = torch.tensor([0, 40, 48], dtype=torch.int32).cuda()
    mla.decode(dc, ql.cuda(), qp.cuda(), ends_ok, 48, 0.3, workspace=ws)
    assert mla.workspace_status(ws) == 0


# ------------------------------------------------- decode with the append

def _oracle_append(oc, kv_new, pe_new, seqs, pos):
    """The oracle's cache write of row pos[i] of sequence seqs[i] (numpy views
    of the oracle cache, so the rows land in place)."""
    for b, t in zip(seqs, pos):
        view = {k: (v[b:b + 1] if isinstance(v, np.ndarray) else v) for k, v in oc.items()}
        orc.cache_append(view, kv_new[b:b + 1], pe_new[b:b + 1], [int(t)])


APPEND_CASES = [  # (fmt, H, end_pos per sequence, max_end_pos, S)
    (0, 128, [1000, 33, 1, 700, 0], 1000, 1024),   # split, single-unit, one row, empty
    (1, 128, [1000, 513, 2, 64], 1000, 1024),
    (2, 128, [900, 47, 48, 49], 900, 960),          # tile edges around the new row
    (0, 64, [300, 1, 129], 300, 320),               # warp-MMA path: an append kernel of its own
    (1, 16, [100, 257, 5], 257, 300),
]


@pytest.mark.parametrize("fmt,H,ends,max_end,S", APPEND_CASES)
def test_decode_append_equals_append_then_decode(fmt, H, ends, max_end, S):
    # the call writes row end_pos - 1 exactly as mla_cache_append would and the
    # decode reads it: the cache-write and MQA-decode excerpts in that order
    B = len(ends)
    seed = 7 * H + S + fmt
    oc = oracle_cache(_rand_bf16((B, S, 512), seed), _rand_bf16((B, S, 64), seed + 1), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), seed + 2), _rand_bf16((B, H, 64), seed + 3)
    kv_new, pe_new = _rand_bf16((B, 512), seed + 4), _rand_bf16((B, 64), seed + 5)
    kv_new[0, :128] = 0.0                                  # an all-zero block
    end_pos = np.array(ends, np.int32)
    ws = mla.alloc_workspace(B, H, max_end)
    out, lse = mla.decode_append(dc, kv_new.cuda(), pe_new.cuda(), ql.cuda(), qp.cuda(),
                                 torch.from_numpy(end_pos).cuda(), max_end, 0.11, workspace=ws)
    ok = (end_pos >= 1) & (end_pos <= max_end)
    _oracle_append(oc, bits(kv_new), bits(pe_new), np.flatnonzero(ok), end_pos[ok] - 1)
    torch.cuda.synchronize()
    if fmt == 0:
        assert np.array_equal(bits(dc.kv.cpu()), oc["kv"])
    else:
        assert np.array_equal(dc.kv.cpu().numpy(), oc["kv"])
        assert np.array_equal(dc.kv_scale.cpu().numpy().view(np.uint32), oc["kv_scale"].view(np.uint32))
    assert np.array_equal(bits(dc.pe.cpu()), oc["pe"])
    want = (0 if ok.all() else mla.DEV_APPEND_SKIPPED) | \
        (0 if ((end_pos >= 0) & (end_pos <= max_end)).all() else mla.DEV_END_POS_CLAMPED)
    assert mla.workspace_status(ws) == want
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), np.clip(end_pos, 0, max_end), 0.11)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


def test_decode_append_skips_clamped_rows():
    # end_pos past max_end_pos: decoded clamped, row not written, both flagged
    B, S, H = 2, 256, 128
    oc = oracle_cache(_rand_bf16((B, S, 512), 141), _rand_bf16((B, S, 64), 142), 1)
    dc = device_cache(oc)
    before = dc.kv.clone(), dc.kv_scale.clone(), dc.pe.clone()
    ql, qp = _rand_bf16((B, H, 512), 143), _rand_bf16((B, H, 64), 144)
    kv_new, pe_new = _rand_bf16((B, 512), 145), _rand_bf16((B, 64), 146)
    ends = torch.tensor([200, 150], dtype=torch.int32).cuda()       # max_end_pos 160
    ws = mla.alloc_workspace(B, H, 160)
    out, lse = mla.decode_append(dc, kv_new.cuda(), pe_new.cuda(), ql.cuda(), qp.cuda(), ends, 160, 0.2,
                                 workspace=ws)
    assert mla.workspace_status(ws) == mla.DEV_APPEND_SKIPPED | mla.DEV_END_POS_CLAMPED
    torch.cuda.synchronize()
    assert torch.equal(dc.kv[0], before[0][0]) and torch.equal(dc.pe[0], before[2][0])
    _oracle_append(oc, bits(kv_new), bits(pe_new), [1], [149])
    assert np.array_equal(dc.kv[1].cpu().numpy(), oc["kv"][1])
    assert np.array_equal(dc.kv_scale[1].cpu().numpy().view(np.uint32), oc["kv_scale"][1].view(np.uint32))
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), np.array([160, 150], np.int32), 0.2)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


SCHEDULE_CASES = [  # (end_pos per slot, max_end_pos, S, new tokens per slot)
    ([4096] * 8, 4096, 4096, 1),
    ([1, 0, 5000, 37, 4096, 48, 49, 2000, 3000], 4096, 4096, 1),    # empty, clamped, tile edges
    (list(np.random.default_rng(151).integers(0, 1000, 33)), 900, 1000, 1),   # two lane blocks
    (list(np.random.default_rng(152).integers(0, 300, 128)), 256, 300, 1),    # the warp's limit
    ([100, 3, 2, 50, 0], 128, 128, 3),                              # multi-token
]


@pytest.mark.parametrize("ends,max_end,S,s", SCHEDULE_CASES)
def test_kernel_schedule_matches_schedule_kernel(ends, max_end, S, s):
    # dense bf16 calls (H = 128, up to 128 sequences) compute the split
    # schedule inside the decode kernel; FP8 calls run the schedule kernel.
    # Both follow one rule, so for the same end_pos the workspace's status
    # word, unit count and per-sequence table must agree byte for byte.
    B, H = len(ends), 128
    end_pos = torch.tensor(ends, dtype=torch.int32).cuda()
    tables = []
    for fmt in (0, 1):
        dc = mla.Cache(B, S, fmt)
        ql = _rand_bf16((B * s, H, 512), 153).cuda() if s == 1 else _rand_bf16((B, s, H, 512), 153).cuda()
        qp = _rand_bf16((B * s, H, 64), 154).cuda() if s == 1 else _rand_bf16((B, s, H, 64), 154).cuda()
        ws = mla.alloc_workspace(B * s, H, max_end)
        if s == 1:
            kv_new, pe_new = _rand_bf16((B, 512), 155).cuda(), _rand_bf16((B, 64), 156).cuda()
            mla.decode_append(dc, kv_new, pe_new, ql, qp, end_pos, max_end, 0.1, workspace=ws)
        else:
            mla.decode_mtp(dc, ql, qp, end_pos, max_end, 0.1, workspace=ws)
        torch.cuda.synchronize()
        tables.append(ws[:256 + 8 * B * s].cpu().numpy())
    hdr = [tb[:8].view(np.int32) for tb in tables]
    assert hdr[0][0] == hdr[1][0] and hdr[0][1] == hdr[1][1], hdr
    assert np.array_equal(tables[0][256:], tables[1][256:])
    seq = tables[0][256:].view(np.int32).reshape(-1, 2)
    assert (seq[:, 1] >= -1).all() and hdr[0][1] >= int((seq[:, 1] != 0).sum())


def test_sparse_kernel_schedule_matches_schedule_kernel():
    # sparse calls of up to 128 sequences compute the split schedule inside the
    # decode kernel from the gather counts; a dense FP8 call with end_pos equal
    # to those counts runs the schedule kernel on the same lengths, so the
    # status word, unit count and per-sequence table must agree byte for byte
    counts = [0, 1, 47, 48, 49, 700, 2048, 95, 96, 1500, 3, 333, 2047, 1024, 511, 5, 0, 1999]
    B, H, S, K = len(counts), 128, 4096, 2048
    rng = np.random.default_rng(157)
    topk = np.full((B, K), -1, np.int32)
    for b, c in enumerate(counts):
        topk[b, :c] = rng.permutation(S)[:c]
    ql, qp = _rand_bf16((B, H, 512), 158).cuda(), _rand_bf16((B, H, 64), 159).cuda()
    tables = []
    ws = mla.alloc_workspace(B, H, S, K)
    mla.decode_sparse(mla.Cache(B, S, 1), ql, qp, torch.full((B,), S, dtype=torch.int32).cuda(), S, 0.1,
                      torch.from_numpy(topk).cuda(), workspace=ws)
    torch.cuda.synchronize()
    tables.append(ws[:256 + 8 * B].cpu().numpy())
    ws = mla.alloc_workspace(B, H, S)
    mla.decode(mla.Cache(B, S, 1), ql, qp, torch.tensor(counts, dtype=torch.int32).cuda(), S, 0.1, workspace=ws)
    torch.cuda.synchronize()
    tables.append(ws[:256 + 8 * B].cpu().numpy())
    hdr = [tb[:8].view(np.int32) for tb in tables]
    assert hdr[0][0] == hdr[1][0] and hdr[0][1] == hdr[1][1], hdr
    assert np.array_equal(tables[0][256:], tables[1][256:])


def test_sparse_more_sequences_than_the_in_kernel_schedule_takes():
    # 130 sequences: the sparse call runs the schedule kernel (the in-kernel
    # schedule holds at most 128 lengths); sampled outputs against the oracle
    B, S, H, K = 130, 512, 128, 64
    oc = oracle_cache(_rand_bf16((B, S, 512), 161), _rand_bf16((B, S, 64), 162), 1)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 163), _rand_bf16((B, H, 64), 164)
    rng = np.random.default_rng(165)
    ends = rng.integers(1, S + 1, B).astype(np.int32)
    topk = rng.integers(-1, S, (B, K)).astype(np.int32)
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.13,
                                 torch.from_numpy(topk).cuda())
    pairs = sample_pairs(B, H, 2, seed=166)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.13, pairs=pairs, topk=topk)
    got = f64(out).reshape(B, H, 512)[pairs[:, 0], pairs[:, 1]]
    check_close(got, ref, "out")
    check_close(f64(lse).reshape(B, H)[pairs[:, 0], pairs[:, 1]], ref_lse, "lse")


@pytest.mark.parametrize("fmt", [0, 1])
def test_bounded_wait_runs_out_and_reports(fmt):
    # the self-test withholds the first unit's first tile: its waits run out
    # (milliseconds), the status word says so, the call completes, and the
    # next decode on the same device and workspace is correct
    B, S, H = 2, 300, 128
    oc = oracle_cache(_rand_bf16((B, S, 512), 131), _rand_bf16((B, S, 64), 132), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 133).cuda(), _rand_bf16((B, H, 64), 134).cuda()
    ends = torch.tensor([300, 200], dtype=torch.int32).cuda()
    ws = mla.alloc_workspace(B, H, S)
    flags = mla.selftest_decode_timeout(dc, ql, qp, ends, S, 0.2, ws)
    assert flags & mla.DEV_PIPELINE_TIMEOUT
    out, lse = mla.decode(dc, ql, qp, ends, S, 0.2, workspace=ws)
    assert mla.workspace_status(ws) == 0
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql.cpu()), bits(qp.cpu()), ends.cpu().numpy(), 0.2)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


def test_workspace_too_small_is_refused():
    oc = oracle_cache(_rand_bf16((1, 32, 512), 41), _rand_bf16((1, 32, 64), 42), 0)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((1, 16, 512), 43).cuda(), _rand_bf16((1, 16, 64), 44).cuda()
    ws = torch.empty(mla.workspace_size(1, 16, 32) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode(dc, ql, qp, torch.tensor([32], dtype=torch.int32).cuda(), 32, 0.1, workspace=ws)
    assert e.value.code == 4


def test_read_ceiling_reads_every_word():
    # the streaming read kernel folds every 32-bit word: its XOR equals the
    # XOR of the buffer (an odd length exercises the tail loop)
    rng = np.random.default_rng(81)
    words = rng.integers(0, 2**32, size=(1 << 22) + 4 * 37, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.read_ceiling(buf, sink)
    torch.cuda.synchronize()
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(np.bitwise_xor.reduce(words))


# ------------------------------------------------------ multi-token decode

@pytest.mark.parametrize("fmt,H,s", [(0, 128, 2), (1, 128, 3), (0, 16, 2), (1, 64, 4), (0, 128, 40),
                                     (1, 16, 24)])
def test_multi_token_decode_all_outputs(fmt, H, s):
    B, S = 3, 300
    oc = oracle_cache(_rand_bf16((B, S, 512), 101), _rand_bf16((B, S, 64), 102), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, s, H, 512), 103), _rand_bf16((B, s, H, 64), 104)
    ends = np.array([300, 97, 2], np.int32)      # the last: the first tokens see nothing or one row
    out, lse = mla.decode_mtp(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.14)
    ref, ref_lse = orc.decode_absorbed_mtp(oc, bits(ql), bits(qp), ends, 0.14)
    check_close(f64(out).reshape(-1, 512), ref.reshape(-1, 512), "out")
    check_close(f64(lse).reshape(-1), ref_lse.reshape(-1), "lse")


@pytest.mark.parametrize("fmt", [0, 1])
def test_prefill_chunk_more_tokens_than_units(fmt):
    # 200 causal tokens over a 520-position prefix: more (token) sequences than
    # CTA pairs in a wave, so every sequence is one unit and the schedule's
    # unit count is the count of sequences
    B, S, H, s = 1, 520, 128, 200
    oc = oracle_cache(_rand_bf16((B, S, 512), 121), _rand_bf16((B, S, 64), 122), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, s, H, 512), 123), _rand_bf16((B, s, H, 64), 124)
    ends = np.array([S], np.int32)
    ws = mla.alloc_workspace(B * s, H, S)
    out, lse = mla.decode_mtp(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.1, workspace=ws)
    torch.cuda.synchronize()
    header = ws[:8].cpu().numpy().view(np.int32)
    assert header[0] == 0 and header[1] == B * s
    ref, ref_lse = orc.decode_absorbed_mtp(oc, bits(ql), bits(qp), ends, 0.1)
    check_close(f64(out).reshape(-1, 512), ref.reshape(-1, 512), "out")
    check_close(f64(lse).reshape(-1), ref_lse.reshape(-1), "lse")


def test_multi_token_decode_with_one_token_is_the_decode():
    B, S, H = 2, 160, 128
    oc = oracle_cache(_rand_bf16((B, S, 512), 111), _rand_bf16((B, S, 64), 112), 1)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 113), _rand_bf16((B, H, 64), 114)
    ends = torch.tensor([160, 61], dtype=torch.int32).cuda()
    o1, l1 = mla.decode(dc, ql.cuda(), qp.cuda(), ends, S, 0.2)
    om, lm = mla.decode_mtp(dc, ql.view(B, 1, H, 512).cuda(), qp.view(B, 1, H, 64).cuda(), ends, S, 0.2)
    assert torch.equal(o1, om.view(B, H, 512)) and torch.equal(l1, lm.view(B, H))


# ---------------------------------------------------------- small sparse

def test_sparse_small_lists_and_outputs():
    B, S, H, K = 4, 400, 128, 96
    oc = oracle_cache(_rand_bf16((B, S, 512), 51), _rand_bf16((B, S, 64), 52), 1)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 53), _rand_bf16((B, H, 64), 54)
    ends = np.array([400, 37, 1, 250], np.int32)
    rng = np.random.default_rng(55)
    topk = rng.integers(-2, 420, (B, K)).astype(np.int32)
    topk[1, :40] = np.arange(40)                    # covers all of a short sequence (with extras)
    topk[3, 10:20] = topk[3, 0]                     # repeats
    gidx = torch.empty((B, K), dtype=torch.int32, device="cuda")
    gcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.15,
                                 torch.from_numpy(topk).cuda(), gidx=gidx, gcount=gcnt)
    ref_g, ref_c = orc.sparse_gather_lists(topk, ends)
    assert np.array_equal(gidx.cpu().numpy(), ref_g) and np.array_equal(gcnt.cpu().numpy(), ref_c)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.15, topk=topk)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


def test_sparse_empty_split_and_single_unit_sequences():
    # one sequence with nothing to gather (every entry -1 or out of range), one
    # long list split over several units (combined inside the decode kernel),
    # one short list (a single unit); every output and log-sum-exp checked
    B, S, H, K = 3, 4096, 128, 1024
    oc = oracle_cache(_rand_bf16((B, S, 512), 61), _rand_bf16((B, S, 64), 62), 1)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 63), _rand_bf16((B, H, 64), 64)
    ends = np.array([4096, 4096, 4096], np.int32)
    rng = np.random.default_rng(65)
    topk = np.full((B, K), -1, np.int32)
    topk[0, :5] = [4096, 5000, -3, 4097, 9999]          # all out of range: nothing gathered
    topk[1] = rng.permutation(4096)[:K]
    topk[2, :7] = [3, 900, 17, 4095, 2048, 17, 0]
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.15,
                                 torch.from_numpy(topk).cuda())
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.15, topk=topk)
    got = f64(out).reshape(B, H, 512)
    assert np.all(got[0] == 0.0) and np.all(np.isneginf(f64(lse).reshape(B, H)[0]))
    check_close(got[1:].reshape(-1, 512), ref.reshape(B, H, 512)[1:].reshape(-1, 512), "out")
    check_close(f64(lse).reshape(B, H)[1:].reshape(-1), ref_lse.reshape(B, H)[1:].reshape(-1), "lse")


@pytest.mark.parametrize("fmt", [1, 2])
def test_sparse_fused_append_sees_the_new_row(fmt):
    B, S, H, K = 3, 128, 128, 64
    oc = oracle_cache(_rand_bf16((B, S, 512), 61), _rand_bf16((B, S, 64), 62), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 63), _rand_bf16((B, H, 64), 64)
    ends = np.array([128, 50, 7], np.int32)
    topk = inputs.topk_indices(B, K, ends, 65).numpy()
    kv_new, pe_new = _rand_bf16((B, 512), 66), _rand_bf16((B, 64), 67)
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.2,
                                 torch.from_numpy(topk).cuda(), kv_new=kv_new.cuda(), pe_new=pe_new.cuda())
    orc.cache_append(oc, bits(kv_new), bits(pe_new), ends - 1)
    torch.cuda.synchronize()
    assert np.array_equal(dc.kv.cpu().numpy(), oc["kv"])
    assert np.array_equal(dc.kv_scale.cpu().numpy().view(np.uint32), oc["kv_scale"].view(np.uint32))
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.2, topk=topk)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


@pytest.mark.parametrize("fmt,H", [(0, 128), (0, 64), (1, 64)])
def test_sparse_gather_variants_lists_and_fused_append(fmt, H):
    # the gather variants on a bf16 cache (the tensor-memory kernel at
    # H = 128, the warp-MMA kernel below) and on an FP8 cache at H = 64:
    # split and single-unit sequences, last tiles of fewer than 32 and of
    # 32-47 rows, repeats and invalid entries, a one-position sequence, with
    # the step's new rows written by the list prep; every output, log-sum-exp
    # and cache byte checked
    B, S, K = 4, 600, 320
    oc = oracle_cache(_rand_bf16((B, S, 512), 171), _rand_bf16((B, S, 64), 172), fmt)
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 173), _rand_bf16((B, H, 64), 174)
    ends = np.array([600, 45, 230, 1], np.int32)
    rng = np.random.default_rng(175)
    topk = np.full((B, K), -1, np.int32)
    topk[0] = rng.permutation(600)[:K]                 # 320 rows: 6 full tiles + 32
    topk[1, :50] = rng.permutation(50)                 # 45 valid rows (44 is the new row)
    topk[2] = rng.integers(-3, 260, K)                 # repeats, some past end_pos
    topk[3, :3] = [0, 0, 5]                            # only the new row
    kv_new, pe_new = _rand_bf16((B, 512), 176), _rand_bf16((B, 64), 177)
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.17,
                                 torch.from_numpy(topk).cuda(), kv_new=kv_new.cuda(), pe_new=pe_new.cuda())
    orc.cache_append(oc, bits(kv_new), bits(pe_new), ends - 1)
    torch.cuda.synchronize()
    if fmt == 0:
        assert np.array_equal(bits(dc.kv.cpu()), oc["kv"])
    else:
        assert np.array_equal(dc.kv.cpu().numpy(), oc["kv"])
        assert np.array_equal(dc.kv_scale.cpu().numpy().view(np.uint32), oc["kv_scale"].view(np.uint32))
    assert np.array_equal(bits(dc.pe.cpu()), oc["pe"])
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.17, topk=topk)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


def test_sparse_gather_lists_span_bitmap_windows():
    # positions past 2^18 and 2^19: the list prep takes the sequence in
    # windows of 2^18 positions; entries on both sides of each window edge,
    # at T - 1, at T (invalid), negative, and repeated
    B, S, H, K = 1, 530000, 128, 1536
    rng = np.random.default_rng(71)
    topk = rng.integers(-5, S + 10, (B, K)).astype(np.int32)
    edges = [0, 262143, 262144, 262145, 524287, 524288, 529999, 530000, -1]
    topk[0, :len(edges)] = edges
    topk[0, 20:40] = topk[0, 10]
    ends = np.array([S], np.int32)
    # only the rows the list names carry data (the rest stay zero): a small
    # host footprint for a cache of 530000 positions
    kv = np.zeros((B, S, 512), np.uint16)
    pe = np.zeros((B, S, 64), np.uint16)
    used = np.unique(topk[(topk >= 0) & (topk < S)])
    kv[0, used] = bits(_rand_bf16((used.size, 512), 72))
    pe[0, used] = bits(_rand_bf16((used.size, 64), 73))
    q, sc = orc.quantize_rows(kv)
    oc = {"fmt": 1, "kv": q, "kv_scale": sc, "pe": pe}
    dc = device_cache(oc)
    ql, qp = _rand_bf16((B, H, 512), 74), _rand_bf16((B, H, 64), 75)
    gidx = torch.empty((B, K), dtype=torch.int32, device="cuda")
    gcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.12,
                                 torch.from_numpy(topk).cuda(), gidx=gidx, gcount=gcnt)
    ref_g, ref_c = orc.sparse_gather_lists(topk, ends)
    assert np.array_equal(gidx.cpu().numpy(), ref_g) and np.array_equal(gcnt.cpu().numpy(), ref_c)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.12, topk=topk)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")


# ------------------------------------------------------ full-size workloads

def _run_dense_workload(w, per_seq):
    oc, dc = workload_cache(w)
    ql, qp = inputs.queries(w)
    ends = inputs.end_positions(w)
    out, lse = mla.decode(dc, ql.cuda(), qp.cuda(), ends.cuda(), w.S, w.softmax_scale)
    pairs = None if per_seq is None else sample_pairs(w.B, w.H, per_seq, w.index)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends.numpy(), w.softmax_scale,
                                       pairs=pairs)
    o = f64(out)
    l = f64(lse)
    if pairs is None:
        got, got_l = o.reshape(-1, 512), l.reshape(-1)
    else:
        got = np.stack([o[b, h] for b, h in pairs])
        got_l = np.array([l[b, h] for b, h in pairs])
    check_close(got, ref, f"{w.name} out")
    check_close(got_l, ref_lse, f"{w.name} lse")


def test_workload1_tiny_all_outputs():
    _run_dense_workload(inputs.WORKLOADS[1], None)


def test_workload1_fp8_append_row():
    # the tiny workload's one-row FP8 append: row 255 of a 1 x 256 FP8 cache
    w = inputs.WORKLOADS[1]
    oc = oracle_cache(inputs.latent_rows(w), inputs.rotary_rows(w), 1)
    dc = device_cache(oc)
    kv_new, pe_new = inputs.new_rows(w)
    mla.cache_append(dc, kv_new.cuda(), pe_new.cuda(), [255])
    orc.cache_append(oc, bits(kv_new), bits(pe_new), [255])
    torch.cuda.synchronize()
    assert np.array_equal(dc.kv.cpu().numpy(), oc["kv"])
    assert np.array_equal(dc.kv_scale.cpu().numpy(), oc["kv_scale"])


def test_workload2_v3_decode():
    _run_dense_workload(inputs.WORKLOADS[2], 6)


def test_workload3_serving_variable_lengths():
    _run_dense_workload(inputs.WORKLOADS[3], 8)


def test_workload4_long_context():
    _run_dense_workload(inputs.WORKLOADS[4], 4)


def test_workload5_sparse_with_fused_append():
    w = inputs.WORKLOADS[5]
    oc, dc = workload_cache(w)
    ql, qp = inputs.queries(w)
    ends = inputs.end_positions(w)
    topk = inputs.topk_indices(w.B, w.topk, ends, 1000 * w.index + inputs.T_TOPK)
    kv_new, pe_new = inputs.new_rows(w)
    gidx = torch.empty((w.B, w.topk), dtype=torch.int32, device="cuda")
    gcnt = torch.empty((w.B,), dtype=torch.int32, device="cuda")
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), ends.cuda(), w.S, w.softmax_scale,
                                 topk.cuda(), kv_new=kv_new.cuda(), pe_new=pe_new.cuda(),
                                 gidx=gidx, gcount=gcnt)
    orc.cache_append(oc, bits(kv_new), bits(pe_new), ends.numpy() - 1)
    ref_g, ref_c = orc.sparse_gather_lists(topk.numpy(), ends.numpy())
    assert np.array_equal(gidx.cpu().numpy(), ref_g) and np.array_equal(gcnt.cpu().numpy(), ref_c)
    pairs = sample_pairs(w.B, w.H, 3, w.index)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends.numpy(), w.softmax_scale,
                                       pairs=pairs, topk=topk.numpy())
    o, l = f64(out), f64(lse)
    check_close(np.stack([o[b, h] for b, h in pairs]), ref, "out")
    check_close(np.array([l[b, h] for b, h in pairs]), ref_lse, "lse")


def _check_tokens_sampled(w, oc, ql, qp, ends, out, lse, tokens, per_seq):
    o, l = f64(out), f64(lse)
    for j in tokens:
        pairs = sample_pairs(w.B, w.H, per_seq, 1000 * w.index + j)
        ref, ref_lse = orc.decode_absorbed_mtp(oc, bits(ql), bits(qp), ends.numpy(), w.softmax_scale,
                                               token=j, pairs=pairs)
        check_close(np.stack([o[b, j, h] for b, h in pairs]), ref, f"{w.name} token {j} out")
        check_close(np.array([l[b, j, h] for b, h in pairs]), ref_lse, f"{w.name} token {j} lse")


def test_workload6_multi_token_decode():
    w = inputs.WORKLOADS[6]
    oc, dc = workload_cache(w)
    ql, qp = inputs.queries(w)
    ends = inputs.end_positions(w)
    ws = mla.alloc_workspace(w.B * w.mtp, w.H, w.S)
    out, lse = mla.decode_mtp(dc, ql.cuda(), qp.cuda(), ends.cuda(), w.S, w.softmax_scale, workspace=ws)
    _check_tokens_sampled(w, oc, ql, qp, ends, out, lse, range(w.mtp), 4)


def test_workload8_prefill_chunk():
    # first, second, middle and last tokens of the 512-token chunk
    w = inputs.WORKLOADS[8]
    oc, dc = workload_cache(w)
    ql, qp = inputs.queries(w)
    ends = inputs.end_positions(w)
    ws = mla.alloc_workspace(w.B * w.mtp, w.H, w.S)
    out, lse = mla.decode_mtp(dc, ql.cuda(), qp.cuda(), ends.cuda(), w.S, w.softmax_scale, workspace=ws)
    _check_tokens_sampled(w, oc, ql, qp, ends, out, lse, [0, 1, 255, 510, 511], 4)


def test_workload7_attention_step():
    # q_nope -> absorption -> latent decode -> value projection, against the
    # oracle's fp64 chain of the same three steps (its own q_latent and x)
    w = inputs.WORKLOADS[7]
    oc, dc = workload_cache(w)
    qn, wkv = inputs.absorb_inputs(w)
    _, qp = inputs.queries(w)
    ends = inputs.end_positions(w)
    ql = mla.absorb_q(qn.cuda(), wkv.cuda())
    out, _ = mla.decode(dc, ql, qp.cuda(), ends.cuda(), w.S, w.softmax_scale)
    o = f64(mla.project_out(out, wkv.cuda()))
    ql_ref = orc.absorb_q(bits(qn), bits(wkv))
    pairs = sample_pairs(w.B, w.H, 6, w.index)
    x_ref, _ = orc.decode_absorbed(oc, ql_ref, bits(qp), ends.numpy(), w.softmax_scale, pairs=pairs)
    x = np.zeros((w.B, w.H, 512))
    for k, (b, h) in enumerate(pairs):
        x[b, h] = x_ref[k]
    o_ref = orc.project_out(x, bits(wkv))
    check_close(f64(ql).reshape(-1, 512), ql_ref.reshape(-1, 512), "q_latent")
    check_close(np.stack([o[b, h] for b, h in pairs]), np.stack([o_ref[b, h] for b, h in pairs]), "o")


# ---------------------------------------------------------------- limits

def test_limits_longest_list_most_tokens_most_rows():
    # the largest top-k list (8192 entries, with repeats and a ragged length),
    # the largest multi-token call (1024 tokens) and the largest append (2048
    # rows), each against the oracle
    B, S, H, K = 2, 9000, 128, 8192
    oc = oracle_cache(_rand_bf16((B, S, 512), 141), _rand_bf16((B, S, 64), 142), 1)
    dc = device_cache(oc)
    ends = np.array([9000, 8500], np.int32)
    rng = np.random.default_rng(143)
    topk = np.stack([rng.permutation(int(T))[:K] for T in ends]).astype(np.int32)
    topk[1, :100] = topk[1, 100]                            # repeats count once
    ql, qp = _rand_bf16((B, H, 512), 144), _rand_bf16((B, H, 64), 145)
    gidx = torch.empty((B, K), dtype=torch.int32, device="cuda")
    gcnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.13,
                                 torch.from_numpy(topk).cuda(), gidx=gidx, gcount=gcnt)
    ref_g, ref_c = orc.sparse_gather_lists(topk, ends)
    assert np.array_equal(gidx.cpu().numpy(), ref_g) and np.array_equal(gcnt.cpu().numpy(), ref_c)
    pairs = sample_pairs(B, H, 6, 146)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.13, pairs=pairs, topk=topk)
    o, l = f64(out), f64(lse)
    check_close(np.stack([o[b, h] for b, h in pairs]), ref, "sparse out")
    check_close(np.array([l[b, h] for b, h in pairs]), ref_lse, "sparse lse")

    s, T = 1024, 1100
    oc0 = oracle_cache(_rand_bf16((1, T, 512), 147), _rand_bf16((1, T, 64), 148), 0)
    dc0 = device_cache(oc0)
    qm, qpm = _rand_bf16((1, s, H, 512), 149), _rand_bf16((1, s, H, 64), 150)
    e = np.array([T], np.int32)
    om, lm = mla.decode_mtp(dc0, qm.cuda(), qpm.cuda(), torch.from_numpy(e).cuda(), T, 0.13,
                            workspace=mla.alloc_workspace(s, H, T))
    om, lm = f64(om), f64(lm)
    for j in (0, 511, 1023):
        pairs = sample_pairs(1, H, 4, 151 + j)
        ref, ref_lse = orc.decode_absorbed_mtp(oc0, bits(qm), bits(qpm), e, 0.13, token=j, pairs=pairs)
        check_close(np.stack([om[b, j, h] for b, h in pairs]), ref, f"token {j} out")
        check_close(np.array([lm[b, j, h] for b, h in pairs]), ref_lse, f"token {j} lse")

    R = 2048
    oc1 = oracle_cache(_rand_bf16((R, 4, 512), 152), _rand_bf16((R, 4, 64), 153), 1)
    dc1 = device_cache(oc1)
    kv_new, pe_new = _rand_bf16((R, 512), 154), _rand_bf16((R, 64), 155)
    start = np.random.default_rng(156).integers(0, 4, R).astype(np.int32)
    mla.cache_append(dc1, kv_new.cuda(), pe_new.cuda(), start)
    orc.cache_append(oc1, bits(kv_new), bits(pe_new), start)
    torch.cuda.synchronize()
    assert np.array_equal(dc1.kv.cpu().numpy(), oc1["kv"])
    assert np.array_equal(dc1.kv_scale.cpu().numpy().view(np.uint32), oc1["kv_scale"].view(np.uint32))
    assert np.array_equal(bits(dc1.pe.cpu()), oc1["pe"])


# ---------------------------------------------------------- top-k select

def _adversarial_scores(B, S, seed):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((B, S)).astype(np.float32)
    s[0, 10:60] = 0.75                                      # a run of equal scores
    s[1, ::5] = -0.0
    s[1, 2::5] = 0.0
    s[2, rng.integers(0, S, 20)] = np.inf
    s[2, rng.integers(0, S, 20)] = -np.inf
    s[3, rng.integers(0, S, 30)] = np.nan
    s[3, :5] = np.float32(3.0e38)
    return s


@pytest.mark.parametrize("K", [1, 7, 64, 250, 299, 300, 500])
def test_topk_select_bit_exact(K):
    B, S = 5, 300
    scores = _adversarial_scores(B, S, 161)
    ends = np.array([300, 257, 0, 299, 40], np.int32)
    got = mla.topk_select(torch.from_numpy(scores).cuda(), torch.from_numpy(ends).cuda(), K)
    assert np.array_equal(got.cpu().numpy(), orc.topk_select(scores, ends, K))


def test_topk_select_sparse_workload_shape():
    # 16 sequences of 32768 scores, 2048 selected (ties included)
    B, S, K = 16, 32768, 2048
    rng = np.random.default_rng(162)
    scores = rng.standard_normal((B, S)).astype(np.float32)
    scores[:, ::97] = np.round(scores[:, ::97], 1)
    ends = np.array([S] * 12 + [S - 1, 3000, 2048, 100], np.int32)
    got = mla.topk_select(torch.from_numpy(scores).cuda(), torch.from_numpy(ends).cuda(), K)
    assert np.array_equal(got.cpu().numpy(), orc.topk_select(scores, ends, K))


def test_topk_select_feeds_the_sparse_decode():
    # per-position scores -> selection -> gathered decode, on the device and
    # in the oracle (each side selects its own lists from the same scores)
    B, S, H, K = 3, 700, 128, 256
    oc = oracle_cache(_rand_bf16((B, S, 512), 163), _rand_bf16((B, S, 64), 164), 1)
    dc = device_cache(oc)
    scores = np.random.default_rng(165).standard_normal((B, S)).astype(np.float32)
    ends = np.array([700, 301, 120], np.int32)
    ql, qp = _rand_bf16((B, H, 512), 166), _rand_bf16((B, H, 64), 167)
    e_dev = torch.from_numpy(ends).cuda()
    idx = mla.topk_select(torch.from_numpy(scores).cuda(), e_dev, K)
    out, lse = mla.decode_sparse(dc, ql.cuda(), qp.cuda(), e_dev, S, 0.11, idx)
    ref_idx = orc.topk_select(scores, ends, K)
    ref, ref_lse = orc.decode_absorbed(oc, bits(ql), bits(qp), ends, 0.11, topk=ref_idx)
    check_close(f64(out).reshape(-1, 512), ref, "out")
    check_close(f64(lse).reshape(-1), ref_lse, "lse")
