"""Pins for the oracle's number formats and its FP8 block quantiser.

The oracle is checked against things other than itself: hand-worked codes of
the OCP E4M3 format, a brute-force nearest-value search over a code table
built here from the format definition, torch's own CPU float8/bf16 casts (an
independent implementation), and error bounds that follow from the format.
The cache-write step being pinned is the FP8 round trip of the latent in the
cache-write excerpt of "DeepSeek-V3.2-Exp . KV cache".
"""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table():
    """Non-negative finite E4M3 values by code 0x00..0x7E, from the definition."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def _brute_encode(y: float) -> int:
    """Nearest table value; ties to the code with an even mantissa; saturate."""
    tab = _table()
    a = abs(y)
    sign = 0x80 if np.signbit(y) else 0
    if a >= 448.0:
        return sign | 0x7E
    d = np.abs(tab - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int([c for c in best if (c & 1) == 0][0])
    return sign | code


def test_hand_codes():
    with open(os.path.join(GOLDEN, "e4m3_hand_codes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    vals = np.array([eval(v) for v, _ in rows], np.float32)
    want = np.array([int(h, 16) for _, h in rows], np.uint8)
    got = orc.e4m3_encode(vals)
    assert (got == want).all(), list(zip(vals, got, want))


def test_encode_matches_brute_force_search():
    rng = np.random.default_rng(0)
    mags = 2.0 ** rng.uniform(-13, 9.2, 4000)
    vals = (mags * rng.choice([-1, 1], mags.size)).astype(np.float32)
    tab = _table()
    mids = ((tab[1:] + tab[:-1]) / 2).astype(np.float32)  # exact ties
    vals = np.concatenate([vals, mids, -mids, tab.astype(np.float32)])
    got = orc.e4m3_encode(vals)
    want = np.array([_brute_encode(float(v)) for v in vals], np.uint8)
    assert (got == want).all()


def test_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    vals = (rng.standard_normal(200_000) * 2.0 ** rng.uniform(-12, 8, 200_000)).astype(np.float32)
    vals = vals[np.abs(vals) < 464]  # torch's cast turns larger values into NaN (no saturation)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (orc.e4m3_encode(vals) == ref).all()


def test_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    v = orc.e4m3_value(codes)
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    tab = _table()
    assert (v[:0x7F] == tab).all() and (v[0x80:0xFF] == -tab).all()
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert (np.diff(v[:0x7F]) > 0).all()
    finite = np.isfinite(v)
    assert (orc.e4m3_encode(v[finite].astype(np.float32)) == codes[finite]).all()
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(v[finite], ref[finite])


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(100_000) * 2.0 ** rng.uniform(-30, 30, 100_000)).astype(np.float32)
    # exact ties: bf16 value plus half an ulp
    base = f.view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (base | np.uint32(0x8000)).view(np.float32)
    f = np.concatenate([f, ties])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (orc.bf16_round(f) == ref).all()


# ----------------------------------------------------------- quantiser

def _bf16(vals):
    t = torch.tensor(vals, dtype=torch.float32)
    assert torch.equal(t.to(torch.bfloat16).float(), t), "hand values must be exact in bf16"
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantise_hand_blocks():
    row = np.zeros(512, np.float32)
    b0 = [448.0, 1.0, -2.0, 3.0, 1.0625, 1.1875, 2.0 ** -9, 2.0 ** -10]
    row[: len(b0)] = b0               # block 0: amax 448 -> scale exactly 1
    row[128:256] = 0.0                # block 1: all zero -> scale 0, codes 0
    row[256:384] = 1.0                # block 2: all ones -> every code 0x7E
    row[384] = 2.0                    # block 3: amax 2 -> scale 2/448
    row[385] = 1.0
    row[386] = -0.5
    q, s = orc.quantize_rows(_bf16(row)[None])
    q, s = q[0], s[0]
    assert s[0] == np.float32(1.0)
    assert list(q[:8]) == [0x7E, 0x38, 0xC0, 0x44, 0x38, 0x3A, 0x01, 0x00]
    assert (q[8:128] == 0).all()
    assert s[1] == 0.0 and (q[128:256] == 0).all()
    assert s[2] == np.float32(1.0) / np.float32(448.0) and (q[256:384] == 0x7E).all()
    assert s[3] == np.float32(2.0) / np.float32(448.0)
    # 1.0 / (2/448) ~ 224 = 1.75 * 2^7 -> 0x76 ; -0.5 -> ~ -112 = -1.75 * 2^6 -> 0xEE
    assert q[384] == 0x7E and q[385] == 0x76 and q[386] == 0xEE
    assert (q[387:] == 0).all()


def _torch_act_quant(x_bf16: torch.Tensor):
    """The cache-write step restated with torch CPU ops (fp32 division and
    torch's float8 cast) -- an independent implementation of the encoder."""
    x = x_bf16.float().view(-1, 4, 128)
    amax = x.abs().amax(-1, keepdim=True)
    scale = amax / 448.0
    y = torch.where(amax > 0, x / scale, torch.zeros_like(x))
    q = y.to(torch.float8_e4m3fn)
    return q.view(torch.uint8).view(-1, 512), scale.view(-1, 4)


def test_quantise_matches_torch_restatement():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(2048, 512, generator=g) * torch.exp(torch.randn(2048, 1, generator=g) * 3)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quantize_rows(bits)
    tq, ts = _torch_act_quant(x)
    assert np.array_equal(s, ts.numpy())
    assert np.array_equal(q, tq.numpy())


def test_dequant_matches_torch_round_trip():
    # (codes as float32) * scale in fp32, then bf16 -- computed by torch
    g = torch.Generator().manual_seed(4)
    x = torch.randn(512, 512, generator=g).to(torch.bfloat16)
    q, s = orc.quantize_rows(x.view(torch.int16).numpy().view(np.uint16))
    deq = orc.dequant_rows(q, s)
    tq = torch.from_numpy(q).view(torch.float8_e4m3fn).float().view(-1, 4, 128)
    ref = (tq * torch.from_numpy(s).view(-1, 4, 1)).to(torch.bfloat16).view(-1, 512)
    assert np.array_equal(deq, ref.view(torch.int16).numpy().view(np.uint16))


def test_round_trip_error_bound():
    # Normal E4M3 values carry 3 mantissa bits: |y - q| <= 2^-4 |y|; below
    # 2^-6 the spacing is 2^-9 so |y - q| <= 2^-10.  In latent units this is
    # scale * that, plus the final bf16 rounding (2^-9 relative).
    g = torch.Generator().manual_seed(5)
    x = torch.randn(256, 512, generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quantize_rows(bits)
    c = orc.bf16_bits_to_f64(orc.dequant_rows(q, s))
    xv = orc.bf16_bits_to_f64(bits)
    sc = np.repeat(s.astype(np.float64), 128, axis=1)
    y = np.abs(xv) / sc
    bound = np.where(y >= 2.0 ** -6, y * 2.0 ** -4, 2.0 ** -10) * sc * (1 + 2.0 ** -8) + np.abs(xv) * 2.0 ** -8
    assert (np.abs(c - xv) <= bound).all()


# ------------------------------------------- power-of-two scale format

def _pow2_at_least_brute(s: float) -> float:
    """Smallest 2^k (k from -149 up, every fp32 power of two) that is >= s."""
    k = -149
    while 2.0 ** k < s:
        k += 1
    return 2.0 ** k


def test_quantise_pow2_hand_blocks():
    row = np.zeros(512, np.float32)
    row[:4] = [448.0, 1.0, -2.0, 2.0 ** -9]   # block 0: amax 448 -> scale exactly 1
    row[128:256] = 1.0                        # block 1: 1/448 -> 2^-8; 1 / 2^-8 = 256 = 0x78
    row[256] = 450.0                          # block 2: 450/448 -> 2; 225 -> 224 = 0x76
    row[257] = -0.5                           #          -0.25 -> 2^-2 = 0xA8
    row[384] = 2.0 ** -132                    # block 3: fp32(amax/448) = 293 * 2^-149 is
    row[385] = -(2.0 ** -133)                 #          subnormal, rounds up to 2^-140
    q, s = orc.quantize_rows(_bf16(row)[None], pow2=True)
    q, s = q[0], s[0]
    assert s[0] == 1.0 and list(q[:4]) == [0x7E, 0x38, 0xC0, 0x01]
    assert s[1] == 2.0 ** -8 and (q[128:256] == 0x78).all()
    assert s[2] == 2.0 and q[256] == 0x76 and q[257] == 0xA8 and (q[258:384] == 0).all()
    assert s[3] == np.float32(2.0 ** -140) and q[384] == 0x78 and q[385] == 0xF0
    zero = np.zeros((1, 512), np.uint16)
    qz, sz = orc.quantize_rows(zero, pow2=True)
    assert (sz == 0).all() and (qz == 0).all()


def test_quantise_pow2_matches_brute_force():
    # scale: brute-force smallest power of two >= fp32(amax / 448); codes:
    # brute-force nearest table value of x / scale, which is exact here
    g = torch.Generator().manual_seed(6)
    x = (torch.randn(96, 512, generator=g) * torch.exp(torch.randn(96, 1, generator=g) * 6)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quantize_rows(bits, pow2=True)
    xv = orc.bf16_bits_to_f64(bits).reshape(-1, 4, 128)
    amax = np.abs(xv).max(-1).astype(np.float32)
    base = amax / np.float32(448.0)
    want_s = np.array([_pow2_at_least_brute(float(v)) if v > 0 else 0.0 for v in base.ravel()])
    assert np.array_equal(s.ravel().astype(np.float64), want_s)
    for r in range(0, 96, 7):
        for j in range(4):
            for i in range(0, 128, 5):
                y = xv[r, j, i] / float(s[r, j])
                assert q[r, j * 128 + i] == _brute_encode(y), (r, j, i)


def test_dequant_pow2_is_exact():
    # e4m3 values carry 4 significant bits, so value * 2^k is exact in fp32
    # and in bf16: the round trip adds no rounding beyond the e4m3 code's
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(256, 512, generator=g) * 3).to(torch.bfloat16)
    q, s = orc.quantize_rows(x.view(torch.int16).numpy().view(np.uint16), pow2=True)
    got = orc.bf16_bits_to_f64(orc.dequant_rows(q, s))
    want = orc.e4m3_value(q) * np.repeat(s.astype(np.float64), 128, axis=1)
    assert np.array_equal(got, want)


def test_cache_append_pow2_format():
    g = torch.Generator().manual_seed(8)
    kv = torch.randn(2, 512, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pe = torch.randn(2, 64, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    cache = {"fmt": 2, "kv": np.zeros((2, 8, 512), np.uint8), "kv_scale": np.zeros((2, 8, 4), np.float32),
             "pe": np.zeros((2, 8, 64), np.uint16)}
    orc.cache_append(cache, kv, pe, [3, 5])
    q, s = orc.quantize_rows(kv, pow2=True)
    assert np.array_equal(cache["kv"][0, 3], q[0]) and np.array_equal(cache["kv"][1, 5], q[1])
    assert np.array_equal(cache["kv_scale"][1, 5], s[1])
    m, _ = np.frexp(s)
    assert (m == 0.5).all()


def test_footprint_golden():
    # latent-only bytes of one layer; pins the byte accounting used by the bench
    from mla_latent_kv_07_gb300 import layout
    with open(os.path.join(GOLDEN, "p4_footprint.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for tokens, bpv, mib in rows:
        fmt = 0 if int(bpv) == 2 else 1
        got = layout.latent_bytes(int(tokens), fmt) / 2 ** 20
        assert round(got, 2) == pytest.approx(float(mib)), (tokens, bpv, got)
