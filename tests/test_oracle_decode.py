"""Pins for the oracle's absorbed decode, sparse mask and cache append.

What fixes the answers here, independent of the oracle's own code:
  * closed forms (one position, two positions, zero query, end_pos = 0);
  * the absorption identity of "DeepSeek MLA architecture ..." section 4:
    scoring against W_UK-expanded keys and summing W_UV-expanded values equals
    the absorbed latent-space computation followed by W_UV;
  * invariants (weights sum to 1, masked weights exactly 0, output inside the
    convex hull of the attended latents, invariance to permuting positions);
  * the top-k mask of the MQA-decode excerpt of "DeepSeek-V3.2-Exp . KV cache"
    (an index list covering every position equals dense attention; repeated
    and out-of-range indices change nothing);
  * the cache geometry of that page: a call that writes row 1,000 reads rows
    0..1,000;
  * multi-token decode: a brute-force float64 attention with the explicit
    causal mask matrix over the step's s tokens (token j at position
    T-s+j sees positions 0..T-s+j);
  * the per-head products around the decode: identity weights, a brute-force
    loop, and query absorption + latent decode + value projection equal to
    the non-absorbed MHA over W_UK / W_UV-expanded keys and values.
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc

DC, DR = 512, 64


def _bits(x):
    """float array exact in bf16 -> bits."""
    x = np.asarray(x, np.float32)
    b = orc.bf16_round(x)
    assert np.array_equal(orc.bf16_bits_to_f64(b), x.astype(np.float64))
    return b


def _rand_cache(rng, B, S, fmt=0):
    x = rng.standard_normal((B, S, DC)).astype(np.float32)
    kv = orc.bf16_round(x)
    pe = orc.bf16_round(rng.standard_normal((B, S, DR)).astype(np.float32))
    if fmt == 0:
        return {"fmt": 0, "kv": kv, "pe": pe}
    q, s = orc.quantize_rows(kv, pow2=fmt == 2)
    return {"fmt": fmt, "kv": q, "kv_scale": s, "pe": pe}


def _latents(cache):
    if cache["fmt"] == 0:
        return orc.bf16_bits_to_f64(cache["kv"])
    return orc.bf16_bits_to_f64(orc.dequant_rows(cache["kv"], cache["kv_scale"]))


def _rand_q(rng, B, H):
    ql = orc.bf16_round(rng.standard_normal((B, H, DC)).astype(np.float32))
    qp = orc.bf16_round(rng.standard_normal((B, H, DR)).astype(np.float32))
    return ql, qp


def test_single_position_closed_form():
    rng = np.random.default_rng(10)
    cache = _rand_cache(rng, 1, 4)
    ql, qp = _rand_q(rng, 1, 3)
    out, lse = orc.decode_absorbed(cache, ql, qp, [1], 0.3)
    c0 = orc.bf16_bits_to_f64(cache["kv"][0, 0])
    k0 = orc.bf16_bits_to_f64(cache["pe"][0, 0])
    for h in range(3):
        assert np.array_equal(out[h], c0)            # weight 1 on the only position
        s0 = 0.3 * (orc.bf16_bits_to_f64(ql[0, h]) @ c0 + orc.bf16_bits_to_f64(qp[0, h]) @ k0)
        assert lse[h] == pytest.approx(s0, rel=1e-14, abs=1e-14)


def test_two_positions_closed_form():
    # c_0 = e_0, c_1 = 2 e_1 ; rotary keys r_0 = e_0, r_1 = 0 ;
    # q_latent = a e_0 + b e_1, q_pe = d e_0  ->  s_0 = sig (a + d), s_1 = sig 2b
    a, b, d, sig = 1.5, -0.75, 0.5, 0.7
    kv = np.zeros((1, 2, DC), np.float32); kv[0, 0, 0] = 1; kv[0, 1, 1] = 2
    pe = np.zeros((1, 2, DR), np.float32); pe[0, 0, 0] = 1
    cache = {"fmt": 0, "kv": _bits(kv), "pe": _bits(pe)}
    ql = np.zeros((1, 1, DC), np.float32); ql[0, 0, 0] = a; ql[0, 0, 1] = b
    qp = np.zeros((1, 1, DR), np.float32); qp[0, 0, 0] = d
    out, lse = orc.decode_absorbed(cache, _bits(ql), _bits(qp), [2], sig)
    s0, s1 = sig * (a + d), sig * 2 * b
    w0 = 1 / (1 + math.exp(s1 - s0))
    assert out[0, 0] == pytest.approx(w0, rel=1e-14)
    assert out[0, 1] == pytest.approx(2 * (1 - w0), rel=1e-14)
    assert np.all(out[0, 2:] == 0)
    assert lse[0] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), rel=1e-14)


def test_zero_query_is_uniform_mean():
    rng = np.random.default_rng(11)
    for fmt in (0, 1):
        cache = _rand_cache(rng, 2, 37, fmt)
        z = np.zeros((2, 2, DC), np.uint16), np.zeros((2, 2, DR), np.uint16)
        out, lse = orc.decode_absorbed(cache, z[0], z[1], [37, 5], 1.0)
        c = _latents(cache)
        np.testing.assert_allclose(out[0], c[0, :37].mean(0), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out[2], c[1, :5].mean(0), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, [math.log(37)] * 2 + [math.log(5)] * 2, rtol=1e-14)


def test_rotary_term_alone():
    # q_latent = 0: only q_pe . k_R decides.  One key aligned with a large q_pe
    # dominates, so the output is that position's latent.
    rng = np.random.default_rng(12)
    cache = _rand_cache(rng, 1, 16)
    pe = np.zeros((1, 16, DR), np.float32); pe[0, 9, 3] = 64.0
    cache["pe"] = _bits(pe)
    qp = np.zeros((1, 1, DR), np.float32); qp[0, 0, 3] = 64.0
    out, lse = orc.decode_absorbed(cache, np.zeros((1, 1, DC), np.uint16), _bits(qp), [16], 1.0)
    np.testing.assert_allclose(out[0], orc.bf16_bits_to_f64(cache["kv"][0, 9]), rtol=1e-12, atol=1e-300)
    assert lse[0] == pytest.approx(4096.0, rel=1e-12)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_absorbed_equals_naive_mha(fmt):
    rng = np.random.default_rng(20 + fmt)
    B, H, S = 2, 3, 9
    cache = _rand_cache(rng, B, S, fmt)
    end_pos = np.array([9, 4], np.int32)
    wkv_b = rng.standard_normal((H, 256, DC)) * 0.05
    q_nope = rng.standard_normal((B, H, 128))
    q_pe = rng.standard_normal((B, H, DR))
    sig = 192 ** -0.5
    o_naive, lse_naive = orc.decode_naive(cache, wkv_b, q_nope, q_pe, end_pos, sig)
    # absorbed query: q_latent[h] = W_UK[h]^T q_nope[h]  (exact in fp64)
    q_lat = np.einsum("bhd,hdc->bhc", q_nope, wkv_b[:, :128])
    out, lse = orc.decode_absorbed(cache, q_lat, q_pe, end_pos, sig)
    out = out.reshape(B, H, DC)
    o_abs = np.einsum("bhc,hdc->bhd", out, wkv_b[:, 128:])   # W_UV after the sum
    np.testing.assert_allclose(o_abs, o_naive, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B, H), lse_naive, rtol=1e-10)


def test_weight_invariants_and_hull():
    rng = np.random.default_rng(30)
    cache = _rand_cache(rng, 2, 64, 1)
    ql, qp = _rand_q(rng, 2, 4)
    ep = np.array([64, 23], np.int32)
    out, lse, w = orc.decode_absorbed(cache, ql, qp, ep, 0.1352, weights_upto=64)
    c = _latents(cache)
    for p in range(8):
        b = p // 4
        T = ep[b]
        assert w[p].sum() == pytest.approx(1.0, abs=1e-12)
        assert (w[p] >= 0).all() and (w[p, T:] == 0).all()
        np.testing.assert_allclose(out[p], w[p, :T] @ c[b, :T], rtol=1e-12, atol=1e-13)
        lo, hi = c[b, :T].min(0), c[b, :T].max(0)
        assert (out[p] >= lo - 1e-12).all() and (out[p] <= hi + 1e-12).all()


def test_position_permutation_invariance():
    rng = np.random.default_rng(31)
    cache = _rand_cache(rng, 1, 50, 1)
    ql, qp = _rand_q(rng, 1, 2)
    out, lse = orc.decode_absorbed(cache, ql, qp, [50], 0.2)
    perm = rng.permutation(50)
    c2 = {"fmt": 1, "kv": cache["kv"][:, perm], "kv_scale": cache["kv_scale"][:, perm],
          "pe": cache["pe"][:, perm]}
    out2, lse2 = orc.decode_absorbed(c2, ql, qp, [50], 0.2)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)


def test_rows_past_end_pos_are_ignored():
    rng = np.random.default_rng(32)
    cache = _rand_cache(rng, 1, 40, 1)
    ql, qp = _rand_q(rng, 1, 2)
    out, lse = orc.decode_absorbed(cache, ql, qp, [17], 0.5)
    cache["kv"][:, 17:] = 0x7F          # NaN codes beyond end_pos
    cache["kv_scale"][:, 17:] = np.inf
    cache["pe"][:, 17:] = 0x7FC0        # bf16 NaN
    out2, lse2 = orc.decode_absorbed(cache, ql, qp, [17], 0.5)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_empty_sequence():
    rng = np.random.default_rng(33)
    cache = _rand_cache(rng, 2, 8)
    ql, qp = _rand_q(rng, 2, 2)
    out, lse = orc.decode_absorbed(cache, ql, qp, [0, 8], 0.5)
    assert (out[:2] == 0).all() and np.isneginf(lse[:2]).all()
    assert np.isfinite(lse[2:]).all()


@pytest.mark.parametrize("fmt", [1, 2])
def test_fp8_cache_attends_to_round_trip_values(fmt):
    # Decoding the FP8 cache equals decoding a bf16 cache that holds the
    # dequantised latents (the bf16 cache of the cache-write excerpt).
    rng = np.random.default_rng(34)
    c8 = _rand_cache(rng, 2, 30, fmt)
    c16 = {"fmt": 0, "kv": orc.dequant_rows(c8["kv"], c8["kv_scale"]), "pe": c8["pe"]}
    ql, qp = _rand_q(rng, 2, 3)
    a = orc.decode_absorbed(c8, ql, qp, [30, 11], 0.13)
    b = orc.decode_absorbed(c16, ql, qp, [30, 11], 0.13)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_pair_subset_matches_full():
    rng = np.random.default_rng(35)
    cache = _rand_cache(rng, 3, 20, 1)
    ql, qp = _rand_q(rng, 3, 4)
    ep = np.array([20, 7, 13], np.int32)
    full, lfull = orc.decode_absorbed(cache, ql, qp, ep, 0.2)
    pairs = np.array([[2, 1], [0, 3], [1, 0]], np.int32)
    sub, lsub = orc.decode_absorbed(cache, ql, qp, ep, 0.2, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(sub[i], full[b * 4 + h]) and lsub[i] == lfull[b * 4 + h]


# ------------------------------------------------------------- top-k mask

def test_topk_covering_all_positions_equals_dense():
    rng = np.random.default_rng(40)
    cache = _rand_cache(rng, 2, 33, 1)
    ql, qp = _rand_q(rng, 2, 2)
    ep = np.array([33, 19], np.int32)
    topk = np.stack([rng.permutation(40) for _ in range(2)]).astype(np.int32)  # includes >= T
    d = orc.decode_absorbed(cache, ql, qp, ep, 0.2)
    s = orc.decode_absorbed(cache, ql, qp, ep, 0.2, topk=topk)
    np.testing.assert_allclose(s[0], d[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s[1], d[1], rtol=1e-13)


def test_topk_mask_weights_and_duplicates():
    rng = np.random.default_rng(41)
    cache = _rand_cache(rng, 1, 50, 1)
    ql, qp = _rand_q(rng, 1, 3)
    chosen = np.array([3, 17, 49, 20, 0], np.int32)
    topk = np.concatenate([chosen, [17, 3, -1, 50, 1000, -7, 49]]).astype(np.int32)[None]
    out, lse, w = orc.decode_absorbed(cache, ql, qp, [50], 0.3, topk=topk, weights_upto=50)
    mask = np.zeros(50, bool); mask[chosen] = True
    assert (w[:, ~mask] == 0).all() and (w[:, mask] > 0).all()
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)
    out2, lse2 = orc.decode_absorbed(cache, ql, qp, [50], 0.3, topk=chosen[None])
    np.testing.assert_allclose(out, out2, rtol=1e-13, atol=1e-15)
    # brute force over the chosen rows only
    c = _latents(cache)[0, np.sort(chosen)]
    kr = orc.bf16_bits_to_f64(cache["pe"][0, np.sort(chosen)])
    for h in range(3):
        s = 0.3 * (c @ orc.bf16_bits_to_f64(ql[0, h]) + kr @ orc.bf16_bits_to_f64(qp[0, h]))
        ww = np.exp(s - s.max()); ww /= ww.sum()
        np.testing.assert_allclose(out[h], ww @ c, rtol=1e-10, atol=1e-13)


def test_gather_lists_brute_force():
    rng = np.random.default_rng(42)
    B, K = 6, 300
    ep = np.array([0, 1, 50, 299, 1000, 37], np.int32)
    topk = rng.integers(-3, 400, (B, K)).astype(np.int32)
    gidx, gcount = orc.sparse_gather_lists(topk, ep)
    for b in range(B):
        want = sorted({int(t) for t in topk[b] if 0 <= t < ep[b]})
        assert gcount[b] == len(want)
        assert list(gidx[b, :gcount[b]]) == want and (gidx[b, gcount[b]:] == -1).all()


# ------------------------------------------------------------- cache write

def test_append_then_read_geometry():
    # write row 1,000 and read rows 0..1,000 (end_pos = start_pos + 1)
    rng = np.random.default_rng(50)
    S = 1024
    cache = _rand_cache(rng, 1, S, 1)
    kv_new = np.zeros((1, DC), np.float32); kv_new[0, 5] = 3.0
    pe_new = np.zeros((1, DR), np.float32); pe_new[0, 0] = 40.0
    qp = np.zeros((1, 1, DR), np.float32); qp[0, 0, 0] = 40.0
    zq = np.zeros((1, 1, DC), np.uint16)
    before = orc.decode_absorbed(cache, zq, _bits(qp), [1000], 1.0)
    orc.cache_append(cache, _bits(kv_new), _bits(pe_new), [1000])
    out, lse = orc.decode_absorbed(cache, zq, _bits(qp), [1001], 1.0)
    # the new row dominates (score 1600 vs at most ~200 for the rest) and its
    # latent survives the FP8 round trip exactly (3.0 is the block maximum)
    assert out[0, 5] == pytest.approx(3.0, rel=1e-12)
    assert lse[0] == pytest.approx(1600.0, rel=1e-12)
    # a read of rows 0..999 does not see row 1,000
    after = orc.decode_absorbed(cache, zq, _bits(qp), [1000], 1.0)
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    with pytest.raises(IndexError):
        orc.cache_append(cache, _bits(kv_new), _bits(pe_new), [S])


@pytest.mark.parametrize("fmt", [0, 1])
def test_multi_token_decode_brute_force(fmt):
    # brute force: scores of all s tokens against all S cache rows in numpy,
    # masked by the explicit [s, S] causal mask matrix built from positions
    rng = np.random.default_rng(31)
    B, S, H, s = 3, 24, 4, 3
    cache = _rand_cache(rng, B, S, fmt)
    ql = orc.bf16_round(rng.standard_normal((B, s, H, DC)).astype(np.float32))
    qp = orc.bf16_round(rng.standard_normal((B, s, H, DR)).astype(np.float32))
    ends = np.array([24, 9, 2], np.int32)          # the last sequence: token 0 has no position
    out, lse = orc.decode_absorbed_mtp(cache, ql, qp, ends, 0.21)
    lat = _latents(cache)
    rot = orc.bf16_bits_to_f64(cache["pe"])
    qlf, qpf = orc.bf16_bits_to_f64(ql), orc.bf16_bits_to_f64(qp)
    for b in range(B):
        T = int(ends[b])
        pos_tok = T - s + np.arange(s)                          # positions of the new tokens
        mask = np.arange(S)[None, :] <= pos_tok[:, None]         # [s, S]: row t visible to token j
        mask &= np.arange(S)[None, :] < T
        for j in range(s):
            for h in range(H):
                sc = 0.21 * (lat[b] @ qlf[b, j, h] + rot[b] @ qpf[b, j, h])
                if not mask[j].any():
                    assert lse[b, j, h] == -np.inf and np.all(out[b, j, h] == 0)
                    continue
                z = sc[mask[j]]
                m = z.max()
                w = np.exp(z - m)
                ref = (w[:, None] * lat[b][mask[j]]).sum(0) / w.sum()
                assert np.allclose(out[b, j, h], ref, rtol=1e-12, atol=1e-12)
                assert lse[b, j, h] == pytest.approx(m + math.log(w.sum()), rel=1e-12, abs=1e-12)


def test_multi_token_last_token_is_the_single_token_decode():
    rng = np.random.default_rng(32)
    cache = _rand_cache(rng, 2, 30)
    ql = orc.bf16_round(rng.standard_normal((2, 2, 3, DC)).astype(np.float32))
    qp = orc.bf16_round(rng.standard_normal((2, 2, 3, DR)).astype(np.float32))
    ends = np.array([30, 17], np.int32)
    out, lse = orc.decode_absorbed_mtp(cache, ql, qp, ends, 0.3)
    o1, l1 = orc.decode_absorbed(cache, np.ascontiguousarray(ql[:, 1]), np.ascontiguousarray(qp[:, 1]), ends, 0.3)
    assert np.array_equal(out[:, 1].reshape(-1, DC), o1) and np.array_equal(lse[:, 1].reshape(-1), l1)


def test_absorb_and_project_identity_weights():
    rng = np.random.default_rng(41)
    B, H = 2, 3
    w = np.zeros((H, 256, DC), np.float64)
    w[:, np.arange(128), np.arange(128)] = 1.0            # W_UK[h] = [I | 0]
    w[:, 128 + np.arange(128), 128 + np.arange(128)] = 1.0  # W_UV[h] picks c = 128..255
    qn = rng.standard_normal((B, H, 128))
    ql = orc.absorb_q(qn, w)
    assert np.array_equal(ql[..., :128], qn) and np.all(ql[..., 128:] == 0)
    x = rng.standard_normal((B, H, DC))
    assert np.array_equal(orc.project_out(x, w), x[..., 128:256])


def test_absorb_and_project_brute_force():
    rng = np.random.default_rng(42)
    B, H = 2, 2
    w = orc.bf16_round(rng.standard_normal((H, 256, DC)).astype(np.float32))
    qn = orc.bf16_round(rng.standard_normal((B, H, 128)).astype(np.float32))
    x = orc.bf16_round(rng.standard_normal((B, H, DC)).astype(np.float32))
    wf, qf, xf = (orc.bf16_bits_to_f64(a) for a in (w, qn, x))
    ql, o = orc.absorb_q(qn, w), orc.project_out(x, w)
    for b in range(B):
        for h in range(H):
            for c in (0, 77, 511):
                ref = sum(qf[b, h, n] * wf[h, n, c] for n in range(128))
                assert ql[b, h, c] == pytest.approx(ref, rel=1e-12, abs=1e-12)
            for v in (0, 64, 127):
                ref = sum(wf[h, 128 + v, c] * xf[b, h, c] for c in range(DC))
                assert o[b, h, v] == pytest.approx(ref, rel=1e-12, abs=1e-12)


@pytest.mark.parametrize("fmt", [0, 1])
def test_absorbed_pipeline_equals_naive_mha(fmt):
    # q_nope -> absorb -> latent decode -> project equals attention over the
    # expanded keys W_UK c_t and values W_UV c_t (section 4 of the MLA page)
    rng = np.random.default_rng(43)
    B, S, H = 2, 20, 3
    cache = _rand_cache(rng, B, S, fmt)
    w = rng.standard_normal((H, 256, DC)) * 0.05
    qn = rng.standard_normal((B, H, 128))
    qp = orc.bf16_round(rng.standard_normal((B, H, DR)).astype(np.float32))
    ends = np.array([20, 7], np.int32)
    ql = orc.absorb_q(qn, w)
    out, _ = orc.decode_absorbed(cache, ql, qp, ends, 0.2)
    o = orc.project_out(out.reshape(B, H, DC), w)
    o_naive, _ = orc.decode_naive(cache, w, qn, qp, ends, 0.2)
    assert np.allclose(o, o_naive, rtol=1e-10, atol=1e-10)
