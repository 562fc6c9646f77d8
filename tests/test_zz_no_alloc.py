"""mla_decode_noalloc: the decode for callers that cannot allocate device
memory where they decode (so cannot pass a workspace); it uses the library's
own static device scratch instead.

The test calls it through the C ABI twice in a row on the same inputs and
checks both results against the existing entry point (mla_decode with a
caller workspace) with the tolerance the parity tests use.  The file name
makes pytest collect it last, so a run that stops at the first failure has
already run every other test; it also passes when run alone.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_07_gb300 as mla
from mla_latent_kv_07_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_REL, L2_REL = 1e-2, 5e-3


def _close(got, ref, what):
    g = got.double().cpu().numpy().reshape(-1)
    r = ref.double().cpu().numpy().reshape(-1)
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), what
    g, r = g[~ninf], r[~ninf]
    scale = np.abs(r).max()
    assert np.abs(g - r).max() <= MAX_REL * scale, what
    assert np.linalg.norm(g - r) <= L2_REL * np.linalg.norm(r), what


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_latent_kv_07_gb300 import build
    build.build()
    mla.lib()


SCRATCH_BYTES = 32 << 20   # the library's static scratch (include/mla.h)


@pytest.mark.parametrize("fmt,H,ends,S", [(1, 128, [700, 33, 1], 768), (0, 16, [256, 100], 256),
                                          (0, 128, [520, 1, 97, 300], 640)])
def test_noalloc_matches_workspace_decode_twice(fmt, H, ends, S):
    B = len(ends)
    kv = inputs.randn_bf16((B, S, 512), 7001 + H).cuda()
    pe = inputs.randn_bf16((B, S, 64), 7002 + H).cuda()
    if fmt == 0:
        cache = mla.Cache(B, S, 0, kv=kv, pe=pe)
    else:
        cache = mla.Cache(B, S, 1, pe=pe)
        # quantise every row with the append kernel (at most 2048 rows per call)
        rows, kvf, scf, pef = kv.view(B * S, 512), cache.kv.view(B * S, 1, 512), \
            cache.kv_scale.view(B * S, 1, 4), cache.pe.view(B * S, 1, 64)
        for r0 in range(0, B * S, 2048):
            n = min(2048, B * S - r0)
            sub = mla.Cache(n, 1, 1, kv=kvf[r0:r0 + n], kv_scale=scf[r0:r0 + n], pe=pef[r0:r0 + n])
            mla.cache_append(sub, rows[r0:r0 + n], pe.view(B * S, 64)[r0:r0 + n], [0] * n)
    ql = inputs.randn_bf16((B, H, 512), 7003 + H).cuda()
    qp = inputs.randn_bf16((B, H, 64), 7004 + H).cuda()
    end_pos = torch.tensor(ends, dtype=torch.int32).cuda()
    ref_out, ref_lse = mla.decode(cache, ql, qp, end_pos, S, 0.1352)
    for _ in range(2):
        out, lse = mla.decode_noalloc(cache, ql, qp, end_pos, S, 0.1352)
        torch.cuda.synchronize()
        _close(out, ref_out, "out")
        _close(lse, ref_lse, "lse")


def test_noalloc_refuses_batches_beyond_its_scratch():
    B, S, H = 1024, 1, 128
    cache = mla.Cache(B, S, 0)
    ql = torch.zeros((B, H, 512), dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros((B, H, 64), dtype=torch.bfloat16, device="cuda")
    end_pos = torch.ones((B,), dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_noalloc(cache, ql, qp, end_pos, S, 0.1)
    assert e.value.code == 4


def test_noalloc_limit_at_128_heads():
    # the largest batch whose scratch need fits the array runs and matches the
    # workspace decode; one more sequence is refused with MLA_ERR_WORKSPACE
    H, S = 128, 64
    fits = max(b for b in range(1, 512) if mla.workspace_size(b, H, S) <= SCRATCH_BYTES)
    assert mla.workspace_size(fits + 1, H, S) > SCRATCH_BYTES
    kv = inputs.randn_bf16((fits + 1, S, 512), 7101).cuda()
    pe = inputs.randn_bf16((fits + 1, S, 64), 7102).cuda()
    cache = mla.Cache(fits + 1, S, 0, kv=kv, pe=pe)
    ql = inputs.randn_bf16((fits + 1, H, 512), 7103).cuda()
    qp = inputs.randn_bf16((fits + 1, H, 64), 7104).cuda()
    end_pos = torch.arange(1, fits + 2, dtype=torch.int32).remainder(S).add(1).cuda()
    ref_out, ref_lse = mla.decode(cache, ql[:fits], qp[:fits], end_pos[:fits], S, 0.1352)
    out, lse = mla.decode_noalloc(cache, ql[:fits], qp[:fits], end_pos[:fits], S, 0.1352)
    torch.cuda.synchronize()
    _close(out, ref_out, "out at the limit")
    _close(lse, ref_lse, "lse at the limit")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_noalloc(cache, ql, qp, end_pos, S, 0.1352)
    assert e.value.code == 4
