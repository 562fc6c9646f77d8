"""GPU parity of the per-head products around the decode (query absorption
q_latent = q_nope . W_UK and value projection o = W_UV . x) against the CPU
oracle, through the C ABI, and of the whole absorbed pipeline (absorb ->
latent decode -> project) against the oracle's non-absorbed MHA.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_07_gb300 as mla
from mla_latent_kv_07_gb300 import inputs
from oracle import oracle as orc

from mla_cases import bits, check_close, device_cache, f64, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_latent_kv_07_gb300 import build
    build.build()
    mla.lib()


def _weights(H, seed, scale=0.05):
    w = inputs.randn_bf16((H, 256, 512), seed).float() * scale
    return w.to(torch.bfloat16)


@pytest.mark.parametrize("B,H", [(3, 4), (64, 128), (70, 16)])
def test_absorb_q_and_project_out(B, H):
    # B = 70: a full chunk of 64 sequences and a ragged one of 6
    w = _weights(H, 201)
    qn = inputs.randn_bf16((B, H, 128), 202)
    x = inputs.randn_bf16((B, H, 512), 203)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ql = mla.absorb_q(qn.cuda(), w.cuda(), status=status)
    o = mla.project_out(x.cuda(), w.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_close(f64(ql).reshape(-1, 512), orc.absorb_q(bits(qn), bits(w)).reshape(-1, 512), "q_latent")
    check_close(f64(o).reshape(-1, 128), orc.project_out(bits(x), bits(w)).reshape(-1, 128), "o")


@pytest.mark.parametrize("fmt", [0, 1])
def test_absorbed_pipeline_equals_naive_mha(fmt):
    B, S, H = 3, 200, 128
    oc = oracle_cache(inputs.randn_bf16((B, S, 512), 211), inputs.randn_bf16((B, S, 64), 212), fmt)
    dc = device_cache(oc)
    w = _weights(H, 213)
    qn = inputs.randn_bf16((B, H, 128), 214)
    qp = inputs.randn_bf16((B, H, 64), 215)
    ends = np.array([200, 61, 1], np.int32)
    ql = mla.absorb_q(qn.cuda(), w.cuda())
    out, _ = mla.decode(dc, ql, qp.cuda(), torch.from_numpy(ends).cuda(), S, 0.3)
    o = mla.project_out(out, w.cuda())
    ref, _ = orc.decode_naive(oc, orc.bf16_bits_to_f64(bits(w)), orc.bf16_bits_to_f64(bits(qn)), bits(qp),
                              ends, 0.3)
    check_close(f64(o).reshape(-1, 128), ref.reshape(-1, 128), "o")
