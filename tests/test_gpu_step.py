"""gqa_attn_prefill_step: one prefill step from a fresh cache ("mojolearn.transformer",
TransformerBlock.forward with an empty TransformerState) -- keys and values into the
cache, attention over them -- against the fp64 oracle: the output within the parity
bar, cached values bit for bit, cached keys within fp32 rounding of the oracle's
rotated keys, and k and v left as they were.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev, rope_params

pytestmark = pytest.mark.gpu


CASES = [
    # B, H, Hkv, L, D, R, window, cap, softcap, qk_norm, scaling
    (2, 8, 2, 300, 128, 0, 0, 320, 0.0, False, ("llama3", 8.0, 1.0, 4.0, 8192)),
    (1, 4, 4, 129, 64, 0, 0, 129, 30.0, True, None),
    (2, 6, 2, 200, 128, 64, 0, 256, 0.0, False, None),         # partial rotary
    (1, 4, 2, 300, 128, 0, 128, 128, 0.0, True, None),          # ring shorter than the chunk
    (2, 4, 2, 100, 64, 0, 128, 128, 20.0, False, None),         # ring longer than the chunk
    (1, 4, 2, 260, 256, 0, 64, 64, 50.0, True, None),           # D = 256, q rotated in a pass
    (1, 4, 2, 70, 96, 32, 0, 80, 0.0, False, ("linear", 2.0)),  # q rotated in a pass (R % 64)
    (2, 4, 2, 50, 40, 0, 0, 64, 0.0, True, None),               # CUDA-core head dim
]


@pytest.mark.parametrize("B,H,Hkv,L,D,R,window,cap,softcap,qk_norm,scaling", CASES)
def test_prefill_step_matches_the_oracle(B, H, Hkv, L, D, R, window, cap, softcap, qk_norm,
                                         scaling):
    w = syn.Workload(name="step", seed=21, B=B, H=H, Hkv=Hkv, D=D, L=L, rope_dim=R,
                     theta=5e5, scaling=scaling, window=window, softcap=softcap,
                     qk_norm=qk_norm, max_positions=4096)
    inp = syn.prefill_inputs(w)
    rp = rope_params(w)
    table = g.rope_table(rp, D, dev())
    q, k, v = (inp[n].to(dev()) for n in ("q", "k", "v"))
    k0, v0 = k.clone(), v.clone()
    qn = None if inp["q_norm_w"] is None else inp["q_norm_w"].to(dev())
    kn = None if inp["k_norm_w"] is None else inp["k_norm_w"].to(dev())
    kc = torch.full((B, Hkv, cap, D), float("nan"), device=dev())
    vc = torch.full_like(kc, float("nan"))
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.gqa_attn_prefill_step(q, k, v, out, kc, vc, rp, table, qn, kn, 1e-6, window, softcap,
                            0.0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(k, k0) and torch.equal(v, v0)
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=w.R, theta=5e5, scaling=scaling,
                     window=window, softcap=softcap)
    want, _, kr = oracle.prefill(inp["q"], inp["k"], inp["v"], [0] * B, cfg, inp["q_norm_w"],
                                 inp["k_norm_w"])
    assert_close(out, want, "prefill step")
    kcw, vcw, written = oracle.append(kr, inp["v"], [0] * B, cfg, cap)
    wr = written >= 0
    got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    np.testing.assert_array_equal(got_v[wr], vcw[wr])
    assert np.isnan(got_v[~wr]).all() and np.isnan(got_k[~wr]).all()    # nothing else written
    assert np.abs(got_k[wr] - kcw[wr]).max() <= 2e-5


def test_prefill_step_equals_append_then_prefill():
    """The fused step and the two separate calls agree."""
    B, H, Hkv, L, D = 2, 8, 2, 333, 128
    w = syn.Workload(name="step2", seed=22, B=B, H=H, Hkv=Hkv, D=D, L=L, theta=1e4,
                     qk_norm=True, max_positions=4096)
    inp = syn.prefill_inputs(w)
    rp = rope_params(w)
    table = g.rope_table(rp, D, dev())
    q, k, v = (inp[n].to(dev()) for n in ("q", "k", "v"))
    qn, kn = inp["q_norm_w"].to(dev()), inp["k_norm_w"].to(dev())
    kc1 = torch.zeros(B, Hkv, L, D, device=dev())
    vc1 = torch.zeros_like(kc1)
    kc2, vc2 = kc1.clone(), vc1.clone()
    out1 = torch.empty_like(q)
    out2 = torch.empty_like(q)
    g.gqa_attn_prefill_step(q, k, v, out1, kc1, vc1, rp, table, qn, kn)
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    k2 = k.clone()
    g.kv_cache_append(k2, v, st, 0, rp, table, kn, 1e-6, kc2, vc2)
    g.gqa_attn_prefill_rope(q, k2, v, out2, st, 0, rp, table, qn)
    torch.cuda.synchronize()
    assert torch.equal(vc1, vc2)
    assert (kc1 - kc2).abs().max().item() <= 1e-5
    assert (out1 - out2).abs().max().item() <= 2e-3
