"""gqa_block_forward: one decoder block ("mojolearn.transformer",
TransformerBlock.forward with state None) against the fp64 oracle's block:
input RMSNorm, q/k/v projections, attention (q/k norm, RoPE, causal or window,
softcap), o_proj + residual, post RMSNorm, SwiGLU MLP + residual.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


def _weights(seed, dm, H, Hkv, D, IT, qk_norm):
    def mat(name, rows, cols, gain=0.5):
        return syn.normal(seed, name, (rows, cols)) * (gain / np.sqrt(cols))

    w = {
        "input_layernorm.weight": syn.norm_weight(seed, "in_norm", dm),
        "post_attention_layernorm.weight": syn.norm_weight(seed, "post_norm", dm),
        "q_proj.weight": mat("wq", H * D, dm, 1.0),
        "k_proj.weight": mat("wk", Hkv * D, dm, 1.0),
        "v_proj.weight": mat("wv", Hkv * D, dm),
        "o_proj.weight": mat("wo", dm, H * D),
        "gate_proj.weight": mat("wg", IT, dm),
        "up_proj.weight": mat("wu", IT, dm),
        "down_proj.weight": mat("wd", dm, IT),
    }
    if qk_norm:
        w["q_norm.weight"] = syn.norm_weight(seed, "qn", D)
        w["k_norm.weight"] = syn.norm_weight(seed, "kn", D)
    return w


CASES = [
    # B, L, H, Hkv, D, IT, R, window, softcap, qk_norm, offset
    (2, 96, 4, 2, 64, 512, 64, 0, 0.0, False, False),
    (1, 150, 8, 2, 128, 768, 128, 64, 30.0, True, True),
    (2, 40, 2, 1, 40, 96, 32, 0, 0.0, True, False),       # q rotated outside the kernel
]


@pytest.mark.parametrize("B,L,H,Hkv,D,IT,R,window,softcap,qk_norm,offset", CASES + [
    # the Llama-3-8B-shaped block: d_model 4096, 32 query / 8 kv heads, IT 14336
    (1, 256, 32, 8, 128, 14336, 128, 0, 0.0, False, False),
])
def test_block_forward_matches_the_oracle(B, L, H, Hkv, D, IT, R, window, softcap, qk_norm,
                                          offset):
    dm = H * D
    w = _weights(71, dm, H, Hkv, D, IT, qk_norm)
    if offset:                          # Gemma's 1 + w: weights near 0
        for n in ("input_layernorm.weight", "post_attention_layernorm.weight"):
            w[n] = w[n] - 1.0
    x = syn.normal(71, "x", (B, L, dm))
    rp = g.RopeParams.make(theta=1e4, rope_dim=R, max_positions=4096)
    table = g.rope_table(rp, D, dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    wd = {n: t.to(dev()).contiguous() for n, t in w.items()}
    xd = x.to(dev())
    out = torch.empty_like(xd)
    g.gqa_block_forward(xd, out, wd, H, Hkv, rp, table, norm_offset=offset, window=window,
                        softcap=softcap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=R, theta=1e4, window=window,
                     softcap=softcap)
    want = oracle.block_forward(x, w, cfg, norm_offset=offset)
    assert_close(out.cpu().numpy(), want, "decoder block")
