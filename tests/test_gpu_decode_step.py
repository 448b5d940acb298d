"""gqa_attn_decode_step: one decode step ("mojolearn.transformer", TransformerBlock.step)
-- the new token's q and k rotated at position pos[b], k and v stored at their slot,
attention over the cache -- against the fp64 oracle (RoPE, append, decode), per row
at different positions; and a prefill followed by token-by-token steps against one
oracle prefill over the whole sequence.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, D, R, window, cap, softcap, qk_norm, pos
    (4, 64, 8, 128, 64, 0, 2100, 0.0, False, (0, 1, 1030, 2099)),   # 8 heads per KV head
    (3, 32, 8, 128, 0, 0, 700, 30.0, True, (5, 300, 699)),          # 4 heads per KV head
    (2, 8, 4, 64, 0, 0, 300, 0.0, False, (17, 299)),
    (2, 4, 2, 256, 0, 64, 64, 50.0, True, (10, 700)),               # ring, wrapped row
    (2, 4, 2, 40, 0, 0, 600, 0.0, False, (3, 599)),                 # CUDA-core head dim
    (1, 16, 2, 128, 0, 300, 300, 0.0, True, (1000,)),               # ring, 8 heads per KV head
    (2, 32, 2, 128, 64, 0, 600, 0.0, True, (5, 599)),               # 16 heads: two groups write
    (2, 8, 2, 128, 0, 100, 100, 0.0, False, (7, 250)),              # 4 heads, wrapped ring
    (2, 32, 4, 128, 64, 0, 900, 50.0, True, (5, 899)),              # 8 heads, softcap, norms
    # 96 groups of 8 heads: more than fit on the GPU at once as clusters
    (12, 64, 8, 128, 64, 0, 400, 0.0, False, (3, 399, 1, 200, 64, 65, 300, 0, 128, 129, 250, 333)),
]


@pytest.mark.parametrize("B,H,Hkv,D,R,window,cap,softcap,qk_norm,pos", CASES)
def test_decode_step_matches_the_oracle(B, H, Hkv, D, R, window, cap, softcap, qk_norm, pos):
    seed = 31
    R_eff = R or D
    q = syn.normal(seed, "q", (B, H, 1, D))
    k = syn.normal(seed, "k", (B, Hkv, 1, D))
    v = syn.normal(seed, "v", (B, Hkv, 1, D))
    kc = syn.normal(seed, "kc", (B, Hkv, cap, D))
    vc = syn.normal(seed, "vc", (B, Hkv, cap, D))
    qn = syn.norm_weight(seed, "qn", D) if qk_norm else None
    kn = syn.norm_weight(seed, "kn", D) if qk_norm else None
    rp = g.RopeParams.make(theta=5e5, rope_dim=R, max_positions=4096,
                           scaling=("llama3", 8.0, 1.0, 4.0, 8192))
    table = g.rope_table(rp, D, dev())
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    kcd, vcd = kc.to(dev()), vc.to(dev())
    posd = torch.tensor(pos, dtype=torch.int32, device=dev())
    out = torch.full_like(qd, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.gqa_attn_decode_step(qd, kd, vd, out, posd, max(pos), kcd, vcd, rp, table,
                           None if qn is None else qn.to(dev()),
                           None if kn is None else kn.to(dev()), 1e-6, window, softcap, 0.0,
                           status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(qd.cpu(), q) and torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)

    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=1, D=D, rope_dim=R_eff, theta=5e5,
                     scaling=("llama3", 8.0, 1.0, 4.0, 8192), window=window, softcap=softcap)
    qr = oracle.rotate(q, list(pos), cfg, qn)
    kr = oracle.rotate(k, list(pos), cfg, kn)
    kc_o, vc_o, written = oracle.append(kr, v, list(pos), cfg, cap, kc.numpy(), vc.numpy())
    want = oracle.decode(qr, kc_o, vc_o, [p + 1 for p in pos], cfg)
    assert_close(out, want, "decode step")
    got_k, got_v = kcd.cpu().numpy(), vcd.cpu().numpy()
    new = written >= 0
    np.testing.assert_array_equal(got_v, vc_o)                       # v copied, others kept
    np.testing.assert_array_equal(got_k[~new], kc.numpy()[~new])     # untouched slots
    assert np.abs(got_k[new] - kc_o[new]).max() <= 2e-5


@pytest.mark.parametrize("window", [0, 96])
def test_prefill_step_then_decode_steps_equal_one_prefill(window):
    """A 200-token prefill step, then 24 decode steps over the carried cache (full, or a
    96-slot ring that wraps), against the oracle's one-shot prefill of all 224 tokens."""
    B, H, Hkv, D, L0, T = 2, 16, 2, 128, 200, 24
    w = syn.Workload(name="carry", seed=33, B=B, H=H, Hkv=Hkv, D=D, L=L0 + T, theta=1e4,
                     window=window, qk_norm=True, max_positions=1024)
    inp = syn.prefill_inputs(w)
    rp = g.RopeParams.make(theta=1e4, max_positions=1024)
    table = g.rope_table(rp, D, dev())
    cap = window if window else L0 + T
    kc = torch.zeros(B, Hkv, cap, D, device=dev())
    vc = torch.zeros_like(kc)
    qn, kn = inp["q_norm_w"].to(dev()), inp["k_norm_w"].to(dev())
    q, k, v = (inp[n].to(dev()) for n in ("q", "k", "v"))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    out0 = torch.empty(B, H, L0, D, device=dev())
    g.gqa_attn_prefill_step(q[:, :, :L0].contiguous(), k[:, :, :L0].contiguous(),
                            v[:, :, :L0].contiguous(), out0, kc, vc, rp, table, qn, kn, 1e-6,
                            window, status=status)
    outs = [out0]
    ws = torch.empty(g.gqa_attn_decode_step_workspace_size(B, H, Hkv, D, L0 + T, window) // 4
                     + 4, device=dev())
    for t in range(T):
        p = L0 + t
        sl = slice(p, p + 1)
        o = torch.empty(B, H, 1, D, device=dev())
        pos = torch.full((B,), p, dtype=torch.int32, device=dev())
        g.gqa_attn_decode_step(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                               v[:, :, sl].contiguous(), o, pos, p, kc, vc, rp, table, qn, kn,
                               1e-6, window, workspace=ws, status=status)
        outs.append(o)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L0 + T, D=D, theta=1e4, window=window)
    want, _, _ = oracle.prefill(inp["q"], inp["k"], inp["v"], [0] * B, cfg, inp["q_norm_w"],
                                inp["k_norm_w"])
    assert_close(torch.cat(outs, dim=2), want, "prefill + decode steps")


# the prep pass (D = 64); folded into the bulk (4 heads per KV head) and head-pair splits
@pytest.mark.parametrize("H,Hkv,D", [(8, 2, 64), (8, 2, 128), (16, 2, 128)])
def test_decode_step_reports_positions_past_the_table(H, Hkv, D):
    B, cap = 2, 64
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    table = g.rope_table(rp, D, dev())
    q = syn.normal(3, "q", (B, H, 1, D)).to(dev())
    k = syn.normal(3, "k", (B, Hkv, 1, D)).to(dev())
    v = syn.normal(3, "v", (B, Hkv, 1, D)).to(dev())
    kc = torch.zeros(B, Hkv, cap, D, device=dev())
    vc = torch.zeros_like(kc)
    out = torch.full_like(q, 7.0)
    pos = torch.tensor([5, 70], dtype=torch.int32, device=dev())      # 70 >= 64: device check
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.gqa_attn_decode_step(q, k, v, out, pos, 5, kc, vc, rp, table, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & g.DEV_POSITION and st & g.DEV_LENGTH
    assert bool((out[1] == 7.0).all()) and torch.isfinite(out[0]).all()
    assert bool((kc[1] == 0).all())


def test_clustered_decode_step_reports_positions_past_the_table():
    """8 heads per KV head with a row split several ways (the clustered kernel): a row
    whose position is past the table is reported and left alone, the other finished."""
    B, H, Hkv, D, cap = 2, 16, 2, 128, 200
    rp = g.RopeParams.make(theta=1e4, max_positions=256)
    table = g.rope_table(rp, D, dev())
    q = syn.normal(4, "q", (B, H, 1, D)).to(dev())
    k = syn.normal(4, "k", (B, Hkv, 1, D)).to(dev())
    v = syn.normal(4, "v", (B, Hkv, 1, D)).to(dev())
    kc = syn.normal(4, "kc", (B, Hkv, cap, D)).to(dev())
    vc = syn.normal(4, "vc", (B, Hkv, cap, D)).to(dev())
    kc1 = kc[1].clone()
    out = torch.full_like(q, 7.0)
    pos = torch.tensor([150, 300], dtype=torch.int32, device=dev())   # 300 >= 256: device check
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.gqa_attn_decode_step(q, k, v, out, pos, 150, kc, vc, rp, table, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & g.DEV_POSITION and st & g.DEV_LENGTH
    assert bool((out[1] == 7.0).all()) and torch.isfinite(out[0]).all()
    assert torch.equal(kc[1], kc1)


def test_decode_launch_counts():
    """The kernels a decode call and a decode step launch, as the library reports them
    (the bench counts its launches with this)."""
    # 8 heads per KV head at D = 128, 64 groups: one cluster per group, one kernel
    assert g.gqa_attn_decode_launches(8, 64, 8, 128, 1536, 0, 64) == 1
    assert g.gqa_attn_decode_launches(8, 64, 8, 128, 1536, 0) == 1
    # 4 heads per KV head: the split kernel (RoPE/append folded in) and the combine
    assert g.gqa_attn_decode_launches(32, 32, 8, 128, 8192, 0, 128) == 2
    # rotary dims that the split kernel does not fold in: a separate pass first
    assert g.gqa_attn_decode_launches(32, 32, 8, 128, 8192, 0, 4) == 3
    # one split per row: no combine
    assert g.gqa_attn_decode_launches(2, 8, 2, 64, 64, 0) == 1
