"""gqa_attn_prefill_rope: q's RMSNorm + RoPE fused into the prefill.

Checked against the fp64 oracle (norm, rotation and attention from their
definitions), against the unfused sequence attn_rope_apply + gqa_attn_prefill,
and for leaving q untouched. Covers the fused tensor-core path (D % 32 == 0,
D <= 128, rope_dim % 64 == 0) and the shapes that rotate into the workspace
first (D = 256, D = 40, rope_dim 32 or 24)."""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, L, D, R, scaling, norm, window, softcap, start
    (2, 8, 2, 300, 128, 128, ("llama3", 8.0, 1.0, 4.0, 8192), False, 0, 0.0, (0, 100)),
    (1, 4, 2, 257, 64, 64, None, True, 0, 30.0, (5,)),
    (1, 8, 4, 200, 128, 64, None, False, 64, 0.0, (0,)),
    (2, 4, 4, 129, 96, 64, ("linear", 2.0), True, 0, 0.0, (3, 900)),
    (1, 4, 2, 130, 256, 256, None, True, 100, 50.0, (0,)),
    (2, 6, 3, 75, 40, 24, None, False, 0, 0.0, (0, 7)),
    (1, 4, 2, 96, 32, 32, None, False, 0, 0.0, (11,)),
]


@pytest.mark.parametrize("B,H,Hkv,L,D,R,scaling,norm,window,softcap,start", CASES)
def test_prefill_rope_matches_oracle_and_unfused(B, H, Hkv, L, D, R, scaling, norm, window,
                                                 softcap, start):
    theta = 1e4
    q = syn.normal(51, "q", (B, H, L, D))
    k = syn.normal(51, "k", (B, Hkv, L, D))
    v = syn.normal(51, "v", (B, Hkv, L, D))
    qn = syn.norm_weight(51, "qn", D) if norm else None
    kn = syn.norm_weight(51, "kn", D) if norm else None
    st = torch.tensor(start, dtype=torch.int32)
    rp = g.RopeParams.make(theta=theta, rope_dim=R, max_positions=16384, scaling=scaling)
    table = g.rope_table(rp, D, dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    std = st.to(dev())
    qnd = None if qn is None else qn.to(dev())
    knd = None if kn is None else kn.to(dev())
    g.attn_rope_apply(kd, std, int(st.max()), rp, table, knd, 1e-6, status)   # rotated k
    q_before = qd.clone()
    out = torch.empty_like(qd)
    g.gqa_attn_prefill_rope(qd, kd, vd, out, std, int(st.max()), rp, table, qnd, 1e-6, window,
                            softcap, 0.0, status=status)
    # unfused reference on the GPU
    qr = qd.clone()
    g.attn_rope_apply(qr, std, int(st.max()), rp, table, qnd, 1e-6, status)
    out2 = torch.empty_like(qd)
    g.gqa_attn_prefill(qr, kd, vd, out2, window, softcap, 0.0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(qd, q_before), "q was modified"
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=R, theta=theta, scaling=scaling,
                     window=window, softcap=softcap)
    want, _, _ = oracle.prefill(q, k, v, st, cfg, qn, kn)
    assert_close(out, want, "fused prefill vs oracle")
    assert_close(out, out2.double().cpu().numpy(), "fused vs unfused", max_tol=2e-3,
                 mean_tol=5e-5)


def test_prefill_rope_llama_shape_full_size():
    w = syn.WORKLOADS["llama3_8b_prefill"]
    inp = syn.prefill_inputs(w)
    rp = g.RopeParams.make(theta=w.theta, max_positions=w.max_positions, scaling=w.scaling)
    table = g.rope_table(rp, w.D, dev())
    st = torch.zeros(w.B, dtype=torch.int32, device=dev())
    qd, kd, vd = (inp[n].to(dev()) for n in ("q", "k", "v"))
    kc = torch.zeros(w.B, w.Hkv, w.capacity, w.D, device=dev())
    vc = torch.zeros_like(kc)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.kv_cache_append(kd, vd, st, 0, rp, table, None, 1e-6, kc, vc, 0, status)
    out = torch.empty_like(qd)
    g.gqa_attn_prefill_rope(qd, kd, vd, out, st, 0, rp, table, None, 1e-6, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=w.B, H=w.H, Hkv=w.Hkv, L=w.L, D=w.D, theta=w.theta, scaling=w.scaling)
    qr = oracle.rotate(inp["q"], [0] * w.B, cfg)
    kr = oracle.rotate(inp["k"], [0] * w.B, cfg)
    rng = np.random.default_rng(17)
    rows = [(b, int(rng.integers(w.H)), l) for b in range(w.B) for l in (0, 1, 127, 128, 1000,
                                                                          2047)]
    rows += [(int(rng.integers(w.B)), int(rng.integers(w.H)), int(rng.integers(w.L)))
             for _ in range(100)]
    want = oracle.attention_rows(qr, kr, inp["v"], [0] * w.B, cfg, rows)
    o = out.cpu()
    got = np.stack([o[b, h, l].numpy() for b, h, l in rows])
    assert_close(got, want, "fused llama prefill")


def test_prefill_rope_many_units_per_block():
    """512 query tiles on at most one block per SM: every block walks several
    units, so the ring, the Q tiles' own barrier and the cross-unit pipelining
    all come into play (single-unit shapes do not exercise them)."""
    B, H, Hkv, L, D = 1, 64, 8, 1024, 128
    q = syn.normal(61, "q", (B, H, L, D))
    k = syn.normal(61, "k", (B, Hkv, L, D))
    v = syn.normal(61, "v", (B, Hkv, L, D))
    rp = g.RopeParams.make(theta=5e5, max_positions=8192)
    table = g.rope_table(rp, D, dev())
    st = torch.tensor([17], dtype=torch.int32, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    g.attn_rope_apply(kd, st, 17, rp, table, None, 1e-6, status)
    out = torch.empty_like(qd)
    g.gqa_attn_prefill_rope(qd, kd, vd, out, st, 17, rp, table, status=status)
    qr = qd.clone()
    g.attn_rope_apply(qr, st, 17, rp, table, None, 1e-6, status)
    out2 = torch.empty_like(qd)
    g.gqa_attn_prefill(qr, kd, vd, out2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, out2.double().cpu().numpy(), "fused vs unfused", max_tol=2e-3,
                 mean_tol=5e-5)
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, theta=5e5)
    qro = oracle.rotate(q, [17], cfg)
    kro = oracle.rotate(k, [17], cfg)
    rng = np.random.default_rng(3)
    rows = [(0, int(rng.integers(H)), int(rng.integers(L))) for _ in range(64)]
    rows += [(0, h, l) for h in (0, 63) for l in (0, 127, 128, 1023)]
    want = oracle.attention_rows(qro, kro, v, [17], cfg, rows)
    o = out.cpu()
    assert_close(np.stack([o[b, h, l].numpy() for b, h, l in rows]), want, "many units")


@pytest.mark.parametrize("L,start,max_positions", [(300, 212, 512), (3, 1, 4), (130, 0, 130)])
def test_prefill_rope_positions_up_to_the_table_end(L, start, max_positions):
    """The last query position sits on the table's last row (start + L =
    max_positions): accepted, and the rotation matches the oracle's."""
    B, H, Hkv, D = 1, 4, 2, 128
    q = syn.normal(71, "q", (B, H, L, D))
    k = syn.normal(71, "k", (B, Hkv, L, D))
    v = syn.normal(71, "v", (B, Hkv, L, D))
    rp = g.RopeParams.make(theta=1e4, max_positions=max_positions)
    table = g.rope_table(rp, D, dev())
    st = torch.tensor([start], dtype=torch.int32, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    g.attn_rope_apply(kd, st, start, rp, table, None, 1e-6, status)
    out = torch.empty_like(qd)
    g.gqa_attn_prefill_rope(qd, kd, vd, out, st, start, rp, table, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, theta=1e4)
    want, _, _ = oracle.prefill(q, k, v, torch.tensor([start], dtype=torch.int32), cfg)
    assert_close(out, want, "fused prefill at the table end")


@pytest.mark.parametrize("B,H,Hkv,L,D,R,norm,window,softcap", [
    (2, 8, 2, 300, 128, 128, False, 0, 0.0),      # q RoPE inside the kernel
    (1, 4, 2, 130, 96, 32, True, 0, 0.0),         # q rotated into the workspace first
    (1, 4, 2, 260, 256, 256, True, 100, 50.0),    # D = 256 kernel
])
def test_prefill_rope_vt_matches_prefill_rope(B, H, Hkv, L, D, R, norm, window, softcap):
    """gqa_attn_v_transpose + gqa_attn_prefill_rope_vt: vt is v transposed exactly,
    and the attention equals gqa_attn_prefill_rope bit for bit (same kernels)."""
    q = syn.normal(81, "q", (B, H, L, D)).to(dev())
    k = syn.normal(81, "k", (B, Hkv, L, D)).to(dev())
    v = syn.normal(81, "v", (B, Hkv, L, D)).to(dev())
    qn = syn.norm_weight(81, "qn", D).to(dev()) if norm else None
    rp = g.RopeParams.make(theta=1e4, rope_dim=R, max_positions=4096)
    table = g.rope_table(rp, D, dev())
    st = torch.tensor([3] * B, dtype=torch.int32, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    pitch = g.gqa_attn_vt_pitch(L)
    assert pitch >= L and pitch % 4 == 0
    vt = torch.full((B, Hkv, D, pitch), float("nan"), device=dev())
    g.gqa_attn_v_transpose(v, vt)
    torch.cuda.synchronize()
    assert torch.equal(vt[..., :L], v.transpose(2, 3))
    out_vt = torch.empty_like(q)
    g.gqa_attn_prefill_rope_vt(q, k, vt, out_vt, st, 3, rp, table, qn, 1e-6, window, softcap,
                               status=status)
    out = torch.empty_like(q)
    g.gqa_attn_prefill_rope(q, k, v, out, st, 3, rp, table, qn, 1e-6, window, softcap,
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out_vt, out)
