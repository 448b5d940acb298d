"""gqa_attn_prefill_cached: a prefill chunk continuing a carried cache.

The chunk's rows must equal the same rows of one prefill over the whole
sequence (prefix + chunk), computed by the fp64 oracle: for a full cache
(window 0, slot = position) and for a sliding-window ring (slot = position mod
W, the chunk attended before it is appended). Rows may carry different prefix
lengths; the chunk may be longer than the window.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


def _tokens(seed, B, H, Hkv, T, D):
    return (syn.normal(seed, "q", (B, H, T, D)), syn.normal(seed, "k", (B, Hkv, T, D)),
            syn.normal(seed, "v", (B, Hkv, T, D)))


CASES = [
    # B, H, Hkv, D, R, starts, L, window, softcap, norm, fused_rope
    (2, 8, 2, 128, 128, (300, 129), 200, 0, 0.0, False, True),
    (1, 4, 4, 64, 64, (1000,), 257, 0, 30.0, True, True),
    (2, 6, 2, 96, 32, (70, 0), 130, 0, 0.0, False, True),       # q rotated before the kernel
    (2, 8, 2, 128, 128, (100, 40), 150, 64, 0.0, False, True),  # ring, chunk longer than W
    (1, 4, 2, 128, 64, (500,), 300, 256, 50.0, True, True),     # ring with softcap, q/k norm
    (2, 4, 2, 40, 40, (33, 7), 90, 0, 0.0, False, False),       # q pre-rotated, D % 32 != 0
    (1, 4, 2, 256, 256, (300,), 130, 0, 50.0, True, True),      # two output halves per tile
    (2, 4, 2, 192, 64, (200, 50), 100, 128, 0.0, False, False),  # halves over a ring
]


@pytest.mark.parametrize("B,H,Hkv,D,R,starts,L,window,softcap,norm,fused", CASES)
def test_cached_prefill_matches_one_shot_prefill(B, H, Hkv, D, R, starts, L, window, softcap,
                                                 norm, fused):
    theta = 1e4
    max_start = max(starts)
    T = max_start + L
    q_all, k_all, v_all = _tokens(91, B, H, Hkv, T, D)
    qn = syn.norm_weight(91, "qn", D) if norm else None
    kn = syn.norm_weight(91, "kn", D) if norm else None
    rp = g.RopeParams.make(theta=theta, rope_dim=R, max_positions=4096)
    table = g.rope_table(rp, D, dev())
    cap = window if window else max_start + L
    kc = torch.zeros(B, Hkv, cap, D, device=dev())
    vc = torch.zeros_like(kc)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    # row b's sequence: its prefix tokens 0 .. start_b - 1, then the chunk
    q_ch = torch.stack([q_all[b, :, starts[b]:starts[b] + L] for b in range(B)]).contiguous()
    k_ch = torch.stack([k_all[b, :, starts[b]:starts[b] + L] for b in range(B)]).contiguous()
    v_ch = torch.stack([v_all[b, :, starts[b]:starts[b] + L] for b in range(B)]).contiguous()
    zero = torch.zeros(1, dtype=torch.int32, device=dev())
    for b in range(B):                            # each row's prefix, into its cache row
        if starts[b] == 0:
            continue
        kp = k_all[b:b + 1, :, :starts[b]].contiguous().to(dev())
        vp = v_all[b:b + 1, :, :starts[b]].contiguous().to(dev())
        g.kv_cache_append(kp, vp, zero, 0, rp, table, None if kn is None else kn.to(dev()),
                          1e-6, kc[b:b + 1], vc[b:b + 1], window, status)
    st = torch.tensor(starts, dtype=torch.int32, device=dev())
    kd, vd, qd = k_ch.to(dev()), v_ch.to(dev()), q_ch.to(dev())
    knd = None if kn is None else kn.to(dev())
    qnd = None if qn is None else qn.to(dev())
    g.attn_rope_apply(kd, st, max_start, rp, table, knd, 1e-6, status)   # the chunk's keys
    out = torch.empty_like(qd)
    if fused:
        g.gqa_attn_prefill_cached(qd, kd, vd, kc, vc, out, st, max_start, rp, table, qnd, 1e-6,
                                  window, softcap, status=status)
    else:
        qr = qd.clone()
        g.attn_rope_apply(qr, st, max_start, rp, table, qnd, 1e-6, status)
        g.gqa_attn_prefill_cached(qr, kd, vd, kc, vc, out, st, max_start, window=window,
                                  softcap=softcap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy()
    for b in range(B):
        Tb = starts[b] + L
        cfg = oracle.Cfg(B=1, H=H, Hkv=Hkv, L=Tb, D=D, rope_dim=R, theta=theta, window=window,
                         softcap=softcap)
        want, _, _ = oracle.prefill(q_all[b:b + 1, :, :Tb], k_all[b:b + 1, :, :Tb],
                                    v_all[b:b + 1, :, :Tb], [0], cfg, qn, kn)
        assert_close(got[b], want[0, :, starts[b]:], f"row {b} vs one-shot oracle")


def test_cached_prefill_with_empty_prefix_equals_plain_prefill():
    """start = 0 everywhere: the same work as gqa_attn_prefill_rope (same kernel)."""
    B, H, Hkv, L, D = 2, 8, 2, 300, 128
    q, k, v = (t.to(dev()) for t in _tokens(92, B, H, Hkv, L, D))
    rp = g.RopeParams.make(theta=1e4, max_positions=4096)
    table = g.rope_table(rp, D, dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.attn_rope_apply(k, st, 0, rp, table, None, 1e-6, status)
    kc = torch.zeros(B, Hkv, 16, D, device=dev())
    out = torch.empty_like(q)
    g.gqa_attn_prefill_cached(q, k, v, kc, kc, out, st, 0, rp, table, status=status)
    ref = torch.empty_like(q)
    g.gqa_attn_prefill_rope(q, k, v, ref, st, 0, rp, table, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, ref)


def test_cached_prefill_reports_a_start_beyond_max_start():
    B, H, Hkv, L, D = 2, 4, 2, 64, 64
    q, k, v = (t.to(dev()) for t in _tokens(93, B, H, Hkv, L, D))
    kc = torch.zeros(B, Hkv, 128, D, device=dev())
    st = torch.tensor([10, 90], dtype=torch.int32, device=dev())   # 90 > max_start
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    out = torch.empty_like(q)
    g.gqa_attn_prefill_cached(q, k, v, kc, kc, out, st, 20, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & g.DEV_POSITION
    assert torch.isfinite(out).all()
