"""gqa_attn_prefill_ragged: a ragged batch ("mojolearn.transformer",
TransformerBlock.forward with lengths).

Row b is real at positions [0, lengths[b]); each real output must match the
fp64 oracle's row run alone at its own length, and every padding output must
be exactly +0.0. The padding of q, k and v holds NaN here: it must reach no
output. Covers the persistent tensor-core kernel with q RoPE fused and without
(D % 32 != 0 included), the D > 128 kernel and the CUDA-core kernel
(D % 4 != 0), query tiles that hold no real row, and windows and softcap.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, Hkv, L, D):
    return (syn.normal(seed, "q", (B, H, L, D)), syn.normal(seed, "k", (B, Hkv, L, D)),
            syn.normal(seed, "v", (B, Hkv, L, D)))


def _with_nan_padding(t, lengths):
    t = t.clone()
    for b, n in enumerate(lengths):
        t[b, :, n:] = float("nan")
    return t


def _check_padding(out, lengths):
    for b, n in enumerate(lengths):
        pad = out[b, :, n:]
        assert (pad == 0).all(), f"row {b}: padding not zero"
        assert not torch.signbit(pad).any(), f"row {b}: padding holds -0.0"


CASES = [
    # B, H, Hkv, L, D, R, lengths, window, softcap, norm, fused
    (4, 8, 2, 300, 128, 128, (300, 129, 1, 40), 0, 0.0, False, True),
    (3, 4, 4, 260, 64, 64, (5, 260, 128), 0, 30.0, True, True),
    (2, 6, 2, 200, 96, 64, (77, 200), 64, 0.0, False, True),
    (3, 8, 2, 384, 128, 128, (384, 256, 3), 0, 0.0, False, False),   # q rotated beforehand
    (2, 4, 2, 150, 40, 40, (150, 31), 0, 0.0, False, False),          # D % 32 != 0
    (2, 4, 2, 200, 256, 256, (200, 70), 128, 50.0, True, False),      # two output halves
    (3, 4, 2, 300, 200, 128, (1, 300, 150), 0, 0.0, False, False),    # halves, D % 32 != 0
    (2, 4, 2, 70, 6, 6, (70, 33), 0, 0.0, False, False),              # CUDA-core kernel
]


@pytest.mark.parametrize("B,H,Hkv,L,D,R,lengths,window,softcap,norm,fused", CASES)
def test_ragged_prefill_matches_rows_run_alone(B, H, Hkv, L, D, R, lengths, window, softcap,
                                               norm, fused):
    theta = 1e4
    q, k, v = _inputs(95, B, H, Hkv, L, D)
    qn = syn.norm_weight(95, "qn", D) if norm else None
    kn = syn.norm_weight(95, "kn", D) if norm else None
    rp = g.RopeParams.make(theta=theta, rope_dim=R, max_positions=4096)
    table = g.rope_table(rp, D, dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    zero = torch.zeros(B, dtype=torch.int32, device=dev())
    qd, kd, vd = (_with_nan_padding(t, lengths).to(dev()) for t in (q, k, v))
    qnd = None if qn is None else qn.to(dev())
    knd = None if kn is None else kn.to(dev())
    g.attn_rope_apply(kd, zero, 0, rp, table, knd, 1e-6, status)       # rotated keys
    lens = torch.tensor(lengths, dtype=torch.int32, device=dev())
    out = torch.full_like(qd, 7.0)
    if fused:
        g.gqa_attn_prefill_ragged(qd, kd, vd, out, lens, rp, table, qnd, 1e-6, window, softcap,
                                  status=status)
    else:
        qr = qd.clone()
        g.attn_rope_apply(qr, zero, 0, rp, table, qnd, 1e-6, status)
        g.gqa_attn_prefill_ragged(qr, kd, vd, out, lens, window=window, softcap=softcap,
                                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=R, theta=theta, window=window,
                     softcap=softcap)
    want = oracle.prefill_ragged(q, k, v, lengths, cfg, qn, kn)
    got = out.cpu()
    _check_padding(got, lengths)
    for b, n in enumerate(lengths):
        assert_close(got[b, :, :n].numpy(), want[b, :, :n], f"row {b} (length {n})")


def test_ragged_at_full_length_equals_the_plain_fused_prefill():
    """Every row at length L: the same units and the same arithmetic as
    gqa_attn_prefill_rope with start 0, bit for bit."""
    B, H, Hkv, L, D = 2, 8, 2, 333, 128
    q, k, v = (t.to(dev()) for t in _inputs(96, B, H, Hkv, L, D))
    rp = g.RopeParams.make(theta=5e5, max_positions=4096)
    table = g.rope_table(rp, D, dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.attn_rope_apply(k, st, 0, rp, table, None, 1e-6, status)
    out = torch.empty_like(q)
    ref = torch.empty_like(q)
    g.gqa_attn_prefill_ragged(q, k, v, out, torch.full((B,), L, dtype=torch.int32,
                                                       device=dev()), rp, table, status=status)
    g.gqa_attn_prefill_rope(q, k, v, ref, st, 0, rp, table, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, ref)


def test_ragged_reports_lengths_outside_the_sequence():
    B, H, Hkv, L, D = 3, 4, 2, 64, 64
    q, k, v = (t.to(dev()) for t in _inputs(97, B, H, Hkv, L, D))
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    lens = torch.tensor([0, 64, 90], dtype=torch.int32, device=dev())   # 0 and 90 are invalid
    out = torch.empty_like(q)
    g.gqa_attn_prefill_ragged(q, k, v, out, lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & g.DEV_LENGTH
    # length 0 clamps to an all-padding row, 90 to L
    _check_padding(out.cpu(), [0, 64, 64])
    assert torch.isfinite(out).all()
