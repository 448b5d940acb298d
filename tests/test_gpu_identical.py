"""The identical numeric mode ("mojolearn.transformer", TransformerBlock
numeric_mode 'identical': decoding token by token, or a prefill continued from a
carried cache, gives the same bits as one prefill over the whole sequence).

Parity of gqa_attn_prefill_identical / gqa_attn_decode_identical with the fp64
oracle, then the bitwise identities, with keys appended by kv_cache_append and
queries rotated by attn_rope_apply (full cache and window ring, softcap, q/k
norm).
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


def _i32(vals):
    return torch.tensor(vals, dtype=torch.int32, device=dev())


PARITY = [
    # B, H, Hkv, L, D, R, window, softcap, norm
    (2, 8, 2, 150, 128, 128, 0, 0.0, False),
    (1, 4, 4, 90, 64, 32, 32, 30.0, True),
    (2, 6, 2, 70, 6, 6, 0, 0.0, False),
    (1, 4, 2, 40, 256, 256, 16, 0.0, True),
]


@pytest.mark.parametrize("B,H,Hkv,L,D,R,window,softcap,norm", PARITY)
def test_identical_prefill_and_decode_match_the_oracle(B, H, Hkv, L, D, R, window, softcap,
                                                       norm):
    q, k, v = _inputs(98, B, H, Hkv, L, D)
    qn = syn.norm_weight(98, "qn", D) if norm else None
    kn = syn.norm_weight(98, "kn", D) if norm else None
    rp = g.RopeParams.make(theta=1e4, rope_dim=R, max_positions=1024)
    table = g.rope_table(rp, D, dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    zero = _i32([0] * B)
    qd, kd, vd = (t.to(dev()) for t in (q, k, v))
    qnd = None if qn is None else qn.to(dev())
    knd = None if kn is None else kn.to(dev())
    cap = window if window else L
    kc = torch.zeros(B, Hkv, cap, D, device=dev())
    vc = torch.zeros_like(kc)
    g.kv_cache_append(kd, vd, zero, 0, rp, table, knd, 1e-6, kc, vc, window, status)
    g.attn_rope_apply(qd, zero, 0, rp, table, qnd, 1e-6, status)
    out = torch.empty_like(qd)
    g.gqa_attn_prefill_identical(qd, kd, vd, out, window=window, softcap=softcap, status=status)
    # the last position decoded against the cache
    dec = torch.empty(B, H, 1, D, device=dev())
    g.gqa_attn_decode_identical(qd[:, :, L - 1:L].contiguous(), kc, vc, _i32([L] * B), L, dec,
                                window=window, softcap=softcap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=R, theta=1e4, window=window,
                     softcap=softcap)
    want, _, _ = oracle.prefill(q, k, v, [0] * B, cfg, qn, kn)
    assert_close(out.cpu().numpy(), want, "identical prefill")
    assert_close(dec.cpu().numpy(), want[:, :, L - 1:L], "identical decode")


IDENTITY = [
    # B, H, Hkv, L, D, R, window, softcap, norm, split
    (2, 8, 2, 97, 128, 128, 0, 0.0, False, 40),
    (2, 4, 2, 75, 64, 64, 32, 25.0, True, 50),      # ring shorter than the sequence
    (1, 6, 3, 33, 40, 32, 0, 0.0, True, 1),
]


def _rotated_sequence(B, H, Hkv, L, D, R, window, norm):
    """The whole sequence prefilled once: q rotated by attn_rope_apply, k rotated (in place)
    and appended by kv_cache_append. Returns what the identity checks need."""
    q, k, v = _inputs(99, B, H, Hkv, L, D)
    qn = syn.norm_weight(99, "qn", D).to(dev()) if norm else None
    kn = syn.norm_weight(99, "kn", D).to(dev()) if norm else None
    rp = g.RopeParams.make(theta=1e4, rope_dim=R, max_positions=1024)
    table = g.rope_table(rp, D, dev())
    return q.to(dev()), k.to(dev()), v.to(dev()), qn, kn, rp, table


@pytest.mark.parametrize("B,H,Hkv,L,D,R,window,softcap,norm,split", IDENTITY)
def test_decode_token_by_token_equals_one_prefill_bit_for_bit(B, H, Hkv, L, D, R, window,
                                                              softcap, norm, split):
    q, k, v, qn, kn, rp, table = _rotated_sequence(B, H, Hkv, L, D, R, window, norm)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    cap = window if window else L
    # one prefill over the whole sequence
    qp, kp = q.clone(), k.clone()
    kc = torch.zeros(B, Hkv, cap, D, device=dev())
    vc = torch.zeros_like(kc)
    g.kv_cache_append(kp, v, _i32([0] * B), 0, rp, table, kn, 1e-6, kc, vc, window, status)
    g.attn_rope_apply(qp, _i32([0] * B), 0, rp, table, qn, 1e-6, status)
    full = torch.empty_like(q)
    g.gqa_attn_prefill_identical(qp, kp, v, full, window=window, softcap=softcap, status=status)
    # token by token: append the token, then decode it against the cache
    kc2 = torch.zeros_like(kc)
    vc2 = torch.zeros_like(kc)
    dec = torch.empty_like(q)
    for t in range(L):
        pos = _i32([t] * B)
        kt = k[:, :, t:t + 1].clone()
        vt = v[:, :, t:t + 1].contiguous()
        qt = q[:, :, t:t + 1].clone()
        g.kv_cache_append(kt, vt, pos, t, rp, table, kn, 1e-6, kc2, vc2, window, status)
        g.attn_rope_apply(qt, pos, t, rp, table, qn, 1e-6, status)
        ot = torch.empty_like(qt)
        g.gqa_attn_decode_identical(qt, kc2, vc2, _i32([t + 1] * B), t + 1, ot, window=window,
                                    softcap=softcap, status=status)
        dec[:, :, t:t + 1] = ot
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(dec, full), f"max |diff| {(dec - full).abs().max().item():.3e}"
    # the caches built both ways hold the same bits
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)


@pytest.mark.parametrize("B,H,Hkv,L,D,R,window,softcap,norm,split", IDENTITY)
def test_chunked_continuation_equals_one_prefill_bit_for_bit(B, H, Hkv, L, D, R, window,
                                                             softcap, norm, split):
    q, k, v, qn, kn, rp, table = _rotated_sequence(B, H, Hkv, L, D, R, window, norm)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    cap = window if window else L
    qp, kp = q.clone(), k.clone()
    scratch_k = torch.zeros(B, Hkv, cap, D, device=dev())
    scratch_v = torch.zeros_like(scratch_k)
    g.kv_cache_append(kp, v, _i32([0] * B), 0, rp, table, kn, 1e-6, scratch_k, scratch_v,
                      window, status)
    g.attn_rope_apply(qp, _i32([0] * B), 0, rp, table, qn, 1e-6, status)
    full = torch.empty_like(q)
    g.gqa_attn_prefill_identical(qp, kp, v, full, window=window, softcap=softcap, status=status)
    # chunk 1 from an empty cache, then chunk 2 continued from the cache of chunk 1
    kc = torch.zeros(B, Hkv, cap, D, device=dev())
    vc = torch.zeros_like(kc)
    outs = []
    for s0, s1 in ((0, split), (split, L)):
        pos = _i32([s0] * B)
        qc = q[:, :, s0:s1].clone()
        kcx = k[:, :, s0:s1].clone()
        vcx = v[:, :, s0:s1].contiguous()
        g.attn_rope_apply(qc, pos, s0, rp, table, qn, 1e-6, status)
        # rotate the chunk's keys exactly as the cache append does (into a throwaway
        # cache), attend before appending (a ring's new rows may overwrite the prefix)
        tk, tv = torch.zeros_like(kc), torch.zeros_like(vc)
        g.kv_cache_append(kcx, vcx, pos, s0, rp, table, kn, 1e-6, tk, tv, window, status)
        oc = torch.empty_like(qc)
        g.gqa_attn_prefill_identical(qc, kcx, vcx, oc, pos, s0, kc, vc, window=window,
                                     softcap=softcap, status=status)
        outs.append(oc)
        # append the (already rotated) chunk to the carried cache
        g.kv_cache_append(kcx, vcx, pos, s0, None, None, None, 1e-6, kc, vc, window, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = torch.cat(outs, dim=2)
    assert torch.equal(got, full), f"max |diff| {(got - full).abs().max().item():.3e}"
