"""The opt-in non-finite input check ("mojolearn.transformer", TransformerBlock:
non-finite weights, inputs or cache values raise an error before any
computation).

A NaN or inf is planted on the host into one input; with the check on the call
reports ATTN_DEV_NONFINITE and writes nothing (outputs keep a sentinel, tensors
updated in place keep their values). Values the call does not read -- cache
slots beyond a row's length, padding of a ragged row -- are not checked.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import dev

pytestmark = pytest.mark.gpu

SENT = 7.25


@pytest.fixture
def check_on():
    prev = g.attn_set_check_finite(1)
    yield
    g.attn_set_check_finite(prev)


def _status():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def _bits(st):
    torch.cuda.synchronize()
    return int(st.item())


def _decode_inputs(B=3, H=8, Hkv=2, D=64, cap=96):
    kc = syn.normal(3, "kc", (B, Hkv, cap, D))
    vc = syn.normal(3, "vc", (B, Hkv, cap, D))
    q = syn.normal(3, "q", (B, H, 1, D))
    return q, kc, vc


def _decode(q, kc, vc, lens, st):
    B, H, _, D = q.shape
    Hkv, cap = kc.shape[1], kc.shape[2]
    out = torch.full((B, H, 1, D), SENT, device=dev())
    cl = torch.tensor(lens, dtype=torch.int32, device=dev())
    ws = torch.empty(max(4, g.gqa_attn_decode_workspace_size(B, H, Hkv, D, max(lens), 0) // 4),
                     device=dev())
    g.gqa_attn_decode(q.to(dev()), kc.to(dev()), vc.to(dev()), cl, max(lens), out, 0, 0.0,
                      0.0, ws, st)
    return out


@pytest.mark.parametrize("where", ["q", "k_slot", "v_slot", "inf"])
def test_decode_refuses_non_finite_reads(check_on, where):
    q, kc, vc = _decode_inputs()
    lens = (10, 96, 40)
    if where == "q":
        q[1, 3, 0, 5] = float("nan")
    elif where == "k_slot":
        kc[2, 1, 39, 0] = float("nan")          # the last live slot of row 2
    elif where == "v_slot":
        vc[0, 0, 0, 63] = float("nan")
    else:
        kc[1, 0, 95, 7] = float("inf")
    st = _status()
    out = _decode(q, kc, vc, lens, st)
    assert _bits(st) == g.DEV_NONFINITE
    assert bool((out == SENT).all())


def test_decode_ignores_slots_it_does_not_read(check_on):
    q, kc, vc = _decode_inputs()
    lens = (10, 96, 40)
    st0 = _status()
    ref = _decode(q, kc, vc, lens, st0)
    kc[0, 1, 10:, :] = float("nan")              # beyond row 0's length
    vc[2, 0, 40:, 3] = float("inf")
    st = _status()
    out = _decode(q, kc, vc, lens, st)
    assert _bits(st) == 0 and _bits(st0) == 0
    assert torch.equal(out, ref)


def test_check_off_does_not_look():
    prev = g.attn_set_check_finite(0)
    try:
        q, kc, vc = _decode_inputs()
        q[0, 0, 0, 0] = float("nan")
        st = _status()
        out = _decode(q, kc, vc, (10, 96, 40), st)
        assert _bits(st) == 0
        assert torch.isnan(out[0, 0]).all() and torch.isfinite(out[1:]).all()
    finally:
        g.attn_set_check_finite(prev)


def test_bit_stays_and_later_checked_calls_skip(check_on):
    q, kc, vc = _decode_inputs()
    bad = q.clone()
    bad[0, 0, 0, 0] = float("nan")
    st = _status()
    _decode(bad, kc, vc, (10, 96, 40), st)
    out = _decode(q, kc, vc, (10, 96, 40), st)   # clean inputs, same status word
    assert _bits(st) == g.DEV_NONFINITE
    assert bool((out == SENT).all())
    st.zero_()
    out = _decode(q, kc, vc, (10, 96, 40), st)
    assert _bits(st) == 0 and torch.isfinite(out).all()


def test_rope_and_append_leave_everything_untouched(check_on):
    B, H, Hkv, L, D, cap = 2, 4, 2, 24, 64, 32
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    table = g.rope_table(rp, D, dev())
    start = torch.zeros(B, dtype=torch.int32, device=dev())
    x = syn.normal(4, "x", (B, H, L, D)).to(dev())
    x[1, 2, 5, 9] = float("nan")
    x0 = x.clone()
    st = _status()
    g.attn_rope_apply(x, start, 0, rp, table, None, 1e-6, st)
    assert _bits(st) == g.DEV_NONFINITE
    assert torch.equal(torch.nan_to_num(x, nan=-1.0), torch.nan_to_num(x0, nan=-1.0))

    k = syn.normal(4, "k", (B, Hkv, L, D)).to(dev())
    v = syn.normal(4, "v", (B, Hkv, L, D)).to(dev())
    v[0, 1, 23, 0] = float("inf")
    k0 = k.clone()
    kc = torch.full((B, Hkv, cap, D), SENT, device=dev())
    vc = torch.full((B, Hkv, cap, D), SENT, device=dev())
    st = _status()
    g.kv_cache_append(k, v, start, 0, rp, table, None, 1e-6, kc, vc, 0, st)
    assert _bits(st) == g.DEV_NONFINITE
    assert torch.equal(k, k0)
    assert bool((kc == SENT).all()) and bool((vc == SENT).all())


@pytest.mark.parametrize("D", [128, 40])       # tensor-core and CUDA-core prefill
def test_prefill_refuses_non_finite_q(check_on, D):
    B, H, Hkv, L = 2, 4, 2, 150
    q = syn.normal(5, "q", (B, H, L, D)).to(dev())
    k = syn.normal(5, "k", (B, Hkv, L, D)).to(dev())
    v = syn.normal(5, "v", (B, Hkv, L, D)).to(dev())
    q[1, 0, 149, 2] = float("nan")
    out = torch.full_like(q, SENT)
    st = _status()
    g.gqa_attn_prefill(q, k, v, out, status=st)
    assert _bits(st) == g.DEV_NONFINITE
    assert bool((out == SENT).all())


def test_ragged_padding_is_not_checked(check_on):
    B, H, Hkv, L, D = 2, 4, 2, 130, 64
    q = syn.normal(6, "q", (B, H, L, D)).to(dev())
    k = syn.normal(6, "k", (B, Hkv, L, D)).to(dev())
    v = syn.normal(6, "v", (B, Hkv, L, D)).to(dev())
    lengths = torch.tensor([100, 130], dtype=torch.int32, device=dev())
    for t in (q, k, v):
        t[0, :, 100:] = float("nan")
    out = torch.full_like(q, SENT)
    st = _status()
    g.gqa_attn_prefill_ragged(q, k, v, out, lengths, status=st)
    assert _bits(st) == 0
    assert torch.isfinite(out).all()
    k[1, 1, 129, 0] = float("nan")                # a real row of batch row 1
    st = _status()
    out2 = torch.full_like(q, SENT)
    g.gqa_attn_prefill_ragged(q, k, v, out2, lengths, status=st)
    assert _bits(st) == g.DEV_NONFINITE
    assert bool((out2 == SENT).all())


def test_cached_prefill_checks_only_the_prefix_it_reads(check_on):
    B, H, Hkv, L, D, W = 1, 4, 2, 64, 64, 48
    q = syn.normal(8, "q", (B, H, L, D)).to(dev())
    k = syn.normal(8, "k", (B, Hkv, L, D)).to(dev())
    v = syn.normal(8, "v", (B, Hkv, L, D)).to(dev())
    kc = syn.normal(8, "kc", (B, Hkv, W, D)).to(dev())
    vc = syn.normal(8, "vc", (B, Hkv, W, D)).to(dev())
    start = torch.tensor([100], dtype=torch.int32, device=dev())
    # the chunk at 100 reads positions 53..99 of the ring (W - 1 = 47 of them): slots
    # 53 mod 48 = 5 .. 99 mod 48 = 3; slot 4 (position 52) is not read
    kc[0, 0, 4, :] = float("nan")
    out = torch.full_like(q, SENT)
    st = _status()
    g.gqa_attn_prefill_cached(q, k, v, kc, vc, out, start, 100, window=W, status=st)
    assert _bits(st) == 0 and torch.isfinite(out).all()
    kc[0, 0, 5, 1] = float("nan")                 # position 53: read
    out = torch.full_like(q, SENT)
    st = _status()
    g.gqa_attn_prefill_cached(q, k, v, kc, vc, out, start, 100, window=W, status=st)
    assert _bits(st) == g.DEV_NONFINITE
    assert bool((out == SENT).all())


def test_block_refuses_a_non_finite_weight(check_on):
    B, L, H, Hkv, D, IT = 1, 64, 4, 2, 64, 256
    dm = H * D
    w = {
        "input_layernorm.weight": syn.norm_weight(9, "a", dm),
        "post_attention_layernorm.weight": syn.norm_weight(9, "b", dm),
        "q_proj.weight": syn.normal(9, "wq", (dm, dm)) / np.sqrt(dm),
        "k_proj.weight": syn.normal(9, "wk", (Hkv * D, dm)) / np.sqrt(dm),
        "v_proj.weight": syn.normal(9, "wv", (Hkv * D, dm)) / np.sqrt(dm),
        "o_proj.weight": syn.normal(9, "wo", (dm, dm)) / np.sqrt(dm),
        "gate_proj.weight": syn.normal(9, "wg", (IT, dm)) / np.sqrt(dm),
        "up_proj.weight": syn.normal(9, "wu", (IT, dm)) / np.sqrt(dm),
        "down_proj.weight": syn.normal(9, "wd", (dm, IT)) / np.sqrt(IT),
    }
    w["down_proj.weight"][17, 200] = float("nan")
    wd = {n: t.to(dev()).contiguous() for n, t in w.items()}
    rp = g.RopeParams.make(theta=1e4, max_positions=128)
    table = g.rope_table(rp, D, dev())
    x = syn.normal(9, "x", (B, L, dm)).to(dev())
    out = torch.full_like(x, SENT)
    st = _status()
    g.gqa_block_forward(x, out, wd, H, Hkv, rp, table, status=st)
    assert _bits(st) == g.DEV_NONFINITE
    assert bool((out == SENT).all())
