"""GPU parity of every step of the hot path against the fp64 oracle, at sizes
the oracle finishes in seconds that still span several tiles and a ragged
tail. Floating-point outputs must stay within max|err| 5e-3 and mean|err|
5e-4; cache slots and copied values must match bit for bit."""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import Path, assert_close, dev, rope_params

pytestmark = pytest.mark.gpu


def _wl(**kw):
    base = dict(name="t", seed=11, B=2, H=4, Hkv=2, D=64, L=64, theta=1e4)
    base.update(kw)
    return syn.Workload(**base)


def _cfg(w, L=None, B=None):
    return oracle.Cfg(B=w.B if B is None else B, H=w.H, Hkv=w.Hkv, L=w.L if L is None else L,
                      D=w.D, rope_dim=w.R, theta=w.theta, scaling=w.scaling,
                      norm_eps=w.norm_eps, window=w.window, softcap=w.softcap)


# ----------------------------------------------------------------------------- tiny workload


def test_tiny_workload_prefill_then_decode():
    """16-token prefill then 4 decode steps at positions 16..19."""
    w = syn.WORKLOADS["tiny"]
    inp = syn.prefill_inputs(w, L=20)
    p = Path(w, capacity=20)
    out, _ = p.prefill(inp["q"][:, :, :16], inp["k"][:, :, :16], inp["v"][:, :, :16])
    outs = [out]
    for t in range(16, 20):
        sl = slice(t, t + 1)
        outs.append(p.step(inp["q"][:, :, sl], inp["k"][:, :, sl], inp["v"][:, :, sl], t))
    p.check_status()
    got = torch.cat(outs, dim=2)
    want, qr, kr = oracle.prefill(inp["q"], inp["k"], inp["v"], [0], _cfg(w, L=20))
    assert_close(got, want, "tiny")
    # cache: values copied exactly, keys rotated, every slot written once
    np.testing.assert_array_equal(p.vc.cpu().numpy(), inp["v"].numpy())
    assert_close(p.kc, kr, "tiny k cache", max_tol=1e-5, mean_tol=1e-6)


# ----------------------------------------------------------------------------- RoPE


@pytest.mark.parametrize("D,R,scaling,norm,B,H,L", [
    (16, 0, None, False, 1, 4, 20),
    (128, 0, ("llama3", 8.0, 1.0, 4.0, 8192), False, 2, 8, 77),
    (128, 64, None, True, 2, 3, 33),
    (256, 0, None, True, 1, 4, 40),
    (64, 0, ("linear", 4.0), False, 3, 2, 9),
    (6, 2, None, True, 2, 2, 5),
    (40, 24, None, False, 1, 3, 7),
])
def test_rope_apply(D, R, scaling, norm, B, H, L):
    w = _wl(B=B, H=H, Hkv=1, D=D, L=L, rope_dim=R, scaling=scaling, theta=5e5,
            max_positions=16384)
    x = syn.normal(3, "x", (B, H, L, D))
    nw = syn.norm_weight(3, "nw", D) if norm else None
    start = torch.tensor([0, 9000, 123][:B], dtype=torch.int32)
    rp = rope_params(w)
    table = g.rope_table(rp, D, dev())
    xd = x.to(dev())
    st = start.to(dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.attn_rope_apply(xd, st, int(start.max()), rp, table,
                      None if nw is None else nw.to(dev()), 1e-6, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = oracle.rotate(x, start, _cfg(w, B=B), nw)
    assert_close(xd, want, "rope", max_tol=2e-5, mean_tol=1e-6)


def test_rope_position_beyond_table_is_reported():
    w = _wl(max_positions=64)
    rp = rope_params(w)
    table = g.rope_table(rp, w.D, dev())
    x = syn.normal(1, "x", (2, 2, 4, w.D)).to(dev())
    before = x.clone()
    st = torch.tensor([0, 61], dtype=torch.int32, device=dev())   # 61 + 3 >= 64
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.attn_rope_apply(x, st, 0, rp, table, None, 1e-6, status)     # host bound understated
    torch.cuda.synchronize()
    assert int(status.item()) & g.DEV_POSITION
    torch.testing.assert_close(x[1], before[1], rtol=0, atol=0)    # row skipped
    assert not torch.equal(x[0, :, 1:], before[0, :, 1:])          # row 0 rotated


# ----------------------------------------------------------------------------- cache append


@pytest.mark.parametrize("window,L,start,rope,norm", [
    (0, 37, (0, 5), True, False),
    (0, 1, (10, 39), True, True),
    (16, 37, (0, 3), True, True),       # chunk longer than the ring
    (16, 5, (14, 30), True, False),     # wraps around the ring
    (0, 8, (0, 0), False, False),       # keys already rotated
])
def test_kv_cache_append(window, L, start, rope, norm):
    B, Hkv, D = 2, 3, 64
    cap = window if window else 48
    w = _wl(B=B, H=Hkv, Hkv=Hkv, D=D, L=L, window=window, theta=1e4)
    k = syn.normal(5, "k", (B, Hkv, L, D))
    v = syn.normal(5, "v", (B, Hkv, L, D))
    kn = syn.norm_weight(5, "kn", D) if norm else None
    st = torch.tensor(start, dtype=torch.int32)
    rp = rope_params(w) if rope else None
    table = g.rope_table(rp, D, dev()) if rope else None
    kc = torch.full((B, Hkv, cap, D), float("nan"), device=dev())
    vc = torch.full_like(kc, float("nan"))
    kd = k.to(dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.kv_cache_append(kd, v.to(dev()), st.to(dev()), int(st.max()), rp, table,
                      None if kn is None else kn.to(dev()), 1e-6, kc, vc, window, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = _cfg(w)
    kr = oracle.rotate(k, st, cfg, kn) if rope else k.double().numpy()
    okc, ovc, written = oracle.append(kr, v, st, cfg, cap)
    got_written = ~torch.isnan(vc[..., 0]).cpu().numpy()
    np.testing.assert_array_equal(got_written, written >= 0)        # exactly these slots
    m = written >= 0
    np.testing.assert_array_equal(vc.cpu().numpy()[m], ovc[m].astype(np.float32))  # exact copy
    assert_close(kc.cpu().numpy()[m], okc[m], "k cache", max_tol=2e-5, mean_tol=1e-6)
    assert_close(kd, kr, "rotated k", max_tol=2e-5, mean_tol=1e-6)
    # the cached keys are the rotated keys, bit for bit
    for b in range(B):
        for l in range(L):
            pos = start[b] + l
            slot = pos % window if window else pos
            if written[b, 0, slot] == pos:
                assert torch.equal(kc[b, :, slot], kd[b, :, l])


# ----------------------------------------------------------------------------- prefill attention


PREFILL_CASES = [
    # B, H, Hkv, L, D, window, softcap
    (1, 4, 2, 16, 16, 0, 0.0),
    (2, 8, 2, 129, 64, 0, 0.0),
    (1, 4, 4, 300, 128, 0, 0.0),
    (2, 8, 1, 200, 128, 0, 30.0),
    (1, 8, 4, 333, 128, 64, 0.0),
    (1, 4, 2, 257, 256, 100, 50.0),
    # D > 128: two output halves per query tile
    (1, 4, 2, 200, 160, 0, 0.0),
    (2, 8, 4, 300, 192, 64, 0.0),
    (1, 6, 3, 260, 224, 0, 20.0),
    (1, 4, 1, 333, 200, 0, 0.0),
    (1, 4, 2, 129, 172, 40, 0.0),
    (1, 2, 1, 1, 256, 0, 0.0),
    (1, 16, 2, 130, 128, 1, 0.0),
    (1, 2, 1, 1, 128, 0, 0.0),
    (2, 6, 3, 75, 6, 0, 5.0),
    (1, 4, 2, 150, 40, 20, 0.0),
    (1, 32, 4, 96, 32, 0, 0.0),
    (1, 4, 1, 520, 96, 0, 0.0),
]


@pytest.mark.parametrize("B,H,Hkv,L,D,window,softcap", PREFILL_CASES)
def test_prefill_attention(B, H, Hkv, L, D, window, softcap):
    q = syn.normal(21, "q", (B, H, L, D))
    k = syn.normal(21, "k", (B, Hkv, L, D))
    v = syn.normal(21, "v", (B, Hkv, L, D))
    out = torch.empty(B, H, L, D, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.gqa_attn_prefill(q.to(dev()), k.to(dev()), v.to(dev()), out, window, softcap, 0.0,
                       status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=0, window=window, softcap=softcap)
    want = oracle.attention(q, k, v, [0] * B, cfg)
    assert_close(out, want, "prefill")


def test_prefill_explicit_scale():
    B, H, Hkv, L, D = 1, 4, 2, 70, 64
    q, k, v = (syn.normal(4, n, (B, h, L, D)) for n, h in (("q", H), ("k", Hkv), ("v", Hkv)))
    out = torch.empty(B, H, L, D, device=dev())
    g.gqa_attn_prefill(q.to(dev()), k.to(dev()), v.to(dev()), out, 0, 0.0, 0.05)
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=0, scale=0.05)
    assert_close(out, oracle.attention(q, k, v, [0], cfg), "scale")


# ----------------------------------------------------------------------------- decode attention


DECODE_CASES = [
    # B, H, Hkv, D, capacity, window, softcap, lengths
    (3, 4, 2, 16, 20, 0, 0.0, (1, 7, 20)),
    (4, 32, 8, 128, 3000, 0, 0.0, (1, 513, 2999, 3000)),
    (2, 64, 8, 128, 700, 0, 0.0, (640, 77)),
    (3, 16, 8, 256, 64, 64, 50.0, (5, 64, 900)),
    (2, 8, 2, 6, 50, 0, 3.0, (50, 2)),
    (5, 8, 8, 64, 1500, 0, 0.0, (1500, 1, 200, 1024, 1025)),
    (2, 12, 1, 96, 300, 0, 0.0, (300, 129)),
    (2, 6, 2, 192, 400, 0, 0.0, (400, 33)),
    (2, 16, 2, 256, 300, 0, 20.0, (300, 100)),
    (1, 4, 4, 128, 5000, 0, 0.0, (4097,)),
    (2, 8, 4, 128, 96, 96, 0.0, (3000, 17)),
    # groups of 8 or more query heads (the head-pair kernel)
    (2, 16, 2, 64, 256, 256, 30.0, (1000, 3)),
    (3, 32, 2, 128, 600, 0, 0.0, (600, 1, 65)),
    (2, 64, 8, 128, 3000, 0, 0.0, (2999, 1400)),              # past 1280 positions
    (2, 64, 8, 128, 1500, 0, 30.0, (1500, 700)),              # softcap, 16-block clusters
    (2, 64, 8, 128, 1000, 0, 30.0, (1000, 300)),              # softcap, 8-block clusters
    (2, 16, 2, 128, 2000, 2000, 0.0, (3000, 1500)),           # wrapped ring past 1280 slots
    (2, 8, 1, 40, 90, 0, 0.0, (90, 9)),
    # 96 groups of 8 heads (more than fit at once as clusters: the one-warp splits)
    (12, 64, 8, 128, 300, 0, 0.0, (300, 1, 129, 64, 65, 200, 2, 299, 150, 100, 33, 257)),
]


@pytest.mark.parametrize("B,H,Hkv,D,cap,window,softcap,lengths", DECODE_CASES)
def test_decode_attention(B, H, Hkv, D, cap, window, softcap, lengths):
    kc = syn.normal(31, "kc", (B, Hkv, cap, D))
    vc = syn.normal(31, "vc", (B, Hkv, cap, D))
    q = syn.normal(31, "q", (B, H, 1, D))
    cl = torch.tensor(lengths, dtype=torch.int32)
    w = _wl(B=B, H=H, Hkv=Hkv, D=D, window=window, softcap=softcap, capacity=cap)
    p = Path(w, capacity=cap)
    p.kc.copy_(kc)
    p.vc.copy_(vc)
    out = p.decode(q.to(dev()), cl, int(cl.max()))
    p.check_status()
    want = oracle.decode(q, kc, vc, cl, _cfg(w, L=1))
    assert_close(out, want, "decode")


def test_decode_bad_length_is_reported():
    B, H, Hkv, D, cap = 2, 4, 2, 64, 100
    w = _wl(B=B, H=H, Hkv=Hkv, D=D, capacity=cap)
    p = Path(w, capacity=cap)
    q = syn.normal(2, "q", (B, H, 1, D)).to(dev())
    out0 = p.decode(q, torch.tensor([10, 10], dtype=torch.int32), 10)
    torch.cuda.synchronize()
    out = torch.full_like(q, 7.0)
    ws = torch.empty(1024, device=dev())
    cl = torch.tensor([10, 0], dtype=torch.int32, device=dev())     # 0 is not a length
    g.gqa_attn_decode(q, p.kc, p.vc, cl, 10, out, workspace=ws, status=p.status)
    torch.cuda.synchronize()
    assert int(p.status.item()) & g.DEV_LENGTH
    assert torch.all(out[1] == 7.0)
    torch.testing.assert_close(out[0], out0[0], rtol=0, atol=0)


def test_gpu_decode_matches_gpu_prefill():
    """Token-by-token GPU decode over the carried cache vs one GPU prefill."""
    w = _wl(B=2, H=8, Hkv=2, D=128, L=96, theta=5e5, softcap=20.0, qk_norm=True, capacity=96)
    inp = syn.prefill_inputs(w)
    one = Path(w)
    one.set_norms(inp["q_norm_w"], inp["k_norm_w"])
    full, _ = one.prefill(inp["q"], inp["k"], inp["v"])
    inc = Path(w)
    inc.set_norms(inp["q_norm_w"], inp["k_norm_w"])
    pre, _ = inc.prefill(inp["q"][:, :, :40], inp["k"][:, :, :40], inp["v"][:, :, :40])
    outs = [pre]
    for t in range(40, 96):
        sl = slice(t, t + 1)
        outs.append(inc.step(inp["q"][:, :, sl], inp["k"][:, :, sl], inp["v"][:, :, sl], t))
    inc.check_status()
    got = torch.cat(outs, dim=2)
    assert_close(got, full.double().cpu().numpy(), "decode vs prefill")
    # the caches written both ways hold the same keys and values
    assert torch.equal(inc.vc, one.vc)
    torch.testing.assert_close(inc.kc, one.kc, rtol=0, atol=0)
