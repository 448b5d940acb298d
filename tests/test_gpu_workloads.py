"""GPU parity at the full workload sizes, on outputs the oracle computes one
row at a time (first and last rows, tile edges, and a seeded random sample).

Workloads: Llama-3-8B-shaped prefill, 64-row batched decode over random
caches, Gemma-2-shaped sliding-window prefill, and long carried decode
(1024-token prefill, then 1024 single-token steps, checked against one
prefill over all 2048 tokens)."""
import numpy as np
import pytest
import torch

import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import Path, assert_close

pytestmark = pytest.mark.gpu


def _cfg(w, B=None, L=None):
    return oracle.Cfg(B=w.B if B is None else B, H=w.H, Hkv=w.Hkv, L=w.L if L is None else L,
                      D=w.D, rope_dim=w.R, theta=w.theta, scaling=w.scaling,
                      norm_eps=w.norm_eps, window=w.window, softcap=w.softcap)


def _sample_rows(w, L, n_random, seed, extra_l=()):
    rng = np.random.default_rng(seed)
    ls = {0, 1, 63, 64, 127, 128, 129, L // 2, L - 2, L - 1} | set(extra_l)
    ls = sorted(l for l in ls if 0 <= l < L)
    rows = []
    for b in range(w.B):
        for l in ls:
            rows.append((b, int(rng.integers(w.H)), l))
    for _ in range(n_random):
        rows.append((int(rng.integers(w.B)), int(rng.integers(w.H)), int(rng.integers(L))))
    return rows


def _check_rows(out, rows, qr, kr, v, cfg, what):
    want = oracle.attention_rows(qr, kr, v, [0] * cfg.B, cfg, rows)
    o = out.cpu()
    got = np.stack([o[b, h, l].numpy() for b, h, l in rows])
    return assert_close(got, want, what)


def test_llama3_8b_prefill_full_size():
    w = syn.WORKLOADS["llama3_8b_prefill"]
    inp = syn.prefill_inputs(w)
    p = Path(w)
    out, _ = p.prefill(inp["q"], inp["k"], inp["v"])
    p.check_status()
    cfg = _cfg(w)
    qr = oracle.rotate(inp["q"], [0] * w.B, cfg)
    kr = oracle.rotate(inp["k"], [0] * w.B, cfg)
    _check_rows(out, _sample_rows(w, w.L, 160, 1), qr, kr, inp["v"], cfg, "llama prefill")
    # the cache holds every position's rotated key and exact value
    assert torch.equal(p.vc.cpu(), inp["v"])
    kc = p.kc.cpu().numpy()
    assert_close(kc[:, :, ::97], kr[:, :, ::97], "llama k cache", max_tol=1e-5, mean_tol=1e-6)


def test_gemma2_window_full_size():
    w = syn.WORKLOADS["gemma2_window"]
    inp = syn.prefill_inputs(w)
    p = Path(w)
    p.set_norms(inp["q_norm_w"], inp["k_norm_w"])
    out, _ = p.prefill(inp["q"], inp["k"], inp["v"])
    p.check_status()
    cfg = _cfg(w)
    qr = oracle.rotate(inp["q"], [0], cfg, inp["q_norm_w"])
    kr = oracle.rotate(inp["k"], [0], cfg, inp["k_norm_w"])
    rows = _sample_rows(w, w.L, 96, 3, extra_l=(4094, 4095, 4096, 4097, 8191, 12288))
    _check_rows(out, rows, qr, kr, inp["v"], cfg, "gemma window prefill")
    # the ring holds the last 4096 positions, slot = position mod 4096
    vc = p.vc.cpu()
    for pos in (12288, 12289, 16383, 14000):
        assert torch.equal(vc[0, :, pos % 4096], inp["v"][0, :, pos])


def test_batched_decode_full_size():
    w = syn.WORKLOADS["batched_decode"]
    n = syn.cache_lengths(w.seed, w.B, *w.cache_len_range)
    p = Path(w)
    for b in range(w.B):
        p.kc[b].copy_(syn.random_cache_row(w, "k", b))
        p.vc[b].copy_(syn.random_cache_row(w, "v", b))
    tok = syn.decode_token_inputs(w, 0)
    out = p.step(tok["q"], tok["k"], tok["v"], n)        # new token at position n_b
    p.check_status()
    rng = np.random.default_rng(5)
    rows = sorted({int(np.argmin(n)), int(np.argmax(n))} | set(rng.integers(0, w.B, 6).tolist()))
    for b in rows:
        cfg1 = _cfg(w, B=1, L=1)
        kc = syn.random_cache_row(w, "k", b)[None].double().numpy()
        vc = syn.random_cache_row(w, "v", b)[None].double().numpy()
        pos = [int(n[b])]
        kt = oracle.rotate(tok["k"][b:b + 1], pos, cfg1)
        qt = oracle.rotate(tok["q"][b:b + 1], pos, cfg1)
        kc, vc, _ = oracle.append(kt, tok["v"][b:b + 1], pos, cfg1, w.capacity, kc, vc)
        want = oracle.decode(qt, kc, vc, [pos[0] + 1], cfg1)
        assert_close(out[b:b + 1], want, f"batched decode row {b} (n={pos[0]})")


def test_long_carried_decode_full_size():
    w = syn.WORKLOADS["long_decode"]
    T = w.L + w.decode_steps
    inp = syn.prefill_inputs(w, L=T)
    inc = Path(w)
    pre, _ = inc.prefill(inp["q"][:, :, :w.L], inp["k"][:, :, :w.L], inp["v"][:, :, :w.L])
    outs = [pre]
    for t in range(w.L, T):
        sl = slice(t, t + 1)
        outs.append(inc.step(inp["q"][:, :, sl], inp["k"][:, :, sl], inp["v"][:, :, sl], t))
    inc.check_status()
    got = torch.cat(outs, dim=2)
    one = Path(w)
    full, _ = one.prefill(inp["q"], inp["k"], inp["v"])
    one.check_status()
    # decode rows 1024..2047 against the one-shot prefill over 2048 tokens
    assert_close(got[:, :, w.L:].cpu().numpy(), full[:, :, w.L:].double().cpu().numpy(),
                 "carried decode vs one-shot prefill")
    assert torch.equal(inc.vc, one.vc)
    cfg = _cfg(w, L=T)
    qr = oracle.rotate(inp["q"], [0] * w.B, cfg)
    kr = oracle.rotate(inp["k"], [0] * w.B, cfg)
    rows = _sample_rows(w, T, 64, 9, extra_l=(1023, 1024, 1025, 1536))
    _check_rows(got, rows, qr, kr, inp["v"], cfg, "carried decode vs oracle")
