"""Helpers for the GPU parity tests: tolerances and the hot path run through
the library's C ABI (via the package binding)."""
import numpy as np
import torch

import gqa_causal_attention_gb300 as g

# Parity bar against the fp64 oracle on unit-scale outputs.
TOL_MAX = 5e-3
TOL_MEAN = 5e-4


def err_stats(got, want):
    got = got.detach().cpu().numpy() if hasattr(got, "detach") else np.asarray(got)
    want = want.detach().cpu().numpy() if hasattr(want, "detach") else np.asarray(want)
    got = got.astype(np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), "non-finite output"
    e = np.abs(got - want)
    return float(e.max()), float(e.mean())


def assert_close(got, want, what="", max_tol=TOL_MAX, mean_tol=TOL_MEAN):
    mx, mn = err_stats(got, want)
    assert mx <= max_tol and mn <= mean_tol, f"{what}: max|err| {mx:.3e}, mean|err| {mn:.3e}"
    return mx, mn


def dev():
    return torch.device("cuda:0")


def rope_params(w):
    return g.RopeParams.make(theta=w.theta, rope_dim=w.rope_dim, max_positions=w.max_positions,
                             scaling=w.scaling)


class Path:
    """The hot path of one layer on the GPU: q RoPE, K RoPE + cache append,
    prefill attention, and single-token decode over the carried cache."""

    def __init__(self, w, capacity=None, device=None):
        self.w = w
        self.d = device or dev()
        self.rp = rope_params(w)
        self.table = g.rope_table(self.rp, w.D, self.d)
        self.capacity = capacity or (w.window if w.window else w.capacity)
        self.kc = torch.zeros(w.B, w.Hkv, self.capacity, w.D, device=self.d)
        self.vc = torch.zeros_like(self.kc)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.d)
        self.qn = self.kn = None

    def set_norms(self, qn, kn):
        self.qn = None if qn is None else qn.to(self.d)
        self.kn = None if kn is None else kn.to(self.d)

    def prefill(self, q, k, v, start=0):
        """q [B,H,L,D], k, v [B,Hkv,L,D] (host or device); returns (out, rotated k)."""
        w = self.w
        q = q.to(self.d).contiguous().clone()
        k = k.to(self.d).contiguous().clone()
        v = v.to(self.d).contiguous()
        st = torch.full((w.B,), start, dtype=torch.int32, device=self.d)
        g.attn_rope_apply(q, st, start, self.rp, self.table, self.qn, w.norm_eps, self.status)
        g.kv_cache_append(k, v, st, start, self.rp, self.table, self.kn, w.norm_eps, self.kc,
                          self.vc, w.window, self.status)
        out = torch.empty_like(q)
        g.gqa_attn_prefill(q, k, v, out, w.window, w.softcap, 0.0, status=self.status)
        return out, k

    def step(self, q, k, v, pos):
        """One token per row at position pos (int or [B] tensor); returns [B,H,1,D]."""
        w = self.w
        if isinstance(pos, int):
            posv = torch.full((w.B,), pos, dtype=torch.int32, device=self.d)
            maxpos = pos
        else:
            posv = pos.to(self.d, torch.int32)
            maxpos = int(pos.max())
        q = q.to(self.d).contiguous().clone()
        k = k.to(self.d).contiguous().clone()
        v = v.to(self.d).contiguous()
        g.attn_rope_apply(q, posv, maxpos, self.rp, self.table, self.qn, w.norm_eps, self.status)
        g.kv_cache_append(k, v, posv, maxpos, self.rp, self.table, self.kn, w.norm_eps, self.kc,
                          self.vc, w.window, self.status)
        return self.decode(q, posv + 1, maxpos + 1)

    def decode(self, q, cache_len, max_len):
        w = self.w
        nbytes = g.gqa_attn_decode_workspace_size(w.B, w.H, w.Hkv, w.D, max_len, w.window)
        ws = torch.empty(max(4, nbytes // 4), device=self.d)
        out = torch.empty_like(q)
        g.gqa_attn_decode(q, self.kc, self.vc, cache_len.to(self.d, torch.int32), max_len, out,
                          w.window, w.softcap, 0.0, ws, self.status)
        return out

    def check_status(self):
        torch.cuda.synchronize()
        s = int(self.status.item())
        assert s == 0, f"device status {s}"
