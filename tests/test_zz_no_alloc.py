"""The decode entry point that allocates nothing (gqa_attn_decode_static).

It serves callers that cannot allocate device memory, such as a plug-in
inside a framework that owns all device memory, or a serving path that must
not allocate after start-up: its split-KV scratch is a fixed array inside the
library. This file sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.

Two calls in a row, through the C ABI, must give the bits of gqa_attn_decode
(which uses a caller workspace): both run the same kernels with the same split
plan, so any difference would mean a wrong plan or a stale scratch address.
"""
import ctypes

import pytest
import torch

import gqa_causal_attention_gb300 as g
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import dev

pytestmark = pytest.mark.gpu


def _decode_pair(B, H, Hkv, D, cap, window, softcap, lengths, seed):
    kc = syn.normal(seed, "kc", (B, Hkv, cap, D)).to(dev())
    vc = syn.normal(seed, "vc", (B, Hkv, cap, D)).to(dev())
    q = syn.normal(seed, "q", (B, H, 1, D)).to(dev())
    cl = torch.tensor(lengths, dtype=torch.int32, device=dev())
    maxlen = int(max(lengths))
    ws = torch.empty(max(4, g.gqa_attn_decode_workspace_size(B, H, Hkv, D, maxlen, window) // 4),
                     device=dev())
    ref = torch.empty_like(q)
    g.gqa_attn_decode(q, kc, vc, cl, maxlen, ref, window, softcap, 0.0, ws)
    lib = g.load()
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):                   # two calls in a row share the static scratch
        out = torch.full_like(q, float("nan"))
        rc = lib.gqa_attn_decode_static(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
            ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(cl.data_ptr()), maxlen,
            ctypes.c_void_p(out.data_ptr()), B, H, Hkv, D, cap, window, softcap, 0.0,
            ctypes.c_void_p(status.data_ptr()), stream)
        assert rc == 0, g.attn_status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ref, outs


@pytest.mark.parametrize("B,H,Hkv,D,cap,window,softcap,lengths", [
    (4, 32, 8, 128, 3000, 0, 0.0, (1, 513, 2999, 3000)),
    (3, 16, 8, 256, 64, 64, 50.0, (5, 64, 900)),
])
def test_static_scratch_decode_matches_workspace_decode(B, H, Hkv, D, cap, window, softcap,
                                                        lengths):
    ref, outs = _decode_pair(B, H, Hkv, D, cap, window, softcap, lengths, seed=41)
    assert torch.isfinite(ref).all()
    for out in outs:
        assert torch.equal(out, ref), (out - ref).abs().max().item()

