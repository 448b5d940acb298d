"""The decode entry point that allocates nothing (gqa_attn_decode_static).

It serves callers that cannot allocate device memory, such as a plug-in
inside a framework that owns all device memory, or a serving path that must
not allocate after start-up: its split-KV scratch is a fixed array inside the
library. This file sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.

Two calls in a row, through the C ABI, must match gqa_attn_decode (which uses
a caller workspace) within the parity tolerance.
"""
import ctypes

import pytest
import torch

import gqa_causal_attention_gb300 as g
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import TOL_MAX, TOL_MEAN, assert_close, dev

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
    for out in outs:
        assert_close(out, ref.double().cpu().numpy(), "static vs workspace decode",
                     max_tol=TOL_MAX, mean_tol=TOL_MEAN)


def test_static_scratch_refuses_sizes_beyond_the_array():
    # 64 rows x 256 heads x (tens of splits) x 258 floats: far more than 32 MiB
    B, H, Hkv, D, maxlen = 64, 256, 8, 256, 8193
    assert g.gqa_attn_decode_workspace_size(B, H, Hkv, D, maxlen, 0) > (32 << 20)
    lib = g.load()
    P = ctypes.c_void_p(0x100000)        # never dereferenced: refused before any launch
    rc = lib.gqa_attn_decode_static(P, P, P, P, maxlen, P, B, H, Hkv, D, 8193, 0, 0.0, 0.0,
                                    None, None)
    assert rc == -5
