"""Failure detection on the GPU, without a fault.

Every wait of the tensor-core pipelines has a limit: when a barrier is not
signalled in time the block raises its abort flag, its other roles stop
waiting, and ATTN_DEV_TIMEOUT lands in the caller's status word. Here a
self-test launch runs that code on barriers that nothing signals, the host
reads the status, and the same context then runs a prefill that matches the
oracle (the stall left nothing broken behind).
"""
import time

import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

ATTN_DEV_TIMEOUT = 8


def test_stalled_wait_reports_timeout_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.attn_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == ATTN_DEV_TIMEOUT
    assert 1.9 <= waited < 60.0, waited          # the wait limit is 2 s of %globaltimer

    B, H, Hkv, L, D = 2, 4, 2, 200, 64
    q = syn.normal(71, "q", (B, H, L, D))
    k = syn.normal(71, "k", (B, Hkv, L, D))
    v = syn.normal(71, "v", (B, Hkv, L, D))
    out = torch.empty(B, H, L, D, device=dev())
    ok = torch.zeros(1, dtype=torch.int32, device=dev())
    g.gqa_attn_prefill(q.to(dev()), k.to(dev()), v.to(dev()), out, status=ok)
    torch.cuda.synchronize()
    assert int(ok.item()) == 0
    want = oracle.attention(q, k, v, [0] * B, oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D))
    assert_close(out, want, "prefill after the stalled-wait self-test")
