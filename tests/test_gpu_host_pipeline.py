"""gqa_attn_prefill_from_host: a prefill step whose inputs and output live in host memory.

The call copies q, k, v in and the output back chunk by chunk (groups of batch rows, or
slices of a row's kv heads) on two copy streams around the kernels. Checked against the
fp64 oracle, and against the same kernels run over the whole batch from device-resident
inputs (kv_cache_append then gqa_attn_prefill_rope): outputs within the parity bar, caches
and rotated k bit for bit.
Covers kv-head slices (a short last slice too), one-row chunks, two rows per chunk with a
short last chunk, a single chunk (head rows not a whole number of 16-byte units), a window
ring, the CUDA-core head dims, and longer sequences with every start 0."""
import pytest
import torch

import gqa_causal_attention_gb300 as g
import oracle
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, L, D, R, scaling, norm, window, softcap, start, capacity
    (3, 8, 2, 300, 128, 128, ("llama3", 8.0, 1.0, 4.0, 8192), True, 0, 30.0, (0, 5, 40), 400),
    (2, 4, 2, 130, 256, 256, None, True, 100, 50.0, (0, 7), 100),
    (9, 4, 4, 64, 64, 64, None, False, 0, 0.0, (0,) * 9, 64),
    (3, 7, 7, 40, 64, 64, None, False, 0, 0.0, (0, 2, 9), 64),
    (17, 2, 1, 33, 32, 32, None, True, 0, 0.0, tuple(range(17)), 64),
    (2, 2, 1, 3, 6, 6, None, False, 0, 0.0, (0, 1), 5),
    (4, 8, 2, 200, 128, 128, ("llama3", 8.0, 1.0, 4.0, 8192), True, 0, 0.0, (0,) * 4, 256),
    (2, 4, 2, 130, 256, 256, None, True, 64, 50.0, (0, 0), 64),
    (2, 8, 2, 700, 128, 64, None, True, 0, 20.0, (0, 0), 700),
    (1, 4, 1, 2100, 64, 64, ("llama3", 8.0, 1.0, 4.0, 8192), False, 0, 0.0, (0,), 2200),
]


@pytest.mark.parametrize("B,H,Hkv,L,D,R,scaling,norm,window,softcap,start,capacity", CASES)
def test_prefill_from_host_matches_device_path_and_oracle(B, H, Hkv, L, D, R, scaling, norm,
                                                          window, softcap, start, capacity):
    theta, eps = 1e4, 1e-6
    q = syn.normal(61, "q", (B, H, L, D))
    k = syn.normal(61, "k", (B, Hkv, L, D))
    v = syn.normal(61, "v", (B, Hkv, L, D))
    qn = syn.norm_weight(61, "qn", D) if norm else None
    kn = syn.norm_weight(61, "kn", D) if norm else None
    max_start = max(start)
    rp = g.RopeParams.make(theta=theta, rope_dim=R, max_positions=4096, scaling=scaling)
    table = g.rope_table(rp, D, dev())
    st = torch.tensor(start, dtype=torch.int32, device=dev())
    qnd = None if qn is None else qn.to(dev())
    knd = None if kn is None else kn.to(dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())

    # the same kernels over the whole batch, inputs already on the device
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    kc_ref = torch.zeros(B, Hkv, capacity, D, device=dev())
    vc_ref = torch.zeros_like(kc_ref)
    g.kv_cache_append(kd, vd, st, max_start, rp, table, knd, eps, kc_ref, vc_ref, window, status)
    out_ref = torch.empty_like(qd)
    g.gqa_attn_prefill_rope(qd, kd, vd, out_ref, st, max_start, rp, table, qnd, eps, window,
                            softcap, 0.0, status=status)

    # from pinned host memory, twice in a row through the same copy streams
    hq, hk, hv = (t.contiguous().pin_memory() for t in (q, k, v))
    bq, bk, bv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    bout = torch.empty_like(qd)
    kc = torch.zeros_like(kc_ref)
    vc = torch.zeros_like(kc_ref)
    outs = []
    for _ in range(2):
        hout = torch.full(q.shape, float("nan")).pin_memory()
        g.gqa_attn_prefill_from_host(hq, hk, hv, hout, bq, bk, bv, bout, kc, vc, st, max_start,
                                     rp, table, qnd, knd, eps, window, softcap, 0.0,
                                     status=status)
        outs.append(hout)
    torch.cuda.current_stream().synchronize()
    assert int(status.item()) == 0

    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=R, theta=theta, scaling=scaling,
                     window=window, softcap=softcap, norm_eps=eps)
    want, _, _ = oracle.prefill(q, k, v, list(start), cfg, qn, kn)
    for hout in outs:
        assert_close(hout, want, "from-host prefill vs oracle")
        assert_close(hout, out_ref.double().cpu().numpy(), "from host vs device-resident",
                     max_tol=2e-3, mean_tol=5e-5)
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref), "caches differ"
    assert torch.equal(bk, kd), "rotated k differs"
