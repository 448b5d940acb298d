"""The carried cache survives a save and reload mid-decode.

"mojolearn.transformer", TransformerState: the cache buffers are plain fp32 that
round-trip exactly. Here they are saved to a file after some decode steps,
loaded into the buffers of a fresh owner, and decoding goes on; every later
output, and the final caches, carry the same bits as a run that never stopped
(the kernels are deterministic: fixed split plans and reduction orders).
"""
import pytest
import torch

from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import Path

pytestmark = pytest.mark.gpu


def _decode(w, inp, stop, path_file):
    p = Path(w)
    p.set_norms(inp["q_norm_w"], inp["k_norm_w"])
    p.prefill(inp["q"][:, :, :32], inp["k"][:, :, :32], inp["v"][:, :, :32])
    outs = []
    for t in range(32, w.L):
        if t == stop:
            p.check_status()
            torch.save({"k_cache": p.kc.cpu(), "v_cache": p.vc.cpu()}, path_file)
            p = Path(w)                               # a fresh owner with zeroed buffers
            p.set_norms(inp["q_norm_w"], inp["k_norm_w"])
            saved = torch.load(path_file)
            p.kc.copy_(saved["k_cache"])
            p.vc.copy_(saved["v_cache"])
        sl = slice(t, t + 1)
        outs.append(p.step(inp["q"][:, :, sl], inp["k"][:, :, sl], inp["v"][:, :, sl], t))
    p.check_status()
    return torch.cat(outs, dim=2), p


@pytest.mark.parametrize("window", [0, 24])
def test_cache_checkpoint_resumes_decode_bit_for_bit(tmp_path, window):
    w = syn.Workload(name="t", seed=13, B=2, H=8, Hkv=2, D=128, L=80, theta=5e5, softcap=20.0,
                     qk_norm=True, window=window, capacity=80)
    inp = syn.prefill_inputs(w)
    straight, p1 = _decode(w, inp, None, tmp_path / "unused.pt")
    resumed, p2 = _decode(w, inp, 57, tmp_path / "cache.pt")
    assert torch.equal(straight, resumed)
    assert torch.equal(p1.kc, p2.kc) and torch.equal(p1.vc, p2.vc)
