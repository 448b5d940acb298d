"""attn_linear: y = x w^T (+ residual) on the tcgen05 tensor cores, the projection
kernel of the decoder block ("mojolearn.transformer", TransformerBlock: bias-free
linear maps, weights in torch's [out, in] layout), against numpy's fp64 product.

The bound comes from the arithmetic: the tensor core reads TF32 operands (each
value's top 19 bits: relative truncation below 2^-10, so a product is off by less
than 2^-9 of its size) and accumulates K products in fp32 (at most K roundings of
2^-24 each of the running sum, which stays below sum_k |x_k w_k|). So every output
satisfies |err| <= (2^-9 + K 2^-24) sum_k |x_k w_k| (+ one rounding of the
residual add). Tile edges: T not a multiple of 128, N not a multiple of 256, K
not a multiple of 32.
"""
import numpy as np
import pytest
import torch

import gqa_causal_attention_gb300 as g
from gqa_causal_attention_gb300 import synthetic as syn

from gpu_util import dev

pytestmark = pytest.mark.gpu


def _check(x, w, y, res=None):
    x64, w64 = x.double().cpu().numpy(), w.double().cpu().numpy()
    want = x64 @ w64.T
    if res is not None:
        want = want + res.double().cpu().numpy()
    got = y.double().cpu().numpy()
    assert np.isfinite(got).all()
    K = x.shape[1]
    mag = np.abs(x64) @ np.abs(w64).T
    bound = (2.0 ** -9 + K * 2.0 ** -24) * mag * (1 + 1e-6) + 2.0 ** -24 * np.abs(want) + 1e-30
    err = np.abs(got - want)
    assert (err <= bound).all(), float((err / bound).max())
    # and the typical error is that of one TF32 truncation of the result (about
    # 0.8 * 2^-10 rms for these inputs), not the size of the bound
    rel = np.sqrt((err ** 2).mean()) / np.sqrt((want ** 2).mean())
    if err.size >= 4096:
        assert rel < 2.0 ** -9.5, rel
    return rel


@pytest.mark.parametrize("T,N,K,with_res", [
    (1, 4, 4, False),
    (200, 260, 100, False),          # ragged in every dimension
    (300, 512, 1024, True),
    (129, 264, 36, True),
    (1000, 1536, 4096, False),       # several tiles per block, full K loop
])
def test_linear_matches_fp64(T, N, K, with_res):
    x = syn.normal(5, "x", (T, K)).to(dev())
    w = (syn.normal(5, "w", (N, K)) / np.sqrt(K)).to(dev())
    res = syn.normal(5, "r", (T, N)).to(dev()) if with_res else None
    y = torch.full((T, N), float("nan"), device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    g.attn_linear(x, w, y, res, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check(x, w, y, res)


def test_linear_residual_in_place():
    T, N, K = 257, 384, 512
    x = syn.normal(6, "x", (T, K)).to(dev())
    w = (syn.normal(6, "w", (N, K)) / np.sqrt(K)).to(dev())
    y = syn.normal(6, "r", (T, N)).to(dev())
    res = y.clone()
    g.attn_linear(x, w, y, y)
    torch.cuda.synchronize()
    _check(x, w, y, res)


def test_linear_llama_projection_shape():
    """The Llama-3-8B-shaped down projection (K = 14336) on 512 tokens."""
    T, N, K = 512, 4096, 14336
    x = syn.normal(7, "x", (T, K)).to(dev())
    w = (syn.normal(7, "w", (N, K)) / np.sqrt(K)).to(dev())
    y = torch.empty(T, N, device=dev())
    g.attn_linear(x, w, y)
    torch.cuda.synchronize()
    _check(x, w, y)
