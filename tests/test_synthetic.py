"""The seeded input generators (no GPU): deterministic, row-addressable, and
drawn with the distributions the workloads state.

Both the CUDA path and the oracle take their inputs from these generators, and
the full-size GPU tests rebuild single rows of multi-gigabyte tensors from them,
so a row must come out the same whether it is drawn alone or with its batch.
"""
import torch

from gqa_causal_attention_gb300 import synthetic as syn


def test_same_seed_same_bits_and_names_are_independent():
    a = syn.normal(5, "q", (3, 2, 7, 16))
    assert torch.equal(a, syn.normal(5, "q", (3, 2, 7, 16)))
    assert not torch.equal(a, syn.normal(5, "k", (3, 2, 7, 16)))
    assert not torch.equal(a, syn.normal(6, "q", (3, 2, 7, 16)))


def test_a_row_drawn_alone_equals_that_row_of_the_batch():
    shape = (4, 3, 9, 8)
    full = syn.normal(2, "v", shape)
    for b in range(shape[0]):
        assert torch.equal(syn.normal_row(2, "v", shape, b), full[b])
    w = syn.WORKLOADS["llama3_8b_prefill"]
    one = syn.prefill_inputs(w, L=32, B=1)
    two = syn.prefill_inputs(w, L=32, B=2)
    for n in ("q", "k", "v"):
        assert torch.equal(one[n][0], two[n][0])


def test_distributions_match_the_workload_statement():
    x = syn.normal(0, "q", (8, 64, 512))                     # 262,144 draws of N(0, 1)
    assert x.dtype == torch.float32
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    w = syn.norm_weight(0, "q_norm_w", 4096)                # N(1, 0.1)
    assert abs(float(w.mean()) - 1.0) < 0.01 and abs(float(w.std()) - 0.1) < 0.01
    n = syn.cache_lengths(2, 20000, 512, 8192)              # U{512..8192}
    assert n.dtype == torch.int32
    assert int(n.min()) == 512 and int(n.max()) == 8192
    assert abs(float(n.double().mean()) - (512 + 8192) / 2) < 60


def test_workload_shapes():
    llama = syn.WORKLOADS["llama3_8b_prefill"]
    assert (llama.B, llama.L, llama.H, llama.Hkv, llama.D) == (4, 2048, 32, 8, 128)
    assert llama.scaling == ("llama3", 8.0, 1.0, 4.0, 8192) and llama.theta == 5e5
    dec = syn.WORKLOADS["batched_decode"]
    assert (dec.B, dec.H, dec.Hkv, dec.D) == (64, 32, 8, 128)
    assert dec.cache_len_range == (512, 8192) and dec.capacity == 8193
    gem = syn.WORKLOADS["gemma2_window"]
    assert (gem.B, gem.L, gem.H, gem.Hkv, gem.D, gem.window) == (1, 16384, 16, 8, 256, 4096)
    assert gem.softcap == 50.0 and gem.qk_norm
    lng = syn.WORKLOADS["long_decode"]
    assert (lng.B, lng.H, lng.Hkv, lng.D, lng.rope_dim) == (8, 64, 8, 128, 64)
    assert lng.L == 1024 and lng.decode_steps == 1024 and lng.theta == 1e6
