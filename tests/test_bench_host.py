"""The bench's algorithmic work counts, on the host (no GPU).

The roofline figures divide these counts by measured times, so each is pinned
here: the visible (query, key) pairs against a brute-force count of the mask,
and the workloads' totals against their closed forms.
"""
import bench
from gqa_causal_attention_gb300 import synthetic as syn


def _mask_pairs(L, W):
    # query p sees key m when m <= p and (W == 0 or p - m < W)
    return sum(1 for p in range(L) for m in range(L) if m <= p and (W == 0 or p - m < W))


def test_visible_pairs_match_a_brute_force_mask_count():
    for L in (1, 2, 7, 33, 100):
        for W in (0, 1, 2, 5, L - 1, L, L + 3):
            if W >= 0:
                assert bench.visible_pairs(L, W) == _mask_pairs(L, W), (L, W)


def test_workload_totals():
    llama = syn.WORKLOADS["llama3_8b_prefill"]
    # causal: L (L + 1) / 2 pairs per head; 4 FLOP per pair and head dim (QK^T and PV)
    assert bench.prefill_flops(llama) == 4.0 * 4 * 32 * 128 * (2048 * 2049 // 2)
    assert abs(bench.prefill_flops(llama) - 1.375e11) < 1e-3 * 1.375e11
    gemma = syn.WORKLOADS["gemma2_window"]
    # window 4096 over 16384 positions: a full triangle, then 4096 keys per query
    assert bench.visible_pairs(gemma.L, gemma.window) == 4096 * 4097 // 2 + 12288 * 4096
    assert bench.visible_pairs(gemma.L, gemma.window) == 58_722_304
    assert abs(bench.prefill_flops(gemma) - 9.62e11) < 1e-3 * 9.62e11


def test_prefill_bytes_count_inputs_outputs_and_caches():
    w = syn.WORKLOADS["llama3_8b_prefill"]
    q = w.B * w.H * w.L * w.D * 4                 # q and out
    kv = w.B * w.Hkv * w.L * w.D * 4              # k, v and each cache (capacity = L)
    assert bench.prefill_bytes(w) == 2 * q + 4 * kv == 384 * 2 ** 20


def test_reduce_max_without_a_process_group_is_the_identity():
    assert bench.reduce_max(1.5, None) == 1.5
