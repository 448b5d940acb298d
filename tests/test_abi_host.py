"""The C ABI on the host: the library loads without a GPU, exports every
function the header declares, and rejects bad arguments before launching
anything (no test here touches a GPU).

Bad-argument cases pass stand-in pointers, so they run only where no CUDA
device is visible; every case is one the host check must refuse.
"""
import ctypes
import os
import re

import pytest
import torch

import gqa_causal_attention_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")

no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="stand-in pointers are only used without a device")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_four_entry_points():
    fns = declared_functions()
    for name in ("attn_rope_apply", "kv_cache_append", "gqa_attn_prefill", "gqa_attn_decode"):
        assert name in fns


def test_library_exports_every_declared_function():
    lib = g.load()
    raw = ctypes.CDLL(g.library_path())
    missing = [f for f in declared_functions() if not hasattr(raw, f)]
    assert not missing, missing
    assert lib.attn_version().decode().count(".") == 2
    assert "attn_last_cuda_error" in declared_functions()
    assert g.attn_last_cuda_error() == "no CUDA error"     # nothing failed on this thread


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        s = g.attn_status_string(code)
        assert s and s != "unknown status"
    assert g.attn_status_string(-99) == "unknown status"


def test_rope_table_bytes():
    rp = g.RopeParams.make(theta=1e4, max_positions=100)
    assert g.attn_rope_table_bytes(rp, 16) == 100 * 8 * 2 * 4
    rp = g.RopeParams.make(theta=1e4, rope_dim=64, max_positions=0)      # default 8192
    assert g.attn_rope_table_bytes(rp, 128) == 8192 * 32 * 2 * 4
    for bad in (g.RopeParams.make(theta=0.0), g.RopeParams.make(rope_dim=3),
                g.RopeParams.make(rope_dim=32), g.RopeParams.make(scaling=("linear", 0.0)),
                g.RopeParams.make(scaling=("llama3", 8.0, 4.0, 1.0, 8192))):
        assert g.attn_rope_table_bytes(bad, 16) == 0


def test_prefill_workspace_size():
    # tensor-core head dims need V^T with rows padded to a multiple of 4 keys
    assert g.gqa_attn_prefill_workspace_size(2, 8, 130, 128) == 2 * 8 * 128 * 132 * 4
    assert g.gqa_attn_prefill_workspace_size(1, 2, 16, 16) == 16     # CUDA-core path: none
    assert g.gqa_attn_prefill_workspace_size(1, 2, 16, 7) == 0       # odd D: invalid


def test_decode_workspace_size():
    # one split needs no real workspace; many splits need B*H*nsplit*(D+2) floats
    small = g.gqa_attn_decode_workspace_size(1, 4, 2, 16, 20)
    assert 0 < small <= 16
    big = g.gqa_attn_decode_workspace_size(64, 32, 8, 128, 8193)
    assert big % (64 * 32 * 130 * 4) == 0 and big // (64 * 32 * 130 * 4) >= 2
    assert g.gqa_attn_decode_workspace_size(1, 3, 2, 16, 20) == 0     # H % Hkv != 0


P = ctypes.c_void_p(0x100000)        # stand-in, 16-byte aligned, never dereferenced
P_ODD = ctypes.c_void_p(0x100004)    # not 16-byte aligned
S = ctypes.c_void_p(None)


def rp(**kw):
    return ctypes.byref(g.RopeParams.make(**kw))


@no_device
@pytest.mark.parametrize("args,code", [
    # x, B, Hx, L, D, start, max_start, rp, table, norm_w, eps
    ((P, 1, 2, 4, 7, P, 0, rp(), P, None, 1e-6), -2),            # odd D
    ((P, 1, 2, 4, 258, P, 0, rp(), P, None, 1e-6), -2),          # D too large
    ((P, 1, 0, 4, 8, P, 0, rp(), P, None, 1e-6), -2),            # no heads
    ((None, 1, 2, 4, 8, P, 0, rp(), P, None, 1e-6), -1),         # null x
    ((P, 1, 2, 4, 8, None, 0, rp(), P, None, 1e-6), -1),         # null start
    ((P, 1, 2, 4, 8, P, 0, rp(), None, None, 1e-6), -1),         # null table
    ((P, 1, 2, 4, 8, P, 0, rp(rope_dim=10), P, None, 1e-6), -7),  # rope_dim > D
    ((P, 1, 2, 4, 8, P, 0, rp(rope_dim=6, theta=-1.0), P, None, 1e-6), -7),
    ((P_ODD, 1, 2, 4, 8, P, 0, rp(), P, None, 1e-6), -6),        # misaligned
    ((P, 1, 2, 4, 8, P, 8189, rp(), P, None, 1e-6), -3),         # 8189 + 3 >= 8192
    ((P, 1, 2, 4, 8, P, -1, rp(), P, None, 1e-6), -3),
    ((P, 1, 2, 4, 8, P, 97, rp(max_positions=100), P, None, 1e-6), -3),   # 97 + 3 >= 100
])
def test_rope_apply_rejects(args, code):
    lib = g.load()
    assert lib.attn_rope_apply(*args, None, S) == code


@no_device
def test_rope_apply_empty_is_a_no_op():
    lib = g.load()
    assert lib.attn_rope_apply(None, 0, 2, 4, 8, None, 0, rp(), P, None, 1e-6, None, S) == 0
    assert lib.attn_rope_apply(None, 3, 2, 0, 8, None, 0, rp(), P, None, 1e-6, None, S) == 0


@no_device
@pytest.mark.parametrize("over,code", [
    (dict(capacity=10, max_start=7), -4),          # 7 + 4 > 10, no window
    (dict(window=4, capacity=8), -2),               # a ring has exactly W slots
    (dict(window=-1), -2),
    (dict(k=None), -1),
    (dict(v_cache=None), -1),
    (dict(table=None), -1),                         # rp without a table
    (dict(rp=None), -7),                            # a table without rp
    (dict(v=P_ODD), -6),
    (dict(max_start=8190), -3),
    (dict(D=5), -2),
])
def test_append_rejects(over, code):
    a = dict(k=P, v=P, B=1, Hkv=2, L=4, D=8, start=P, max_start=0, rp=rp(), table=P, kn=None,
             eps=1e-6, k_cache=P, v_cache=P, capacity=16, window=0, status=None, stream=S)
    assert set(over) <= set(a)
    a.update(over)
    lib = g.load()
    assert lib.kv_cache_append(*a.values()) == code


@no_device
@pytest.mark.parametrize("over,code", [
    (dict(H=6, Hkv=4), -2),                         # H % Hkv != 0
    (dict(Hkv=0), -2),
    (dict(D=3), -2),
    (dict(window=-2), -2),
    (dict(q=None), -1),
    (dict(out=P_ODD), -6),
    (dict(softcap=float("inf")), -7),
    (dict(scale=float("nan")), -7),
    (dict(D=64, workspace=None), -5),               # the tensor-core path needs V^T scratch
    (dict(D=64, ws_bytes=64), -5),
    (dict(D=64, workspace=P_ODD), -6),
])
def test_prefill_rejects(over, code):
    a = dict(q=P, k=P, v=P, out=P, B=1, H=4, Hkv=2, L=8, D=16, window=0, softcap=0.0,
             scale=0.0, workspace=P, ws_bytes=1 << 30, status=None, stream=S)
    assert set(over) <= set(a)
    a.update(over)
    assert g.load().gqa_attn_prefill(*a.values()) == code


@no_device
@pytest.mark.parametrize("over,code", [
    (dict(max_cache_len=0), -2),
    (dict(max_cache_len=5000, capacity=4096), -4),  # beyond the cache, no window
    (dict(window=8, capacity=16), -2),
    (dict(H=5), -2),
    (dict(cache_len=None), -1),
    (dict(workspace=None), -5),
    (dict(ws_bytes=64), -5),
    (dict(k_cache=P_ODD), -6),
])
def test_decode_rejects(over, code):
    a = dict(q=P, k_cache=P, v_cache=P, cache_len=P, max_cache_len=4000, out=P, B=8, H=4, Hkv=2, D=64,
             capacity=4096, window=0, softcap=0.0, scale=0.0, workspace=P, ws_bytes=1 << 30,
             status=None, stream=S)
    assert set(over) <= set(a)
    a.update(over)
    assert g.load().gqa_attn_decode(*a.values()) == code


def test_binding_refuses_other_dtypes():
    x = torch.zeros(1, 2, 3, 4, dtype=torch.float64)
    with pytest.raises(TypeError):
        g.gqa_attn_prefill(x, x, x, x)
    xb = torch.zeros(1, 2, 3, 4, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        g.gqa_attn_prefill(xb, xb, xb, xb)


@no_device
def test_vt_entry_points_refuse_before_launch():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)
    assert lib.gqa_attn_vt_pitch(10) == 12 and lib.gqa_attn_vt_pitch(16) == 16
    # head dims the tensor-core kernels do not take
    assert lib.gqa_attn_v_transpose(P, P, 1, 2, 16, 6, None) == -2       # ATTN_ERR_SHAPE
    assert lib.gqa_attn_v_transpose(P, P, 1, 2, 16, 20, None) == -2
    assert lib.gqa_attn_v_transpose(P, None, 1, 2, 16, 64, None) == -1    # ATTN_ERR_NULL
    assert lib.gqa_attn_v_transpose(P, ctypes.c_void_p(0x100004), 1, 2, 16, 64, None) == -6
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    st = P
    args = (P, P, P, P, 1, 4, 2, 16, 20, st, 0, ctypes.byref(rp), P, None, 1e-6, 0, 0.0, 0.0,
            None, 0, None, None)
    assert lib.gqa_attn_prefill_rope_vt(*args) == -2                       # D = 20
    # fused shape: no workspace needed; unfused (rope_dim 32): workspace refused
    assert lib.gqa_attn_prefill_rope_vt_workspace_size(1, 4, 16, 64, ctypes.byref(rp)) == 16
    rp32 = g.RopeParams.make(theta=1e4, rope_dim=32, max_positions=64)
    assert lib.gqa_attn_prefill_rope_vt_workspace_size(1, 4, 16, 64, ctypes.byref(rp32)) == \
        4 * 16 * 64 * 4
    args32 = (P, P, P, P, 1, 4, 2, 16, 64, st, 0, ctypes.byref(rp32), P, None, 1e-6, 0, 0.0, 0.0,
              None, 0, None, None)
    assert lib.gqa_attn_prefill_rope_vt(*args32) == -5                     # ATTN_ERR_WORKSPACE


@no_device
def test_cached_prefill_refuses_before_launch():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)

    def call(D=64, capacity=128, max_start=32, window=0, ws=None, wbytes=0, L=16):
        return lib.gqa_attn_prefill_cached(P, P, P, P, P, capacity, P, 1, 4, 2, L, D, P,
                                           max_start, None, None, None, 1e-6, window, 0.0, 0.0,
                                           ws, wbytes, None, None)

    assert call(D=260) == -2                      # head dims past 256
    assert call(D=256) == -5                      # wide heads too (here: no workspace)
    assert call(D=20) == -2
    assert call(window=64, capacity=128) == -2    # a ring holds exactly window slots
    assert call(max_start=200) == -4              # prefix positions without cache slots
    assert call() == -5                           # no workspace
    need = lib.gqa_attn_prefill_cached_workspace_size(1, 4, 2, 16, 64, 32, 0, None)
    # pre [B] + K rows (32 prefix + 16 chunk) + V^T rows of the same keys
    assert need >= 2 * 2 * 48 * 64 * 4
    assert lib.gqa_attn_prefill_cached_workspace_size(1, 4, 2, 16, 64, 1000, 64, None) < need * 3
    assert call(ws=ctypes.c_void_p(0x100004), wbytes=need) == -6


def test_ragged_prefill_refuses_before_launch():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)

    def call(lengths=P, H=4, Hkv=2, D=64, window=0, ws=None, wbytes=0, rp=None, table=None):
        return lib.gqa_attn_prefill_ragged(P, P, P, P, 2, H, Hkv, 16, D, lengths, rp, table,
                                           None, 1e-6, window, 0.0, 0.0, ws, wbytes, None, None)

    assert call(H=6, Hkv=4) == -2                 # H % Hkv != 0
    assert call(D=7) == -2                        # odd head dim
    assert call(window=-1) == -2
    assert call(lengths=None) == -1               # lengths are required
    assert call() == -5                           # no workspace
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    plain = lib.gqa_attn_prefill_ragged_workspace_size(2, 4, 2, 16, 64, None)
    roped = lib.gqa_attn_prefill_ragged_workspace_size(2, 4, 2, 16, 64, ctypes.byref(rp))
    # start = 0 per row, then V^T (2 rows x 2 kv heads x 64 dims x 16 keys)
    assert plain >= 256 + 2 * 2 * 64 * 16 * 4 and roped >= plain
    assert call(ws=ctypes.c_void_p(0x100004), wbytes=plain) == -6
    bad = g.RopeParams.make(theta=1e4, rope_dim=66, max_positions=64)   # R > D
    assert call(rp=ctypes.byref(bad)) == -7
    assert lib.gqa_attn_prefill_ragged(P, P, P, P, 0, 4, 2, 16, 64, None, None, None, None,
                                       1e-6, 0, 0.0, 0.0, None, 0, None, None) == 0   # empty


def test_identical_mode_refuses_before_launch():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)

    def pre(kc=None, vc=None, cap=0, start=None, max_start=0, window=0, H=4, Hkv=2, D=64):
        return lib.gqa_attn_prefill_identical(P, P, P, kc, vc, cap, P, 1, H, Hkv, 16, D, start,
                                              max_start, window, 0.0, 0.0, None, None)

    assert pre(H=6, Hkv=4) == -2
    assert pre(D=9) == -2
    assert pre(kc=P, vc=P, cap=0, start=P) == -2          # a cache needs capacity
    assert pre(kc=P, vc=P, cap=64, start=P, window=32) == -2   # a ring holds window slots
    assert pre(kc=P, vc=None, cap=64, start=P) == -1      # both caches or neither
    assert pre(kc=P, vc=P, cap=64) == -1                  # a cached prefix needs start
    assert pre(max_start=3) == -3                         # start NULL means position 0
    assert pre(kc=P, vc=P, cap=64, start=P, max_start=65) == -4

    def dec(cap=64, max_len=10, window=0, cl=P):
        return lib.gqa_attn_decode_identical(P, P, P, cl, max_len, P, 1, 4, 2, 64, cap, window,
                                             0.0, 0.0, None, None)

    assert dec(max_len=0) == -2
    assert dec(max_len=65) == -4
    assert dec(window=32) == -2
    assert dec(cl=None) == -1


def test_block_forward_refuses_before_launch():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)
    P2 = ctypes.c_void_p(0x200000)
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    w = g._BlockWeights(*([0x100000] * 9 + [0, 0]))

    def call(H=4, Hkv=2, D=16, IT=32, L=8, weights=w, params=rp, ws=None, wbytes=0, out=P2):
        return lib.gqa_block_forward(P, out, 2, L, H, Hkv, D, IT,
                                     None if weights is None else ctypes.byref(weights), 0, 1e-6,
                                     None if params is None else ctypes.byref(params), P, 0, 0.0,
                                     0.0, ws, wbytes, None, None)

    assert call(H=6, Hkv=4) == -2
    assert call(IT=0) == -2
    assert call(IT=30) == -2                       # 16-byte rows for the projections
    assert call(H=1, Hkv=1, D=2) == -2             # d_model = 2
    assert call(weights=None) == -1
    assert call(params=None) == -1
    assert call(out=P) == -2                       # out must not be x
    assert call(L=65) == -3                        # positions reach max_positions
    assert call() == -5                            # no workspace
    need = lib.gqa_block_forward_workspace_size(2, 8, 4, 2, 16, 32, ctypes.byref(rp))
    # normed rows, q, k, v, attention output, activations
    assert need >= 2 * 8 * (3 * 64 + 2 * 32 + 32) * 4
    w2 = g._BlockWeights(*([0x100000] * 8 + [0, 0, 0]))          # no down_proj
    assert call(weights=w2, ws=P, wbytes=need) == -1
    w3 = g._BlockWeights(*([0x100000] * 8 + [0x100004, 0, 0]))   # misaligned down_proj
    assert call(weights=w3, ws=P, wbytes=need) == -6


@no_device
def test_linear_refuses_before_launch():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)

    def call(T=8, N=16, K=32, x=P, w=P, r=None, y=P):
        return lib.attn_linear(x, w, r, y, T, N, K, None, None)

    assert call(K=30) == -2 and call(N=6) == -2 and call(K=0) == -2 and call(T=-1) == -2
    assert call(x=None) == -1 and call(w=None) == -1 and call(y=None) == -1
    assert call(r=ctypes.c_void_p(0x100008)) == -6
    assert call(T=0, x=None) == 0                  # empty: nothing to do


@no_device
def test_prefill_from_host_refuses_before_any_copy():
    lib = g.load()
    P = ctypes.c_void_p(0x100000)
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    need = lib.gqa_attn_prefill_from_host_workspace_size(4, 8, 2, 16, 64, 64, ctypes.byref(rp))
    # 4 rows of 2 kv heads: 8 chunks of one kv head and its 4 query heads each
    assert need == lib.gqa_attn_prefill_rope_workspace_size(1, 4, 1, 16, 64, ctypes.byref(rp))
    # 32 rows: 16 chunks of 2 rows; L * D not a multiple of 4: one chunk of every row
    assert lib.gqa_attn_prefill_from_host_workspace_size(32, 8, 2, 16, 64, 64, ctypes.byref(rp)) \
        == lib.gqa_attn_prefill_rope_workspace_size(2, 8, 2, 16, 64, ctypes.byref(rp))
    assert lib.gqa_attn_prefill_from_host_workspace_size(4, 8, 2, 3, 6, 64, ctypes.byref(rp)) \
        == lib.gqa_attn_prefill_rope_workspace_size(4, 8, 2, 3, 6, ctypes.byref(rp))

    def call(B=4, H=8, Hkv=2, L=16, D=64, max_start=0, capacity=64, window=0, ws=P,
             wbytes=need, qh=P, table=P, dev_q=P, rpp=ctypes.byref(rp)):
        return lib.gqa_attn_prefill_from_host(qh, P, P, P, dev_q, P, P, P, B, H, Hkv, L, D, P,
                                              max_start, rpp, table, None, None, 1e-6, P, P,
                                              capacity, window, 0.0, 0.0, ws, wbytes, None, None)

    assert call(H=6, Hkv=4) == -2                 # H % Hkv != 0
    assert call(D=7) == -2                        # odd head dim
    assert call(window=32, capacity=64) == -2     # a ring holds exactly window slots
    assert call(qh=None) == -1                    # host buffers are required
    assert call(table=None) == -1
    assert call(dev_q=ctypes.c_void_p(0x100004)) == -6
    assert call(max_start=60) == -3               # positions reach max_positions
    assert call(capacity=8) == -4                 # positions without cache slots
    assert call(ws=None) == -5
    assert call(wbytes=need - 4) == -5
    bad = g.RopeParams.make(theta=1e4, rope_dim=66, max_positions=64)
    assert call(rpp=ctypes.byref(bad)) == -7
    assert call(B=0) == 0 and call(L=0) == 0      # empty: nothing to do


@no_device
def test_static_scratch_refuses_sizes_beyond_the_array():
    # 64 rows x 256 heads x (tens of splits) x 258 floats: far more than 32 MiB
    B, H, Hkv, D, maxlen = 64, 256, 8, 256, 8193
    assert g.gqa_attn_decode_workspace_size(B, H, Hkv, D, maxlen, 0) > (32 << 20)
    lib = g.load()
    P = ctypes.c_void_p(0x100000)        # never dereferenced: refused before any launch
    rc = lib.gqa_attn_decode_static(P, P, P, P, maxlen, P, B, H, Hkv, D, 8193, 0, 0.0, 0.0,
                                    None, None)
    assert rc == -5


@no_device
def test_static_scratch_refuses_like_the_workspace_decode():
    """Host refusals come from gqa_attn_decode's own checks, before the size
    check: a bad shape or capacity reports that, not the scratch size."""
    lib = g.load()
    P = ctypes.c_void_p(0x100000)        # never dereferenced: refused before any launch
    big = (64, 256, 8, 256, 8193)        # scratch far beyond the array
    B, H, Hkv, D, maxlen = big
    # H % Hkv != 0 -> shape, even though the scratch would also be too large
    assert lib.gqa_attn_decode_static(P, P, P, P, maxlen, P, B, H, 7, D, 8193, 0, 0.0, 0.0,
                                      None, None) == -2
    # positions beyond the capacity without a window -> capacity
    assert lib.gqa_attn_decode_static(P, P, P, P, maxlen, P, B, H, Hkv, D, 100, 0, 0.0, 0.0,
                                      None, None) == -4
    # a NULL tensor -> null
    assert lib.gqa_attn_decode_static(None, P, P, P, maxlen, P, B, H, Hkv, D, 8193, 0, 0.0,
                                      0.0, None, None) == -1
    # an empty batch is a no-op, as for the workspace decode
    assert lib.gqa_attn_decode_static(None, None, None, None, 0, None, 0, H, Hkv, D, 8193, 0,
                                      0.0, 0.0, None, None) == 0


def test_decode_workspace_sizes_never_shrink_as_the_length_grows():
    """One buffer sized for the largest length must serve every shorter one: the split
    plan's chunk grows in steps, which drops the split count, but the sizes do not."""
    for B, H, Hkv, D, window in ((8, 64, 8, 128, 0), (1, 32, 8, 128, 0), (32, 32, 8, 128, 0),
                                 (3, 12, 3, 96, 0), (2, 16, 2, 256, 1500)):
        prev = prev_step = 0
        for n in list(range(1, 9000, 7)) + [16384, 16385, 40000, 100000]:
            size = g.gqa_attn_decode_workspace_size(B, H, Hkv, D, n, window)
            step = g.gqa_attn_decode_step_workspace_size(B, H, Hkv, D, n - 1, window)
            assert size >= prev and step >= prev_step, (B, H, Hkv, D, window, n)
            prev, prev_step = size, step
    # at the edge of a chunk band the plan's own need drops; the reported size does not
    assert g.gqa_attn_decode_workspace_size(8, 64, 8, 128, 4097, 0) == \
        g.gqa_attn_decode_workspace_size(8, 64, 8, 128, 4096, 0)


def test_decode_launch_count_refuses_sizes_no_call_accepts():
    lib = g.load()
    assert lib.gqa_attn_decode_launches(0, 8, 2, 128, 100, 0, -1) == -2     # no rows
    assert lib.gqa_attn_decode_launches(2, 8, 3, 128, 100, 0, -1) == -2     # H % Hkv
    assert lib.gqa_attn_decode_launches(2, 8, 2, 7, 100, 0, -1) == -2       # odd D
    assert lib.gqa_attn_decode_launches(2, 8, 2, 128, 0, 0, -1) == -2       # no positions
    assert lib.gqa_attn_decode_launches(2, 8, 2, 128, 100, -1, -1) == -2    # window
    assert lib.gqa_attn_decode_launches(2, 8, 2, 64, 100, 0, 66) == -2      # rotary dims > D
    assert lib.gqa_attn_decode_launches(2, 8, 2, 64, 100, 0, 5) == -2       # odd rotary dims


def test_wait_timeout_selftest_needs_a_status_word():
    assert g.load().attn_selftest_wait_timeout(None, None) == -1      # ATTN_ERR_NULL


def test_no_cpu_fallback_host_tensors_are_refused():
    """Every compute entry point of the binding takes device tensors only: host tensors are
    refused with an error, never computed some other way."""
    q = torch.zeros(1, 4, 8, 64)
    k = torch.zeros(1, 2, 8, 64)
    st = torch.zeros(1, dtype=torch.int32)
    rp = g.RopeParams.make(theta=1e4, max_positions=64)
    calls = [
        lambda: g.gqa_attn_prefill(q, k, k, q),
        lambda: g.attn_rope_apply(q, st, 0, rp, torch.zeros(64 * 32 * 2)),
        lambda: g.kv_cache_append(k, k, st, 0, rp, torch.zeros(64 * 32 * 2), None, 1e-6,
                                  torch.zeros(1, 2, 8, 64), torch.zeros(1, 2, 8, 64)),
        lambda: g.gqa_attn_decode(q[:, :, :1], k, k, torch.ones(1, dtype=torch.int32), 1,
                                  q[:, :, :1].clone()),
        lambda: g.gqa_attn_decode_static(q[:, :, :1], k, k, torch.ones(1, dtype=torch.int32),
                                         1, q[:, :, :1].clone()),
    ]
    for call in calls:
        with pytest.raises((ValueError, TypeError)):
            call()


def test_missing_library_fails_loudly(tmp_path):
    """Without the built CUDA library the package raises on load; nothing runs in its place."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "gqa_causal_attention_gb300"
    shutil.copytree(os.path.join(ROOT, "gqa_causal_attention_gb300"), pkg,
                    ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so"))
    code = ("import gqa_causal_attention_gb300 as g\n"
            "try:\n"
            "    g.load(build_if_missing=False)\n"
            "except OSError as e:\n"
            "    print('refused', type(e).__name__)\n"
            "else:\n"
            "    print('loaded')\n")
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    out = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.stdout.strip() == "refused OSError", out.stdout + out.stderr


def test_every_declared_function_has_a_binding_of_the_same_name():
    missing = [f for f in declared_functions()
               if f not in g.__all__ or not callable(getattr(g, f, None))]
    assert not missing, missing


def test_from_host_chunk_plan_follows_the_documented_rule():
    """At most 16 chunks: groups of ceil(B / 16) rows when B >= 16; with fewer rows, slices of
    ceil(Hkv / (16 // B)) kv heads of one row; one chunk of everything when a head's rows
    (L * D or capacity * D floats) are not whole 16-byte units. Seen through the workspace
    size, which is the prefill workspace of the largest chunk (rope_dim 32 < D keeps q's
    rotation out of the kernel, so the size grows with the chunk's query heads)."""
    lib = g.load()
    G = 2
    cases = [(64, g.RopeParams.make(theta=1e4, rope_dim=32, max_positions=4096),
              ((64, 64), (33, 64), (3, 66), (64, 5))),
             (6, g.RopeParams.make(theta=1e4, max_positions=4096),      # CUDA-core head dim
              ((64, 64), (33, 64), (64, 33), (2, 2)))]
    shapes = [(D, rp, L, cap, B, Hkv) for D, rp, sizes in cases for L, cap in sizes
              for B in (1, 2, 3, 5, 8, 15, 16, 17, 40) for Hkv in (1, 2, 3, 8)]
    for D, rp, L, cap, B, Hkv in shapes:
        H = G * Hkv
        if (L * D) % 4 or (cap * D) % 4:
            rows, heads = B, Hkv
        elif B >= 16:
            rows, heads = -(-B // 16), Hkv
        else:
            rows, heads = 1, -(-Hkv // (16 // B))
        want = lib.gqa_attn_prefill_rope_workspace_size(rows, heads * G, heads, L, D,
                                                        ctypes.byref(rp))
        got = lib.gqa_attn_prefill_from_host_workspace_size(B, H, Hkv, L, D, cap,
                                                            ctypes.byref(rp))
        assert got == want, (D, B, Hkv, L, cap, got, want)


def test_check_finite_switch_follows_the_environment(tmp_path):
    """ATTN_CHECK_FINITE turns the non-finite check on at first use; unset, empty or "0"
    leaves it off (fresh processes, so the process-wide switch starts unread)."""
    import subprocess
    import sys
    code = ("import gqa_causal_attention_gb300 as g\n"
            "print(g.attn_set_check_finite(-1))\n")
    for val, want in ((None, "0"), ("", "0"), ("0", "0"), ("1", "1"), ("yes", "1")):
        env = {k: v for k, v in os.environ.items() if k != "ATTN_CHECK_FINITE"}
        if val is not None:
            env["ATTN_CHECK_FINITE"] = val
        env["PYTHONPATH"] = ROOT
        out = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, env=env,
                             capture_output=True, text=True, timeout=300)
        assert out.stdout.strip() == want, (val, out.stdout, out.stderr)


@no_device
def test_check_finite_needs_a_status_word():
    """With the check on, a computing call without a status word is refused before any
    launch; with it off the same call goes on to launch (which fails here, with no GPU)."""
    lib = g.load()
    P = ctypes.c_void_p(0x100000)
    prev = g.attn_set_check_finite(1)
    try:
        assert g.attn_set_check_finite(-1) == 1
        assert lib.gqa_attn_decode(P, P, P, P, 10, P, 2, 4, 2, 64, 64, 0, 0.0, 0.0, P, 1 << 20,
                                   None, None) == -1
        assert lib.attn_linear(P, P, None, P, 8, 16, 32, None, None) == -1
        rp = g.RopeParams.make(theta=1e4, max_positions=64)
        assert lib.attn_rope_apply(P, 1, 2, 8, 16, P, 0, ctypes.byref(rp), P, None, 1e-6, None,
                                   None) == -1
        g.attn_set_check_finite(0)
        assert lib.gqa_attn_decode(P, P, P, P, 10, P, 2, 4, 2, 64, 64, 0, 0.0, 0.0, P, 1 << 20,
                                   None, None) == -8
    finally:
        g.attn_set_check_finite(prev)
