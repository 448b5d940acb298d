"""Pins of the fp64 oracle against things other than itself (no GPU).

Each test checks the oracle against a hand-worked fixture, a closed form, an
invariant of the mathematics, an independent brute-force loop written here,
or a library routine (torch's CPU scaled_dot_product_attention in float64).
The cases are chosen so that a dropped term, a wrong sign, a wrong index or
pairing, or a transposed operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _fixture(name):
    rows = {}
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            rows[key] = rest
    return rows


def _eval(expr):
    return eval(expr, {"__builtins__": {}}, {"cos": math.cos, "sin": math.sin,
                                               "sqrt": math.sqrt})


# ----------------------------------------------------------------------------- RoPE


def test_rope_rotate_half_hand_case():
    fx = _fixture("rope_rotate_half_d4.txt")
    x = np.array([float(t) for t in fx["x"].split()]).reshape(1, 1, 1, 4)
    p = int(fx["p"])
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=4, theta=10000.0)
    y = oracle.rotate(x, [p], cfg).reshape(-1)
    want = [_eval(fx[f"y{i}"]) for i in range(4)]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-14)


def test_rope_partial_rotary_hand_case():
    fx = _fixture("rope_partial_d8_r4.txt")
    x = np.array([float(t) for t in fx["x"].split()]).reshape(1, 1, 1, 8)
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=8, rope_dim=4, theta=100.0)
    y = oracle.rotate(x, [int(fx["p"])], cfg).reshape(-1)
    want = [_eval(fx[f"y{i}"]) for i in range(8)]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-14)


def test_rotate_half_is_the_printed_interleaved_rope_up_to_a_dim_permutation():
    """"Core Layers -- Deep Reference", RoPE, prints pairs (2i, 2i+1) turned by p * theta_i;
    the oracle pairs (i, i + R/2). Laying dims out so that interleaved dim 2i is half dim i and
    2i+1 is half dim i + R/2 makes the two the same rotation, and since scores are dot
    products, the same attention for q and k permuted alike."""
    B, H, L, D, theta = 1, 2, 6, 8, 100.0
    R = D
    x_int = RNG.standard_normal((B, H, L, D))
    perm = [2 * i for i in range(R // 2)] + [2 * i + 1 for i in range(R // 2)]
    x_half = x_int[..., perm]                     # half dim j holds interleaved dim perm[j]
    y_half = oracle.rotate(x_half, [3], oracle.Cfg(B=B, H=H, Hkv=H, L=L, D=D, theta=theta))
    want = np.empty_like(x_int)                   # the printed interleaved form
    for l in range(L):
        p = 3 + l
        for i in range(R // 2):
            ang = p * theta ** (-2.0 * i / R)
            a, b = x_int[..., l, 2 * i], x_int[..., l, 2 * i + 1]
            want[..., l, 2 * i] = a * math.cos(ang) - b * math.sin(ang)
            want[..., l, 2 * i + 1] = a * math.sin(ang) + b * math.cos(ang)
    np.testing.assert_allclose(y_half, want[..., perm], rtol=0, atol=1e-13)


def test_rope_two_dims_turn_by_the_absolute_position():
    """At D = 2 the one pair has frequency theta^0 = 1, so the angle is the position itself:
    (1, 0) at position p becomes (cos p, sin p), with p = start[b] + l for every row."""
    B, H, L = 3, 2, 4
    start = [0, 5, 11]
    x = np.zeros((B, H, L, 2))
    x[..., 0] = 1.0
    y = oracle.rotate(x, start, oracle.Cfg(B=B, H=H, Hkv=H, L=L, D=2, theta=123.0))
    for b in range(B):
        for h in range(H):
            for l in range(L):
                p = start[b] + l
                np.testing.assert_allclose(y[b, h, l], [math.cos(p), math.sin(p)], rtol=0,
                                           atol=1e-15)


@pytest.mark.parametrize("D,R", [(16, 16), (64, 32), (128, 64)])
def test_rope_preserves_norm_and_position_zero_is_identity(D, R):
    L = 7
    x = RNG.standard_normal((2, 3, L, D))
    cfg = oracle.Cfg(B=2, H=3, Hkv=3, L=L, D=D, rope_dim=R, theta=5e5,
                     scaling=("llama3", 8.0, 1.0, 4.0, 8192))
    y = oracle.rotate(x, [0, 11], cfg)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1),
                               rtol=1e-13)
    np.testing.assert_allclose(y[0, :, 0], x[0, :, 0], rtol=0, atol=0)


@pytest.mark.parametrize("scaling", [None, ("linear", 4.0), ("llama3", 8.0, 1.0, 4.0, 64)])
def test_rope_relative_position_invariance(scaling):
    """rope(q, p+d) . rope(k, m+d) == rope(q, p) . rope(k, m): the dot product
    depends only on p - m ("Core Layers -- Deep Reference", RoPE)."""
    D = 32
    q = RNG.standard_normal((1, 1, 1, D))
    k = RNG.standard_normal((1, 1, 1, D))
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=D, theta=1e4, scaling=scaling)

    def dot(p, m):
        return float((oracle.rotate(q, [p], cfg) * oracle.rotate(k, [m], cfg)).sum())

    base = dot(9, 4)
    for d in (1, 17, 300, 4095):
        assert abs(dot(9 + d, 4 + d) - base) < 1e-9
    assert abs(dot(9, 5) - base) > 1e-6     # it does depend on p - m


def test_rope_linear_scaling_is_position_division():
    D, f = 16, 4.0
    x = RNG.standard_normal((1, 2, 1, D))
    lin = oracle.Cfg(B=1, H=2, Hkv=2, L=1, D=D, theta=1e4, scaling=("linear", f))
    plain = oracle.Cfg(B=1, H=2, Hkv=2, L=1, D=D, theta=1e4)
    for k in (1, 5, 250):
        np.testing.assert_allclose(oracle.rotate(x, [int(f) * k], lin),
                                   oracle.rotate(x, [k], plain), rtol=0, atol=1e-12)


def test_llama3_scaling_special_cases():
    """The Llama-3 ramp: factor 1 is no scaling; short wavelengths are kept;
    long ones are divided by the factor; the ramp is continuous at both ends."""
    D, theta = 128, 5e5
    plain = oracle.inv_freq(oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=D, theta=theta))
    one = oracle.inv_freq(oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=D, theta=theta,
                                     scaling=("llama3", 1.0, 1.0, 4.0, 8192)))
    np.testing.assert_allclose(one, plain, rtol=1e-15)

    orig, lo, hi, fac = 8192.0, 1.0, 4.0, 8.0
    sc = oracle.inv_freq(oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=D, theta=theta,
                                    scaling=("llama3", fac, lo, hi, orig)))
    wl = 2 * math.pi / plain
    short = wl < orig / hi
    long_ = wl > orig / lo
    assert short.any() and long_.any() and (~short & ~long_).any()
    np.testing.assert_array_equal(sc[short], plain[short])
    np.testing.assert_allclose(sc[long_], plain[long_] / fac, rtol=1e-15)
    mid = ~short & ~long_
    # inside the ramp the frequency lies between the two branches
    assert np.all(sc[mid] <= plain[mid]) and np.all(sc[mid] >= plain[mid] / fac)

    # continuity: move the base so one frequency's wavelength crosses each end
    for edge in (orig / hi, orig / lo):
        i = 1
        # theta such that 2*pi / theta^(-2i/D) == edge
        th_edge = (edge / (2 * math.pi)) ** (D / (2 * i))
        vals = []
        for th in (th_edge * (1 - 1e-9), th_edge * (1 + 1e-9)):
            cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=D, theta=th,
                             scaling=("llama3", fac, lo, hi, orig))
            vals.append(oracle.inv_freq(cfg)[i])
        assert abs(vals[0] - vals[1]) <= 1e-7 * abs(vals[0])


def test_llama3_ramp_interior_hand_worked():
    """Three frequencies inside the Llama-3 ramp of the Llama-3-8B-shaped
    workload, worked by hand from the published Llama 3.1 rule (linear blend
    in frequency), fix the interior arithmetic: a blend in wavelength or in
    log-frequency stays continuous and bounded but misses these values."""
    fx = _fixture("llama3_ramp_interior.txt")
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=128, theta=5e5,
                     scaling=("llama3", 8.0, 1.0, 4.0, 8192))
    inv = oracle.inv_freq(cfg)
    for i in (32, 29, 34):
        want = float(fx[f"f{i}"])
        assert abs(inv[i] - want) <= 1e-12 * want, (i, inv[i], want)


def test_llama3_ramp_ratio_is_affine_in_frequency():
    """Inside the ramp s is affine in 1/wavelength, i.e. in f, so the published
    rule makes f'/f = 1/factor + (1 - 1/factor) * s an affine function of f.
    Checked over every interior pair, for two bases (no fixed values)."""
    for theta in (5e5, 2.5e5):
        cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=128, theta=theta,
                         scaling=("llama3", 8.0, 1.0, 4.0, 8192))
        plain = oracle.inv_freq(oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=128, theta=theta))
        sc = oracle.inv_freq(cfg)
        wl = 2 * math.pi / plain
        mid = (wl >= 8192 / 4.0) & (wl <= 8192 / 1.0)
        assert mid.sum() >= 4
        f, ratio = plain[mid], sc[mid] / plain[mid]
        slope, icpt = np.polyfit(f, ratio, 1)
        np.testing.assert_allclose(ratio, slope * f + icpt, rtol=0, atol=1e-12)
        # the line is fixed too: ratio 1/factor where s = 0 (f = 2*pi*low/orig) and
        # 1 where s = 1 (f = 2*pi*high/orig)
        np.testing.assert_allclose(slope * (2 * math.pi * 1.0 / 8192) + icpt, 1 / 8.0,
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(slope * (2 * math.pi * 4.0 / 8192) + icpt, 1.0,
                                   rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- RMSNorm


def test_rmsnorm_hand_case():
    fx = _fixture("rmsnorm_d2.txt")
    x = np.array([float(t) for t in fx["x"].split()]).reshape(1, 1, 1, 2)
    w = np.array([float(t) for t in fx["w"].split()])
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=2, rope_dim=0, norm_eps=0.0)
    y = oracle.rotate(x, [0], cfg, norm_w=w).reshape(-1)
    np.testing.assert_allclose(y, [_eval(fx["y0"]), _eval(fx["y1"])], rtol=1e-15)


def test_rmsnorm_eps_hand_case():
    """eps sits inside the square root, added to the mean of squares."""
    fx = _fixture("rmsnorm_eps_d2.txt")
    x = np.array([float(t) for t in fx["x"].split()]).reshape(1, 1, 1, 2)
    w = np.array([float(t) for t in fx["w"].split()])
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=2, rope_dim=0, norm_eps=float(fx["eps"]))
    y = oracle.rotate(x, [0], cfg, norm_w=w).reshape(-1)
    np.testing.assert_allclose(y, [_eval(fx["y0"]), _eval(fx["y1"])], rtol=1e-14)


def test_rmsnorm_unit_rms_and_scale_invariance():
    D = 64
    x = RNG.standard_normal((1, 2, 3, D))
    w = 1.0 + 0.1 * RNG.standard_normal(D)
    cfg = oracle.Cfg(B=1, H=2, Hkv=2, L=3, D=D, rope_dim=0, norm_eps=0.0)
    y = oracle.rotate(x, [0], cfg, norm_w=w)
    np.testing.assert_allclose(np.sqrt(np.mean((y / w) ** 2, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rotate(37.5 * x, [0], cfg, norm_w=w), y, rtol=1e-13)


def test_norm_comes_before_rope():
    """q/k RMSNorm runs before RoPE ("mojolearn.transformer", qk_norm)."""
    D = 8
    x = RNG.standard_normal((1, 1, 1, D))
    w = np.arange(1, D + 1, dtype=np.float64)       # not rotation-symmetric
    cfg = oracle.Cfg(B=1, H=1, Hkv=1, L=1, D=D, theta=10.0, norm_eps=0.0)
    y = oracle.rotate(x, [5], cfg, norm_w=w)
    normed = x / np.sqrt(np.mean(x ** 2)) * w
    rot_only = oracle.rotate(normed, [5], cfg)
    np.testing.assert_allclose(y, rot_only, rtol=1e-13)


# ----------------------------------------------------------------------------- attention


def brute_force(q, k, v, start, H, Hkv, window=0, softcap=0.0, scale=None):
    """Independent per-query loop: explicit repeat-KV, a materialised mask."""
    B, _, L, D = q.shape
    G = H // Hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = np.zeros_like(q)
    for b in range(B):
        pos = [start[b] + j for j in range(L)]
        mask = [[(pos[j] <= pos[i]) and (window == 0 or pos[j] > pos[i] - window)
                 for j in range(L)] for i in range(L)]
        for h in range(H):
            kk = [list(k[b, h // G, j]) for j in range(L)]        # repeat-KV
            vv = [list(v[b, h // G, j]) for j in range(L)]
            for i in range(L):
                qi = list(q[b, h, i])
                logits = []
                for j in range(L):
                    s = sum(a * c for a, c in zip(qi, kk[j])) * scale
                    if softcap > 0:
                        s = softcap * math.tanh(s / softcap)
                    logits.append(s if mask[i][j] else -math.inf)
                m = max(logits)
                e = [math.exp(s - m) if s != -math.inf else 0.0 for s in logits]
                z = sum(e)
                for d in range(D):
                    out[b, h, i, d] = sum(e[j] * vv[j][d] for j in range(L)) / z
    return out


@pytest.mark.parametrize("H,Hkv,L,D,window,softcap,start", [
    (4, 2, 9, 4, 0, 0.0, (0,)),
    (4, 2, 9, 6, 3, 0.0, (0,)),
    (6, 2, 8, 4, 0, 2.0, (0, 5)),
    (4, 1, 7, 8, 2, 1.5, (3,)),
    (2, 2, 5, 2, 1, 0.0, (0,)),
])
def test_attention_matches_brute_force(H, Hkv, L, D, window, softcap, start):
    B = len(start)
    q = 2.0 * RNG.standard_normal((B, H, L, D))
    k = 2.0 * RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=window, softcap=softcap)
    got = oracle.attention(q, k, v, list(start), cfg)
    want = brute_force(q, k, v, list(start), H, Hkv, window, softcap)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_attention_matches_brute_force_random_sweep():
    """40 random small problems: head dims, group sizes, lengths (1 included), windows from 1
    to past L, softcap on or off, explicit scales, per-row starts."""
    rng = np.random.default_rng(77)
    for _ in range(40):
        D = int(rng.choice([2, 4, 6, 8, 10]))
        Hkv = int(rng.integers(1, 3))
        H = Hkv * int(rng.integers(1, 5))
        L = int(rng.integers(1, 11))
        B = int(rng.integers(1, 3))
        window = int(rng.choice([0, 0, 1, 2, 3, L, L + 2]))
        softcap = float(rng.choice([0.0, 0.0, 0.7, 4.0]))
        scale = float(rng.choice([0.0, 0.0, 0.2, 1.3]))
        start = [int(x) for x in rng.integers(0, 50, B)]
        q = 2.0 * rng.standard_normal((B, H, L, D))
        k = 2.0 * rng.standard_normal((B, Hkv, L, D))
        v = rng.standard_normal((B, Hkv, L, D))
        cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=window, softcap=softcap,
                         scale=scale)
        got = oracle.attention(q, k, v, start, cfg)
        want = brute_force(q, k, v, start, H, Hkv, window, softcap,
                           scale if scale > 0 else None)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("B,H,Hkv,L,D", [(2, 8, 2, 37, 16), (1, 4, 4, 20, 32), (1, 8, 1, 33, 8)])
def test_attention_matches_torch_sdpa(B, H, Hkv, L, D):
    q = RNG.standard_normal((B, H, L, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D)
    got = oracle.attention(q, k, v, [0] * B, cfg)
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True,
        enable_gqa=True).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_explicit_scale_matches_torch_sdpa():
    B, H, Hkv, L, D = 1, 4, 2, 12, 8
    q, k, v = (RNG.standard_normal((B, n, L, D)) for n in (H, Hkv, Hkv))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, scale=0.3)
    got = oracle.attention(q, k, v, [0], cfg)
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True,
        enable_gqa=True, scale=0.3).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_default_scale_under_partial_rotary_is_full_head_dim():
    """Partial rotary narrows only the rotation: the default score scale stays 1/sqrt(D),
    torch SDPA's default for head dimension D."""
    B, H, Hkv, L, D = 1, 4, 2, 10, 16
    q, k, v = (RNG.standard_normal((B, n, L, D)) for n in (H, Hkv, Hkv))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, rope_dim=4)
    got = oracle.attention(q, k, v, [0], cfg)
    want = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True,
        enable_gqa=True).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_sampled_rows_equal_the_full_prefill_rows():
    """attention_rows computes chosen (b, h, l) rows alone; they equal those rows of the
    whole prefill, with the query's batch row, head and position all taken from the triple."""
    B, H, Hkv, L, D = 3, 6, 3, 13, 8
    q = RNG.standard_normal((B, H, L, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    start = [0, 4, 9]
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=5, softcap=2.0)
    full = oracle.attention(q, k, v, start, cfg)
    rows = [(0, 0, 0), (2, 5, 12), (1, 3, 7), (2, 0, 4), (0, 4, 11), (1, 1, 0)]
    got = oracle.attention_rows(q, k, v, start, cfg, rows)
    for i, (b, h, l) in enumerate(rows):
        np.testing.assert_array_equal(got[i], full[b, h, l])


def test_gqa_equals_mha_over_repeated_kv():
    B, H, Hkv, L, D = 1, 8, 2, 11, 8
    q = RNG.standard_normal((B, H, L, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    gqa = oracle.attention(q, k, v, [0], oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=4,
                                                    softcap=3.0))
    krep, vrep = np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1)
    mha = oracle.attention(q, krep, vrep, [0], oracle.Cfg(B=B, H=H, Hkv=H, L=L, D=D, window=4,
                                                          softcap=3.0))
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=0)


def test_special_cases():
    B, H, Hkv, L, D = 1, 4, 2, 10, 8
    q = 3 * RNG.standard_normal((B, H, L, D))
    k = 3 * RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    causal = oracle.attention(q, k, v, [0], oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D))
    # position 0 sees only itself
    for h in range(H):
        np.testing.assert_array_equal(causal[0, h, 0], v[0, h // 2, 0])
    # window 1: every query sees only itself
    w1 = oracle.attention(q, k, v, [0], oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=1))
    for h in range(H):
        np.testing.assert_array_equal(w1[0, h], v[0, h // 2])
    # a window as long as the sequence is plain causal
    wl = oracle.attention(q, k, v, [0], oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=L))
    np.testing.assert_array_equal(wl, causal)
    # a huge softcap is no softcap
    big = oracle.attention(q, k, v, [0], oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D,
                                                    softcap=1e9))
    np.testing.assert_allclose(big, causal, rtol=1e-9, atol=1e-12)
    # a small softcap does change the result
    small = oracle.attention(q, k, v, [0], oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D,
                                                      softcap=0.5))
    assert np.abs(small - causal).max() > 1e-3


def test_window_width_fixture():
    fx = _fixture("window_mean_l8_w3.txt")
    ps = [int(t) for t in fx["p"].split()]
    want = [float(t) for t in fx["mean"].split()]
    L, D = len(ps), 2
    q = RNG.standard_normal((1, 1, L, D))
    k = np.ones((1, 1, L, D))                     # every key equal
    v = np.zeros((1, 1, L, D))
    v[0, 0, :, 0] = np.arange(L)
    out = oracle.attention(q, k, v, [0], oracle.Cfg(B=1, H=1, Hkv=1, L=L, D=D, window=3))
    np.testing.assert_allclose(out[0, 0, :, 0], want, rtol=0, atol=1e-14)


def test_softcap_two_key_closed_form():
    """Two keys: softmax of c*tanh(s/c) written out by hand."""
    D, c = 2, 1.5
    q = np.array([[[[2.0, 0.0], [1.0, -1.0]]]])
    k = np.array([[[[0.5, 1.0], [3.0, 2.0]]]])
    v = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    out = oracle.attention(q, k, v, [0], oracle.Cfg(B=1, H=1, Hkv=1, L=2, D=D, softcap=c))
    sc = 1 / math.sqrt(2)
    s0 = c * math.tanh((1.0 * 0.5 - 1.0 * 1.0) * sc / c)
    s1 = c * math.tanh((1.0 * 3.0 - 1.0 * 2.0) * sc / c)
    w1 = math.exp(s1) / (math.exp(s0) + math.exp(s1))
    np.testing.assert_allclose(out[0, 0, 1], [1 - w1, w1], rtol=1e-14)


# ----------------------------------------------------------------------------- cache and decode


@pytest.mark.parametrize("window,L", [(0, 12), (5, 12), (4, 3), (12, 12)])
def test_carried_decode_equals_prefill(window, L):
    """Token-by-token decode over a carried cache gives the prefill's rows
    ("mojolearn.transformer": step is forward with L = 1 at cached_tokens)."""
    B, H, Hkv, D = 2, 4, 2, 8
    q = RNG.standard_normal((B, H, L, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    full = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, theta=100.0, window=window, softcap=2.0)
    want, qr, kr = oracle.prefill(q, k, v, [0] * B, full)
    cap = window if window else L
    one = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=1, D=D, theta=100.0, window=window, softcap=2.0)
    kc = vc = wr = None
    for t in range(L):
        kt = oracle.rotate(k[:, :, t:t + 1], [t] * B, one)
        qt = oracle.rotate(q[:, :, t:t + 1], [t] * B, one)
        kc, vc, wr = oracle.append(kt, v[:, :, t:t + 1], [t] * B, one, cap, kc, vc, wr)
        got = oracle.decode(qt, kc, vc, [t + 1] * B, one)
        np.testing.assert_allclose(got[:, :, 0], want[:, :, t], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("window", [0, 6])
def test_decode_rows_each_use_their_own_cache_length(window):
    """Rows of one decode call at different lengths: row b's query sits at cache_len[b] - 1
    and sees only positions up to it, so it equals that position's row of the prefill over
    the whole sequence (causality), whatever the other rows' lengths."""
    B, H, Hkv, L, D = 3, 4, 2, 14, 8
    q = RNG.standard_normal((B, H, L, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, theta=100.0, window=window, softcap=3.0)
    want, qr, kr = oracle.prefill(q, k, v, [0] * B, cfg)
    lens = [5, 14, 9]
    # each row's cache after its first lens[b] tokens, filled here slot by slot (slot = m, or
    # m mod W in a ring of W slots)
    cap = window or L
    kc = np.zeros((B, Hkv, cap, D))
    vc = np.zeros((B, Hkv, cap, D))
    for b, n in enumerate(lens):
        for m in range(n):
            kc[b, :, m % cap] = kr[b, :, m]
            vc[b, :, m % cap] = v[b, :, m]
    qsel = np.stack([qr[b, :, n - 1] for b, n in enumerate(lens)])[:, :, None]
    got = oracle.decode(qsel, kc, vc, lens, oracle.Cfg(**{**cfg.__dict__, "L": 1}))
    for b, n in enumerate(lens):
        np.testing.assert_allclose(got[b, :, 0], want[b, :, n - 1], rtol=1e-12, atol=1e-13)


def test_ring_slots_hold_the_last_window_positions():
    """Under a window the cache is a ring of W slots, slot = position % W
    ("mojolearn.transformer", TransformerState)."""
    B, Hkv, L, D, W = 1, 2, 11, 4, 4
    kr = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    cfg = oracle.Cfg(B=B, H=Hkv, Hkv=Hkv, L=L, D=D, window=W)
    kc, vc, wr = oracle.append(kr, v, [0], cfg, W)
    for s in range(W):
        m = max(p for p in range(L) if p % W == s)
        assert (wr[0, :, s] == m).all()
        np.testing.assert_array_equal(vc[0, :, s], v[0, :, m])
    # in ascending position order, the slots are the last W positions
    order = sorted(range(W), key=lambda s: wr[0, 0, s])
    assert [wr[0, 0, s] for s in order] == list(range(L - W, L))


def test_append_full_cache_positions():
    B, Hkv, L, D = 2, 1, 5, 4
    kr = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    cfg = oracle.Cfg(B=B, H=1, Hkv=Hkv, L=L, D=D)
    kc, vc, wr = oracle.append(kr, v, [0, 3], cfg, 9)
    assert list(wr[0, 0]) == [0, 1, 2, 3, 4, -1, -1, -1, -1]
    assert list(wr[1, 0]) == [-1, -1, -1, 3, 4, 5, 6, 7, -1]
    np.testing.assert_array_equal(kc[1, 0, 3:8], kr[1, 0])


# ----------------------------------------------------------------------------- ragged batch


def _ragged_inputs(B, H, Hkv, L, D):
    return (RNG.standard_normal((B, H, L, D)), RNG.standard_normal((B, Hkv, L, D)),
            RNG.standard_normal((B, Hkv, L, D)))


def test_ragged_full_lengths_is_the_plain_prefill():
    """lengths == L everywhere: no padding, the ordinary prefill."""
    B, H, Hkv, L, D = 3, 4, 2, 9, 8
    q, k, v = _ragged_inputs(B, H, Hkv, L, D)
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=4, softcap=5.0)
    want, _, _ = oracle.prefill(q, k, v, [0] * B, cfg)
    got = oracle.prefill_ragged(q, k, v, [L] * B, cfg)
    np.testing.assert_array_equal(got, want)


def test_ragged_length_one_row_is_its_first_value():
    """A row of length 1 has one real query, which sees only itself: its output is v at
    position 0 (weight 1), and the rest of the row is +0.0."""
    B, H, Hkv, L, D = 2, 4, 2, 6, 8
    q, k, v = _ragged_inputs(B, H, Hkv, L, D)
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D)
    got = oracle.prefill_ragged(q, k, v, [1, L], cfg)
    for h in range(H):
        np.testing.assert_array_equal(got[0, h, 0], v[0, h // 2, 0])
    assert (got[0, :, 1:] == 0).all() and not np.signbit(got[0, :, 1:]).any()


def test_ragged_real_rows_are_the_causal_prefix_and_ignore_padding():
    """Causal attention at position l reads positions <= l only, so a row of length n equals
    the first n positions of the full-length prefill of that row; padding holds NaN here and
    must not reach any output, and padding outputs are exactly +0.0."""
    B, H, Hkv, L, D = 3, 6, 2, 12, 8
    q, k, v = _ragged_inputs(B, H, Hkv, L, D)
    lengths = [5, 12, 1]
    for window, softcap in ((0, 0.0), (3, 0.0), (0, 2.0)):
        cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, window=window, softcap=softcap,
                         rope_dim=4)
        full, _, _ = oracle.prefill(q, k, v, [0] * B, cfg)
        qn, kn, vn = q.copy(), k.copy(), v.copy()
        for b, n in enumerate(lengths):
            qn[b, :, n:] = np.nan
            kn[b, :, n:] = np.nan
            vn[b, :, n:] = np.nan
        got = oracle.prefill_ragged(qn, kn, vn, lengths, cfg)
        for b, n in enumerate(lengths):
            np.testing.assert_allclose(got[b, :, :n], full[b, :, :n], rtol=1e-12, atol=1e-13)
            pad = got[b, :, n:]
            assert (pad == 0).all() and not np.signbit(pad).any()


# ----------------------------------------------------------------------------- decoder block


def _block_weights(dm, H, Hkv, D, IT, qk_norm=False, scale=0.3):
    w = {
        "input_layernorm.weight": 1.0 + 0.1 * RNG.standard_normal(dm),
        "post_attention_layernorm.weight": 1.0 + 0.1 * RNG.standard_normal(dm),
        "q_proj.weight": scale * RNG.standard_normal((H * D, dm)) / np.sqrt(dm),
        "k_proj.weight": scale * RNG.standard_normal((Hkv * D, dm)) / np.sqrt(dm),
        "v_proj.weight": scale * RNG.standard_normal((Hkv * D, dm)) / np.sqrt(dm),
        "o_proj.weight": scale * RNG.standard_normal((dm, H * D)) / np.sqrt(H * D),
        "gate_proj.weight": scale * RNG.standard_normal((IT, dm)) / np.sqrt(dm),
        "up_proj.weight": scale * RNG.standard_normal((IT, dm)) / np.sqrt(dm),
        "down_proj.weight": scale * RNG.standard_normal((dm, IT)) / np.sqrt(IT),
    }
    if qk_norm:
        w["q_norm.weight"] = 1.0 + 0.1 * RNG.standard_normal(D)
        w["k_norm.weight"] = 1.0 + 0.1 * RNG.standard_normal(D)
    return w


def test_block_with_zero_output_projections_is_the_identity():
    B, L, H, Hkv, D, IT = 2, 7, 4, 2, 8, 24
    dm = H * D
    w = _block_weights(dm, H, Hkv, D, IT)
    w["o_proj.weight"][:] = 0.0
    w["down_proj.weight"][:] = 0.0
    x = RNG.standard_normal((B, L, dm))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D)
    np.testing.assert_array_equal(oracle.block_forward(x, w, cfg), x)


def test_block_single_token_closed_form():
    """One token attends to itself only (weight 1), so attention returns its value row: the
    block is x + Wo . repeat_kv(Wv . n1(x)) followed by the MLP. Checks the head layout of
    the projections and the grouping of query heads onto kv heads."""
    B, L, H, Hkv, D, IT = 3, 1, 6, 2, 4, 10
    dm = H * D
    w = _block_weights(dm, H, Hkv, D, IT, qk_norm=True)
    x = RNG.standard_normal((B, L, dm))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D, softcap=3.0, window=5)
    got = oracle.block_forward(x, w, cfg)
    eps = cfg.norm_eps
    for b in range(B):
        xt = x[b, 0]
        n1 = xt / np.sqrt(np.mean(xt * xt) + eps) * w["input_layernorm.weight"]
        vh = (w["v_proj.weight"] @ n1).reshape(Hkv, D)
        attn = np.concatenate([vh[h // (H // Hkv)] for h in range(H)])
        hmid = xt + w["o_proj.weight"] @ attn
        n2 = hmid / np.sqrt(np.mean(hmid * hmid) + eps) * w["post_attention_layernorm.weight"]
        gt, up = w["gate_proj.weight"] @ n2, w["up_proj.weight"] @ n2
        want = hmid + w["down_proj.weight"] @ (gt / (1 + np.exp(-gt)) * up)
        np.testing.assert_allclose(got[b, 0], want, rtol=1e-12, atol=1e-12)


def test_block_is_causal():
    """Changing the tokens from position t on leaves every earlier output unchanged."""
    B, L, H, Hkv, D, IT = 1, 9, 4, 1, 8, 16
    dm = H * D
    w = _block_weights(dm, H, Hkv, D, IT)
    x = RNG.standard_normal((B, L, dm))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D)
    base = oracle.block_forward(x, w, cfg)
    x2 = x.copy()
    x2[:, 5:] = RNG.standard_normal((B, L - 5, dm))
    other = oracle.block_forward(x2, w, cfg)
    np.testing.assert_array_equal(other[:, :5], base[:, :5])
    assert np.abs(other[:, 5:] - base[:, 5:]).max() > 1e-3


def test_block_mlp_is_per_token_and_linear_in_up():
    """With W_v = 0 attention adds nothing, so the block maps each token alone: permuting the
    tokens permutes the outputs, and scaling W_up scales the MLP's contribution (SiLU acts on
    the gate branch only)."""
    B, L, H, Hkv, D, IT = 1, 6, 2, 2, 8, 20
    dm = H * D
    w = _block_weights(dm, H, Hkv, D, IT)
    w["v_proj.weight"][:] = 0.0
    x = RNG.standard_normal((B, L, dm))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D)
    base = oracle.block_forward(x, w, cfg)
    perm = RNG.permutation(L)
    np.testing.assert_allclose(oracle.block_forward(x[:, perm], w, cfg), base[:, perm],
                               rtol=1e-13, atol=1e-13)
    w3 = dict(w, **{"up_proj.weight": 3.0 * w["up_proj.weight"]})
    np.testing.assert_allclose(oracle.block_forward(x, w3, cfg) - x, 3.0 * (base - x),
                               rtol=1e-12, atol=1e-12)


def test_block_offset_norm_with_zero_weight_is_plain_unit_norm():
    B, L, H, Hkv, D, IT = 1, 4, 2, 1, 8, 12
    dm = H * D
    w = _block_weights(dm, H, Hkv, D, IT)
    x = RNG.standard_normal((B, L, dm))
    cfg = oracle.Cfg(B=B, H=H, Hkv=Hkv, L=L, D=D)
    w0 = dict(w, **{"input_layernorm.weight": np.zeros(dm),
                    "post_attention_layernorm.weight": np.zeros(dm)})
    w1 = dict(w, **{"input_layernorm.weight": np.ones(dm),
                    "post_attention_layernorm.weight": np.ones(dm)})
    np.testing.assert_array_equal(oracle.block_forward(x, w0, cfg, norm_offset=True),
                                  oracle.block_forward(x, w1, cfg))
