"""fp64 CPU oracle for grouped-query causal attention.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The
CUDA library and its Python binding never import it, and the two share no
code: only the seeded input generators feed both sides.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one loop per
definition). This module compiles it with gcc, converts numpy/torch inputs to
float64 and calls it through ctypes.

Functions follow these pages (cited by title and section):

* "mojolearn.transformer" -- TransformerBlock (window, rope_theta,
  rope_scaling, rope_dim, qk_norm, attn_softcap, norm_eps), step,
  TransformerState (cache slots, window ring).
* "Core Layers -- Deep Reference" -- RMSNorm, RoPE, MHA and GQA grouping,
  sliding window attention, static KV cache.
* "dew.nn.backbones.causal_transformer" -- LayerKind.window,
  partial_rotary_factor, attention_scale.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` (OpenMP if gcc has it)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("L", ctypes.c_int), ("D", ctypes.c_int),
        ("rope_dim", ctypes.c_int),
        ("theta", ctypes.c_double),
        ("scaling_type", ctypes.c_int),
        ("factor", ctypes.c_double),
        ("low_freq_factor", ctypes.c_double),
        ("high_freq_factor", ctypes.c_double),
        ("original_max_positions", ctypes.c_double),
        ("norm_eps", ctypes.c_double),
        ("window", ctypes.c_int),
        ("softcap", ctypes.c_double),
        ("scale", ctypes.c_double),
    ]


@dataclass
class Cfg:
    """Problem description, in the vocabulary of the mojolearn TransformerBlock.

    rope_dim = 0 turns rotation off; scaling is None, ("linear", f) or
    ("llama3", factor, low_freq_factor, high_freq_factor, original_max).
    window = 0 is full causal; softcap <= 0 is off; scale <= 0 is 1/sqrt(D).
    """
    B: int
    H: int
    Hkv: int
    L: int
    D: int
    rope_dim: int = -1            # -1: the full head dimension
    theta: float = 10000.0
    scaling: tuple | None = None
    norm_eps: float = 1e-6
    window: int = 0
    softcap: float = 0.0
    scale: float = 0.0

    def c(self) -> _Cfg:
        st, f, lo, hi, orig = 0, 1.0, 1.0, 1.0, 1.0
        if self.scaling is not None:
            if self.scaling[0] == "linear":
                st, f = 1, float(self.scaling[1])
            elif self.scaling[0] == "llama3":
                st = 2
                f, lo, hi, orig = (float(x) for x in self.scaling[1:5])
            else:
                raise ValueError(f"unknown rope scaling {self.scaling[0]!r}")
        R = self.D if self.rope_dim < 0 else self.rope_dim
        return _Cfg(self.B, self.H, self.Hkv, self.L, self.D, R, float(self.theta), st, f, lo,
                    hi, orig, float(self.norm_eps), int(self.window), float(self.softcap),
                    float(self.scale))


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            d, i, l = P(ctypes.c_double), P(ctypes.c_int), P(ctypes.c_long)
            c = P(_Cfg)
            _lib.orc_inv_freq.argtypes = [c, d]
            _lib.orc_rotate_rows.argtypes = [c, d, ctypes.c_int, i, d, d]
            _lib.orc_prefill.argtypes = [c, d, d, d, i, d]
            _lib.orc_prefill_rows.argtypes = [c, d, d, d, i, ctypes.c_int, i, d]
            _lib.orc_append.argtypes = [c, d, d, i, ctypes.c_int, d, d, l]
            _lib.orc_decode.argtypes = [c, d, d, d, i, ctypes.c_int, d]
            _lib.orc_num_threads.restype = ctypes.c_int
    return _lib


def num_threads() -> int:
    return int(lib().orc_num_threads())


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def inv_freq(cfg: Cfg) -> np.ndarray:
    """Rotary frequencies theta_i (with scaling), length R/2."""
    cc = cfg.c()
    out = np.zeros(max(cc.rope_dim // 2, 1), dtype=np.float64)
    lib().orc_inv_freq(ctypes.byref(cc), _dp(out))
    return out[: cc.rope_dim // 2]


def rotate(x, start, cfg: Cfg, norm_w=None) -> np.ndarray:
    """RMSNorm (if norm_w) then RoPE of x [B, NH, L, D] at positions start[b] + l."""
    x = _f64(x)
    B, NH, L, D = x.shape
    assert B == cfg.B and L == cfg.L and D == cfg.D
    st = _i32(start)
    y = np.empty_like(x)
    w = None if norm_w is None else _f64(norm_w)
    lib().orc_rotate_rows(ctypes.byref(cfg.c()), _dp(x), NH, _ip(st),
                          None if w is None else _dp(w), _dp(y))
    return y


def attention(qr, kr, v, start, cfg: Cfg) -> np.ndarray:
    """Prefill attention over the chunk's own keys: out [B, H, L, D] (float64)."""
    qr, kr, v, st = _f64(qr), _f64(kr), _f64(v), _i32(start)
    out = np.empty_like(qr)
    lib().orc_prefill(ctypes.byref(cfg.c()), _dp(qr), _dp(kr), _dp(v), _ip(st), _dp(out))
    return out


def attention_rows(qr, kr, v, start, cfg: Cfg, rows) -> np.ndarray:
    """The prefill outputs of selected rows [(b, h, l), ...] -> [n, D]."""
    qr, kr, v, st = _f64(qr), _f64(kr), _f64(v), _i32(start)
    r = _i32(np.asarray(rows).reshape(-1, 3))
    out = np.empty((r.shape[0], cfg.D), dtype=np.float64)
    lib().orc_prefill_rows(ctypes.byref(cfg.c()), _dp(qr), _dp(kr), _dp(v), _ip(st),
                           r.shape[0], _ip(r), _dp(out))
    return out


def prefill(q, k, v, start, cfg: Cfg, q_norm_w=None, k_norm_w=None):
    """The whole prefill path: (out, rotated q, rotated k), all float64."""
    H, Hkv = cfg.H, cfg.Hkv
    qr = rotate(q, start, cfg, q_norm_w)
    kr = rotate(k, start, cfg, k_norm_w)
    assert qr.shape[1] == H and kr.shape[1] == Hkv
    return attention(qr, kr, v, start, cfg), qr, kr


def prefill_ragged(q, k, v, lengths, cfg: Cfg, q_norm_w=None, k_norm_w=None) -> np.ndarray:
    """A ragged batch ("mojolearn.transformer", TransformerBlock.forward, lengths): row b is
    real at positions [0, lengths[b]) and padding after. Each real output is row b run alone
    at its own length (a fresh sequence, start 0), and every padding output is exactly +0.0.
    Raw q, k, v (normalised and rotated here) -> out [B, H, L, D] float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    out = np.zeros(q.shape, dtype=np.float64)
    for b, n in enumerate(int(x) for x in lengths):
        assert 1 <= n <= cfg.L
        alone = Cfg(**{**cfg.__dict__, "B": 1, "L": n})
        o, _, _ = prefill(q[b:b + 1, :, :n], k[b:b + 1, :, :n], v[b:b + 1, :, :n], [0], alone,
                          q_norm_w, k_norm_w)
        out[b, :, :n] = o[0]
    return out


def rmsnorm(x, w, eps: float, offset: bool = False) -> np.ndarray:
    """RMSNorm over the last axis ("Core Layers -- Deep Reference", RMSNorm): x / sqrt(mean x^2
    + eps) times w, or times 1 + w ("mojolearn.transformer", norm='rmsnorm_offset', Gemma)."""
    x = _f64(x)
    scale = (1.0 + _f64(w)) if offset else _f64(w)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * scale


def block_forward(x, weights: dict, cfg: Cfg, norm_offset: bool = False) -> np.ndarray:
    """One decoder block ("mojolearn.transformer", TransformerBlock.forward with state None,
    computing Hugging Face's LlamaDecoderLayer.forward): input RMSNorm, q/k/v projections,
    (q/k norm,) RoPE and causal grouped-query attention over positions 0 .. L-1, output
    projection, residual; post-attention RMSNorm, SiLU-gated MLP, residual.

    x [B, L, d_model]; weights keyed by the Hugging Face names in torch's [out, in] layout
    (q_norm.weight / k_norm.weight optional). Matrix products are numpy's; returns float64.
    """
    x = _f64(x)
    B, L, dm = x.shape
    H, Hkv, D = cfg.H, cfg.Hkv, cfg.D
    W = {n: _f64(t) for n, t in weights.items()}
    eps = cfg.norm_eps
    n1 = rmsnorm(x, W["input_layernorm.weight"], eps, norm_offset)

    def heads(y, nh):                      # [B, L, nh * D] -> [B, nh, L, D]
        return y.reshape(B, L, nh, D).transpose(0, 2, 1, 3)

    q = heads(n1 @ W["q_proj.weight"].T, H)
    k = heads(n1 @ W["k_proj.weight"].T, Hkv)
    v = heads(n1 @ W["v_proj.weight"].T, Hkv)
    attn, _, _ = prefill(q, k, v, [0] * B, Cfg(**{**cfg.__dict__, "B": B, "L": L}),
                         W.get("q_norm.weight"), W.get("k_norm.weight"))
    h = x + attn.transpose(0, 2, 1, 3).reshape(B, L, H * D) @ W["o_proj.weight"].T
    n2 = rmsnorm(h, W["post_attention_layernorm.weight"], eps, norm_offset)
    gate = n2 @ W["gate_proj.weight"].T
    up = n2 @ W["up_proj.weight"].T
    act = gate / (1.0 + np.exp(-gate)) * up          # SiLU(gate) * up
    return h + act @ W["down_proj.weight"].T


def append(kr, v, start, cfg: Cfg, capacity: int, k_cache=None, v_cache=None, written=None):
    """Store rotated k and raw v at their cache slots. Returns (k_cache, v_cache, written).

    Caches are float64 [B, Hkv, capacity, D]; written [B, Hkv, capacity] holds the
    position stored in each slot, -1 where nothing was written.
    """
    kr, v, st = _f64(kr), _f64(v), _i32(start)
    B, Hkv, D = cfg.B, cfg.Hkv, cfg.D
    kc = np.zeros((B, Hkv, capacity, D)) if k_cache is None else _f64(k_cache).copy()
    vc = np.zeros((B, Hkv, capacity, D)) if v_cache is None else _f64(v_cache).copy()
    wr = (np.full((B, Hkv, capacity), -1, dtype=np.int64) if written is None
          else np.ascontiguousarray(np.asarray(written, dtype=np.int64)).copy())
    lib().orc_append(ctypes.byref(cfg.c()), _dp(kr), _dp(v), _ip(st), int(capacity),
                     _dp(kc), _dp(vc), wr.ctypes.data_as(ctypes.POINTER(ctypes.c_long)))
    return kc, vc, wr


def decode(qr, k_cache, v_cache, cache_len, cfg: Cfg) -> np.ndarray:
    """Single-token attention of rotated qr [B, H, D] (or [B, H, 1, D]) over the cache."""
    qr, kc, vc, cl = _f64(qr), _f64(k_cache), _f64(v_cache), _i32(cache_len)
    shape = qr.shape
    capacity = kc.shape[2]
    out = np.empty((cfg.B, cfg.H, cfg.D), dtype=np.float64)
    lib().orc_decode(ctypes.byref(cfg.c()), _dp(qr.reshape(cfg.B, cfg.H, cfg.D)), _dp(kc),
                     _dp(vc), _ip(cl), int(capacity), _dp(out))
    return out.reshape(shape)
