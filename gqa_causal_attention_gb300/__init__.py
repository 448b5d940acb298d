"""Python binding of libgqa_attn.so: grouped-query causal attention on GB300.

Every function here has the name of the C entry point it wraps (see
``include/gqa_attn.h``) and does argument marshalling only: it checks dtypes,
devices and contiguity, passes tensor pointers (device memory, and the host buffers
of gqa_attn_prefill_from_host) and the current CUDA stream,
and raises ``AttnError`` on a non-zero return code. All arithmetic runs in the
library's CUDA kernels; there is no fallback of any kind. If the library is
missing or cannot load, every call raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _build

__all__ = [
    "AttnError", "RopeParams", "load", "library_path",
    "attn_rope_table_bytes", "attn_rope_table_init", "attn_rope_apply", "kv_cache_append",
    "gqa_attn_prefill", "gqa_attn_prefill_workspace_size", "gqa_attn_decode_workspace_size",
    "gqa_attn_decode", "gqa_attn_prefill_rope", "gqa_attn_prefill_rope_workspace_size",
    "gqa_attn_decode_static", "gqa_attn_vt_pitch", "gqa_attn_v_transpose",
    "gqa_attn_prefill_rope_vt", "gqa_attn_prefill_rope_vt_workspace_size",
    "gqa_attn_prefill_cached", "gqa_attn_prefill_cached_workspace_size",
    "gqa_attn_prefill_ragged", "gqa_attn_prefill_ragged_workspace_size",
    "gqa_attn_prefill_identical", "gqa_attn_decode_identical",
    "gqa_block_forward", "gqa_block_forward_workspace_size", "BLOCK_WEIGHT_NAMES",
    "attn_linear", "attn_set_check_finite", "DEV_NONFINITE",
    "gqa_attn_prefill_step", "gqa_attn_prefill_step_workspace_size",
    "gqa_attn_decode_step", "gqa_attn_decode_step_workspace_size", "gqa_attn_decode_launches",
    "gqa_attn_prefill_from_host", "gqa_attn_prefill_from_host_workspace_size",
    "attn_selftest_wait_timeout",
    "attn_status_string", "attn_version", "attn_last_cuda_error", "rope_table", "ROPE_SCALING",
    "DEV_POSITION", "DEV_CAPACITY", "DEV_LENGTH", "DEV_TIMEOUT",
]

DEV_POSITION, DEV_CAPACITY, DEV_LENGTH, DEV_TIMEOUT, DEV_NONFINITE = 1, 2, 4, 8, 16
ROPE_SCALING = {None: 0, "none": 0, "linear": 1, "llama3": 2}


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = f"{fn}: {attn_status_string(code)} (code {code})"
        if code == -8:
            msg += f": {attn_last_cuda_error()}"
        super().__init__(msg)
        self.code = code


class RopeParams(ctypes.Structure):
    """Mirror of ``attn_rope_params``."""
    _fields_ = [
        ("theta", ctypes.c_double),
        ("rope_dim", ctypes.c_int32),
        ("max_positions", ctypes.c_int32),
        ("scaling_type", ctypes.c_int32),
        ("original_max_positions", ctypes.c_int32),
        ("factor", ctypes.c_double),
        ("low_freq_factor", ctypes.c_double),
        ("high_freq_factor", ctypes.c_double),
    ]

    @classmethod
    def make(cls, theta=10000.0, rope_dim=0, max_positions=8192, scaling=None):
        """scaling: None, ("linear", f) or ("llama3", factor, low, high, original_max)."""
        p = cls(theta=float(theta), rope_dim=int(rope_dim), max_positions=int(max_positions),
                scaling_type=0, original_max_positions=0, factor=1.0, low_freq_factor=1.0,
                high_freq_factor=1.0)
        if scaling is not None:
            p.scaling_type = ROPE_SCALING[scaling[0]]
            if scaling[0] == "linear":
                p.factor = float(scaling[1])
            elif scaling[0] == "llama3":
                p.factor, p.low_freq_factor, p.high_freq_factor = map(float, scaling[1:4])
                p.original_max_positions = int(scaling[4])
        return p


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgqa_attn.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_missing else _build.LIB
        lib = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        rp = ctypes.POINTER(RopeParams)
        f = ctypes.c_float
        sig = {
            "attn_rope_table_bytes": (sz, [rp, i32]),
            "attn_rope_table_init": (i32, [rp, i32, vp, sz, vp]),
            "attn_rope_apply": (i32, [vp, i32, i32, i32, i32, vp, ctypes.c_int32, rp, vp, vp, f,
                                      vp, vp]),
            "kv_cache_append": (i32, [vp, vp, i32, i32, i32, i32, vp, ctypes.c_int32, rp, vp,
                                      vp, f, vp, vp, i32, i32, vp, vp]),
            "gqa_attn_prefill_workspace_size": (sz, [i32, i32, i32, i32]),
            "gqa_attn_prefill": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f, f, vp,
                                       sz, vp, vp]),
            "gqa_attn_prefill_rope_workspace_size": (sz, [i32, i32, i32, i32, i32, rp]),
            "gqa_attn_prefill_rope": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                            ctypes.c_int32, rp, vp, vp, f, i32, f, f, vp, sz, vp,
                                            vp]),
            "gqa_attn_vt_pitch": (i32, [i32]),
            "gqa_attn_v_transpose": (i32, [vp, vp, i32, i32, i32, i32, vp]),
            "gqa_attn_prefill_rope_vt_workspace_size": (sz, [i32, i32, i32, i32, rp]),
            "gqa_attn_prefill_rope_vt": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                               ctypes.c_int32, rp, vp, vp, f, i32, f, f, vp, sz,
                                               vp, vp]),
            "gqa_attn_prefill_from_host_workspace_size": (sz, [i32, i32, i32, i32, i32, i32,
                                                               rp]),
            "gqa_attn_prefill_from_host": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                 i32, i32, vp, ctypes.c_int32, rp, vp, vp, vp, f,
                                                 vp, vp, i32, i32, f, f, vp, sz, vp, vp]),
            "gqa_attn_prefill_cached_workspace_size": (sz, [i32, i32, i32, i32, i32,
                                                            ctypes.c_int32, i32, rp]),
            "gqa_attn_prefill_cached": (i32, [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                              i32, vp, ctypes.c_int32, rp, vp, vp, f, i32, f, f,
                                              vp, sz, vp, vp]),
            "gqa_attn_prefill_ragged_workspace_size": (sz, [i32, i32, i32, i32, i32, rp]),
            "gqa_attn_prefill_ragged": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, rp,
                                              vp, vp, f, i32, f, f, vp, sz, vp, vp]),
            "gqa_attn_prefill_identical": (i32, [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                                 i32, i32, vp, ctypes.c_int32, i32, f, f, vp,
                                                 vp]),
            "gqa_attn_decode_identical": (i32, [vp, vp, vp, vp, ctypes.c_int32, vp, i32, i32,
                                                i32, i32, i32, i32, f, f, vp, vp]),
            "gqa_block_forward_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, rp]),
            "gqa_block_forward": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, f, rp,
                                        vp, i32, f, f, vp, sz, vp, vp]),
            "attn_linear": (i32, [vp, vp, vp, vp, ctypes.c_long, i32, i32, vp, vp]),
            "gqa_attn_prefill_step_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, rp]),
            "gqa_attn_decode_step_workspace_size": (sz, [i32, i32, i32, i32, ctypes.c_int32,
                                                         i32]),
            "gqa_attn_decode_step": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, vp,
                                           ctypes.c_int32, rp, vp, vp, vp, f, vp, vp, i32, i32,
                                           f, f, vp, sz, vp, vp]),
            "gqa_attn_prefill_step": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, rp, vp, vp,
                                            vp, f, vp, vp, i32, i32, f, f, vp, sz, vp, vp]),
            "attn_set_check_finite": (i32, [i32]),
            "gqa_attn_decode_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
            "gqa_attn_decode_launches": (i32, [i32, i32, i32, i32, ctypes.c_int32, i32, i32]),
            "gqa_attn_decode": (i32, [vp, vp, vp, vp, ctypes.c_int32, vp, i32, i32, i32, i32,
                                      i32, i32, f, f, vp, sz, vp, vp]),
            "gqa_attn_decode_static": (i32, [vp, vp, vp, vp, ctypes.c_int32, vp, i32, i32, i32,
                                             i32, i32, i32, f, f, vp, vp]),
            "attn_selftest_wait_timeout": (i32, [vp, vp]),
            "attn_status_string": (ctypes.c_char_p, [i32]),
            "attn_version": (ctypes.c_char_p, []),
            "attn_last_cuda_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _rp(params):
    """RoPE parameters by reference, or NULL."""
    return None if params is None else ctypes.byref(params)


def _ptr(t) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _f32(name: str, t, ndim: int | None = None):
    if t is None:
        return
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


def _i32(name: str, t):
    if t is None:
        return
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")


def _check(fn: str, rc: int):
    if rc != 0:
        raise AttnError(fn, rc)


def attn_status_string(code: int) -> str:
    return load().attn_status_string(int(code)).decode()


def attn_set_check_finite(on: int) -> int:
    """Turn the non-finite input check on (1) or off (0), or query it (< 0); returns the
    previous setting. With it on, every computing call needs a status tensor."""
    return int(load().attn_set_check_finite(int(on)))


def attn_version() -> str:
    return load().attn_version().decode()


def attn_last_cuda_error() -> str:
    """The CUDA error behind the last ATTN_ERR_CUDA on this thread."""
    return load().attn_last_cuda_error().decode()


def attn_selftest_wait_timeout(status, stream=None) -> None:
    """Run the kernels' bounded-wait failure path on purpose: after the wait limit (2 s)
    the launched block ORs ATTN_DEV_TIMEOUT into status (device int32 [1])."""
    _i32("status", status)
    _check("attn_selftest_wait_timeout",
           load().attn_selftest_wait_timeout(_ptr(status), _stream(stream)))


def attn_rope_table_bytes(params: RopeParams, D: int) -> int:
    return int(load().attn_rope_table_bytes(ctypes.byref(params), int(D)))


def attn_rope_table_init(params: RopeParams, D: int, table: torch.Tensor, stream=None) -> None:
    _f32("table", table)
    rc = load().attn_rope_table_init(ctypes.byref(params), int(D), _ptr(table),
                                     table.numel() * 4, _stream(stream))
    _check("attn_rope_table_init", rc)


def rope_table(params: RopeParams, D: int, device="cuda", stream=None) -> torch.Tensor:
    """Allocate (with torch) and fill the cos/sin table for ``params``."""
    n = attn_rope_table_bytes(params, D)
    if n == 0:
        raise AttnError("attn_rope_table_bytes", -7)
    t = torch.empty(n // 4, dtype=torch.float32, device=device)
    attn_rope_table_init(params, D, t, stream)
    return t


def attn_rope_apply(x, start, max_start: int, params: RopeParams, table, norm_w=None,
                    norm_eps: float = 1e-6, status=None, stream=None) -> None:
    """In place on x [B, Hx, L, D]: optional RMSNorm (norm_w), then RoPE at start[b] + l."""
    _f32("x", x, 4); _f32("table", table); _f32("norm_w", norm_w); _i32("start", start)
    _i32("status", status)
    B, Hx, L, D = x.shape
    rc = load().attn_rope_apply(_ptr(x), B, Hx, L, D, _ptr(start), int(max_start),
                                ctypes.byref(params), _ptr(table), _ptr(norm_w),
                                float(norm_eps), _ptr(status), _stream(stream))
    _check("attn_rope_apply", rc)


def kv_cache_append(k, v, start, max_start: int, params, table, k_norm_w, norm_eps, k_cache,
                    v_cache, window: int = 0, status=None, stream=None) -> None:
    """Rotate k [B, Hkv, L, D] in place (if params) and store k, v at their cache slots."""
    _f32("k", k, 4); _f32("v", v, 4); _f32("k_cache", k_cache, 4); _f32("v_cache", v_cache, 4)
    _f32("table", table); _f32("k_norm_w", k_norm_w); _i32("start", start)
    _i32("status", status)
    B, Hkv, L, D = k.shape
    if tuple(v.shape) != (B, Hkv, L, D) or k_cache.shape != v_cache.shape \
            or tuple(k_cache.shape[:2]) != (B, Hkv) or k_cache.shape[3] != D:
        raise ValueError("kv_cache_append: inconsistent shapes")
    rc = load().kv_cache_append(_ptr(k), _ptr(v), B, Hkv, L, D, _ptr(start), int(max_start),
                                _rp(params), _ptr(table),
                                _ptr(k_norm_w), float(norm_eps), _ptr(k_cache), _ptr(v_cache),
                                int(k_cache.shape[2]), int(window), _ptr(status),
                                _stream(stream))
    _check("kv_cache_append", rc)


def gqa_attn_prefill_workspace_size(B: int, Hkv: int, L: int, D: int) -> int:
    return int(load().gqa_attn_prefill_workspace_size(B, Hkv, L, D))


def gqa_attn_prefill(q, k, v, out, window: int = 0, softcap: float = 0.0, scale: float = 0.0,
                     workspace=None, status=None, stream=None) -> None:
    """out [B, H, L, D] = causal (or windowed) GQA attention of rotated q, k and v.

    workspace: device scratch of gqa_attn_prefill_workspace_size bytes; when None a
    torch tensor of that size is taken from the caching allocator for this call."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _f32(n, t, 4)
    _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_prefill: inconsistent shapes")
    if workspace is None:
        n = gqa_attn_prefill_workspace_size(B, Hkv, L, D)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Hkv, L, D,
                                 int(window), float(softcap), float(scale), _ptr(workspace),
                                 wbytes, _ptr(status), _stream(stream))
    _check("gqa_attn_prefill", rc)


def gqa_attn_prefill_rope_workspace_size(B: int, H: int, Hkv: int, L: int, D: int,
                                         params: RopeParams) -> int:
    return int(load().gqa_attn_prefill_rope_workspace_size(B, H, Hkv, L, D,
                                                           _rp(params)))


def gqa_attn_prefill_rope(q, k, v, out, start, max_start: int, params: RopeParams, table,
                          q_norm_w=None, norm_eps: float = 1e-6, window: int = 0,
                          softcap: float = 0.0, scale: float = 0.0, workspace=None, status=None,
                          stream=None) -> None:
    """Prefill attention of raw q (RMSNorm + RoPE applied inside; q is not modified) over
    rotated k and v. workspace: gqa_attn_prefill_rope_workspace_size bytes, or None to take
    one from torch's caching allocator for this call."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _f32(n, t, 4)
    _f32("table", table); _f32("q_norm_w", q_norm_w); _i32("start", start); _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_prefill_rope: inconsistent shapes")
    if workspace is None:
        n = gqa_attn_prefill_rope_workspace_size(B, H, Hkv, L, D, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Hkv, L, D,
                                      _ptr(start), int(max_start), _rp(params),
                                      _ptr(table), _ptr(q_norm_w), float(norm_eps), int(window),
                                      float(softcap), float(scale), _ptr(workspace), wbytes,
                                      _ptr(status), _stream(stream))
    _check("gqa_attn_prefill_rope", rc)


def gqa_attn_prefill_ragged_workspace_size(B: int, H: int, Hkv: int, L: int, D: int,
                                           params: RopeParams = None) -> int:
    return int(load().gqa_attn_prefill_ragged_workspace_size(
        B, H, Hkv, L, D, _rp(params)))


def gqa_attn_prefill_ragged(q, k, v, out, lengths, params: RopeParams = None, table=None,
                            q_norm_w=None, norm_eps: float = 1e-6, window: int = 0,
                            softcap: float = 0.0, scale: float = 0.0, workspace=None,
                            status=None, stream=None) -> None:
    """Prefill of a ragged batch: row b is real at positions [0, lengths[b]) (lengths: int32
    CUDA tensor [B]) and its padding outputs are +0.0. With params, q is raw (RMSNorm + RoPE
    at position l applied inside); without, q is already rotated. workspace:
    gqa_attn_prefill_ragged_workspace_size bytes, or None to take one from torch's caching
    allocator for this call."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _f32(n, t, 4)
    _f32("table", table); _f32("q_norm_w", q_norm_w); _i32("lengths", lengths)
    _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_prefill_ragged: inconsistent shapes")
    if lengths is None or lengths.numel() != B:
        raise ValueError("gqa_attn_prefill_ragged: lengths must hold B values")
    if workspace is None:
        n = gqa_attn_prefill_ragged_workspace_size(B, H, Hkv, L, D, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill_ragged(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Hkv, L, D,
                                        _ptr(lengths),
                                        _rp(params),
                                        _ptr(table), _ptr(q_norm_w), float(norm_eps),
                                        int(window), float(softcap), float(scale),
                                        _ptr(workspace), wbytes, _ptr(status), _stream(stream))
    _check("gqa_attn_prefill_ragged", rc)


def gqa_attn_vt_pitch(L: int) -> int:
    """Row pitch (floats) of the transposed v that the tensor-core prefill reads."""
    return int(load().gqa_attn_vt_pitch(int(L)))


def gqa_attn_v_transpose(v, vt, stream=None) -> None:
    """vt[b, hkv, d, m] = v[b, hkv, m, d]; vt holds B * Hkv * D * gqa_attn_vt_pitch(L) floats."""
    _f32("v", v, 4)
    B, Hkv, L, D = v.shape
    if not vt.is_cuda or vt.dtype != torch.float32 or not vt.is_contiguous() or \
            vt.numel() < B * Hkv * D * gqa_attn_vt_pitch(L):
        raise ValueError("vt must be a contiguous float32 CUDA tensor of "
                         "B * Hkv * D * gqa_attn_vt_pitch(L) elements")
    _check("gqa_attn_v_transpose",
           load().gqa_attn_v_transpose(_ptr(v), _ptr(vt), B, Hkv, L, D, _stream(stream)))


def gqa_attn_prefill_rope_vt_workspace_size(B: int, H: int, L: int, D: int,
                                            params: RopeParams) -> int:
    return int(load().gqa_attn_prefill_rope_vt_workspace_size(B, H, L, D, _rp(params)))


def gqa_attn_prefill_rope_vt(q, k, vt, out, start, max_start: int, params: RopeParams, table,
                             q_norm_w=None, norm_eps: float = 1e-6, window: int = 0,
                             softcap: float = 0.0, scale: float = 0.0, workspace=None,
                             status=None, stream=None) -> None:
    """gqa_attn_prefill_rope with v given transposed (from gqa_attn_v_transpose)."""
    for n, t in (("q", q), ("k", k), ("out", out)):
        _f32(n, t, 4)
    _f32("table", table); _f32("q_norm_w", q_norm_w); _i32("start", start); _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, D) or out.shape != q.shape:
        raise ValueError("gqa_attn_prefill_rope_vt: inconsistent shapes")
    if not vt.is_cuda or vt.dtype != torch.float32 or not vt.is_contiguous() or \
            vt.numel() < B * Hkv * D * gqa_attn_vt_pitch(L):
        raise ValueError("vt must be a contiguous float32 CUDA tensor of "
                         "B * Hkv * D * gqa_attn_vt_pitch(L) elements")
    if workspace is None:
        n = gqa_attn_prefill_rope_vt_workspace_size(B, H, L, D, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill_rope_vt(_ptr(q), _ptr(k), _ptr(vt), _ptr(out), B, H, Hkv, L, D,
                                         _ptr(start), int(max_start), _rp(params),
                                         _ptr(table), _ptr(q_norm_w), float(norm_eps),
                                         int(window), float(softcap), float(scale),
                                         _ptr(workspace), wbytes, _ptr(status), _stream(stream))
    _check("gqa_attn_prefill_rope_vt", rc)


def gqa_attn_prefill_from_host_workspace_size(B: int, H: int, Hkv: int, L: int, D: int,
                                              capacity: int, params: RopeParams) -> int:
    return int(load().gqa_attn_prefill_from_host_workspace_size(B, H, Hkv, L, D, capacity,
                                                                ctypes.byref(params)))


def gqa_attn_prefill_from_host(q_host, k_host, v_host, out_host, q, k, v, out, k_cache, v_cache,
                               start, max_start: int, params: RopeParams, table, q_norm_w=None,
                               k_norm_w=None, norm_eps: float = 1e-6, window: int = 0,
                               softcap: float = 0.0, scale: float = 0.0, workspace=None,
                               status=None, stream=None) -> None:
    """One prefill step from host memory: q_host, k_host, v_host (CPU float32, pinned for
    the copies to overlap the kernels) are copied into the device buffers q, k, v chunk by
    chunk (rows, or kv-head slices of a row), k/v are appended to the caches (k rotated in place), the attention with
    q's RoPE fused writes out, and out is copied back into out_host. Returns once enqueued;
    out_host is complete when `stream` has passed the call."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("k_cache", k_cache),
                 ("v_cache", v_cache)):
        _f32(n, t, 4)
    for n, t, d in (("q_host", q_host, q), ("k_host", k_host, k), ("v_host", v_host, v),
                    ("out_host", out_host, out)):
        if t.dtype != torch.float32 or t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous CPU float32 tensor")
        if t.shape != d.shape:
            raise ValueError(f"{n} must have the shape of its device buffer {tuple(d.shape)}")
    _f32("table", table); _f32("q_norm_w", q_norm_w); _f32("k_norm_w", k_norm_w)
    _i32("start", start); _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape \
            or k_cache.shape != v_cache.shape or tuple(k_cache.shape[:2]) != (B, Hkv) \
            or k_cache.shape[3] != D:
        raise ValueError("gqa_attn_prefill_from_host: inconsistent shapes")
    cap = int(k_cache.shape[2])
    if workspace is None:
        n = gqa_attn_prefill_from_host_workspace_size(B, H, Hkv, L, D, cap, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill_from_host(
        _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host), _ptr(q), _ptr(k), _ptr(v),
        _ptr(out), B, H, Hkv, L, D, _ptr(start), int(max_start), ctypes.byref(params),
        _ptr(table), _ptr(q_norm_w), _ptr(k_norm_w), float(norm_eps), _ptr(k_cache),
        _ptr(v_cache), cap, int(window), float(softcap), float(scale), _ptr(workspace), wbytes,
        _ptr(status), _stream(stream))
    _check("gqa_attn_prefill_from_host", rc)


def gqa_attn_prefill_cached_workspace_size(B: int, H: int, Hkv: int, L: int, D: int,
                                           max_start: int, window: int = 0,
                                           params: RopeParams = None) -> int:
    return int(load().gqa_attn_prefill_cached_workspace_size(
        B, H, Hkv, L, D, int(max_start), int(window),
        _rp(params)))


def gqa_attn_prefill_cached(q, k, v, k_cache, v_cache, out, start, max_start: int,
                            params: RopeParams = None, table=None, q_norm_w=None,
                            norm_eps: float = 1e-6, window: int = 0, softcap: float = 0.0,
                            scale: float = 0.0, workspace=None, status=None, stream=None) -> None:
    """Prefill of a chunk (q [B,H,L,D], rotated k and v [B,Hkv,L,D]) continuing the cache
    (k_cache, v_cache [B,Hkv,capacity,D]) after start[b] positions. params/table: q's RoPE
    applied inside (q raw), or None (q already rotated)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("out", out)):
        _f32(n, t, 4)
    _f32("table", table); _f32("q_norm_w", q_norm_w); _i32("start", start); _i32("status", status)
    B, H, L, D = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape or \
            tuple(k_cache.shape) != (B, Hkv, cap, D) or v_cache.shape != k_cache.shape:
        raise ValueError("gqa_attn_prefill_cached: inconsistent shapes")
    if workspace is None:
        n = gqa_attn_prefill_cached_workspace_size(B, H, Hkv, L, D, max_start, window, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill_cached(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), cap, _ptr(out), B, H, Hkv, L, D,
        _ptr(start), int(max_start), _rp(params),
        _ptr(table), _ptr(q_norm_w), float(norm_eps), int(window), float(softcap), float(scale),
        _ptr(workspace), wbytes, _ptr(status), _stream(stream))
    _check("gqa_attn_prefill_cached", rc)


def gqa_attn_decode_workspace_size(B: int, H: int, Hkv: int, D: int, max_cache_len: int,
                                   window: int = 0) -> int:
    return int(load().gqa_attn_decode_workspace_size(B, H, Hkv, D, int(max_cache_len),
                                                     int(window)))


def gqa_attn_decode(q, k_cache, v_cache, cache_len, max_cache_len: int, out, window: int = 0,
                    softcap: float = 0.0, scale: float = 0.0, workspace=None, status=None,
                    stream=None) -> None:
    """out [B, H, 1, D]: one query per row against the first cache_len[b] positions."""
    _f32("q", q, 4); _f32("out", out, 4); _f32("k_cache", k_cache, 4)
    _f32("v_cache", v_cache, 4); _i32("cache_len", cache_len); _i32("status", status)
    B, H, one, D = q.shape
    Bc, Hkv, cap, Dc = k_cache.shape
    if one != 1 or Bc != B or Dc != D or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_decode: inconsistent shapes")
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len),
                                int(max_cache_len), _ptr(out), B, H, Hkv, D, cap, int(window),
                                float(softcap), float(scale), _ptr(workspace), wbytes,
                                _ptr(status), _stream(stream))
    _check("gqa_attn_decode", rc)


def gqa_attn_prefill_identical(q, k, v, out, start=None, max_start: int = 0, k_cache=None,
                               v_cache=None, window: int = 0, softcap: float = 0.0,
                               scale: float = 0.0, status=None, stream=None) -> None:
    """Prefill attention in the identical numeric mode (bit-for-bit equal to token-by-token
    gqa_attn_decode_identical and to chunked continuations). q, k, v rotated; with k_cache /
    v_cache the positions before start[b] are read from the cache."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("k_cache", k_cache),
                 ("v_cache", v_cache)):
        _f32(n, t, 4)
    _i32("start", start); _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_prefill_identical: inconsistent shapes")
    cap = 0
    if k_cache is not None:
        if v_cache is None or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or \
                k_cache.shape[1] != Hkv or k_cache.shape[3] != D:
            raise ValueError("gqa_attn_prefill_identical: inconsistent cache shapes")
        cap = k_cache.shape[2]
    rc = load().gqa_attn_prefill_identical(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache),
                                           _ptr(v_cache), cap, _ptr(out), B, H, Hkv, L, D,
                                           _ptr(start), int(max_start), int(window),
                                           float(softcap), float(scale), _ptr(status),
                                           _stream(stream))
    _check("gqa_attn_prefill_identical", rc)


def gqa_attn_decode_identical(q, k_cache, v_cache, cache_len, max_cache_len: int, out,
                              window: int = 0, softcap: float = 0.0, scale: float = 0.0,
                              status=None, stream=None) -> None:
    """gqa_attn_decode in the identical numeric mode (no workspace)."""
    _f32("q", q, 4); _f32("out", out, 4); _f32("k_cache", k_cache, 4)
    _f32("v_cache", v_cache, 4); _i32("cache_len", cache_len); _i32("status", status)
    B, H, one, D = q.shape
    Bc, Hkv, cap, Dc = k_cache.shape
    if one != 1 or Bc != B or Dc != D or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_decode_identical: inconsistent shapes")
    rc = load().gqa_attn_decode_identical(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len),
                                          int(max_cache_len), _ptr(out), B, H, Hkv, D, cap,
                                          int(window), float(softcap), float(scale),
                                          _ptr(status), _stream(stream))
    _check("gqa_attn_decode_identical", rc)


# attn_block_weights field -> Hugging Face parameter name
BLOCK_WEIGHT_NAMES = (
    ("input_norm", "input_layernorm.weight"), ("post_norm", "post_attention_layernorm.weight"),
    ("wq", "q_proj.weight"), ("wk", "k_proj.weight"), ("wv", "v_proj.weight"),
    ("wo", "o_proj.weight"), ("w_gate", "gate_proj.weight"), ("w_up", "up_proj.weight"),
    ("w_down", "down_proj.weight"), ("q_norm", "q_norm.weight"), ("k_norm", "k_norm.weight"),
)


class _BlockWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f, _ in BLOCK_WEIGHT_NAMES]


def gqa_attn_prefill_step_workspace_size(B: int, H: int, Hkv: int, L: int, D: int,
                                         window: int, params: RopeParams) -> int:
    return int(load().gqa_attn_prefill_step_workspace_size(B, H, Hkv, L, D, int(window),
                                                           _rp(params)))


def gqa_attn_prefill_step(q, k, v, out, k_cache, v_cache, params: RopeParams, table,
                          q_norm_w=None, k_norm_w=None, norm_eps: float = 1e-6,
                          window: int = 0, softcap: float = 0.0, scale: float = 0.0,
                          workspace=None, status=None, stream=None) -> None:
    """One prefill step from a fresh cache at positions 0 .. L-1: k, v (raw, read only)
    enter the caches rotated / as they are, and out = attention of raw q over them."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("k_cache", k_cache),
                 ("v_cache", v_cache)):
        _f32(n, t, 4)
    _f32("table", table); _f32("q_norm_w", q_norm_w); _f32("k_norm_w", k_norm_w)
    _i32("status", status)
    B, H, L, D = q.shape
    Hkv = k.shape[1]
    cap = k_cache.shape[2]
    if tuple(k.shape) != (B, Hkv, L, D) or v.shape != k.shape or out.shape != q.shape or \
            tuple(k_cache.shape) != (B, Hkv, cap, D) or v_cache.shape != k_cache.shape:
        raise ValueError("gqa_attn_prefill_step: inconsistent shapes")
    if workspace is None:
        n = gqa_attn_prefill_step_workspace_size(B, H, Hkv, L, D, window, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_prefill_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Hkv, L, D,
                                      _rp(params), _ptr(table), _ptr(q_norm_w), _ptr(k_norm_w),
                                      float(norm_eps), _ptr(k_cache), _ptr(v_cache), cap,
                                      int(window), float(softcap), float(scale),
                                      _ptr(workspace), wbytes, _ptr(status), _stream(stream))
    _check("gqa_attn_prefill_step", rc)


def gqa_attn_decode_launches(B: int, H: int, Hkv: int, D: int, max_cache_len: int,
                             window: int = 0, step_rope_dim: int = -1) -> int:
    """Kernels one gqa_attn_decode call (step_rope_dim < 0) or one gqa_attn_decode_step
    call (step_rope_dim = its rope_dim, 0 meaning D; max_cache_len = max_pos + 1) launches."""
    n = int(load().gqa_attn_decode_launches(B, H, Hkv, D, int(max_cache_len), int(window),
                                            int(step_rope_dim)))
    _check("gqa_attn_decode_launches", min(n, 0))
    return n


def gqa_attn_decode_step_workspace_size(B: int, H: int, Hkv: int, D: int, max_pos: int,
                                        window: int = 0) -> int:
    return int(load().gqa_attn_decode_step_workspace_size(B, H, Hkv, D, int(max_pos),
                                                          int(window)))


def gqa_attn_decode_step(q, k, v, out, pos, max_pos: int, k_cache, v_cache, params: RopeParams,
                         table, q_norm_w=None, k_norm_w=None, norm_eps: float = 1e-6,
                         window: int = 0, softcap: float = 0.0, scale: float = 0.0,
                         workspace=None, status=None, stream=None) -> None:
    """One decode step: the new token of row b (raw q [B,H,1,D], k, v [B,Hkv,1,D], read only)
    at position pos[b] enters the caches and out = its attention over the cache."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("k_cache", k_cache),
                 ("v_cache", v_cache)):
        _f32(n, t, 4)
    _f32("table", table); _f32("q_norm_w", q_norm_w); _f32("k_norm_w", k_norm_w)
    _i32("pos", pos); _i32("status", status)
    B, H, one, D = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    if one != 1 or tuple(k.shape) != (B, Hkv, 1, D) or v.shape != k.shape or \
            out.shape != q.shape or tuple(k_cache.shape) != (B, Hkv, cap, D) or \
            v_cache.shape != k_cache.shape or pos.numel() != B:
        raise ValueError("gqa_attn_decode_step: inconsistent shapes")
    if workspace is None:
        n = gqa_attn_decode_step_workspace_size(B, H, Hkv, D, max_pos, window)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_attn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Hkv, D,
                                     _ptr(pos), int(max_pos), _rp(params), _ptr(table),
                                     _ptr(q_norm_w), _ptr(k_norm_w), float(norm_eps),
                                     _ptr(k_cache), _ptr(v_cache), cap, int(window),
                                     float(softcap), float(scale), _ptr(workspace), wbytes,
                                     _ptr(status), _stream(stream))
    _check("gqa_attn_decode_step", rc)


def attn_linear(x, w, y, residual=None, status=None, stream=None) -> None:
    """y = x w^T (+ residual) on the tensor cores: x [T, K], w [N, K] (torch's [out, in]),
    y and residual [T, N]; K and N multiples of 4."""
    _f32("x", x, 2); _f32("w", w, 2); _f32("y", y, 2); _f32("residual", residual, 2)
    _i32("status", status)
    T, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or tuple(y.shape) != (T, N) or (
            residual is not None and tuple(residual.shape) != (T, N)):
        raise ValueError("attn_linear: x [T, K], w [N, K], y and residual [T, N]")
    rc = load().attn_linear(_ptr(x), _ptr(w), _ptr(residual), _ptr(y), T, N, K, _ptr(status),
                            _stream(stream))
    _check("attn_linear", rc)


def gqa_block_forward_workspace_size(B: int, L: int, H: int, Hkv: int, D: int, IT: int,
                                     params: RopeParams) -> int:
    return int(load().gqa_block_forward_workspace_size(B, L, H, Hkv, D, IT,
                                                       ctypes.byref(params)))


def gqa_block_forward(x, out, weights: dict, n_heads: int, n_kv_heads: int,
                      params: RopeParams, table, norm_offset: bool = False,
                      norm_eps: float = 1e-6, window: int = 0, softcap: float = 0.0,
                      scale: float = 0.0, workspace=None, status=None, stream=None) -> None:
    """One decoder block (TransformerBlock.forward, state None): x, out [B, L, d_model];
    weights: float32 CUDA tensors keyed by the Hugging Face names (q_norm / k_norm
    optional)."""
    _f32("x", x, 3); _f32("out", out, 3); _f32("table", table); _i32("status", status)
    B, L, dm = x.shape
    H, Hkv = int(n_heads), int(n_kv_heads)
    if dm % H or out.shape != x.shape:
        raise ValueError("gqa_block_forward: d_model must be n_heads * head_dim")
    D = dm // H
    IT = weights["gate_proj.weight"].shape[0]
    shapes = {"input_layernorm.weight": (dm,), "post_attention_layernorm.weight": (dm,),
              "q_proj.weight": (H * D, dm), "k_proj.weight": (Hkv * D, dm),
              "v_proj.weight": (Hkv * D, dm), "o_proj.weight": (dm, H * D),
              "gate_proj.weight": (IT, dm), "up_proj.weight": (IT, dm),
              "down_proj.weight": (dm, IT), "q_norm.weight": (D,), "k_norm.weight": (D,)}
    w = _BlockWeights()
    for field, name in BLOCK_WEIGHT_NAMES:
        t = weights.get(name)
        if t is None:
            if name in ("q_norm.weight", "k_norm.weight"):
                continue
            raise ValueError(f"gqa_block_forward: missing {name}")
        _f32(name, t)
        if tuple(t.shape) != shapes[name] or not t.is_contiguous():
            raise ValueError(f"gqa_block_forward: {name} must be contiguous {shapes[name]}")
        setattr(w, field, t.data_ptr())
    if workspace is None:
        n = gqa_block_forward_workspace_size(B, L, H, Hkv, D, IT, params)
        workspace = torch.empty(max(4, n // 4), dtype=torch.float32, device=x.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    wbytes = workspace.numel() * workspace.element_size()
    rc = load().gqa_block_forward(_ptr(x), _ptr(out), B, L, H, Hkv, D, IT, ctypes.byref(w),
                                  int(bool(norm_offset)), float(norm_eps), ctypes.byref(params),
                                  _ptr(table), int(window), float(softcap), float(scale),
                                  _ptr(workspace), wbytes, _ptr(status), _stream(stream))
    _check("gqa_block_forward", rc)


def gqa_attn_decode_static(q, k_cache, v_cache, cache_len, max_cache_len: int, out,
                           window: int = 0, softcap: float = 0.0, scale: float = 0.0,
                           status=None, stream=None) -> None:
    """gqa_attn_decode for callers that cannot allocate: the split-KV scratch is a
    fixed 32 MiB array inside the library (shared by all calls; calls that overlap
    on the GPU race on it). The first call on a device sets it up."""
    _f32("q", q, 4); _f32("out", out, 4); _f32("k_cache", k_cache, 4)
    _f32("v_cache", v_cache, 4); _i32("cache_len", cache_len); _i32("status", status)
    B, H, one, D = q.shape
    Bc, Hkv, cap, Dc = k_cache.shape
    if one != 1 or Bc != B or Dc != D or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("gqa_attn_decode_static: inconsistent shapes")
    rc = load().gqa_attn_decode_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len),
                                       int(max_cache_len), _ptr(out), B, H, Hkv, D, cap,
                                       int(window), float(softcap), float(scale), _ptr(status),
                                       _stream(stream))
    _check("gqa_attn_decode_static", rc)
