"""B300-native attention for Wan-style video diffusion transformers.

Thin ctypes binding over ``libwan_attn.so`` (the C ABI in ``include/wan_attn.h``).
The functions named like the C entry points only marshal arguments: tensors
become device pointers, streams become ``cudaStream_t`` handles, and the C
status code is returned (or raised, in the ``*_checked`` helpers). Every step
of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and importing a function whose library is missing raises.

The convenience wrappers at the bottom (``attention_forward`` and friends)
allocate outputs and workspace with PyTorch and call the same entry points.
"""
from __future__ import annotations

import ctypes
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
RELEASE_LIB_PATH = os.path.join(HERE, "libwan_attn.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libwan_attn_debug.so")  # built with -DWAN_DEBUG
# Which build to load: WAN_ATTN_LIB may name another build of the same C ABI
# (the debug library, for instance); by default the release library.
LIB_PATH = os.environ.get("WAN_ATTN_LIB") or RELEASE_LIB_PATH

WAN_OK = 0
WAN_ERR_INVALID = 1
WAN_ERR_UNSUPPORTED = 2
WAN_ERR_CUDA = 3
WAN_ERR_TIMEOUT = 4
WAN_ERR_DEVICE_CHECK = 5
WAN_OP_FWD = 0
WAN_OP_BWD = 1
WAN_OP_FWD_FP8 = 2
HEAD_DIM = 128
DEFAULT_THETA = 10000.0

EXPORTED = (
    "wan_status_str", "wan_version", "wan_rope3d_tables_size", "wan_rope3d_tables",
    "wan_attn_workspace_size", "wan_attn_fwd", "wan_xattn_fwd", "wan_attn_bwd",
    "wan_get_device_status", "wan_profile_set_events", "wan_debug_inject_stall", "wan_attn_fwd_noalloc",
    "wan_attn_fwd_ring_step", "wan_xattn_fwd_dual", "wan_attn_fwd_fp8", "wan_vae_causal_conv3d",
    "wan_profile_set_pass_events", "wan_vae_time_downsample", "wan_debug_build", "wan_debug_inject_check",
    "wan_debug_check_line",
)
WAN_PASS_MAIN = 0
WAN_PASS_ROPE = 1
WAN_PASS_ROWS = 2
WAN_PASS_POST = 3
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
NOALLOC_MAX_ROW_HEADS = NOALLOC_SCRATCH_BYTES // 256


class WanError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}" if where else status_str(status))


class wan_grid_t(ctypes.Structure):
    _fields_ = [("F", ctypes.c_int), ("Hp", ctypes.c_int), ("Wp", ctypes.c_int)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m long_sequence_attention_02_b300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.wan_status_str.argtypes, lib.wan_status_str.restype = [i32], ctypes.c_char_p
    lib.wan_version.argtypes, lib.wan_version.restype = [], i32
    lib.wan_rope3d_tables_size.argtypes, lib.wan_rope3d_tables_size.restype = [wan_grid_t, i32], sz
    lib.wan_rope3d_tables.argtypes = [wan_grid_t, i32, ctypes.c_double, vp, vp]
    lib.wan_attn_workspace_size.argtypes = [i32, i32, wan_grid_t, i32, i32]
    lib.wan_attn_workspace_size.restype = sz
    lib.wan_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, wan_grid_t, i32, i32, vp, f32, vp, sz, vp]
    lib.wan_xattn_fwd.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, wan_grid_t, i32, i32, f32, vp]
    lib.wan_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, wan_grid_t, i32, i32, vp, f32, vp, sz,
                                 vp]
    lib.wan_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, wan_grid_t, i32, i32, vp, f32, vp]
    lib.wan_attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i32, wan_grid_t, i32, i32, vp, f32, vp, sz, vp]
    lib.wan_attn_fwd_ring_step.argtypes = [vp, vp, vp, vp, vp, i32, wan_grid_t, i32, i32, vp, f32, i32, i32, i32,
                                           i32, i32, vp, sz, vp]
    lib.wan_xattn_fwd_dual.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, vp, i32, wan_grid_t, i32, i32,
                                       f32, vp]
    lib.wan_vae_causal_conv3d.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.wan_vae_time_downsample.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.wan_get_device_status.argtypes = [vp]
    lib.wan_debug_inject_stall.argtypes = [i32, i32]
    lib.wan_debug_build.argtypes = []
    lib.wan_debug_inject_check.argtypes = [i32]
    lib.wan_debug_check_line.argtypes = []
    lib.wan_profile_set_events.argtypes = [vp, vp]
    lib.wan_profile_set_pass_events.argtypes = [i32, vp, vp]
    for name in ("wan_rope3d_tables", "wan_attn_fwd", "wan_xattn_fwd", "wan_attn_bwd",
                 "wan_get_device_status", "wan_profile_set_events", "wan_debug_inject_stall",
                 "wan_attn_fwd_noalloc", "wan_attn_fwd_ring_step", "wan_xattn_fwd_dual", "wan_attn_fwd_fp8",
                 "wan_vae_causal_conv3d", "wan_profile_set_pass_events", "wan_vae_time_downsample",
                 "wan_debug_build", "wan_debug_inject_check", "wan_debug_check_line"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# Argument marshalling


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _grid(g) -> wan_grid_t:
    if isinstance(g, wan_grid_t):
        return g
    F, Hp, Wp = g
    return wan_grid_t(int(F), int(Hp), int(Wp))


# ---------------------------------------------------------------------------
# The C entry points, same names and argument order


def status_str(status: int) -> str:
    return load_library().wan_status_str(int(status)).decode()


wan_status_str = status_str


def wan_version() -> int:
    return load_library().wan_version()


def wan_rope3d_tables_size(grid, head_dim: int = HEAD_DIM) -> int:
    return load_library().wan_rope3d_tables_size(_grid(grid), head_dim)


def wan_rope3d_tables(grid, head_dim, theta, tables_dev, stream=None) -> int:
    return load_library().wan_rope3d_tables(_grid(grid), head_dim, float(theta), _ptr(tables_dev), _stream(stream))


def wan_attn_workspace_size(op, B, grid, H, head_dim=HEAD_DIM) -> int:
    return load_library().wan_attn_workspace_size(op, B, _grid(grid), H, head_dim)


def wan_attn_fwd(q, k, v, o, lse, B, grid, H, head_dim, tables, scale, workspace, ws_bytes, stream=None) -> int:
    return load_library().wan_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, _grid(grid), H, head_dim,
                                       _ptr(tables), float(scale), _ptr(workspace), int(ws_bytes), _stream(stream))


def wan_xattn_fwd(q, k, v, kv_lens, Lk, o, lse, B, grid, H, head_dim, scale, stream=None) -> int:
    return load_library().wan_xattn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_lens), Lk, _ptr(o), _ptr(lse), B,
                                        _grid(grid), H, head_dim, float(scale), _stream(stream))


def wan_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, grid, H, head_dim, tables, scale, workspace, ws_bytes,
                 stream=None) -> int:
    return load_library().wan_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                       _ptr(dk), _ptr(dv), B, _grid(grid), H, head_dim, _ptr(tables), float(scale),
                                       _ptr(workspace), int(ws_bytes), _stream(stream))


def wan_attn_fwd_noalloc(q, k, v, o, lse, B, grid, H, head_dim, tables, scale, stream=None) -> int:
    """wan_attn_fwd without a workspace: the library's fixed device scratch
    holds the rotated keys (B * L * H <= NOALLOC_MAX_ROW_HEADS)."""
    return load_library().wan_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, _grid(grid), H,
                                                head_dim, _ptr(tables), float(scale), _stream(stream))


def wan_attn_fwd_fp8(q, k, v, o, lse, B, grid, H, head_dim, tables, scale, workspace, ws_bytes, stream=None) -> int:
    return load_library().wan_attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, _grid(grid), H,
                                            head_dim, _ptr(tables), float(scale), _ptr(workspace), int(ws_bytes),
                                            _stream(stream))


def wan_vae_causal_conv3d(x, cache, weight, bias, y, cache_out, B, T, H, W, c_in, c_out, stream=None) -> int:
    return load_library().wan_vae_causal_conv3d(_ptr(x), _ptr(cache), _ptr(weight), _ptr(bias), _ptr(y),
                                                 _ptr(cache_out), B, T, H, W, c_in, c_out, _stream(stream))


def wan_vae_time_downsample(x, cache, weight, bias, y, cache_out, B, T, H, W, c_in, c_out, stream=None) -> int:
    return load_library().wan_vae_time_downsample(_ptr(x), _ptr(cache), _ptr(weight), _ptr(bias), _ptr(y),
                                                   _ptr(cache_out), B, T, H, W, c_in, c_out, _stream(stream))


def wan_attn_fwd_ring_step(q, k, v, o, lse, B, grid, H, head_dim, tables, scale, q_start, q_len, kv_start, kv_len,
                           accumulate, workspace, ws_bytes, stream=None) -> int:
    return load_library().wan_attn_fwd_ring_step(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, _grid(grid), H,
                                                  head_dim, _ptr(tables), float(scale), int(q_start), int(q_len),
                                                  int(kv_start), int(kv_len), int(accumulate), _ptr(workspace),
                                                  int(ws_bytes), _stream(stream))


def wan_xattn_fwd_dual(q, k_txt, v_txt, lens_txt, Lk_txt, k_img, v_img, lens_img, Lk_img, o, lse, B, grid, H,
                       head_dim, scale, stream=None) -> int:
    return load_library().wan_xattn_fwd_dual(_ptr(q), _ptr(k_txt), _ptr(v_txt), _ptr(lens_txt), int(Lk_txt),
                                              _ptr(k_img), _ptr(v_img), _ptr(lens_img), int(Lk_img), _ptr(o),
                                              _ptr(lse), B, _grid(grid), H, head_dim, float(scale), _stream(stream))


def wan_get_device_status(stream=None) -> int:
    return load_library().wan_get_device_status(_stream(stream))


def wan_profile_set_events(start, stop) -> int:
    """start/stop: torch.cuda.Event (created with enable_timing and recorded
    at least once, so that its handle exists) or None."""
    handles = [None if e is None else e.cuda_event for e in (start, stop)]
    if any(h == 0 for h in handles):
        raise ValueError("wan_profile_set_events: event has no CUDA handle yet (record it once first)")
    return load_library().wan_profile_set_events(*handles)


def wan_profile_set_pass_events(pass_, start, stop) -> int:
    """Events around one pass (WAN_PASS_*) of the next entry-point call; same
    event rules as wan_profile_set_events."""
    handles = [None if e is None else e.cuda_event for e in (start, stop)]
    if any(h == 0 for h in handles):
        raise ValueError("wan_profile_set_pass_events: event has no CUDA handle yet (record it once first)")
    return load_library().wan_profile_set_pass_events(int(pass_), *handles)


def wan_debug_inject_stall(count: int, timeout_ms: int) -> int:
    return load_library().wan_debug_inject_stall(count, timeout_ms)


def wan_debug_build() -> int:
    return load_library().wan_debug_build()


def wan_debug_inject_check(count: int) -> int:
    return load_library().wan_debug_inject_check(count)


def wan_debug_check_line() -> int:
    return load_library().wan_debug_check_line()


def check(status: int, where: str = "") -> None:
    if status != WAN_OK:
        raise WanError(status, where)


# ---------------------------------------------------------------------------
# Convenience wrappers (PyTorch allocates; the library computes)


def rope_tables(grid, theta=DEFAULT_THETA, device="cuda", stream=None):
    import torch

    n = wan_rope3d_tables_size(grid)
    if n == 0:
        raise WanError(WAN_ERR_INVALID, "wan_rope3d_tables_size")
    t = torch.empty(n // 4, dtype=torch.float32, device=device)
    check(wan_rope3d_tables(grid, HEAD_DIM, theta, t, stream), "wan_rope3d_tables")
    return t


def attention_forward(q, k, v, grid, tables=None, scale=None, theta=DEFAULT_THETA, lse=True, stream=None):
    """Self-attention with 3D RoPE. q, k, v: bf16 [B, L, H, 128] on the GPU."""
    import torch

    B, L, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if tables is None:
        tables = rope_tables(grid, theta, q.device, stream)
    o = torch.empty_like(q)
    lse_t = torch.empty(B, H, L, dtype=torch.float32, device=q.device) if lse else None
    ws_bytes = wan_attn_workspace_size(WAN_OP_FWD, B, grid, H, d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    check(wan_attn_fwd(q, k, v, o, lse_t, B, grid, H, d, tables, scale, ws, ws_bytes, stream), "wan_attn_fwd")
    return o, lse_t


def cross_attention_forward(q, k, v, kv_lens, grid, scale=None, lse=True, stream=None):
    """Cross-attention; q [B, Lq, H, 128], k, v [B, Lk, H, 128], kv_lens int32 [B] or None."""
    import torch

    B, Lq, H, d = q.shape
    Lk = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse_t = torch.empty(B, H, Lq, dtype=torch.float32, device=q.device) if lse else None
    check(wan_xattn_fwd(q, k, v, kv_lens, Lk, o, lse_t, B, grid, H, d, scale, stream), "wan_xattn_fwd")
    return o, lse_t


def attention_forward_fp8(q, k, v, grid, tables=None, scale=None, theta=DEFAULT_THETA, lse=True, stream=None):
    """FP8 (e4m3) self-attention with 3D RoPE. q, k, v: bf16 [B, L, H, 128] on the GPU."""
    import torch

    B, L, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if tables is None:
        tables = rope_tables(grid, theta, q.device, stream)
    o = torch.empty_like(q)
    lse_t = torch.empty(B, H, L, dtype=torch.float32, device=q.device) if lse else None
    ws_bytes = wan_attn_workspace_size(WAN_OP_FWD_FP8, B, grid, H, d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    check(wan_attn_fwd_fp8(q, k, v, o, lse_t, B, grid, H, d, tables, scale, ws, ws_bytes, stream), "wan_attn_fwd_fp8")
    return o, lse_t


def attention_backward(q, k, v, o, lse, dout, grid, tables=None, scale=None, theta=DEFAULT_THETA, stream=None):
    """Gradients of self-attention with 3D RoPE w.r.t. the pre-RoPE q, k and v."""
    import torch

    B, L, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if tables is None:
        tables = rope_tables(grid, theta, q.device, stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = wan_attn_workspace_size(WAN_OP_BWD, B, grid, H, d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    check(wan_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, grid, H, d, tables, scale, ws, ws_bytes, stream),
          "wan_attn_bwd")
    return dq, dk, dv


def causal_conv3d(x, weight, bias=None, cache=None, stream=None):
    """One causal 3x3x3 Conv3d layer of the Wan-VAE on one chunk of frames.

    x: bf16 [B, T, H, W, C_in] on the GPU; weight: bf16 [C_out, 3, 3, 3, C_in];
    bias: fp32 [C_out] or None; cache: bf16 [B, 2, H, W, C_in] from the previous
    chunk, or None for a first chunk. Returns (y [B, T, H, W, C_out], the cache
    for the next chunk).
    """
    import torch

    B, T, H, W, c_in = x.shape
    c_out = weight.shape[0]
    y = torch.empty(B, T, H, W, c_out, dtype=torch.bfloat16, device=x.device)
    new_cache = torch.empty(B, 2, H, W, c_in, dtype=torch.bfloat16, device=x.device)
    check(wan_vae_causal_conv3d(x, cache, weight, bias, y, new_cache, B, T, H, W, c_in, c_out, stream),
          "wan_vae_causal_conv3d")
    return y, new_cache


def time_downsample(x, weight, bias=None, cache=None, stream=None):
    """One time-downsampling layer (3 x 1 x 1 taps, stride 2 in time) of the
    Wan-VAE encoder on one chunk of frames.

    x: bf16 [B, T, H, W, C_in] on the GPU; weight: bf16 [C_out, 3, C_in];
    bias: fp32 [C_out] or None; cache: bf16 [B, 1, H, W, C_in] from the
    previous chunk, or None for a first chunk (one frame, passed through).
    Returns (y [B, T/2, H, W, C_out] (x itself for a first chunk), the cache
    for the next chunk).
    """
    import torch

    B, T, H, W, c_in = x.shape
    c_out = c_in if cache is None else weight.shape[0]
    t_out = T if cache is None else T // 2
    y = torch.empty(B, t_out, H, W, c_out, dtype=torch.bfloat16, device=x.device)
    new_cache = torch.empty(B, 1, H, W, c_in, dtype=torch.bfloat16, device=x.device)
    check(wan_vae_time_downsample(x, cache, weight, bias, y, new_cache, B, T, H, W, c_in, c_out, stream),
          "wan_vae_time_downsample")
    return y, new_cache
