"""The C-ABI library: it loads, exports what the header declares, and rejects
bad arguments on the host before touching CUDA (no GPU needed)."""
import os
import re

import pytest

import long_sequence_attention_02_b300 as wan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wan_attn.h")


@pytest.fixture(scope="module")
def lib():
    from long_sequence_attention_02_b300 import build

    build.build_attn()
    return wan.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wan_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(wan.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert wan.status_str(0) == "WAN_OK"
    for code in (1, 2, 3, 4, 5):
        assert wan.status_str(code).startswith("WAN_ERR")
    assert wan.wan_version() >= 100


def test_table_and_workspace_sizes(lib):
    assert wan.wan_rope3d_tables_size((3, 8, 8)) == (3 * 22 + 8 * 21 + 8 * 21) * 8
    assert wan.wan_rope3d_tables_size((21, 45, 80)) == (21 * 22 + 45 * 21 + 80 * 21) * 8
    assert wan.wan_rope3d_tables_size((0, 8, 8)) == 0
    assert wan.wan_rope3d_tables_size((3, 8, 8), 64) == 0
    n = 1 * 75600 * 40 * 128 * 2
    assert wan.wan_attn_workspace_size(wan.WAN_OP_FWD, 1, (21, 45, 80), 40) >= n
    assert wan.wan_attn_workspace_size(wan.WAN_OP_BWD, 1, (4, 4, 4), 2) > 0
    assert wan.wan_attn_workspace_size(7, 1, (4, 4, 4), 2) == 0


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every case fails validation first


def test_fwd_rejects_bad_arguments(lib):
    g = (2, 4, 4)
    ws = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, 1, g, 2)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, grid=g, H=2, head_dim=128, tables=FAKE,
              scale=0.088, workspace=FAKE, ws_bytes=ws, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_attn_fwd(**a)

    assert call(q=None) == wan.WAN_ERR_INVALID
    assert call(tables=None) == wan.WAN_ERR_INVALID
    assert call(workspace=None) == wan.WAN_ERR_INVALID
    assert call(q=FAKE + 8) == wan.WAN_ERR_INVALID
    assert call(o=FAKE + 2) == wan.WAN_ERR_INVALID
    assert call(ws_bytes=ws - 1) == wan.WAN_ERR_INVALID
    assert call(grid=(0, 4, 4)) == wan.WAN_ERR_INVALID
    assert call(grid=(2, -1, 4)) == wan.WAN_ERR_INVALID
    assert call(H=0) == wan.WAN_ERR_INVALID
    assert call(B=-1) == wan.WAN_ERR_INVALID
    assert call(scale=0.0) == wan.WAN_ERR_INVALID
    assert call(scale=float("nan")) == wan.WAN_ERR_INVALID
    assert call(head_dim=64) == wan.WAN_ERR_UNSUPPORTED
    # zero work is a no-op that launches nothing
    assert call(B=0, q=None, k=None, v=None, o=None, lse=None, workspace=None, ws_bytes=0) == wan.WAN_OK


def test_xattn_rejects_bad_arguments(lib):
    g = (2, 4, 4)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, kv_lens=None, Lk=77, o=FAKE, lse=None, B=2, grid=g, H=2, head_dim=128,
              scale=0.088, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_xattn_fwd(**a)

    assert call(Lk=0) == wan.WAN_ERR_INVALID
    assert call(Lk=513) == wan.WAN_ERR_INVALID
    assert call(k=None) == wan.WAN_ERR_INVALID
    assert call(kv_lens=FAKE + 2) == wan.WAN_ERR_INVALID
    assert call(lse=FAKE + 1) == wan.WAN_ERR_INVALID
    assert call(head_dim=96) == wan.WAN_ERR_UNSUPPORTED
    assert call(B=0, q=None) == wan.WAN_OK


def test_bwd_rejects_bad_arguments(lib):
    g = (2, 4, 4)
    ws = wan.wan_attn_workspace_size(wan.WAN_OP_BWD, 1, g, 2)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, grid=g, H=2,
              head_dim=128, tables=FAKE, scale=0.088, workspace=FAKE, ws_bytes=ws, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_attn_bwd(**a)

    for name in ("q", "k", "v", "o", "lse", "dout", "dq", "dk", "dv", "tables", "workspace"):
        assert call(**{name: None}) == wan.WAN_ERR_INVALID, name
    assert call(dq=FAKE + 4) == wan.WAN_ERR_INVALID
    assert call(ws_bytes=ws - 16) == wan.WAN_ERR_INVALID
    assert call(head_dim=256) == wan.WAN_ERR_UNSUPPORTED


def test_tables_reject_bad_arguments(lib):
    assert wan.wan_rope3d_tables((3, 8, 8), 128, 10000.0, None, 0) == wan.WAN_ERR_INVALID
    assert wan.wan_rope3d_tables((3, 8, 8), 128, 0.5, FAKE, 0) == wan.WAN_ERR_INVALID
    assert wan.wan_rope3d_tables((3, 0, 8), 128, 1e4, FAKE, 0) == wan.WAN_ERR_INVALID
    assert wan.wan_rope3d_tables((3, 8, 8), 100, 1e4, FAKE, 0) == wan.WAN_ERR_UNSUPPORTED


def test_profile_pass_hook_argument_checks(lib):
    assert lib.wan_profile_set_pass_events(4, None, None) == wan.WAN_ERR_INVALID
    assert lib.wan_profile_set_pass_events(-1, None, None) == wan.WAN_ERR_INVALID
    assert lib.wan_profile_set_pass_events(wan.WAN_PASS_ROPE, 1, None) == wan.WAN_ERR_INVALID
    for p in (wan.WAN_PASS_MAIN, wan.WAN_PASS_ROPE, wan.WAN_PASS_ROWS, wan.WAN_PASS_POST):
        assert lib.wan_profile_set_pass_events(p, None, None) == wan.WAN_OK


def test_debug_hook_argument_checks(lib):
    assert wan.wan_debug_inject_stall(-1, 10) == wan.WAN_ERR_INVALID
    assert wan.wan_debug_inject_stall(1, 0) == wan.WAN_ERR_INVALID
    assert wan.wan_debug_inject_stall(0, 100) == wan.WAN_OK


def test_fp8_workspace_size(lib):
    # e4m3 Q and K [B, L, H, 128], V transposed to [B, H, 128, Lpad] (Lpad = L rounded up to 16)
    # and the per-head amax triples, each region 256-byte aligned
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for B, g, H in [(1, (21, 45, 80), 40), (2, (3, 7, 9), 3), (1, (1, 1, 1), 1)]:
        L = g[0] * g[1] * g[2]
        lpad = (L + 15) // 16 * 16
        n = B * L * H * 128
        want = up(n) + up(n) + up(B * H * 128 * lpad) + up(B * H * 3 * 4)
        assert wan.wan_attn_workspace_size(wan.WAN_OP_FWD_FP8, B, g, H) == want


def test_fp8_rejects_bad_arguments(lib):
    g = (2, 4, 4)
    ws = wan.wan_attn_workspace_size(wan.WAN_OP_FWD_FP8, 1, g, 2)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, grid=g, H=2, head_dim=128, tables=FAKE,
              scale=0.088, workspace=FAKE, ws_bytes=ws, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_attn_fwd_fp8(**a)

    assert call(k=None) == wan.WAN_ERR_INVALID
    assert call(workspace=None) == wan.WAN_ERR_INVALID
    assert call(v=FAKE + 4) == wan.WAN_ERR_INVALID
    assert call(lse=FAKE + 2) == wan.WAN_ERR_INVALID
    assert call(ws_bytes=ws - 1) == wan.WAN_ERR_INVALID
    assert call(grid=(2, 0, 4)) == wan.WAN_ERR_INVALID
    assert call(scale=float("inf")) == wan.WAN_ERR_INVALID
    assert call(head_dim=256) == wan.WAN_ERR_UNSUPPORTED
    assert call(B=0, q=None, k=None, v=None, o=None, lse=None, workspace=None, ws_bytes=0) == wan.WAN_OK


def test_ring_step_rejects_bad_ranges(lib):
    g = (2, 4, 4)  # 32 tokens
    ok = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, grid=g, H=1, head_dim=128, tables=FAKE, scale=0.088,
              q_start=0, q_len=4, kv_start=0, kv_len=4, accumulate=0, workspace=FAKE, ws_bytes=1 << 16, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_attn_fwd_ring_step(**a)

    for bad in [dict(q_start=-1), dict(q_len=0), dict(q_start=30, q_len=3), dict(kv_start=29, kv_len=4),
                dict(kv_len=0), dict(accumulate=2), dict(lse=None), dict(ws_bytes=4 * 256 - 1)]:
        assert call(**bad) == wan.WAN_ERR_INVALID, bad


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    # one row-head more than the fixed scratch holds fails before any device work
    assert wan.NOALLOC_MAX_ROW_HEADS == 262144
    g = (1, 1, 2049)  # 2049 tokens x 128 heads = 262,272 row-heads
    assert wan.wan_attn_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, g, 128, 128, FAKE, 0.088) == wan.WAN_ERR_INVALID
    assert wan.wan_attn_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, (0, 4, 4), 2, 128, FAKE, 0.088) == \
        wan.WAN_ERR_INVALID


def test_conv3d_rejects_bad_arguments(lib):
    # x [1, 4, 8, 16, 64], y [1, 4, 8, 16, 128], cache [1, 2, 8, 16, 64], weight [128, 27, 64]
    frame = 8 * 16 * 64 * 2
    X, Y, C, Wt = FAKE, FAKE + (1 << 24), FAKE + (2 << 24), FAKE + (3 << 24)
    ok = dict(x=X, cache=C, weight=Wt, bias=FAKE + (4 << 24), y=Y, cache_out=C, B=1, T=4, H=8, W=16, c_in=64,
              c_out=128, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_vae_causal_conv3d(**a)

    assert call(x=None) == wan.WAN_ERR_INVALID
    assert call(weight=None) == wan.WAN_ERR_INVALID
    assert call(y=None) == wan.WAN_ERR_INVALID
    assert call(x=X + 8) == wan.WAN_ERR_INVALID
    assert call(bias=FAKE + 2) == wan.WAN_ERR_INVALID
    assert call(T=0) == wan.WAN_ERR_INVALID
    assert call(H=-1) == wan.WAN_ERR_INVALID
    assert call(c_in=80) == wan.WAN_ERR_UNSUPPORTED         # channels must be multiples of 32
    assert call(c_out=48) == wan.WAN_ERR_UNSUPPORTED
    assert call(c_out=8224) == wan.WAN_ERR_UNSUPPORTED       # more than 8192 output channels
    assert call(y=X + frame) == wan.WAN_ERR_INVALID          # output overlapping the input
    assert call(cache_out=X) == wan.WAN_ERR_INVALID          # next cache over the input
    assert call(cache_out=C + 64) == wan.WAN_ERR_INVALID     # partly over the cache it reads
    assert call(B=0, x=None, weight=None, y=None) == wan.WAN_OK


def test_time_downsample_rejects_bad_arguments(lib):
    # x [1, 4, 8, 16, 64], y [1, 2, 8, 16, 128], cache [1, 1, 8, 16, 64], weight [128, 3, 64]
    frame = 8 * 16 * 64 * 2
    X, Y, C, Wt = FAKE, FAKE + (1 << 24), FAKE + (2 << 24), FAKE + (3 << 24)
    ok = dict(x=X, cache=C, weight=Wt, bias=FAKE + (4 << 24), y=Y, cache_out=C, B=1, T=4, H=8, W=16, c_in=64,
              c_out=128, stream=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return wan.wan_vae_time_downsample(**a)

    assert call(x=None) == wan.WAN_ERR_INVALID
    assert call(weight=None) == wan.WAN_ERR_INVALID          # a later chunk needs its weights
    assert call(y=None) == wan.WAN_ERR_INVALID
    assert call(x=X + 8) == wan.WAN_ERR_INVALID
    assert call(bias=FAKE + 2) == wan.WAN_ERR_INVALID
    assert call(T=3) == wan.WAN_ERR_INVALID                  # later chunks hold an even number of frames
    assert call(cache=None, cache_out=None) == wan.WAN_ERR_INVALID         # a first chunk is one frame
    assert call(cache=None, cache_out=None, T=1) == wan.WAN_ERR_INVALID    # ... and keeps its channels
    assert call(c_in=80) == wan.WAN_ERR_UNSUPPORTED
    assert call(c_out=48) == wan.WAN_ERR_UNSUPPORTED
    assert call(y=X + frame) == wan.WAN_ERR_INVALID          # output overlapping the input
    assert call(cache_out=X + 3 * frame) == wan.WAN_ERR_INVALID   # next cache over the input
    assert call(cache_out=C + 64) == wan.WAN_ERR_INVALID     # partly over the cache it reads
    assert call(B=0, x=None, weight=None, y=None) == wan.WAN_OK


def test_debug_build_exports_every_declared_symbol_and_says_so(lib):
    """The -DWAN_DEBUG library is the same C ABI; only it accepts the forced
    device-check hook (host-side calls only, no GPU needed)."""
    import ctypes

    from long_sequence_attention_02_b300 import build

    dbg = ctypes.CDLL(build.build_attn(debug=True))
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert dbg.wan_debug_build() == 1
    assert lib.wan_debug_build() == 0
    assert lib.wan_debug_inject_check(1) == wan.WAN_ERR_UNSUPPORTED     # release: no checks to force
    assert dbg.wan_debug_inject_check(-1) == wan.WAN_ERR_INVALID
    assert dbg.wan_debug_inject_check(0) == wan.WAN_OK
    assert dbg.wan_debug_check_line() == 0
    dbg.wan_status_str.restype = ctypes.c_char_p
    assert dbg.wan_status_str(wan.WAN_ERR_DEVICE_CHECK).decode().startswith("WAN_ERR_DEVICE_CHECK")
