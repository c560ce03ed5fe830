"""The C-ABI library: it loads, exports every symbol the headers in include/ declare, and its host-side
argument checks and size queries behave as documented.  No kernel runs here (no GPU needed):
every call below returns from the host checks before any CUDA work is enqueued."""
import ctypes
import os
import re

import pytest

import bit_quantized_expert_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            with open(os.path.join(ROOT, "include", h)) as f:
                src = f.read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b((?:moe|gqa|gdn)_\w+)\s*\(", src, re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from bit_quantized_expert_gb300 import build
        build.build()
    return moe.load_library()


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert set(declared) == set(moe.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_wait_probe_host_checks(lib):
    """moe_wait_timeout_probe refuses a limit outside 1 .. 4e9 cycles and a missing, short or
    misaligned workspace before launching anything."""
    f = lib.moe_wait_timeout_probe
    assert f(256, 256, 0, None) == 1 and f(256, 256, 4000000001, None) == 1 and f(256, 256, -5, None) == 1
    assert f(None, 256, 1000, None) == 4
    assert f(256, 255, 1000, None) == 4
    assert f(264, 256, 1000, None) == 3


def test_status_strings(lib):
    for code, name in moe.STATUS.items():
        assert lib.moe_status_string(code).decode().startswith(name)


def test_workspace_and_tile_bounds(lib):
    dm = moe.dims(4096, 2048, 256, 8, 512, 512)
    ws = moe.workspace_bytes(dm)
    T, k, d, F = 4096, 8, 2048, 512
    slots = T * k + T
    assert ws >= slots * F * 2 + slots * d * 2 + slots * d * 2   # h, fp16 expert outputs, x rows per slot
    assert moe.max_tiles(dm, 128) == T * k // 128 + min(256, T * k) + T // 128
    assert moe.max_tiles(dm, 16) == T * k // 16 + min(256, T * k) + T // 16
    assert moe.max_tiles(dm, 17) == 0 and moe.max_tiles(dm, 256) == 0


def test_workspace_holds_decode_partials_per_token(lib):
    """Up to eight tokens run one decode launch that keeps, per token, one partial of every row of y
    per expert slot and cluster ((k+1) slots x F/512 clusters of 16 CTAs at F = 512, rows in
    128-row slices): the workspace grows by at least that much per token up to eight, and the
    host-buffer entry point's workspace adds room for x, logits and y behind it."""
    d, E, k, F = 2048, 256, 8, 512
    part = (k + 1) * (F // 512) * d * 4
    sizes = [moe.workspace_bytes(moe.dims(T, d, E, k, F, F)) for T in range(1, 10)]
    for T in range(1, 9):
        assert sizes[T - 1] >= T * part, T
    for T in (1, 3, 8, 9, 64):
        dm = moe.dims(T, d, E, k, F, F)
        assert lib.moe_workspace_bytes_host(ctypes.byref(dm)) >= moe.workspace_bytes(dm) + T * (d * 2 + E * 4 + d * 4)


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(k=0), dict(k=17, E=16), dict(d=200), dict(F=192), dict(F_shared=256),
    dict(E=2000), dict(k=40, E=64)])
def test_invalid_dims_rejected(lib, bad):
    args = dict(T=4, d=256, E=16, k=2, F=128, F_shared=128)
    args.update(bad)
    assert lib.moe_workspace_bytes(ctypes.byref(moe.dims(**args))) == 0


def test_route_host_checks(lib):
    dm = moe.dims(4, 256, 16, 2, 128, 128)
    ws_n = moe.workspace_bytes(dm)
    good = moe.RoutingC(16, 16, 16, 16, 16, 16, 16, 16, 128)
    # null logits
    assert lib.moe_route(ctypes.byref(dm), None, ctypes.byref(good), 16, ws_n, None) == 1
    # misaligned logits
    assert lib.moe_route(ctypes.byref(dm), 20, ctypes.byref(good), 16, ws_n, None) == 3
    # workspace too small / missing
    assert lib.moe_route(ctypes.byref(dm), 16, ctypes.byref(good), 16, ws_n - 1, None) == 4
    assert lib.moe_route(ctypes.byref(dm), 16, ctypes.byref(good), None, ws_n, None) == 4
    # bad tile_n
    bad = moe.RoutingC(16, 16, 16, 16, 16, 16, 16, 16, 24)
    assert lib.moe_route(ctypes.byref(dm), 16, ctypes.byref(bad), 16, ws_n, None) == 1
    # T == 0 is a no-op
    dm0 = moe.dims(0, 256, 16, 2, 128, 128)
    assert lib.moe_route(ctypes.byref(dm0), None, ctypes.byref(good), None, 0, None) == 0


def test_layer_host_checks(lib):
    dm = moe.dims(4, 256, 16, 2, 128, 128)
    ws_n = moe.workspace_bytes(dm)
    q = moe.QMat(16, 16, 16)
    ex = moe.ExpertsC(q, q, q)
    call = lambda **kw: lib.moe_layer_forward(
        ctypes.byref(kw.get("dm", dm)), kw.get("x", 16), kw.get("lg", 16), ctypes.byref(kw.get("re", ex)),
        kw.get("se", ctypes.byref(ex)), kw.get("wsg", 16), kw.get("y", 16), None, kw.get("ws", 16),
        kw.get("wsn", ws_n), None)
    assert call(x=None) == 1
    assert call(y=8) == 3
    assert call(wsg=None) == 1
    assert call(re=moe.ExpertsC(moe.QMat(16, 16, 0), q, q)) == 1
    assert call(re=moe.ExpertsC(moe.QMat(16, 24, 16), q, q)) == 3
    assert call(se=None) == 1                  # dims say there is a shared expert
    assert call(wsn=ws_n - 256) == 4
    dm_ns = moe.dims(4, 256, 16, 2, 128, 0)
    assert call(dm=dm_ns) == 1                 # a shared expert given but dims say none


def test_layer_options_host_checks(lib):
    """moe_layer_forward_opts: an unknown option bit is refused before anything else; with a known
    one the argument checks of moe_layer_forward apply (these calls fail on the host, no launch)."""
    dm = moe.dims(4, 256, 16, 2, 128, 128)
    ws_n = moe.workspace_bytes(dm)
    q = moe.QMat(16, 16, 16)
    ex = moe.ExpertsC(q, q, q)
    call = lambda opts, **kw: lib.moe_layer_forward_opts(
        ctypes.byref(dm), kw.get("x", 16), 16, ctypes.byref(ex), ctypes.byref(ex), 16, kw.get("y", 16), None, 16,
        ws_n, None, opts)
    assert moe.OPT_BF16_OPERANDS == 1
    for bad in (2, 4, 0x80000000, 0xFFFFFFFF):
        assert call(bad) == 1, bad
    assert call(moe.OPT_BF16_OPERANDS, x=None) == 1
    assert call(moe.OPT_BF16_OPERANDS, y=8) == 3
    assert call(0, y=8) == 3


def test_layer_host_entry_checks(lib):
    """The host-buffer entry point refuses what it must before touching the GPU."""
    dm = moe.dims(4, 256, 16, 2, 128, 128)
    ws_n, ws_h = moe.workspace_bytes(dm), moe.workspace_bytes_host(dm)
    # staging for x (bf16), logits (fp32) and y (fp32), each padded to 256 bytes
    assert ws_h >= ws_n + 4 * 256 * 2 + 4 * 16 * 4 + 4 * 256 * 4
    q = moe.QMat(16, 16, 16)
    ex = moe.ExpertsC(q, q, q)
    call = lambda **kw: lib.moe_layer_forward_host(
        ctypes.byref(kw.get("dm", dm)), kw.get("x", 16), kw.get("lg", 16), ctypes.byref(ex), ctypes.byref(ex),
        16, kw.get("y", 16), kw.get("ws", 16), kw.get("wsn", ws_h), None)
    assert call(x=None) == 1
    assert call(lg=None) == 1
    assert call(y=None) == 1
    assert call(ws=None) == 4
    assert call(wsn=ws_h - 1) == 4
    assert call(wsn=ws_n) == 4
    assert call(dm=moe.dims(0, 256, 16, 2, 128, 128)) == 0   # T == 0: nothing to do
    # moe_layer_forward_host_opts: unknown option bits refused first; the known one checks alike
    opts = lambda o, **kw: lib.moe_layer_forward_host_opts(
        ctypes.byref(kw.get("dm", dm)), kw.get("x", 16), 16, ctypes.byref(ex), ctypes.byref(ex), 16, 16,
        kw.get("ws", 16), ws_h, None, o)
    assert moe.OPT_HOST_INPUTS_READY == 1
    for bad in (2, 0x80000000, 0xFFFFFFFF):
        assert opts(bad) == 1, bad
    assert opts(1, x=None) == 1 and opts(1, ws=None) == 4
    assert opts(1, dm=moe.dims(0, 256, 16, 2, 128, 128)) == 0


def test_gqa_workspace_bytes(lib):
    """256-byte head, then Hkv * min(ceil(N / 64), 256) blocks of 4160 bytes (1024 + 16 floats)."""
    for Hq, Hkv, N in ((16, 2, 1), (16, 2, 64), (16, 2, 65), (16, 2, 32768), (16, 2, 131072), (8, 8, 1000)):
        gd = moe.gqa_dims(Hq, Hkv, 128, N)
        assert lib.gqa_decode_workspace_bytes(ctypes.byref(gd)) == 256 + Hkv * min(-(-N // 64), 256) * 4160


@pytest.mark.parametrize("bad", [
    dict(head_dim=64), dict(n_heads=18), dict(n_heads=32), dict(n_ctx=0), dict(n_ctx=10, capacity=9),
    dict(n_kv_heads=0), dict(n_ctx=-1)])
def test_gqa_invalid_dims_rejected(lib, bad):
    args = dict(n_heads=16, n_kv_heads=2, head_dim=128, n_ctx=100, capacity=100)
    args.update(bad)
    gd = moe.GqaDims(**{k: int(v) for k, v in args.items()})
    assert lib.gqa_decode_workspace_bytes(ctypes.byref(gd)) == 0


def test_gqa_host_checks(lib):
    """Statuses of include/gqa_attention.h, all returned before any CUDA work: 1 for a null pointer,
    Hq % Hkv != 0, N < 1 or N > capacity; 2 for head_dim != 128 or more than 8 query heads per
    key/value head; 3 for a misaligned pointer; 4 for a short workspace."""
    gd = moe.gqa_dims(16, 2, 128, 100)
    n = lib.gqa_decode_workspace_bytes(ctypes.byref(gd))
    call = lambda dims=gd, q=16, k=16, v=16, o=16, ws=16, nb=n: lib.gqa_decode_attention(
        ctypes.byref(dims), q, k, v, o, ws, nb, None)
    assert call(q=None) == 1 and call(k=None) == 1 and call(v=None) == 1 and call(o=None) == 1
    assert call(ws=None) == 1
    assert call(q=18) == 3 and call(k=24) == 3 and call(o=20) == 3 and call(ws=8) == 3
    assert call(nb=n - 1) == 4
    assert call(dims=moe.gqa_dims(16, 3, 128, 100)) == 1
    assert call(dims=moe.gqa_dims(16, 2, 128, 0)) == 1
    assert call(dims=moe.gqa_dims(16, 2, 128, 101, 100)) == 1
    assert call(dims=moe.gqa_dims(16, 2, 64, 100)) == 2
    assert call(dims=moe.gqa_dims(32, 2, 128, 100)) == 2


def test_gdn_workspace_and_host_checks(lib):
    """include/deltanet_scan.h: the workspace is the 256-byte error-word head; 1 for a null pointer,
    T < 0 or H < 1; 2 for sizes other than 128; 3 for a misaligned pointer; 4 for a short workspace."""
    gd = moe.gdn_dims(64, 16)
    assert lib.gdn_scan_workspace_bytes(ctypes.byref(gd)) == 256
    for bad in (moe.gdn_dims(-1, 16), moe.gdn_dims(4, 0), moe.gdn_dims(4, 16, 64), moe.gdn_dims(4, 16, 128, 256)):
        assert lib.gdn_scan_workspace_bytes(ctypes.byref(bad)) == 0
    call = lambda dims=gd, q=16, k=16, v=16, g=16, b=16, si=16, so=16, o=16, ws=16, nb=256: lib.gdn_scan(
        ctypes.byref(dims), q, k, v, g, b, si, so, o, ws, nb, None)
    assert call(q=None) == 1 and call(si=None) == 1 and call(so=None) == 1 and call(ws=None) == 1
    assert call(dims=moe.gdn_dims(-3, 16)) == 1 and call(dims=moe.gdn_dims(3, 0)) == 1
    assert call(dims=moe.gdn_dims(3, 16, 64, 64)) == 2
    assert call(k=24) == 3 and call(g=20) == 3 and call(so=8) == 3
    assert call(nb=255) == 4
    # gdn_scan_opts: an unknown option bit is refused; with the known one the same checks apply
    opts = lambda o, **kw: lib.gdn_scan_opts(ctypes.byref(kw.get("dims", gd)), kw.get("q", 16), 16, 16, 16, 16, 16, 16,
                                             16, 16, kw.get("nb", 256), None, o)
    assert moe.GDN_OPT_STATE_EARLY == 1
    assert opts(2) == 1 and opts(0x80000000) == 1
    assert opts(1, q=None) == 1 and opts(1, q=24) == 3 and opts(1, nb=255) == 4
