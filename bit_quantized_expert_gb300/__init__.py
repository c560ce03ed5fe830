"""Python binding of the GB300 4-bit MoE layer library (libmoe_gb300.so).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
Tensors are torch CUDA tensors; bf16 data may be passed as torch.bfloat16 or as 16-bit
integer bit patterns.  The C declarations and contracts are in include/moe.h.

There is no fallback: importing works without a GPU (so the exported symbols can be
inspected), but every call needs the built library and a CUDA device, and raises otherwise.
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoe_gb300.so")

# Symbols declared in include/moe.h, include/gqa_attention.h, include/deltanet_scan.h and
# include/moe_probe.h.
EXPORTED = ("moe_status_string", "moe_max_tiles", "moe_workspace_bytes", "moe_route",
            "moe_expert_forward", "moe_layer_forward", "moe_layer_forward_opts", "moe_rmsnorm_router",
            "moe_clear_error_flags",
            "moe_read_error_flags", "moe_layer_forward_decode_noalloc", "moe_workspace_bytes_host",
            "moe_layer_forward_host", "moe_decode_stream_probe", "gqa_decode_workspace_bytes",
            "gqa_decode_attention", "gdn_scan_workspace_bytes", "gdn_scan", "gdn_scan_opts",
            "moe_wait_timeout_probe", "moe_layer_forward_host_opts")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_MISALIGNED",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA"}
ERR_WAIT_TIMEOUT, ERR_FP16_RANGE, ERR_BAD_ROUTING, ERR_NON_FINITE = 1, 2, 4, 8
OPT_BF16_OPERANDS = 1
OPT_HOST_INPUTS_READY = 1
_OPERAND_OPTS = {"fp16": 0, "bf16": OPT_BF16_OPERANDS}


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("F", ctypes.c_int32), ("F_shared", ctypes.c_int32)]


class QMat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class ExpertsC(ctypes.Structure):
    _fields_ = [("gate", QMat), ("up", QMat), ("down", QMat)]


class GqaDims(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("n_ctx", ctypes.c_int32), ("capacity", ctypes.c_int32)]


class GdnDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32)]


class RoutingC(ctypes.Structure):
    _fields_ = [("idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("perm", ctypes.c_void_p), ("inv", ctypes.c_void_p),
                ("tiles", ctypes.c_void_p), ("num_tiles", ctypes.c_void_p), ("tile_n", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build it with `python -m bit_quantized_expert_gb300.build`")
    try:
        import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    except Exception:
        pass
    lib = ctypes.CDLL(path)
    P, S, I32, VP = ctypes.POINTER, ctypes.c_size_t, ctypes.c_int32, ctypes.c_void_p
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_max_tiles.restype = S
    lib.moe_max_tiles.argtypes = [P(Dims), I32]
    lib.moe_workspace_bytes.restype = S
    lib.moe_workspace_bytes.argtypes = [P(Dims)]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_route.argtypes = [P(Dims), VP, P(RoutingC), VP, S, VP]
    lib.moe_expert_forward.restype = ctypes.c_int
    lib.moe_expert_forward.argtypes = [P(Dims), VP, P(RoutingC), P(ExpertsC), P(ExpertsC), VP, VP, S, VP]
    lib.moe_layer_forward.restype = ctypes.c_int
    lib.moe_layer_forward.argtypes = [P(Dims), VP, VP, P(ExpertsC), P(ExpertsC), VP, VP, P(RoutingC), VP, S, VP]
    lib.moe_layer_forward_opts.restype = ctypes.c_int
    lib.moe_layer_forward_opts.argtypes = [P(Dims), VP, VP, P(ExpertsC), P(ExpertsC), VP, VP, P(RoutingC), VP, S, VP,
                                           ctypes.c_uint32]
    lib.moe_rmsnorm_router.restype = ctypes.c_int
    lib.moe_rmsnorm_router.argtypes = [P(Dims), VP, VP, VP, VP, ctypes.c_float, VP, VP, VP, S, VP]
    lib.moe_workspace_bytes_host.restype = S
    lib.moe_workspace_bytes_host.argtypes = [P(Dims)]
    lib.moe_layer_forward_host.restype = ctypes.c_int
    lib.moe_layer_forward_host.argtypes = [P(Dims), VP, VP, P(ExpertsC), P(ExpertsC), VP, VP, VP, S, VP]
    lib.moe_layer_forward_host_opts.restype = ctypes.c_int
    lib.moe_layer_forward_host_opts.argtypes = [P(Dims), VP, VP, P(ExpertsC), P(ExpertsC), VP, VP, VP, S, VP,
                                                ctypes.c_uint32]
    lib.moe_layer_forward_decode_noalloc.restype = ctypes.c_int
    lib.moe_layer_forward_decode_noalloc.argtypes = [P(Dims), VP, VP, P(ExpertsC), P(ExpertsC), VP, VP, VP]
    lib.moe_decode_stream_probe.restype = ctypes.c_int
    lib.moe_decode_stream_probe.argtypes = [P(Dims), VP, P(ExpertsC), P(ExpertsC), VP, S, VP]
    lib.moe_wait_timeout_probe.restype = ctypes.c_int
    lib.moe_wait_timeout_probe.argtypes = [VP, S, ctypes.c_longlong, VP]
    lib.gqa_decode_workspace_bytes.restype = S
    lib.gqa_decode_workspace_bytes.argtypes = [P(GqaDims)]
    lib.gqa_decode_attention.restype = ctypes.c_int
    lib.gqa_decode_attention.argtypes = [P(GqaDims), VP, VP, VP, VP, VP, S, VP]
    lib.gdn_scan_workspace_bytes.restype = S
    lib.gdn_scan_workspace_bytes.argtypes = [P(GdnDims)]
    lib.gdn_scan.restype = ctypes.c_int
    lib.gdn_scan.argtypes = [P(GdnDims), VP, VP, VP, VP, VP, VP, VP, VP, VP, S, VP]
    lib.gdn_scan_opts.restype = ctypes.c_int
    lib.gdn_scan_opts.argtypes = [P(GdnDims), VP, VP, VP, VP, VP, VP, VP, VP, VP, S, VP, ctypes.c_uint32]
    lib.moe_clear_error_flags.restype = ctypes.c_int
    lib.moe_clear_error_flags.argtypes = [VP, S, VP]
    lib.moe_read_error_flags.restype = ctypes.c_int
    lib.moe_read_error_flags.argtypes = [VP, S, P(ctypes.c_uint32), VP]
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise MoeError(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    """A torch stream, a raw cudaStream_t handle (int), or None for torch's current stream."""
    if isinstance(stream, int):
        return stream
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def dims(T, d, E, k, F, F_shared) -> Dims:
    return Dims(int(T), int(d), int(E), int(k), int(F), int(F_shared))


def experts_struct(ex: dict | None) -> ExpertsC | None:
    """{"gate"|"up"|"down": {"codes", "scales", "biases"}} of CUDA tensors -> C struct."""
    if ex is None:
        return None

    def q(m):
        return QMat(_ptr(m["codes"]), _ptr(m["scales"]), _ptr(m["biases"]))

    return ExpertsC(q(ex["gate"]), q(ex["up"]), q(ex["down"]))


def routing_struct(r: dict) -> RoutingC:
    return RoutingC(_ptr(r["idx"]), _ptr(r["w"]), _ptr(r["counts"]), _ptr(r["offsets"]), _ptr(r["perm"]),
                    _ptr(r["inv"]), _ptr(r["tiles"]), _ptr(r["num_tiles"]), int(r["tile_n"]))


def max_tiles(dm: Dims, tile_n: int) -> int:
    return load_library().moe_max_tiles(ctypes.byref(dm), int(tile_n))


def workspace_bytes(dm: Dims) -> int:
    n = load_library().moe_workspace_bytes(ctypes.byref(dm))
    if n == 0:
        raise MoeError(1, "moe_workspace_bytes")
    return n


def alloc_workspace(dm: Dims, device="cuda"):
    """Workspace for these dims with its error word cleared."""
    import torch
    ws = torch.empty(workspace_bytes(dm), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def workspace_bytes_host(dm: Dims) -> int:
    n = load_library().moe_workspace_bytes_host(ctypes.byref(dm))
    if n == 0:
        raise MoeError(1, "moe_workspace_bytes_host")
    return n


def alloc_workspace_host(dm: Dims, device="cuda"):
    """Workspace (with the host-call staging area) for these dims, its error word cleared."""
    import torch
    ws = torch.empty(workspace_bytes_host(dm), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def _host_ptr(t) -> int:
    if t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def clear_error_flags(workspace, stream=None):
    _check(load_library().moe_clear_error_flags(_ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_clear_error_flags")


def alloc_routing(dm: Dims, tile_n: int = 128, device="cuda") -> dict:
    import torch
    T, k, E = dm.T, dm.k, dm.E
    i32 = dict(dtype=torch.int32, device=device)
    return {"idx": torch.empty((T, k), **i32), "w": torch.empty((T, k), dtype=torch.float32, device=device),
            "counts": torch.empty(E, **i32), "offsets": torch.empty(E + 1, **i32),
            "perm": torch.empty(T * k, **i32), "inv": torch.empty(T * k, **i32),
            "tiles": torch.empty((max(1, max_tiles(dm, tile_n)), 4), **i32),
            "num_tiles": torch.empty(1, **i32), "tile_n": tile_n}


def route(dm: Dims, logits, routing: dict, workspace, stream=None):
    r = routing_struct(routing)
    _check(load_library().moe_route(ctypes.byref(dm), _ptr(logits), ctypes.byref(r), _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "moe_route")


def expert_forward(dm: Dims, x, routing: dict, routed: dict, shared: dict | None, y_perm, workspace,
                   stream=None):
    r = routing_struct(routing)
    re, se = experts_struct(routed), experts_struct(shared)
    _check(load_library().moe_expert_forward(ctypes.byref(dm), _ptr(x), ctypes.byref(r), ctypes.byref(re),
                                             ctypes.byref(se) if se is not None else None, _ptr(y_perm),
                                             _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_expert_forward")


def layer_forward(dm: Dims, x, logits, routed: dict, shared: dict | None, w_sg, y, workspace,
                  routing: dict | None = None, stream=None, operands: str = "fp16"):
    """operands: the grouped-GEMM path's tensor-core operand type, "fp16" (moe_layer_forward) or
    "bf16" (moe_layer_forward_opts with MOE_OPT_BF16_OPERANDS)."""
    re, se = experts_struct(routed), experts_struct(shared)
    r = routing_struct(routing) if routing is not None else None
    _check(load_library().moe_layer_forward_opts(ctypes.byref(dm), _ptr(x), _ptr(logits), ctypes.byref(re),
                                                 ctypes.byref(se) if se is not None else None, _ptr(w_sg), _ptr(y),
                                                 ctypes.byref(r) if r is not None else None, _ptr(workspace),
                                                 workspace.numel(), _stream(stream), _OPERAND_OPTS[operands]),
           "moe_layer_forward_opts")


def rmsnorm_router(dm: Dims, x_resid, y_prev, gamma, w_router, eps: float, h_out, logits_out, workspace,
                   stream=None):
    _check(load_library().moe_rmsnorm_router(ctypes.byref(dm), _ptr(x_resid), _ptr(y_prev), _ptr(gamma),
                                             _ptr(w_router), float(eps), _ptr(h_out), _ptr(logits_out),
                                             _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_rmsnorm_router")


def layer_forward_decode_noalloc(dm: Dims, x, logits, routed: dict, shared: dict | None, w_sg, y, stream=None):
    """One-token layer call without a workspace (scratch is a library-owned device array)."""
    re, se = experts_struct(routed), experts_struct(shared)
    _check(load_library().moe_layer_forward_decode_noalloc(
        ctypes.byref(dm), _ptr(x), _ptr(logits), ctypes.byref(re), ctypes.byref(se) if se is not None else None,
        _ptr(w_sg), _ptr(y), _stream(stream)), "moe_layer_forward_decode_noalloc")


def decode_stream_probe(dm: Dims, idx, routed: dict, shared: dict | None, workspace, stream=None):
    """Loads-only replica of the one-token decode launch (include/moe_probe.h): moves the weight
    bytes of the experts in idx (int32 [k]) and nothing else."""
    re, se = experts_struct(routed), experts_struct(shared)
    _check(load_library().moe_decode_stream_probe(ctypes.byref(dm), _ptr(idx), ctypes.byref(re),
                                                  ctypes.byref(se) if se is not None else None, _ptr(workspace),
                                                  workspace.numel(), _stream(stream)), "moe_decode_stream_probe")


def wait_timeout_probe(workspace, limit_cycles: int, stream=None):
    """Make the library's bounded device wait run out after limit_cycles SM cycles: the error word
    of the workspace gets the timeout bit (ERR_WAIT_TIMEOUT) and nothing else changes."""
    _check(load_library().moe_wait_timeout_probe(_ptr(workspace), workspace.numel(), int(limit_cycles),
                                                 _stream(stream)), "moe_wait_timeout_probe")


def gqa_dims(n_heads, n_kv_heads, head_dim, n_ctx, capacity=None) -> GqaDims:
    return GqaDims(int(n_heads), int(n_kv_heads), int(head_dim), int(n_ctx),
                   int(n_ctx if capacity is None else capacity))


def gqa_workspace_bytes(gd: GqaDims) -> int:
    n = load_library().gqa_decode_workspace_bytes(ctypes.byref(gd))
    if n == 0:
        raise MoeError(1, "gqa_decode_workspace_bytes")
    return n


def alloc_gqa_workspace(gd: GqaDims, device="cuda"):
    """Workspace of the decode attention for these dims, its error word cleared."""
    import torch
    ws = torch.empty(gqa_workspace_bytes(gd), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def gqa_decode_attention(gd: GqaDims, q, k_cache, v_cache, o, workspace, stream=None):
    """o[h] = softmax(q[h] . K[g] / sqrt(128)) V[g] over the first n_ctx cached positions, g = h // (Hq/Hkv).
    q bf16 [Hq, 128]; caches bf16 [Hkv, capacity, 128]; o fp32 [Hq, 128]."""
    _check(load_library().gqa_decode_attention(ctypes.byref(gd), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o),
                                               _ptr(workspace), workspace.numel(), _stream(stream)),
           "gqa_decode_attention")


def gdn_dims(T, H, d_k=128, d_v=128) -> GdnDims:
    return GdnDims(int(T), int(H), int(d_k), int(d_v))


def alloc_gdn_workspace(gd: GdnDims, device="cuda"):
    """Workspace of the Gated DeltaNet scan (its error word), cleared."""
    import torch
    n = load_library().gdn_scan_workspace_bytes(ctypes.byref(gd))
    if n == 0:
        raise MoeError(1, "gdn_scan_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


GDN_OPT_STATE_EARLY = 1


def gdn_scan(gd: GdnDims, q, k, v, g, beta, state_in, state_out, o, workspace, stream=None, early_state=False):
    """Gated delta rule over gd.T tokens: q, k, v bf16 [T, H, 128]; g, beta fp32 [T, H];
    state_in / state_out fp32 [H, 128, 128] (may be the same tensor); o fp32 [T, H, 128].
    early_state: GDN_OPT_STATE_EARLY (gdn_scan_opts): the state is read before the preceding work on
    the stream finishes, which must then not write it."""
    lib = load_library()
    args = (ctypes.byref(gd), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in), _ptr(state_out), _ptr(o),
            _ptr(workspace), workspace.numel(), _stream(stream))
    if early_state:
        _check(lib.gdn_scan_opts(*args, GDN_OPT_STATE_EARLY), "gdn_scan_opts")
    else:
        _check(lib.gdn_scan(*args), "gdn_scan")


def read_error_flags(workspace, stream=None) -> int:
    """Synchronise, return the sticky error word and clear it."""
    out = ctypes.c_uint32(0)
    _check(load_library().moe_read_error_flags(_ptr(workspace), workspace.numel(), ctypes.byref(out),
                                               _stream(stream)), "moe_read_error_flags")
    return out.value


class Layer:
    """Device-resident weights of one MoE layer plus the dims, for repeated calls."""

    def __init__(self, routed: dict, shared: dict | None, w_sg, d: int, E: int, k: int, F: int):
        self.routed, self.shared, self.w_sg = routed, shared, w_sg
        self.d, self.E, self.k, self.F = d, E, k, F
        self._re = experts_struct(routed)
        self._se = experts_struct(shared)
        self._se_ref = ctypes.byref(self._se) if self._se is not None else None
        self._dims = {}   # T -> Dims, reused by forward_host

    def dims(self, T: int) -> Dims:
        return dims(T, self.d, self.E, self.k, self.F, self.F if self.shared is not None else 0)

    def forward_host(self, x_host, logits_host, y_host, workspace, stream=None, inputs_ready=False):
        """The layer on host tensors, queued on the stream (a torch stream, a raw handle, or None
        for the current one).  Pinned, 16-byte-aligned tensors at T = 1 are read and written by
        the decode kernel in place; otherwise the library stages them with copies (asynchronous
        for pinned memory).  inputs_ready: MOE_OPT_HOST_INPUTS_READY (moe_layer_forward_host_opts):
        x_host and logits_host are final when the call is made, so they may be read before the
        preceding work on the stream finishes."""
        T = x_host.shape[0]
        dm = self._dims.get(T)
        if dm is None:
            dm = self._dims[T] = self.dims(T)
        lib = load_library()
        args = (ctypes.byref(dm), _host_ptr(x_host), _host_ptr(logits_host), ctypes.byref(self._re), self._se_ref,
                _ptr(self.w_sg), _host_ptr(y_host), _ptr(workspace), workspace.numel(), _stream(stream))
        if inputs_ready:
            _check(lib.moe_layer_forward_host_opts(*args, OPT_HOST_INPUTS_READY), "moe_layer_forward_host_opts")
        else:
            _check(lib.moe_layer_forward_host(*args), "moe_layer_forward_host")

    def forward(self, x, logits, y, workspace, routing: dict | None = None, stream=None, operands: str = "fp16"):
        """operands: "fp16" (moe_layer_forward) or "bf16" (moe_layer_forward_opts with bf16
        tensor-core operands on the grouped-GEMM path)."""
        dm = self.dims(x.shape[0])
        r = routing_struct(routing) if routing is not None else None
        lib = load_library()
        args = (ctypes.byref(dm), _ptr(x), _ptr(logits), ctypes.byref(self._re),
                ctypes.byref(self._se) if self._se is not None else None, _ptr(self.w_sg), _ptr(y),
                ctypes.byref(r) if r is not None else None, _ptr(workspace), workspace.numel(), _stream(stream))
        if operands == "fp16":
            _check(lib.moe_layer_forward(*args), "moe_layer_forward")
        else:
            _check(lib.moe_layer_forward_opts(*args, _OPERAND_OPTS[operands]), "moe_layer_forward_opts")


def to_device_layer(layer: dict, device="cuda") -> dict:
    """numpy layer (synth.make_layer) -> the same nesting of contiguous CUDA tensors."""
    import numpy as np
    import torch

    def t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint32:
            a = a.view(np.int32)
        elif a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(device)

    def ex(e):
        if e is None:
            return None
        return {m: {f: t(e[m][f]) for f in ("codes", "scales", "biases")} for m in ("gate", "up", "down")}

    return {"routed": ex(layer["routed"]), "shared": ex(layer.get("shared")), "w_sg": t(layer["w_sg"])}
