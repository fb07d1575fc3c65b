"""Python binding of the GB300 MoE layer library (include/moe.h).

Thin ctypes marshalling over libmoe_gb300.so: each function takes torch CUDA
tensors, checks dtype / device / contiguity / shape, and passes raw pointers,
sizes and the current torch stream to the C function of the same name.  Every
step of the layer runs in the library's CUDA kernels; nothing here computes.

The library must be built (``serving_router_gate_gb300._build.build()``, or
``__graft_entry__.build()``); importing this module without it raises
ImportError -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_WORKSPACE", "MOE_ERR_CUDA",
    "MOE_ERR_DEVICE_BOUNDS", "MOE_ERR_TIMEOUT", "MOE_NONLOCAL_SKIP", "MOE_NONLOCAL_MOD", "MoEError",
    "lib_path", "moe_workspace_size", "moe_workspace_init", "moe_get_device_status", "moe_get_route_stats",
    "moe_route", "moe_permute", "moe_forward", "moe_grouped_fc1", "moe_grouped_fc2", "moe_finalize",
    "moe_debug_wait_timeout", "moe_set_wait_timeout_ns", "moe_route_noalloc", "moe_set_gemm_pair_mode",
    "moe_set_pdl", "moe_get_launch_count", "moe_permute_on_input", "moe_route_grouped", "moe_forward_fp8",
    "moe_quantize_fp8_rows", "moe_forward_w8a8", "moe_quantize_act_rows", "moe_grouped_fc1_fp8",
    "moe_forward_nvfp4", "moe_quantize_nvfp4_rows", "nvfp4_sf_row_bytes", "MOE_WS_HEADER_BYTES",
    "moe_grouped_fc2_fp8", "moe_grouped_fc1_w8a8", "moe_grouped_fc2_w8a8", "moe_launch_events_arm",
    "moe_launch_events_mark", "moe_launch_events_used", "EXPORTED_SYMBOLS", "moe_a2a_regroup",
    "moe_grouped_fc2_scatter", "moe_ep_signal", "moe_ep_reduce", "moe_ipc_export", "moe_ipc_import",
    "moe_ipc_close", "MOE_IPC_HANDLE_BYTES",
    "MOE_A2A_TO_GEMM", "MOE_A2A_TO_EXCHANGE",
]

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_BOUNDS = 8
MOE_ERR_TIMEOUT = 16
MOE_NONLOCAL_SKIP = 0
MOE_NONLOCAL_MOD = 1
MOE_A2A_TO_GEMM = 0
MOE_A2A_TO_EXCHANGE = 1
MOE_LAUNCH_LABEL_BYTES = 48  # bytes per label written by moe_launch_events_used
MOE_WS_HEADER_BYTES = 256    # the workspace header (status word, counters) a caller never writes
MOE_IPC_HANDLE_BYTES = 64    # bytes of a handle moe_ipc_export writes

EXPORTED_SYMBOLS = (
    "moe_status_string", "moe_workspace_size", "moe_workspace_init", "moe_get_device_status",
    "moe_get_route_stats", "moe_route", "moe_permute", "moe_forward", "moe_grouped_fc1", "moe_grouped_fc2",
    "moe_finalize", "moe_debug_wait_timeout", "moe_set_wait_timeout_ns", "moe_route_noalloc",
    "moe_set_gemm_pair_mode", "moe_set_pdl", "moe_get_launch_count", "moe_permute_on_input", "moe_route_grouped",
    "moe_forward_fp8", "moe_quantize_fp8_rows", "moe_grouped_fc1_fp8", "moe_grouped_fc2_fp8",
    "moe_forward_nvfp4", "moe_quantize_nvfp4_rows",
    "moe_forward_w8a8", "moe_quantize_act_rows", "moe_grouped_fc1_w8a8", "moe_grouped_fc2_w8a8",
    "moe_launch_events_arm", "moe_launch_events_mark", "moe_launch_events_used", "moe_a2a_regroup",
    "moe_grouped_fc2_scatter", "moe_ep_signal", "moe_ep_reduce", "moe_ipc_export", "moe_ipc_import",
    "moe_ipc_close",
)


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_lib.moe_status_string(status).decode()} (status {status})")


def lib_path() -> str:
    """The library this process loads: the bounds-checked build when MOE_CHECKED=1."""
    return _build.CHECKED_LIB_PATH if os.environ.get("MOE_CHECKED") == "1" else _build.LIB_PATH


def _load():
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} is missing (run serving_router_gate_gb300._build.build("
                          f"{'checked=True' if path == _build.CHECKED_LIB_PATH else ''}))")
    lib = ctypes.CDLL(path)
    P, i32, i64, sz, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint64
    sig = {
        "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "moe_workspace_size": ([i64, i32, i32, i32, i32, i32, i32], sz),
        "moe_workspace_init": ([P, sz, P], i32),
        "moe_get_device_status": ([P, P, P], i32),
        "moe_get_route_stats": ([P, P, P], i32),
        "moe_route": ([P, P, P, i64, i32, i32, i32, i32, P, P, P, sz, P], i32),
        "moe_route_grouped": ([P, P, P, i64, i32, i32, i32, i32, i32, i32, P, P, P, sz, P], i32),
        "moe_permute": ([P, P, i64, i32, i32, P, P, i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P, sz, P], i32),
        "moe_permute_on_input": ([P, P, i64, i32, i32, P, P, i32, i32, i32, i32, P, i32, P, P, P, P, P, P, P, sz, P],
                                 i32),
        "moe_forward": ([P, P, i32, i64, P, P, i32, i32, P, P, i64, i32, P, P, P, i32, P, P, P, sz, P], i32),
        "moe_forward_fp8": ([P, P, i32, i64, P, P, P, P, i32, i32, P, P, i64, i32, P, P, P, P, P, i32, P, P, P, sz, P],
                            i32),
        "moe_quantize_fp8_rows": ([P, i64, i32, P, P, P], i32),
        "moe_forward_w8a8": ([P, P, i32, i64, P, P, P, P, i32, i32, P, P, i64, i32, P, P, P, P, P, i32, P, P, P, sz,
                              P], i32),
        "moe_quantize_act_rows": ([P, i64, i32, P, P, P], i32),
        "moe_forward_nvfp4": ([P, P, i32, i64, P, P, P, P, P, P, i32, i32, P, P, i64, i32, P, P, P, P, P, P, P, i32,
                               P, P, P, sz, P], i32),
        "moe_quantize_nvfp4_rows": ([P, i64, i32, i32, P, P, P, P], i32),
        "moe_grouped_fc1_w8a8": ([P, P, i64, P, i32, P, P, i32, i32, P, P, i64, P, P, i32, P, P, P, sz, P], i32),
        "moe_grouped_fc2_w8a8": ([P, P, i64, P, i32, P, P, i32, i32, P, P, i64, P, P, i32, P, P, P, sz, P], i32),
        "moe_grouped_fc1_fp8": ([P, i64, P, i32, P, P, i32, i32, P, i64, P, P, i32, P, P, P, sz, P], i32),
        "moe_grouped_fc2_fp8": ([P, i64, P, i32, P, P, i32, i32, P, i64, P, P, i32, P, P, P, sz, P], i32),
        "moe_grouped_fc1": ([P, i64, P, i32, P, i32, i32, P, i64, P, i32, P, P, P, sz, P], i32),
        "moe_grouped_fc2": ([P, i64, P, i32, P, i32, i32, P, i64, P, i32, P, P, P, sz, P], i32),
        "moe_finalize": ([P, i64, P, P, i64, i32, i32, P, P, P, P, P, sz, P], i32),
        "moe_a2a_regroup": ([P, i32, i32, P, P, i64, i32, i32, P, P, P, sz, P], i32),
        "moe_grouped_fc2_scatter": ([P, i64, P, i32, P, i32, i32, P, i64, P, i32, P, P, P, P, sz, P], i32),
        "moe_ep_signal": ([P, i32, i32, i32, P], i32),
        "moe_ep_reduce": ([P, i32, P, i32, i64, i64, i32, P, P, sz, P], i32),
        "moe_ipc_export": ([P, P, P], i32),
        "moe_ipc_import": ([P, i64, P], i32),
        "moe_ipc_close": ([P, i64], i32),
        "moe_debug_wait_timeout": ([P, sz, u64, P], i32),
        "moe_set_wait_timeout_ns": ([u64], None),
        "moe_route_noalloc": ([P, P, P, i64, i32, i32, i32, i32, P, P, P], i32),
        "moe_set_gemm_pair_mode": ([i32], i32),
        "moe_set_pdl": ([i32], i32),
        "moe_get_launch_count": ([], ctypes.c_uint64),
        "moe_launch_events_arm": ([P, i32], i32),
        "moe_launch_events_mark": ([P], i32),
        "moe_launch_events_used": ([P, i32], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


# ----------------------------------------------------------------------------- marshalling helpers

def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t, name, dtype=None, shape=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn, status):
    if status != MOE_OK:
        raise MoEError(fn, status)


_bf16, _f32, _i32 = torch.bfloat16, torch.float32, torch.int32


# ----------------------------------------------------------------------------- API (names of include/moe.h)

def moe_workspace_size(max_T, H, I, E, S, k, I_shared_total=0) -> int:
    n = _lib.moe_workspace_size(max_T, H, I, E, S, k, I_shared_total)
    if n == 0:
        raise MoEError("moe_workspace_size", MOE_ERR_UNSUPPORTED)
    return int(n)


def moe_workspace_init(ws, stream=None):
    _check("moe_workspace_init", _lib.moe_workspace_init(_ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream)))


def moe_get_device_status(ws, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("moe_get_device_status",
           _lib.moe_get_device_status(_ptr(ws, "ws", torch.uint8), _stream(stream), ctypes.byref(v)))
    return int(v.value)


def moe_get_route_stats(ws, stream=None) -> int:
    v = ctypes.c_int64(0)
    _check("moe_get_route_stats",
           _lib.moe_get_route_stats(_ptr(ws, "ws", torch.uint8), _stream(stream), ctypes.byref(v)))
    return int(v.value)


def moe_route(x, gate_w, logit_bias, k, renorm, topk_ids, topk_w, ws, stream=None):
    T, H = x.shape
    E = gate_w.shape[0]
    st = _lib.moe_route(_ptr(x, "x", _bf16, (T, H)), _ptr(gate_w, "gate_w", _f32, (E, H)),
                        _ptr(logit_bias, "logit_bias", _f32, (E,), allow_none=True), T, H, E, k, int(bool(renorm)),
                        _ptr(topk_ids, "topk_ids", _i32, (T, k)), _ptr(topk_w, "topk_w", _f32, (T, k)),
                        _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_route", st)


def moe_route_grouped(x, gate_w, logit_bias, k, renorm, n_group, topk_group, topk_ids, topk_w, ws, stream=None):
    """Group-limited top-k routing: only experts of the topk_group best of n_group groups are eligible."""
    T, H = x.shape
    E = gate_w.shape[0]
    st = _lib.moe_route_grouped(_ptr(x, "x", _bf16, (T, H)), _ptr(gate_w, "gate_w", _f32, (E, H)),
                                _ptr(logit_bias, "logit_bias", _f32, (E,), allow_none=True), T, H, E, k,
                                int(bool(renorm)), int(n_group), int(topk_group),
                                _ptr(topk_ids, "topk_ids", _i32, (T, k)), _ptr(topk_w, "topk_w", _f32, (T, k)),
                                _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_route_grouped", st)


def moe_route_noalloc(x, gate_w, logit_bias, k, renorm, topk_ids, topk_w, stream=None):
    """moe_route without a workspace: scratch in the library's own fixed 16 MiB device array."""
    T, H = x.shape
    E = gate_w.shape[0]
    st = _lib.moe_route_noalloc(_ptr(x, "x", _bf16, (T, H)), _ptr(gate_w, "gate_w", _f32, (E, H)),
                                _ptr(logit_bias, "logit_bias", _f32, (E,), allow_none=True), T, H, E, k,
                                int(bool(renorm)), _ptr(topk_ids, "topk_ids", _i32, (T, k)),
                                _ptr(topk_w, "topk_w", _f32, (T, k)), _stream(stream))
    _check("moe_route_noalloc", st)


def moe_permute(topk_ids, topk_w, E, rep_offset, rep_slots, S, local_start, local_count, nonlocal_mode, x,
                slot_ids, counts, offsets, perm_src, pair_row, x_perm, ws, stream=None, on_input=False):
    """moe_permute, or moe_permute_on_input when on_input (rows scaled by the routing weights).
    x_perm=None (not with on_input): only the routing tables are written, no rows copied."""
    T, k = topk_ids.shape
    H = x.shape[1]
    S_local = local_count if local_count >= 0 else S
    fn = _lib.moe_permute_on_input if on_input else _lib.moe_permute
    st = fn(_ptr(topk_ids, "topk_ids", _i32, (T, k)), _ptr(topk_w, "topk_w", _f32, (T, k)), T, k, E,
                          _ptr(rep_offset, "rep_offset", _i32, (E + 1,), allow_none=True),
                          _ptr(rep_slots, "rep_slots", _i32, (S,), allow_none=True), S, local_start, local_count,
                          nonlocal_mode, _ptr(x, "x", _bf16, (T, H)), H,
                          _ptr(slot_ids, "slot_ids", _i32, (T, k)), _ptr(counts, "counts", _i32, (S_local,)),
                          _ptr(offsets, "offsets", _i32, (S_local + 1,)), _ptr(perm_src, "perm_src", _i32, (T * k,)),
                          _ptr(pair_row, "pair_row", _i32, (T, k)),
                          _ptr(x_perm, "x_perm", _bf16, (T * k, H), allow_none=True),
                          _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_permute_on_input" if on_input else "moe_permute", st)


def moe_forward(x_perm, offsets, W1, W2, pair_row, topk_w, x, W1s, W2s, shared_gate_w, out, ws, stream=None):
    P_cap, H = x_perm.shape
    S_local = offsets.shape[0] - 1
    I = W2.shape[2]
    T, k = pair_row.shape
    I_sh = 0 if W2s is None else W2s.shape[1]
    st = _lib.moe_forward(_ptr(x_perm, "x_perm", _bf16), _ptr(offsets, "offsets", _i32), S_local, P_cap,
                          _ptr(W1, "W1", _bf16, (S_local, 2 * I, H)), _ptr(W2, "W2", _bf16, (S_local, H, I)), H, I,
                          _ptr(pair_row, "pair_row", _i32), _ptr(topk_w, "topk_w", _f32, (T, k), allow_none=True),
                          T, k,
                          _ptr(x, "x", _bf16, (T, H), allow_none=True),
                          _ptr(W1s, "W1s", _bf16, (2 * I_sh, H), allow_none=True),
                          _ptr(W2s, "W2s", _bf16, (H, I_sh), allow_none=True), I_sh,
                          _ptr(shared_gate_w, "shared_gate_w", _bf16, (H,), allow_none=True),
                          _ptr(out, "out", _bf16, (T, H)), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_forward", st)



def moe_forward_fp8(x_perm, offsets, W1q, s1, W2q, s2, pair_row, topk_w, x, W1sq, s1s, W2sq, s2s, shared_gate_w,
                    out, ws, stream=None):
    """moe_forward with E4M3 weights (uint8 tensors) and fp32 row scales (moe_quantize_fp8_rows)."""
    _forward_q("moe_forward_fp8", x_perm, offsets, W1q, s1, W2q, s2, pair_row, topk_w, x, W1sq, s1s, W2sq, s2s,
               shared_gate_w, out, ws, stream)


def moe_forward_w8a8(x_perm, offsets, W1q, s1, W2q, s2, pair_row, topk_w, x, W1sq, s1s, W2sq, s2s, shared_gate_w,
                     out, ws, stream=None):
    """moe_forward_fp8 with the activations quantised to E4M3 per row as well (moe_quantize_act_rows)."""
    _forward_q("moe_forward_w8a8", x_perm, offsets, W1q, s1, W2q, s2, pair_row, topk_w, x, W1sq, s1s, W2sq, s2s,
               shared_gate_w, out, ws, stream)


def _forward_q(fn, x_perm, offsets, W1q, s1, W2q, s2, pair_row, topk_w, x, W1sq, s1s, W2sq, s2s, shared_gate_w,
               out, ws, stream):
    S_local = offsets.shape[0] - 1
    I = W2q.shape[2]
    T, k = pair_row.shape
    P_cap, H = x_perm.shape if x_perm is not None else (T * k, x.shape[1])
    I_sh = 0 if W2sq is None else W2sq.shape[1]
    u8 = torch.uint8
    st = getattr(_lib, fn)(_ptr(x_perm, "x_perm", _bf16, allow_none=True), _ptr(offsets, "offsets", _i32), S_local,
                           P_cap,
                              _ptr(W1q, "W1q", u8, (S_local, 2 * I, H)), _ptr(s1, "W1_scale", _f32, (S_local, 2 * I)),
                              _ptr(W2q, "W2q", u8, (S_local, H, I)), _ptr(s2, "W2_scale", _f32, (S_local, H)), H, I,
                              _ptr(pair_row, "pair_row", _i32), _ptr(topk_w, "topk_w", _f32, (T, k), allow_none=True),
                              T, k, _ptr(x, "x", _bf16, (T, H), allow_none=True),
                              _ptr(W1sq, "W1sq", u8, (2 * I_sh, H), allow_none=True),
                              _ptr(s1s, "W1s_scale", _f32, (2 * I_sh,), allow_none=True),
                              _ptr(W2sq, "W2sq", u8, (H, I_sh), allow_none=True),
                              _ptr(s2s, "W2s_scale", _f32, (H,), allow_none=True), I_sh,
                              _ptr(shared_gate_w, "shared_gate_w", _bf16, (H,), allow_none=True),
                              _ptr(out, "out", _bf16, (T, H)), _ptr(ws, "ws", torch.uint8), ws.numel(),
                              _stream(stream))
    _check(fn, st)


def moe_grouped_fc1_fp8(a, offsets, W1q, s1, a_shared, W1sq, s1s, h, h_shared, ws, stream=None):
    rows_cap, H = a.shape
    G = offsets.shape[0] - 1
    I = W1q.shape[1] // 2
    T = 0 if a_shared is None else a_shared.shape[0]
    I_sh = 0 if W1sq is None else W1sq.shape[0] // 2
    u8 = torch.uint8
    st = _lib.moe_grouped_fc1_fp8(_ptr(a, "a", _bf16), rows_cap, _ptr(offsets, "offsets", _i32), G,
                                  _ptr(W1q, "W1q", u8, (G, 2 * I, H)), _ptr(s1, "W1_scale", _f32, (G, 2 * I)), H, I,
                                  _ptr(a_shared, "a_shared", _bf16, (T, H), allow_none=True), T,
                                  _ptr(W1sq, "W1sq", u8, (2 * I_sh, H), allow_none=True),
                                  _ptr(s1s, "W1s_scale", _f32, (2 * I_sh,), allow_none=True), I_sh,
                                  _ptr(h, "h", _bf16, (rows_cap, I)),
                                  _ptr(h_shared, "h_shared", _bf16, (T, I_sh), allow_none=True),
                                  _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc1_fp8", st)


def moe_grouped_fc2_fp8(h, offsets, W2q, s2, h_shared, W2sq, s2s, y, y_shared, ws, stream=None):
    rows_cap, I = h.shape
    G = offsets.shape[0] - 1
    H = W2q.shape[1]
    T = 0 if h_shared is None else h_shared.shape[0]
    I_sh = 0 if W2sq is None else W2sq.shape[1]
    u8 = torch.uint8
    st = _lib.moe_grouped_fc2_fp8(_ptr(h, "h", _bf16), rows_cap, _ptr(offsets, "offsets", _i32), G,
                                  _ptr(W2q, "W2q", u8, (G, H, I)), _ptr(s2, "W2_scale", _f32, (G, H)), H, I,
                                  _ptr(h_shared, "h_shared", _bf16, (T, I_sh), allow_none=True), T,
                                  _ptr(W2sq, "W2sq", u8, (H, I_sh), allow_none=True),
                                  _ptr(s2s, "W2s_scale", _f32, (H,), allow_none=True), I_sh,
                                  _ptr(y, "y", _bf16, (rows_cap, H)),
                                  _ptr(y_shared, "y_shared", _bf16, (T, H), allow_none=True),
                                  _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc2_fp8", st)


def moe_grouped_fc1_w8a8(aq, a_scale, offsets, W1q, s1, a_shared_q, a_shared_scale, W1sq, s1s, h, h_shared, ws,
                         stream=None):
    """FC1 + SwiGLU on E4M3 activation rows (with their scales) and E4M3 weights."""
    rows_cap, H = aq.shape
    G = offsets.shape[0] - 1
    I = W1q.shape[1] // 2
    T = 0 if a_shared_q is None else a_shared_q.shape[0]
    I_sh = 0 if W1sq is None else W1sq.shape[0] // 2
    u8 = torch.uint8
    st = _lib.moe_grouped_fc1_w8a8(_ptr(aq, "aq", u8), _ptr(a_scale, "a_scale", _f32, (rows_cap,)), rows_cap,
                                   _ptr(offsets, "offsets", _i32), G,
                                   _ptr(W1q, "W1q", u8, (G, 2 * I, H)), _ptr(s1, "W1_scale", _f32, (G, 2 * I)), H, I,
                                   _ptr(a_shared_q, "a_shared_q", u8, (T, H), allow_none=True),
                                   _ptr(a_shared_scale, "a_shared_scale", _f32, (T,), allow_none=True), T,
                                   _ptr(W1sq, "W1sq", u8, (2 * I_sh, H), allow_none=True),
                                   _ptr(s1s, "W1s_scale", _f32, (2 * I_sh,), allow_none=True), I_sh,
                                   _ptr(h, "h", _bf16, (rows_cap, I)),
                                   _ptr(h_shared, "h_shared", _bf16, (T, I_sh), allow_none=True),
                                   _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc1_w8a8", st)


def moe_grouped_fc2_w8a8(hq, h_scale, offsets, W2q, s2, h_shared_q, h_shared_scale, W2sq, s2s, y, y_shared, ws,
                         stream=None):
    """FC2 on E4M3 intermediate rows (with their scales) and E4M3 weights."""
    rows_cap, I = hq.shape
    G = offsets.shape[0] - 1
    H = W2q.shape[1]
    T = 0 if h_shared_q is None else h_shared_q.shape[0]
    I_sh = 0 if W2sq is None else W2sq.shape[1]
    u8 = torch.uint8
    st = _lib.moe_grouped_fc2_w8a8(_ptr(hq, "hq", u8), _ptr(h_scale, "h_scale", _f32, (rows_cap,)), rows_cap,
                                   _ptr(offsets, "offsets", _i32), G,
                                   _ptr(W2q, "W2q", u8, (G, H, I)), _ptr(s2, "W2_scale", _f32, (G, H)), H, I,
                                   _ptr(h_shared_q, "h_shared_q", u8, (T, I_sh), allow_none=True),
                                   _ptr(h_shared_scale, "h_shared_scale", _f32, (T,), allow_none=True), T,
                                   _ptr(W2sq, "W2sq", u8, (H, I_sh), allow_none=True),
                                   _ptr(s2s, "W2s_scale", _f32, (H,), allow_none=True), I_sh,
                                   _ptr(y, "y", _bf16, (rows_cap, H)),
                                   _ptr(y_shared, "y_shared", _bf16, (T, H), allow_none=True),
                                   _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc2_w8a8", st)


def moe_quantize_act_rows(v, q, scale, stream=None):
    """Row-wise E4M3 quantisation of activations [..., K] bf16 with power-of-two scales into q (uint8, same
    shape) and scale ([...] fp32)."""
    K = v.shape[-1]
    rows = v.numel() // K
    st = _lib.moe_quantize_act_rows(_ptr(v, "v", _bf16), rows, K, _ptr(q, "q", torch.uint8, tuple(v.shape)),
                                    _ptr(scale, "scale", _f32, tuple(v.shape[:-1])), _stream(stream))
    _check("moe_quantize_act_rows", st)


def nvfp4_sf_row_bytes(K: int) -> int:
    """Bytes of one row of NVFP4 block scales of K elements (MOE_NVFP4_SF_ROW_BYTES)."""
    return 16 * ((K + 255) // 256)


def moe_quantize_nvfp4_rows(v, q, sb, scale, pow2=False, stream=None):
    """NVFP4 quantisation of a bf16 tensor [..., K]: q [..., K/2] uint8 (packed E2M1 codes), sb
    [..., nvfp4_sf_row_bytes(K)] uint8 (E4M3 block scales, zero-padded), scale [...] fp32 row scales
    (amax / 2688, or powers of two with pow2)."""
    K = v.shape[-1]
    rows = v.numel() // K
    lead = tuple(v.shape[:-1])
    st = _lib.moe_quantize_nvfp4_rows(_ptr(v, "v", _bf16), rows, K, int(bool(pow2)),
                                      _ptr(q, "q", torch.uint8, lead + (K // 2,)),
                                      _ptr(sb, "sb", torch.uint8, lead + (nvfp4_sf_row_bytes(K),)),
                                      _ptr(scale, "scale", _f32, lead), _stream(stream))
    _check("moe_quantize_nvfp4_rows", st)


def moe_forward_nvfp4(x_perm, offsets, W1q, W1sf, s1, W2q, W2sf, s2, pair_row, topk_w, x, W1sq, W1ssf, s1s,
                      W2sq, W2ssf, s2s, shared_gate_w, out, ws, stream=None):
    """moe_forward with NVFP4 weights (moe_quantize_nvfp4_rows, pow2=False) and NVFP4 activations.
    With topk_w and x given, each token row of x is quantised once for its pairs' rows and
    x_perm is not read (it may be None)."""
    S_local = offsets.shape[0] - 1
    I = 2 * W2q.shape[2]
    T, k = pair_row.shape
    P_cap, H = x_perm.shape if x_perm is not None else (T * k, x.shape[1])
    I_sh = 0 if W2sq is None else 2 * W2sq.shape[1]
    u8 = torch.uint8
    fh, fi, fs = nvfp4_sf_row_bytes(H), nvfp4_sf_row_bytes(I), nvfp4_sf_row_bytes(I_sh) if I_sh else 0
    st = _lib.moe_forward_nvfp4(
        _ptr(x_perm, "x_perm", _bf16, allow_none=True), _ptr(offsets, "offsets", _i32), S_local, P_cap,
        _ptr(W1q, "W1q", u8, (S_local, 2 * I, H // 2)), _ptr(W1sf, "W1_sf", u8, (S_local, 2 * I, fh)),
        _ptr(s1, "W1_scale", _f32, (S_local, 2 * I)),
        _ptr(W2q, "W2q", u8, (S_local, H, I // 2)), _ptr(W2sf, "W2_sf", u8, (S_local, H, fi)),
        _ptr(s2, "W2_scale", _f32, (S_local, H)), H, I,
        _ptr(pair_row, "pair_row", _i32), _ptr(topk_w, "topk_w", _f32, (T, k), allow_none=True), T, k,
        _ptr(x, "x", _bf16, (T, H), allow_none=True),
        _ptr(W1sq, "W1sq", u8, (2 * I_sh, H // 2), allow_none=True),
        _ptr(W1ssf, "W1s_sf", u8, (2 * I_sh, fh), allow_none=True),
        _ptr(s1s, "W1s_scale", _f32, (2 * I_sh,), allow_none=True),
        _ptr(W2sq, "W2sq", u8, (H, I_sh // 2), allow_none=True),
        _ptr(W2ssf, "W2s_sf", u8, (H, fs), allow_none=True),
        _ptr(s2s, "W2s_scale", _f32, (H,), allow_none=True), I_sh,
        _ptr(shared_gate_w, "shared_gate_w", _bf16, (H,), allow_none=True),
        _ptr(out, "out", _bf16, (T, H)), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_forward_nvfp4", st)


def moe_quantize_fp8_rows(w, q, scale, stream=None):
    """Row-wise E4M3 quantisation of a bf16 tensor [..., K] into q (uint8, same shape) and scale ([...] fp32)."""
    K = w.shape[-1]
    rows = w.numel() // K
    st = _lib.moe_quantize_fp8_rows(_ptr(w, "w", _bf16), rows, K, _ptr(q, "q", torch.uint8, tuple(w.shape)),
                                    _ptr(scale, "scale", _f32, tuple(w.shape[:-1])), _stream(stream))
    _check("moe_quantize_fp8_rows", st)

def moe_grouped_fc1(a, offsets, W1, a_shared, W1s, h, h_shared, ws, stream=None):
    rows_cap, H = a.shape
    G = offsets.shape[0] - 1
    I = W1.shape[1] // 2
    T = 0 if a_shared is None else a_shared.shape[0]
    I_sh = 0 if W1s is None else W1s.shape[0] // 2
    st = _lib.moe_grouped_fc1(_ptr(a, "a", _bf16), rows_cap, _ptr(offsets, "offsets", _i32), G,
                              _ptr(W1, "W1", _bf16, (G, 2 * I, H)), H, I,
                              _ptr(a_shared, "a_shared", _bf16, (T, H), allow_none=True), T,
                              _ptr(W1s, "W1s", _bf16, (2 * I_sh, H), allow_none=True), I_sh,
                              _ptr(h, "h", _bf16, (rows_cap, I)),
                              _ptr(h_shared, "h_shared", _bf16, (T, I_sh), allow_none=True),
                              _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc1", st)


def moe_grouped_fc2(h, offsets, W2, h_shared, W2s, y, y_shared, ws, stream=None):
    rows_cap, I = h.shape
    G = offsets.shape[0] - 1
    H = W2.shape[1]
    T = 0 if h_shared is None else h_shared.shape[0]
    I_sh = 0 if W2s is None else W2s.shape[1]
    st = _lib.moe_grouped_fc2(_ptr(h, "h", _bf16), rows_cap, _ptr(offsets, "offsets", _i32), G,
                              _ptr(W2, "W2", _bf16, (G, H, I)), H, I,
                              _ptr(h_shared, "h_shared", _bf16, (T, I_sh), allow_none=True), T,
                              _ptr(W2s, "W2s", _bf16, (H, I_sh), allow_none=True), I_sh,
                              _ptr(y, "y", _bf16, (rows_cap, H)),
                              _ptr(y_shared, "y_shared", _bf16, (T, H), allow_none=True),
                              _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc2", st)


def moe_finalize(y, pair_row, topk_w, y_shared, x, shared_gate_w, out, ws, stream=None):
    rows_cap, H = y.shape
    T, k = pair_row.shape
    st = _lib.moe_finalize(_ptr(y, "y", _bf16), rows_cap, _ptr(pair_row, "pair_row", _i32, (T, k)),
                           _ptr(topk_w, "topk_w", _f32, (T, k), allow_none=True), T, k, H,
                           _ptr(y_shared, "y_shared", _bf16, (T, H), allow_none=True),
                           _ptr(x, "x", _bf16, (T, H), allow_none=True),
                           _ptr(shared_gate_w, "shared_gate_w", _bf16, (H,), allow_none=True),
                           _ptr(out, "out", _bf16, (T, H)), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_finalize", st)


def moe_a2a_regroup(recv_counts, src, dst, direction, offsets, ws, stream=None, row_map=None):
    """Rows of an all-to-all expert-parallel rank from exchange order to GEMM order
    (direction MOE_A2A_TO_GEMM, offsets [S_local+1] written unless None) or back
    (MOE_A2A_TO_EXCHANGE).  recv_counts [N, S_local] int32; src, dst [rows_cap, H] bf16;
    row_map [rows_cap] int32 (or None): the src row of each dst row."""
    N, S_l = recv_counts.shape
    rows_cap, H = src.shape
    st = _lib.moe_a2a_regroup(_ptr(recv_counts, "recv_counts", _i32, (N, S_l)), N, S_l, _ptr(src, "src", _bf16),
                              _ptr(dst, "dst", _bf16, (rows_cap, H)), rows_cap, H, int(direction),
                              _ptr(offsets, "offsets", _i32, (S_l + 1,), allow_none=True),
                              _ptr(row_map, "row_map", _i32, (rows_cap,), allow_none=True),
                              _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_a2a_regroup", st)


def moe_grouped_fc2_scatter(h, offsets, W2, h_shared, W2s, y_row, y, y_shared, ws, stream=None):
    """moe_grouped_fc2 with routed output row r stored at y row y_row[r]."""
    rows_cap, I = h.shape
    G = offsets.shape[0] - 1
    H = W2.shape[1]
    T = 0 if h_shared is None else h_shared.shape[0]
    I_sh = 0 if W2s is None else W2s.shape[1]
    st = _lib.moe_grouped_fc2_scatter(_ptr(h, "h", _bf16), rows_cap, _ptr(offsets, "offsets", _i32), G,
                                      _ptr(W2, "W2", _bf16, (G, H, I)), H, I,
                                      _ptr(h_shared, "h_shared", _bf16, (T, I_sh), allow_none=True), T,
                                      _ptr(W2s, "W2s", _bf16, (H, I_sh), allow_none=True), I_sh,
                                      _ptr(y_row, "y_row", _i32, (rows_cap,)), _ptr(y, "y", _bf16, (rows_cap, H)),
                                      _ptr(y_shared, "y_shared", _bf16, (T, H), allow_none=True),
                                      _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_grouped_fc2_scatter", st)


def _ptr_array(ptrs, name):
    """A host array of device addresses: ints (e.g. peer-mapped addresses) or CUDA tensors."""
    vals = []
    for i, p in enumerate(ptrs):
        if isinstance(p, torch.Tensor):
            if not p.is_cuda or not p.is_contiguous():
                raise ValueError(f"{name}[{i}] must be a contiguous CUDA tensor")
            p = p.data_ptr()
        vals.append(int(p))
    return (ctypes.c_void_p * len(vals))(*vals)


def moe_ep_signal(peer_flags, rank, epoch, stream=None):
    """Raise this rank's flag to `epoch` in every rank's flag array (peer_flags[n]: the
    address on this GPU of rank n's int32 flags)."""
    arr = _ptr_array(peer_flags, "peer_flags")
    _check("moe_ep_signal", _lib.moe_ep_signal(arr, len(peer_flags), int(rank), int(epoch), _stream(stream)))


def moe_ep_reduce(partials, flags, epoch, row0, row1, out, ws, stream=None):
    """out rows [row0, row1) = bf16 of the rank-order fp32 sum of the ranks' bf16 partials
    [T, H] (addresses or tensors), once flags (this rank's [N] int32) all reach epoch."""
    N = len(partials)
    T, H = out.shape
    if not 0 <= row0 <= row1 <= T:
        raise ValueError(f"rows [{row0}, {row1}) outside [0, {T})")
    arr = _ptr_array(partials, "partials")
    st = _lib.moe_ep_reduce(arr, N, _ptr(flags, "flags", _i32, (N,)), int(epoch), int(row0), int(row1), H,
                            _ptr(out, "out", _bf16), _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check("moe_ep_reduce", st)


def moe_ipc_export(t: torch.Tensor):
    """(handle bytes, offset) that let another process map the CUDA tensor t's memory."""
    buf = ctypes.create_string_buffer(MOE_IPC_HANDLE_BYTES)
    off = ctypes.c_int64(0)
    _check("moe_ipc_export", _lib.moe_ipc_export(_ptr(t, "t"), buf, ctypes.byref(off)))
    return bytes(buf.raw), int(off.value)


def moe_ipc_import(handle: bytes, offset: int) -> int:
    """Map another process's exported memory here; returns the address of its tensor."""
    if len(handle) != MOE_IPC_HANDLE_BYTES:
        raise ValueError("bad IPC handle")
    p = ctypes.c_void_p(0)
    _check("moe_ipc_import", _lib.moe_ipc_import(handle, int(offset), ctypes.byref(p)))
    return int(p.value)


def moe_ipc_close(addr: int, offset: int) -> None:
    _check("moe_ipc_close", _lib.moe_ipc_close(ctypes.c_void_p(int(addr)), int(offset)))


def moe_debug_wait_timeout(ws, timeout_ns, stream=None):
    _check("moe_debug_wait_timeout",
           _lib.moe_debug_wait_timeout(_ptr(ws, "ws", torch.uint8), ws.numel(), int(timeout_ns), _stream(stream)))


def moe_set_wait_timeout_ns(timeout_ns: int) -> None:
    _lib.moe_set_wait_timeout_ns(int(timeout_ns))


def moe_set_pdl(enable: bool) -> None:
    """Launch kernels with programmatic dependent launch (default) or in plain stream order."""
    _check("moe_set_pdl", _lib.moe_set_pdl(int(bool(enable))))


def moe_get_launch_count() -> int:
    """Kernel launches the library has issued in this process (counted on the host)."""
    return int(_lib.moe_get_launch_count())


_armed_events: list = []


def moe_launch_events_arm(events) -> None:
    """Arm the per-launch timing hook with torch.cuda.Event objects created with
    enable_timing=True; each must have been recorded once (torch creates the CUDA
    event on first record).  While armed, every library launch first records the
    next event on its stream.  None or an empty list disarms."""
    global _armed_events
    evs = list(events or [])
    handles = []
    for e in evs:
        h = int(e.cuda_event)
        if not h:
            raise ValueError("record each event once before arming it (its CUDA event is created on first record)")
        handles.append(h)
    arr = (ctypes.c_void_p * len(handles))(*handles) if handles else None
    _check("moe_launch_events_arm", _lib.moe_launch_events_arm(arr, len(handles)))
    _armed_events = evs  # the events must outlive their use by the library


def moe_launch_events_mark(stream=None) -> None:
    """Record the next armed event on `stream` now (closes the last launch's interval)."""
    _check("moe_launch_events_mark", _lib.moe_launch_events_mark(_stream(stream)))


def moe_launch_events_used() -> list:
    """Labels of the events recorded since arming: kernel names, and "mark" for marks."""
    n = int(_lib.moe_launch_events_used(None, 0))
    w = MOE_LAUNCH_LABEL_BYTES
    buf = ctypes.create_string_buffer(w * max(1, n))
    _lib.moe_launch_events_used(buf, n)
    return [buf.raw[w * i:w * (i + 1)].split(b"\0", 1)[0].decode() for i in range(n)]


def moe_set_gemm_pair_mode(mode: int) -> None:
    """0: one CTA per tile (default); 1: 2-SM CTA pairs for large launches; 2: pairs whenever possible."""
    _check("moe_set_gemm_pair_mode", _lib.moe_set_gemm_pair_mode(int(mode)))
