"""fp64 CPU oracle for the MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The CUDA library never imports, links or
calls it, and the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, per-token loops); this
module compiles it with gcc (``build()``) and marshals numpy arrays through
ctypes.  Each wrapper names the C function it calls; the C file cites the
passage of the source pages each step follows.

Parity status of each function (see tests/test_oracle_pins.py for the pins):
  route, slot_map, local_mask, permute, expert_mlp, moe_tokens, bf16 rounding,
  the E4M3 and NVFP4 quantisers and expert MLPs, a2a_regroup: pinned (closed
  forms, brute force, invariants, hand-worked examples, independent
  numpy/torch routines).  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")

NONLOCAL_SKIP = 0
NONLOCAL_MOD = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_route.argtypes = [P, P, P, i64, i32, i32, i32, i32, P, P, P]
        lib.oracle_route.restype = None
        lib.oracle_route_grouped.argtypes = [P, P, P, i64, i32, i32, i32, i32, i32, i32, P, P, P]
        lib.oracle_route_grouped.restype = None
        lib.oracle_slot_map.argtypes = [P, i64, i32, P, P, P]
        lib.oracle_slot_map.restype = None
        lib.oracle_local_mask.argtypes = [P, P, i64, i32, i32, i32, P, P, P]
        lib.oracle_local_mask.restype = None
        lib.oracle_permute.argtypes = [P, i64, i32, P, P, P, P]
        lib.oracle_permute.restype = None
        lib.oracle_expert_mlp.argtypes = [P, P, P, i32, i32, P, P]
        lib.oracle_expert_mlp.restype = None
        lib.oracle_moe_tokens.argtypes = [P, i64, i32, P, P, i32, i32, i32, i32, i32, i32, P, P, i32, i32, i32,
                                          P, P, i32, i32, P, P, i32, P, P, P, P, P, P, P, P, P,
                                          P, P, P, P, i32, P, i64, P, P, P, P]
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_quantize_fp8_rows.argtypes = [P, i64, i32, P, P]
        lib.oracle_quantize_fp8_rows.restype = None
        lib.oracle_expert_mlp_fp8.argtypes = [P, P, P, P, P, i32, i32, P, P]
        lib.oracle_expert_mlp_fp8.restype = None
        lib.oracle_expert_mlp_w8a8.argtypes = [P, P, P, P, P, i32, i32, P, P]
        lib.oracle_expert_mlp_w8a8.restype = None
        lib.oracle_quantize_act_rows.argtypes = [P, i64, i32, P, P]
        lib.oracle_quantize_act_rows.restype = None
        lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_e2m1.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_e2m1.restype = ctypes.c_uint8
        lib.oracle_quantize_nvfp4_rows.argtypes = [P, i64, i32, i32, P, P, P]
        lib.oracle_quantize_nvfp4_rows.restype = None
        lib.oracle_expert_mlp_nvfp4.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, P, P]
        lib.oracle_expert_mlp_nvfp4.restype = None
        lib.oracle_moe_tokens.restype = None
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_set_threads.restype = None
        lib.oracle_get_threads.argtypes = []
        lib.oracle_get_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 numpy array (accepts a torch bf16 tensor)."""
    if a is None:
        return None
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def _np(a, dtype):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def bf16_to_f64(b: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(b)))


def f64_to_bf16(v: float) -> int:
    """Round to nearest bf16, ties to even; returns the bf16 bit pattern."""
    return int(_load().oracle_f64_to_bf16(float(v)))


def route(x, Wg, bias, k: int, renorm: bool, n_group: int = 1, topk_group: int = 1):
    """C oracle_route (n_group <= 1) or oracle_route_grouped (group-limited top-k):
    returns (ids [T,k] int32, w [T,k] float64, logits [T,E] float64)."""
    lib = _load()
    x = _u16(x)
    Wg = _np(Wg, np.float32)
    bias = _np(bias, np.float32)
    T, H = x.shape
    E = Wg.shape[0]
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float64)
    if n_group > 1:
        lib.oracle_route_grouped(_ptr(x), _ptr(Wg), _ptr(bias), T, H, E, k, int(bool(renorm)), n_group, topk_group,
                                 _ptr(ids), _ptr(w), _ptr(logits))
    else:
        lib.oracle_route(_ptr(x), _ptr(Wg), _ptr(bias), T, H, E, k, int(bool(renorm)),
                         _ptr(ids), _ptr(w), _ptr(logits))
    return ids, w, logits


def slot_map(ids, rep_offset=None, rep_slots=None):
    """C oracle_slot_map: expert id -> expert slot (identity when rep_offset is None)."""
    lib = _load()
    ids = _np(ids, np.int32)
    T, k = ids.shape
    ro = _np(rep_offset, np.int32)
    rs = _np(rep_slots, np.int32)
    out = np.empty((T, k), np.int32)
    lib.oracle_slot_map(_ptr(ids), T, k, _ptr(ro), _ptr(rs), _ptr(out))
    return out


def local_mask(slots, w, start: int, count: int, mode: int = NONLOCAL_SKIP):
    """C oracle_local_mask: returns (slots_out, w_out, mask) with the input's shape."""
    lib = _load()
    slots = _np(slots, np.int32)
    w = _np(w, np.float64)
    shape = slots.shape
    P = slots.size
    so = np.empty(shape, np.int32)
    wo = np.empty(shape, np.float64)
    m = np.empty(shape, np.uint8)
    lib.oracle_local_mask(_ptr(slots), _ptr(w), P, start, count, mode, _ptr(so), _ptr(wo), _ptr(m))
    return so, wo, m.astype(bool)


def permute(slots, S: int):
    """C oracle_permute: returns (counts [S], offsets [S+1], perm_src [total], pair_row [P])."""
    lib = _load()
    slots = _np(slots, np.int32).reshape(-1)
    P = slots.size
    counts = np.empty(S, np.int32)
    offsets = np.empty(S + 1, np.int32)
    perm_src = np.full(max(P, 1), -1, np.int32)
    pair_row = np.empty(max(P, 1), np.int32)
    lib.oracle_permute(_ptr(slots), P, S, _ptr(counts), _ptr(offsets), _ptr(perm_src), _ptr(pair_row))
    total = int(offsets[S])
    return counts, offsets, perm_src[:total].copy(), pair_row[:P].copy()


def a2a_regroup(recv_counts):
    """The GEMM order of the rows one rank receives in the all-to-all dispatch.

    recv_counts [N, S_local]: rows source rank n sent for local slot c.  The rows
    arrive source by source, each source's rows grouped by slot (the order of its
    own permutation), so exchange row q belongs to local slot c of the block (n, c)
    that holds it.  The experts take the rows grouped by slot, each slot's rows in
    arrival order: a stable grouping by slot -- oracle_permute with one pair per
    row.  Returns (offsets [S_local+1], gemm_row [R]: the GEMM-order row of each
    exchange-order row, exch_row [R]: the inverse)."""
    rc = np.asarray(recv_counts, dtype=np.int64)
    N, S_l = rc.shape
    if (rc < 0).any():
        raise ValueError("negative count")
    slot_of_row = [c for n in range(N) for c in range(S_l) for _ in range(int(rc[n, c]))]
    slots = np.asarray(slot_of_row, dtype=np.int32).reshape(-1, 1)
    counts, offsets, perm_src, pair_row = permute(slots, S_l)
    return offsets, pair_row, perm_src


def expert_mlp(x_row, W1, W2):
    """C oracle_expert_mlp: one token through one SwiGLU expert. Returns (y [H] f64, h [I] bf16 bits)."""
    lib = _load()
    x_row = _u16(x_row).reshape(-1)
    W1 = _u16(W1)
    W2 = _u16(W2)
    H = x_row.size
    I = W1.shape[0] // 2
    assert W1.shape == (2 * I, H) and W2.shape == (H, I)
    y = np.empty(H, np.float64)
    h = np.empty(I, np.uint16)
    lib.oracle_expert_mlp(_ptr(x_row), _ptr(W1), _ptr(W2), H, I, _ptr(y), _ptr(h))
    return y, h


def e4m3_to_f64(q: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(q)))


def f64_to_e4m3(v: float) -> int:
    """Nearest E4M3 value, ties to even, saturated at +-448; returns the byte."""
    return int(_load().oracle_f64_to_e4m3(float(v)))


def quantize_fp8_rows(w):
    """C oracle_quantize_fp8_rows on a bf16 matrix [..., K]: returns (q uint8 same shape,
    scale float32 [...]) with scale = amax/448 per row and q = e4m3(w / scale)."""
    lib = _load()
    w16 = _u16(w)
    shape = w16.shape
    K = shape[-1]
    rows = int(np.prod(shape[:-1]))
    q = np.empty(shape, np.uint8)
    sc = np.empty(shape[:-1], np.float32)
    lib.oracle_quantize_fp8_rows(_ptr(np.ascontiguousarray(w16)), rows, K, _ptr(q), _ptr(sc))
    return q, sc


def quantize_act_rows(v):
    """C oracle_quantize_act_rows on a bf16 matrix [..., K]: returns (q uint8 same shape,
    scale float32 [...]) with a power-of-two scale 2^e per row, e the smallest integer
    >= -126 with amax <= 448 * 2^e, and q = e4m3(v / 2^e)."""
    lib = _load()
    v16 = np.ascontiguousarray(_u16(v))
    shape = v16.shape
    K = shape[-1]
    rows = int(np.prod(shape[:-1]))
    q = np.empty(shape, np.uint8)
    sc = np.empty(shape[:-1], np.float32)
    lib.oracle_quantize_act_rows(_ptr(v16), rows, K, _ptr(q), _ptr(sc))
    return q, sc


def expert_mlp_fp8(x_row, W1q, s1, W2q, s2, act8=False):
    """C oracle_expert_mlp_fp8 (or, act8, oracle_expert_mlp_w8a8: x and h quantised to
    E4M3 per row too): one token through one SwiGLU expert with E4M3 weights."""
    lib = _load()
    x_row = _u16(x_row).reshape(-1)
    W1q, W2q = _np(W1q, np.uint8), _np(W2q, np.uint8)
    s1, s2 = _np(s1, np.float32), _np(s2, np.float32)
    H = x_row.size
    I = W1q.shape[0] // 2
    y = np.empty(H, np.float64)
    h = np.empty(I, np.uint16)
    fn = lib.oracle_expert_mlp_w8a8 if act8 else lib.oracle_expert_mlp_fp8
    fn(_ptr(x_row), _ptr(W1q), _ptr(s1), _ptr(W2q), _ptr(s2), H, I, _ptr(y), _ptr(h))
    return y, h


def e2m1_to_f64(q: int) -> float:
    return float(_load().oracle_e2m1_to_f64(int(q)))


def f64_to_e2m1(v: float) -> int:
    """Nearest E2M1 value, ties to even, saturated at +-6; returns the 4-bit code."""
    return int(_load().oracle_f64_to_e2m1(float(v)))


def quantize_nvfp4_rows(v, pow2=False):
    """C oracle_quantize_nvfp4_rows on a bf16 matrix [..., K] (K a multiple of 16):
    returns (q uint8 [..., K] E2M1 codes, sb uint8 [..., K/16] E4M3 block scales,
    s float32 [...] row scales), s = amax / 2688 (pow2, for activations: the
    smallest 2^e, e >= -126, with amax <= 2688 * 2^e), sb = e4m3(amax_b / (6 s)),
    q = e2m1(v / (sb s)); the value of an element is e2m1(q) * sb * s."""
    lib = _load()
    v16 = np.ascontiguousarray(_u16(v))
    shape = v16.shape
    K = shape[-1]
    assert K % 16 == 0, "NVFP4 rows hold whole 16-element blocks"
    rows = int(np.prod(shape[:-1]))
    q = np.empty(shape, np.uint8)
    sb = np.empty(shape[:-1] + (K // 16,), np.uint8)
    sc = np.empty(shape[:-1], np.float32)
    lib.oracle_quantize_nvfp4_rows(_ptr(v16), rows, K, int(bool(pow2)), _ptr(q), _ptr(sb), _ptr(sc))
    return q, sb, sc


def expert_mlp_nvfp4(x_row, W1q, W1sb, s1, W2q, W2sb, s2, act4=False):
    """C oracle_expert_mlp_nvfp4: one token through one SwiGLU expert with NVFP4
    weights (codes, block scales, row scales as quantize_nvfp4_rows returns them);
    act4: x and h quantised to NVFP4 per row as well (power-of-two row scales).  Returns (y [H] f64, h [I] bf16 bits)."""
    lib = _load()
    x_row = _u16(x_row).reshape(-1)
    W1q, W2q = _np(W1q, np.uint8), _np(W2q, np.uint8)
    W1sb, W2sb = _np(W1sb, np.uint8), _np(W2sb, np.uint8)
    s1, s2 = _np(s1, np.float32), _np(s2, np.float32)
    H = x_row.size
    I = W1q.shape[0] // 2
    assert W1q.shape == (2 * I, H) and W2q.shape == (H, I) and H % 16 == 0 and I % 16 == 0
    assert W1sb.shape == (2 * I, H // 16) and W2sb.shape == (H, I // 16)
    y = np.empty(H, np.float64)
    h = np.empty(I, np.uint16)
    lib.oracle_expert_mlp_nvfp4(_ptr(x_row), _ptr(W1q), _ptr(W1sb), _ptr(s1), _ptr(W2q), _ptr(W2sb), _ptr(s2),
                                H, I, int(bool(act4)), _ptr(y), _ptr(h))
    return y, h


def moe_tokens(x, Wg, bias, k, renorm, W1, W2, tokens=None, rep_offset=None, rep_slots=None,
               local_start=0, local_count=-1, mode=NONLOCAL_SKIP,
               W1s=None, W2s=None, shared_gate_w=None, n_group=1, topk_group=1, on_input=False, fp8=None,
               nvfp4=None):
    """C oracle_moe_tokens: full layer output (float64) for the listed tokens.

    n_group / topk_group: group-limited top-k (n_group <= 1: plain top-k).
    on_input: the routing weight scales each expert's input (rounded to bf16)
    and the expert outputs are summed unweighted.
    fp8: None, or a dict of E4M3 weights with row scales (W1q, s1, W2q, s2 and,
    with shared experts, W1sq, s1s, W2sq, s2s) used in place of W1/W2/W1s/W2s;
    with act8=True in it, the activations are quantised to E4M3 per row as well.
    nvfp4: None, or a dict of NVFP4 weights as quantize_nvfp4_rows returns them (W1q,
    W1sb, s1, W2q, W2sb, s2 and, with shared experts, W1sq, W1ssb, s1s, W2sq, W2ssb,
    s2s); with act4=True in it, the activations are quantised to NVFP4 per row as well.

    W1 [S_local, 2I, H], W2 [S_local, H, I] are indexed by local slot.
    W1s [n_shared, 2*I_sh, H] / W2s [n_shared, H, I_sh] (or None).
    Returns dict(out [n,H] f64, ids [n,k], w [n,k] f64 (after the mask), slots [n,k]).
    """
    lib = _load()
    x = _u16(x)
    T, H = x.shape
    Wg = _np(Wg, np.float32)
    bias = _np(bias, np.float32)
    E = Wg.shape[0]
    W1 = _u16(W1)
    W2 = _u16(W2)
    I = W1.shape[1] // 2
    if tokens is None:
        tokens = np.arange(T, dtype=np.int64)
    tokens = _np(tokens, np.int64).reshape(-1)
    n = tokens.size
    ro = _np(rep_offset, np.int32)
    rs = _np(rep_slots, np.int32)
    n_shared, I_sh = 0, 0
    if W1s is not None:
        W1s = _u16(W1s)
        W2s = _u16(W2s)
        n_shared = W1s.shape[0]
        I_sh = W1s.shape[1] // 2
    gw = _u16(shared_gate_w)
    out = np.empty((n, H), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    sl = np.empty((n, k), np.int32)
    assert fp8 is None or nvfp4 is None, "one weight format at a time"
    f = fp8 or nvfp4 or {}
    keys = ("W1q", "s1", "W2q", "s2", "W1sq", "s1s", "W2sq", "s2s", "W1sb", "W2sb", "W1ssb", "W2ssb")
    fq = {key: (_np(f[key], np.float32) if key.startswith("s") else _np(f[key], np.uint8))
          if f.get(key) is not None else None for key in keys}
    act = bool(f.get("act4", False)) if nvfp4 is not None else bool(f.get("act8", False))
    lib.oracle_moe_tokens(_ptr(x), T, H, _ptr(Wg), _ptr(bias), E, k, int(bool(renorm)),
                          int(n_group), int(topk_group), int(bool(on_input)),
                          _ptr(ro), _ptr(rs), local_start, local_count, mode,
                          _ptr(W1), _ptr(W2), I, n_shared, _ptr(W1s), _ptr(W2s), I_sh, _ptr(gw),
                          _ptr(fq["W1q"]), _ptr(fq["s1"]), _ptr(fq["W2q"]), _ptr(fq["s2"]),
                          _ptr(fq["W1sq"]), _ptr(fq["s1s"]), _ptr(fq["W2sq"]), _ptr(fq["s2s"]),
                          _ptr(fq["W1sb"]), _ptr(fq["W2sb"]), _ptr(fq["W1ssb"]), _ptr(fq["W2ssb"]),
                          int(act), _ptr(tokens), n, _ptr(out), _ptr(ids), _ptr(w), _ptr(sl))
    return dict(out=out, ids=ids, w=w, slots=sl)


def moe_layer(x, Wg, bias, k, renorm, W1, W2, rep_offset=None, rep_slots=None,
              local_start=0, local_count=-1, mode=NONLOCAL_SKIP,
              W1s=None, W2s=None, shared_gate_w=None, S=None, n_group=1, topk_group=1, on_input=False,
              fp8=None, nvfp4=None):
    """The whole layer on a batch: routing, slot map, mask, permutation and outputs.

    Composes the C steps in the order the layer runs them; returns a dict with
    ids, w (router weights), slots/w_masked (after slot map and mask), counts,
    offsets, perm_src, pair_row and out [T, H] (float64).
    """
    ids, w, logits = route(x, Wg, bias, k, renorm, n_group, topk_group)
    slots = slot_map(ids, rep_offset, rep_slots)
    if S is None:
        S = Wg.shape[0] if rep_offset is None else int(np.asarray(rep_offset)[-1])
    if local_count is not None and local_count >= 0:
        slots_l, w_l, mask = local_mask(slots, w, local_start, local_count, mode)
        S_local = local_count
    else:
        slots_l, w_l, mask = slots, w, np.ones_like(slots, dtype=bool)
        S_local = S
    counts, offsets, perm_src, pair_row = permute(slots_l, S_local)
    res = moe_tokens(x, Wg, bias, k, renorm, W1, W2, None, rep_offset, rep_slots,
                     local_start, local_count if local_count is not None else -1, mode,
                     W1s, W2s, shared_gate_w, n_group, topk_group, on_input, fp8, nvfp4)
    return dict(ids=ids, w=w, logits=logits, slots_global=slots, slots=slots_l, w_masked=w_l,
                mask=mask, counts=counts, offsets=offsets, perm_src=perm_src,
                pair_row=pair_row.reshape(ids.shape), out=res["out"])
