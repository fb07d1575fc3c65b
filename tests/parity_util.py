"""Helpers of the GPU parity tests: run the CUDA layer, run the oracle on the
same seeded inputs, and compare.

Bars (all written here, used by every parity test):
  * ids, slot ids, counts, offsets, perm_src, pair_row: bit-exact;
  * x_perm rows: bitwise copies of the source token rows;
  * routing weights: |w_gpu - w_oracle| <= rel_w(t) * w_oracle + 1e-7, where
    rel_w(t) = exp(2 B_t) - 1 + 64 u32 and B_t is the worst-case rounding
    error of one fp32 logit of token t (the router's certified bound
    gamma_n (||x_t|| max_e ||w_e|| + max_e |b_e|), n the logit's rounding
    depth): a softmax weight moves by at most a factor exp(+-2 B_t);
  * layer outputs: |gpu - oracle| <= 1e-2 * max|oracle| + 1e-3 elementwise.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import moe_inputs as mi
import oracle
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.layer import layer_from_inputs

U32 = 2.0 ** -24
U64 = 2.0 ** -53


def oracle_threads():
    oracle.set_threads(os.cpu_count() or 1)


def to_cpu(inp: dict) -> dict:
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def router_bound(x: torch.Tensor, Wg: torch.Tensor, bias, H: int) -> np.ndarray:
    """Upper bound B_t of |fp32 logit - exact logit| per token (any split plan)."""
    # deepest rounding chain the router can use: 32-term chunks, 8-chunk groups,
    # up to ceil(H/256) groups, up to 32 split partials, the bias
    n = 32 + 8 + math.ceil(H / 256) + 32 + 1
    g32 = n * U32 / (1 - n * U32)
    g64 = (H + 2) * U64 / (1 - (H + 2) * U64)
    xn = torch.linalg.vector_norm(x.double(), dim=1).numpy()
    wmax = float(torch.linalg.vector_norm(Wg.double(), dim=1).max())
    bmax = 0.0 if bias is None else float(bias.double().abs().max())
    return (g32 + g64) * (xn * wmax + bmax) * 1.01


def check_weights(w_gpu: np.ndarray, w_ref: np.ndarray, B: np.ndarray):
    rel = np.expm1(2.0 * B)[:, None] + 64 * U32
    err = np.abs(w_gpu.astype(np.float64) - w_ref)
    bad = err > rel * np.abs(w_ref) + 1e-7
    assert not bad.any(), f"routing weights off at {np.argwhere(bad)[:5]}: max rel err {(err / np.maximum(w_ref, 1e-30)).max()}"
    return float((err / np.maximum(np.abs(w_ref), 1e-30)).max())


def check_out(out_gpu: torch.Tensor, ref: np.ndarray, what="out"):
    g = out_gpu.float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    err = np.abs(g - ref)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    assert err.max() <= tol, f"{what}: max |gpu - oracle| = {err.max():.3e} > {tol:.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    return float(err.max()), tol


def run_gpu(inp: dict, local_start=0, local_count=-1, mode=0, layer=None, on_input=None):
    """Route, permute and forward on the GPU; returns CPU copies of every output."""
    if layer is None:
        layer = layer_from_inputs(inp, "cuda", local_start=local_start, local_count=local_count,
                                  nonlocal_mode=mode, on_input=on_input)
    x = inp["x"].cuda()
    out = layer.forward(x)
    torch.cuda.synchronize()
    T = x.shape[0]
    v = layer.views(T)
    rows = int(v["offsets"][-1])
    res = {k: t.cpu().clone() for k, t in v.items() if k not in ("x_perm", "out")}
    res["rows"] = rows
    res["out"] = out.cpu().clone()
    # None: the layer's experts read the token rows through pair_row and no rows were copied
    res["x_perm"] = None if layer.rows_from_tokens(T) else v["x_perm"][:rows]
    res["layer"] = layer
    return res


def permute_with_rows(layer, x):
    """Route and permute x through the layer with the rows copied into layer.x_perm (as
    moe_permute does for every layer whose experts read x_perm); returns the views."""
    v = layer.route(x)
    moe.moe_permute(v["topk_ids"], v["topk_w"], layer.E, layer.rep_offset, layer.rep_slots, layer.S,
                    layer.local_start, layer.local_count, layer.mode, x, v["slot_ids"], v["counts"], v["offsets"],
                    v["perm_src"], v["pair_row"], v["x_perm"], layer.ws)
    return v


def oracle_layer(inp_cpu: dict, local_start=0, local_count=-1, mode=0, tokens=None, on_input=None):
    cfg = inp_cpu["cfg"]
    if on_input is None:
        on_input = cfg.on_input
    W1, W2 = inp_cpu["W1"], inp_cpu["W2"]
    if local_count >= 0:
        W1 = W1[local_start:local_start + local_count]
        W2 = W2[local_start:local_start + local_count]
    W1s, W2s = inp_cpu["W1s"], inp_cpu["W2s"]
    fp8 = None
    if cfg.fp8:
        # the GPU runs the shared experts as one MLP (rows / columns concatenated), and row
        # scales depend on that layout: the oracle gets the same single MLP
        if W1s is not None:
            from moe_inputs import shared_concat
            c1, c2 = shared_concat(W1s, W2s)
            W1s, W2s = c1[None], c2[None]
        q1, s1 = oracle.quantize_fp8_rows(W1)
        q2, s2 = oracle.quantize_fp8_rows(W2)
        fp8 = dict(W1q=q1, s1=s1, W2q=q2, s2=s2, act8=cfg.act8)
        if W1s is not None:
            q1s, s1s = oracle.quantize_fp8_rows(W1s)
            q2s, s2s = oracle.quantize_fp8_rows(W2s)
            fp8.update(W1sq=q1s, s1s=s1s, W2sq=q2s, s2s=s2s)
    nvfp4 = None
    if cfg.fp4:
        nvfp4 = nvfp4_weights(W1, W2, W1s, W2s)
        if W1s is not None:
            from moe_inputs import shared_concat
            c1, c2 = shared_concat(W1s, W2s)
            W1s, W2s = c1[None], c2[None]
    kw = dict(rep_offset=inp_cpu["rep_offset"], rep_slots=inp_cpu["rep_slots"], local_start=local_start,
              local_count=local_count, mode=mode, W1s=W1s, W2s=W2s,
              shared_gate_w=inp_cpu["w_s"], n_group=cfg.n_group, topk_group=cfg.topk_group, on_input=on_input,
              fp8=fp8, nvfp4=nvfp4)
    if tokens is None:
        return oracle.moe_layer(inp_cpu["x"], inp_cpu["Wg"], inp_cpu["bias"], cfg.k, cfg.renorm, W1, W2,
                                S=cfg.slots, **kw)
    return oracle.moe_tokens(inp_cpu["x"], inp_cpu["Wg"], inp_cpu["bias"], cfg.k, cfg.renorm, W1, W2,
                             tokens=tokens, **kw)


def nvfp4_weights(W1, W2, W1s=None, W2s=None):
    """The oracle's NVFP4 quantisation of the expert weights (the shared experts as the one
    concatenated MLP the GPU runs: its row and block scales depend on that layout), with
    NVFP4 activations."""
    d = {}
    d["W1q"], d["W1sb"], d["s1"] = oracle.quantize_nvfp4_rows(W1)
    d["W2q"], d["W2sb"], d["s2"] = oracle.quantize_nvfp4_rows(W2)
    if W1s is not None:
        from moe_inputs import shared_concat
        c1, c2 = shared_concat(W1s, W2s)
        d["W1sq"], d["W1ssb"], d["s1s"] = oracle.quantize_nvfp4_rows(c1[None])
        d["W2sq"], d["W2ssb"], d["s2s"] = oracle.quantize_nvfp4_rows(c2[None])
    d["act4"] = True
    return d


def unpack_e2m1(q: np.ndarray) -> np.ndarray:
    """Packed E2M1 bytes [..., K/2] -> one code per element [..., K] (low nibble first)."""
    q = np.asarray(q, np.uint8)
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],), np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def oracle_routing(inp_cpu: dict, local_start=0, local_count=-1, mode=0):
    """Routing + slot map + mask + permutation of every token (no expert MLPs)."""
    cfg = inp_cpu["cfg"]
    ids, w, _ = oracle.route(inp_cpu["x"], inp_cpu["Wg"], inp_cpu["bias"], cfg.k, cfg.renorm, cfg.n_group,
                             cfg.topk_group)
    slots = oracle.slot_map(ids, inp_cpu["rep_offset"], inp_cpu["rep_slots"])
    if local_count >= 0:
        slots, w_m, _ = oracle.local_mask(slots, w, local_start, local_count, mode)
        S_local = local_count
    else:
        w_m, S_local = w, cfg.slots
    counts, offsets, perm_src, pair_row = oracle.permute(slots, S_local)
    return dict(ids=ids, w=w, w_masked=w_m, slots=slots, counts=counts, offsets=offsets, perm_src=perm_src,
                pair_row=pair_row.reshape(ids.shape))


def check_routing(g: dict, ref: dict, inp_cpu: dict, masked: bool):
    cfg = inp_cpu["cfg"]
    assert np.array_equal(g["topk_ids"].numpy(), ref["ids"]), "topk ids differ"
    assert np.array_equal(g["slot_ids"].numpy(), ref["slots"]), "slot ids differ"
    assert np.array_equal(g["counts"].numpy(), ref["counts"]), "counts differ"
    assert np.array_equal(g["offsets"].numpy(), ref["offsets"]), "offsets differ"
    assert g["rows"] == int(ref["offsets"][-1])
    assert np.array_equal(g["perm_src"].numpy()[:g["rows"]], ref["perm_src"]), "perm_src differs"
    assert np.array_equal(g["pair_row"].numpy(), ref["pair_row"]), "pair_row differs"
    B = router_bound(inp_cpu["x"], inp_cpu["Wg"], inp_cpu["bias"], cfg.H)
    return check_weights(g["topk_w"].numpy(), ref["w_masked"] if masked else ref["w"], B)


def check_x_perm(g: dict, x_dev: torch.Tensor, k: int):
    rows = g["rows"]
    if rows == 0 or g["x_perm"] is None:
        return
    src = g["perm_src"][:rows].to(torch.int64).cuda() // k
    want = x_dev.index_select(0, src)
    assert torch.equal(g["x_perm"].view(torch.int16), want.view(torch.int16)), "x_perm rows are not copies of x"


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    if T <= n:
        return np.arange(T, dtype=np.int64)
    g = np.random.default_rng(seed)
    s = set([0, T - 1])
    while len(s) < n:
        s.add(int(g.integers(0, T)))
    return np.array(sorted(s), dtype=np.int64)


def make(cfg_name_or_cfg, device="cpu", weights_device=None, **over):
    cfg = mi.CONFIGS[cfg_name_or_cfg] if isinstance(cfg_name_or_cfg, str) else cfg_name_or_cfg
    if over:
        cfg = cfg.with_(**over)
    return mi.make_inputs(cfg, device=device, weights_device=weights_device)
