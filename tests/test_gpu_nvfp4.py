"""GPU parity of the NVFP4 experts (E2M1 weights and activations, E4M3 scales per
16 elements, fp32 row scales; tcgen05.mma kind::mxf4nvf4) against the fp64 oracle.

The quantiser must reproduce the oracle's codes, block scales and row scales
bit for bit (weights with amax / 2688 row scales, activations with power-of-two
ones).  The layer runs every routing variant on NVFP4 experts and must match
the oracle's NVFP4 layer (which quantises the same activation rows) within the
output tolerance of tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import serving_router_gate_gb300 as moe
from serving_router_gate_gb300.layer import layer_from_inputs

from parity_util import (check_out, check_routing, make, oracle_layer, oracle_threads, permute_with_rows, run_gpu,
                         sample_tokens, to_cpu, unpack_e2m1)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _threads():
    oracle_threads()


def _check(inp, local_start=0, local_count=-1, mode=0):
    g = run_gpu(inp, local_start, local_count, mode)
    ref = oracle_layer(to_cpu(inp), local_start, local_count, mode)
    check_routing(g, dict(ids=ref["ids"], w=ref["w"], w_masked=ref["w_masked"], slots=ref["slots"],
                          counts=ref["counts"], offsets=ref["offsets"], perm_src=ref["perm_src"],
                          pair_row=ref["pair_row"]), to_cpu(inp), masked=local_count >= 0)
    # weights at the output: the layer quantises token rows through pair_row and leaves
    # x_perm unwritten; routing on the input: x_perm holds the scaled rows (checked by
    # the permute tests)
    check_out(g["out"], ref["out"])
    st = moe.moe_get_device_status(g["layer"].ws)
    assert st == 0, f"device status {st}"
    return g, ref


def _quantize_gpu(v, pow2):
    K = v.shape[-1]
    d = v.cuda()
    q = torch.empty(v.shape[:-1] + (K // 2,), dtype=torch.uint8, device="cuda")
    sb = torch.full(v.shape[:-1] + (moe.nvfp4_sf_row_bytes(K),), 0xAB, dtype=torch.uint8, device="cuda")
    sc = torch.empty(v.shape[:-1], dtype=torch.float32, device="cuda")
    moe.moe_quantize_nvfp4_rows(d, q, sb, sc, pow2=pow2)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sb.cpu().numpy(), sc.cpu().numpy()


def _special_rows(K, g):
    v = torch.randn(12, K, generator=g) * 0.02
    v[0] = 0.0                                              # an all-zero row
    v[1, : K // 2] = 0.0                                    # zero blocks in a live row
    v[2] = torch.randn(K, generator=g) * 3000.0             # large values
    v[3] = torch.full((K,), 2.0 ** -130)                    # bf16 subnormals
    v[4] = torch.linspace(-6.0, 6.0, K)                     # many E2M1 ties at scale 1
    v[5, 0] = 1.0                                           # one element dominating its row
    v[6] = torch.randn(K, generator=g) * 1e-30
    return v.to(torch.bfloat16)


@pytest.mark.parametrize("K", [64, 192, 1408, 2048])
@pytest.mark.parametrize("pow2", [False, True])
def test_quantize_nvfp4_rows_bit_exact(K, pow2):
    g = torch.Generator().manual_seed(K + (1000 if pow2 else 0))
    v = torch.cat([_special_rows(K, g), (torch.randn(100, K, generator=g) * 0.05).to(torch.bfloat16)])
    q, sb, sc = _quantize_gpu(v, pow2)
    rq, rsb, rsc = oracle.quantize_nvfp4_rows(v, pow2=pow2)
    assert np.array_equal(unpack_e2m1(q), rq), "E2M1 codes differ"
    assert np.array_equal(sb[:, : K // 16], rsb), "block scales differ"
    assert not sb[:, K // 16:].any(), "block-scale padding is not zero"
    assert np.array_equal(sc.view(np.uint32), rsc.view(np.uint32)), "row scales differ"


def _threshold_rows(K):
    """Rows whose quotients v / (sb s) land exactly on the E2M1 rounding thresholds
    (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5; round-half-even decides them) under block
    scales that are not powers of two, so a quotient formed as v * (1 / (sb s))
    misses the tie by a few ulps: the row amax 2688 makes s = 1 in both modes, and
    each block's maximum 6 c makes its scale exactly c."""
    t = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    cs = [1.25, 1.5, 1.75, 1.875, 3.0, 3.5, 5.0, 7.0, 0.875, 0.625, 0.5625, 13.0, 0.1875, 26.0, 112.0]
    rows = []
    for r in range(2):
        row = []
        for b in range(K // 16):
            if b == 0:
                blk = [2688.0] + [0.0] * 15                 # sets s = 1
            else:
                c = cs[(b + 3 * r) % len(cs)]
                blk = [6.0 * c] + [x * c for x in t] + [-x * c for x in t] + [0.5 * c]
            row += blk
        rows.append(row)
    v = torch.tensor(rows, dtype=torch.float64)
    assert torch.equal(v.to(torch.bfloat16).double(), v), "threshold values are not bf16 values"
    return v.to(torch.bfloat16)


@pytest.mark.parametrize("pow2", [False, True])
def test_quantize_nvfp4_rows_exact_ties_under_odd_block_scales(pow2):
    v = _threshold_rows(256)
    q, sb, sc = _quantize_gpu(v, pow2)
    rq, rsb, rsc = oracle.quantize_nvfp4_rows(v, pow2=pow2)
    assert np.array_equal(sc.view(np.uint32), rsc.view(np.uint32)) and (rsc == 1.0).all()
    assert np.array_equal(sb[:, :16], rsb), "block scales differ"
    assert np.array_equal(unpack_e2m1(q), rq), "E2M1 codes differ at the rounding ties"


def _every_value_under_every_block_scale():
    """Rows of 16 blocks: the first block's 2688 makes s = 1; every other block is
    [6 c, v1 .. v15] with c an E4M3 value (so the block scale is exactly c) and the v
    running through every finite bf16 magnitude up to 6 c, for every positive E4M3 c,
    with alternating signs."""
    mags = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    blocks = []
    for code in range(1, 127):
        e, m = code >> 3, code & 7
        c = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        v = mags[mags <= 6 * c].copy()
        v[1::2] *= -1.0
        v = np.concatenate([v, np.zeros((-len(v)) % 15, np.float32)]).reshape(-1, 15)
        blocks.append(np.concatenate([np.full((len(v), 1), 6 * c, np.float32), v], axis=1))
    blocks = np.concatenate(blocks)
    blocks = np.concatenate([blocks, np.zeros(((-len(blocks)) % 15, 16), np.float32)]).reshape(-1, 15 * 16)
    first = np.zeros((len(blocks), 16), np.float32)
    first[:, 0] = 2688.0
    v = torch.from_numpy(np.concatenate([first, blocks], axis=1))
    assert torch.equal(v.to(torch.bfloat16).float(), v)
    return v.to(torch.bfloat16)


def test_quantize_nvfp4_division_free_codes_exhaustive_over_block_scales():
    # power-of-two row scales take the reciprocal-and-residual path: it must give the
    # codes of the binary32 division for every (value, block scale) pair
    v = _every_value_under_every_block_scale()
    q, sb, sc = _quantize_gpu(v, True)
    rq, rsb, rsc = oracle.quantize_nvfp4_rows(v, pow2=True)
    assert (rsc == 1.0).all() and np.array_equal(sc.view(np.uint32), rsc.view(np.uint32))
    assert np.array_equal(sb[:, :16], rsb), "block scales differ"
    assert np.array_equal(unpack_e2m1(q), rq), "E2M1 codes differ from the division's"


@pytest.mark.parametrize("pow2", [False, True])
def test_quantize_nvfp4_rows_bit_exact_large_random(pow2):
    g = torch.Generator().manual_seed(77 + pow2)
    rows, K = 2048, 4096
    scale = torch.exp(torch.empty(rows, 1).uniform_(-12.0, 12.0, generator=g))
    v = torch.randn(rows, K, generator=g) * scale
    v[::7] = torch.empty(rows // 7 + 1, K).uniform_(-1.0, 1.0, generator=g) * scale[::7]
    v = v.to(torch.bfloat16)
    q, sb, sc = _quantize_gpu(v, pow2)
    rq, rsb, rsc = oracle.quantize_nvfp4_rows(v, pow2=pow2)
    assert np.array_equal(sc.view(np.uint32), rsc.view(np.uint32)), "row scales differ"
    assert np.array_equal(sb[:, : K // 16], rsb), "block scales differ"
    assert np.array_equal(unpack_e2m1(q), rq), "E2M1 codes differ"


def test_quantize_nvfp4_expert_stack_as_one_matrix():
    inp = mi.make_inputs(mi.MoEConfig("q4stack", T=4, H=256, I=128, E=3, k=1, renorm=True))
    q, sb, sc = _quantize_gpu(inp["W1"], False)
    rq, rsb, rsc = oracle.quantize_nvfp4_rows(inp["W1"])
    assert np.array_equal(unpack_e2m1(q), rq) and np.array_equal(sb[..., :16], rsb)
    assert np.array_equal(sc.view(np.uint32), rsc.view(np.uint32))


NV_MID = mi.MoEConfig("mid_nvfp4", T=1000, H=512, I=384, E=12, k=3, renorm=True, n_shared=1, I_shared=256,
                      shared_gate=True, fp4=True)


def test_nvfp4_mid_layer():
    _check(mi.make_inputs(NV_MID))


def test_nvfp4_ragged_k_partial_tiles_two_shared_experts():
    # FC2's K = I = 320: a stage of 256 elements and a second one zero-filled past K;
    # H = 320: partial N tiles; two shared experts
    cfg = mi.MoEConfig("odd_nvfp4", T=200, H=320, I=320, E=5, k=2, renorm=False, n_shared=2, I_shared=192,
                       fp4=True)
    _check(mi.make_inputs(cfg))


@pytest.mark.parametrize("T", [1, 5, 32])
def test_nvfp4_small_batches(T):
    cfg = mi.MoEConfig(f"sb_nvfp4_{T}", T=T, H=512, I=256, E=16, k=4, renorm=True, n_shared=2, I_shared=256,
                       fp4=True)
    _check(mi.make_inputs(cfg))


def test_nvfp4_local_ranges_routing_on_input_and_replicas():
    inp = mi.make_inputs(NV_MID)
    _check(inp, 4, 5, moe.MOE_NONLOCAL_SKIP)
    _check(inp, 4, 5, moe.MOE_NONLOCAL_MOD)
    _check(mi.make_inputs(NV_MID.with_(name="mid_nvfp4_oi", on_input=True)))
    rep = mi.MoEConfig("rep_nvfp4", T=700, H=256, I=256, E=10, S=13, n_hot=3, zipf_s=1.1, k=4, renorm=True,
                       fp4=True)
    _check(mi.make_inputs(rep))


def _forward_from_x_perm(layer, x):
    """The layer's forward with the expert input rows copied into x_perm by moe_permute and
    quantised row by row (x = None: no shared experts, so nothing reads the token rows)."""
    v = permute_with_rows(layer, x)
    (q1, f1, s1), (q2, f2, s2) = layer.W1f, layer.W2f
    moe.moe_forward_nvfp4(v["x_perm"], v["offsets"], q1, f1, s1, q2, f2, s2, v["pair_row"], v["topk_w"], None,
                          None, None, None, None, None, None, None, v["out"], layer.ws)
    torch.cuda.synchronize()
    return v["out"].clone()


@pytest.mark.parametrize("T,H,local", [(3, 512, None), (700, 512, (3, 9, 0)), (700, 512, (3, 9, 1)),
                                       (4096, 2048, None)])
def test_nvfp4_token_rows_equal_permuted_rows(T, H, local):
    # each token row quantised once and placed at its pairs' rows (moe_permute copies no
    # rows) must give the bits of quantising the permuted copies one by one; 4096 x 2048
    # takes the warp-per-row quantiser, the smaller batches the spread one
    cfg = mi.MoEConfig(f"tok_nvfp4_{T}", T=T, H=H, I=256, E=16, k=4, renorm=True, fp4=True)
    inp = mi.make_inputs(cfg)
    ls, lc, mode = local if local else (0, -1, moe.MOE_NONLOCAL_SKIP)
    layer = layer_from_inputs(inp, "cuda", local_start=ls, local_count=lc, nonlocal_mode=mode)
    assert layer.rows_from_tokens(T)
    x = inp["x"].cuda()
    a = layer.forward(x).clone()
    b = _forward_from_x_perm(layer, x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_get_device_status(layer.ws) == 0


def test_nvfp4_zero_tokens_determinism_and_poisoned_workspace():
    layer = layer_from_inputs(mi.make_inputs(NV_MID), "cuda")
    assert layer.forward(torch.zeros((0, NV_MID.H), dtype=torch.bfloat16, device="cuda")).shape[0] == 0
    x = mi.make_inputs(NV_MID)["x"].cuda()
    a = layer.forward(x).clone()
    layer.ws[moe.MOE_WS_HEADER_BYTES:].fill_(0xFF)  # nothing the forward reads may come from before it
    b = layer.forward(x).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_get_device_status(layer.ws) == 0


@pytest.mark.parametrize("name", ["dsv2_lite_like_decode_t1_nvfp4", "dsv2_lite_like_decode_t32_nvfp4"])
def test_nvfp4_decode_full(name):
    _check(make(name))


def test_nvfp4_qwen2_moe_like_prefill_full_size():
    cfg = mi.CONFIGS["qwen2_moe_like_prefill_nvfp4"]
    inp = mi.make_inputs(cfg, device="cpu", weights_device="cuda")
    inp_cpu = to_cpu(inp)
    g = run_gpu(inp)
    tok = sample_tokens(cfg.T, 32)
    part = oracle_layer(inp_cpu, tokens=tok)
    check_out(g["out"][tok], part["out"])
    assert moe.moe_get_device_status(g["layer"].ws) == 0
