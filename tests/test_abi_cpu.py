"""Host-only checks of the C ABI: the library loads, exports every function
include/moe.h declares, sizes workspaces, and rejects bad arguments on the host
before any kernel launch (every case here fails validation, so no pointer is
ever dereferenced and no CUDA call is reached)."""
import ctypes
import os
import re

import pytest

import serving_router_gate_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_API[^(]*?\b(moe_[a-z0-9_]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ("moe_route", "moe_permute", "moe_forward", "moe_workspace_size", "moe_get_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(moe.lib_path())
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(moe.EXPORTED_SYMBOLS) == _declared()


def test_status_strings():
    for code in (0, 1, 2, 3, 4, 8, 16):
        assert moe._lib.moe_status_string(code)


def test_workspace_size():
    n2 = moe.moe_workspace_size(4096, 2048, 1408, 60, 60, 4, 5632)
    # at least h and y of every pair plus the shared expert's h and y
    assert n2 >= 2 * (4096 * 4 * (1408 + 2048) + 4096 * (5632 + 2048))
    n5 = moe.moe_workspace_size(16384, 7168, 2048, 256, 288, 8, 0)
    assert n5 >= 2 * 16384 * 8 * (2048 + 7168)
    assert moe.moe_workspace_size(1, 2048, 1408, 64, 64, 6, 5632) > 0
    assert moe.moe_workspace_size(0, 256, 512, 8, 8, 2, 0) > 0
    for bad in ((64, 100, 512, 8, 8, 2, 0),      # H not a multiple of 64
                (64, 256, 500, 8, 8, 2, 0),      # I not a multiple of 64
                (64, 256, 512, 8, 8, 9, 0),      # k > E
                (64, 256, 512, 600, 600, 2, 0),  # E > 512
                (64, 256, 512, 8, 2000, 2, 0),   # S > 1024
                (-1, 256, 512, 8, 8, 2, 0)):
        assert moe._lib.moe_workspace_size(*bad) == 0


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails host validation first


def test_route_rejects_bad_arguments_on_host():
    r = moe._lib.moe_route
    assert r(FAKE, FAKE, None, 16, 256, 8, 9, 1, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert r(FAKE, FAKE, None, -1, 256, 8, 2, 1, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert r(FAKE, FAKE, None, 16, 100, 8, 2, 1, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    assert r(FAKE, FAKE, None, 16, 256, 600, 2, 1, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    assert r(None, FAKE, None, 16, 256, 8, 2, 1, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert r(FAKE, FAKE, None, 16, 256, 8, 2, 1, FAKE, FAKE, None, 1 << 30, None) == moe.MOE_ERR_WORKSPACE
    assert r(FAKE, FAKE, None, 16, 256, 8, 2, 1, FAKE, FAKE, FAKE, 64, None) == moe.MOE_ERR_WORKSPACE
    assert r(None, None, None, 0, 256, 8, 2, 1, None, None, None, 0, None) == moe.MOE_OK  # T = 0: no-op


def test_permute_rejects_bad_arguments_on_host():
    p = moe._lib.moe_permute

    def call(T=16, k=2, E=8, ro=None, rs=None, S=8, ls=0, lc=-1, mode=0, H=256, ws=FAKE, wsb=1 << 30, ids=FAKE):
        return p(ids, FAKE, T, k, E, ro, rs, S, ls, lc, mode, FAKE, H, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                 ws, wsb, None)

    assert call(S=9) == moe.MOE_ERR_INVALID_ARG                    # no table but S != E
    assert call(ro=FAKE, rs=None, S=9) == moe.MOE_ERR_INVALID_ARG  # table without slots
    assert call(mode=2) == moe.MOE_ERR_INVALID_ARG
    assert call(ls=6, lc=4) == moe.MOE_ERR_INVALID_ARG             # range past S
    assert call(ls=-1, lc=4) == moe.MOE_ERR_INVALID_ARG
    assert call(lc=0) == moe.MOE_ERR_INVALID_ARG
    assert call(H=96) == moe.MOE_ERR_UNSUPPORTED
    assert call(k=33, E=64, S=64) == moe.MOE_ERR_UNSUPPORTED
    assert call(ids=None) == moe.MOE_ERR_INVALID_ARG
    assert call(ws=None) == moe.MOE_ERR_WORKSPACE
    assert call(wsb=300) == moe.MOE_ERR_WORKSPACE


def test_forward_and_stages_reject_bad_arguments_on_host():
    f = moe._lib.moe_forward

    def call(S_local=8, P_cap=32, H=256, I=512, T=16, k=2, x=FAKE, W1s=None, W2s=None, I_sh=0, gate=None,
             ws=FAKE, wsb=1 << 30, out=FAKE):
        return f(FAKE, FAKE, S_local, P_cap, FAKE, FAKE, H, I, FAKE, FAKE, T, k, x, W1s, W2s, I_sh, gate, out,
                 ws, wsb, None)

    assert call(S_local=0) == moe.MOE_ERR_INVALID_ARG
    assert call(I=100) == moe.MOE_ERR_UNSUPPORTED
    assert call(I_sh=256) == moe.MOE_ERR_INVALID_ARG         # shared size without shared weights
    assert call(gate=FAKE) == moe.MOE_ERR_INVALID_ARG        # gate without a shared expert
    assert call(out=None) == moe.MOE_ERR_INVALID_ARG
    assert call(ws=None) == moe.MOE_ERR_WORKSPACE
    assert call(wsb=1000) == moe.MOE_ERR_WORKSPACE
    assert call(T=0) == moe.MOE_OK
    fc1 = moe._lib.moe_grouped_fc1
    assert fc1(FAKE, 32, FAKE, 2000, FAKE, 256, 512, None, 0, None, 0, FAKE, None, FAKE, 1 << 20,
               None) == moe.MOE_ERR_UNSUPPORTED
    assert fc1(FAKE, 32, None, 4, FAKE, 256, 512, None, 0, None, 0, FAKE, None, FAKE, 1 << 20,
               None) == moe.MOE_ERR_INVALID_ARG
    assert fc1(FAKE, 32, FAKE, 4, FAKE, 256, 512, None, 0, None, 0, FAKE, None, None, 0,
               None) == moe.MOE_ERR_WORKSPACE
    fin = moe._lib.moe_finalize
    assert fin(FAKE, 32, FAKE, FAKE, 16, 2, 256, None, None, FAKE, FAKE, FAKE, 1 << 20,
               None) == moe.MOE_ERR_INVALID_ARG  # gate without x / y_shared
    assert fin(FAKE, 32, FAKE, FAKE, 16, 40, 256, None, None, None, FAKE, FAKE, 1 << 20,
               None) == moe.MOE_ERR_UNSUPPORTED
    dbg = moe._lib.moe_debug_wait_timeout
    assert dbg(FAKE, 1 << 20, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert dbg(None, 0, 1000, None) == moe.MOE_ERR_WORKSPACE


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        moe.moe_route(x, torch.zeros(8, 256), None, 2, True, torch.zeros(4, 2, dtype=torch.int32),
                      torch.zeros(4, 2), torch.zeros(1 << 20, dtype=torch.uint8))


def test_rejected_calls_launch_nothing():
    """Calls refused by host validation never reach a kernel launch, so the
    library's launch count does not move."""
    before = moe.moe_get_launch_count()
    assert before >= 0
    r = moe._lib.moe_route
    assert r(None, FAKE, None, 16, 256, 8, 2, 1, FAKE, FAKE, FAKE, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert r(FAKE, FAKE, None, 16, 256, 8, 2, 1, FAKE, FAKE, FAKE, 64, None) == moe.MOE_ERR_WORKSPACE
    assert moe.moe_get_launch_count() == before


def test_route_grouped_rejects_bad_group_parameters_on_host():
    r = moe._lib.moe_route_grouped
    args = lambda E, k, ng, tg: (FAKE, FAKE, None, 16, 256, E, k, 1, ng, tg, FAKE, FAKE, FAKE, 1 << 30, None)  # noqa: E731
    assert r(*args(32, 4, 5, 2)) == moe.MOE_ERR_INVALID_ARG    # E not a multiple of n_group
    assert r(*args(32, 4, 8, 9)) == moe.MOE_ERR_INVALID_ARG    # topk_group > n_group
    assert r(*args(32, 9, 8, 2)) == moe.MOE_ERR_INVALID_ARG    # k > topk_group * E / n_group
    assert r(*args(128, 4, 64, 2)) == moe.MOE_ERR_INVALID_ARG  # n_group > 32
    assert r(*args(32, 4, 0, 1)) == moe.MOE_ERR_INVALID_ARG
    assert r(None, None, None, 0, 256, 32, 4, 1, 8, 2, None, None, None, 0, None) == moe.MOE_OK  # T = 0


def test_permute_without_x_perm_and_nvfp4_token_rows_validation():
    p = moe._lib.moe_permute
    args = lambda x, xp: (FAKE, FAKE, 16, 2, 8, None, None, 8, 0, -1, 0, x, 256, FAKE, FAKE, FAKE, FAKE, FAKE, xp,
                          None, 1 << 30, None)
    assert p(*args(None, FAKE)) == moe.MOE_ERR_INVALID_ARG  # rows to copy but no token rows
    assert p(*args(FAKE, FAKE)[:19], None, 300, None) == moe.MOE_ERR_WORKSPACE
    assert p(*args(None, None)[:19], FAKE, 300, None) == moe.MOE_ERR_WORKSPACE  # tables only: x not needed
    # routing on the input scales the copied rows: x_perm is required
    assert moe._lib.moe_permute_on_input(*args(FAKE, None)) == moe.MOE_ERR_INVALID_ARG
    f = moe._lib.moe_forward_nvfp4
    odd = ctypes.c_void_p(FAKE.value + 2)

    def fwd(x_perm, topk_w, x):
        return f(x_perm, FAKE, 4, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 256, FAKE, topk_w, 16, 2, x, None,
                 None, None, None, None, None, 0, None, FAKE, FAKE, 1 << 30, None)

    assert fwd(None, FAKE, None) == moe.MOE_ERR_INVALID_ARG   # token rows need x
    assert fwd(None, None, FAKE) == moe.MOE_ERR_INVALID_ARG   # and the weights at the output
    assert fwd(None, FAKE, odd) == moe.MOE_ERR_INVALID_ARG    # x must be 16-byte aligned
    assert fwd(odd, None, None) == moe.MOE_ERR_INVALID_ARG    # x_perm too, when it is read


def test_permute_on_input_shares_the_host_validation():
    p = moe._lib.moe_permute_on_input
    # S != E without a slot table
    assert p(FAKE, FAKE, 16, 2, 8, None, None, 9, 0, -1, 0, FAKE, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
             FAKE, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG


def test_a2a_regroup_rejects_bad_arguments_on_host():
    f = moe._lib.moe_a2a_regroup
    other = ctypes.c_void_p(0x2000)
    odd = ctypes.c_void_p(0x2002)
    before = moe.moe_get_launch_count()

    def call(N=4, S_l=8, src=FAKE, dst=other, rows=64, H=256, direction=moe.MOE_A2A_TO_GEMM, counts=FAKE,
             ws=FAKE, ws_bytes=1 << 20):
        return f(counts, N, S_l, src, dst, rows, H, direction, None, None, ws, ws_bytes, None)

    assert call(N=0) == moe.MOE_ERR_INVALID_ARG
    assert call(S_l=0) == moe.MOE_ERR_INVALID_ARG
    assert call(rows=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(direction=2) == moe.MOE_ERR_INVALID_ARG
    assert call(counts=None) == moe.MOE_ERR_INVALID_ARG
    assert call(N=64, S_l=65) == moe.MOE_ERR_UNSUPPORTED       # more blocks than the tables hold
    assert call(H=100) == moe.MOE_ERR_UNSUPPORTED              # H not a multiple of 64
    assert call(rows=1 << 31) == moe.MOE_ERR_UNSUPPORTED       # rows beyond int32
    assert call(dst=FAKE) == moe.MOE_ERR_INVALID_ARG           # in place
    assert call(src=None) == moe.MOE_ERR_INVALID_ARG
    assert call(dst=odd) == moe.MOE_ERR_INVALID_ARG            # not 16-byte aligned
    assert call(ws=None) == moe.MOE_ERR_WORKSPACE
    assert call(ws_bytes=64) == moe.MOE_ERR_WORKSPACE
    # FC2 with a row map: the map is required when there are rows
    fs = moe._lib.moe_grouped_fc2_scatter
    assert fs(FAKE, 64, FAKE, 4, FAKE, 256, 256, None, 0, None, 0, None, other, None, FAKE, 1 << 20,
              None) == moe.MOE_ERR_INVALID_ARG
    assert fs(FAKE, 64, FAKE, 4, FAKE, 256, 250, None, 0, None, 0, FAKE, other, None, FAKE, 1 << 20,
              None) == moe.MOE_ERR_UNSUPPORTED  # I not a multiple of 64
    assert moe.moe_get_launch_count() == before


def test_ep_signal_reduce_and_ipc_reject_bad_arguments_on_host():
    lib = moe._lib
    before = moe.moe_get_launch_count()
    two = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    odd = (ctypes.c_void_p * 2)(0x1000, 0x2002)
    nul = (ctypes.c_void_p * 2)(0x1000, 0)
    assert lib.moe_ep_signal(None, 2, 0, 1, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_ep_signal(two, 0, 0, 1, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_ep_signal(two, 17, 0, 1, None) == moe.MOE_ERR_INVALID_ARG   # more than 16 ranks
    assert lib.moe_ep_signal(two, 2, 2, 1, None) == moe.MOE_ERR_INVALID_ARG    # rank outside the world
    assert lib.moe_ep_signal(nul, 2, 0, 1, None) == moe.MOE_ERR_INVALID_ARG
    r = lib.moe_ep_reduce

    def red(parts=two, N=2, flags=FAKE, r0=0, r1=8, H=256, out=FAKE, ws=FAKE, ws_bytes=1 << 20):
        return r(parts, N, flags, 1, r0, r1, H, out, ws, ws_bytes, None)

    assert red(parts=None) == moe.MOE_ERR_INVALID_ARG
    assert red(flags=None) == moe.MOE_ERR_INVALID_ARG
    assert red(r0=9) == moe.MOE_ERR_INVALID_ARG                # row1 < row0
    assert red(H=100) == moe.MOE_ERR_UNSUPPORTED
    assert red(ws=None) == moe.MOE_ERR_WORKSPACE
    assert red(parts=odd) == moe.MOE_ERR_INVALID_ARG           # partials 16-byte aligned
    assert red(out=None) == moe.MOE_ERR_INVALID_ARG
    assert red(r0=4, r1=4) == moe.MOE_OK                        # no rows: nothing to do
    assert moe.moe_get_launch_count() == before
    assert lib.moe_ipc_export(None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_ipc_import(None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_ipc_close(None, 0) == moe.MOE_ERR_INVALID_ARG


def test_launch_event_hook_host_side():
    lib = moe._lib
    assert lib.moe_launch_events_arm(None, -1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_launch_events_arm(None, 3) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_launch_events_arm(None, 0) == moe.MOE_OK
    assert lib.moe_launch_events_mark(None) == moe.MOE_OK      # disarmed: records nothing, calls no CUDA
    assert lib.moe_launch_events_used(None, 0) == 0
    # arming only stores the handles (no CUDA call); nothing is recorded until a launch or a mark
    handles = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    assert lib.moe_launch_events_arm(handles, 2) == moe.MOE_OK
    assert lib.moe_launch_events_used(None, 0) == 0
    assert lib.moe_launch_events_arm(None, 0) == moe.MOE_OK
    assert moe.moe_launch_events_used() == []


def test_import_without_the_built_library_fails_loudly(tmp_path):
    # a copy of the Python package with no compiled library next to it: the import must
    # raise ImportError (no fallback path exists)
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "serving_router_gate_gb300")
    dst = tmp_path / "serving_router_gate_gb300"
    dst.mkdir()
    for name in os.listdir(src):
        if name.endswith(".py"):
            shutil.copy(os.path.join(src, name), dst / name)
    code = ("import sys; sys.path.insert(0, sys.argv[1])\n"
            "try:\n    import serving_router_gate_gb300\nexcept ImportError as e:\n"
            "    print('ImportError:', e); sys.exit(0)\n"
            "sys.exit(3)\n")
    r = subprocess.run([sys.executable, "-c", code, str(tmp_path)], capture_output=True, text=True, timeout=300,
                       cwd=str(tmp_path))
    assert r.returncode == 0, r.stdout + r.stderr
    assert "not built" in r.stdout
