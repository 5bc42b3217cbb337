"""The C-ABI library: it loads, exports every entry point that include/*.h
declare, and rejects bad arguments on the host before anything is enqueued.
No call here reaches the GPU (every case fails validation first)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def _declared():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_expert_gemm_gb300 as m
    return m


def test_header_declares_the_path(moe):
    names = _declared()
    for required in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine",
                     "moe_combine_backward", "moe_dispatch_backward"]:
        assert required in names


def test_library_exports_every_declared_symbol(moe):
    lib = moe.lib()
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(moe.EXPORTED) <= set(_declared())


def _shape(moe, **kw):
    base = dict(T=64, d=128, N=8, K=2, h=256, cap=20)
    base.update(kw)
    return moe.Shape(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), 1), (dict(K=17, N=32), 1), (dict(N=1025), 1), (dict(K=9, N=8), 1),
    (dict(T=-1), 1), (dict(cap=-1), 1), (dict(d=100), 2), (dict(h=12), 2),
    (dict(T=1 << 28, K=8, N=16), 1),
])
def test_shape_validation(moe, kw, code):
    s = _shape(moe, **kw)
    lib = moe.lib()
    assert lib.moe_route_workspace_bytes(ctypes.byref(s)) == 0
    P = ctypes.c_void_p(16)
    assert lib.moe_dispatch(ctypes.byref(s), P, P, P, None) == code
    assert lib.moe_combine(ctypes.byref(s), P, P, P, P, None) == code


def test_buffer_rows_is_the_smaller_bound(moe):
    """Capacity buffers hold min(N*cap, T*K) rows: the packed prefix never
    exceeds the per-expert caps nor one row per route."""
    lib = moe.lib()
    for kw, rows in [(dict(), 64 * 2), (dict(cap=10), 8 * 10), (dict(cap=0), 0),
                     (dict(N=1024, K=2, cap=1 << 21), 128), (dict(K=0), -1)]:
        s = _shape(moe, **kw)
        assert lib.moe_buffer_rows(ctypes.byref(s)) == rows, kw
        if rows >= 0:
            assert s.R == rows


def test_route_logits_offset_lies_inside_the_workspace(moe):
    """The logits [T, N] fp32 sit 256-aligned past the status word and the
    per-block counts, and end inside moe_route_workspace_bytes."""
    lib = moe.lib()
    for kw in [dict(), dict(T=1000, N=64, K=8), dict(T=257, d=136, N=33, K=5), dict(T=0),
               dict(T=300, N=1024, K=16, d=64)]:
        s = _shape(moe, **kw)
        off = lib.moe_route_logits_offset(ctypes.byref(s))
        nblk = (s.T + 255) // 256
        assert off == 256 + ((4 * nblk * s.N + 255) // 256) * 256, kw
        assert off % 256 == 0
        assert off + 4 * s.T * s.N <= lib.moe_route_workspace_bytes(ctypes.byref(s)), kw
    assert lib.moe_route_logits_offset(ctypes.byref(_shape(moe, K=0))) == 0


def test_checked_calls_want_a_status_workspace(moe):
    """The checked row movements refuse a missing or misaligned status
    workspace (MOE_ERR_WORKSPACE) before anything is enqueued."""
    s = _shape(moe)
    lib = moe.lib()
    P = ctypes.c_void_p(256)
    for bad in (None, ctypes.c_void_p(4096 + 16)):
        assert lib.moe_dispatch_checked(ctypes.byref(s), P, P, P, bad, None) == 3
        assert lib.moe_combine_checked(ctypes.byref(s), P, P, P, P, bad, None) == 3
        assert lib.moe_combine_backward_checked(ctypes.byref(s), P, P, P, P, P, P, bad, None) == 3
        assert lib.moe_dispatch_backward_checked(ctypes.byref(s), P, P, P, bad, None) == 3
    assert b"ROUTE_RANGE" in lib.moe_status_string(7)


def test_router_backward_argument_errors(moe):
    s = _shape(moe)
    lib = moe.lib()
    P, Q = ctypes.c_void_p(256), ctypes.c_void_p(264)
    ws_n = lib.moe_router_backward_workspace_bytes(ctypes.byref(s))
    assert ws_n >= 256
    args = [P] * 8 + [None]                            # x .. dw_router, dbias = NULL
    bad = list(args); bad[7] = None                    # dw_router
    assert lib.moe_router_backward(ctypes.byref(s), *bad, P, ws_n, None) == 1
    bad = list(args); bad[5] = None                    # dlogit
    assert lib.moe_router_backward(ctypes.byref(s), *bad, P, ws_n, None) == 1
    bad = list(args); bad[6] = Q                       # dx misaligned
    assert lib.moe_router_backward(ctypes.byref(s), *bad, P, ws_n, None) == 2
    assert lib.moe_router_backward(ctypes.byref(s), *args, P, ws_n - 1, None) == 3
    assert lib.moe_router_backward(ctypes.byref(s), *args, Q, ws_n, None) == 3
    assert lib.moe_router_backward(ctypes.byref(_shape(moe, K=0)), *args, P, ws_n, None) == 1


def test_null_and_alignment_and_workspace_errors(moe):
    s = _shape(moe)
    lib = moe.lib()
    A = ctypes.c_void_p(4096)
    mis = ctypes.c_void_p(4096 + 4)
    assert lib.moe_dispatch(ctypes.byref(s), None, A, A, None) == 1
    assert lib.moe_dispatch(ctypes.byref(s), mis, A, A, None) == 2
    assert lib.moe_combine(ctypes.byref(s), A, A, A, mis, None) == 2
    assert lib.moe_dispatch_backward(ctypes.byref(s), A, A, None, None) == 1
    assert lib.moe_combine_backward(ctypes.byref(s), A, A, A, A, A, None, None) == 1
    ws_need = lib.moe_route_workspace_bytes(ctypes.byref(s))
    assert ws_need >= 256
    args = [A] * 9
    assert lib.moe_route(ctypes.byref(s), *args, A, ws_need - 1, None) == 3
    assert lib.moe_route(ctypes.byref(s), *args, ctypes.c_void_p(4096 + 16), ws_need, None) == 3
    assert lib.moe_route(ctypes.byref(s), *args, None, ws_need, None) == 1
    # expert FFN: tensor-core tiles need d, h multiples of 64
    s2 = _shape(moe, d=136)
    assert lib.moe_expert_ffn(ctypes.byref(s2), *([A] * 10), A, 256, None) == 5
    # g_save without u_save
    ffn = [A, A, A, A, A, A, A, A, None, A]
    assert lib.moe_expert_ffn(ctypes.byref(s), *ffn, A, 256, None) == 1
    assert lib.moe_read_device_error(None, None, None) == 1


def test_status_strings(moe):
    lib = moe.lib()
    for c in range(7):
        assert lib.moe_status_string(c).decode().startswith("MOE_")
    with pytest.raises(moe.MoEError, match="MOE_ERR_ALIGNMENT"):
        moe._check(2, "x")


def test_capacity_formula(moe):
    import synth
    for cfg in synth.CONFIGS.values():
        assert moe.capacity(cfg.T, cfg.K, cfg.N, cfg.cf_num, cfg.cf_den) == cfg.cap
    assert synth.CONFIGS["tiny"].cap == 80 and synth.CONFIGS["olmoe"].cap == 1280
    assert synth.CONFIGS["fine_zipf"].cap == 1024 and synth.CONFIGS["wide"].cap == 6144


def test_product_path_refuses_to_run_without_library(tmp_path):
    """A copy of the binding without its built library raises on import
    instead of falling back to anything."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "combine_expert_gemm_gb300"
    pkg.mkdir()
    for f in ("__init__.py", "build.py"):
        shutil.copy(os.path.join(ROOT, "combine_expert_gemm_gb300", f), pkg / f)
    r = subprocess.run([sys.executable, "-c", "import combine_expert_gemm_gb300"],
                       capture_output=True, text=True, cwd=tmp_path)
    assert r.returncode != 0 and "no CPU fallback" in r.stderr


def test_fused_entry_points_argument_errors(moe):
    """moe_expert_ffn_gather, moe_dispatch_router_backward and
    moe_router_weight_backward refuse bad arguments before enqueuing anything
    (every call here fails validation, so nothing reaches a GPU)."""
    s = _shape(moe)
    lib = moe.lib()
    A, mis = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 8)
    ws_g = lib.moe_expert_ffn_gather_workspace_bytes(ctypes.byref(s))
    assert ws_g >= 256 + 4 * s.R
    args = [A] * 11                                    # x .. y_disp
    assert lib.moe_expert_ffn_gather(ctypes.byref(s), *args, A, ws_g - 1, None) == 3
    assert lib.moe_expert_ffn_gather(ctypes.byref(s), *args, mis, ws_g, None) == 3
    bad = list(args); bad[1] = None                    # route_row
    assert lib.moe_expert_ffn_gather(ctypes.byref(s), *bad, A, ws_g, None) == 1
    bad = list(args); bad[0] = mis                     # x misaligned
    assert lib.moe_expert_ffn_gather(ctypes.byref(s), *bad, A, ws_g, None) == 2
    bad = list(args); bad[8] = None                    # g_save given without u_save
    assert lib.moe_expert_ffn_gather(ctypes.byref(s), *bad, A, ws_g, None) == 1
    s2 = _shape(moe, d=136)
    assert lib.moe_expert_ffn_gather(ctypes.byref(s2), *args, A, ws_g, None) == 5

    d8 = [A] * 8                                       # dx_disp .. dx
    bad = list(d8); bad[3] = None                      # topk_idx
    assert lib.moe_dispatch_router_backward(ctypes.byref(s), *bad, None) == 1
    bad = list(d8); bad[6] = mis                       # dlogit misaligned
    assert lib.moe_dispatch_router_backward(ctypes.byref(s), *bad, None) == 2
    assert lib.moe_dispatch_router_backward(ctypes.byref(_shape(moe, K=0)), *d8, None) == 1

    ws_r = lib.moe_router_backward_workspace_bytes(ctypes.byref(s))
    w5 = [A] * 4 + [None]                              # x, topk_idx, dlogit, dw_router, dbias
    assert lib.moe_router_weight_backward(ctypes.byref(s), *w5, A, ws_r - 1, None) == 3
    bad = list(w5); bad[3] = None                      # dw_router
    assert lib.moe_router_weight_backward(ctypes.byref(s), *bad, A, ws_r, None) == 1
    bad = list(w5); bad[0] = mis                       # x misaligned
    assert lib.moe_router_weight_backward(ctypes.byref(s), *bad, A, ws_r, None) == 2


def test_mxfp8_entry_points_argument_errors(moe):
    """The MXFP8 calls (include/moe_mxfp8.h) refuse bad arguments before
    enqueuing anything; the accepted empty cases return without a launch."""
    s = _shape(moe)                                    # d = 128, h = 256, R = 128
    lib = moe.lib()
    A, mis = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 8)
    # scale-chunk bytes: (ceil(R / 128) + N) * (k / 128) * 512
    assert lib.moe_mx_act_scale_bytes(ctypes.byref(s), 128) == (1 + 8) * 1 * 512
    assert lib.moe_mx_act_scale_bytes(ctypes.byref(s), 256) == (1 + 8) * 2 * 512
    assert lib.moe_mx_act_scale_bytes(ctypes.byref(s), 100) == 0
    assert lib.moe_mx_act_scale_bytes(ctypes.byref(_shape(moe, K=0)), 128) == 0

    q = lib.moe_mx_quantize_weights
    assert q(-1, 128, 128, A, A, A, None) == 1
    assert q(1, 100, 128, A, A, A, None) == 5          # rows not a multiple of 128
    assert q(1, 128, 96, A, A, A, None) == 5           # k not a multiple of 128
    assert q(1, 128, 128, None, A, A, None) == 1
    assert q(1, 128, 128, A, mis, A, None) == 2
    assert q(0, 128, 128, None, None, None, None) == 0  # nothing to do, nothing enqueued

    d7 = [A] * 7                                       # x .. x_sf
    bad = list(d7); bad[1] = None                      # route_row
    assert lib.moe_dispatch_mxfp8(ctypes.byref(s), *bad, None) == 1
    bad = list(d7); bad[0] = mis                       # x misaligned
    assert lib.moe_dispatch_mxfp8(ctypes.byref(s), *bad, None) == 2
    assert lib.moe_dispatch_mxfp8(ctypes.byref(_shape(moe, d=136)), *d7, None) == 5
    assert lib.moe_dispatch_mxfp8(ctypes.byref(_shape(moe, cap=0)), *([None] * 7), None) == 0

    f14 = [A] * 14                                     # x_q .. y_scale
    assert lib.moe_expert_ffn_mxfp8(ctypes.byref(s), *f14, None, 256, None) == 1
    assert lib.moe_expert_ffn_mxfp8(ctypes.byref(s), *f14, A, 255, None) == 3
    assert lib.moe_expert_ffn_mxfp8(ctypes.byref(s), *f14, mis, 256, None) == 3
    bad = list(f14); bad[5] = None                     # w_gate_sf
    assert lib.moe_expert_ffn_mxfp8(ctypes.byref(s), *bad, A, 256, None) == 1
    bad = list(f14); bad[11] = mis                     # h_sf misaligned
    assert lib.moe_expert_ffn_mxfp8(ctypes.byref(s), *bad, A, 256, None) == 2
    assert lib.moe_expert_ffn_mxfp8(ctypes.byref(_shape(moe, h=200)), *f14, A, 256, None) == 5

    c5 = [A] * 5                                       # y_q .. y
    bad = list(c5); bad[4] = None                      # y
    assert lib.moe_combine_mxfp8(ctypes.byref(s), *bad, None) == 1
    bad = list(c5); bad[1] = mis                       # y_scale misaligned
    assert lib.moe_combine_mxfp8(ctypes.byref(s), *bad, None) == 2
    assert lib.moe_combine_mxfp8(ctypes.byref(_shape(moe, d=136)), *c5, None) == 5


def test_binding_refuses_tensors_of_another_device(moe, monkeypatch):
    """The binding passes raw pointers to kernels on the current device, so a
    tensor that lives on another GPU is refused before any call."""
    import torch

    class OnDevice(torch.Tensor):
        index = 0

        @property
        def device(self):
            return torch.device("cuda", type(self).index)

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    t = torch.Tensor._make_subclass(OnDevice, torch.zeros(4, dtype=torch.int32))
    assert moe._ptr(t, torch.int32, "route_row") == t.data_ptr()
    OnDevice.index = 1
    with pytest.raises(ValueError, match="route_row: on cuda:1"):
        moe._ptr(t, torch.int32, "route_row")
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        moe._ptr(torch.zeros(4), None, "x")


def test_expert_backward_workspace_holds_map_slots(moe):
    """moe_expert_ffn_backward's workspace is the status word, dG and dU
    ([R, h] bf16 each, 256-byte aligned) and 1 MiB of tensor-map copies for
    the weight-gradient kernels; one byte short is refused before anything is
    enqueued (every call here fails validation, so nothing reaches a GPU)."""
    s = _shape(moe)
    lib = moe.lib()
    align = lambda n: (n + 255) // 256 * 256
    ws = lib.moe_expert_ffn_backward_workspace_bytes(ctypes.byref(s))
    assert ws == 256 + 2 * align(s.R * s.h * 2) + (1 << 20)
    A = ctypes.c_void_p(4096)
    args = [A] * 14                                     # x_disp .. dw_down
    assert lib.moe_expert_ffn_backward(ctypes.byref(s), *args, A, ws - 1, None) == 3
    assert lib.moe_expert_ffn_backward(ctypes.byref(s), *args, ctypes.c_void_p(4096 + 128), ws,
                                       None) == 3
