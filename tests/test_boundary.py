"""The C ABI without a GPU: the library loads, exports every function that
include/moe.h declares, and rejects bad arguments on the host before any
launch (these calls never reach the CUDA runtime)."""
import ctypes
import os
import re
import subprocess

import pytest

import mixture_experts_routing_warp_gb300 as moe
from mixture_experts_routing_warp_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    cuda_build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_compiles_as_c99(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "moe.h"\nint main(void) { moe_params p = {0}; (void)p; '
                   'return moe_abi_version() == MOE_ABI_VERSION ? 0 : 1; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    f"-I{os.path.join(ROOT, 'include')}", "-c", str(src), "-o",
                    str(tmp_path / "t.o")], check=True)


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert len(names) >= 10, names
    for name in names:
        assert hasattr(L, name), f"{name} declared in moe.h but not exported"
    assert set(names) == set(moe._binding.SIGNATURES), "binding and header disagree"


def test_abi_and_status_strings(L):
    assert L.moe_abi_version() == 4
    for code in range(7):
        s = moe.status_string(code)
        assert s.startswith("MOE_"), s
    assert moe.status_string(99) == "unknown moe_status"


def test_workspace_size(L):
    assert moe.workspace_size(33, 8, 2, 64, 128) > 0
    for bad in [(-1, 8, 2, 64, 128), (33, 0, 2, 64, 128), (33, 300, 2, 64, 128),
                (33, 8, 9, 64, 128), (33, 4, 5, 64, 128), (33, 8, 2, 65, 128),
                (33, 8, 2, 64, 100), (1 << 30, 8, 4, 64, 64)]:
        assert moe.workspace_size(*bad) == 0, bad
    a = moe.workspace_size(1000, 8, 1, 512, 1408)
    b = moe.workspace_size(1000, 8, 2, 512, 1408)
    assert b > a   # per-slot outputs only when k > 1
    assert moe.workspace_size(0, 8, 2, 64, 128) > 0


@pytest.mark.parametrize("sizes", [(33, 8, 2, 64, 128), (1, 32, 4, 2880, 2880),
                                   (8191, 256, 8, 192, 320), (0, 4, 1, 64, 64)])
def test_workspace_regions(L, sizes):
    """Regions in layout order, each 256-byte aligned and inside the
    workspace, none overlapping the next; sized for the arrays they hold."""
    n, E, k, H, I_ = sizes
    reg = moe.workspace_regions(*sizes)
    total = moe.workspace_size(*sizes)
    N = n * k
    assert reg["x_sorted"][1] == N * H * 2 and reg["h"][1] == N * I_ * 2
    assert reg["y_flat"][1] == N * H * 2 and reg["col_sorted"][1] == N * 4
    assert reg["offs"][1] == (E + 1) * 4 and reg["gate_scal"][1] == N * 2
    spans = list(reg.values())
    for (o, b), (o2, _) in zip(spans, spans[1:] + [(total, 0)]):
        assert o % 256 == 0 and o + b <= o2, (o, b, o2)
    with pytest.raises(moe.MoEError):
        moe.workspace_regions(33, 0, 2, 64, 128)


def _p(v):
    return ctypes.c_void_p(v)


def test_route_rejects_before_launch(L):
    good = _p(1 << 20)
    # invalid sizes / enums
    assert L.moe_route(good, 4, 0, 1, 0, good, good, None) == 1
    assert L.moe_route(good, 4, 8, 9, 0, good, good, None) == 1
    assert L.moe_route(good, 4, 4, 5, 0, good, good, None) == 1
    assert L.moe_route(good, -1, 8, 2, 0, good, good, None) == 1
    assert L.moe_route(good, 4, 8, 2, 7, good, good, None) == 1
    # null and misaligned pointers
    assert L.moe_route(None, 4, 8, 2, 0, good, good, None) == 1
    assert L.moe_route(_p((1 << 20) + 2), 4, 8, 2, 0, good, good, None) == 6
    # n = 0 is a no-op
    assert L.moe_route(None, 0, 8, 2, 0, None, None, None) == 0


def test_forward_launch_count_host_rules(L):
    assert L.moe_forward_launch_count(0, 8, 2, 64, 128) == 0
    for bad in [(10, 8, 9, 64, 64), (10, 0, 1, 64, 64), (10, 8, 2, 96, 64), (-1, 8, 2, 64, 64)]:
        assert L.moe_forward_launch_count(*bad) == -1, bad


def test_ffn_plan_host_rules(L):
    """moe_ffn_plan validates like moe_forward, reports the tokens-on-M
    kernel's fixed tiling, and flags the decode tiling (n*k <= 32 E) on the
    host alone."""
    plan = (ctypes.c_int32 * 6)()
    p = ctypes.byref(moe.make_params())
    assert L.moe_ffn_plan(8, 0, 1, 128, 128, p, plan) == 1      # E < 1
    assert L.moe_ffn_plan(8, 4, 2, 96, 128, p, plan) == 1       # H not a multiple of 64
    assert L.moe_ffn_plan(8, 4, 2, 128, 128, p, None) == 1      # no output
    assert L.moe_ffn_plan(8, 4, 2, 128, 128, ctypes.byref(moe.make_params(ffn_kernel="tiled")),
                          plan) == 0
    assert list(plan) == [128, 128, 0, 0, 0, 0]
    assert L.moe_ffn_plan(1, 32, 4, 2880, 2880, p, plan) == 0
    assert plan[4] == 1 and plan[0] == plan[1] == 32 and plan[2] == plan[3] == 0
    assert plan[5] == 1  # decode: both contractions in one launch
    assert L.moe_ffn_plan(256, 32, 4, 2880, 2880, p, plan) == 0  # n*k = 32 E: still decode
    assert plan[4] == 1
    assert L.moe_ffn_plan(257, 32, 4, 2880, 2880, p, plan) == 0
    assert plan[4] == 0


def test_ffn_and_forward_parameter_rules(L):
    good = _p(1 << 20)
    ws = _p(1 << 20)
    meta = moe.RoutingMeta(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    big = moe.workspace_size(8, 4, 2, 64, 64)

    def ffn(params, **kw):
        a = dict(n=8, E=4, k=2, H=64, I=64, ws_bytes=big)
        a.update(kw)
        return L.moe_grouped_ffn(good, ctypes.byref(meta), good, good, a["n"], a["E"], a["k"],
                                 a["H"], a["I"], ctypes.byref(params), good, ws, a["ws_bytes"],
                                 None)

    # SwiGLU takes a clamp limit ("SILU + clamp"), which must be >= 0 and not NaN;
    # ReLU2 takes none
    assert ffn(moe.make_params(act="swiglu", limit=-1.0)) == 1
    assert ffn(moe.make_params(act="swiglu", limit=float("nan"))) == 1
    assert ffn(moe.make_params(act="relu2", limit=3.0)) == 2
    bad = moe.make_params()
    bad.activation = 3
    assert ffn(bad) == 1
    # alpha / beta are not parameters of plain SwiGLU: ignored, and n = 0 is a no-op
    assert ffn(moe.make_params(act="swiglu", alpha=2.0), n=0) == 0
    assert ffn(moe.make_params(act="swiglu_oai", limit=-1.0)) == 1
    assert ffn(moe.make_params(act="swiglu_oai", alpha=float("nan"))) == 1
    bad = moe.make_params()
    bad.w13_layout = 5
    assert ffn(bad) == 1
    bad = moe.make_params()
    bad.set = 8
    assert ffn(bad) == 1
    bad = moe.make_params()
    bad.ffn_kernel = 3
    assert ffn(bad) == 1
    assert ffn(moe.make_params(), ws_bytes=big - 1) == 3
    assert ffn(moe.make_params(), H=96) == 1
    assert L.moe_grouped_ffn(_p((1 << 20) + 8), ctypes.byref(meta), good, good, 8, 4, 2, 64, 64,
                             ctypes.byref(moe.make_params()), good, ws, big, None) == 6
    assert L.moe_grouped_ffn(good, None, good, good, 8, 4, 2, 64, 64,
                             ctypes.byref(moe.make_params()), good, ws, big, None) == 1
    # forward: topk outputs come as a pair
    assert L.moe_forward(good, good, good, good, 8, 4, 2, 64, 64,
                         ctypes.byref(moe.make_params()), good, good, None, None, ws, big,
                         None) == 1
    # expert map: n_local_experts in [1, E], a 4-byte aligned map (checked
    # before the n = 0 shortcut, so no launch is needed to see it)
    def fwd(params, n=0):
        return L.moe_forward(good, good, good, good, n, 4, 2, 64, 64, ctypes.byref(params), good,
                             None, None, None, ws, big, None)

    emap = moe.make_params()
    emap.expert_map = 1 << 20
    for n_local, rc in ((0, 1), (5, 1), (1, 0), (4, 0)):
        emap.n_local_experts = n_local
        assert fwd(emap) == rc, n_local
    emap.expert_map = (1 << 20) + 2
    assert fwd(emap) == 6
    assert L.moe_combine(good, 8, 2, 100, good, None) == 1
    assert L.moe_combine(None, 0, 2, 64, None, None) == 0
    assert L.moe_read_status(None, 0, 0, None) == 1
    assert L.moe_selftest_wait_timeout(ws, 4096, 0, None) == 1
    assert L.moe_selftest_wait_timeout(ws, 4096, 10 ** 10, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe._binding, "_LIB", None)
    monkeypatch.setattr(moe._binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.lib()


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "mixture_experts_routing_warp_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "moe_oracle" not in text, f
