"""moe_build_metadata_noalloc: routing metadata for callers that cannot
allocate device memory.

Some callers have no way to give the library a workspace: a plugin that
enqueues work inside a framework whose allocator owns all device memory, or
a latency-critical path where a cudaMalloc (which can synchronise the
device) is not allowed. The no-allocation entry point keeps its scratch in
a fixed array inside the library instead. This test calls it through the C
ABI, twice in a row on different routings (the array keeps the previous
call's contents), and checks that each result equals, bit for bit, what the
workspace-based moe_build_metadata produces for the same input, and that
the reported device status is MOE_OK. Collected last on purpose; it passes
alone in a fresh process as well as after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_routing_warp_gb300 as moe
import moe_inputs as I

pytestmark = pytest.mark.gpu

KEYS = ("col_sum", "offs", "col_sorted", "row_sorted", "gate_scal")


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return torch.equal(a, b)


@pytest.mark.parametrize("calls", [[(16384, 128, 4, 0), (4099, 32, 4, 7)],
                                   [(300_000, 64, 8, 3), (1, 8, 2, 5)]])
def test_noalloc_matches_workspace_metadata_on_consecutive_calls(calls):
    L = moe.lib()
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for n, E, k, seed in calls:
        logits = torch.from_numpy(I.route_logits(n, E, seed=seed, tie_heavy=True)).to(dev)
        indx, vals = moe.route(logits, k)

        ws = moe.workspace(n, E, k, 64, 64, dev)
        want = moe.build_metadata(indx, vals, E, ws)

        got = moe.empty_meta(n * k, E, dev)
        for t in got.values():   # stale-looking contents: the call must overwrite them
            t.view(torch.uint8).fill_(0xA5)
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        rc = L.moe_build_metadata_noalloc(indx.data_ptr(), vals.data_ptr(), n, E, k,
                                          ctypes.byref(moe._binding._meta_struct(got)),
                                          status.data_ptr(), stream)
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert moe.read_status(ws) == 0
        for key in KEYS:
            assert _same(got[key], want[key]), (n, E, k, key)
        assert int(got["offs"][-1].item()) == n * k
        np.testing.assert_array_equal(got["col_sum"].cpu().numpy(),
                                      np.bincount(indx.cpu().numpy().ravel(), minlength=E))


def test_noalloc_rejects_sizes_beyond_its_limits():
    L = moe.lib()
    meta = moe.RoutingMeta(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    p = ctypes.c_void_p(1 << 20)
    for n, E, k in [(10, 257, 4), (10, 8, 9), (10, 4, 5), (1 << 29, 8, 8), (-1, 8, 2)]:
        assert L.moe_build_metadata_noalloc(p, p, n, E, k, ctypes.byref(meta), None,
                                            None) == 1
