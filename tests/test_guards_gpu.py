"""Out-of-bounds writes, checked with canaries (a stand-in for a memory checker).

Every buffer the library writes is carved out of a larger allocation whose
bytes before and after it hold a canary pattern (0xA5), and the workspace's
own gaps -- the bytes between one internal region's end (X_sorted, h,
y_flat, the metadata arrays, ...) and the next region's start -- hold it too.
After forwards and stage calls at ragged sizes (slot counts that are no
multiple of 32 or 256, experts with no token, E = 256 with k = 8, decode
tiles, CTA-pair tiles, the routing kernel's row copy, k = 1 where the w2
contraction writes the output itself), every canary byte must be intact, the
device status word 0 and the output within the parity tolerance of the
oracle."""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_routing_warp_gb300 as moe
import moe_inputs as I
import oracle

from helpers import assert_layer_close, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

CANARY = 0xA5
GUARD = 4096   # canary bytes on each side of a buffer (keeps 256-byte alignment)


class Guarded:
    """Device buffers with canary bytes on both sides."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        t = raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
        self.bufs.append((raw, nbytes, f"{tuple(shape)} {dtype}"))
        return t

    def workspace(self, n, E, k, H, I_):
        size = moe.workspace_size(n, E, k, H, I_)
        raw = torch.full((size + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        ws = raw[GUARD:GUARD + size]
        st = moe.lib().moe_workspace_init(ws.data_ptr(), size,
                                          ctypes.c_void_p(torch.cuda.current_stream()
                                                          .cuda_stream))
        assert st == 0
        self.bufs.append((raw, size, "workspace"))
        self.ws_raw, self.ws_regions = raw, moe.workspace_regions(n, E, k, H, I_)
        return ws

    def check(self):
        torch.cuda.synchronize()
        for raw, nbytes, what in self.bufs:
            head = raw[:GUARD].cpu().numpy()
            tail = raw[GUARD + nbytes:].cpu().numpy()
            assert (head == CANARY).all(), f"{what}: write before the buffer"
            assert (tail == CANARY).all(), \
                f"{what}: write past the end at +{int(np.nonzero(tail != CANARY)[0][0])}"
        if hasattr(self, "ws_raw"):
            host = self.ws_raw[GUARD:].cpu().numpy()
            spans = list(self.ws_regions.items())
            total = self.ws_raw.numel() - 2 * GUARD
            for i, (name, (off, used)) in enumerate(spans):
                nxt = spans[i + 1][1][0] if i + 1 < len(spans) else total
                gap = host[off + used:nxt]
                assert (gap == CANARY).all(), f"workspace region {name}: write past its end"


def _case(name, n, H, E, k, I_, act="swiglu", layout="packed", seed=0):
    return I.LayerCase(name, n=n, H=H, E=E, k=k, I=I_, act=act, layout=layout, w_std=0.05,
                       seed=seed)


def _routed(case, counts, seed=0):
    """Inputs whose top-1 slot sends counts[e] tokens to expert e."""
    h = I.layer_inputs(case)
    n, E, k = case.n, case.E, case.k
    owner = np.random.default_rng(seed).permutation(np.repeat(np.arange(E), counts))
    logits = np.zeros((n, E), dtype=np.float32)
    for t in range(n):
        for j in range(k):
            logits[t, (owner[t] + j) % E] = float(k - j) + 1.0
    h["logits"] = logits
    return h


CASES = [
    # ragged slot counts through the 256-row tiles (N = 3000)
    (_case("ragged_n1000", 1000, 192, 8, 3, 320), None, "auto"),
    (_case("ragged_n1000_tiled", 1000, 192, 8, 3, 320), None, "tiled"),
    # the cooperative routing kernel copies the dispatch rows (N = 16380)
    (_case("rows_in_routing_n4095", 4095, 256, 32, 4, 128, "swiglu_oai", "interleaved"), None,
     "auto"),
    # experts without tokens, k = 1: the w2 epilogue writes the output
    (_case("empty_experts_k1", 606, 128, 5, 1, 192), (0, 600, 0, 5, 1), "auto"),
    (_case("empty_experts_k1_tiled", 606, 128, 5, 1, 192), (0, 600, 0, 5, 1), "tiled"),
    # the largest expert count and top-k
    (_case("e256_k8", 77, 64, 256, 8, 64), None, "auto"),
    # decode: stream-K w13, rows gathered inside w13 (n k <= 2 E), 32-row tiles
    (_case("decode_n1", 1, 256, 32, 4, 128, "swiglu_oai", "interleaved"), None, "auto"),
    (_case("decode_n3", 3, 256, 32, 4, 128, "swiglu_oai", "interleaved"), None, "auto"),
    (_case("decode_n37", 37, 256, 32, 4, 128, "swiglu_oai", "interleaved"), None, "auto"),
    # CTA-pair tiles with a ragged last tile per expert
    (_case("pairs_n2047", 2047, 384, 8, 4, 192, "swiglu_oai", "interleaved", seed=3), None,
     "auto"),
    (_case("relu2_n301", 301, 192, 8, 3, 320, "relu2"), None, "auto"),
]


@pytest.mark.parametrize("case,counts,ffn_kernel", CASES, ids=[c[0].name for c in CASES])
def test_forward_writes_stay_in_bounds(case, counts, ffn_kernel):
    c = case
    h = I.layer_inputs(c) if counts is None else _routed(c, counts)
    x, logits = dev_bf16(h["x"]), dev(h["logits"])
    w13, w2 = dev_bf16(h["w13"]), dev_bf16(h["w2"])
    params = moe.make_params(c.gating, c.act, c.layout, ffn_kernel=ffn_kernel)
    g = Guarded()
    ws = g.workspace(c.n, c.E, c.k, c.H, c.I)
    out = g.empty((c.n, c.H), torch.bfloat16)
    indx = g.empty((c.n, c.k), torch.int32)
    vals = g.empty((c.n, c.k), torch.bfloat16)
    N = c.n * c.k
    meta = {"col_sum": g.empty((c.E,), torch.int32), "offs": g.empty((c.E + 1,), torch.int32),
            "col_sorted": g.empty((N,), torch.int32), "row_sorted": g.empty((N,), torch.int32),
            "gate_scal": g.empty((N,), torch.bfloat16)}
    moe.forward(x, logits, w13, w2, c.k, params, ws, out=out, topk=(indx, vals), meta=meta)
    g.check()
    assert moe.read_status(ws) == 0
    if counts is not None:
        np.testing.assert_array_equal(meta["col_sum"].cpu().numpy(), np.array(counts))
    ref = oracle.ffn(h["x"], indx.cpu().numpy(), host_bits(vals), h["w13"], h["w2"],
                     act=c.act, layout=c.layout)
    assert_layer_close(host_bits(out), ref, c.name)


@pytest.mark.parametrize("case,counts,ffn_kernel", CASES[:4] + CASES[6:8],
                         ids=[c[0].name for c in CASES[:4] + CASES[6:8]])
def test_stage_writes_stay_in_bounds(case, counts, ffn_kernel):
    """route -> build_metadata -> grouped_ffn -> combine into guarded
    buffers (y_flat included), then the same canary checks."""
    c = case
    h = I.layer_inputs(c) if counts is None else _routed(c, counts)
    x, logits = dev_bf16(h["x"]), dev(h["logits"])
    w13, w2 = dev_bf16(h["w13"]), dev_bf16(h["w2"])
    params = moe.make_params(c.gating, c.act, c.layout, ffn_kernel=ffn_kernel)
    g = Guarded()
    ws = g.workspace(c.n, c.E, c.k, c.H, c.I)
    N = c.n * c.k
    indx = g.empty((c.n, c.k), torch.int32)
    vals = g.empty((c.n, c.k), torch.bfloat16)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert moe.lib().moe_route(logits.data_ptr(), c.n, c.E, c.k, 0, indx.data_ptr(),
                               vals.data_ptr(), stream) == 0
    meta = {"col_sum": g.empty((c.E,), torch.int32), "offs": g.empty((c.E + 1,), torch.int32),
            "col_sorted": g.empty((N,), torch.int32), "row_sorted": g.empty((N,), torch.int32),
            "gate_scal": g.empty((N,), torch.bfloat16)}
    moe.build_metadata(indx, vals, c.E, ws, meta=meta)
    y_flat = g.empty((N, c.H), torch.bfloat16)
    moe.grouped_ffn(x, meta, w13, w2, c.k, ws, params, y_flat=y_flat)
    out = g.empty((c.n, c.H), torch.bfloat16)
    moe.combine(y_flat, c.n, c.k, out=out)
    g.check()
    assert moe.read_status(ws) == 0
    ref = oracle.ffn(h["x"], indx.cpu().numpy(), host_bits(vals), h["w13"], h["w2"],
                     act=c.act, layout=c.layout)
    assert_layer_close(host_bits(out), ref, c.name)
