"""Capture safety of the public calls (ggq.h: after ggq_reserve no call
allocates or synchronises, so a decode step can be captured in a CUDA graph;
ggq_reserve refuses to grow the pool while its stream is capturing).

The calls are captured once, replayed, and the replay must reproduce the eager
results bit for bit (same kernels, same launch parameters, no atomics in any
result); replaying after new inputs are copied in place must follow them.
"""
import numpy as np
import pytest

import ggq_synth as syn
from tests.gpu_util import to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quant_ggq_gb300 as ggq  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gguf_block_quant_ggq_gb300 import _build
    _build.build()
    c = ggq.Context(0)
    yield c
    c.close()


def _step(ctx, w8, cfg, E, inputs, outs):
    """One decode-like step through the public calls."""
    W, N, K = inputs["W"], inputs["N"], inputs["K"]
    ctx.quantize_act("Q8_K", inputs["x4"], out=outs["xq4"])
    ctx.mul_mat_vec_q("Q4_K", W, N, K, outs["xq4"], 4, Y=outs["y4"])
    ctx.mul_mat_vec("Q4_K", W, N, K, inputs["x1"], Y=outs["y1"])
    H, I, k = cfg["H"], cfg["I"], cfg["k"]
    for T in (1, 3, 8):  # one token, the direct route, expert-sorted tiles
        ctx.moe_experts(w8, E, H, I, k, inputs[f"mx{T}"], logits=inputs[f"lg{T}"], Y=outs[f"my{T}"])


def _inputs(cfg, E, seed):
    g = syn.rng(80, seed)
    N, K, H = 300, 1024, cfg["H"]
    d = {"N": N, "K": K,
         "x4": to_dev(syn.activations(4, K, g)), "x1": to_dev(syn.activations(1, K, g))}
    for T in (1, 3, 8):
        d[f"mx{T}"] = to_dev(syn.activations(T, H, g))
        d[f"lg{T}"] = to_dev(syn.router_logits(T, E, g))
    return d


def test_public_calls_replay_from_a_graph_bit_identically(ctx):
    cfg, E = syn.MOE_DECODE, 16
    H, I, k = cfg["H"], cfg["I"], cfg["k"]
    g = syn.rng(80, 100)
    banks = [to_dev(syn.expert_bank(cfg[n], E, r, c, g)) for n, r, c in (("gate", I, H), ("up", I, H), ("down", H, I))]
    w8 = ctx.moe_weights(cfg["gate"], banks[0], cfg["up"], banks[1], cfg["down"], banks[2])
    W = to_dev(syn.weights("Q4_K", 300, 1024, g))
    ctx.reserve(max_tokens=8, max_k=1024)
    ctx.reserve(max_tokens=8, n_experts=E, hidden=H, inter=I, top_k=k)
    inp = _inputs(cfg, E, 0)
    inp["W"] = W
    outs = {"xq4": torch.empty((4, syn.row_bytes("Q8_K", 1024)), dtype=torch.uint8, device="cuda"),
            "y4": torch.empty((4, 300), dtype=torch.float32, device="cuda"),
            "y1": torch.empty((1, 300), dtype=torch.float32, device="cuda")}
    for T in (1, 3, 8):
        outs[f"my{T}"] = torch.empty((T, H), dtype=torch.float32, device="cuda")

    # eager reference
    _step(ctx, w8, cfg, E, inp, outs)
    torch.cuda.synchronize()
    ctx.sync_status()
    eager = {n: to_host(t).copy() for n, t in outs.items()}

    # capture once, then replay
    for t in outs.values():
        t.fill_(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        _step(ctx, w8, cfg, E, inp, outs)
    graph.replay()
    torch.cuda.synchronize()
    ctx.sync_status()
    for n, ref in eager.items():
        assert np.array_equal(to_host(outs[n]), ref), f"{n}: graph replay differs from the eager call"

    # new inputs copied in place: the replay follows them
    new = _inputs(cfg, E, 1)
    for n in ("x4", "x1", "mx1", "mx3", "mx8", "lg1", "lg3", "lg8"):
        inp[n].copy_(new[n])
    graph.replay()
    torch.cuda.synchronize()
    ctx.sync_status()
    replayed = {n: to_host(t).copy() for n, t in outs.items()}
    _step(ctx, w8, cfg, E, inp, outs)
    torch.cuda.synchronize()
    ctx.sync_status()
    for n, got in replayed.items():
        assert np.array_equal(got, to_host(outs[n])), f"{n}: replay on new inputs differs from the eager call"
        assert not np.array_equal(got, eager[n]), f"{n}: replay did not follow the new inputs"


def test_reserve_refuses_to_grow_while_capturing():
    fresh = ggq.Context(0)
    try:
        fresh.reserve(max_tokens=1, max_k=256)
        before = fresh.scratch_bytes()
        lib = ggq.load()
        side = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        statuses = []
        with torch.cuda.graph(graph, stream=side):
            # a plan that fits is a no-op; one that needs a larger pool is refused, not allocated
            small = ggq.ggq_plan(1, 256, 0, 0, 0, 0)
            large = ggq.ggq_plan(8, 65536, 0, 0, 0, 0)
            import ctypes
            sh = ctypes.c_void_p(side.cuda_stream)
            statuses.append(lib.ggq_reserve(fresh.handle, ctypes.byref(small), sh))
            statuses.append(lib.ggq_reserve(fresh.handle, ctypes.byref(large), sh))
        assert statuses == [0, 7], statuses  # GGQ_OK, GGQ_ERR_CAPTURE_ALLOC
        assert b"capturing" in lib.ggq_last_error(fresh.handle)
        assert fresh.scratch_bytes() == before
        fresh.reserve(max_tokens=8, max_k=65536)  # outside the capture it grows
        assert fresh.scratch_bytes() > before
    finally:
        fresh.close()
