"""The scratch-free GEMV entry point (ggq_mul_mat_vec_noalloc).

Some callers cannot allocate device memory (graph capture that forbids
cudaMalloc, frameworks that own every device byte, request paths with a fixed
HBM budget), so this entry point keeps its quantized activations in a fixed
array inside the library instead of a context's pool.  Its output must match
the pooled entry point, ggq_mul_mat_vec, within the tolerance every GEMV test
uses, on two calls in a row (the second call finds the first call's data in
the shared array).  Kept in a file of its own that runs last.
"""
import ctypes

import numpy as np
import pytest

import ggq_synth as syn
import oracle as orc
from tests.gpu_util import RTOL_ABS, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quant_ggq_gb300 as ggq  # noqa: E402


def test_noalloc_gemv_matches_pooled_entry_point():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gguf_block_quant_ggq_gb300 import _build
    _build.build()
    lib = ggq.load()
    ctx = ggq.Context(0)
    try:
        # different calls in a row: each overwrites the previous one's scratch; the
        # last has rows too long for whole-row stages (streamed in chunks)
        for call, (fmt, N, K, T) in enumerate([("Q4_K", 300, 4096, 8), ("Q4_0", 77, 1024, 3),
                                               ("Q8_0", 37, 14336, 2)]):
            W = syn.weights(fmt, N, K, syn.rng(70, call))
            x = syn.activations(T, K, syn.rng(70, 10 + call))
            dW, dx = to_dev(W), to_dev(x)
            y_pool = to_host(ctx.mul_mat_vec(fmt, dW, N, K, dx))
            y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            st = lib.ggq_mul_mat_vec_noalloc(ggq.TYPE[fmt], dW.data_ptr(), N, K, dx.data_ptr(), T, y.data_ptr(),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == 0, ggq.STATUS.get(st, st)
            torch.cuda.synchronize()
            y = to_host(y).astype(np.float64)
            _, absdot = orc.gemv_dequant(fmt, W, N, K, orc.quantize(orc.act_type(fmt), x), T)
            assert np.all(np.isfinite(y))
            assert np.all(np.abs(y - y_pool) <= RTOL_ABS * absdot), f"call {call} ({fmt}) differs"
        # beyond the fixed array: refused before any launch
        big = torch.zeros((8, 32768), dtype=torch.float32, device="cuda")
        yb = torch.zeros((8, 16), dtype=torch.float32, device="cuda")
        Wb = to_dev(syn.weights("Q4_K", 16, 32768, syn.rng(70, 99)))
        st = lib.ggq_mul_mat_vec_noalloc(ggq.TYPE["Q4_K"], Wb.data_ptr(), 16, 32768, big.data_ptr(), 8,
                                         yb.data_ptr(), None)
        assert st == 6  # GGQ_ERR_CAPACITY
    finally:
        ctx.close()
