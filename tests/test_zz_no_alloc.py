"""The scratch-free GEMV entry point (ggq_mul_mat_vec_noalloc).

Some callers cannot allocate device memory: code running inside a CUDA graph
capture that forbids cudaMalloc, plugins whose host framework owns every
device byte through its own allocator, and serving processes whose HBM is
split up front with no allocation allowed on the request path.  This entry
point keeps its quantized activations in a fixed array inside the library
instead of a context's pool.  Its output must match the oracle at the
tolerance every GEMV test uses, and the pooled entry point (ggq_mul_mat_vec)
within the same tolerance, on calls in a row: each later call finds the
previous call's data in the shared array.  Kept in a file of its own that
pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import ggq_synth as syn
import oracle as orc
from tests.gpu_util import RTOL_ABS, check_outputs, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quant_ggq_gb300 as ggq  # noqa: E402

CALLS = [  # (fmt, N, K, T), run one after the other
    ("Q4_K", 300, 4096, 8),
    ("Q4_K", 16 * 9 + 5, 4096, 1),  # one token: activations held in registers
    ("Q6_K", 16 * 7 + 3, 2048, 4),
    ("MXFP4", 16 * 5 + 9, 4096, 2),   # two tokens: both in registers, warp pairs split the units
    ("Q6_K", 16 * 7 + 3, 3072, 2),
    ("Q5_K", 61, 1024, 1),
    ("Q4_0", 77, 1024, 3),
    ("Q8_0", 37, 14336, 2),         # rows too long for whole-row stages: row chunks
    ("Q2_K", 16 * 6 + 1, 4096, 3),
    ("Q3_K", 45, 2048, 1),
]


def test_noalloc_gemv_matches_oracle_and_pooled_entry_point():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gguf_block_quant_ggq_gb300 import _build
    _build.build()
    lib = ggq.load()
    ctx = ggq.Context(0)
    try:
        for call, (fmt, N, K, T) in enumerate(CALLS):
            W = syn.weights(fmt, N, K, syn.rng(70, call))
            x = syn.activations(T, K, syn.rng(70, 10 + call))
            dW, dx = to_dev(W), to_dev(x)
            y_pool = to_host(ctx.mul_mat_vec(fmt, dW, N, K, dx)).astype(np.float64)
            y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            st = lib.ggq_mul_mat_vec_noalloc(ggq.TYPE[fmt], dW.data_ptr(), N, K, dx.data_ptr(), T, y.data_ptr(),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == 0, ggq.STATUS.get(st, st)
            torch.cuda.synchronize()
            y = to_host(y).astype(np.float64)
            ref, absdot = orc.gemv_dequant(fmt, W, N, K, orc.quantize(orc.act_type(fmt), x), T)
            assert np.all(np.isfinite(y)), f"call {call} ({fmt}) left rows unwritten"
            check_outputs(y, ref, absdot, f"noalloc call {call} ({fmt} N={N} K={K} T={T})")
            assert np.all(np.abs(y - y_pool) <= 2 * RTOL_ABS * absdot), f"call {call} ({fmt}) differs from the pooled call"
        # beyond the fixed array: refused before any launch, Y untouched
        big = torch.zeros((8, 32768), dtype=torch.float32, device="cuda")
        yb = torch.full((8, 16), 7.0, dtype=torch.float32, device="cuda")
        Wb = to_dev(syn.weights("Q4_K", 16, 32768, syn.rng(70, 99)))
        st = lib.ggq_mul_mat_vec_noalloc(ggq.TYPE["Q4_K"], Wb.data_ptr(), 16, 32768, big.data_ptr(), 8,
                                         yb.data_ptr(), None)
        assert st == 6  # GGQ_ERR_CAPACITY
        torch.cuda.synchronize()
        assert bool(torch.all(yb == 7.0))
    finally:
        ctx.close()
