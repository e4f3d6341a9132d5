"""GPU parity of the quantizers, the dequantizer, the integer block dots and the
decode GEMV (ggq_mul_mat_vec / _q / ggq_block_dots) against the CPU oracle.

Bars: quantized activation bytes and per-block int32 coefficients bit-exact;
fp32 outputs within 1e-5 * sum |w x| per output and NMSE <= 1e-10."""
import numpy as np
import pytest

import ggq_synth as syn
import oracle as orc
from tests.gpu_util import check_outputs, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quant_ggq_gb300 as ggq  # noqa: E402

FORMATS = list(syn.WEIGHT_FORMATS)


@pytest.fixture(scope="module")
def ctx():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gguf_block_quant_ggq_gb300 import _build
    _build.build()
    orc.set_threads(__import__("os").cpu_count() or 1)
    c = ggq.Context(0)
    yield c
    c.close()


def _acts(T, K, seed, scale=1.0):
    g = syn.rng(50, seed)
    x = syn.activations(T, K, g) * np.float32(scale)
    if T > 1:
        x[1, :32] = 0.0                       # an all-zero Q8_1 block
        x[-1, 40:48] = np.float32(2.5)        # exact ties of |x| = amax
    return x.astype(np.float32)


@pytest.mark.parametrize("act,K,T", [("Q8_1", 4096, 3), ("Q8_1", 32, 1), ("Q8_K", 4096, 8), ("Q8_K", 256, 5),
                                     ("Q8_K", 768, 2)])
def test_quantize_act_bytes_bit_exact(ctx, act, K, T):
    for scale in (1.0, 1e-3, 300.0):
        x = _acts(T, K, K + T, scale)
        got = to_host(ctx.quantize_act(act, to_dev(x)))
        ref = orc.quantize(act, x)
        assert np.array_equal(got, ref), f"{act}: {np.count_nonzero(got != ref)} bytes differ"


@pytest.mark.parametrize("fmt", FORMATS)
def test_dequant_matches_oracle(ctx, fmt):
    K = 512 if syn.BLOCK_ELEMS[fmt] == 256 else 96
    rows = 37
    W = syn.weights(fmt, rows, K, syn.rng(51, FORMATS.index(fmt)))
    got = to_host(ctx.dequant(fmt, to_dev(W), rows, K)).astype(np.float64)
    ref = orc.dequant(fmt, W, rows, K)
    # fp32 products of exact fp16/int fields: relative error of one or two roundings
    assert np.all(np.abs(got - ref) <= 3e-7 * (np.abs(ref) + 1e-30) + 1e-12 * np.abs(ref).max())


def _case(fmt, N, K, T, seed):
    g = syn.rng(52, seed)
    W = syn.weights(fmt, N, K, g)
    x = _acts(T, K, seed)
    return W, x


SHAPES = [  # (N, K, T): several 16-row tiles with a ragged tail; one and several superblocks
    (16 * 9 + 5, 1024, 1), (16 * 9 + 5, 1024, 2), (101, 512, 3), (67, 2048, 4), (33, 768, 5), (16 * 20 + 7, 1024, 8),
    (1, 256, 1), (17, 4096, 6), (50, 256, 7),
    (16 * 11 + 3, 1024, 3), (40, 2048, 5), (16 * 9 + 9, 3072, 7),
    (37, 8192, 3), (16 * 5 + 3, 8192, 8),  # K beyond the tensor-path GEMV: the grouped int8 kernel
    # two tokens above 32 units a row: warp pairs split the units (K = 3072: the odd warp's
    # upper 16 lanes idle); 16 * 7 + 3 rows leave the last tile's second warp pair a row alone
    (16 * 7 + 3, 4096, 2), (45, 3072, 2),
]
Q4_0_ODD_SHAPES = [(21, 96, 2), (40, 32, 1), (35, 160, 8)]  # K % 64 == 32: a half 64-weight unit per row


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N,K,T", SHAPES)
def test_block_dots_bit_exact_and_gemv_within_tolerance(ctx, fmt, N, K, T):
    W, x = _case(fmt, N, K, T, N * 31 + K + T + FORMATS.index(fmt))
    act = orc.act_type(fmt)
    xq = orc.quantize(act, x)
    dW, dxq = to_dev(W), to_dev(xq)
    # integer core
    coefs = to_host(ctx.block_dots(fmt, dW, N, K, dxq, T))
    ref_coefs = orc.gemv_coefs(fmt, W, N, K, xq, T)
    assert np.array_equal(coefs, ref_coefs), f"{np.count_nonzero(coefs != ref_coefs)} coefficients differ"
    # prequantized GEMV and the full call (quantize inside)
    ref, absdot = orc.gemv_dequant(fmt, W, N, K, xq, T)
    y_q = to_host(ctx.mul_mat_vec_q(fmt, dW, N, K, dxq, T))
    check_outputs(y_q, ref, absdot, f"{fmt} mul_mat_vec_q N={N} K={K} T={T}")
    y = to_host(ctx.mul_mat_vec(fmt, dW, N, K, to_dev(x)))
    check_outputs(y, ref, absdot, f"{fmt} mul_mat_vec N={N} K={K} T={T}")


def _extreme_block(fmt, sign):
    """One block of the largest integer products the format allows: every code
    at its extreme, every 6-bit scale and min 63 (K-quants), scales 127 or -128
    (Q6_K), fp16 scale 1.  With activations of one sign at +-127 each integer
    dot reaches its bound (e.g. Q4_K: 256 * 945 * 127 > 2^24 per superblock)."""
    bb = syn.BLOCK_BYTES[fmt]
    b = np.zeros(bb, np.uint8)
    one = np.array([1.0], np.float16).view(np.uint8)
    if fmt == "Q4_0":
        b[0:2], b[2:] = one, 0xFF if sign > 0 else 0x00
    elif fmt == "Q8_0":
        b[0:2], b[2:] = one, (0x7F if sign > 0 else 0x80)
    elif fmt == "MXFP4":
        b[0], b[1:] = 127, (0x77 if sign > 0 else 0xFF)  # E2M1 codes 7 (6.0) or 15 (-6.0)
    elif fmt in ("Q4_K", "Q5_K"):
        b[0:2], b[2:4], b[4:] = one, np.array([0.0], np.float16).view(np.uint8), 0xFF
    elif fmt == "Q6_K":
        b[0:192] = 0xFF if sign > 0 else 0x00  # codes 63 (31 after the offset) or 0 (-32)
        b[192:208] = 127
        b[208:210] = one
    elif fmt == "Q2_K":
        b[0:16] = 0xFF  # scale 15, min 15 in every group
        b[16:80] = 0xFF  # every 2-bit code 3
        b[80:82], b[82:84] = one, one
    elif fmt == "Q3_K":
        b[0:32] = 0xFF if sign > 0 else 0x00  # high bits: codes 3 or -4 (with low bits 3 / 0)
        b[32:96] = 0xFF if sign > 0 else 0x00
        b[96:108] = 0x00  # every 6-bit scale 0: signed scale -32, the largest magnitude
        b[108:110] = one
    return b


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("T", [1, 2, 3, 8])
def test_block_dots_exact_at_the_integer_bounds(ctx, fmt, T):
    """Blocks at the formats' extremes against activations quantized to +-127:
    the largest integer sums the kernels' accumulators can meet.  The tensor
    paths hold them in f32 chains short enough to stay exact (below 2^24), so
    the dumped coefficients equal the oracle's integers bit for bit."""
    K = 8192 if T == 3 else 4096  # T = 3 at K = 8192 takes the grouped int8 kernel
    N = 35
    W = np.stack([np.tile(_extreme_block(fmt, 1 if (r % 3) else -1), K // syn.BLOCK_ELEMS[fmt]) for r in range(N)])
    x = np.full((T, K), 3.0, np.float32)
    x[:, 1::7] = -3.0  # a few negatives: mixed signs inside blocks, still quantized to +-127
    if T > 1:
        x[1] = 5.0  # one token of a single sign: the bound itself
    xq = orc.quantize(orc.act_type(fmt), x)
    dW, dxq = to_dev(W), to_dev(xq)
    coefs = to_host(ctx.block_dots(fmt, dW, N, K, dxq, T))
    ref_coefs = orc.gemv_coefs(fmt, W, N, K, xq, T)
    assert np.array_equal(coefs, ref_coefs), f"{np.count_nonzero(coefs != ref_coefs)} coefficients differ"
    ref, absdot = orc.gemv_dequant(fmt, W, N, K, xq, T)
    check_outputs(to_host(ctx.mul_mat_vec_q(fmt, dW, N, K, dxq, T)), ref, absdot, f"{fmt} extremes T={T}")


Q8_0_ACT_CASES = [  # (fmt, N, K, T): Q8_0 activation blocks (Q4_0 x Q8_0, Q8_0 x Q8_0)
    ("Q4_0", 16 * 9 + 5, 1024, 1), ("Q4_0", 21, 96, 2), ("Q4_0", 35, 160, 8), ("Q4_0", 77, 4096, 3),
    ("Q8_0", 16 * 9 + 5, 1024, 1), ("Q8_0", 40, 4096, 2), ("Q8_0", 33, 768, 5), ("Q8_0", 16 * 20 + 7, 2048, 8),
    ("Q8_0", 37, 14336, 2),  # rows streamed in chunks
    ("Q4_0", 21, 16384, 1),
]


@pytest.mark.parametrize("fmt,N,K,T", Q8_0_ACT_CASES)
def test_q8_0_activations_bit_exact_and_within_tolerance(ctx, fmt, N, K, T):
    """The Q8_0 activation quantizer (bytes bit-exact) and the Q4_0 x Q8_0 /
    Q8_0 x Q8_0 GEMV: per-block int32 coefficients bit-exact, outputs within
    the fp32 tolerance of the oracle."""
    W, x = _case(fmt, N, K, T, 3 * N + K + T + 11)
    xq = orc.quantize("Q8_0", x)
    got = to_host(ctx.quantize_act("Q8_0", to_dev(x)))
    assert np.array_equal(got, xq), f"{np.count_nonzero(got != xq)} Q8_0 activation bytes differ"
    dW, dxq = to_dev(W), to_dev(xq)
    if K <= 4096:  # the dump stages whole rows (long rows stream in chunks only for the GEMV)
        coefs = to_host(ctx.block_dots_qa(fmt, "Q8_0", dW, N, K, dxq, T))
        assert np.array_equal(coefs, orc.gemv_coefs(fmt, W, N, K, xq, T, act="Q8_0"))
    ref, absdot = orc.gemv_dequant(fmt, W, N, K, xq, T, act="Q8_0")
    y = to_host(ctx.mul_mat_vec_qa(fmt, "Q8_0", dW, N, K, dxq, T))
    check_outputs(y, ref, absdot, f"{fmt} x Q8_0 N={N} K={K} T={T}")
    ctx.sync_status()


def test_unsupported_activation_pairings_are_refused(ctx):
    W = to_dev(syn.weights("Q4_K", 16, 256, syn.rng(57, 0)))
    xq = to_dev(orc.quantize("Q8_0", syn.activations(1, 256, syn.rng(57, 1))))
    with pytest.raises(ggq.GGQError, match="UNSUPPORTED"):
        ctx.mul_mat_vec_qa("Q4_K", "Q8_0", W, 16, 256, xq, 1)
    assert ggq.supported("Q8_0", "Q8_0", "mul_mat_vec") and ggq.supported("Q4_0", "Q8_0", "mul_mat_vec")
    assert not ggq.supported("Q4_K", "Q8_0", "mul_mat_vec") and ggq.supported("Q4_0", "Q8_0", "quantize_act")


LONG_ROWS = [  # (fmt, N, K, T): rows too long for whole-row stages, streamed in row chunks
    ("Q8_0", 16 * 160 + 7, 14336, 1),  # more tiles than SMs (a CTA streams several), ragged tail
    ("Q8_0", 37, 14336, 2),
    ("Q8_0", 45, 14336, 8),            # 28 chunks per tile: the ring wraps many times
    ("Q4_K", 45, 28672, 1),
    ("Q4_K", 29, 28672, 4),
    ("Q6_K", 16 * 160 + 3, 14336, 1),  # 8-superblock chunks
    ("Q5_K", 53, 14336, 3),
    ("Q4_0", 21, 16384, 1),
    ("MXFP4", 40, 16384, 2),
    ("Q2_K", 16 * 40 + 9, 28672, 1),   # 4-superblock chunks
    ("Q3_K", 37, 28672, 2),            # 8-superblock chunks
    # rows that are not 16-byte multiples: chunk ends copied byte by byte
    ("Q2_K", 35, 26368, 1),            # 103 superblocks: 8652-byte rows
    ("Q3_K", 16 * 9 + 7, 26368, 3),    # 11330-byte rows
    ("Q6_K", 16 * 9 + 7, 18944, 1),    # 74 superblocks: 15540-byte rows
    ("Q6_K", 35, 18944, 4),
    ("MXFP4", 40, 23296, 2),           # 12376-byte rows
    # the staged activations of all tokens do not fit: tokens run in groups
    ("Q4_K", 29, 28672, 8),            # 4 + 4
    ("Q6_K", 35, 18944, 8),
    ("MXFP4", 40, 23296, 7),           # 3 + 4
]


@pytest.mark.parametrize("fmt,N,K,T", LONG_ROWS)
def test_long_rows_stream_in_chunks(ctx, fmt, N, K, T):
    W, x = _case(fmt, N, K, T, N + K + T + FORMATS.index(fmt))
    xq = orc.quantize(orc.act_type(fmt), x)
    dW = to_dev(W)
    ref, absdot = orc.gemv_dequant(fmt, W, N, K, xq, T)
    y_q = to_host(ctx.mul_mat_vec_q(fmt, dW, N, K, to_dev(xq), T))
    check_outputs(y_q, ref, absdot, f"{fmt} long rows mul_mat_vec_q N={N} K={K} T={T}")
    y = to_host(ctx.mul_mat_vec(fmt, dW, N, K, to_dev(x)))
    check_outputs(y, ref, absdot, f"{fmt} long rows mul_mat_vec N={N} K={K} T={T}")
    ctx.sync_status()


def test_rows_too_long_for_one_token_are_refused(ctx):
    # one token's staged activations (about 1.52 bytes per input) plus two
    # chunked stages no longer fit in one SM's shared memory beyond K = 146432
    K, T = 147456, 1
    W = to_dev(syn.weights("Q8_0", 16, K, syn.rng(56, 0)))
    xq = to_dev(orc.quantize("Q8_K", syn.activations(T, K, syn.rng(56, 1))))
    with pytest.raises(ggq.GGQError, match="SHAPE"):
        ctx.mul_mat_vec_q("Q8_0", W, 16, K, xq, T)
    ctx.sync_status()


@pytest.mark.parametrize("N,K,T", Q4_0_ODD_SHAPES)
def test_q4_0_widths_with_a_half_unit(ctx, N, K, T):
    W, x = _case("Q4_0", N, K, T, 7 * N + K)
    xq = orc.quantize("Q8_1", x)
    dW, dxq = to_dev(W), to_dev(xq)
    assert np.array_equal(to_host(ctx.block_dots("Q4_0", dW, N, K, dxq, T)), orc.gemv_coefs("Q4_0", W, N, K, xq, T))
    ref, absdot = orc.gemv_dequant("Q4_0", W, N, K, xq, T)
    check_outputs(to_host(ctx.mul_mat_vec("Q4_0", dW, N, K, to_dev(x))), ref, absdot, f"Q4_0 N={N} K={K} T={T}")


def test_q4_0_workload_1024x4096(ctx):
    cfg = syn.GEMV_Q4_0
    g = syn.rng(cfg["index"], 0)
    W = syn.weights("Q4_0", cfg["N"], cfg["K"], g)
    x = syn.activations(1, cfg["K"], syn.rng(cfg["index"], 1))
    xq = orc.quantize("Q8_1", x)
    ref, absdot = orc.gemv_dequant("Q4_0", W, cfg["N"], cfg["K"], xq, 1)
    y = to_host(ctx.mul_mat_vec("Q4_0", to_dev(W), cfg["N"], cfg["K"], to_dev(x)))
    check_outputs(y, ref, absdot, "Q4_0 1024x4096")
    assert np.array_equal(to_host(ctx.quantize_act("Q8_1", to_dev(x))), xq)


@pytest.mark.parametrize("fmt", ["Q8_0", "Q4_K", "Q5_K", "Q6_K", "Q2_K", "Q3_K"])
def test_full_size_14336x4096_sampled_rows(ctx, fmt):
    """Full workload size in the bench's launch configuration (T = 8, 2 and 1);
    the oracle computes a sample of rows one by one, including both ends."""
    cfg = syn.GEMV_KQUANT
    N, K = cfg["N"], cfg["K"]
    W = syn.weights(fmt, N, K, syn.rng(cfg["index"], FORMATS.index(fmt)))
    dW = to_dev(W)
    rows = np.unique(np.concatenate([[0, 1, 15, 16, N - 17, N - 1], syn.rng(53, 0).integers(0, N, 58)]))
    for T in (8, 2, 1):
        x = syn.activations(T, K, syn.rng(cfg["index"], 100 + T))
        y = to_host(ctx.mul_mat_vec(fmt, dW, N, K, to_dev(x)))
        xq = orc.quantize("Q8_K", x)
        Ws = np.ascontiguousarray(W[rows])
        ref, absdot = orc.gemv_dequant(fmt, Ws, len(rows), K, xq, T)
        check_outputs(y[:, rows], ref, absdot, f"{fmt} full-size sampled T={T}")
        assert np.all(np.isfinite(y))


def test_errors_are_refused_loudly(ctx):
    W = to_dev(syn.weights("Q4_K", 16, 256, syn.rng(54, 0)))
    x = to_dev(np.zeros((9, 256), np.float32))
    with pytest.raises(ggq.GGQError, match="SHAPE"):
        ctx.mul_mat_vec("Q4_K", W, 16, 256, x)  # T = 9
    with pytest.raises(ggq.GGQError, match="SHAPE"):
        ctx.mul_mat_vec("Q4_K", W, 16, 255, x[:1])
    with pytest.raises(KeyError):
        ctx.mul_mat_vec("IQ2_XXS", W, 16, 256, x[:1])
    h = ggq.load()
    y = torch.empty((1, 16), dtype=torch.float32, device="cuda")
    st = h.ggq_mul_mat_vec(ctx.handle, 16, W.data_ptr(), 16, 256, x.data_ptr(), 1, y.data_ptr(), None)  # IQ2_XXS
    assert st == 3 and b"supported" in h.ggq_last_error(ctx.handle)
    fresh = ggq.Context(0)
    try:  # no reserve yet: the call refuses instead of allocating
        st = h.ggq_mul_mat_vec(fresh.handle, 12, W.data_ptr(), 16, 256, x.data_ptr(), 1, y.data_ptr(), None)
        assert st == 6
    finally:
        fresh.close()
    ctx.sync_status()


def test_empty_inputs(ctx):
    """Empty quantize/dequant calls are no-ops (NULL pointers allowed); the
    GEMV, whose contract is 1 <= T <= 8 and N >= 1, refuses T = 0 and N = 0."""
    h = ggq.load()
    Q8_1, Q8_K, Q4_K = ggq.TYPE["Q8_1"], ggq.TYPE["Q8_K"], ggq.TYPE["Q4_K"]
    assert h.ggq_quantize_act(ctx.handle, Q8_K, None, 0, 4096, None, None) == 0
    assert h.ggq_quantize_act(ctx.handle, Q8_1, None, 3, 0, None, None) == 0
    assert h.ggq_dequant(ctx.handle, Q4_K, None, 0, 256, None, None) == 0
    # an empty call writes nothing: a sentinel-filled buffer stays as it was
    out = torch.full((4, 292), 7, dtype=torch.uint8, device="cuda")
    x = to_dev(np.ones((1, 256), np.float32))
    assert h.ggq_quantize_act(ctx.handle, Q8_K, x.data_ptr(), 0, 256, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert bool(torch.all(out == 7))
    W = to_dev(syn.weights("Q4_K", 16, 256, syn.rng(55, 0)))
    y = torch.empty((1, 16), dtype=torch.float32, device="cuda")
    assert h.ggq_mul_mat_vec(ctx.handle, Q4_K, W.data_ptr(), 16, 256, x.data_ptr(), 0, y.data_ptr(), None) == 2
    assert h.ggq_mul_mat_vec(ctx.handle, Q4_K, W.data_ptr(), 0, 256, x.data_ptr(), 1, y.data_ptr(), None) == 2
    ctx.sync_status()

