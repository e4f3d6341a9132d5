"""GPU parity of the routed-expert layer (ggq_moe_experts / _routed) against the
CPU oracle, stage by stage and teacher-forced (the GPU's own intermediate is
fed to the oracle's next stage), then end to end.

  (i)   expert ids bit-exact, routing weights to fp32 rounding;
  (ii)  x^ bytes bit-exact; g and u within 1e-5 * sum |w x| and NMSE 1e-10;
        h = silu(g) * u from the GPU's own g, u to a few fp32 ulps;
  (iii) the oracle quantizer on the GPU's fp32 h equals the GPU's Q8_K bytes;
  (iv)  down outputs o within tolerance of the oracle's down on the GPU's h^;
  (v)   y within tolerance of the oracle's combine of (iv);
  and the free-running oracle y, where int8 flips of h^ at fp32 ties are
  counted and the remaining difference bounded.
"""
import numpy as np
import pytest

import ggq_synth as syn
import oracle as orc
from tests.gpu_util import check_outputs, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quant_ggq_gb300 as ggq  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from gguf_block_quant_ggq_gb300 import _build
    _build.build()
    orc.set_threads(__import__("os").cpu_count() or 1)
    c = ggq.Context(0)
    yield c
    c.close()


_BANKS = {}


def _banks(cfg, E):
    key = (cfg["index"], E, cfg["gate"], cfg["up"], cfg["down"])
    if key not in _BANKS:
        g = syn.rng(cfg["index"], 1000 + E)
        H, I = cfg["H"], cfg["I"]
        host = {
            "gate": syn.expert_bank(cfg["gate"], E, I, H, g),
            "up": syn.expert_bank(cfg["up"], E, I, H, g),
            "down": syn.expert_bank(cfg["down"], E, H, I, g),
        }
        _BANKS.clear()
        _BANKS[key] = (host, {k: to_dev(v) for k, v in host.items()})
    return _BANKS[key]


def _ncoef(fmt, K):
    return K // syn.BLOCK_ELEMS[fmt] * orc.coefs_per_block(fmt)


COEF_BYTES_MAX = 1 << 30  # integer-core dumps larger than this are skipped (full-size prefill)


def _dump_buffers(T, k, H, I, cfg=None):
    P = T * k
    z = lambda *s, dt=torch.float32: torch.full(s, -7, dtype=dt, device="cuda")  # noqa: E731
    d = {
        "ids": z(T, k, dt=torch.int32), "weights": z(T, k), "xq": z(T, H // 256 * 292, dt=torch.uint8),
        "g": z(P, I), "u": z(P, I), "h": z(P, I), "hq": z(P, I // 256 * 292, dt=torch.uint8), "o": z(P, H),
    }
    if cfg is not None:
        ng, nd = _ncoef(cfg["gate"], H), _ncoef(cfg["down"], I)
        if 4 * P * (2 * I * ng + H * nd) <= COEF_BYTES_MAX:
            d["coefs_gate"] = z(P, I, ng, dt=torch.int32)
            d["coefs_up"] = z(P, I, ng, dt=torch.int32)
            d["coefs_down"] = z(P, H, nd, dt=torch.int32)
    return d


def _run_and_check(ctx, cfg, E, T, routed=False, seed=0, sample_tokens=None):
    """Run the layer with every dump, then check stage by stage.  With
    sample_tokens, the per-pair oracle checks cover only the pairs of that many
    seeded tokens (routing is per token, so a token's whole layer can be
    recomputed on its own); ids, weights, x^ and h^ are always checked in full."""
    H, I, k = cfg["H"], cfg["I"], cfg["k"]
    host, dev = _banks(cfg, E)
    g = syn.rng(cfg["index"], 2000 + 17 * T + seed)
    x = syn.activations(T, H, g)
    logits = syn.router_logits(T, E, g, cfg.get("zipf"))
    ids_ref, w_ref = orc.router(logits, k)
    w8 = ctx.moe_weights(cfg["gate"], dev["gate"], cfg["up"], dev["up"], cfg["down"], dev["down"])
    d = _dump_buffers(T, k, H, I, cfg)
    if routed:
        y = ctx.moe_experts(w8, E, H, I, k, to_dev(x), ids=to_dev(ids_ref),
                            route_w=to_dev(w_ref.astype(np.float32)), dump=d)
    else:
        y = ctx.moe_experts(w8, E, H, I, k, to_dev(x), logits=to_dev(logits), dump=d)
    ctx.sync_status()
    y = to_host(y).astype(np.float64)
    r = {n: to_host(t) for n, t in d.items()}
    toks = np.arange(T) if sample_tokens is None else np.unique(
        np.concatenate([[0, T - 1], syn.rng(61, T).integers(0, T, sample_tokens)]))

    # (i) routing
    assert np.array_equal(r["ids"], ids_ref)
    assert np.all(np.abs(r["weights"] - w_ref) <= 2e-6 * w_ref + 1e-9)
    # (ii) x^ and gate/up
    xq = orc.quantize("Q8_K", x)
    assert np.array_equal(r["xq"], xq)
    P = T * k
    pairs = np.array([t * k + j for t in toks for j in range(k)])
    coefs = "coefs_gate" in r
    for p in pairs:
        t, e = p // k, int(ids_ref.flat[p])
        if coefs:  # the gate/up kernels' own integer core, bit-exact
            for m in ("gate", "up"):
                cref = orc.gemv_coefs(cfg[m], host[m][e], I, H, xq[t:t + 1], 1)[0]
                assert np.array_equal(r["coefs_" + m][p], cref), \
                    f"{m} pair {p}: {np.count_nonzero(r['coefs_' + m][p] != cref)} integer coefficients differ"
        gref, gabs = orc.gemv_dequant(cfg["gate"], host["gate"][e], I, H, xq[t:t + 1], 1)
        uref, uabs = orc.gemv_dequant(cfg["up"], host["up"][e], I, H, xq[t:t + 1], 1)
        check_outputs(r["g"][p][None], gref, gabs, f"gate pair {p}")
        check_outputs(r["u"][p][None], uref, uabs, f"up pair {p}")
    gg, uu = r["g"][pairs].astype(np.float64), r["u"][pairs].astype(np.float64)
    h64 = gg / (1.0 + np.exp(-gg)) * uu
    assert np.all(np.abs(r["h"][pairs] - h64) <= 6e-7 * np.abs(h64) + 1e-30)
    # (iii) h^ = Q8_K(h) bit-exact on the GPU's own h (every pair)
    assert np.array_equal(orc.quantize("Q8_K", r["h"].astype(np.float32)), r["hq"])
    # (iv) down on the GPU's h^
    o_tf = np.zeros((P, H))
    o_abs = np.zeros((P, H))
    for p in pairs:
        e = int(ids_ref.flat[p])
        if coefs:  # the down kernel's integer core on the GPU's own h^, bit-exact
            cref = orc.gemv_coefs(cfg["down"], host["down"][e], H, I, r["hq"][p:p + 1], 1)[0]
            assert np.array_equal(r["coefs_down"][p], cref), \
                f"down pair {p}: {np.count_nonzero(r['coefs_down'][p] != cref)} integer coefficients differ"
        oref, oabs = orc.gemv_dequant(cfg["down"], host["down"][e], H, I, r["hq"][p:p + 1], 1)
        check_outputs(r["o"][p][None], oref, oabs, f"down pair {p}")
        o_tf[p], o_abs[p] = oref[0], oabs[0]
    # (v) combine
    y_tf = orc.moe_combine(o_tf, w_ref, T, k, H)[toks]
    y_abs = orc.moe_combine(o_abs, w_ref, T, k, H)[toks]
    # routing weights carry fp32 rounding (<= 2e-6 relative): widen the scale by 30 %
    check_outputs(y[toks], y_tf, 1.3 * y_abs, "combine")
    # (v') the same layer without dumps takes the fused down path (no per-pair
    # outputs; partials added straight into the token sums): same h^, same bar
    if routed:
        y2 = ctx.moe_experts(w8, E, H, I, k, to_dev(x), ids=to_dev(ids_ref), route_w=to_dev(w_ref.astype(np.float32)))
    else:
        y2 = ctx.moe_experts(w8, E, H, I, k, to_dev(x), logits=to_dev(logits))
    ctx.sync_status()
    check_outputs(to_host(y2).astype(np.float64)[toks], y_tf, 1.3 * y_abs, "combine (fused down)")
    # (v'') with every dump but the per-pair down outputs, the layer takes the
    # same kernels as without dumps: routing, x^, g, u, h and h^ are
    # bit-identical to the fully dumped run above, and y to the run without dumps
    d3 = {n: t for n, t in _dump_buffers(T, k, H, I).items() if n != "o" and not n.startswith("coefs")}
    if routed:
        y3 = ctx.moe_experts(w8, E, H, I, k, to_dev(x), ids=to_dev(ids_ref), route_w=to_dev(w_ref.astype(np.float32)),
                             dump=d3)
    else:
        y3 = ctx.moe_experts(w8, E, H, I, k, to_dev(x), logits=to_dev(logits), dump=d3)
    ctx.sync_status()
    for n, t in d3.items():
        assert np.array_equal(to_host(t), r[n]), f"{n} differs from the fully dumped run"
    assert np.array_equal(to_host(y3), to_host(y2)), "y differs with and without the dumps"
    # free running against the whole oracle layer on the checked tokens
    ref = orc.moe(cfg["gate"], host["gate"], cfg["up"], host["up"], cfg["down"], host["down"], E, H, I, k,
                  x[toks], logits[toks])
    # The GPU's fp32 h differs from the oracle's double h within the gate/up
    # tolerance, so a few quants sitting at a rounding boundary land on the
    # neighbouring integer.  Every such flip must be a +-1 step of a block whose
    # scale agrees, and the flips must stay rare; the teacher-forced checks above
    # are the acceptance.
    nP = len(pairs)
    gq = r["hq"][pairs].reshape(nP, I // 256, 292)
    oq = ref["hq"].reshape(nP, I // 256, 292)
    d_gpu, d_orc = gq[..., :4].copy().view(np.float32), oq[..., :4].copy().view(np.float32)
    same_d = np.abs(d_gpu - d_orc) <= 1e-5 * np.abs(d_orc)
    qg = gq[..., 4:260].view(np.int8).astype(int)
    qo = oq[..., 4:260].view(np.int8).astype(int)
    diff = np.abs(qg - qo)
    assert np.all(diff[same_d[..., 0]] <= 1), "an h^ quant moved by more than one step"
    flips = int(np.count_nonzero(diff))
    assert flips <= 0.01 * nP * I, f"{flips} of {nP * I} h^ quants differ from the free-running oracle"
    nmse = float(np.sum((y[toks] - ref["y"]) ** 2) / np.sum(ref["y"] ** 2))
    print(f"free-running: {flips} of {nP * I} h^ quants flipped at fp32 ties, NMSE {nmse:.3e}")
    assert nmse <= (1e-10 if flips == 0 else 1e-4), f"free-running NMSE {nmse:.3e} with {flips} flips"
    return flips


@pytest.mark.parametrize("T", [1, 2, 3, 4, 6, 13])
def test_moe_decode_q4k_q6k(ctx, T):
    """The decode layer on the direct route: one launch pair up to 4 tokens,
    calls of at most 4 tokens above (6 = 4 + 2, 13 = 4 + 4 + 4 + 1), every
    dumped array written at its tokens' rows."""
    cfg = syn.MOE_DECODE
    _run_and_check(ctx, cfg, cfg["E"], T)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5])
def test_moe_mxfp4_reduced_bank(ctx, T):
    """MXFP4 experts at full H and I over a 32-expert bank (the routing of the
    256-expert bank is exercised at full size below)."""
    _run_and_check(ctx, syn.MOE_MXFP4, 32, T)


def test_moe_routed_entry_matches(ctx):
    _run_and_check(ctx, syn.MOE_DECODE, syn.MOE_DECODE["E"], 3, routed=True, seed=1)


def test_moe_q8_0_gate_q4k_down_decode(ctx):
    cfg = dict(syn.MOE_PREFILL)
    cfg["E"] = 16
    for T in (1, 4):
        _run_and_check(ctx, cfg, 16, T)


@pytest.mark.parametrize("T", [5, 40])
def test_moe_q8_0_gate_q4k_down_sorted(ctx, T):
    """Expert-sorted route with the prefill formats over a 16-expert bank: Q8_0
    gate/up on the tcgen05 grouped GEMM, Q4_K down on the f16 grouped GEMM."""
    cfg = dict(syn.MOE_PREFILL)
    cfg["E"] = 16
    _run_and_check(ctx, cfg, 16, T, sample_tokens=None if T <= 8 else 6)


def test_moe_q8_0_banks_sorted(ctx):
    """Q8_0 gate/up and Q8_0 down on the expert-sorted route (16 experts): the
    down bank takes the f16 mma.sync grouped GEMM."""
    cfg = dict(syn.MOE_PREFILL)
    cfg["E"] = 16
    cfg["down"] = "Q8_0"
    _run_and_check(ctx, cfg, 16, 24, sample_tokens=6)


@pytest.mark.parametrize("T", [5, 8, 32, 64, 128])
def test_moe_sorted_route_mxfp4(ctx, T):
    """MXFP4 over a 32-expert bank: 5 and 8 tokens as direct-route calls of 4
    tokens (pairs <= 2 E), 32 and up on expert-sorted tiles, on the grouped
    int8 tensor-core kernel below 16 (token, expert) pairs per expert (T = 32)
    and on the tcgen05 grouped GEMM with bf16 operands from there (64, 128)."""
    _run_and_check(ctx, syn.MOE_MXFP4, 32, T, sample_tokens=None if T <= 8 else 6)


def test_moe_q5k_banks_sorted(ctx):
    """Q5_K gate/up and down on the expert-sorted route (grouped int8 kernel)."""
    cfg = dict(syn.MOE_DECODE)
    cfg.update(E=16, gate="Q5_K", up="Q5_K", down="Q5_K")
    _run_and_check(ctx, cfg, 16, 12, sample_tokens=5)


@pytest.mark.parametrize("T,dmax", [(5, 32), (16, 32), (5, 4), (16, 4), (40, 32)])
def test_moe_sorted_route_q4k_q6k(ctx, T, dmax):
    """The 128-expert decode layer above 4 tokens: calls of 4 tokens on the
    direct route at 5 and 16 tokens by default, expert-sorted tiles with the
    direct route held to 4 tokens (the ds4 page's split) and at 40 (pairs > 2 E)."""
    ctx.set_direct_route_max_tokens(dmax)
    try:
        _sorted_q4k_q6k(ctx, T)
    finally:
        ctx.set_direct_route_max_tokens(32)


def _sorted_q4k_q6k(ctx, T):
    cfg = syn.MOE_DECODE
    _run_and_check(ctx, cfg, cfg["E"], T, sample_tokens=None if T <= 8 else 6)


def test_moe_sorted_route_routed_entry(ctx):
    _run_and_check(ctx, syn.MOE_MXFP4, 32, 9, routed=True, seed=3)


def test_moe_prefill_4096_tokens_zipf(ctx):
    """The prefill workload at full size: 4096 tokens, 128 experts, Zipf(1.1)
    expert bias, Q8_0 gate/up and Q4_K down; sampled tokens against the oracle."""
    cfg = syn.MOE_PREFILL
    _run_and_check(ctx, cfg, cfg["E"], cfg["T"][0], sample_tokens=5)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 32, 128, 512])
def test_moe_mxfp4_full_bank_256_experts(ctx, T):
    """The MXFP4 workload at full size (256 experts, H 4096, I 2048, top-8) at
    every token count it names: 1-4 on the direct route, 5 and 32 as direct
    calls of 4 tokens, 128 and 512 on expert-sorted tiles; larger counts check
    the pairs of sampled tokens."""
    cfg = syn.MOE_MXFP4
    _run_and_check(ctx, cfg, cfg["E"], T, sample_tokens=None if T <= 5 else 6)


@pytest.mark.parametrize("T", [5, 32])
def test_moe_mxfp4_full_bank_sorted_tiles(ctx, T):
    """The MXFP4 workload at 5 and 32 tokens on the route it names, expert-sorted
    tiles (the direct route held to 4 tokens)."""
    cfg = syn.MOE_MXFP4
    ctx.set_direct_route_max_tokens(4)
    try:
        _run_and_check(ctx, cfg, cfg["E"], T, sample_tokens=None if T <= 5 else 6)
    finally:
        ctx.set_direct_route_max_tokens(32)


def test_direct_route_limit_is_checked(ctx):
    for bad in (3, 33, 0):
        with pytest.raises(ggq.GGQError, match="INVALID_ARG"):
            ctx.set_direct_route_max_tokens(bad)
    ctx.set_direct_route_max_tokens(32)


def test_moe_all_experts_uniform_equals_dense(ctx):
    """top_k = E with equal logits: uniform weights 1/E, every expert used."""
    cfg = dict(syn.MOE_DECODE)
    E, H, I = 8, 512, 256
    cfg.update(E=E, H=H, I=I, k=8)
    g = syn.rng(60, 0)
    gate = syn.expert_bank("Q4_K", E, I, H, g)
    up = syn.expert_bank("Q4_K", E, I, H, g)
    down = syn.expert_bank("Q6_K", E, H, I, g)
    x = syn.activations(2, H, g)
    logits = np.zeros((2, E), np.float32)
    banks = [to_dev(gate), to_dev(up), to_dev(down)]  # keep the device copies alive: the struct holds raw pointers
    w8 = ctx.moe_weights("Q4_K", banks[0], "Q4_K", banks[1], "Q6_K", banks[2])
    d = _dump_buffers(2, E, H, I)
    y = to_host(ctx.moe_experts(w8, E, H, I, E, to_dev(x), logits=to_dev(logits), dump=d)).astype(np.float64)
    assert np.array_equal(to_host(d["ids"]), np.tile(np.arange(E, dtype=np.int32), (2, 1)))
    assert np.allclose(to_host(d["weights"]), 1.0 / E, rtol=1e-6, atol=0)
    ref = orc.moe("Q4_K", gate, "Q4_K", up, "Q6_K", down, E, H, I, E, x, logits)
    assert np.sum((y - ref["y"]) ** 2) / np.sum(ref["y"] ** 2) <= 1e-4


@pytest.mark.parametrize("T", [1, 3, 8, 40])
def test_moe_prequantized_entry_is_bit_identical(ctx, T):
    """ggq_moe_experts_q on x^ from ggq_quantize_act gives the very bytes of
    ggq_moe_experts on x (the same kernels take the same x^), on the direct
    route (1 and 3 tokens, 8 as two calls of 4) and on expert-sorted tiles (40)."""
    cfg = syn.MOE_DECODE
    E, H, I, k = cfg["E"], cfg["H"], cfg["I"], cfg["k"]
    host, dev = _banks(cfg, E)
    w8 = ctx.moe_weights(cfg["gate"], dev["gate"], cfg["up"], dev["up"], cfg["down"], dev["down"])
    g = syn.rng(cfg["index"], 5000 + T)
    x = to_dev(syn.activations(T, H, g))
    lg = to_dev(syn.router_logits(T, E, g))
    y = to_host(ctx.moe_experts(w8, E, H, I, k, x, logits=lg))
    xq = ctx.quantize_act("Q8_K", x)
    d = {"xq": torch.full((T, H // 256 * 292), 7, dtype=torch.uint8, device="cuda")}
    yq = to_host(ctx.moe_experts_q(w8, E, H, I, k, xq, lg, dump=d))
    ctx.sync_status()
    assert np.array_equal(yq, y)
    assert np.array_equal(to_host(d["xq"]), to_host(xq))


def test_moe_expert_load_counters(ctx):
    """Expert-load telemetry: pairs per expert, calls and distinct experts per
    call, accumulated on the device over direct-route and expert-sorted calls,
    against the oracle's routing of the same logits."""
    cfg = syn.MOE_DECODE
    E, H, I, k = cfg["E"], cfg["H"], cfg["I"], cfg["k"]
    host, dev = _banks(cfg, E)
    w8 = ctx.moe_weights(cfg["gate"], dev["gate"], cfg["up"], dev["up"], cfg["down"], dev["down"])
    pairs = torch.zeros(E, dtype=torch.int64, device="cuda")
    calls = torch.zeros(2, dtype=torch.int64, device="cuda")
    ctx.set_moe_counters(pairs, calls)
    want_pairs = np.zeros(E, np.int64)
    want_calls = np.zeros(2, np.int64)
    try:
        g = syn.rng(cfg["index"], 4242)
        for T in (1, 2, 3, 4, 16, 40, 1):  # 16: direct calls of 4 tokens, 40: expert-sorted tiles
            x = syn.activations(T, H, g)
            logits = syn.router_logits(T, E, g)
            ids, _ = orc.router(logits, k)
            ctx.moe_experts(w8, E, H, I, k, to_dev(x), logits=to_dev(logits))
            want_pairs += np.bincount(ids.ravel(), minlength=E)
            want_calls += [1, len(np.unique(ids))]
        ctx.sync_status()
        assert np.array_equal(to_host(pairs), want_pairs)
        assert np.array_equal(to_host(calls), want_calls)
        # a layer with more experts than the buffer holds is refused while the telemetry is on
        with pytest.raises(ggq.GGQError, match="SHAPE"):
            ctx.moe_experts(w8, E + 1, H, I, k, to_dev(np.zeros((1, H), np.float32)),
                            logits=to_dev(np.zeros((1, E + 1), np.float32)))
    finally:
        ctx.set_moe_counters(None, None)
    # off: further calls leave the buffers alone
    x = syn.activations(2, H, syn.rng(cfg["index"], 4243))
    ctx.moe_experts(w8, E, H, I, k, to_dev(x), logits=to_dev(syn.router_logits(2, E, syn.rng(cfg["index"], 4244))))
    ctx.sync_status()
    assert np.array_equal(to_host(pairs), want_pairs) and np.array_equal(to_host(calls), want_calls)


def test_moe_rejects_bad_arguments(ctx):
    cfg = syn.MOE_DECODE
    host, dev = _banks(cfg, cfg["E"])
    w8 = ctx.moe_weights("Q4_0", dev["gate"], "Q4_0", dev["up"], "Q6_K", dev["down"])
    x = to_dev(np.zeros((1, cfg["H"]), np.float32))
    lg = to_dev(np.zeros((1, cfg["E"]), np.float32))
    with pytest.raises(ggq.GGQError, match="UNSUPPORTED"):
        ctx.moe_experts(w8, cfg["E"], cfg["H"], cfg["I"], 8, x, logits=lg)
    w8 = ctx.moe_weights("Q4_K", dev["gate"], "Q4_K", dev["up"], "Q6_K", dev["down"])
    with pytest.raises(ggq.GGQError, match="SHAPE"):
        ctx.moe_experts(w8, cfg["E"], cfg["H"], 700, 8, x, logits=lg)
    with pytest.raises(ggq.GGQError, match="SHAPE"):
        ctx.moe_experts(w8, cfg["E"], cfg["H"], cfg["I"], 9, x, logits=lg)
    # widths beyond the kernels' shared-memory plans are refused before anything
    # is enqueued (direct route, Q8_0 gate/up rows of H = 8192): Y keeps its bytes
    dummy = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    wide = ctx.moe_weights("Q8_0", dummy, "Q8_0", dummy, "Q4_K", dummy)
    xw = torch.zeros((1, 8192), dtype=torch.float32, device="cuda")
    lgw = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    yw = torch.full((1, 8192), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(ggq.GGQError, match="SHAPE"):
        ctx.moe_experts(wide, 16, 8192, 256, 8, xw, logits=lgw, Y=yw)
    torch.cuda.synchronize()
    assert bool(torch.all(yw == 7.0))
    # an out-of-range routed id is caught on the device and reported
    ids = to_dev(np.array([[cfg["E"] + 3, 0, 1, 2, 3, 4, 5, 6]], np.int32))
    wts = to_dev(np.full((1, 8), 0.125, np.float32))
    ctx.moe_experts(w8, cfg["E"], cfg["H"], cfg["I"], 8, x, ids=ids, route_w=wts)
    with pytest.raises(ggq.GGQError, match="DEVICE"):
        ctx.sync_status()
    ctx.sync_status()  # the word was cleared
