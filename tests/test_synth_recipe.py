"""The seeded input recipe (ggq_synth) on CPU: shapes, field ranges and
determinism of the synthetic workloads, read straight from the block bytes.

The recipe follows the workload definitions: fp16 scales uniform in their
ranges (Q2_K: d and dmin after the 80 bytes of scales and quants; Q3_K: d
after 108), Q6_K int8 sub-scales in [-32, 31], MXFP4 E8M0 exponent bytes in
117..123 (scales 2^-10 .. 2^-4), uniform quant bytes, N(0, 1) activations and
logits, and for the prefill workload a Zipf(1.1) expert bias over a seeded
permutation of ranks.
"""
import numpy as np
import pytest

import ggq_synth as syn


def _f16(field):
    return field.copy().view(np.float16).astype(np.float64).ravel()


@pytest.mark.parametrize("fmt", list(syn.WEIGHT_FORMATS))
def test_weight_fields_stay_in_their_ranges(fmt):
    rows, K = 64, 1024
    W = syn.weights(fmt, rows, K, syn.rng(90, syn.WEIGHT_FORMATS.index(fmt)))
    bb = syn.BLOCK_BYTES[fmt]
    assert W.shape == (rows, K // syn.BLOCK_ELEMS[fmt] * bb) and W.dtype == np.uint8
    B = W.reshape(-1, bb)
    lo, hi = (1e-3, 1e-2) if fmt == "Q4_0" else (1e-4, 1e-2)
    lo16, hi16 = float(np.float16(lo)), float(np.float16(hi))
    if fmt in ("Q4_0", "Q8_0"):
        d = _f16(B[:, 0:2])
        assert d.min() >= lo16 and d.max() <= hi16
        quants = B[:, 2:]
    elif fmt in ("Q4_K", "Q5_K"):
        for off in (0, 2):  # d, dmin
            v = _f16(B[:, off:off + 2])
            assert v.min() >= lo16 and v.max() <= hi16
        quants = B[:, 4:]
    elif fmt == "Q6_K":
        d = _f16(B[:, 208:210])
        assert d.min() >= lo16 and d.max() <= hi16
        sc = B[:, 192:208].view(np.int8)
        assert sc.min() == -32 and sc.max() == 31
        quants = B[:, 0:192]
    elif fmt == "Q2_K":  # scales[16], qs[64], d, dmin
        for off in (80, 82):
            v = _f16(B[:, off:off + 2])
            assert v.min() >= lo16 and v.max() <= hi16
        quants = B[:, 0:80]
    elif fmt == "Q3_K":  # hmask[32], qs[64], scales[12], d
        d = _f16(B[:, 108:110])
        assert d.min() >= lo16 and d.max() <= hi16
        quants = B[:, 0:108]
    else:  # MXFP4
        e = B[:, 0]
        assert e.min() == 117 and e.max() == 123
        quants = B[:, 1:]
    # quant bytes uniform over all 256 values: every value present, no value far off its share
    counts = np.bincount(quants.ravel(), minlength=256)
    assert np.all(counts > 0)
    assert counts.max() < 2.0 * counts.mean()


def test_inputs_are_seeded_and_independent_per_stream():
    a = syn.weights("Q4_K", 8, 512, syn.rng(1, 10))
    b = syn.weights("Q4_K", 8, 512, syn.rng(1, 10))
    c = syn.weights("Q4_K", 8, 512, syn.rng(1, 11))
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    x = syn.activations(4, 4096, syn.rng(2, 0))
    assert x.dtype == np.float32 and abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05


def test_expert_bank_is_rows_of_one_weight_draw():
    g1, g2 = syn.rng(3, 0), syn.rng(3, 0)
    bank = syn.expert_bank("Q6_K", 4, 16, 512, g1)
    flat = syn.weights("Q6_K", 4 * 16, 512, g2)
    assert bank.shape == (4, 16, syn.row_bytes("Q6_K", 512))
    assert np.array_equal(bank.reshape(64, -1), flat)


def test_zipf_bias_follows_a_seeded_rank_permutation():
    E, T = 128, 2048
    plain = syn.router_logits(T, E, syn.rng(4, 0))
    biased = syn.router_logits(T, E, syn.rng(4, 0), 1.1)
    bias = (biased - plain)[0]
    assert np.allclose(biased - plain, bias[None, :], atol=1e-6)
    # the bias takes the values -1.1 ln r for a permutation of the ranks 1..E
    ranks = np.rint(np.exp(-bias.astype(np.float64) / 1.1)).astype(int)
    assert sorted(ranks.tolist()) == list(range(1, E + 1))
    assert bias.max() == pytest.approx(0.0, abs=1e-6)
    # skew: the top-ranked experts are chosen far more often than the bottom ones
    top = np.argsort(-biased, axis=1, kind="stable")[:, :8]
    hits = np.bincount(top.ravel(), minlength=E)
    order = np.argsort(ranks)
    assert hits[order[:8]].sum() > 10 * hits[order[-64:]].sum()


def test_workload_shapes():
    assert (syn.GEMV_Q4_0["N"], syn.GEMV_Q4_0["K"]) == (1024, 4096)
    assert (syn.GEMV_KQUANT["N"], syn.GEMV_KQUANT["K"]) == (14336, 4096)
    assert syn.GEMV_KQUANT["T"] == (1, 2, 4, 8)
    for cfg, shape in ((syn.MOE_DECODE, (128, 2048, 768, 8)), (syn.MOE_MXFP4, (256, 4096, 2048, 8)),
                       (syn.MOE_PREFILL, (128, 4096, 1536, 8))):
        assert (cfg["E"], cfg["H"], cfg["I"], cfg["k"]) == shape
    assert syn.MOE_PREFILL["T"] == (4096,) and syn.MOE_PREFILL["zipf"] == 1.1
