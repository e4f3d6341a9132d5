"""Pins of the CPU oracle against what the format definitions and mathematics fix.

Each test checks the oracle against something other than itself: hand-worked
fixtures under tests/golden/, numpy's independent IEEE binary16 conversion,
exhaustive enumeration of codes and bit positions, inverse encoders, the
identity between the integer-dot form and the dequantize-then-double form,
closed-form router properties, special cases that reduce to a dense FFN, and
brute force on tiny MoE layers.
"""
import itertools
import math
import os

import numpy as np
import pytest

import ggq_synth as syn
import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows, header = [], {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "bytes":
            header["bytes"] = bytes(int(b, 16) for b in parts[1:])
        else:
            rows.append(parts)
    return header, rows


# ------------------------------------------------------------- scalars

def test_half_decode_matches_numpy_for_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_half_golden_values():
    _, rows = _read_pairs("fp16_examples.txt")
    for h, v in rows:
        assert orc.half_to_double(int(h, 16)) == float(v)
        assert orc.float_to_half(float(v)) == int(h, 16)


def test_half_encode_round_to_nearest_even_matches_numpy():
    g = np.random.default_rng(1)
    xs = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-8, 5, 20000).astype(np.float32),
        np.array([65504, 65519.99, 65520, 70000, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8, 1e-9, -0.0, 0.0,
                  1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 2048 + 1, 2048 + 3], dtype=np.float32),
    ]).astype(np.float32)
    # exact ties in the subnormal and normal ranges
    ties = (np.arange(1, 200, dtype=np.float64) + 0.5) * 2.0 ** -24
    xs = np.concatenate([xs, ties.astype(np.float32), -ties.astype(np.float32)])
    with np.errstate(over="ignore"):  # values past 65519.99 round to infinity on purpose
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([orc.float_to_half(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_e2m1_golden_table():
    _, rows = _read_pairs("e2m1_codes.txt")
    assert len(rows) == 16
    for c, v in rows:
        got = orc.e2m1(int(c))
        assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v))


# ------------------------------------------------------------- block formats

def test_q4_0_golden_block():
    hdr, rows = _read_pairs("q4_0_worked.txt")
    vals = orc.dequant("Q4_0", np.frombuffer(hdr["bytes"], dtype=np.uint8), 1, 32)[0]
    assert len(rows) == 32
    for i, v in rows:
        assert vals[int(i)] == float(v)


def test_q4_0_closed_form_every_code_every_position():
    d = np.float16(0.0078125)  # exact power of two
    for code in range(16):
        blk = np.zeros(18, np.uint8)
        blk[0:2] = np.array([d]).view(np.uint8)
        blk[2:] = code | (((code + 5) % 16) << 4)
        v = orc.dequant("Q4_0", blk, 1, 32)[0]
        assert np.all(v[:16] == (code - 8) * float(d))
        assert np.all(v[16:] == (((code + 5) % 16) - 8) * float(d))


def test_q8_0_closed_form_all_int8_values():
    for start in range(0, 256, 32):
        blk = np.zeros(34, np.uint8)
        blk[0:2] = np.array([np.float16(0.3)]).view(np.uint8)
        q = np.arange(start, start + 32, dtype=np.uint8)
        blk[2:] = q
        v = orc.dequant("Q8_0", blk, 1, 32)[0]
        assert np.array_equal(v, q.view(np.int8).astype(np.float64) * float(np.float16(0.3)))


def _pack_kq_scales(sc, m):
    """Inverse of the 6-bit unpack: 8 scales and 8 mins (0..63) -> 12 bytes."""
    b = np.zeros(12, np.uint8)
    for s in range(4):
        b[s] = (sc[s] & 63) | ((sc[s + 4] >> 4) << 6)
        b[s + 4] = (m[s] & 63) | ((m[s + 4] >> 4) << 6)
        b[s + 8] = (sc[s + 4] & 15) | ((m[s + 4] & 15) << 4)
    return b


def test_q4_k_scale_golden():
    hdr, rows = _read_pairs("q4_k_scales_worked.txt")
    b = np.frombuffer(hdr["bytes"], dtype=np.uint8)
    for s, sc, m in rows:
        assert orc.kq_scale_min(b, int(s)) == (int(sc), int(m))


def test_q4_k_scale_roundtrip_exhaustive():
    g = np.random.default_rng(2)
    for s in range(8):
        for v in range(64):
            for which in ("sc", "m"):
                sc = g.integers(0, 64, 8)
                m = g.integers(0, 64, 8)
                (sc if which == "sc" else m)[s] = v
                b = _pack_kq_scales(sc, m)
                for t in range(8):
                    assert orc.kq_scale_min(b, t) == (sc[t], m[t])


def _kq_block(fmt, d, dmin, sc, m, nib, hb=None):
    """Build one Q4_K / Q5_K block from integer fields (inverse of the layout)."""
    bb = 144 if fmt == "Q4_K" else 176
    blk = np.zeros(bb, np.uint8)
    blk[0:2] = np.array([np.float16(d)]).view(np.uint8)
    blk[2:4] = np.array([np.float16(dmin)]).view(np.uint8)
    blk[4:16] = _pack_kq_scales(sc, m)
    qs_off = 16 if fmt == "Q4_K" else 48
    for i in range(256):
        s, l = divmod(i, 32)
        c = s // 2
        if s % 2 == 0:
            blk[qs_off + 32 * c + l] |= nib[i] & 15
        else:
            blk[qs_off + 32 * c + l] |= (nib[i] & 15) << 4
        if fmt == "Q5_K" and hb is not None and hb[i]:
            blk[16 + l] |= 1 << s
    return blk


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K"])
def test_kquant_element_closed_form(fmt):
    g = np.random.default_rng(3)
    d, dmin = np.float16(0.0123), np.float16(0.0071)
    for rep in range(8):
        sc = g.integers(0, 64, 8)
        m = g.integers(0, 64, 8)
        sc[rep % 8], m[(rep + 3) % 8] = 63, 0
        nib = np.tile(np.arange(16), 16)[g.permutation(256)]
        hb = g.integers(0, 2, 256) if fmt == "Q5_K" else np.zeros(256, int)
        v = orc.dequant(fmt, _kq_block(fmt, d, dmin, sc, m, nib, hb), 1, 256)[0]
        q = nib + 16 * hb
        s = np.arange(256) // 32
        expect = float(d) * sc[s] * q - float(dmin) * m[s]
        assert np.array_equal(v, expect)


def test_q5_k_every_high_bit_position():
    d, dmin = np.float16(0.5), np.float16(0.25)
    sc = np.arange(1, 9)
    m = np.arange(8)
    zero = np.zeros(256, int)
    base = orc.dequant("Q5_K", _kq_block("Q5_K", d, dmin, sc, m, zero), 1, 256)[0]
    for s in range(8):
        for l in range(32):
            blk = _kq_block("Q5_K", d, dmin, sc, m, zero)
            blk[16 + l] |= 1 << s  # one high bit: element 32*s + l gains 16
            v = orc.dequant("Q5_K", blk, 1, 256)[0]
            diff = np.nonzero(v != base)[0]
            assert list(diff) == [32 * s + l]
            assert v[32 * s + l] - base[32 * s + l] == 16 * float(d) * sc[s]


def test_q6_k_every_bit_field_position():
    """One-hot ql nibbles and qh bit pairs: exactly one element moves, at the
    index the layout defines: ql byte b, nibble n -> 128*(b//64) + 64*n + b%64;
    qh byte j, bit pair p -> 128*(j//32) + 32*p + j%32; value d*sc_(i//16)*(q-32)."""
    blk = np.zeros(210, np.uint8)
    scales = (np.arange(16) - 7).astype(np.int8)
    blk[192:208] = scales.view(np.uint8)
    blk[208:210] = np.array([np.float16(0.25)]).view(np.uint8)
    base = orc.dequant("Q6_K", blk, 1, 256)[0]
    assert np.array_equal(base, 0.25 * scales[np.arange(256) // 16] * -32.0)
    for b in range(128):
        for n in range(2):
            x = blk.copy()
            x[b] |= 0x5 << (4 * n)
            v = orc.dequant("Q6_K", x, 1, 256)[0]
            i = 128 * (b // 64) + 64 * n + b % 64
            assert list(np.nonzero(v != base)[0]) == [i] or scales[i // 16] == 0
            assert v[i] == 0.25 * scales[i // 16] * (5 - 32)
    for j in range(64):
        for p in range(4):
            x = blk.copy()
            x[128 + j] |= 0x2 << (2 * p)
            v = orc.dequant("Q6_K", x, 1, 256)[0]
            i = 128 * (j // 32) + 32 * p + j % 32
            assert v[i] == 0.25 * scales[i // 16] * (32 - 32)
            assert np.count_nonzero(v != base) == (1 if scales[i // 16] != 0 else 0)


def _pack_q3k_scales(sc6):
    """Inverse of the Q3_K scale layout: 16 unsigned 6-bit scales -> 12 bytes."""
    b = np.zeros(12, np.uint8)
    for s in range(16):
        v = int(sc6[s])
        if s < 8:
            b[s] |= v & 15
        else:
            b[s - 8] |= (v & 15) << 4
        b[8 + s % 4] |= ((v >> 4) & 3) << (2 * (s // 4))
    return b


def test_q3_k_scale_golden():
    hdr, rows = _read_pairs("q3_k_scales_worked.txt")
    b = np.frombuffer(hdr["bytes"], dtype=np.uint8)
    for s, sc in rows:
        assert orc.q3k_scale(b, int(s)) == int(sc)


def test_q3_k_scale_roundtrip_exhaustive():
    g = np.random.default_rng(5)
    for s in range(16):
        for v in range(64):
            sc6 = g.integers(0, 64, 16)
            sc6[s] = v
            b = _pack_q3k_scales(sc6)
            assert [orc.q3k_scale(b, t) for t in range(16)] == [int(x) for x in sc6]


def _low_k_block(fmt, d, dmin, sc, m, q):
    """Build one Q2_K / Q3_K block from integer fields (inverse of the layout):
    element i = 128n + 32j + l holds its two low bits at bits 2j of qs[32n + l];
    Q3_K's q in -4..3 keeps bit 4n + j of hmask[l] set for q >= 0 (q + 4 - 4)
    and clear for q < 0 (low bits q + 4).  sc, m: per 16-element group (Q2_K:
    4-bit scale and min; Q3_K: unsigned 6-bit scale, signed value sc - 32)."""
    blk = np.zeros(84 if fmt == "Q2_K" else 110, np.uint8)
    qs_off = 16 if fmt == "Q2_K" else 32
    for i in range(256):
        n, j, l = i // 128, (i % 128) // 32, i % 32
        v = int(q[i])
        if fmt == "Q3_K":
            if v >= 0:
                blk[l] |= 1 << (4 * n + j)
            else:
                v += 4
        blk[qs_off + 32 * n + l] |= (v & 3) << (2 * j)
    if fmt == "Q2_K":
        blk[0:16] = (np.asarray(sc) & 15) | ((np.asarray(m) & 15) << 4)
        blk[80:82] = np.array([np.float16(d)]).view(np.uint8)
        blk[82:84] = np.array([np.float16(dmin)]).view(np.uint8)
    else:
        blk[96:108] = _pack_q3k_scales(sc)
        blk[108:110] = np.array([np.float16(d)]).view(np.uint8)
    return blk


@pytest.mark.parametrize("fmt", ["Q2_K", "Q3_K"])
def test_low_bit_kquant_element_closed_form(fmt):
    g = np.random.default_rng(7)
    d, dmin = np.float16(0.0137), np.float16(0.0059)
    grp = np.arange(256) // 16
    for rep in range(8):
        if fmt == "Q2_K":
            sc, m = g.integers(0, 16, 16), g.integers(0, 16, 16)
            sc[rep], m[(rep + 5) % 16] = 15, 0
            q = np.tile(np.arange(4), 64)[g.permutation(256)]
            expect = float(d) * sc[grp] * q - float(dmin) * m[grp]
        else:
            sc, m = g.integers(0, 64, 16), None
            sc[rep], sc[(rep + 9) % 16] = 63, 0
            q = np.tile(np.arange(-4, 4), 32)[g.permutation(256)]
            expect = float(d) * (sc[grp] - 32) * q
        v = orc.dequant(fmt, _low_k_block(fmt, d, dmin, sc, m, q), 1, 256)[0]
        assert np.array_equal(v, expect)


@pytest.mark.parametrize("fmt", ["Q2_K", "Q3_K"])
def test_low_bit_kquant_every_bit_position(fmt):
    """One-hot bit pairs of qs (and, for Q3_K, bits of hmask): exactly one
    element moves, at the index the layout defines: qs byte 32n + l, bit pair
    j -> element 128n + 32j + l; hmask byte l, bit 4n + j -> the same element."""
    d, dmin = np.float16(0.5), np.float16(0.25)
    grp = np.arange(256) // 16
    sc = np.arange(16) % 13 + 1 if fmt == "Q2_K" else (np.arange(16) * 3 + 33) % 64
    m = np.arange(16) % 5 if fmt == "Q2_K" else None
    zero = np.zeros(256, int) if fmt == "Q2_K" else np.full(256, -4)
    blk = _low_k_block(fmt, d, dmin, sc, m, zero)
    base = orc.dequant(fmt, blk, 1, 256)[0]
    qs_off = 16 if fmt == "Q2_K" else 32
    scale = (sc if fmt == "Q2_K" else sc - 32)[grp]
    for byte in range(64):
        for j in range(4):
            x = blk.copy()
            x[qs_off + byte] |= 1 << (2 * j)  # low bit of the pair: +1
            v = orc.dequant(fmt, x, 1, 256)[0]
            i = 128 * (byte // 32) + 32 * j + byte % 32
            assert list(np.nonzero(v != base)[0]) == [i]
            assert v[i] - base[i] == float(d) * scale[i]
    if fmt == "Q3_K":
        for l in range(32):
            for bit in range(8):
                x = blk.copy()
                x[l] |= 1 << bit  # high bit: -4 -> 0
                v = orc.dequant(fmt, x, 1, 256)[0]
                i = 128 * (bit // 4) + 32 * (bit % 4) + l
                diff = np.nonzero(v != base)[0]
                assert list(diff) == ([i] if scale[i] != 0 else [])
                assert v[i] - base[i] == 4 * float(d) * scale[i]


def test_mxfp4_every_code_and_exponent():
    _, rows = _read_pairs("e2m1_codes.txt")
    table = {int(c): float(v) for c, v in rows}
    for e in (1, 117, 120, 123, 127, 200):
        for code in range(16):
            blk = np.zeros(17, np.uint8)
            blk[0] = e
            blk[1:] = code | (((15 - code)) << 4)
            v = orc.dequant("MXFP4", blk, 1, 32)[0]
            assert np.all(v[:16] == table[code] * 2.0 ** (e - 127))
            assert np.all(v[16:] == table[15 - code] * 2.0 ** (e - 127))


# ------------------------------------------------------------- quantizers

def _q8k_fields(b):
    d = b[0:4].view(np.float32)[0]
    q = b[4:260].view(np.int8).astype(np.int64)
    bs = b[260:292].view(np.int16).astype(np.int64)
    return d, q, bs


def _q8_1_fields(b):
    d = b[0:2].view(np.float16)[0]
    s = b[2:4].view(np.float16)[0]
    q = b[4:36].view(np.int8).astype(np.int64)
    return d, s, q


def _random_acts(g, T, K):
    x = g.standard_normal((T, K)).astype(np.float32)
    x[0, :256] = 0.0                                   # an all-zero block
    x[-1, 256:512] *= np.float32(1e-30)                # tiny magnitudes
    x[-1, 512:768] = np.float32(3.0) * np.sign(x[-1, 512:768])  # many ties of |x| = amax
    return x


@pytest.mark.parametrize("act", ["Q8_K", "Q8_1", "Q8_0"])
def test_quantizer_invariants(act):
    g = np.random.default_rng(4)
    T, K = 3, 1024
    x = _random_acts(g, T, K)
    out = orc.quantize(act, x)
    blk = 256 if act == "Q8_K" else 32
    bb = {"Q8_K": 292, "Q8_1": 36, "Q8_0": 34}[act]
    for t in range(T):
        for j in range(K // blk):
            b = out[t, j * bb:(j + 1) * bb]
            xs = x[t, j * blk:(j + 1) * blk].astype(np.float64)
            amax = np.max(np.abs(xs))
            d32 = np.float32(np.float32(amax) / np.float32(127.0))
            if act == "Q8_K":
                d, q, bs = _q8k_fields(b)
                assert d == d32
                assert np.array_equal(bs, q.reshape(16, 16).sum(1))
            elif act == "Q8_0":  # fp16 d, then the 32 quants (the Q8_0 weight layout)
                d, q = b[0:2].view(np.float16)[0], b[2:34].view(np.int8).astype(int)
                assert d == np.float16(d32)
            else:
                d, s, q = _q8_1_fields(b)
                assert d == np.float16(d32)
                assert s == np.float16(np.float32(d32 * np.float32(q.sum())))
                # independent of that formula: s stands for the block's sum, so it lies
                # within the 32 quantization errors (and its own fp16 rounding) of sum(x)
                assert abs(float(s) - xs.sum()) <= 16 * float(d32) * (1 + 1e-5) + abs(float(s)) * 2.0 ** -11 + 1e-7
            assert np.all(np.abs(q) <= 127)
            if amax == 0:
                assert np.all(q == 0) and float(d) == 0.0
                continue
            i = int(np.argmax(np.abs(xs)))
            assert abs(q[i]) == 127 and np.sign(q[i]) == np.sign(xs[i])
            # reconstruction within half a step (fp32 rounding of x * (1/d) adds a hair)
            assert np.all(np.abs(xs - q * float(d32)) <= float(d32) * (0.5 + 1e-6))


def test_quantizer_rounds_ties_away_from_zero():
    # amax = 127 makes d = 1 and 1/d = 1 exactly, so x * id = x.
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 127.0
    x[0, 1:7] = [2.5, -2.5, 0.5, -0.5, 126.5, -1.5]
    q = _q8k_fields(orc.quantize("Q8_K", x)[0])[1]
    assert list(q[:7]) == [127, 3, -3, 1, -1, 127, -2]


# ------------------------------------------------------------- integer dots

@pytest.mark.parametrize("fmt", list(syn.WEIGHT_FORMATS))
def test_integer_form_equals_dequant_form(fmt):
    g = syn.rng(99, syn.WEIGHT_FORMATS.index(fmt))
    N, K, T = 7, 768, 3
    W = syn.weights(fmt, N, K, g)
    if fmt == "Q8_0":
        W[0, 2:34] = 0x80  # -128 quants: the extreme of the int8 range
    x = syn.activations(T, K, g) * np.float32(4.0)
    xq = orc.quantize(orc.act_type(fmt), x)
    Yi = orc.gemv(fmt, W, N, K, xq, T)
    Yd, A = orc.gemv_dequant(fmt, W, N, K, xq, T)
    assert np.all(np.abs(Yi - Yd) <= 1e-12 * A)
    # and the coefficients are the ones whose scale epilogue gives Yi
    C = orc.gemv_coefs(fmt, W, N, K, xq, T)
    assert C.shape == (T, N, K // syn.BLOCK_ELEMS[fmt] * orc.coefs_per_block(fmt))


@pytest.mark.parametrize("fmt,act", [("Q4_0", "Q8_1"), ("Q8_0", "Q8_K"), ("MXFP4", "Q8_K"), ("Q4_0", "Q8_0"),
                                     ("Q8_0", "Q8_0")])
def test_block_coefs_brute_force_32_block_formats(fmt, act):
    """S_b = sum of integer quants products, recovered element by element from the
    dequantized values: w / d_w (resp. w / 2^(e-128)) and x / d_x are integers."""
    g = syn.rng(98, 0)
    N, K, T = 3, 512, 2
    W = syn.weights(fmt, N, K, g)
    x = syn.activations(T, K, g)
    xq = orc.quantize(act, x)
    C = orc.gemv_coefs(fmt, W, N, K, xq, T, act=act)
    wd = orc.dequant(fmt, W, N, K)
    xd = orc.dequant(act, xq, T, K)
    nb = K // 32
    for n in range(N):
        for b in range(nb):
            blk = W[n, b * syn.BLOCK_BYTES[fmt]:(b + 1) * syn.BLOCK_BYTES[fmt]]
            unit = 2.0 ** (int(blk[0]) - 128) if fmt == "MXFP4" else float(blk[0:2].view(np.float16)[0])
            qw = wd[n, 32 * b:32 * b + 32] / unit
            assert np.array_equal(qw, np.round(qw))
            for t in range(T):
                if act == "Q8_1":
                    dx = float(xq[t, b * 36:b * 36 + 2].view(np.float16)[0])
                elif act == "Q8_0":
                    dx = float(xq[t, b * 34:b * 34 + 2].view(np.float16)[0])
                else:
                    dx = float(xq[t, (b // 8) * 292:(b // 8) * 292 + 4].view(np.float32)[0])
                qx = np.round(xd[t, 32 * b:32 * b + 32] / dx)
                assert C[t, n, b] == int(np.dot(qw, qx))


@pytest.mark.parametrize("fmt", ["Q4_0", "Q8_0"])
def test_q8_0_activation_pairings_integer_form_equals_dequant_form(fmt):
    """The Q8_0 activation blocks ([VC523] What changed: Q8_0 x Q8_0) pair with
    Q4_0 and Q8_0 weights; the integer form equals the dequantized dot."""
    g = syn.rng(97, 1 + (fmt == "Q8_0"))
    N, K, T = 9, 1024, 3
    W = syn.weights(fmt, N, K, g)
    x = syn.activations(T, K, g) * np.float32(2.5)
    xq = orc.quantize("Q8_0", x)
    Yi = orc.gemv(fmt, W, N, K, xq, T, act="Q8_0")
    Yd, A = orc.gemv_dequant(fmt, W, N, K, xq, T, act="Q8_0")
    assert np.all(np.abs(Yi - Yd) <= 1e-12 * A)
    # the same dot through the Q8_1 blocks of the same x: Q8_1 and Q8_0 share d and q
    q81 = orc.quantize("Q8_1", x).reshape(T, K // 32, 36)
    q80 = xq.reshape(T, K // 32, 34)
    assert np.array_equal(q81[..., 0:2], q80[..., 0:2]) and np.array_equal(q81[..., 4:], q80[..., 2:])
    if fmt == "Q4_0":
        assert np.array_equal(orc.gemv_coefs(fmt, W, N, K, xq, T, act="Q8_0"),
                              orc.gemv_coefs(fmt, W, N, K, q81.reshape(T, -1), T))
    with pytest.raises(ValueError):
        orc.gemv("Q4_K", syn.weights("Q4_K", 1, 256, g), 1, 256, orc.quantize("Q8_0", x[:1, :256]), 1, act="Q8_0")


# ------------------------------------------------------------- router

def test_router_matches_exhaustive_subset_search():
    g = np.random.default_rng(5)
    E, k = 7, 3
    logits = g.standard_normal((40, E)).astype(np.float32)
    logits[3] = 0.5                       # all tied
    logits[4, [1, 4]] = logits[4, 2]      # partial ties
    ids, w = orc.router(logits, k)
    for t in range(logits.shape[0]):
        l = logits[t].astype(np.float64)
        # the top-k set: largest sum of logits; among equal sums, the one whose
        # sorted index list is smallest (ties go to the lower expert index)
        best = max(itertools.combinations(range(E), k),
                   key=lambda S: (sorted(l[list(S)], reverse=True), [-i for i in sorted(S)]))
        assert sorted(ids[t]) == sorted(best)
        # order: descending logit, ties by index
        assert [(-l[i], i) for i in ids[t]] == sorted((-l[i], i) for i in ids[t])
        assert abs(w[t].sum() - 1.0) < 1e-15
        for a in range(k):
            for b in range(k):
                assert abs(w[t, a] / w[t, b] - math.exp(l[ids[t, a]] - l[ids[t, b]])) < 1e-13
    assert list(ids[3]) == [0, 1, 2] and np.allclose(w[3], 1.0 / 3, rtol=0, atol=1e-16)


# ------------------------------------------------------------- MoE

def _dense_ffn(gtype, Wg, utype, Wu, dtype, Wd, H, I, x):
    """One dense FFN on x^ = Q8_K(x) from the pinned GEMV and quantizer."""
    xq = orc.quantize("Q8_K", x)
    T = x.shape[0]
    gv = orc.gemv(gtype, Wg, I, H, xq, T)
    uv = orc.gemv(utype, Wu, I, H, xq, T)
    h = np.vectorize(orc.silu)(gv) * uv
    hq = orc.quantize("Q8_K", h.astype(np.float32))
    return orc.gemv(dtype, Wd, H, I, hq, T)


@pytest.mark.parametrize("types", [("Q4_K", "Q4_K", "Q6_K"), ("MXFP4", "MXFP4", "MXFP4"), ("Q8_0", "Q8_0", "Q4_K")])
def test_moe_all_experts_uniform_reduces_to_dense_ffn(types):
    gt, ut, dt = types
    g = syn.rng(97, 0)
    E, H, I, T = 4, 256, 512, 3
    Wg = syn.weights(gt, I, H, g)
    Wu = syn.weights(ut, I, H, g)
    Wd = syn.weights(dt, H, I, g)
    gate = np.stack([Wg] * E)
    up = np.stack([Wu] * E)
    down = np.stack([Wd] * E)
    x = syn.activations(T, H, g)
    logits = np.zeros((T, E), np.float32)
    r = orc.moe(gt, gate, ut, up, dt, down, E, H, I, E, x, logits)
    assert np.all(r["ids"] == np.arange(E)) and np.all(r["weights"] == 1.0 / E)
    dense = _dense_ffn(gt, Wg, ut, Wu, dt, Wd, H, I, x)
    scale = np.abs(dense).max()
    assert np.max(np.abs(r["y"] - dense)) <= 1e-12 * scale


@pytest.mark.parametrize("types", [("Q8_0", "MXFP4", "Q6_K"), ("Q4_K", "Q5_K", "MXFP4")])
def test_moe_brute_force_two_experts(types):
    """Two experts, H = I = 256, every output by naive loops over dequantized
    elements and an exhaustive top-k search."""
    gt, ut, dt = types
    g = syn.rng(96, 0)
    E, H, I, T = 2, 256, 256, 3
    gate = syn.expert_bank(gt, E, I, H, g)
    up = syn.expert_bank(ut, E, I, H, g)
    down = syn.expert_bank(dt, E, H, I, g)
    x = syn.activations(T, H, g)
    logits = syn.router_logits(T, E, g)
    for k in (1, 2):
        r = orc.moe(gt, gate, ut, up, dt, down, E, H, I, k, x, logits)
        Wg = [orc.dequant(gt, gate[e], I, H) for e in range(E)]
        Wu = [orc.dequant(ut, up[e], I, H) for e in range(E)]
        Wd = [orc.dequant(dt, down[e], H, I) for e in range(E)]
        xq = orc.quantize("Q8_K", x)
        xd = orc.dequant("Q8_K", xq, T, H)
        for t in range(T):
            l = logits[t].astype(np.float64)
            S = max(itertools.combinations(range(E), k), key=lambda S: (sorted(l[list(S)], reverse=True),
                                                                      [-i for i in sorted(S)]))
            S = sorted(S, key=lambda e: (-l[e], e))
            p = np.array([math.exp(l[e] - l.max()) for e in S])
            wts = p / p.sum()
            y = np.zeros(H)
            for j, e in enumerate(S):
                gv = np.array([sum(Wg[e][i, c] * xd[t, c] for c in range(H)) for i in range(I)])
                uv = Wu[e] @ xd[t]
                h = np.array([gv[i] / (1 + math.exp(-gv[i])) * uv[i] for i in range(I)])
                hq = orc.quantize("Q8_K", h.astype(np.float32)[None, :])
                hd = orc.dequant("Q8_K", hq, 1, I)[0]
                y += wts[j] * (Wd[e] @ hd)
            assert list(r["ids"][t]) == S
            assert np.max(np.abs(r["y"][t] - y)) <= 1e-11 * np.abs(y).max()
