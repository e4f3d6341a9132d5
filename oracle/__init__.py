"""CPU oracle for the keep-quant GEMV / MoE routed-expert path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The product library never
imports, links or runs anything here.  The arithmetic lives in plain C
(``ggq_oracle.c``, double precision, no code shared with the CUDA path); this
module only builds it with gcc and marshals numpy arrays through ctypes.

Parity status: pinned by the CPU tests in ``tests/test_oracle_pins.py``,
except layout agreement with real GGUF files (no such file is available):
parity unpinned for that one property.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ggq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libggq_oracle.so")
_lock = threading.Lock()
_lib = None

# The oracle's own format tags (see ggq_oracle.h).
FMT = {"Q4_0": 0, "Q8_0": 1, "Q4_K": 2, "Q5_K": 3, "Q6_K": 4, "MXFP4": 5, "Q8_1": 6, "Q8_K": 7, "Q2_K": 8, "Q3_K": 9}
BLOCK_ELEMS = {"Q4_0": 32, "Q8_0": 32, "MXFP4": 32, "Q8_1": 32, "Q4_K": 256, "Q5_K": 256, "Q6_K": 256, "Q8_K": 256,
               "Q2_K": 256, "Q3_K": 256}
BLOCK_BYTES = {"Q4_0": 18, "Q8_0": 34, "MXFP4": 17, "Q8_1": 36, "Q4_K": 144, "Q5_K": 176, "Q6_K": 210, "Q8_K": 292,
               "Q2_K": 84, "Q3_K": 110}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE: no contraction, no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "ggq_oracle.h"))
    ):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=gnu99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            "-fno-strict-aliasing", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # GGQ_ORACLE_LIB: load another build of the oracle (the pin tests'
            # mutation check runs them against deliberately broken builds)
            L = ctypes.CDLL(os.environ.get("GGQ_ORACLE_LIB") or build())
            i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            sig = {
                "orc_set_threads": (None, [i32]),
                "orc_get_threads": (i32, []),
                "orc_half_to_double": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_float_to_half": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_e2m1": (ctypes.c_double, [i32]),
                "orc_kq_scale_min": (None, [p, i32, p, p]),
                "orc_q3k_scale": (i32, [p, i32]),
                "orc_coefs_per_block": (i32, [i32]),
                "orc_block_bytes": (i32, [i32]),
                "orc_dequant": (None, [i32, p, i64, i64, p]),
                "orc_quantize_q8_1": (None, [p, i64, i64, p]),
                "orc_quantize_q8_k": (None, [p, i64, i64, p]),
                "orc_quantize_q8_0": (None, [p, i64, i64, p]),
                "orc_pair_ok": (i32, [i32, i32]),
                "orc_gemv_a": (None, [i32, i32, p, i64, i64, p, i64, p]),
                "orc_gemv_coefs_a": (None, [i32, i32, p, i64, i64, p, i64, p]),
                "orc_gemv_dequant_a": (None, [i32, i32, p, i64, i64, p, i64, p, p]),
                "orc_row_coefs": (None, [i32, p, p, i64, p]),
                "orc_gemv": (None, [i32, p, i64, i64, p, i64, p]),
                "orc_gemv_coefs": (None, [i32, p, i64, i64, p, i64, p]),
                "orc_gemv_dequant": (None, [i32, p, i64, i64, p, i64, p, p]),
                "orc_router": (None, [p, i64, i64, i32, p, p]),
                "orc_silu": (ctypes.c_double, [ctypes.c_double]),
                "orc_moe_gate_up": (None, [i32, p, i32, p, i64, i64, p, i64, p, i32, p, p, p]),
                "orc_moe_down": (None, [i32, p, i64, i64, p, i64, p, i32, p]),
                "orc_moe_combine": (None, [p, p, i64, i32, i64, p]),
                "orc_moe": (None, [i32, p, i32, p, i32, p, i64, i64, i64, i32, p, p, i64, p, p, p, p, p, p, p]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def threads() -> int:
    return lib().orc_get_threads()


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(int(h))


def float_to_half(f: float) -> int:
    return lib().orc_float_to_half(float(f))


def e2m1(code: int) -> float:
    return lib().orc_e2m1(int(code))


def kq_scale_min(scales12: np.ndarray, s: int) -> tuple[int, int]:
    a = np.ascontiguousarray(scales12, dtype=np.uint8)
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().orc_kq_scale_min(_p(a), int(s), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def q3k_scale(scales12: np.ndarray, s: int) -> int:
    """Unsigned 6-bit scale of 16-element group s of a Q3_K block (signed: - 32)."""
    a = np.ascontiguousarray(scales12, dtype=np.uint8)
    return int(lib().orc_q3k_scale(_p(a), int(s)))


def act_type(wtype: str) -> str:
    return "Q8_1" if wtype == "Q4_0" else "Q8_K"


def coefs_per_block(wtype: str) -> int:
    return int(lib().orc_coefs_per_block(FMT[wtype]))


def row_bytes(fmt: str, K: int) -> int:
    return K // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]


def dequant(fmt: str, blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    assert b.size >= rows * row_bytes(fmt, K)
    out = np.empty((rows, K), dtype=np.float64)
    lib().orc_dequant(FMT[fmt], _p(b), rows, K, _p(out))
    return out


def quantize(act: str, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, K = x.reshape(-1, x.shape[-1]).shape
    out = np.zeros((T, row_bytes(act, K)), dtype=np.uint8)
    if act == "Q8_1":
        lib().orc_quantize_q8_1(_p(x), T, K, _p(out))
    elif act == "Q8_0":
        lib().orc_quantize_q8_0(_p(x), T, K, _p(out))
    elif act == "Q8_K":
        lib().orc_quantize_q8_k(_p(x), T, K, _p(out))
    else:
        raise ValueError(act)
    return out


def _act(wtype: str, act: str | None) -> str:
    a = act or act_type(wtype)
    if not lib().orc_pair_ok(FMT[wtype], FMT[a]):
        raise ValueError(f"{wtype} weights do not pair with {a} activations")
    return a


def gemv(wtype: str, W: np.ndarray, N: int, K: int, Xq: np.ndarray, T: int, act: str | None = None) -> np.ndarray:
    """Integer-dot form: Y[T][N] in float64 (act: the activation format of Xq, default the weight's)."""
    a = _act(wtype, act)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    assert W.size >= N * row_bytes(wtype, K) and Xq.size >= T * row_bytes(a, K)
    Y = np.empty((T, N), dtype=np.float64)
    lib().orc_gemv_a(FMT[wtype], FMT[a], _p(W), N, K, _p(Xq), T, _p(Y))
    return Y


def gemv_coefs(wtype: str, W: np.ndarray, N: int, K: int, Xq: np.ndarray, T: int, act: str | None = None) -> np.ndarray:
    """Per-block int32 coefficients: [T][N][K/blk * coefs_per_block]."""
    a = _act(wtype, act)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    assert W.size >= N * row_bytes(wtype, K) and Xq.size >= T * row_bytes(a, K)
    nc = K // BLOCK_ELEMS[wtype] * coefs_per_block(wtype)
    out = np.empty((T, N, nc), dtype=np.int32)
    lib().orc_gemv_coefs_a(FMT[wtype], FMT[a], _p(W), N, K, _p(Xq), T, _p(out))
    return out


def gemv_dequant(wtype: str, W: np.ndarray, N: int, K: int, Xq: np.ndarray, T: int, act: str | None = None):
    """Dequantize-then-double form: returns (Y, sum |w*x|), each [T][N]."""
    a = _act(wtype, act)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    assert W.size >= N * row_bytes(wtype, K) and Xq.size >= T * row_bytes(a, K)
    Y = np.empty((T, N), dtype=np.float64)
    A = np.empty((T, N), dtype=np.float64)
    lib().orc_gemv_dequant_a(FMT[wtype], FMT[a], _p(W), N, K, _p(Xq), T, _p(Y), _p(A))
    return Y, A


def router(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().orc_router(_p(logits), T, E, k, _p(ids), _p(w))
    return ids, w


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def moe_gate_up(gtype, gate_bank, utype, up_bank, H, I, xq, T, ids, k, want_gu=False):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    h = np.empty((T * k, I), dtype=np.float64)
    g = np.empty((T * k, I), dtype=np.float64) if want_gu else None
    u = np.empty((T * k, I), dtype=np.float64) if want_gu else None
    lib().orc_moe_gate_up(FMT[gtype], _p(np.ascontiguousarray(gate_bank)), FMT[utype],
                          _p(np.ascontiguousarray(up_bank)), H, I, _p(np.ascontiguousarray(xq)), T, _p(ids), k,
                          _p(g), _p(u), _p(h))
    return (g, u, h) if want_gu else h


def moe_down(dtype, down_bank, H, I, hq, T, ids, k):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    o = np.empty((T * k, H), dtype=np.float64)
    lib().orc_moe_down(FMT[dtype], _p(np.ascontiguousarray(down_bank)), H, I, _p(np.ascontiguousarray(hq)), T,
                       _p(ids), k, _p(o))
    return o


def moe_combine(o, weights, T, k, H):
    o = np.ascontiguousarray(o, dtype=np.float64)
    w = np.ascontiguousarray(weights, dtype=np.float64)
    y = np.empty((T, H), dtype=np.float64)
    lib().orc_moe_combine(_p(o), _p(w), T, k, H, _p(y))
    return y


def moe(gtype, gate_bank, utype, up_bank, dtype, down_bank, E, H, I, k, x, logits):
    """The whole routed-expert layer; returns a dict of every intermediate."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T = x.shape[0]
    r = {
        "ids": np.empty((T, k), dtype=np.int32),
        "weights": np.empty((T, k), dtype=np.float64),
        "xq": np.empty((T, row_bytes("Q8_K", H)), dtype=np.uint8),
        "h": np.empty((T * k, I), dtype=np.float64),
        "hq": np.empty((T * k, row_bytes("Q8_K", I)), dtype=np.uint8),
        "o": np.empty((T * k, H), dtype=np.float64),
        "y": np.empty((T, H), dtype=np.float64),
    }
    lib().orc_moe(FMT[gtype], _p(np.ascontiguousarray(gate_bank)), FMT[utype], _p(np.ascontiguousarray(up_bank)),
                  FMT[dtype], _p(np.ascontiguousarray(down_bank)), E, H, I, k, _p(x), _p(logits), T,
                  _p(r["ids"]), _p(r["weights"]), _p(r["xq"]), _p(r["h"]), _p(r["hq"]), _p(r["o"]), _p(r["y"]))
    return r
