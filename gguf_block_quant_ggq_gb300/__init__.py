"""Python binding of libggq: keep-quant GEMV and MoE routed-expert GEMM over
GGUF block-quantized weights on one GB300 (sm_103a).

Argument marshalling only.  Every step of every call runs in the CUDA kernels
of ``libggq.so`` (built in-tree by ``_build.build()``); there is no CPU path.
Loading fails loudly when the library is missing.  Functions keep the C names
of ``include/ggq.h`` and take device pointers as Python ints; ``Context`` wraps
them for torch tensors (torch supplies device memory and streams only).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libggq.so")

TYPE = {"Q4_0": 2, "Q8_0": 8, "Q8_1": 9, "Q2_K": 10, "Q3_K": 11, "Q4_K": 12, "Q5_K": 13, "Q6_K": 14, "Q8_K": 15,
        "MXFP4": 39}
OP = {"quantize_act": 0, "dequant": 1, "mul_mat_vec": 2, "moe": 3}
STATUS = {0: "GGQ_OK", 1: "GGQ_ERR_INVALID_ARG", 2: "GGQ_ERR_SHAPE", 3: "GGQ_ERR_UNSUPPORTED", 4: "GGQ_ERR_ARCH",
          5: "GGQ_ERR_CUDA", 6: "GGQ_ERR_CAPACITY", 7: "GGQ_ERR_CAPTURE_ALLOC", 8: "GGQ_ERR_DEVICE"}
BLOCK_ELEMS = {"Q4_0": 32, "Q8_0": 32, "MXFP4": 32, "Q8_1": 32, "Q4_K": 256, "Q5_K": 256, "Q6_K": 256, "Q8_K": 256,
               "Q2_K": 256, "Q3_K": 256}
BLOCK_BYTES = {"Q4_0": 18, "Q8_0": 34, "MXFP4": 17, "Q8_1": 36, "Q4_K": 144, "Q5_K": 176, "Q6_K": 210, "Q8_K": 292,
               "Q2_K": 84, "Q3_K": 110}

# Every entry point the header declares, with its ctypes signature.
_P, _I64, _I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
SIGNATURES = {
    "ggq_create": (_I32, [ctypes.POINTER(ctypes.c_void_p), _I32]),
    "ggq_destroy": (_I32, [_P]),
    "ggq_last_error": (ctypes.c_char_p, [_P]),
    "ggq_reserve": (_I32, [_P, _P, _P]),
    "ggq_scratch_bytes": (ctypes.c_size_t, [_P]),
    "ggq_set_static_weights": (_I32, [_P, _I32]),
    "ggq_set_direct_route_max_tokens": (_I32, [_P, _I32]),
    "ggq_supported": (_I32, [_I32, _I32, _I32]),
    "ggq_quantize_act": (_I32, [_P, _I32, _P, _I64, _I64, _P, _P]),
    "ggq_dequant": (_I32, [_P, _I32, _P, _I64, _I64, _P, _P]),
    "ggq_mul_mat_vec": (_I32, [_P, _I32, _P, _I64, _I64, _P, _I64, _P, _P]),
    "ggq_mul_mat_vec_q": (_I32, [_P, _I32, _P, _I64, _I64, _P, _I64, _P, _P]),
    "ggq_block_dots": (_I32, [_P, _I32, _P, _I64, _I64, _P, _I64, _P, _P]),
    "ggq_moe_experts": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _P, _P]),
    "ggq_moe_experts_routed": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _I64, _P, _P, _P]),
    "ggq_sync_status": (_I32, [_P, _P]),
    "ggq_mul_mat_vec_noalloc": (_I32, [_I32, _P, _I64, _I64, _P, _I64, _P, _P]),
    "ggq_set_moe_counters": (_I32, [_P, _P, _I64, _P]),
    "ggq_moe_experts_q": (_I32, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _I64, _P, _P, _P]),
    "ggq_mul_mat_vec_qa": (_I32, [_P, _I32, _I32, _P, _I64, _I64, _P, _I64, _P, _P]),
    "ggq_block_dots_qa": (_I32, [_P, _I32, _I32, _P, _I64, _I64, _P, _I64, _P, _P]),
}


class ggq_plan(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int64), ("max_k", ctypes.c_int64), ("n_experts", ctypes.c_int64),
                ("hidden", ctypes.c_int64), ("inter", ctypes.c_int64), ("top_k", ctypes.c_int64)]


class ggq_moe_weights(ctypes.Structure):
    _fields_ = [("gate_type", ctypes.c_int32), ("up_type", ctypes.c_int32), ("down_type", ctypes.c_int32),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p)]


class ggq_moe_dump(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("ids", "weights", "xq", "g", "u", "h", "hq", "o", "coefs_gate",
                                               "coefs_up", "coefs_down")]


class GGQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load libggq.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libggq is not built ({path} missing): run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _bind(name):
    def call(*args):
        return getattr(load(), name)(*args)
    call.__name__ = name
    return call


for _name in SIGNATURES:
    globals()[_name] = _bind(_name)


def row_bytes(fmt: str, K: int) -> int:
    return K // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]


def act_type(wfmt: str) -> str:
    return "Q8_1" if wfmt == "Q4_0" else "Q8_K"


def _ptr(t, dtype: str | None = None):
    """Device address of a torch CUDA tensor (None passes NULL).  The C calls
    read and write dense rows from that address, so the tensor must be on a
    CUDA device and contiguous; `dtype` (a torch dtype name) is checked where
    the call has a fixed element type.  Packed weight blocks may have any dtype."""
    if t is None:
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"libggq takes CUDA tensors (device memory), got one on {getattr(t, 'device', type(t))}")
    if not t.is_contiguous():
        raise ValueError("libggq reads and writes dense rows: pass a contiguous tensor")
    if dtype is not None and str(t.dtype) != "torch." + dtype:
        raise ValueError(f"expected a {dtype} tensor, got {t.dtype}")
    return t.data_ptr()


class Context:
    """A libggq context on one CUDA device; methods take torch CUDA tensors and
    enqueue on torch's current stream (or the given one)."""

    def __init__(self, device: int = 0):
        import torch  # device memory and streams only

        self._torch = torch
        self.device = device
        h = ctypes.c_void_p()
        st = load().ggq_create(ctypes.byref(h), device)
        if st != 0:
            raise GGQError(st, f"ggq_create(device={device}) failed")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            load().ggq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self, stream):
        if stream is None:
            stream = self._torch.cuda.current_stream(self.device)
        return ctypes.c_void_p(stream.cuda_stream)

    def _check(self, st):
        if st != 0:
            raise GGQError(st, load().ggq_last_error(self.handle).decode())

    def reserve(self, max_tokens=0, max_k=0, n_experts=0, hidden=0, inter=0, top_k=0, stream=None):
        plan = ggq_plan(max_tokens, max_k, n_experts, hidden, inter, top_k)
        self._check(load().ggq_reserve(self.handle, ctypes.byref(plan), self._stream(stream)))

    def set_static_weights(self, on: bool = True):
        self._check(load().ggq_set_static_weights(self.handle, 1 if on else 0))

    def set_direct_route_max_tokens(self, max_tokens: int = 32):
        self._check(load().ggq_set_direct_route_max_tokens(self.handle, int(max_tokens)))

    def scratch_bytes(self) -> int:
        return load().ggq_scratch_bytes(self.handle)

    def set_moe_counters(self, pairs=None, calls=None):
        """Expert-load telemetry: int64 CUDA tensors pairs [E] and calls [2], or None to stop."""
        n = 0 if pairs is None else pairs.numel()
        self._check(load().ggq_set_moe_counters(self.handle, _ptr(pairs, "int64"), n, _ptr(calls, "int64")))

    def sync_status(self, stream=None):
        self._check(load().ggq_sync_status(self.handle, self._stream(stream)))

    def quantize_act(self, act: str, x, out=None, stream=None):
        T, K = x.shape
        if out is None:
            out = self._torch.empty((T, row_bytes(act, K)), dtype=self._torch.uint8, device=x.device)
        self._check(load().ggq_quantize_act(self.handle, TYPE[act], _ptr(x, "float32"), T, K, _ptr(out, "uint8"),
                                            self._stream(stream)))
        return out

    def dequant(self, fmt: str, blocks, rows: int, K: int, out=None, stream=None):
        if out is None:
            out = self._torch.empty((rows, K), dtype=self._torch.float32, device=blocks.device)
        self._check(load().ggq_dequant(self.handle, TYPE[fmt], _ptr(blocks), rows, K, _ptr(out, "float32"),
                                       self._stream(stream)))
        return out

    def mul_mat_vec(self, fmt: str, W, N: int, K: int, X, Y=None, stream=None, reserve=True):
        T = X.shape[0]
        if Y is None:
            Y = self._torch.empty((T, N), dtype=self._torch.float32, device=X.device)
        if reserve:
            self.reserve(max_tokens=T, max_k=K, stream=stream)
        self._check(load().ggq_mul_mat_vec(self.handle, TYPE[fmt], _ptr(W), N, K, _ptr(X, "float32"), T,
                                           _ptr(Y, "float32"), self._stream(stream)))
        return Y

    def mul_mat_vec_q(self, fmt: str, W, N: int, K: int, Xq, T: int, Y=None, stream=None):
        if Y is None:
            Y = self._torch.empty((T, N), dtype=self._torch.float32, device=Xq.device)
        self._check(load().ggq_mul_mat_vec_q(self.handle, TYPE[fmt], _ptr(W), N, K, _ptr(Xq), T, _ptr(Y, "float32"),
                                             self._stream(stream)))
        return Y

    def mul_mat_vec_qa(self, fmt: str, act: str, W, N: int, K: int, Xq, T: int, Y=None, stream=None):
        if Y is None:
            Y = self._torch.empty((T, N), dtype=self._torch.float32, device=Xq.device)
        self._check(load().ggq_mul_mat_vec_qa(self.handle, TYPE[fmt], TYPE[act], _ptr(W), N, K, _ptr(Xq), T,
                                              _ptr(Y, "float32"), self._stream(stream)))
        return Y

    def block_dots_qa(self, fmt: str, act: str, W, N: int, K: int, Xq, T: int, stream=None):
        nc = K // BLOCK_ELEMS[fmt] * (2 if fmt in ("Q4_K", "Q5_K", "Q2_K") else 1)
        out = self._torch.empty((T, N, nc), dtype=self._torch.int32, device=Xq.device)
        self._check(load().ggq_block_dots_qa(self.handle, TYPE[fmt], TYPE[act], _ptr(W), N, K, _ptr(Xq), T,
                                             _ptr(out), self._stream(stream)))
        return out

    def block_dots(self, fmt: str, W, N: int, K: int, Xq, T: int, stream=None):
        nc = K // BLOCK_ELEMS[fmt] * (2 if fmt in ("Q4_K", "Q5_K", "Q2_K") else 1)
        out = self._torch.empty((T, N, nc), dtype=self._torch.int32, device=Xq.device)
        self._check(load().ggq_block_dots(self.handle, TYPE[fmt], _ptr(W), N, K, _ptr(Xq), T, _ptr(out),
                                          self._stream(stream)))
        return out

    def moe_weights(self, gate_fmt, gate, up_fmt, up, down_fmt, down):
        return ggq_moe_weights(TYPE[gate_fmt], TYPE[up_fmt], TYPE[down_fmt], _ptr(gate), _ptr(up), _ptr(down))

    def moe_experts(self, weights: ggq_moe_weights, E, H, I, top_k, X, logits=None, ids=None, route_w=None,
                    Y=None, dump: dict | None = None, stream=None, reserve=True):
        T = X.shape[0]
        if Y is None:
            Y = self._torch.empty((T, H), dtype=self._torch.float32, device=X.device)
        if reserve:
            self.reserve(max_tokens=T, n_experts=E, hidden=H, inter=I, top_k=top_k, stream=stream)
        d = None
        if dump is not None:
            d = ggq_moe_dump(**{k: _ptr(v) for k, v in dump.items()})
        dp = ctypes.byref(d) if d is not None else None
        if logits is not None:
            st = load().ggq_moe_experts(self.handle, ctypes.byref(weights), E, H, I, top_k, _ptr(X, "float32"),
                                        _ptr(logits, "float32"), T, _ptr(Y, "float32"), dp, self._stream(stream))
        else:
            st = load().ggq_moe_experts_routed(self.handle, ctypes.byref(weights), E, H, I, top_k, _ptr(X, "float32"),
                                               _ptr(ids, "int32"), _ptr(route_w, "float32"), T, _ptr(Y, "float32"),
                                               dp, self._stream(stream))
        self._check(st)
        return Y


def _moe_q(ctx, weights, E, H, I, top_k, Xq, logits, Y=None, dump=None, stream=None, reserve=True):
    """ggq_moe_experts_q: the layer on pre-quantized Q8_K activations Xq [T][H/256*292] (uint8)."""
    T = Xq.shape[0]
    if Y is None:
        Y = ctx._torch.empty((T, H), dtype=ctx._torch.float32, device=Xq.device)
    if reserve:
        ctx.reserve(max_tokens=T, n_experts=E, hidden=H, inter=I, top_k=top_k, stream=stream)
    d = ggq_moe_dump(**{k: _ptr(v) for k, v in dump.items()}) if dump is not None else None
    ctx._check(load().ggq_moe_experts_q(ctx.handle, ctypes.byref(weights), E, H, I, top_k, _ptr(Xq, "uint8"),
                                        _ptr(logits, "float32"), T, _ptr(Y, "float32"),
                                        ctypes.byref(d) if d is not None else None, ctx._stream(stream)))
    return Y


Context.moe_experts_q = _moe_q


def supported(w: str, act: str, op: str) -> bool:
    return bool(load().ggq_supported(TYPE.get(w, -1), TYPE.get(act, -1), OP[op]))
