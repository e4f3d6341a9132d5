"""CPU checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and answers the per-format support query.  No compute call
runs here (there is no GPU)."""
import os
import re

import pytest

import gguf_block_quant_ggq_gb300 as ggq
from gguf_block_quant_ggq_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ggq.load()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "ggq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ggq_[a-z_]+)\s*\(", text)))


def test_header_declares_the_bound_entry_points():
    assert _declared_symbols() == sorted(ggq.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_support_query_per_format(lib):
    ok = [("Q4_0", "Q8_1"), ("Q8_0", "Q8_K"), ("Q4_K", "Q8_K"), ("Q5_K", "Q8_K"), ("Q6_K", "Q8_K"),
          ("MXFP4", "Q8_K"), ("Q4_0", "Q8_0"), ("Q8_0", "Q8_0"), ("Q2_K", "Q8_K"), ("Q3_K", "Q8_K")]
    for w in ggq.TYPE:
        for a in ggq.TYPE:
            assert ggq.supported(w, a, "mul_mat_vec") == ((w, a) in ok)
            moe_ok = a == "Q8_K" and w in ("Q8_0", "Q4_K", "Q5_K", "Q6_K", "MXFP4")
            assert ggq.supported(w, a, "moe") == moe_ok
        assert ggq.supported(w, "Q8_K", "dequant") == (w in ("Q4_0", "Q8_0", "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K",
                                                             "MXFP4"))
    assert ggq.supported("Q4_0", "Q8_1", "quantize_act") and ggq.supported("Q4_0", "Q8_K", "quantize_act")
    assert ggq.supported("Q4_0", "Q8_0", "quantize_act")
    assert not ggq.supported("Q4_0", "Q4_0", "quantize_act")
    # formats outside the eight (e.g. Q4_1 = 3, IQ2_XXS = 16) are refused, not mapped
    assert lib.ggq_supported(16, ggq.TYPE["Q8_K"], 2) == 0
    assert lib.ggq_supported(3, ggq.TYPE["Q8_1"], 2) == 0


def test_type_ids_are_gguf_tensor_types():
    assert ggq.TYPE == {"Q4_0": 2, "Q8_0": 8, "Q8_1": 9, "Q2_K": 10, "Q3_K": 11, "Q4_K": 12, "Q5_K": 13,
                        "Q6_K": 14, "Q8_K": 15, "MXFP4": 39}


def test_null_context_is_rejected_without_touching_a_device(lib):
    assert lib.ggq_reserve(None, None, None) == 1
    assert lib.ggq_destroy(None) == 1
    assert lib.ggq_last_error(None) == b"null context"


def test_binding_refuses_host_tensors_before_any_call():
    # the C calls take device pointers: a host tensor is refused by the binding
    # itself, before any pointer reaches the library; None passes NULL
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="CUDA tensors"):
        ggq._ptr(torch.zeros(4))
    assert ggq._ptr(None) is None
