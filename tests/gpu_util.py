"""Helpers shared by the GPU parity tests: device transfer, tolerance checks."""
import numpy as np

RTOL_ABS = 1e-5   # max |err| <= RTOL_ABS * sum |w * x| per output
NMSE_MAX = 1e-10  # sum err^2 / sum ref^2


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t):
    return t.detach().cpu().numpy()


def check_outputs(got, ref, absdot, what=""):
    """The fp32 acceptance: per-output error against sum |w x| and the NMSE."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > RTOL_ABS * absdot + 1e-30
    assert not bad.any(), (f"{what}: {bad.sum()} outputs over tolerance; worst ratio "
                           f"{np.max(err / np.maximum(absdot, 1e-30)):.3e}")
    den = float(np.sum(ref * ref))
    nmse = float(np.sum(err * err)) / den if den > 0 else float(np.sum(err * err))
    assert nmse <= NMSE_MAX, f"{what}: NMSE {nmse:.3e}"
    return nmse
