"""Helpers shared by the GPU parity tests: the tolerance rule and host<->device
marshalling of bf16 bit patterns."""
import numpy as np
import torch

# Attention tolerance (fp32 accumulation over bf16 inputs): an element passes
# when |gpu - oracle| <= ATOL + RTOL * |oracle|.  With an fp32 output the
# maximum absolute error must also stay within ATOL.  A bf16 output adds its
# own rounding (up to 2^-8 relative), which the RTOL term covers.
ATOL = 2e-3
RTOL = 1e-2


def to_bits(t):
    """uint16 NumPy copy of a bf16 tensor's bits (any device)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def out_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_attention_close(got, ref, f32_out, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    d = np.abs(got - ref)
    bad = d > ATOL + RTOL * np.abs(ref)
    big = np.abs(ref) > 1e-2
    max_rel = float((d[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    msg = "%s: max abs %.3g, max rel(|ref|>1e-2) %.3g, %d/%d outside tolerance" % (
        what, d.max(), max_rel, int(bad.sum()), d.size)
    assert not bad.any(), msg
    if f32_out:
        assert d.max() <= ATOL, msg
    return float(d.max()), max_rel
