"""Helpers for the GPU parity tests: device copies and bound checks."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def dev(a, offset_bytes: int = 0):
    """numpy array -> cuda tensor.  With offset_bytes > 0 the data starts that
    many bytes into a larger allocation (to exercise unaligned bases); the
    returned object is (tensor_holding_memory, data_pointer_int)."""
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if offset_bytes == 0:
        return t
    raw = np.ascontiguousarray(a).view(np.uint8).ravel()
    buf = torch.zeros(raw.size + offset_bytes + 16, dtype=torch.uint8, device="cuda")
    buf[offset_bytes:offset_bytes + raw.size] = torch.from_numpy(raw).cuda()
    return buf, buf.data_ptr() + offset_bytes


def empty(shape, dtype=torch.float32):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda") if dtype.is_floating_point \
        else torch.zeros(shape, dtype=dtype, device="cuda")


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_within(got, ref, bound, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside bound; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} err {err[tuple(i)]:.3e} "
                             f"bound {np.broadcast_to(bound, got.shape)[tuple(i)]:.3e}")
    return float((err / bound).max()) if err.size else 0.0


def status_clean(lq):
    rc, bits = lq.lq_device_status()
    assert rc == 0 and bits == 0, f"device status rc={rc} bits={bits}"
