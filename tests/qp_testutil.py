"""Helpers shared by the GPU parity tests: device copies, NaN-guarded output
buffers, and the GEMM tolerance check."""
import numpy as np

F32_NAN = 0x7FC00000
F16_NAN = 0x7E00


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(n, dtype, cols):
    """A device buffer holding n elements with a NaN guard band of one output
    row plus 4 KiB on each side; returns (buffer, interior view, guard)."""
    import torch
    esize = 4 if dtype == torch.float32 else 2
    g = cols + 4096 // esize
    g = (g + 15) // 16 * 16                 # keeps the interior 64-byte aligned
    if dtype == torch.float32:
        buf = torch.full((n + 2 * g,), F32_NAN, dtype=torch.int32, device="cuda").view(torch.float32)
    else:
        buf = torch.full((n + 2 * g,), F16_NAN, dtype=torch.int16, device="cuda").view(torch.float16)
    return buf, buf[g:g + n], g


def guard_intact(buf, g, n):
    import torch
    bits = buf.view(torch.int32 if buf.dtype == torch.float32 else torch.int16).cpu().numpy()
    nan = F32_NAN if buf.dtype == torch.float32 else np.int16(F16_NAN)
    return bool(np.all(bits[:g] == nan) and np.all(bits[g + n:] == nan))


def gemm_errors(Y, Yref, A):
    """(relative Frobenius error, max of |Y - Yref| / (4e-3 * A))."""
    Y = np.asarray(Y, np.float64)
    err = Y - Yref
    rel = np.linalg.norm(err) / max(np.linalg.norm(Yref), 1e-300)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(A > 0, np.abs(err) / (4e-3 * A), np.where(err == 0, 0.0, np.inf))
    return rel, float(ratio.max()) if ratio.size else 0.0


def assert_gemm_within_tolerance(Y, Yref, A, what=""):
    """The acceptance bar for the projection: relative Frobenius error <= 1e-3
    and every |y - y_ref| <= 4e-3 * sum_k |x||w| against the fp64 oracle."""
    rel, ratio = gemm_errors(Y, Yref, A)
    assert rel <= 1e-3, "%s: relative Frobenius error %.3g > 1e-3" % (what, rel)
    assert ratio <= 1.0, "%s: elementwise error reaches %.3g of the 4e-3*sum|x||w| bound" % (what, ratio)
    return rel, ratio


class GemmErrorTally:
    """The projection's acceptance bar over an output checked piece by piece
    (row blocks): the relative Frobenius error of the whole, and the worst
    elementwise |y - y_ref| / (4e-3 * sum_k |x||w|)."""

    def __init__(self, what=""):
        self.what = what
        self.se = 0.0
        self.sr = 0.0
        self.worst = 0.0
        self.n = 0

    def add(self, Y, Yref, A):
        Y = np.asarray(Y, np.float64)
        assert np.isfinite(Y).all(), "%s: non-finite output" % self.what
        err = Y - Yref
        self.se += float(np.sum(err * err))
        self.sr += float(np.sum(Yref * Yref))
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(A > 0, np.abs(err) / (4e-3 * A), np.where(err == 0, 0.0, np.inf))
        if ratio.size:
            self.worst = max(self.worst, float(ratio.max()))
        self.n += Y.size

    def check(self):
        rel = (self.se / self.sr) ** 0.5 if self.sr > 0 else (0.0 if self.se == 0 else float("inf"))
        assert self.n > 0
        assert rel <= 1e-3, "%s: relative Frobenius error %.3g > 1e-3" % (self.what, rel)
        assert self.worst <= 1.0, "%s: elementwise error reaches %.3g of the bound" % (self.what, self.worst)
        return rel, self.worst
