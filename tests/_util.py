"""Shared helpers for the GPU parity tests (tolerances, conversions, canaries)."""
import numpy as np
import torch

# Parity tolerance on fp32 outputs: |y - y_ref| <= REL * sum_b |d_w d_x s_b| + ABS.
REL = 1e-4
ABS = 1e-6


def np_(t):
    return t.detach().cpu().numpy()


def wd_bits(wd):
    """float16 scale tensor -> uint16 bit patterns (numpy)."""
    return np_(wd.contiguous().view(torch.int16)).view(np.uint16)


def bf16_bits_np(x):
    return np_(x.contiguous().view(torch.int16)).view(np.uint16)


def abs_terms(s, wd_u16, xd):
    """sum_b |d_w[n,b] d_x[m,b] s[m,n,b]| as fp64 [M, N] from int32 block sums."""
    c = wd_u16.view(np.float16).astype(np.float64)[None, :, :] * \
        xd.astype(np.float64)[:, None, :]
    return np.abs(c * s.astype(np.float64)).sum(axis=2)


def nvfp4_terms(orc, oc, os_, og, oxq, oxd):
    """sum over 16-element half-blocks of |(g/2) s d_x S| as fp64 [M, N], S the exact sum of
    twice the E2M1 values times the activation quants (the NVFP4 product's terms)."""
    N, K = oc.shape[0], oc.shape[1] * 2
    M = oxq.shape[0]
    c2 = orc.unpack_nvfp4(oc).astype(np.float64).reshape(N, K // 16, 16)
    S = np.einsum("nbi,mbi->mnb", c2, oxq.astype(np.float64).reshape(M, K // 16, 16))
    s = orc.e4m3_to_f32(os_).astype(np.float64)
    dx = np.repeat(oxd.astype(np.float64), 2, axis=1)
    return np.abs(0.5 * float(og) * s[None] * dx[:, None, :] * S).sum(axis=2)


def assert_within(y, y_ref, terms, what=""):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    err = np.abs(y - y_ref)
    tol = REL * np.asarray(terms, np.float64) + ABS
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError("%s: %d of %d outside tolerance; worst at %s: got %r want %r "
                             "(tol %r)" % (what, int(bad.sum()), bad.size, i, y[i], y_ref[i],
                                           tol[i]))


class Guarded:
    """A CUDA buffer with sentinel guard bands on both sides of the view handed out,
    to catch out-of-bounds writes without a sanitizer."""

    def __init__(self, shape, dtype, guard_bytes=256, fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        esize = torch.empty((), dtype=dtype).element_size()
        self.g = guard_bytes // esize
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self._sentinel(self.buf)
        self.view = self.buf[self.g:self.g + n].view(shape)
        if fill is not None:
            self.view.fill_(fill)

    @staticmethod
    def _sentinel(t):
        if t.dtype.is_floating_point:
            t.fill_(-12345.0)
        else:
            t.fill_(-77)

    def intact(self):
        ref = torch.empty(self.g, dtype=self.buf.dtype, device="cuda")
        self._sentinel(ref)
        return bool(torch.equal(self.buf[:self.g], ref) and torch.equal(self.buf[-self.g:], ref))
