"""Shared helpers of the parity tests: moving arrays between NumPy and the
device, exact comparison of float bit patterns, and the spec float
tolerance."""
import numpy as np

RTOL, ATOL = 1e-5, 1e-7  # float buffers after many steps


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().cpu().numpy()


def u32(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype in (np.float32, np.int32) else a.astype(np.uint32)


def assert_bits_equal(got, want, what=""):
    g, w = u32(got).ravel(), u32(want).ravel()
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.nonzero(g != w)[0]
    if bad.size:
        i = bad[0]
        gf = np.ascontiguousarray(got).ravel()[i]
        wf = np.ascontiguousarray(want).ravel()[i]
        raise AssertionError(f"{what}: {bad.size} of {g.size} differ; first at {i}: "
                             f"got {gf!r} ({g[i]:#010x}) want {wf!r} ({w[i]:#010x})")


def assert_close(got, want, what="", rtol=RTOL, atol=ATOL):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want)
    lim = atol + rtol * np.abs(want)
    bad = np.nonzero(~(err <= lim))[0] if got.ndim == 1 else np.argwhere(~(err <= lim))
    assert bad.size == 0, f"{what}: {len(bad)} outside rel {rtol} / abs {atol}; first {bad[:3]}"


def bf16_tensor(bits_u16):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).cuda().view(torch.bfloat16)


GUARD = 64  # elements of poisoned margin on each side of a guarded buffer
POISON = 0xA5


class Guarded:
    """A device buffer with GUARD poisoned elements (bytes 0xA5) on each side,
    for catching stray writes just outside an output (compute-sanitizer
    stand-in): `t` is the buffer itself, `intact()` checks both margins.
    The margin is a multiple of 16 bytes for 4-byte types, so the buffer
    keeps the alignment of the allocation."""

    def __init__(self, shape, dtype, value=None):
        import torch
        shape = (shape,) if isinstance(shape, int) else tuple(shape)
        count = int(np.prod(shape))
        isz = torch.empty((), dtype=dtype).element_size()
        self.mb = GUARD * isz
        self.raw = torch.full((count * isz + 2 * self.mb,), POISON, dtype=torch.uint8,
                              device="cuda")
        self.t = self.raw[self.mb:self.mb + count * isz].view(dtype).view(shape)
        if value is not None:
            v = torch.as_tensor(np.ascontiguousarray(value)).to(self.t.device)
            self.t.copy_(v.view(self.t.dtype).view(shape) if v.dtype != self.t.dtype and
                         v.element_size() == isz else v.view(shape))

    def intact(self):
        m = host(self.raw[: self.mb]), host(self.raw[-self.mb:])
        return bool((m[0] == POISON).all() and (m[1] == POISON).all())


def assert_guards(what, *guarded):
    for i, g in enumerate(guarded):
        assert g.intact(), f"{what}: a write landed in the margin of guarded buffer {i}"
