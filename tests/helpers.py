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
