"""Helpers for the GPU parity tests: device upload/download of bf16 bit
patterns and the tolerance check.

Tolerance (for the bf16-input / fp32-accumulate path, element-wise against
the fp64 oracle on the identical bf16 inputs):
  relative L2 error  ||gpu - ref|| / ||ref||  <= 5e-3, and
  |gpu - ref| <= 1e-2 * S  per element, S = the sum of |product| terms of that
  element (plus |bias| for pooled outputs).
"""
import numpy as np

REL_L2 = 5e-3
ELEM = 1e-2


def torch_mod():
    import torch
    return torch


def dev_bf16(u16):
    torch = torch_mod()
    a = np.ascontiguousarray(u16, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def dev(a):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16_f64(t):
    torch = torch_mod()
    u = t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def empty_bf16(shape, fill=None):
    torch = torch_mod()
    t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t


def assert_close(gpu, ref, S, what, rel_l2=REL_L2, elem=ELEM):
    gpu = np.asarray(gpu, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    S = np.asarray(S, np.float64).ravel()
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    assert rel <= rel_l2, f"{what}: relative L2 error {rel:.3e} > {rel_l2}"
    bound = elem * S + 1e-30
    bad = err > bound
    if np.any(bad):
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {int(bad.sum())} elements over 1e-2*S; worst at {i}: "
                             f"gpu={gpu[i]!r} ref={ref[i]!r} S={S[i]!r}")
    return rel


GUARD_BYTES = 4096
GUARD_FILL = 0xA5


def guarded(shape, dtype, fill=None):
    """A device tensor of `shape`/`dtype` placed between two 4 KB guard bands of
    a sentinel byte (in place of a memory checker: a kernel that writes past
    either end of its output changes them).  Returns (tensor, check); check()
    asserts both bands are intact.  The tensor starts 4 KB into the buffer, so
    it keeps the 16-byte alignment the library requires."""
    torch = torch_mod()
    n = int(np.prod(shape)) if len(shape) else 1
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8, device="cuda")
    t = buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
    if fill is not None:
        t.fill_(fill)

    def check(what="output"):
        head = buf[:GUARD_BYTES]
        tail = buf[GUARD_BYTES + nbytes:]
        assert bool((head == GUARD_FILL).all()), f"{what}: write before the start of the tensor"
        assert bool((tail == GUARD_FILL).all()), f"{what}: write past the end of the tensor"
    return t, check


def tile_cover_pts(rng, c_out, c_in, k_min=512, co_blk=64, ci_blk=32):
    """Filter elements (co, kd, kh, kw, ci) with at least one in every
    (c_out block x tap x c_in block) tile of the weight gradient -- the unit of
    its split-K partials and of the MMA accumulators -- topped up with uniform
    random elements to at least k_min."""
    pts = []
    for cb in range(0, c_out, co_blk):
        for t in range(27):
            for ib in range(0, c_in, ci_blk):
                co = int(rng.integers(cb, min(cb + co_blk, c_out)))
                ci = int(rng.integers(ib, min(ib + ci_blk, c_in)))
                pts.append((co, t // 9, (t // 3) % 3, t % 3, ci))
    while len(pts) < k_min:
        pts.append((int(rng.integers(0, c_out)), int(rng.integers(0, 3)), int(rng.integers(0, 3)),
                    int(rng.integers(0, 3)), int(rng.integers(0, c_in))))
    return np.array(pts, dtype=np.int64)
