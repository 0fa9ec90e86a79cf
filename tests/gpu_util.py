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
