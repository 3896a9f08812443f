"""Helpers of the GPU parity tests: device copies with guard bands and controlled base alignment, and the bitwise
comparison rule (every non-NaN output bit-exact; NaN outputs at exactly the same positions, payload and sign not
compared, since x86/Arm fmaf propagates an input NaN's payload while the GPU returns its canonical NaN)."""

from __future__ import annotations

import numpy as np
import torch

GUARD = 64                       # floats of guard band on each side
CANARY = np.uint32(0x7FC0DEAD)   # a quiet-NaN pattern no kernel writes


class DevArray:
    """A float32 device copy of a numpy array inside a guarded buffer; `offset_floats` past a 256-byte boundary."""

    def __init__(self, a: np.ndarray, offset_floats: int = 0, row_pad: int = 0):
        a = np.ascontiguousarray(a, np.float32)
        self.shape = a.shape
        if row_pad:
            N, R, W = a.shape
            ld = W + row_pad
            body = np.zeros((N, R, ld), np.float32)
            body[:, :, :W] = a
            self.ld = ld
        else:
            body = a
            self.ld = a.shape[-1]
        n = body.size
        self.buf = torch.empty(n + 2 * GUARD + 64 + 256 // 4, dtype=torch.float32, device="cuda")
        base = self.buf.data_ptr()
        start = (-(base // 4)) % (256 // 4) + GUARD + offset_floats
        self.start = start
        self.n = n
        guard = torch.from_numpy(np.full(self.buf.numel(), CANARY, np.uint32).view(np.float32)).cuda()
        self.buf.copy_(guard)
        flat = self.buf[start:start + n]
        flat.copy_(torch.from_numpy(body.reshape(-1)).cuda())
        self.body = flat.view(body.shape)
        if row_pad:
            self.t = self.body[:, :, :self.shape[-1]]
        else:
            self.t = self.body

    def host(self) -> np.ndarray:
        return np.ascontiguousarray(self.t.cpu().numpy())

    def guards_intact(self) -> bool:
        b = self.buf.cpu().numpy().view(np.uint32)
        lo = b[:self.start]
        hi = b[self.start + self.n:]
        if not (np.all(lo == CANARY) and np.all(hi == CANARY)):
            return False
        if self.ld != self.shape[-1]:   # row padding must be untouched too (it was zero)
            pad = self.body[:, :, self.shape[-1]:].cpu().numpy()
            if np.any(pad != 0):
                return False
        return True


def assert_bitwise(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (got.shape, want.shape)
    gn, wn = np.isnan(got), np.isnan(want)
    if not np.array_equal(gn, wn):
        idx = np.argwhere(gn != wn)[:5]
        raise AssertionError(f"{what}: NaN positions differ at {idx.tolist()}")
    m = ~gn
    gb = got[m].view(np.uint32)
    wb = want[m].view(np.uint32)
    bad = np.flatnonzero(gb != wb)
    if bad.size:
        k = bad[:5]
        raise AssertionError(f"{what}: {bad.size} of {gb.size} outputs differ; got {got[m][k]} want {want[m][k]}")
