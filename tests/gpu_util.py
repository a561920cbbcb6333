"""Helpers for the GPU parity tests: device buffers at chosen alignments and the tolerance."""
import numpy as np
import torch

TOL_REL = 1e-5
TOL_ABS = 1e-6


# worst |y - y_ref| / bound seen per check (printed in the session summary by conftest)
WORST_RATIO = {}


def assert_within_tolerance(y, y_ref, a_ref, what=""):
    """|y - y_ref| <= 1e-5 * sum|w x| + 1e-6, element by element (the stated GEMV bound).
    Returns the worst ratio of error to bound (recorded under `what`)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = TOL_REL * a_ref + TOL_ABS
    ratio = float(np.max(err / bound)) if err.size else 0.0
    if what:
        WORST_RATIO[what] = max(ratio, WORST_RATIO.get(what, 0.0))
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    return ratio


def device_bytes(arr: np.ndarray, offset: int = 0, device="cuda"):
    """Copy host bytes to a device buffer whose start is `offset` bytes past a 256-byte
    aligned address; returns (view tensor, backing tensor)."""
    raw = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
    back = torch.zeros(raw.size + offset + 256, dtype=torch.uint8, device=device)
    base = (-back.data_ptr()) % 256
    view = back[base + offset: base + offset + raw.size]
    view.copy_(torch.from_numpy(raw))
    assert (view.data_ptr() - offset) % 256 == 0
    return view, back


def f32_with_canary(rows, cols, device="cuda", guard=64):
    """fp32 [rows][cols] output buffer followed by `guard` canary words."""
    buf = torch.full((rows * cols + guard,), float("nan"), dtype=torch.float32, device=device)
    canary = torch.tensor([1234.5], dtype=torch.float32, device=device)
    buf[rows * cols:] = canary
    return buf, buf[: rows * cols].view(rows, cols)


def canary_intact(buf, n):
    return bool(torch.all(buf[n:] == 1234.5).item())
