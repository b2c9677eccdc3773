"""Shared helpers for the tests: tolerance check and tensor plumbing."""
import numpy as np

# fp16 error bound: |y - y_ref| <= 4e-3 * sum_k |w_mk * x_kn| + 1e-5 per element
REL = 4e-3
ABS = 1e-5


def within_bound(y_f16: np.ndarray, y_ref: np.ndarray, sumabs: np.ndarray) -> np.ndarray:
    y = y_f16.astype(np.float64)
    return np.abs(y - y_ref) <= REL * sumabs + ABS


def assert_within_bound(y_f16, y_ref, sumabs, what=""):
    ok = within_bound(y_f16, y_ref, sumabs)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(tuple(int(i) for i in b), float(y_f16[tuple(b)]), float(y_ref[tuple(b)]),
                   float(sumabs[tuple(b)])) for b in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside the bound, e.g. {detail}")


def to_dev_f16(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).to(dev)


def to_dev(a: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def sample_rows(M: int, per_strip: int, seed: int) -> np.ndarray:
    """per_strip distinct rows from every 64-row strip (all strips covered)."""
    g = np.random.Generator(np.random.PCG64(seed))
    rows = [s * 64 + np.sort(g.choice(64, size=per_strip, replace=False)) for s in range(M // 64)]
    return np.concatenate(rows)


_TUNE_DEFAULTS = {}


def tune(knob: str, value=None):
    """Set a process-wide tuning knob of the library (bsp_set_tuning; names
    as in ``bitmap_encoded_unstructured_gb300.TUNE``); value None restores
    the value it had when the first test touched the knobs."""
    import bitmap_encoded_unstructured_gb300 as bsp
    if not _TUNE_DEFAULTS:
        _TUNE_DEFAULTS.update({k: bsp.get_tuning(k) for k in bsp.TUNE})
    bsp.set_tuning(knob, _TUNE_DEFAULTS[knob] if value is None else int(value))


def restore_tuning():
    """Every knob back to its starting value (after a test that changed some)."""
    if _TUNE_DEFAULTS:
        import bitmap_encoded_unstructured_gb300 as bsp
        for k, v in _TUNE_DEFAULTS.items():
            bsp.set_tuning(k, v)
