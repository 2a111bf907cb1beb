"""Helpers shared by the GPU parity tests: host<->device moves and metrics."""
import numpy as np


def to_dev(a, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.uint16:
        t = t.view(torch.bfloat16)
    return t.to(device)


def to_host(t) -> np.ndarray:
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(h) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def norm_max_abs(a, b) -> float:
    """max |a - b| divided by the RMS of b."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    rms = np.sqrt(np.mean(b * b))
    return float(np.max(np.abs(a - b)) / (rms if rms > 0 else 1.0))


def bf16_ulp_diff(a, b) -> np.ndarray:
    """Distance in BF16 units in the last place (sign-magnitude ordered)."""
    def ordered(h):
        h = np.asarray(h, np.int32)
        return np.where(h & 0x8000, -(h & 0x7FFF), h & 0x7FFF)
    return np.abs(ordered(a) - ordered(b))


# Per-layer bar: relative L2 <= 5e-3 literally, and max-abs <= 3e-2 measured on
# outputs normalised by the oracle's RMS (the raw outputs have RMS in the
# thousands, where one BF16 unit in the last place is far above 3e-2).
LAYER_REL_L2 = 5e-3
LAYER_NORM_MAX_ABS = 3e-2
STEP_REL_L2 = 2e-2


def assert_layer_close(gpu_bf16, ref_bf16, what="", flipped_rows=(), max_abs_bar=None):
    """The per-layer bar on every row whose quantisation decisions match the
    oracle's; rows listed in `flipped_rows` (a row scale differs because the
    row's absmax element differs by one BF16 unit upstream) are held to the
    step bar instead, since one such flip moves every INT8 code of the row."""
    a = bf16_to_f64(gpu_bf16)
    b = bf16_to_f64(ref_bf16)
    a2 = a.reshape(a.shape[0], -1)
    b2 = b.reshape(b.shape[0], -1)
    keep = np.ones(a2.shape[0], bool)
    keep[list(flipped_rows)] = False
    r = rel_l2(a2[keep], b2[keep])
    m = norm_max_abs(a2[keep], b2[keep])
    assert r <= LAYER_REL_L2, f"{what}: rel-L2 {r:.3e} > {LAYER_REL_L2}"
    bar = LAYER_NORM_MAX_ABS if max_abs_bar is None else max_abs_bar
    assert m <= bar, f"{what}: normalised max-abs {m:.3e} > {bar}"
    for row in flipped_rows:
        rr = rel_l2(a2[row], b2[row])
        assert rr <= STEP_REL_L2, f"{what}: row {row} with a flipped scale: rel-L2 {rr:.3e}"
    return r, m


def bf16_close(gpu_bf16, ref_bf16, ulps: float, rel_floor: float) -> np.ndarray:
    """Elementwise |a - b| <= ulps BF16 units of max(|b|, rel_floor * rms(b)).

    Plain unit-in-the-last-place distances blow up for values near zero
    (cancellation, or a float32 exp that underflows where the double one does
    not); the floor measures those against the tensor's own scale."""
    a = bf16_to_f64(gpu_bf16)
    b = bf16_to_f64(ref_bf16)
    rms = np.sqrt(np.mean(b * b)) if b.size else 0.0
    mag = np.maximum(np.abs(b), max(rel_floor * rms, 1e-30))
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    return np.abs(a - b) <= ulps * ulp
