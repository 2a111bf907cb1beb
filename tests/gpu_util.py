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


# ---------------------------------------------------------------------------
# Element-wise bounds for float32 sums of exact products
# ---------------------------------------------------------------------------

# The LM head multiplies BF16 operands on the tensor cores with float32
# accumulation; each product is exact and the accumulated value is within a
# small multiple of the float32 unit of the absolute sum. 2^-20 of sum |h w|
# leaves room for a few dozen accumulation roundings in a row while a wrong
# operand (a permuted column, a dropped K block) moves a logit by a sizeable
# share of |h w| for that column, far above it.
LM_HEAD_REL = 2.0 ** -20


def abs_dot(x_bf16, W_bf16, chunk: int = 8192) -> np.ndarray:
    """sum_k |x[m,k]| |W[n,k]| for BF16 operands, float64, W chunked by rows."""
    xa = np.abs(bf16_to_f64(x_bf16)).astype(np.float32)
    out = np.empty((xa.shape[0], W_bf16.shape[0]), np.float64)
    for n0 in range(0, W_bf16.shape[0], chunk):
        wa = np.abs(bf16_to_f64(W_bf16[n0:n0 + chunk])).astype(np.float32)
        out[:, n0:n0 + chunk] = (xa @ wa.T).astype(np.float64)
    return out


def check_lm_head(fh_bf16, W_lm, g_logits, g_next, o_logits=None):
    """GPU logits against the oracle's LM head evaluated on the GPU's own final
    hidden rows, element by element within LM_HEAD_REL * sum |h w|, and the
    GPU's token equal to the oracle's argmax except where the oracle's top two
    are closer than twice that bound. Returns (max |diff| / bound, #near ties)."""
    import oracle
    if o_logits is None:
        o_logits = oracle.lm_head(fh_bf16, W_lm)
    bound = LM_HEAD_REL * abs_dot(fh_bf16, W_lm)
    diff = np.abs(np.asarray(g_logits, np.float64) - o_logits)
    worst = float(np.max(diff / np.maximum(bound, 1e-300)))
    assert (diff <= bound).all(), f"LM head: logits beyond the float32 bound (worst {worst:.3g}x)"
    o_next = oracle.argmax_f64(o_logits)
    ties = 0
    for b in range(o_logits.shape[0]):
        if g_next[b] != o_next[b]:
            gap = o_logits[b, o_next[b]] - o_logits[b, g_next[b]]
            assert gap <= 2 * max(bound[b, o_next[b]], bound[b, g_next[b]]), \
                f"row {b}: GPU token {g_next[b]} vs oracle {o_next[b]}, gap {gap:.3g}"
            ties += 1
    return worst, ties


def proj_error_bound(x_bf16, W_bf16, K: int) -> np.ndarray:
    """Bound on |float32 sum - exact sum| of sum_k x[m,k] W[n,k] with exact
    products: gamma_K * sum |x w|, gamma_K = K u / (1 - K u), u = 2^-24
    (any summation order), plus one more u for a residual add."""
    u = 2.0 ** -24
    gamma = (K + 1) * u / (1 - (K + 1) * u)
    return gamma * abs_dot(x_bf16, W_bf16)


def bf16_ulp_at(v) -> np.ndarray:
    """One BF16 unit in the last place at |v| (normal range)."""
    mag = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(mag)) - 7)
