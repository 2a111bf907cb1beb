"""CPU oracle of device-side sampling beyond greedy (test infrastructure).

Reading of the pages' serving step ("Add native Qwen3 14B A8W8 serving path",
pypto-serving PR #48, "Performance": greedy decoding at temperature 0, top_p 1;
"Add Qwen3 A8W8 L2 runner foundation", pypto-serving PR #61, "Related":
sampling on the device): for one logits row l over the vocabulary,
  * temperature T <= 0: greedy argmax (lowest index on ties);
  * otherwise z = (l - max l) / T, p = exp(z) (unnormalised, max 1);
  * top_p < 1 keeps the nucleus: with p32 = float32(p), the largest threshold
    tau among the p32 values such that the tokens with p32 >= tau carry at
    least top_p of the total mass (ties at tau all kept);
  * the token is drawn from softmax(z) restricted to the nucleus by the
    Gumbel-max rule: argmax over the nucleus of z_i + g_i, with g_i =
    -log(-log(u_i)) and u_i uniform in (0, 1) (Gumbel 1954; the argmax of
    Gumbel-perturbed log-probabilities is distributed as the softmax).
u_i comes from the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror
and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011): key =
(seed low 32 bits, seed high 32 bits), counter = (i, row, step low, step high),
output word 0 = x, u = (floor(x / 2^8) + 1/2) / 2^24 (24 bits, exact in
float32, never 0 or 1).
Arithmetic here is float64 (the real-valued definition); the device evaluates
the exponentials and masses in two-float arithmetic and the Gumbel noise in
float32.
"""
from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on arrays of 32-bit counter words (uint64
    arrays holding 32-bit values) and a 32-bit key pair; returns four words."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK for c in (c0, c1, c2, c3))
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0            # < 2^64: exact in uint64
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & _MASK, lo1, (hi0 ^ c3 ^ k1) & _MASK, lo0
    return c0, c1, c2, c3


def uniforms(n: int, row: int, seed: int, step: int) -> np.ndarray:
    """u_i in (0, 1), i < n, for one row of one step (float64)."""
    i = np.arange(n, dtype=np.uint64)
    x, _, _, _ = philox4x32_10(i, np.full(n, row, np.uint64), np.full(n, step & 0xFFFFFFFF, np.uint64),
                               np.full(n, (step >> 32) & 0xFFFFFFFF, np.uint64),
                               seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    return ((x >> np.uint64(8)).astype(np.float64) + 0.5) / 16777216.0


def nucleus(z: np.ndarray, top_p: float) -> np.ndarray:
    """Boolean mask of the nucleus of exp(z) (z <= 0, max 0) at top_p."""
    p = np.exp(z)
    if top_p >= 1.0:
        return np.ones(z.shape, bool)
    p32 = p.astype(np.float32)
    order = np.argsort(-p32, kind="stable")
    cum = np.cumsum(p[order])
    need = top_p * p.sum()
    k = int(np.searchsorted(cum, need))          # first position reaching the mass
    k = min(k, len(order) - 1)
    tau = p32[order[k]]
    return p32 >= tau


def sample_rows(logits, temperature: float, top_p: float, seed: int, step: int) -> np.ndarray:
    """Next token of each logits row [B, V] (float32) -> int32 [B]."""
    logits = np.asarray(logits, dtype=np.float32)
    B, V = logits.shape
    # the device receives both parameters as float32
    temperature = float(np.float32(temperature))
    top_p = float(np.float32(top_p))
    out = np.empty(B, dtype=np.int32)
    for b in range(B):
        row = logits[b].astype(np.float64)
        if temperature <= 0.0:
            out[b] = int(np.argmax(row))      # first maximum
            continue
        z = (row - row.max()) / float(temperature)
        keep = nucleus(z, top_p)
        g = -np.log(-np.log(uniforms(V, b, seed, step)))
        key = np.where(keep, z + g, -np.inf)
        out[b] = int(np.argmax(key))
    return out
