"""Oracle: the packed 4-bit group-quantized weight format, in plain fp64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Why a format of our own
    The pages store experts as EXL3 trellis codes (GLM-5.3-Flash EXL3 3.05bpw on
    1x RTX PRO 6000 recipe, ``summary`` and ``config.expert_cache.layout``: about
    9 MiB per expert at 3.05 bits per weight), but they never define the codebook
    (the glm53-flash-offload README, "CPU tier" bullet, names the trellis variant
    and nothing more).  This library therefore defines a plain symmetric 4-bit group format
    with fp16 scales.  It is a weight-only quantization, as on the pages.

Definition (for a weight matrix ``W`` of shape ``[N, K]``, fp32, K contiguous)
    * groups are ``G`` consecutive elements along K (``G`` divides K);
    * scale ``s = fp16_RNE(max|w in group| / 7)``, the division done in fp64 and the
      fp64 quotient rounded to fp16 with round-to-nearest-even;
    * a group whose scale rounds to 0 stores ``q = 0`` for every element;
    * otherwise ``q = clamp(round_half_even(w / s), -8, 7)``, ``w / s`` in fp64;
    * nibble ``u = q + 8`` in [0, 15]; element ``(n, k)`` goes to byte
      ``(n*K + k) // 2`` of the packed array, even k in the low nibble;
    * scales are stored fp16, row-major ``[N, K // G]``;
    * dequantized weight ``w_hat = (u - 8) * s``, exact in fp32 and fp64.

    A scale that is not finite (non-finite weights, or ``max|w| / 7`` beyond the
    fp16 range) is an error.

Gate/up interleave
    The gate and up projections of one expert (each ``[I, H]``) are stored as one
    ``[2I, H]`` matrix whose rows alternate in blocks of 16: combined row ``r``
    belongs to block ``b = r // 32``; offset ``o = r % 32``; rows with ``o < 16``
    are gate row ``16*b + o``, the others up row ``16*b + o - 16``.  The row order
    is a storage choice only; ``deinterleave_rows`` reads it back with its own
    index formula.
"""

from __future__ import annotations

import numpy as np

QMIN = -8
QMAX = 7
INTERLEAVE = 16


def group_scales(W: np.ndarray, G: int) -> np.ndarray:
    """fp16 scales ``[N, K//G]``: RNE of ``max|w| / 7`` computed in fp64."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % G:
        raise ValueError(f"K={K} is not a multiple of the group size {G}")
    amax = np.abs(W.astype(np.float64)).reshape(N, K // G, G).max(axis=2)
    with np.errstate(over="ignore", invalid="ignore"):
        s16 = (amax / 7.0).astype(np.float16)
    if not np.all(np.isfinite(s16)):
        raise ValueError("a group scale is not finite (non-finite weight or |w| beyond 7*65504)")
    return s16


def quantize_codes(W: np.ndarray, G: int) -> tuple[np.ndarray, np.ndarray]:
    """Signed codes ``q`` (int8, ``[N, K]``) and fp16 scales ``[N, K//G]``."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    s16 = group_scales(W, G)
    s = s16.astype(np.float64)[:, :, None]                     # [N, K//G, 1]
    Wg = W.astype(np.float64).reshape(N, K // G, G)
    safe = np.where(s > 0.0, s, 1.0)
    q = np.clip(np.rint(Wg / safe), QMIN, QMAX)                # rint: half to even
    q = np.where(s > 0.0, q, 0.0)
    return q.reshape(N, K).astype(np.int8), s16


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """``[N, K]`` signed codes -> ``[N, K//2]`` bytes; even k in the low nibble."""
    q = np.asarray(q)
    N, K = q.shape
    if K % 2:
        raise ValueError("K must be even")
    u = (q.astype(np.int16) + 8).astype(np.uint8)
    if u.max(initial=0) > 15:
        raise ValueError("code out of range")
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray, K: int) -> np.ndarray:
    """``[N, K//2]`` bytes -> ``[N, K]`` unsigned nibbles ``u`` in [0, 15]."""
    packed = np.asarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    u = np.empty((N, K), dtype=np.uint8)
    u[:, 0::2] = packed & 0x0F
    u[:, 1::2] = packed >> 4
    return u


def quantize_matrix(W: np.ndarray, G: int) -> tuple[np.ndarray, np.ndarray]:
    """fp32 ``[N, K]`` -> (packed uint8 ``[N, K//2]``, fp16 scales ``[N, K//G]``)."""
    q, s16 = quantize_codes(W, G)
    return pack_nibbles(q), s16


def dequantize_matrix(packed: np.ndarray, scales: np.ndarray, K: int, G: int) -> np.ndarray:
    """Exact dequantized weights ``(u - 8) * s`` as fp64 ``[N, K]``."""
    u = unpack_nibbles(packed, K).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    N = u.shape[0]
    return ((u - 8.0).reshape(N, K // G, G) * s[:, :, None]).reshape(N, K)


def interleave_rows(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """Stack gate and up row-blocks of 16 alternately: ``[I, ...] x 2 -> [2I, ...]``."""
    gate = np.asarray(gate)
    up = np.asarray(up)
    I = gate.shape[0]
    if up.shape != gate.shape or I % INTERLEAVE:
        raise ValueError("gate and up must have the same shape with rows a multiple of 16")
    out = np.empty((2 * I,) + gate.shape[1:], dtype=gate.dtype)
    for r in range(2 * I):
        b, o = divmod(r, 2 * INTERLEAVE)
        src = gate if o < INTERLEAVE else up
        out[r] = src[INTERLEAVE * b + (o % INTERLEAVE)]
    return out


def deinterleave_rows(comb: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Inverse of :func:`interleave_rows`: ``[2I, ...] -> (gate [I, ...], up [I, ...])``."""
    comb = np.asarray(comb)
    I = comb.shape[0] // 2
    gate = np.empty((I,) + comb.shape[1:], dtype=comb.dtype)
    up = np.empty_like(gate)
    for i in range(I):
        b, o = divmod(i, INTERLEAVE)
        gate[i] = comb[2 * INTERLEAVE * b + o]
        up[i] = comb[2 * INTERLEAVE * b + INTERLEAVE + o]
    return gate, up


def quantize_expert(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, G: int) -> dict:
    """Quantize one expert into the stored layout.

    ``Wg``, ``Wu``: ``[I, H]``; ``Wd``: ``[H, I]`` (all fp32).  Returns a dict with
    ``w_gate_up`` (uint8 ``[2I, H//2]``), ``s_gate_up`` (fp16 ``[2I, H//G]``),
    ``w_down`` (uint8 ``[H, I//2]``) and ``s_down`` (fp16 ``[H, I//G]``).
    Quantization is row-wise, so interleaving before or after it is the same.
    """
    pg, sg = quantize_matrix(Wg, G)
    pu, su = quantize_matrix(Wu, G)
    pd, sd = quantize_matrix(Wd, G)
    return {
        "w_gate_up": interleave_rows(pg, pu),
        "s_gate_up": interleave_rows(sg, su),
        "w_down": pd,
        "s_down": sd,
    }


def dequantize_expert(ex: dict, H: int, I: int, G: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Stored expert -> exact fp64 ``(Wg_hat [I,H], Wu_hat [I,H], Wd_hat [H,I])``."""
    comb = dequantize_matrix(ex["w_gate_up"], ex["s_gate_up"], H, G)
    Wg, Wu = deinterleave_rows(comb)
    Wd = dequantize_matrix(ex["w_down"], ex["s_down"], I, G)
    return Wg, Wu, Wd
