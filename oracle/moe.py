"""Oracle: the routed MoE layer in plain fp64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What the pages fix, and what this module reads into them
    * 288 routed experts, top-8 per token per layer (GLM-5.3-Flash EXL3 3.05bpw on
      1x RTX 3090 recipe, ``summary``: each token takes 8 experts per layer); a shared
      expert that runs beside the routed ones (glm53-flash-offload README,
      "Decode kernels" bullet: the shared expert moved to a side stream).
    * Picks are deduplicated per layer into one expert union that all tokens of
      the batch share (README, "Elastic CLOCK expert cache" and "Batched decode").
    * Experts are addressed through per-expert pointer tables (RTX PRO 6000 recipe,
      ``config.expert_cache.mechanism``).
    * The routed partial results are summed in fp32 after the experts (README,
      "CPU tier" bullet: the fp32 partial is added back after its experts).
    The router function itself is not on the pages.  This library reads it as:
    sigmoid scores, an optional selection-only bias, top-k with ties to the lower
    expert id, and the selected (unbiased) scores renormalised to sum to 1.

Definitions (per token t; x_t is the exact bf16 value)
    l_e   = sum_h x_th * Wr[e, h]                      (fp64)
    s_e   = 1 / (1 + exp(-l_e))
    sel_e = s_e + b_e                                  (b = 0 when no bias)
    S_t   = the k experts of largest sel, ties to the lower id, listed ascending
    w_te  = s_e / sum_{e' in S_t} s_e'
    FFN_e(x) = Wd_e @ (silu(Wg_e @ x) * (Wu_e @ x)),  silu(z) = z / (1 + exp(-z))
    y_t   = sum_{e in S_t} w_te FFN_e(x_t) + FFN_shared(x_t)
Dispatch orders the T*k pick ids p = t*k + j stably by (expert, p); the routed
expert outputs are listed in that order, followed by the shared expert's output
for tokens 0..T-1.
"""

from __future__ import annotations

import numpy as np

from . import quant


def bf16_bits_to_f64(x_bits: np.ndarray) -> np.ndarray:
    """bf16 stored as uint16 bit patterns -> exact fp64 values."""
    b = np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(y: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 with round-to-nearest-even; returns uint16 bits.

    Written from the IEEE definition: keep the top 16 bits of the fp32 pattern and
    round on the 16 dropped bits, ties to the even kept pattern.  NaN stays NaN.
    """
    f = np.asarray(y, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep = u >> 16
    rest = u & 0xFFFF
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & 1) == 1))
    out = (keep + up.astype(np.uint64)) & 0xFFFF
    nan = np.isnan(f)
    out = np.where(nan, (keep | 0x40) & 0xFFFF, out)
    return out.astype(np.uint16)


def sigmoid(z: np.ndarray) -> np.ndarray:
    """Logistic function 1 / (1 + exp(-z)) in fp64."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU / swish: z * sigmoid(z) = z / (1 + exp(-z)), fp64."""
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """``l = x @ Wr^T`` in fp64; ``x`` [T,H] fp64, ``w_router`` [E,H] (fp32 values)."""
    return np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T


def route(x: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None, k: int) -> dict:
    """Sigmoid top-k routing with renormalised weights.

    Returns a dict:
      ``idx``   int32 [T,k]  selected experts, ascending id;
      ``w``     fp64  [T,k]  routing weights s_e / sum s over the selection;
      ``score`` fp64  [T,E]  sigmoid scores s;
      ``sel``   fp64  [T,E]  selection scores s + b;
      ``gap``   fp64  [T]    sel of the k-th pick minus sel of the (k+1)-th
                             (+inf when k == E): the margin that decides S_t.
    """
    logits = router_logits(x, w_router)
    s = sigmoid(logits)
    T, E = s.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    sel = s if bias is None else s + np.asarray(bias, np.float64)[None, :]
    # Descending by sel; a stable sort on -sel keeps equal values in ascending id.
    order = np.argsort(-sel, axis=1, kind="stable")
    top = np.sort(order[:, :k], axis=1)
    picked = np.take_along_axis(s, top, axis=1)
    w = picked / picked.sum(axis=1, keepdims=True)
    rows = np.arange(T)
    kth = sel[rows, order[:, k - 1]]
    gap = kth - sel[rows, order[:, k]] if k < E else np.full(T, np.inf)
    return {"idx": top.astype(np.int32), "w": w, "score": s, "sel": sel, "gap": gap}


def dispatch(idx: np.ndarray, n_experts: int) -> dict:
    """Histogram, exclusive offsets, stable permutation and active-expert list.

    ``perm[q]`` is the pick id ``p = t*k + j`` at sorted position ``q`` (sorted by
    expert, then by p); ``inv_perm[p]`` is its position.  ``active`` lists the
    experts with at least one pick, ascending.
    """
    idx = np.asarray(idx, dtype=np.int64)
    flat = idx.reshape(-1)
    P = flat.size
    counts = np.bincount(flat, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat * max(P, 1) + np.arange(P), kind="stable")
    inv = np.empty(P, dtype=np.int64)
    inv[perm] = np.arange(P)
    active = np.nonzero(counts)[0]
    return {
        "counts": counts.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "perm": perm.astype(np.int32),
        "inv_perm": inv.astype(np.int32),
        "active": active.astype(np.int32),
        "n_active": int(active.size),
    }


def expert_ffn(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """SwiGLU expert on rows of ``x`` [M,H]: ``(silu(x Wg^T) * (x Wu^T)) Wd^T`` in fp64."""
    x = np.asarray(x, np.float64)
    g = x @ np.asarray(Wg, np.float64).T
    u = x @ np.asarray(Wu, np.float64).T
    h = silu(g) * u
    return h @ np.asarray(Wd, np.float64).T


def expert_hidden(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray) -> np.ndarray:
    """The SwiGLU activation ``silu(x Wg^T) * (x Wu^T)`` alone, fp64 ``[M, I]``."""
    x = np.asarray(x, np.float64)
    return silu(x @ np.asarray(Wg, np.float64).T) * (x @ np.asarray(Wu, np.float64).T)


def combine(expert_out: np.ndarray, w: np.ndarray, inv_perm: np.ndarray, T: int, k: int) -> np.ndarray:
    """``y_t = sum_j w[t,j] * expert_out[inv_perm[t*k+j]] + expert_out[T*k + t]`` in fp64."""
    eo = np.asarray(expert_out, np.float64)
    w = np.asarray(w, np.float64)
    y = eo[T * k: T * k + T].copy()
    for t in range(T):
        for j in range(k):
            y[t] += w[t, j] * eo[inv_perm[t * k + j]]
    return y


class DequantCache:
    """Dequantizes stored experts on demand (fp64), keeping a few recent ones."""

    def __init__(self, experts, H: int, I: int, G: int, keep: int = 4):
        self.experts, self.H, self.I, self.G, self.keep = experts, H, I, G, keep
        self._cache: dict[int, tuple] = {}

    def __call__(self, e: int):
        if e not in self._cache:
            if len(self._cache) >= self.keep:
                self._cache.pop(next(iter(self._cache)))
            self._cache[e] = quant.dequantize_expert(self.experts[e], self.H, self.I, self.G)
        return self._cache[e]


def moe_layer(x_bits: np.ndarray, w_router: np.ndarray, bias, experts, shared: dict,
              H: int, I: int, E: int, k: int, G: int, tokens=None) -> dict:
    """The whole layer for bf16 input bits ``x_bits`` [T,H].

    ``experts``: sequence (or mapping) of E stored experts (see
    ``quant.quantize_expert``); ``shared``: the shared expert in the same layout.
    ``tokens``: optional subset of token indices whose outputs ``y`` are computed
    (routing and dispatch always cover all tokens); ``None`` means all.

    Returns routing, dispatch, ``expert_out`` (fp64, rows in dispatch order
    followed by the shared rows, only for the requested tokens; other rows NaN)
    and ``y`` (fp64 [T,H]; rows of tokens not requested are NaN).
    """
    x = bf16_bits_to_f64(x_bits)
    T = x.shape[0]
    r = route(x, w_router, bias, k)
    d = dispatch(r["idx"], E)
    want = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    wanted = np.zeros(T, dtype=bool)
    wanted[want] = True
    eo = np.full((T * k + T, H), np.nan)
    deq = DequantCache(experts, H, I, G)
    flat = r["idx"].reshape(-1)
    for e in d["active"]:
        lo, hi = d["offsets"][e], d["offsets"][e + 1]
        picks = d["perm"][lo:hi]
        toks = picks // k
        sel = wanted[toks]
        if not sel.any():
            continue
        assert np.all(flat[picks] == e)
        Wg, Wu, Wd = deq(int(e))
        eo[lo:hi][sel] = expert_ffn(x[toks[sel]], Wg, Wu, Wd)
    Sg, Su, Sd = quant.dequantize_expert(shared, H, I, G)
    eo[T * k + want] = expert_ffn(x[want], Sg, Su, Sd)
    y = np.full((T, H), np.nan)
    yw = combine(np.nan_to_num(eo, nan=0.0), r["w"], d["inv_perm"], T, k)
    y[want] = yw[want]
    return {**r, **d, "expert_out": eo, "y": y, "x": x}
