"""fp64 forward pass of the decoder for one batched step (oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may import it.

What it computes, per row r = (slot s, token t, position p):

    x = E[t]
    per layer:
        h = x / sqrt(mean(x^2) + eps) * g_attn
        q, k, v = h Wq^T, h Wk^T, h Wv^T           (no biases)
        q, k = RoPE(q, p), RoPE(k, p)               (rotate-half, base^(-2i/hd))
        K_s[p], V_s[p] = bf16(k), bf16(v)           (KV is persistent bf16 state)
        o_i = sum_{j<=p} softmax_j(q_i . K_s[j]_g / sqrt(hd)) V_s[j]_g,
              g = i // (H_q / H_kv)                 (grouped-query attention)
        x = x + o Wo^T
        h = x / sqrt(mean(x^2) + eps) * g_ffn
        x = x + (silu(h Wg^T) * (h Wu^T)) Wd^T
    z = (x / sqrt(mean(x^2) + eps) * g_final) Wlm^T     (sampled rows only)

Batching (page "0.8MB 跑通 Qwen 第 14-1 篇", section 1 and section 3): one step
serves a dynamic set of rows, each with its own KV; the result must equal
running every row on its own.  Paging ("20.3 服务、批处理与流式", section
20.3.2) is a storage detail, so this oracle keeps each sequence's KV
contiguous.  All arithmetic is fp64 over the bf16 weights; the only rounding
is KV storage to bf16, which mirrors the persistent bf16 KV state.

Rows of one step are processed layer by layer: every row's k, v for a layer
is stored before any row of that layer attends, so a prefill row at position
p sees the earlier rows of its own chunk (causal chunked prefill).

Int8 weights ("RWKV Runner Albatross 后端", 边界与后续路线: int8-quantised
weights are listed among the backend's next steps; "大模型推理为什么需要
Continuous Batching", section 6: quantisation shrinks the bytes a step moves).
The pages name int8 and no scheme, so this oracle takes the plainest one:
weight-only, symmetric, one scale per output channel (row) of every matrix the
step streams (wq, wk, wv, wo, w_gate, w_up, w_down, lm_head; the embedding
table and the norm gains are unchanged).  With ``weight_format="int8"`` each
such matrix is replaced by q * s, computed by ``quantize_int8_rows``.

FP8 KV ("大模型推理为什么需要 Continuous Batching", section 6: quantising the
KV cache, e.g. to FP8, fits more sequences at a small precision cost): with
``kv_format="e4m3"`` K and V are stored as FP8 E4M3 values instead of bf16
(round to nearest even, finite values beyond the largest magnitude 448
saturate; no scale factor -- the page names none, and this model's K and V
are O(1)).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_base: float = 10000.0
    rms_eps: float = 1e-6


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as fp64."""
    b = np.ascontiguousarray(bits).view(np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    bf16 keeps 8 significant bits and fp32's exponent range, so a value
    m * 2^e with m in [0.5, 1) rounds to rint(m * 2^8) * 2^(e-8).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_to_e4m3(x) -> np.ndarray:
    """Round fp64 values to the nearest FP8 E4M3 value (ties to even), as fp64.

    E4M3 (the OCP 8-bit format without infinities): sign, 4 exponent bits
    with bias 7, 3 fraction bits.  A normal value 1.f * 2^E (E >= -6) has 4
    significant bits, so its spacing is 2^(E-3); below 2^-6 the subnormals
    are multiples of 2^-9.  The largest finite magnitude is 448 (exponent
    field 15 with fraction 110; 111 there is NaN); larger finite inputs
    saturate to +-448.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                     # a = m * 2^e, m in [0.5, 1): E = e - 1
    quantum = np.maximum(e - 4, -9)        # log2 of the spacing at a
    r = np.ldexp(np.rint(np.ldexp(a, -quantum)), quantum)
    r = np.minimum(r, 448.0)
    return np.where(np.isnan(x), x, np.copysign(r, x))


INT8_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "lm_head")


def quantize_int8_rows(w) -> tuple:
    """Symmetric per-row int8 quantisation of a matrix of bf16 values.

    For each row r:  a = max_k |w[r, k]| (exact);  s = a / 127 rounded to
    fp32 (one IEEE single-precision division, nearest even);
    q[r, k] = w[r, k] / s rounded to the nearest integer, ties to even (the
    quotient evaluated in fp64), clamped to [-127, 127].  A row of zeros gets
    s = 0 and q = 0.  Returns (q as int8, s as float32); the dequantised
    matrix is q * s, exact in fp64.
    """
    w = np.asarray(w, dtype=np.float64)
    a = np.max(np.abs(w), axis=1)
    s = (a.astype(np.float32) / np.float32(127.0)).astype(np.float32)
    s64 = s.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(w / s64[:, None])
    q = np.where(s64[:, None] > 0, q, 0.0)
    q = np.clip(q, -127, 127).astype(np.int8)
    return q, s


def dequantize_int8_rows(q, s) -> np.ndarray:
    """q * s per row, in fp64 (exact: 8-bit by 24-bit products)."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float32).astype(np.float64)[:, None]


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half rotary embedding.

    x: [n, heads, hd]; pos: [n].  Dimension i < hd/2 is paired with
    i + hd/2 and the pair is turned by the angle pos * base^(-2i/hd):
        (a, b) -> (a cos - b sin, b cos + a sin).
    """
    hd = x.shape[-1]
    half = hd // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Grouped-query attention of one row.

    q: [H_q, hd]; K, V: [n_pos, H_kv, hd] holding positions 0..n_pos-1.
    Query head i reads KV head i // (H_q / H_kv).  Returns [H_q, hd].
    """
    hq, hd = q.shape
    group = hq // K.shape[1]
    Kg = np.repeat(K, group, axis=1)          # [n_pos, H_q, hd]
    Vg = np.repeat(V, group, axis=1)
    s = np.einsum("hd,jhd->hj", q, Kg) / math.sqrt(hd)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return np.einsum("hj,jhd->hd", p, Vg)


class SequenceKV:
    """Contiguous KV of one sequence: per layer K, V of shape [cap, H_kv, hd]."""

    def __init__(self, cfg: ModelConfig, capacity: int):
        shape = (capacity, cfg.n_kv_heads, cfg.head_dim)
        self.K = [np.zeros(shape) for _ in range(cfg.n_layers)]
        self.V = [np.zeros(shape) for _ in range(cfg.n_layers)]
        self.length = 0          # positions 0..length-1 hold valid KV

    def ensure(self, n: int) -> None:
        cap = self.K[0].shape[0]
        if n <= cap:
            return
        new = max(n, 2 * cap)
        for arrs in (self.K, self.V):
            for i, a in enumerate(arrs):
                b = np.zeros((new,) + a.shape[1:])
                b[:cap] = a
                arrs[i] = b


class OracleModel:
    """The decoder's weights as exact fp64 values of bf16 parameters.

    ``weights`` maps names to bf16 bit arrays (uint16) or arrays whose
    values are exactly representable in bf16:
      embed [V, d], lm_head [V, d], final_norm [d], and per layer l
      "l.attn_norm" [d], "l.wq" [H_q*hd, d], "l.wk" [H_kv*hd, d],
      "l.wv" [H_kv*hd, d], "l.wo" [d, H_q*hd], "l.ffn_norm" [d],
      "l.w_gate" [F, d], "l.w_up" [F, d], "l.w_down" [d, F].
    With ``cache=False`` each layer is upcast on use and dropped (bounds RAM
    for the 7B shape); ``weights`` may then also be a callable name -> array.
    ``weight_format="int8"`` replaces every streamed matrix by its per-row
    int8 quantisation q * s (``quantize_int8_rows``).
    """

    LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm",
                  "w_gate", "w_up", "w_down")

    def __init__(self, cfg: ModelConfig, weights, cache: bool = True, kv_format: str = "bf16",
                 weight_format: str = "bf16"):
        if kv_format not in ("bf16", "e4m3"):
            raise ValueError(kv_format)
        if weight_format not in ("bf16", "int8"):
            raise ValueError(weight_format)
        self.cfg = cfg
        self.int8 = weight_format == "int8"
        self.kv_round = round_to_bf16 if kv_format == "bf16" else round_to_e4m3
        self._src = weights
        self._cache = {} if cache else None

    def _get(self, name: str) -> np.ndarray:
        if self._cache is not None and name in self._cache:
            return self._cache[name]
        src = self._src(name) if callable(self._src) else self._src[name]
        a = np.asarray(src)
        arr = bf16_bits_to_f64(a) if a.dtype in (np.uint16, np.int16) else a.astype(np.float64)
        if self.int8 and name.split(".")[-1] in INT8_MATRICES:
            arr = dequantize_int8_rows(*quantize_int8_rows(arr))
        if self._cache is not None:
            self._cache[name] = arr
        return arr

    def layer(self, l: int) -> dict:
        return {k: self._get(f"{l}.{k}") for k in self.LAYER_KEYS}

    def embed_rows(self, tokens) -> np.ndarray:
        src = self._src("embed_rows", tokens) if callable(self._src) else None
        if src is not None:
            return bf16_bits_to_f64(src)
        return self._get("embed")[np.asarray(tokens)]


def step(model: OracleModel, kv: dict, rows) -> np.ndarray:
    """One batched step.

    rows: sequence of (slot, token, pos, sample) -- the step's row set, in any
    order; positions of one slot must be distinct.  kv: slot -> SequenceKV,
    extended in place (positions written by this step become valid).
    Returns the fp64 logits of the rows with sample != 0, in row order,
    shape [m, V].
    """
    cfg = model.cfg
    rows = [tuple(int(v) for v in r) for r in rows]
    n = len(rows)
    slots = [r[0] for r in rows]
    toks = [r[1] for r in rows]
    pos = np.array([r[2] for r in rows], dtype=np.int64)
    hq, hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    for s, p in zip(slots, pos):
        kv[s].ensure(int(p) + 1)

    x = model.embed_rows(toks).reshape(n, cfg.d_model).astype(np.float64)
    for l in range(cfg.n_layers):
        w = model.layer(l)
        h = rmsnorm(x, w["attn_norm"], cfg.rms_eps)
        q = rope((h @ w["wq"].T).reshape(n, hq, hd), pos, cfg.rope_base)
        k = rope((h @ w["wk"].T).reshape(n, hkv, hd), pos, cfg.rope_base)
        v = (h @ w["wv"].T).reshape(n, hkv, hd)
        for r in range(n):                          # store all KV first
            kv[slots[r]].K[l][pos[r]] = model.kv_round(k[r])
            kv[slots[r]].V[l][pos[r]] = model.kv_round(v[r])
        o = np.empty((n, hq * hd))
        for r in range(n):                          # then attend causally
            S = kv[slots[r]]
            o[r] = attend(q[r], S.K[l][: pos[r] + 1], S.V[l][: pos[r] + 1]).reshape(-1)
        x = x + o @ w["wo"].T
        h = rmsnorm(x, w["ffn_norm"], cfg.rms_eps)
        x = x + (silu(h @ w["w_gate"].T) * (h @ w["w_up"].T)) @ w["w_down"].T
    for s, p in zip(slots, pos):
        kv[s].length = max(kv[s].length, int(p) + 1)
    sel = [r for r in range(n) if rows[r][3]]
    if not sel:
        return np.zeros((0, cfg.vocab))
    hf = rmsnorm(x[sel], model._get("final_norm"), cfg.rms_eps)
    return hf @ model._get("lm_head").T


def prefill(model: OracleModel, kv: dict, slot: int, tokens, start: int = 0,
            chunk: int | None = None) -> np.ndarray:
    """Run ``tokens`` at positions start.. through ``step`` in chunks.

    Returns the logits of the last token.  ``chunk=None`` is one chunk.
    """
    tokens = list(tokens)
    chunk = chunk or len(tokens)
    z = None
    for c0 in range(0, len(tokens), chunk):
        part = tokens[c0:c0 + chunk]
        last = c0 + len(part) == len(tokens)
        rows = [(slot, t, start + c0 + i, 1 if (last and i == len(part) - 1) else 0)
                for i, t in enumerate(part)]
        out = step(model, kv, rows)
        if last:
            z = out[0]
    return z
