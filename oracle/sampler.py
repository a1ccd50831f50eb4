"""Per-row sampling with decayed occurrence penalties (oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may import it.

Parameters come from "RWKV Runner Albatross 后端",
section "适配器": temperature 1.0, top_p 0.3, top_k 0, frequency penalty 1,
penalty decay 0.996 are the defaults; section "Worker 主循环" applies
presence / frequency penalties and then samples every row of the batch.  The
pages fix the parameter set but not the order of operations, so this module
states one (each is a reading listed in the design notes):

1. Penalty, in fp32 with every operation rounded separately (no fused
   multiply-add):  l1 = l - (presence if cnt > 0 else 0);  l2 = l1 - freq*cnt.
2. Greedy when temperature == 0 or top_k == 1: the largest l2, ties to the
   lowest token id.
3. Otherwise z = l2 / T (fp32 division), then top-k (k > 0): keep the k
   largest by (z descending, id ascending).
4. Probabilities are the softmax of the kept z (fp64 here).  Top-p keeps the
   shortest prefix of the kept tokens ordered by (p descending, id ascending)
   whose cumulative probability reaches top_p; at least one token.
5. Draw: with u in [0, 1), walk the kept tokens in ascending id order and
   return the first whose cumulative probability exceeds u * (sum of kept).
6. Counters: every entry of the slot's row is multiplied by the decay
   (fp32), then the drawn token's entry gains 1.0 (fp32).

Greedy and sampled rows both update the counters.

Forbidden tokens (section "Worker 主循环" masks them before the penalties):
0. A forbidden id is removed from the candidates before step 1 -- its logit
   counts as -inf, so it is never the greedy choice, carries no probability
   and is never drawn; the remaining steps run over the other ids unchanged.
   The counters of forbidden ids still decay like every other entry.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class SamplingParams:
    temperature: float = 1.0
    top_p: float = 0.3
    top_k: int = 0
    presence_penalty: float = 0.0
    frequency_penalty: float = 1.0
    penalty_decay: float = 0.996
    seed: int = 0
    request_id: int = 0
    token_index: int = 0


def penalize(logits, counters, presence: float, frequency: float) -> np.ndarray:
    """Step 1: fp32, one rounding per operation."""
    l = np.asarray(logits, dtype=np.float32)
    c = np.asarray(counters, dtype=np.float32)
    pres = np.where(c > np.float32(0), np.float32(presence), np.float32(0))
    l1 = (l - pres).astype(np.float32)
    prod = (np.float32(frequency) * c).astype(np.float32)
    return (l1 - prod).astype(np.float32)


def is_greedy(p: SamplingParams) -> bool:
    return p.temperature == 0.0 or p.top_k == 1


def kept_set(l2, p: SamplingParams):
    """Steps 3-4: returns (kept ids ascending, their probabilities, details).

    details = (z (fp32), order of the top-k survivors, cumulative p in that
    order, nucleus length) for near-tie checks in tests.
    """
    z = (np.asarray(l2, dtype=np.float32) / np.float32(p.temperature)).astype(np.float32)
    V = z.shape[0]
    ids = np.arange(V)
    order = np.lexsort((ids, -z.astype(np.float64)))    # z desc, then id asc
    if 0 < p.top_k < V:
        order = order[: p.top_k]
    zk = z[order].astype(np.float64)
    e = np.exp(zk - zk.max())
    prob = e / e.sum()
    cum = np.cumsum(prob)
    hit = np.nonzero(cum >= p.top_p)[0]
    n_keep = int(hit[0]) + 1 if hit.size else len(order)
    n_keep = max(1, n_keep)
    keep = order[:n_keep]
    pk = prob[:n_keep]
    asc = np.argsort(keep, kind="stable")
    return keep[asc], pk[asc], (z, order, cum, n_keep)


def draw(kept_ids, kept_p, u: float) -> int:
    """Step 5: inverse CDF over the kept set in ascending id order."""
    cum = np.cumsum(kept_p)
    target = u * cum[-1]
    j = int(np.searchsorted(cum, target, side="right"))
    return int(kept_ids[min(j, len(kept_ids) - 1)])


def mask_forbidden(logits, forbidden) -> np.ndarray:
    """Step 0: forbidden ids get -inf (fp32)."""
    l = np.array(logits, dtype=np.float32)
    if forbidden is not None and len(forbidden):
        l[np.asarray(forbidden, dtype=np.int64)] = -np.inf
    return l


def sample_row(logits, counters, p: SamplingParams, u: float, forbidden=None) -> int:
    """Steps 0-5 for one row; returns the token id."""
    l2 = penalize(mask_forbidden(logits, forbidden), counters, p.presence_penalty, p.frequency_penalty)
    if is_greedy(p):
        return int(np.argmax(l2))            # argmax returns the first maximum
    ids, pk, _ = kept_set(l2, p)
    return draw(ids, pk, u)


def update_counters(counters, token: int, decay: float) -> np.ndarray:
    """Step 6: decay every entry (fp32), then add 1.0 to the drawn token."""
    c = (np.asarray(counters, dtype=np.float32) * np.float32(decay)).astype(np.float32)
    c[token] = np.float32(c[token] + np.float32(1.0))
    return c
