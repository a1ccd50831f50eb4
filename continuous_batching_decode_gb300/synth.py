"""Seeded synthetic inputs shared by the tests, the bench and the smoke run.

This module holds shapes, random draws and request traces only -- none of the
step's arithmetic.  Both the CUDA path and the CPU oracle are fed from here;
neither imports the other.

Model shapes (random-init, bf16 weights ~ N(0, 0.02), norm gains 1.0):
  tiny  2 layers, d 256, 4 q / 2 KV heads, head_dim 64, FFN 768, vocab 4096
  1b    16 layers, d 2048, 32 q / 8 KV heads, head_dim 64, FFN 8192, vocab 65536
  7b    32 layers, d 4096, 32 q / 8 KV heads, head_dim 128, FFN 14336, vocab 65536
"""
from __future__ import annotations

import numpy as np

MODEL_SHAPES = {
    "tiny": dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64,
                 ffn_dim=768, vocab=4096),
    # head_dim 128 and 4 query heads per KV head, as in the 7B shape, at toy size
    "hd128": dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128,
                  ffn_dim=1024, vocab=4096),
    "1b": dict(n_layers=16, d_model=2048, n_heads=32, n_kv_heads=8, head_dim=64,
               ffn_dim=8192, vocab=65536),
    "7b": dict(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128,
               ffn_dim=14336, vocab=65536),
}
ROPE_BASE = 10000.0
RMS_EPS = 1e-6
BLOCK = 32

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def weight_shapes(s: dict) -> dict:
    """name -> shape; per-layer names are "<layer>.<key>"."""
    d, hq, hkv, hd, F, V = (s["d_model"], s["n_heads"], s["n_kv_heads"], s["head_dim"],
                            s["ffn_dim"], s["vocab"])
    out = {"embed": (V, d)}
    for l in range(s["n_layers"]):
        out.update({
            f"{l}.attn_norm": (d,), f"{l}.wq": (hq * hd, d), f"{l}.wk": (hkv * hd, d),
            f"{l}.wv": (hkv * hd, d), f"{l}.wo": (d, hq * hd), f"{l}.ffn_norm": (d,),
            f"{l}.w_gate": (F, d), f"{l}.w_up": (F, d), f"{l}.w_down": (d, F),
        })
    out["final_norm"] = (d,)
    out["lm_head"] = (V, d)
    return out


def make_weights(s: dict, seed: int = 0, device: str = "cpu", std: float = 0.02) -> dict:
    """Random-init bf16 weights as torch tensors (norm gains exactly 1.0)."""
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    out = {}
    for name, shape in weight_shapes(s).items():
        if name.endswith("norm"):
            out[name] = torch.ones(shape, dtype=torch.bfloat16, device=device)
        else:
            t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            out[name] = (t * std).to(torch.bfloat16)
    return out


def bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (host copy)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def random_tokens(rng: np.random.Generator, n: int, vocab: int) -> list:
    return [int(v) for v in rng.integers(0, vocab, size=n)]


def permuted_tables(n_blocks_needed: dict, n_pool_blocks: int, max_blocks_per_seq: int,
                    rng: np.random.Generator):
    """Place every slot's logical blocks on distinct, randomly chosen physical
    blocks.  Returns (tables [max_slot+1][max_blocks_per_seq] int32 with -1
    padding, n_blocks_per_slot)."""
    total = sum(n_blocks_needed.values())
    if total > n_pool_blocks:
        raise ValueError("pool too small for the requested contexts")
    phys = rng.permutation(n_pool_blocks)[:total]
    n_slots = max(n_blocks_needed) + 1 if n_blocks_needed else 0
    tables = np.full((n_slots, max_blocks_per_seq), -1, dtype=np.int32)
    nbs = np.zeros(n_slots, dtype=np.int32)
    k = 0
    for slot in sorted(n_blocks_needed):
        nb = n_blocks_needed[slot]
        tables[slot, :nb] = phys[k:k + nb]
        nbs[slot] = nb
        k += nb
    return tables, nbs


def tiny_step(seed: int = 0) -> dict:
    """The tiny workload: 4 decode slots at contexts 5/17/33/64 (random prior
    tokens, to be prefilled) plus one 40-token prefill chunk in slot 4.  Slots
    0-3 decode greedily; slot 4's last prompt row is sampled with
    temperature 1.0, top_p 0.3, frequency penalty 1, decay 0.996, and its
    counters are pre-loaded by replaying 16 prior tokens."""
    rng = np.random.default_rng(seed)
    V = MODEL_SHAPES["tiny"]["vocab"]
    contexts = [5, 17, 33, 64]
    prior = [random_tokens(rng, c, V) for c in contexts]
    next_tok = random_tokens(rng, 4, V)
    prompt = random_tokens(rng, 40, V)
    replay = random_tokens(rng, 16, V)
    return dict(contexts=contexts, prior=prior, next_tokens=next_tok, prompt=prompt,
                replay=replay, pool_blocks=32, seed=seed)


def decode_batch(B: int, ctx_lo: int, ctx_hi: int, vocab: int, seed: int) -> dict:
    """B decode rows with cached contexts ~ U[ctx_lo, ctx_hi] and random
    current tokens."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=B)
    return dict(contexts=[int(c) for c in ctx], tokens=random_tokens(rng, B, vocab))


def request_trace(n: int, vocab: int, seed: int, prompt_choices=(20, 50, 200, 1000),
                  mean_out: float = 128.0, cap: int = 512, rate: float | None = None) -> list:
    """Requests with prompt lengths drawn uniformly from ``prompt_choices``,
    output lengths min(Geometric(1/mean_out), cap) and Poisson arrivals at
    ``rate`` per second (all at t=0 when rate is None).  Returns dicts with
    id, arrival, prompt, max_tokens."""
    rng = np.random.default_rng(seed)
    t = 0.0
    out = []
    for i in range(n):
        if rate:
            t += float(rng.exponential(1.0 / rate))
        P = int(rng.choice(prompt_choices))
        m = int(min(rng.geometric(1.0 / mean_out), cap))
        out.append(dict(id=i, arrival=t, prompt=random_tokens(rng, P, vocab), max_tokens=m))
    return out
