"""Helpers for the GPU parity tests: build an engine from seeded weights,
drive prefill through the C ABI, read the paged pool back as contiguous KV,
and compare with the oracle at the stated tolerance."""
import numpy as np
import torch

import continuous_batching_decode_gb300 as cbd
from continuous_batching_decode_gb300 import synth
from oracle import model as om
from oracle import philox
from oracle import sampler as osamp

# Logit tolerance: max-abs <= 1e-2 * max|z| and mean-abs <= 2e-3.
TOL_MAX_REL = 1e-2
TOL_MEAN_ABS = 2e-3
NEAR_TIE = 1e-3


class Model:
    def __init__(self, name, max_rows=64, max_slots=8, mbps=8, seed=0, device_weights=True, kv_fp8=False,
                 layers=None, weights_int8=False):
        self.shape = dict(synth.MODEL_SHAPES[name])
        if layers:
            self.shape["n_layers"] = layers
        self.kv_fp8 = kv_fp8
        self.int8 = weights_int8
        self.w = synth.make_weights(self.shape, seed=seed, device="cuda" if device_weights else "cpu")
        self.cfg = cbd.make_config(self.shape, max_rows, max_slots, mbps, kv_fp8=kv_fp8, weights_int8=weights_int8)
        self.e = cbd.engine_create(self.cfg, self.w)
        self.mbps = mbps
        self._oracle = None

    def oracle(self, cache=True):
        if self._oracle is None:
            bits = {k: synth.bf16_bits(v) for k, v in self.w.items()}
            self._oracle = om.OracleModel(om.ModelConfig(**self.shape), bits, cache=cache,
                                          kv_format="e4m3" if self.kv_fp8 else "bf16",
                                          weight_format="int8" if self.int8 else "bf16")
        return self._oracle

    def close(self):
        cbd.engine_destroy(self.e)

    def pool(self, n_blocks):
        return Pool(self, n_blocks)


class Pool:
    def __init__(self, model, n_blocks):
        self.m = model
        self.p = cbd.kv_pool_create(model.e, n_blocks)
        base, nbytes, nb = cbd.kv_pool_data(self.p)
        s = model.shape
        hd = s["head_dim"]
        self.fp8 = model.kv_fp8
        r = np.arange(32)[:, None]
        d = np.arange(hd)[None, :]
        if self.fp8:
            # E4M3 bytes; K tile rows = positions (hd bytes), V tile rows =
            # dims (32 bytes); 16-byte chunks swizzled per row (include/cbd.h)
            self.view = cbd.device_view(base, (s["n_layers"], nb, s["n_kv_heads"], 2, 32 * hd), "u8")
            kswz = (r % 8) if hd == 128 else ((r // 2) % 4)
            k_idx = r * hd + (((d // 16) ^ kswz) * 16) + d % 16
            v_idx = d * 32 + (((r // 16) ^ ((d // 4) % 2)) * 16) + r % 16
            self.tile_index_kv = [torch.as_tensor(k_idx.reshape(-1), device="cuda"),
                                  torch.as_tensor(v_idx.reshape(-1), device="cuda")]
        else:
            # [L][n_blocks][H_kv][K|V][tile]; a tile stores (position, dim) at a
            # 128-byte-swizzled offset (see cbd_kv_pool_data in include/cbd.h)
            self.view = cbd.device_view(base, (s["n_layers"], nb, s["n_kv_heads"], 2, 32 * hd), "bf16")
            self.tile_index = torch.as_tensor(((d // 64) * 2048 + r * 64 + ((((d % 64) // 8) ^ (r % 8)) * 8) + d % 8)
                                              .reshape(-1), device="cuda")

    def close(self):
        cbd.kv_pool_destroy(self.p)

    def gather(self, tables, slot, n_pos):
        """Contiguous K, V of a slot: lists per layer of [n_pos, H_kv, hd] fp64."""
        nb = (n_pos + 31) // 32
        ids = torch.as_tensor(tables[slot][:nb].astype(np.int64), device="cuda")
        L, _, hkv, _, te = self.view.shape
        hd = te // 32
        if self.fp8:
            t = self.view[:, ids]
            k = t[:, :, :, 0][..., self.tile_index_kv[0]]
            v = t[:, :, :, 1][..., self.tile_index_kv[1]]
            kv = torch.stack([k, v], dim=3).contiguous().view(torch.float8_e4m3fn).float()
            kv = kv.reshape(L, nb, hkv, 2, 32, hd)
        else:
            kv = self.view[:, ids][..., self.tile_index].reshape(L, nb, hkv, 2, 32, hd)   # unswizzled
        kv = kv.permute(0, 3, 1, 4, 2, 5).reshape(L, 2, nb * 32, hkv, hd)
        kv = kv[:, :, :n_pos].float().cpu().numpy().astype(np.float64)
        return [kv[l, 0] for l in range(L)], [kv[l, 1] for l in range(L)]


def gpu_prefill(model, pool, slot, tokens, tables, nbps, start=0, chunk=512):
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c0 in range(0, len(tokens), chunk):
        part = tokens[c0:c0 + chunk]
        rows = [(slot, int(t), start + c0 + i, 1, 0) for i, t in enumerate(part)]
        cbd.step(model.e, pool.p, rows, tables, nbps, [], None, dummy)
        cbd.engine_check(model.e)       # a kernel-flagged error fails at the step that raised it


def run_step(model, pool, rows, tables, nbps, sampling, uniforms=None):
    m = sum(1 for r in rows if r[4])
    tok = torch.zeros(max(m, 1), dtype=torch.int32, device="cuda")
    lg = torch.zeros(max(m, 1), model.shape["vocab"], dtype=torch.float32, device="cuda")
    cbd.step(model.e, pool.p, rows, tables, nbps, sampling, uniforms, tok, lg)
    cbd.engine_check(model.e)
    return tok[:m].cpu().numpy(), lg[:m].cpu().numpy().astype(np.float64)


def oracle_kv_from_gpu(model, pool, tables, slot_ctx):
    """Oracle KV state for slots given the GPU pool contents."""
    cfg = model.oracle().cfg
    kv = {}
    for slot, n in slot_ctx.items():
        s = om.SequenceKV(cfg, n + 64)
        K, V = pool.gather(tables, slot, n)
        for l in range(cfg.n_layers):
            s.K[l][:n] = K[l]
            s.V[l][:n] = V[l]
        s.length = n
        kv[slot] = s
    return kv


def assert_logits_close(z_gpu, z_ref, what=""):
    err = np.abs(z_gpu - z_ref)
    mx = np.abs(z_ref).max()
    assert err.max() <= TOL_MAX_REL * mx, f"{what} max-abs {err.max():.4g} > {TOL_MAX_REL} * {mx:.4g}"
    assert err.mean() <= TOL_MEAN_ABS, f"{what} mean-abs {err.mean():.4g} > {TOL_MEAN_ABS}"
    return err.max(), err.mean()


def greedy_near_tie(z):
    t = np.sort(z)[-2:]
    return t[1] - t[0] < NEAR_TIE


def sampling_near_tie(logits_f32, counters, p: osamp.SamplingParams, u: float) -> bool:
    """Draws whose decision sits within the tolerance of a boundary."""
    l2 = osamp.penalize(logits_f32, counters, p.presence_penalty, p.frequency_penalty)
    if osamp.is_greedy(p):
        return greedy_near_tie(l2.astype(np.float64))
    ids, pk, (z, order, cum, n_keep) = osamp.kept_set(l2, p)
    if p.top_p < 1.0:
        if abs(cum[n_keep - 1] - p.top_p) < 1e-6 or (n_keep >= 2 and abs(cum[n_keep - 2] - p.top_p) < 1e-6):
            return True
        if n_keep < len(order) and z[order[n_keep - 1]] == z[order[n_keep]]:
            return True
    c = np.cumsum(pk)
    S = c[-1]
    return bool(np.any(np.abs(c - u * S) <= 1e-6 * S))


def sampling_params(d) -> osamp.SamplingParams:
    return osamp.SamplingParams(temperature=d.get("temperature", 0.0), top_p=d.get("top_p", 1.0),
                                top_k=d.get("top_k", 0), presence_penalty=d.get("presence_penalty", 0.0),
                                frequency_penalty=d.get("frequency_penalty", 0.0),
                                penalty_decay=d.get("penalty_decay", 1.0), seed=d.get("seed", 0),
                                request_id=d.get("request_id", 0), token_index=d.get("token_index", 0))


def uniform_of(d) -> float:
    return philox.sampler_uniform(d.get("seed", 0), d.get("request_id", 0), d.get("token_index", 0))


def counters_view(model):
    s = model.shape
    return cbd.device_view(cbd.engine_counters(model.e), (model.cfg.max_slots, s["vocab"]), "f32")
