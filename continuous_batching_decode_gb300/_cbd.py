"""ctypes binding of libcbd (argument marshalling only).

Every function here forwards to the C entry point of the same name in
``include/cbd.h`` (without the ``cbd_`` prefix) and raises ``CbdError`` on a
negative status.  The step itself runs entirely in libcbd's kernels; torch
is used only to hold device buffers and to name the current CUDA stream.
There is no fallback: if libcbd.so is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcbd.so")

OK, EINVAL, ENOMEM, ECUDA, EPOOL, EUNSUPPORTED, EDEVICE, EDEADLOCK, ESTATE, EBUSY = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9
FINISH_LENGTH, FINISH_FALLBACK, FINISH_ABORTED, FINISH_TIMEOUT, FINISH_LAGGING = 1, 2, 3, 4, 5
POLICY_FORMA, POLICY_ALBATROSS = 0, 1


class CbdError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libcbd status {status}: {msg}")
        self.status = status


c_i32, c_u32, c_u64, c_f32, c_vp = ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p


class Config(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("d_model", c_i32), ("n_heads", c_i32), ("n_kv_heads", c_i32),
                ("head_dim", c_i32), ("ffn_dim", c_i32), ("vocab", c_i32), ("rope_base", c_f32),
                ("rms_eps", c_f32), ("block_size", c_i32), ("max_rows", c_i32), ("max_slots", c_i32),
                ("max_blocks_per_seq", c_i32), ("kv_fp8", c_i32), ("weights_int8", c_i32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")]


class Weights(ctypes.Structure):
    _fields_ = [("on_device", c_i32), ("embed", c_vp), ("final_norm", c_vp), ("lm_head", c_vp),
                ("layers", ctypes.POINTER(LayerWeights))]


TOKEN_LAST = -1       # cbd_row.token: the token the engine last sampled for the row's slot


class Row(ctypes.Structure):
    _fields_ = [("slot", c_i32), ("token", c_i32), ("pos", c_i32), ("is_prefill", c_i32), ("sample", c_i32)]


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", c_f32), ("top_p", c_f32), ("top_k", c_i32), ("presence_penalty", c_f32),
                ("frequency_penalty", c_f32), ("penalty_decay", c_f32), ("seed", c_u64), ("request_id", c_u64),
                ("token_index", c_u32), ("reserved", c_u32)]


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class SchedConfig(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("n_blocks", "block_size", "max_slots", "max_rows", "chunk", "answer_budget",
                                     "max_blocks_per_seq", "reserve_answer", "stall_fallback",
                                     "queue_per_slot", "queue_timeout_ms", "out_buffer",
                                     "policy", "max_prefill", "prefill_every", "short_prompt")]


class Request(ctypes.Structure):
    _fields_ = [("id", c_u64), ("prompt", ctypes.POINTER(c_i32)), ("prompt_len", c_i32), ("max_tokens", c_i32),
                ("sampling", Sampling)]


class Plan(ctypes.Structure):
    _fields_ = [("n_rows", c_i32), ("rows", ctypes.POINTER(Row)), ("n_sampled", c_i32),
                ("sampling", ctypes.POINTER(Sampling)), ("sampled_ids", ctypes.POINTER(c_u64)),
                ("table_slots", c_i32), ("block_tables", ctypes.POINTER(c_i32)),
                ("n_blocks_per_slot", ctypes.POINTER(c_i32)), ("n_resets", c_i32),
                ("reset_slots", ctypes.POINTER(c_i32)), ("n_stopped", c_i32), ("stopped_ids", ctypes.POINTER(c_u64))]


class Finished(ctypes.Structure):
    _fields_ = [("id", c_u64), ("reason", c_i32), ("n_tokens", c_i32)]


class SchedStats(ctypes.Structure):
    _fields_ = [("running", c_i32), ("waiting", c_i32), ("free_blocks", c_i32), ("allocated", c_i32),
                ("reserved", c_i32), ("outstanding", c_i32), ("steps", ctypes.c_int64),
                ("rows_prefill", ctypes.c_int64), ("rows_decode", ctypes.c_int64),
                ("fallback_stops", ctypes.c_int64), ("stalled_rows", ctypes.c_int64),
                ("rejected_busy", ctypes.c_int64), ("timed_out", ctypes.c_int64), ("aborted", ctypes.c_int64),
                ("lagging", ctypes.c_int64)]


_P = ctypes.POINTER
PROTOS = {
    "cbd_last_error": (ctypes.c_char_p, []),
    "cbd_version": (ctypes.c_char_p, []),
    "cbd_engine_create": (c_i32, [_P(Config), _P(Weights), _P(c_vp)]),
    "cbd_engine_destroy": (c_i32, [c_vp]),
    "cbd_engine_check": (c_i32, [c_vp]),
    "cbd_engine_counters": (c_i32, [c_vp, _P(c_vp)]),
    "cbd_slot_reset": (c_i32, [c_vp, c_i32, c_vp]),
    "cbd_engine_profile": (c_i32, [c_vp, c_i32]),
    "cbd_engine_set_gemm_path": (c_i32, [c_vp, c_i32, c_i32]),
    "cbd_engine_set_rows_gemm": (c_i32, [c_vp, c_i32, c_i32]),
    "cbd_engine_set_prefill_attention": (c_i32, [c_vp, c_i32]),
    "cbd_engine_set_attention_path": (c_i32, [c_vp, c_i32]),
    "cbd_engine_set_l2_prefetch": (c_i32, [c_vp, c_u64]),
    "cbd_engine_set_fused_norm": (c_i32, [c_vp, c_i32]),
    "cbd_engine_set_gemm_chain": (c_i32, [c_vp, c_i32]),
    "cbd_engine_set_forbidden": (c_i32, [c_vp, _P(c_i32), c_i32]),
    "cbd_engine_profile_read": (c_i32, [c_vp, _P(KernelStat), c_i32, _P(c_i32)]),
    "cbd_kv_pool_create": (c_i32, [c_vp, c_i32, _P(c_vp)]),
    "cbd_kv_pool_destroy": (c_i32, [c_vp]),
    "cbd_kv_pool_data": (c_i32, [c_vp, _P(c_vp), _P(c_u64), _P(c_i32)]),
    "cbd_step": (c_i32, [c_vp, c_vp, _P(Row), c_i32, _P(c_i32), c_i32, _P(c_i32), _P(Sampling), _P(c_f32),
                         c_vp, c_vp, c_vp]),
    "cbd_batch_create": (c_i32, [c_vp, c_vp, _P(Row), c_i32, _P(c_i32), c_i32, _P(c_i32), _P(Sampling),
                                 _P(c_f32), _P(c_vp), c_vp]),
    "cbd_batch_run": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "cbd_batch_destroy": (c_i32, [c_vp]),
    "cbd_batch_launches": (c_i32, [c_vp, _P(c_i32)]),
    "cbd_batch_set_graph": (c_i32, [c_vp, c_i32]),
    "cbd_engine_set_step_graph": (c_i32, [c_vp, c_i32]),
    "cbd_engine_step_graph_captures": (c_i32, [c_vp, _P(c_i32)]),
    "cbd_batch_captures": (c_i32, [c_vp, _P(c_i32)]),
    "cbd_sample": (c_i32, [c_vp, c_vp, c_i32, _P(c_i32), _P(Sampling), _P(c_f32), c_vp, c_vp]),
    "cbd_sample_static": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_i32, _P(c_i32), _P(Sampling), _P(c_f32), c_vp, c_vp]),
    "cbd_sample_static_check": (c_i32, [c_vp]),
    "cbd_engine_test_wait_timeout": (c_i32, [c_vp, ctypes.c_int64, c_vp]),
    "cbd_engine_read_weight": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_vp]),
    "cbd_sched_create": (c_i32, [_P(SchedConfig), _P(c_vp)]),
    "cbd_sched_destroy": (c_i32, [c_vp]),
    "cbd_sched_submit": (c_i32, [c_vp, _P(Request)]),
    "cbd_sched_plan": (c_i32, [c_vp, _P(Plan)]),
    "cbd_sched_commit": (c_i32, [c_vp, _P(c_i32), c_i32, _P(Finished), c_i32, _P(c_i32)]),
    "cbd_sched_output": (c_i32, [c_vp, c_u64, _P(c_i32), c_i32, _P(c_i32)]),
    "cbd_sched_stats_get": (c_i32, [c_vp, _P(SchedStats)]),
    "cbd_sched_abort": (c_i32, [c_vp, c_u64]),
    "cbd_sched_set_time": (c_i32, [c_vp, ctypes.c_int64]),
    "cbd_sched_read": (c_i32, [c_vp, c_u64, _P(c_i32), c_i32, _P(c_i32)]),
    "cbd_sched_finished": (c_i32, [c_vp, _P(Finished), c_i32, _P(c_i32)]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libcbd.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise CbdError(ECUDA, f"{LIB_PATH} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != OK:
        raise CbdError(status, lib().cbd_last_error().decode(errors="replace"))


def _ptr(t) -> int:
    """Raw device/host address of a torch tensor (None -> NULL)."""
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def last_error() -> str:
    return lib().cbd_last_error().decode(errors="replace")


def version() -> str:
    return lib().cbd_version().decode()


# ------------------------------------------------------------------ engine
def make_config(shape: dict, max_rows: int, max_slots: int, max_blocks_per_seq: int,
                rope_base: float = 10000.0, rms_eps: float = 1e-6, kv_fp8: bool = False,
                weights_int8: bool = False) -> Config:
    return Config(shape["n_layers"], shape["d_model"], shape["n_heads"], shape["n_kv_heads"], shape["head_dim"],
                  shape["ffn_dim"], shape["vocab"], rope_base, rms_eps, 32, max_rows, max_slots, max_blocks_per_seq,
                  1 if kv_fp8 else 0, 1 if weights_int8 else 0)


def engine_create(cfg: Config, weights: dict):
    """weights: name -> bf16 torch tensor, all on the current CUDA device or
    all on the host (names as in the synthetic generator: embed, lm_head,
    final_norm, "<l>.wq", ...)."""
    L = cfg.n_layers
    on_dev = bool(weights["embed"].is_cuda)
    keep = [w.contiguous() for w in weights.values()]     # keep-alive
    byname = dict(zip(weights.keys(), keep))
    layers = (LayerWeights * L)()
    for l in range(L):
        for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
            setattr(layers[l], k, _ptr(byname[f"{l}.{k}"]))
    w = Weights(1 if on_dev else 0, _ptr(byname["embed"]), _ptr(byname["final_norm"]), _ptr(byname["lm_head"]),
                layers)
    out = c_vp()
    _check(lib().cbd_engine_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(out)))
    return out.value


def engine_destroy(e) -> None:
    _check(lib().cbd_engine_destroy(e))


def engine_set_forbidden(e, ids) -> None:
    """Token ids the sampler never draws (empty: none); see include/cbd.h."""
    ia, ip = _i32(list(ids) or [0])
    _check(lib().cbd_engine_set_forbidden(e, ip, len(list(ids))))


def engine_check(e) -> None:
    _check(lib().cbd_engine_check(e))


def engine_test_wait_timeout(e, limit_cycles: int, stream=None) -> None:
    _check(lib().cbd_engine_test_wait_timeout(e, int(limit_cycles), _stream(stream)))


WEIGHT_QKV, WEIGHT_O, WEIGHT_GATE_UP, WEIGHT_DOWN, WEIGHT_LM_HEAD = 0, 1, 2, 3, 4


def engine_read_weight(e, which: int, layer: int, rows: int, cols: int, int8: bool):
    """The engine's copy of a streamed matrix in its row order (see
    cbd_engine_read_weight): (uint16 bf16 bits or int8 array [rows][cols],
    fp32 scales [rows] or None)."""
    m = np.zeros((rows, cols), dtype=np.int8 if int8 else np.uint16)
    sc = np.zeros(rows, dtype=np.float32) if int8 else None
    _check(lib().cbd_engine_read_weight(e, which, layer, m.ctypes.data,
                                        sc.ctypes.data if sc is not None else None))
    return m, sc


def engine_counters(e) -> int:
    p = c_vp()
    _check(lib().cbd_engine_counters(e, ctypes.byref(p)))
    return p.value


def engine_set_gemm_path(e, path: int, gemv_max_rows: int = 0) -> None:
    """0 automatic, 1 CUDA-core GEMV only, 2 tcgen05 only."""
    _check(lib().cbd_engine_set_gemm_path(e, path, gemv_max_rows))


def engine_set_prefill_attention(e, enable: bool) -> None:
    """Prefill runs on the prefill attention kernel (attention path 0, bf16 K/V)."""
    _check(lib().cbd_engine_set_prefill_attention(e, 1 if enable else 0))


def engine_set_rows_gemm(e, min_rows: int, force: bool = False) -> None:
    """tcgen05 path: the 128-row-tile kernel from min_rows rows (0 = never),
    for the GEMMs it fills the GPU well for (every GEMM with force)."""
    _check(lib().cbd_engine_set_rows_gemm(e, min_rows, 1 if force else 0))


def engine_set_attention_path(e, path: int) -> None:
    """0 streaming tensor-core kernel (default), 1 CUDA cores, 2 one CTA per chunk."""
    _check(lib().cbd_engine_set_attention_path(e, path))


def engine_set_fused_norm(e, enable: bool) -> None:
    """RMSNorm folded into the tensor-core GEMM epilogues (default on)."""
    _check(lib().cbd_engine_set_fused_norm(e, 1 if enable else 0))


def engine_set_gemm_chain(e, enable: bool) -> None:
    """Decode layers' O, gate/up, down and next-QKV contractions as one persistent launch (default off)."""
    _check(lib().cbd_engine_set_gemm_chain(e, 1 if enable else 0))


def engine_set_l2_prefetch(e, nbytes: int) -> None:
    """Bytes of the next weight contraction each kernel prefetches into L2 (0: off)."""
    _check(lib().cbd_engine_set_l2_prefetch(e, nbytes))


def engine_profile(e, enable: bool) -> None:
    _check(lib().cbd_engine_profile(e, 1 if enable else 0))


def engine_profile_read(e) -> dict:
    """kernel class -> (launches, total ms)."""
    buf = (KernelStat * 32)()
    n = c_i32()
    _check(lib().cbd_engine_profile_read(e, buf, 32, ctypes.byref(n)))
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n.value)}


def slot_reset(e, slot: int, stream=None) -> None:
    _check(lib().cbd_slot_reset(e, slot, _stream(stream)))


def kv_pool_create(e, n_blocks: int):
    out = c_vp()
    _check(lib().cbd_kv_pool_create(e, n_blocks, ctypes.byref(out)))
    return out.value


def kv_pool_destroy(p) -> None:
    _check(lib().cbd_kv_pool_destroy(p))


def kv_pool_data(p):
    base, nbytes, nb = c_vp(), c_u64(), c_i32()
    _check(lib().cbd_kv_pool_data(p, ctypes.byref(base), ctypes.byref(nbytes), ctypes.byref(nb)))
    return base.value, nbytes.value, nb.value


# ------------------------------------------------------------------ step
# NumPy views of cbd_row and cbd_sampling with the C layout: a caller may
# build its step inputs once as such arrays and update fields in place
# (tokens, positions, token_index) instead of passing Python tuples and
# dicts that are converted on every call.
ROW_DTYPE = np.dtype({"names": [n for n, _ in Row._fields_],
                      "formats": ["<i4"] * 5,
                      "offsets": [getattr(Row, n).offset for n, _ in Row._fields_],
                      "itemsize": ctypes.sizeof(Row)})
SAMPLING_DTYPE = np.dtype({"names": [n for n, _ in Sampling._fields_],
                           "formats": ["<f4", "<f4", "<i4", "<f4", "<f4", "<f4", "<u8", "<u8", "<u4", "<u4"],
                           "offsets": [getattr(Sampling, n).offset for n, _ in Sampling._fields_],
                           "itemsize": ctypes.sizeof(Sampling)})


def rows_table(rows) -> np.ndarray:
    """rows as a ROW_DTYPE array (a copy; fields may then be updated in place)."""
    a = np.zeros(len(rows), ROW_DTYPE)
    for i, r in enumerate(rows):
        a[i] = tuple(int(v) for v in r)
    return a


def sampling_table(params) -> np.ndarray:
    """Sampling dicts as a SAMPLING_DTYPE array (missing fields -> defaults)."""
    params = list(params)
    a = np.zeros(max(1, len(params)), SAMPLING_DTYPE)
    for i, p in enumerate(params):
        a[i] = (float(p.get("temperature", 0.0)), float(p.get("top_p", 1.0)), int(p.get("top_k", 0)),
                float(p.get("presence_penalty", 0.0)), float(p.get("frequency_penalty", 0.0)),
                float(p.get("penalty_decay", 1.0)), int(p.get("seed", 0)), int(p.get("request_id", 0)),
                int(p.get("token_index", 0)), 0)
    return a if params else a[:0]


def _rows_arg(rows):
    """(keep-alive, pointer, count) for cbd_row inputs: a ROW_DTYPE array or a
    ctypes Row array as they are, anything else converted."""
    if isinstance(rows, np.ndarray):
        if rows.dtype != ROW_DTYPE:
            raise TypeError(f"rows array dtype {rows.dtype} is not ROW_DTYPE")
        a = np.ascontiguousarray(rows)
        return a, a.ctypes.data_as(_P(Row)), len(a)
    if isinstance(rows, ctypes.Array) and rows._type_ is Row:
        return rows, rows, len(rows)
    ra = rows_array(rows)
    return ra, ra, len(ra)


def _sampling_arg(params):
    if isinstance(params, np.ndarray):
        if params.dtype != SAMPLING_DTYPE:
            raise TypeError(f"sampling array dtype {params.dtype} is not SAMPLING_DTYPE")
        a = np.ascontiguousarray(params)
        if len(a) == 0:
            a = np.zeros(1, SAMPLING_DTYPE)
        return a, a.ctypes.data_as(_P(Sampling))
    if isinstance(params, ctypes.Array) and params._type_ is Sampling:
        return params, params
    sa = sampling_array(params)
    return sa, sa


def rows_array(rows) -> ctypes.Array:
    """rows: iterable of (slot, token, pos, is_prefill, sample)."""
    rows = [tuple(int(v) for v in r) for r in rows]
    arr = (Row * len(rows))()
    for i, r in enumerate(rows):
        arr[i] = Row(*r)
    return arr


def sampling_array(params) -> ctypes.Array:
    """params: iterable of dicts with the cbd_sampling fields (missing -> 0)."""
    params = list(params)
    arr = (Sampling * max(1, len(params)))()
    for i, p in enumerate(params):
        arr[i] = Sampling(float(p.get("temperature", 0.0)), float(p.get("top_p", 1.0)), int(p.get("top_k", 0)),
                          float(p.get("presence_penalty", 0.0)), float(p.get("frequency_penalty", 0.0)),
                          float(p.get("penalty_decay", 1.0)), int(p.get("seed", 0)), int(p.get("request_id", 0)),
                          int(p.get("token_index", 0)), 0)
    return arr


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(c_i32))


def _f32(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(c_f32))


def step(e, pool, rows, block_tables, n_blocks_per_slot, sampling, uniforms, out_tokens, out_logits=None,
         stream=None) -> None:
    """One batched step.  rows: (slot, token, pos, is_prefill, sample)
    tuples, or a ROW_DTYPE / ctypes Row array; block_tables [S][max_blocks_per_seq] int32;
    n_blocks_per_slot [S]; sampling: one dict per sampled row (row order), or
    a SAMPLING_DTYPE / ctypes Sampling array; uniforms: None or [m] floats;
    out_tokens / out_logits: device tensors (int32 [m], fp32 [m][V])."""
    ra, rp, nr = _rows_arg(rows)
    bt, btp = _i32(block_tables)
    nb, nbp = _i32(n_blocks_per_slot)
    sa, sp = _sampling_arg(sampling)
    ua, uap = _f32(uniforms)
    _check(lib().cbd_step(e, pool, rp, nr, btp, int(bt.shape[0]), nbp, sp, uap, _ptr(out_tokens),
                          _ptr(out_logits), _stream(stream)))


def batch_create(e, pool, rows, block_tables, n_blocks_per_slot, sampling, uniforms=None, stream=None):
    ra, rp, nr = _rows_arg(rows)
    bt, btp = _i32(block_tables)
    nb, nbp = _i32(n_blocks_per_slot)
    sa, sp = _sampling_arg(sampling)
    ua, uap = _f32(uniforms)
    out = c_vp()
    _check(lib().cbd_batch_create(e, pool, rp, nr, btp, int(bt.shape[0]), nbp, sp, uap, ctypes.byref(out),
                                  _stream(stream)))
    return out.value


def batch_run(e, pool, b, out_tokens, out_logits=None, stream=None) -> None:
    _check(lib().cbd_batch_run(e, pool, b, _ptr(out_tokens), _ptr(out_logits), _stream(stream)))


def batch_destroy(b) -> None:
    _check(lib().cbd_batch_destroy(b))


def batch_launches(b) -> int:
    n = c_i32()
    _check(lib().cbd_batch_launches(b, ctypes.byref(n)))
    return n.value


def batch_set_graph(b, enable: bool = True) -> None:
    _check(lib().cbd_batch_set_graph(b, 1 if enable else 0))


def engine_set_step_graph(e, enable: bool = True) -> None:
    _check(lib().cbd_engine_set_step_graph(e, 1 if enable else 0))


def engine_step_graph_captures(e) -> int:
    n = c_i32()
    _check(lib().cbd_engine_step_graph_captures(e, ctypes.byref(n)))
    return n.value


def batch_captures(b) -> int:
    n = c_i32()
    _check(lib().cbd_batch_captures(b, ctypes.byref(n)))
    return n.value


def sample(e, logits, slots, sampling, uniforms, out_tokens, stream=None) -> None:
    sl, slp = _i32(slots)
    sa = sampling_array(sampling)
    ua, uap = _f32(uniforms)
    _check(lib().cbd_sample(e, _ptr(logits), len(sl), slp, sa, uap, _ptr(out_tokens), _stream(stream)))


SAMPLE_STATIC_MAX_ROWS = 16
SAMPLE_STATIC_MAX_VOCAB = 65536


def sample_static(logits, counters, slots, sampling, uniforms, out_tokens, stream=None) -> None:
    """Allocation-free sampler: logits [m][V] and counters [rows][V] are
    caller-owned device tensors; see cbd_sample_static in include/cbd.h."""
    sl, slp = _i32(slots)
    sa = sampling_array(sampling)
    ua, uap = _f32(uniforms)
    _check(lib().cbd_sample_static(_ptr(logits), len(sl), int(logits.shape[1]), _ptr(counters),
                                   int(counters.shape[0]), slp, sa, uap, _ptr(out_tokens), _stream(stream)))


def sample_static_check(stream=None) -> None:
    """Raise CbdError (EDEVICE) if a cbd_sample_static call since the last
    check found no token for a row; clears the error word."""
    _check(lib().cbd_sample_static_check(_stream(stream)))


# ------------------------------------------------------------------ scheduler
def sched_create(n_blocks, block_size=32, max_slots=64, max_rows=2048, chunk=512, answer_budget=128,
                 max_blocks_per_seq=1024, reserve_answer=True, stall_fallback=True, queue_per_slot=0,
                 queue_timeout_ms=0, out_buffer=0, policy="forma", max_prefill=0, prefill_every=0, short_prompt=0):
    pol = {"forma": POLICY_FORMA, "albatross": POLICY_ALBATROSS}[policy] if isinstance(policy, str) else policy
    cfg = SchedConfig(n_blocks, block_size, max_slots, max_rows, chunk, answer_budget, max_blocks_per_seq,
                      1 if reserve_answer else 0, 1 if stall_fallback else 0, queue_per_slot, queue_timeout_ms,
                      out_buffer, pol, max_prefill, prefill_every, short_prompt)
    out = c_vp()
    _check(lib().cbd_sched_create(ctypes.byref(cfg), ctypes.byref(out)))
    _sched_width[out.value] = max_blocks_per_seq
    return out.value


_sched_width = {}


def sched_destroy(s) -> None:
    _sched_width.pop(s, None)
    _check(lib().cbd_sched_destroy(s))


def sched_submit(s, req_id: int, prompt, max_tokens: int, sampling: dict | None = None) -> None:
    pa, pp = _i32(prompt)
    sa = sampling_array([sampling or {}])
    r = Request(req_id, pp, len(pa), max_tokens, sa[0])
    _check(lib().cbd_sched_submit(s, ctypes.byref(r)))


def sched_plan(s) -> dict:
    p = Plan()
    _check(lib().cbd_sched_plan(s, ctypes.byref(p)))
    rows = [(p.rows[i].slot, p.rows[i].token, p.rows[i].pos, p.rows[i].is_prefill, p.rows[i].sample)
            for i in range(p.n_rows)]
    samp = [{f: getattr(p.sampling[i], f) for f, _ in Sampling._fields_} for i in range(p.n_sampled)]
    S = p.table_slots
    W = _sched_width[s]
    nbps = np.ctypeslib.as_array(p.n_blocks_per_slot, shape=(S,)).copy()
    tables = np.ctypeslib.as_array(p.block_tables, shape=(S, W)).copy()
    return dict(rows=rows, sampling=samp, sampled_ids=[p.sampled_ids[i] for i in range(p.n_sampled)],
                block_tables=tables, n_blocks_per_slot=nbps,
                resets=[p.reset_slots[i] for i in range(p.n_resets)],
                stopped=[p.stopped_ids[i] for i in range(p.n_stopped)])


def sched_plan_raw(s) -> Plan:
    """The next plan as the scheduler's own C struct (no Python copies of the
    rows or tables); valid until the next plan / commit.  See step_plan."""
    p = Plan()
    _check(lib().cbd_sched_plan(s, ctypes.byref(p)))
    return p


def step_plan(e, pool, p: Plan, out_tokens, out_logits=None, stream=None) -> None:
    """cbd_step over a plan from sched_plan_raw: its rows, block tables and
    sampling parameters go to the engine straight from the scheduler's
    arrays."""
    _check(lib().cbd_step(e, pool, p.rows, p.n_rows, p.block_tables, p.table_slots, p.n_blocks_per_slot,
                          p.sampling, None, _ptr(out_tokens), _ptr(out_logits), _stream(stream)))


def sched_commit(s, tokens, cap: int = 4096) -> list:
    ta, tp = _i32(tokens)
    fin = (Finished * cap)()
    n = c_i32()
    _check(lib().cbd_sched_commit(s, tp, len(ta), fin, cap, ctypes.byref(n)))
    return [(fin[i].id, fin[i].reason, fin[i].n_tokens) for i in range(n.value)]


def sched_output(s, req_id: int) -> list:
    n = c_i32()
    _check(lib().cbd_sched_output(s, req_id, None, 0, ctypes.byref(n)))
    buf = (c_i32 * max(1, n.value))()
    _check(lib().cbd_sched_output(s, req_id, buf, n.value, ctypes.byref(n)))
    return list(buf[: n.value])


def sched_abort(s, req_id: int) -> None:
    _check(lib().cbd_sched_abort(s, req_id))


def sched_set_time(s, now_ms: int) -> None:
    _check(lib().cbd_sched_set_time(s, int(now_ms)))


def sched_read(s, req_id: int, cap: int = 4096) -> list:
    buf = (c_i32 * max(1, cap))()
    n = c_i32()
    _check(lib().cbd_sched_read(s, req_id, buf, cap, ctypes.byref(n)))
    return list(buf[: n.value])


def sched_finished(s, cap: int = 4096) -> list:
    fin = (Finished * max(1, cap))()
    n = c_i32()
    _check(lib().cbd_sched_finished(s, fin, cap, ctypes.byref(n)))
    return [(fin[i].id, fin[i].reason, fin[i].n_tokens) for i in range(n.value)]


def sched_stats(s) -> dict:
    st = SchedStats()
    _check(lib().cbd_sched_stats_get(s, ctypes.byref(st)))
    return {f: getattr(st, f) for f, _ in SchedStats._fields_}


# ------------------------------------------------------------------ views
class _CAI:
    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 3, "strides": None}


def device_view(ptr: int, shape: tuple, dtype: str):
    """A torch view of libcbd-owned device memory (dtype: 'f32', 'bf16', 'i32', 'u8')."""
    import torch
    typestr = {"f32": "<f4", "bf16": "<i2", "i32": "<i4", "u8": "|u1"}[dtype]
    t = torch.as_tensor(_CAI(ptr, shape, typestr), device="cuda")
    return t.view(torch.bfloat16) if dtype == "bf16" else t
