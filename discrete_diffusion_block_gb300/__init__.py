"""Python binding of libdg, the GB300 (sm_103a) block text-diffusion decoder.

Argument marshalling only: every step of the decoding path runs in the CUDA
library behind include/dg.h.  Functions keep the C names.  Host buffers are
numpy arrays; device buffers are torch CUDA tensors (PyTorch provides device
memory and streams, nothing else).  If the compiled library is missing the
import of this module still works but every call raises: there is no CPU
fallback.
"""
import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdg.so")

DG_OK, DG_EINVAL, DG_ENOMEM, DG_ECUDA, DG_ESTATE, DG_ECAPACITY, DG_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
DG_K_CLASSES = 13
(DG_W_EMBED, DG_W_LM_HEAD, DG_W_FINAL_NORM, DG_W_WQKV, DG_W_WO, DG_W_ROUTER, DG_W_GATE_UP,
 DG_W_DOWN, DG_W_ATTN_NORM, DG_W_MOE_NORM) = range(10)


class DgError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"dg error {code}: {msg}")
        self.code = code


class dg_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "n_experts", "top_k",
        "d_ff", "vocab", "page_size", "max_context", "max_requests", "expert_fp8")] + [
        ("rope_base", ctypes.c_float), ("rms_eps", ctypes.c_float), ("init_std", ctypes.c_float),
        ("weight_seed", ctypes.c_uint64)]


class dg_sampler_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "canvas_len", "budget_N", "stable_steps", "adaptive", "eos_id", "commit_causal")] + [
        ("conf_threshold", ctypes.c_float), ("temp_start", ctypes.c_float), ("temp_end", ctypes.c_float),
        ("sample_seed", ctypes.c_uint64)]


class dg_stats(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("total_steps", ctypes.c_int32), ("n_forwards", ctypes.c_int32),
                ("effective_steps", ctypes.c_double), ("tpf", ctypes.c_double),
                ("prefill_seconds", ctypes.c_double), ("decode_seconds", ctypes.c_double),
                ("steps_per_s", ctypes.c_double), ("tokens_per_s", ctypes.c_double),
                ("canvas_loop_syncs", ctypes.c_int32),
                ("N_k", ctypes.POINTER(ctypes.c_int32)), ("C_k", ctypes.POINTER(ctypes.c_int32))]


@dataclass
class Config:
    """Model shape (mirrors dg_config)."""
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    d_ff: int
    vocab: int
    page_size: int = 128
    max_context: int = 4096
    max_requests: int = 1
    expert_fp8: int = 0
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    init_std: float = 0.02
    weight_seed: int = 0

    def to_c(self):
        return dg_config(**{f: getattr(self, f) for f, _ in dg_config._fields_})


@dataclass
class SamplerConfig:
    """Sampler of one canvas (mirrors dg_sampler_config)."""
    canvas_len: int = 256
    budget_N: int = 48
    stable_steps: int = 2
    adaptive: int = 1
    eos_id: int = -1
    commit_causal: int = 1
    conf_threshold: float = 0.9
    temp_start: float = 1.0
    temp_end: float = 1.0
    sample_seed: int = 0

    def to_c(self):
        return dg_sampler_config(**{f: getattr(self, f) for f, _ in dg_sampler_config._fields_})


def tiny_config(**kw):
    """2 layers, d=256, 4/2 heads of 64, 8 experts top-2, SwiGLU 512, vocab 1024."""
    base = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64, n_experts=8,
                top_k=2, d_ff=512, vocab=1024, max_context=1024)
    base.update(kw)
    return Config(**base)


def full_config(**kw):
    """30 layers, d=2816, 16/8 heads of 128, 128 experts top-8, FFN 704, vocab 262144."""
    base = dict(n_layers=30, d_model=2816, n_q_heads=16, n_kv_heads=8, head_dim=128,
                n_experts=128, top_k=8, d_ff=704, vocab=262144, max_context=4096)
    base.update(kw)
    return Config(**base)


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_SIGS = {
    "dg_last_error": (ctypes.c_char_p, []),
    "dg_init_model": (_I, [ctypes.POINTER(dg_config), ctypes.POINTER(dg_sampler_config), _P, _P,
                           ctypes.POINTER(_P)]),
    "dg_free_model": (None, [_P]),
    "dg_prefill": (_I, [_P, _P, _I]),
    "dg_denoise_step": (_I, [_P, _P]),
    "dg_denoise_canvas": (_I, [_P, _P]),
    "dg_prefill_batch": (_I, [_P, _P, _P]),
    "dg_denoise_canvas_batch": (_I, [_P, _P]),
    "dg_commit_canvas_batch": (_I, [_P, _P, _P]),
    "dg_generate_batch": (_I, [_P, _P, _P, _I, _P, _P]),
    "dg_commit_canvas": (_I, [_P, _P, _P]),
    "dg_generate": (_I, [_P, _P, _I, _I, _P, ctypes.POINTER(dg_stats)]),
    "dg_set_sampler": (_I, [_P, ctypes.POINTER(dg_sampler_config)]),
    "dg_rewind": (_I, [_P, _I]),
    "dg_read_canvas": (_I, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "dg_write_canvas": (_I, [_P, _P, _P, _P, _P, _I, _I]),
    "dg_read_step_outputs": (_I, [_P, _P, _P, _P]),
    "dg_canvas_logits": (_I, [_P, _P]),
    "dg_read_kv": (_I, [_P, _I, _I, _I, _P, _P]),
    "dg_read_routing": (_I, [_P, _I, _P, _I, _P]),
    "dg_read_moe_input": (_I, [_P, _P, _I, _P, _P]),
    "dg_read_page_table": (_I, [_P, _P, _I, _P]),
    "dg_get_weight": (_I, [_P, _I, _I, ctypes.POINTER(_P), ctypes.POINTER(_SZ)]),
    "dg_kernel_class_name": (ctypes.c_char_p, [_I]),
    "dg_profile": (_I, [_P, _I]),
    "dg_profile_read": (_I, [_P, _P, _P]),
    "dg_profile_experts": (_I, [_P, _P, _P]),
    "dg_op_fill_weights": (_I, [_P, _U64, _U64, ctypes.c_uint32, _U64, _F, _P]),
    "dg_op_attention_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "dg_op_status": (_I, [_P]),
    "dg_op_wait_selftest": (_I, [ctypes.c_int64, _P]),
    "dg_op_canvas_attention": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "dg_op_canvas_attention_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "dg_op_moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "dg_op_moe": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "dg_op_fill_moe_weights": (_I, [_P, _P, _P, _I, _I, _I, _I, _U64, _F, _P]),
    "dg_op_lm_head_partials": (_I, [_P, _P, _P, _I, _I, _I, _U64, _I, _I, _F, _P, _P, _P]),
    "dg_op_logits_partials": (_I, [_P, _I, _I, _U64, _I, _I, _F, _P, _P]),
    "dg_op_gumbel_noise": (_I, [_P, _P, _U64, _P]),
    "dg_op_quantize_rows_e4m3": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "dg_op_fill_tiled_weights": (_I, [_P, _I, _I, _U64, ctypes.c_uint32, _F, _P]),
    "dg_op_sampler_update": (_I, [_P, _I, _I, _I, ctypes.POINTER(dg_sampler_config), _P, _P, _P,
                                  _P, _P, _P, _P, _P, _P]),
    "dg_op_kv_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
}


def exported_symbols():
    return sorted(_SIGS)


def load(path=LIB_PATH):
    """Load libdg.so (built by discrete_diffusion_block_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run discrete_diffusion_block_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(code):
    if code != DG_OK:
        raise DgError(code, load().dg_last_error().decode())


def _ptr(a):
    """Address of a numpy array, torch tensor or raw int (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    assert a.is_contiguous()
    return a.data_ptr()


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32(a):
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


# ---- model-level calls -------------------------------------------------------

class Model:
    """Owner of a dg_model*; freed on close() / garbage collection."""

    def __init__(self, handle, cfg, scfg):
        self.handle, self.cfg, self.scfg = handle, cfg, scfg

    def close(self):
        if self.handle:
            load().dg_free_model(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def n_weight_tensors(cfg):
    """Entries of dg_init_model's borrowed-weights array."""
    return 3 + 7 * cfg.n_layers


def dg_init_model(cfg, scfg=None, stream=None, weights=None):
    """weights: None (seeded weights owned by the model) or a sequence of
    n_weight_tensors(cfg) device tensors / addresses in the DG_W_* order
    (borrowed: they must outlive the model)."""
    scfg = scfg or SamplerConfig()
    c, s = cfg.to_c(), scfg.to_c()
    h = ctypes.c_void_p()
    arr = None
    if weights is not None:
        assert len(weights) == n_weight_tensors(cfg)
        arr = (ctypes.c_void_p * len(weights))(*[_ptr(w) for w in weights])
    _check(load().dg_init_model(ctypes.byref(c), ctypes.byref(s), arr, _stream(stream), ctypes.byref(h)))
    model = Model(h.value, cfg, scfg)
    model.borrowed = weights          # keeps borrowed tensors alive as long as the model
    return model


def dg_free_model(m):
    m.close()


def dg_prefill(m, prompt_ids):
    p = _i32(prompt_ids)
    _check(load().dg_prefill(m.handle, _ptr(p) if len(p) else None, len(p)))


def dg_denoise_step(m):
    done = ctypes.c_int32()
    _check(load().dg_denoise_step(m.handle, ctypes.byref(done)))
    return bool(done.value)


def dg_denoise_canvas(m):
    """Denoise the current canvas to the end on the device; returns the steps taken."""
    n = ctypes.c_int32()
    _check(load().dg_denoise_canvas(m.handle, ctypes.byref(n)))
    return n.value


def dg_commit_canvas(m):
    ids = np.zeros(m.scfg.canvas_len, np.int32)
    valid = ctypes.c_int32()
    _check(load().dg_commit_canvas(m.handle, _ptr(ids), ctypes.byref(valid)))
    return ids, valid.value


def dg_generate(m, prompt, K_max):
    p = _i32(prompt)
    out = np.zeros((K_max, m.scfg.canvas_len), np.int32)
    Nk, Ck = np.zeros(K_max, np.int32), np.zeros(K_max, np.int32)
    st = dg_stats()
    st.N_k = Nk.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    st.C_k = Ck.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    _check(load().dg_generate(m.handle, _ptr(p) if len(p) else None, len(p), K_max, _ptr(out),
                              ctypes.byref(st)))
    K = st.K
    stats = dict(K=K, total_tokens=st.total_tokens, total_steps=st.total_steps,
                 n_forwards=st.n_forwards, effective_steps=st.effective_steps, tpf=st.tpf,
                 prefill_seconds=st.prefill_seconds, decode_seconds=st.decode_seconds,
                 steps_per_s=st.steps_per_s, tokens_per_s=st.tokens_per_s,
                 canvas_loop_syncs=st.canvas_loop_syncs,
                 N_k=Nk[:K].tolist(), C_k=Ck[:K].tolist())
    return out[:K], stats


def _prompt_arrays(prompts):
    ps = [_i32(p) for p in prompts]
    ptrs = (ctypes.c_void_p * len(ps))(*[p.ctypes.data if len(p) else None for p in ps])
    lens = np.array([len(p) for p in ps], np.int32)
    return ps, ptrs, lens


def dg_prefill_batch(m, prompts):
    ps, ptrs, lens = _prompt_arrays(prompts)
    _check(load().dg_prefill_batch(m.handle, ptrs, _ptr(lens)))


def dg_denoise_canvas_batch(m):
    """Steps at which each request's canvas finished."""
    n = np.zeros(m.cfg.max_requests or 1, np.int32)
    _check(load().dg_denoise_canvas_batch(m.handle, _ptr(n)))
    return n.tolist()


def dg_commit_canvas_batch(m):
    B = m.cfg.max_requests or 1
    ids = np.zeros((B, m.scfg.canvas_len), np.int32)
    valid = np.zeros(B, np.int32)
    _check(load().dg_commit_canvas_batch(m.handle, _ptr(ids), _ptr(valid)))
    return ids, valid.tolist()


def dg_generate_batch(m, prompts, K_max):
    """(ids [B][K_max][C] (canvases past a request's K are not reported), per-request stats)."""
    B = m.cfg.max_requests or 1
    assert len(prompts) == B
    ps, ptrs, lens = _prompt_arrays(prompts)
    out = np.zeros((B, K_max, m.scfg.canvas_len), np.int32)
    Nk, Ck = np.zeros((B, K_max), np.int32), np.zeros((B, K_max), np.int32)
    sts = (dg_stats * B)()
    for b in range(B):
        sts[b].N_k = Nk[b].ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        sts[b].C_k = Ck[b].ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    _check(load().dg_generate_batch(m.handle, ptrs, _ptr(lens), K_max, _ptr(out), sts))
    stats = []
    for b in range(B):
        st = sts[b]
        stats.append(dict(K=st.K, total_tokens=st.total_tokens, total_steps=st.total_steps,
                          n_forwards=st.n_forwards, effective_steps=st.effective_steps, tpf=st.tpf,
                          prefill_seconds=st.prefill_seconds, decode_seconds=st.decode_seconds,
                          steps_per_s=st.steps_per_s, tokens_per_s=st.tokens_per_s,
                          canvas_loop_syncs=st.canvas_loop_syncs, N_k=Nk[b][:st.K].tolist(),
                          C_k=Ck[b][:st.K].tolist()))
    return out, stats


def dg_set_sampler(m, scfg):
    s = scfg.to_c()
    _check(load().dg_set_sampler(m.handle, ctypes.byref(s)))
    m.scfg = scfg


def dg_rewind(m, n_prefix):
    _check(load().dg_rewind(m.handle, n_prefix))


def dg_read_canvas(m):
    C = m.scfg.canvas_len
    ids, com = np.zeros(C, np.int32), np.zeros(C, np.uint8)
    last, stab = np.zeros(C, np.int32), np.zeros(C, np.int32)
    step, k, pre = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().dg_read_canvas(m.handle, _ptr(ids), _ptr(com), _ptr(last), _ptr(stab),
                                 ctypes.byref(step), ctypes.byref(k), ctypes.byref(pre)))
    return dict(ids=ids, committed=com, last=last, stable=stab, step=step.value,
                canvas_index=k.value, prefix_len=pre.value)


def dg_write_canvas(m, ids, committed, last, stable, step, canvas_index):
    a, b = _i32(ids), np.ascontiguousarray(committed, dtype=np.uint8)
    c, d = _i32(last), _i32(stable)
    _check(load().dg_write_canvas(m.handle, _ptr(a), _ptr(b), _ptr(c), _ptr(d), step, canvas_index))


def dg_read_step_outputs(m):
    C = m.scfg.canvas_len
    a, conf, g = np.zeros(C, np.int32), np.zeros(C, np.float32), np.zeros(C, np.int32)
    _check(load().dg_read_step_outputs(m.handle, _ptr(a), _ptr(conf), _ptr(g)))
    return a, conf, g


def dg_canvas_logits(m, logits_dev):
    _check(load().dg_canvas_logits(m.handle, _ptr(logits_dev)))


def dg_read_kv(m, layer, pos0, n):
    shape = (n, m.cfg.n_kv_heads, m.cfg.head_dim)
    k, v = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    _check(load().dg_read_kv(m.handle, layer, pos0, n, _ptr(k), _ptr(v)))
    return k, v


def dg_read_moe_input(m):
    """(bf16 bits [rows][d_model] uint16, layer) of the last MoE input."""
    n, L = ctypes.c_int32(), ctypes.c_int32()
    _check(load().dg_read_moe_input(m.handle, None, 0, ctypes.byref(n), ctypes.byref(L)))
    rows = np.zeros((n.value, m.cfg.d_model), np.uint16)
    _check(load().dg_read_moe_input(m.handle, _ptr(rows), n.value, ctypes.byref(n), ctypes.byref(L)))
    return rows, L.value


def dg_read_routing(m, layer):
    n = ctypes.c_int32()
    _check(load().dg_read_routing(m.handle, layer, None, 0, ctypes.byref(n)))
    ids = np.zeros((n.value, m.cfg.top_k), np.int32)
    _check(load().dg_read_routing(m.handle, layer, _ptr(ids), n.value, ctypes.byref(n)))
    return ids


def dg_read_page_table(m, max_entries=1 << 16):
    t = np.zeros(max_entries, np.int32)
    n = ctypes.c_int32()
    _check(load().dg_read_page_table(m.handle, _ptr(t), max_entries, ctypes.byref(n)))
    return t[:n.value]


def dg_get_weight(m, which, layer=0):
    p, b = ctypes.c_void_p(), ctypes.c_size_t()
    _check(load().dg_get_weight(m.handle, which, layer, ctypes.byref(p), ctypes.byref(b)))
    return p.value, b.value


def dg_kernel_class_name(cls):
    return load().dg_kernel_class_name(cls).decode()


def dg_profile(m, enable):
    _check(load().dg_profile(m.handle, int(enable)))


def dg_profile_read(m):
    """{class name: (device ms, kernel launches)} since the last dg_profile(m, 1)."""
    ms, n = np.zeros(DG_K_CLASSES, np.float64), np.zeros(DG_K_CLASSES, np.int64)
    _check(load().dg_profile_read(m.handle, _ptr(ms), _ptr(n)))
    return {dg_kernel_class_name(i): (float(ms[i]), int(n[i])) for i in range(DG_K_CLASSES)}


def dg_profile_experts(m):
    """(experts touched, rows routed) summed over MoE launches since dg_profile(m, 1)."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(load().dg_profile_experts(m.handle, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


# ---- kernel-level calls (torch CUDA tensors for device buffers) --------------

def dg_op_fill_weights(dst, seed, tensor_id, e0=0, std=0.02, stream=None):
    _check(load().dg_op_fill_weights(_ptr(dst), dst.numel(), seed, tensor_id, e0, std, _stream(stream)))


def dg_op_attention_workspace_bytes(n_prefix, n_new, Hq, Hkv, hd):
    return load().dg_op_attention_workspace_bytes(n_prefix, n_new, Hq, Hkv, hd)


def dg_op_status(stream=None):
    """Raises DgError if a kernel-level call since the last check recorded a
    device-side failure (bounded wait timeout, bad page index)."""
    _check(load().dg_op_status(_stream(stream)))


def dg_op_wait_selftest(limit_cycles, stream=None):
    _check(load().dg_op_wait_selftest(limit_cycles, _stream(stream)))


def dg_op_canvas_attention(q, k_pool, v_pool, page_table, n_prefix, n_new, Hq, Hkv, hd, page_size,
                           causal, out, workspace, stream=None, n_pages=None):
    n_pages = k_pool.shape[0] if n_pages is None else n_pages     # pools [n_pages][Hkv][pg][hd]
    _check(load().dg_op_canvas_attention(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                         n_prefix, n_new, Hq, Hkv, hd, page_size, n_pages, int(causal),
                                         _ptr(out), _ptr(workspace), _nbytes(workspace),
                                         _stream(stream)))


def dg_op_canvas_attention_noalloc(q, k_pool, v_pool, page_table, n_prefix, n_new, Hq, Hkv, hd,
                                   page_size, causal, out, stream=None, n_pages=None):
    """dg_op_canvas_attention without a workspace argument; allocates nothing."""
    n_pages = k_pool.shape[0] if n_pages is None else n_pages
    _check(load().dg_op_canvas_attention_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                                 _ptr(page_table), n_prefix, n_new, Hq, Hkv, hd,
                                                 page_size, n_pages, int(causal), _ptr(out),
                                                 _stream(stream)))


def dg_op_moe_workspace_bytes(T, d, E, k, F):
    return load().dg_op_moe_workspace_bytes(T, d, E, k, F)


def dg_op_moe(xn, w_router, w_gate_up, w_down, T, d, E, k, F, y, ids, gates, workspace, stream=None):
    _check(load().dg_op_moe(_ptr(xn), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down), T, d, E, k, F,
                            _ptr(y), _ptr(ids), _ptr(gates), _ptr(workspace), _nbytes(workspace),
                            _stream(stream)))


def dg_op_fill_moe_weights(w_router, w_gate_up, w_down, d, E, F, layer, seed, std=0.02, stream=None):
    _check(load().dg_op_fill_moe_weights(_ptr(w_router), _ptr(w_gate_up), _ptr(w_down), d, E, F,
                                         layer, seed, std, _stream(stream)))


def partials_bytes(rows, V):
    return rows * (V // 256) * 20


def dg_op_lm_head_partials(xn, w_out, rows, d, V, seed, canvas, step, partials, stream=None,
                           xn_lo=None, logits=None, inv_tau=1.0):
    _check(load().dg_op_lm_head_partials(_ptr(xn), _ptr(xn_lo), _ptr(w_out), rows, d, V, seed, canvas,
                                         step, inv_tau, _ptr(partials), _ptr(logits), _stream(stream)))


def dg_op_logits_partials(logits, rows, V, seed, canvas, step, partials, stream=None, inv_tau=1.0):
    _check(load().dg_op_logits_partials(_ptr(logits), rows, V, seed, canvas, step, inv_tau, _ptr(partials),
                                        _stream(stream)))


def dg_op_fill_tiled_weights(dst, rows, cols, seed, tensor_id, std=0.02, stream=None):
    _check(load().dg_op_fill_tiled_weights(_ptr(dst), rows, cols, seed, tensor_id, std, _stream(stream)))


def to_operand_tiles(x):
    """Row-major [rows][cols] numpy array (cols a multiple of 64) -> the
    library's operand-tile order (128-row blocks, the last one partial; per
    block cols/64 tiles of (block rows) x 64, the 16-byte chunk c of row r at
    chunk position c ^ (r % 8)), flattened.  Host-side layout marshalling."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    out = []
    for b0 in range(0, rows, 128):
        blk = x[b0:b0 + 128]
        n = blk.shape[0]
        t = blk.reshape(n, cols // 64, 8, 8).transpose(1, 0, 2, 3)          # [kt][row][chunk][8]
        pos = np.arange(8)[None, :] ^ (np.arange(n)[:, None] % 8)           # stored position of chunk c
        o = np.empty_like(t)
        o[:, np.arange(n)[:, None], pos, :] = t
        out.append(o.reshape(-1))
    return np.concatenate(out)


def dg_op_gumbel_noise(words, out, stream=None):
    _check(load().dg_op_gumbel_noise(_ptr(words), _ptr(out), words.numel(), _stream(stream)))


def dg_op_quantize_rows_e4m3(src_tiles, n_mat, rows, cols, dst, exps, stream=None):
    """bf16 operand tiles of n_mat [rows][cols] matrices -> e4m3 operand tiles
    (dst: rows * cols bytes each) and row scale exponents (exps int32)."""
    _check(load().dg_op_quantize_rows_e4m3(_ptr(src_tiles), n_mat, rows, cols, _ptr(dst), _ptr(exps),
                                           _stream(stream)))


def dg_op_sampler_update(partials, C, V, step, scfg, x, committed, last, stable, argmax, conf,
                         gumbel, done, stream=None):
    s = scfg.to_c()
    _check(load().dg_op_sampler_update(_ptr(partials), C, V, step, ctypes.byref(s), _ptr(x),
                                       _ptr(committed), _ptr(last), _ptr(stable), _ptr(argmax),
                                       _ptr(conf), _ptr(gumbel), _ptr(done), _stream(stream)))


def dg_op_kv_append(k_new, v_new, k_pool, v_pool, page_table, n_layers, n_pages, pos0, n_new, Hkv,
                    hd, page_size, stream=None):
    _check(load().dg_op_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                  _ptr(page_table), n_layers, n_pages, pos0, n_new, Hkv, hd,
                                  page_size, _stream(stream)))
