"""Python binding of libmk, the persistent MoE decode megakernel (C ABI in include/mk.h).

Argument marshalling only: every step of the decode path runs in the CUDA
library.  Functions keep the C names.  Device buffers may be given as torch
tensors (their data_ptr() is passed) or as integer addresses; host arrays as
numpy arrays.  Errors raise MkError carrying the mk_status code.

There is no CPU fallback: if the library has not been built, importing works
but every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(BUILD, "libmk.so")

ARCH = "-gencode=arch=compute_103a,code=sm_103a"
SOURCES = ["mk_kernel.cu", "mk_api.cpp", "mk_schedule.cpp", "mk_noalloc.cu"]

MK_OK = 0
STATUS_NAMES = {0: "MK_OK", 1: "MK_ERR_INVALID_ARG", 2: "MK_ERR_BATCH", 3: "MK_ERR_PAGE_OOB",
                4: "MK_ERR_NO_SCHEDULE", 5: "MK_ERR_CUDA", 6: "MK_ERR_DEVICE_TIMEOUT",
                7: "MK_ERR_BAD_TASK", 8: "MK_ERR_UNSUPPORTED", 9: "MK_ERR_NO_DEVICE",
                10: "MK_ERR_SCRATCH_LIMIT", 11: "MK_ERR_BAD_TOKEN"}
MK_ERR_INVALID_ARG, MK_ERR_BATCH, MK_ERR_PAGE_OOB, MK_ERR_NO_SCHEDULE = 1, 2, 3, 4
MK_ERR_CUDA, MK_ERR_DEVICE_TIMEOUT, MK_ERR_BAD_TASK, MK_ERR_UNSUPPORTED = 5, 6, 7, 8
MK_ERR_NO_DEVICE = 9
MK_ERR_SCRATCH_LIMIT = 10
MK_ERR_BAD_TOKEN = 11


def build_commands() -> List[List[str]]:
    """nvcc commands: one object per source (run them in parallel), then the link."""
    os.makedirs(BUILD, exist_ok=True)
    cmds = []
    objs = []
    for s in SOURCES:
        obj = os.path.join(BUILD, s + ".o")
        objs.append(obj)
        cmds.append(["nvcc", ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, s), "-o", obj])
    link = ["nvcc", ARCH, "-shared", "-o", LIB_PATH] + objs + ["-lcudart"]
    return cmds + [link]


def build(verbose: bool = False) -> None:
    cmds = build_commands()
    procs = [subprocess.Popen(c, stdout=None if verbose else subprocess.PIPE,
                              stderr=subprocess.STDOUT) for c in cmds[:-1]]
    for p, c in zip(procs, cmds):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("libmk build failed: " + " ".join(c) + "\n" + (out or b"").decode())
    subprocess.check_call(cmds[-1])


class MkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


# ------------------------------------------------------------------- C structs


class mk_model_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "n_experts",
                 "top_k", "d_ffn", "vocab", "page_size", "max_batch", "num_pages",
                 "max_pages_per_seq")] + [("rope_base", ctypes.c_float),
                                          ("rms_eps", ctypes.c_float)]


class mk_layer_ptrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("norm", "wq", "wk", "wv", "wo", "w_router", "router_bias", "w_gate", "w_up",
                 "w_down", "k_cache", "v_cache")]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("layers", ctypes.POINTER(mk_layer_ptrs)),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


class mk_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("sum_experts", ctypes.c_uint64),
                ("rebuilds", ctypes.c_uint64)]


class mk_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_cta", "tasks_per_cta", "n_layer_tasks_max", "n_qkv", "n_router", "n_attn",
                 "n_up", "n_out", "n_lm", "n_attn_slots", "n_down")]


EXPORTS = ["mk_create", "mk_build_schedule", "mk_decode_step", "mk_sync", "mk_destroy",
           "mk_status_string", "mk_set_wait_limit_ns", "mk_debug_routing", "mk_debug_dump",
           "mk_get_stats", "mk_debug_poison_wait", "mk_plan", "mk_decode_step_static",
           "mk_set_trace", "mk_get_trace", "mk_set_stage_trace_cta"]

_lib = None


def lib():
    """The loaded libmk (raises if it was not built: no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        L.mk_create.argtypes = [ctypes.POINTER(mk_model_dims), ctypes.POINTER(mk_weights), vp,
                                ctypes.POINTER(vp)]
        L.mk_build_schedule.argtypes = [vp, i32, vp, vp]
        L.mk_decode_step.argtypes = [vp, vp, vp, vp]
        L.mk_sync.argtypes = [vp]
        L.mk_destroy.argtypes = [vp]
        L.mk_destroy.restype = None
        L.mk_status_string.argtypes = [i32]
        L.mk_status_string.restype = ctypes.c_char_p
        L.mk_set_wait_limit_ns.argtypes = [vp, u64]
        L.mk_debug_routing.argtypes = [vp, vp, vp]
        L.mk_debug_dump.argtypes = [vp, i32, vp, u64]
        L.mk_get_stats.argtypes = [vp, ctypes.POINTER(mk_stats)]
        L.mk_debug_poison_wait.argtypes = [vp, i32, i32]
        L.mk_plan.argtypes = [ctypes.POINTER(mk_model_dims), i32, i32, vp,
                              ctypes.POINTER(mk_plan_info), vp, i64]
        L.mk_decode_step_static.argtypes = [ctypes.POINTER(mk_model_dims),
                                            ctypes.POINTER(mk_weights), i32, vp, vp, vp, vp, vp,
                                            vp]
        L.mk_set_trace.argtypes = [vp, i32]
        L.mk_get_trace.argtypes = [vp, vp, u64, vp, vp]
        L.mk_set_stage_trace_cta.argtypes = [vp, i32]
        for n in EXPORTS:
            if n not in ("mk_destroy", "mk_status_string"):
                getattr(L, n).restype = i32
        _lib = L
    return _lib


def _addr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _check(rc: int, where: str) -> None:
    if rc != MK_OK:
        raise MkError(rc, where)


def status_string(code: int) -> str:
    if _lib is None and not os.path.exists(LIB_PATH):
        return "library not built"
    return lib().mk_status_string(code).decode()


mk_status_string = status_string


def make_dims(n_layers, d_model, n_q_heads, n_kv_heads, head_dim, n_experts, top_k, d_ffn, vocab,
              page_size, max_batch, num_pages, max_pages_per_seq, rope_base=10000.0,
              rms_eps=1e-6) -> mk_model_dims:
    return mk_model_dims(n_layers, d_model, n_q_heads, n_kv_heads, head_dim, n_experts, top_k,
                         d_ffn, vocab, page_size, max_batch, num_pages, max_pages_per_seq,
                         rope_base, rms_eps)


class Weights:
    """Keeps the mk_weights struct and its layer array alive."""

    def __init__(self, embed, layers: Sequence[dict], final_norm, lm_head):
        n = len(layers)
        self.layer_arr = (mk_layer_ptrs * n)()
        for i, ly in enumerate(layers):
            for f in mk_layer_ptrs._fields_:
                setattr(self.layer_arr[i], f[0], _addr(ly.get(f[0])))
        self.c = mk_weights(_addr(embed), self.layer_arr, _addr(final_norm), _addr(lm_head))


def mk_create(dims: mk_model_dims, weights: Weights, stream=None) -> int:
    ctx = ctypes.c_void_p()
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else (stream or 0)
    _check(lib().mk_create(ctypes.byref(dims), ctypes.byref(weights.c), s, ctypes.byref(ctx)),
           "mk_create")
    return ctx.value


def mk_build_schedule(ctx: int, batch: int, seq_lens, page_tables) -> None:
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    pt = np.ascontiguousarray(page_tables, dtype=np.int32)
    _check(lib().mk_build_schedule(ctx, batch, sl.ctypes.data, pt.ctypes.data),
           "mk_build_schedule")


def mk_decode_step(ctx: int, token_ids, out_logits, out_next_tokens) -> None:
    _check(lib().mk_decode_step(ctx, _addr(token_ids), _addr(out_logits), _addr(out_next_tokens)),
           "mk_decode_step")


def mk_sync(ctx: int) -> None:
    _check(lib().mk_sync(ctx), "mk_sync")


def mk_destroy(ctx: int) -> None:
    if ctx:
        lib().mk_destroy(ctx)


def mk_set_wait_limit_ns(ctx: int, ns: int) -> None:
    _check(lib().mk_set_wait_limit_ns(ctx, ns), "mk_set_wait_limit_ns")


def mk_debug_poison_wait(ctx: int, layer: int, delta: int) -> None:
    _check(lib().mk_debug_poison_wait(ctx, layer, delta), "mk_debug_poison_wait")


def mk_debug_routing(ctx: int, n_layers: int, batch: int, top_k: int):
    ids = np.empty((n_layers, batch, top_k), np.int32)
    w = np.empty((n_layers, batch, top_k), np.float32)
    _check(lib().mk_debug_routing(ctx, ids.ctypes.data, w.ctypes.data), "mk_debug_routing")
    return ids, w


def mk_debug_dump(ctx: int, what: int, shape, dtype) -> np.ndarray:
    out = np.empty(shape, dtype)
    _check(lib().mk_debug_dump(ctx, what, out.ctypes.data, out.nbytes), "mk_debug_dump")
    return out


def mk_get_stats(ctx: int) -> mk_stats:
    st = mk_stats()
    _check(lib().mk_get_stats(ctx, ctypes.byref(st)), "mk_get_stats")
    return st


def mk_decode_step_static(dims: mk_model_dims, weights: Weights, batch: int, seq_lens,
                          page_tables, token_ids, out_logits, out_next_tokens,
                          stream=None) -> None:
    """One decode step with no allocation by the library (see include/mk.h)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    pt = np.ascontiguousarray(page_tables, dtype=np.int32)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else (stream or 0)
    _check(lib().mk_decode_step_static(ctypes.byref(dims), ctypes.byref(weights.c), batch,
                                       sl.ctypes.data, pt.ctypes.data, _addr(token_ids),
                                       _addr(out_logits), _addr(out_next_tokens), s),
           "mk_decode_step_static")


def mk_set_trace(ctx: int, events_per_cta: int) -> None:
    _check(lib().mk_set_trace(ctx, events_per_cta), "mk_set_trace")


STAGE_TRACE_EVENTS = 4096


def mk_set_stage_trace_cta(ctx: int, cta: int) -> None:
    _check(lib().mk_set_stage_trace_cta(ctx, cta), "mk_set_stage_trace_cta")


def mk_get_trace(ctx: int):
    """The last step's trace: (task events uint64 [n_cta][events][8], CTA 0's
    stage events uint64 [STAGE_TRACE_EVENTS][8])."""
    n_cta, ev = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().mk_get_trace(ctx, None, 0, ctypes.byref(n_cta), ctypes.byref(ev)), "mk_get_trace")
    n_task = n_cta.value * ev.value * 8
    out = np.zeros(n_task + STAGE_TRACE_EVENTS * 8, np.uint64)
    _check(lib().mk_get_trace(ctx, out.ctypes.data, out.size, None, None), "mk_get_trace")
    return (out[:n_task].reshape(n_cta.value, ev.value, 8),
            out[n_task:].reshape(STAGE_TRACE_EVENTS, 8))


def mk_plan(dims: mk_model_dims, n_sm: int, batch: int, seq_lens):
    """Host-only schedule: (info, table [n_cta][tasks_per_cta][32])."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    info = mk_plan_info()
    _check(lib().mk_plan(ctypes.byref(dims), n_sm, batch, sl.ctypes.data, ctypes.byref(info),
                         None, 0), "mk_plan")
    table = np.empty((info.n_cta, info.tasks_per_cta, 32), np.int32)
    _check(lib().mk_plan(ctypes.byref(dims), n_sm, batch, sl.ctypes.data, ctypes.byref(info),
                         table.ctypes.data, table.size), "mk_plan")
    return info, table


class Decoder:
    """Convenience wrapper: marshals a dict of device tensors (names embed,
    lm_head, final_norm, l{i}.norm / wq / wk / wv / wo / wr / wg / wu / wd /
    kpool / vpool) into mk_create and forwards the other calls.  No
    computation happens here."""

    LAYER_FIELDS = {"norm": "norm", "wq": "wq", "wk": "wk", "wv": "wv", "wo": "wo",
                    "w_router": "wr", "w_gate": "wg", "w_up": "wu", "w_down": "wd",
                    "k_cache": "kpool", "v_cache": "vpool"}

    def __init__(self, dims, tensors: dict, num_pages: int, max_pages_per_seq: int,
                 max_batch: int, bias_tensors=None, stream=None):
        self.dims = dims
        self.cdims = make_dims(dims.n_layers, dims.d_model, dims.n_q_heads, dims.n_kv_heads,
                               dims.head_dim, dims.n_experts, dims.top_k, dims.d_ffn, dims.vocab,
                               dims.page_size, max_batch, num_pages, max_pages_per_seq,
                               dims.rope_base, dims.rms_eps)
        layers = []
        for l in range(dims.n_layers):
            ly = {c: tensors[f"l{l}.{n}"] for c, n in self.LAYER_FIELDS.items()}
            ly["router_bias"] = None if bias_tensors is None else bias_tensors[l]
            layers.append(ly)
        self._keep = (tensors, bias_tensors)
        self.weights = Weights(tensors["embed"], layers, tensors["final_norm"], tensors["lm_head"])
        self.ctx = None
        self.ctx = mk_create(self.cdims, self.weights, stream)
        self.batch = 0

    def build_schedule(self, seq_lens, page_tables):
        self.batch = len(seq_lens)
        mk_build_schedule(self.ctx, self.batch, seq_lens, page_tables)

    def decode_step(self, token_ids, out_logits, out_next_tokens):
        mk_decode_step(self.ctx, token_ids, out_logits, out_next_tokens)

    def sync(self):
        mk_sync(self.ctx)

    def routing(self):
        return mk_debug_routing(self.ctx, self.dims.n_layers, self.batch, self.dims.top_k)

    def dump_h(self):
        d = self.dims
        return mk_debug_dump(self.ctx, 0, (d.n_layers + 1, self.batch, d.d_model), np.uint16)

    def dump_o(self):
        d = self.dims
        return mk_debug_dump(self.ctx, 1, (d.n_layers, self.batch, d.n_q_heads * d.head_dim),
                             np.uint16)

    def dump_router_logits(self):
        d = self.dims
        return mk_debug_dump(self.ctx, 2, (d.n_layers, self.batch, d.n_experts), np.float32)

    def dump_qkv(self):
        d = self.dims
        return mk_debug_dump(self.ctx, 3, (d.n_layers, self.batch,
                                           (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim),
                             np.uint16)

    def dump_attn_moe(self):
        d = self.dims
        shp = (d.n_layers, self.batch, d.d_model)
        return (mk_debug_dump(self.ctx, 4, shp, np.uint16), mk_debug_dump(self.ctx, 5, shp, np.uint16))

    def stats(self):
        return mk_get_stats(self.ctx)

    def close(self):
        if self.ctx:
            mk_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
