"""Python access to the CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package; the product library never
does, and it never imports the product.  The oracle's inputs come from the
seeded generator in ``synth`` (or from host arrays the harness made with it).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, List, Optional, Sequence

import numpy as np

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
BUILT_LIB = os.path.join(BUILD, "liboracle.so")
# The mutation test points this at a deliberately broken build of the oracle.
LIB = os.environ.get("MK_ORACLE_LIB_OVERRIDE", BUILT_LIB)


def build_commands() -> List[List[str]]:
    os.makedirs(BUILD, exist_ok=True)
    return [["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
             os.path.join(HERE, "oracle.cpp"), "-o", BUILT_LIB]]


def build() -> None:
    for c in build_commands():
        subprocess.check_call(c)


class Dims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("rope_base", ctypes.c_double), ("rms_eps", ctypes.c_float)]


class Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("seed", ctypes.c_uint64), ("tid", ctypes.c_uint64),
                ("sigma", ctypes.c_double), ("is_const", ctypes.c_int32),
                ("const_bits", ctypes.c_uint16)]


class Layer(ctypes.Structure):
    _fields_ = [("norm", Tensor), ("wq", Tensor), ("wk", Tensor), ("wv", Tensor),
                ("wo", Tensor), ("wr", Tensor), ("router_bias", ctypes.c_void_p),
                ("wg", Tensor), ("wu", Tensor), ("wd", Tensor),
                ("kpool", Tensor), ("vpool", Tensor)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", Tensor), ("final_norm", Tensor), ("lm_head", Tensor),
                ("layers", ctypes.POINTER(Layer))]


class StepOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "next_tokens", "argmax_margin", "route_ids", "route_w",
                 "route_margin", "router_logits", "h", "n", "q", "k", "v", "o", "attn",
                 "moe")] + [("route_mismatch", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} missing: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.orc_create.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights), i32, vp, vp, i32, i32]
        L.orc_create.restype = vp
        L.orc_destroy.argtypes = [vp]
        L.orc_step.argtypes = [vp, vp, vp, ctypes.c_float, ctypes.POINTER(StepOut)]
        L.orc_step.restype = i32
        L.orc_layer_step.argtypes = [vp, i32, vp, vp, ctypes.c_float, i32, vp,
                                     ctypes.POINTER(StepOut)]
        L.orc_layer_step.restype = i32
        L.orc_head.argtypes = [vp, vp, ctypes.POINTER(StepOut)]
        L.orc_head.restype = i32
        L.orc_advance.argtypes = [vp]
        L.orc_advance.restype = i32
        L.orc_reset_seq.argtypes = [vp, i32, i32, vp]
        L.orc_reset_seq.restype = i32
        L.orc_rmsnorm.argtypes = [vp, vp, i32, ctypes.c_float, i32, vp]
        L.orc_gemv.argtypes = [vp, i32, i32, vp, i32, vp]
        L.orc_rope.argtypes = [vp, i32, i32, i64, ctypes.c_double]
        L.orc_attention_head.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.orc_route.argtypes = [vp, i32, i32, vp, vp, vp]
        L.orc_silu.argtypes = [ctypes.c_float]
        L.orc_silu.restype = ctypes.c_float
        L.orc_expert.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------ building blocks


def rmsnorm(h_bits, g_bits, eps, accum_double=False) -> np.ndarray:
    h, g = _c(h_bits, np.uint16), _c(g_bits, np.uint16)
    out = np.empty_like(h)
    lib().orc_rmsnorm(_ptr(h), _ptr(g), h.size, eps, int(accum_double), _ptr(out))
    return out


def gemv(w_bits, x_bits, accum_double=False) -> np.ndarray:
    w, x = _c(w_bits, np.uint16), _c(x_bits, np.uint16)
    out = np.empty(w.shape[0], dtype=np.float32)
    lib().orc_gemv(_ptr(w), w.shape[0], w.shape[1], _ptr(x), int(accum_double), _ptr(out))
    return out


def rope(x_bits, n_heads, head_dim, pos, base) -> np.ndarray:
    x = _c(x_bits, np.uint16).copy()
    lib().orc_rope(_ptr(x), n_heads, head_dim, pos, base)
    return x


def attention_head(q_bits, k_bits, v_bits, accum_double=False) -> np.ndarray:
    q, k, v = _c(q_bits, np.uint16), _c(k_bits, np.uint16), _c(v_bits, np.uint16)
    out = np.empty(q.size, dtype=np.uint16)
    lib().orc_attention_head(_ptr(q), _ptr(k), _ptr(v), k.shape[0], q.size, int(accum_double),
                             _ptr(out))
    return out


def route(logits, k):
    r = _c(logits, np.float32)
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float32)
    margin = np.empty(1, dtype=np.float32)
    lib().orc_route(_ptr(r), r.size, k, _ptr(ids), _ptr(w), _ptr(margin))
    return ids, w, float(margin[0])


def silu(x: float) -> float:
    return float(lib().orc_silu(x))


def expert(n_bits, wg_bits, wu_bits, wd_bits, accum_double=False) -> np.ndarray:
    n, wg, wu, wd = (_c(a, np.uint16) for a in (n_bits, wg_bits, wu_bits, wd_bits))
    d, f = n.size, wg.shape[0]
    y = np.empty(d, dtype=np.float32)
    lib().orc_expert(_ptr(n), _ptr(wg), _ptr(wu), _ptr(wd), d, f, int(accum_double), _ptr(y))
    return y


# ----------------------------------------------------------------- decode state


def _tensor(src, seed: int) -> Tensor:
    """src: a numpy uint16 array (materialised) or a synth.TensorSpec (generated)."""
    t = Tensor()
    if isinstance(src, np.ndarray):
        t.data = src.ctypes.data
    elif src.const_bits is not None:
        t.is_const, t.const_bits = 1, src.const_bits
    else:
        t.seed, t.tid, t.sigma = seed, src.tid, src.sigma
    return t


class Oracle:
    """One decode state.  ``tensors`` maps names (synth.weight_specs / kv_specs)
    to host uint16 arrays or to TensorSpecs that the oracle regenerates."""

    def __init__(self, dims: synth.Dims, tensors: Dict[str, object], seq_lens: Sequence[int],
                 page_tables: np.ndarray, router_biases: Optional[List] = None,
                 accum_double: bool = False, seed: int = 0, reverse: bool = False):
        """accum_double: sums in double; reverse: fp32 sums in descending
        index order (otherwise fp32 in ascending order)."""
        self.dims = dims
        self.B = len(seq_lens)
        self._keep = [v for v in tensors.values() if isinstance(v, np.ndarray)]
        self.cd = Dims(dims.n_layers, dims.d_model, dims.n_q_heads, dims.n_kv_heads,
                       dims.head_dim, dims.n_experts, dims.top_k, dims.d_ffn, dims.vocab,
                       dims.page_size, dims.rope_base, dims.rms_eps)
        L = dims.n_layers
        self.layers = (Layer * L)()
        self._bias = []
        for l in range(L):
            ly = self.layers[l]
            for f in ("norm", "wq", "wk", "wv", "wo", "wr", "wg", "wu", "wd", "kpool", "vpool"):
                setattr(ly, f, _tensor(tensors[f"l{l}.{f}"], seed))
            b = None if router_biases is None else router_biases[l]
            if b is not None:
                b = _c(b, np.float32)
                self._bias.append(b)
                ly.router_bias = b.ctypes.data
        self.w = Weights(_tensor(tensors["embed"], seed), _tensor(tensors["final_norm"], seed),
                         _tensor(tensors["lm_head"], seed), self.layers)
        self.seq_lens = _c(seq_lens, np.int32)
        self.pt = _c(page_tables, np.int32)
        self.h = lib().orc_create(ctypes.byref(self.cd), ctypes.byref(self.w), self.B,
                                  _ptr(self.seq_lens), _ptr(self.pt), self.pt.shape[1],
                                  1 if accum_double else (2 if reverse else 0))
        if not self.h:
            raise ValueError("orc_create rejected the arguments")

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_destroy(self.h)
            self.h = None

    def step(self, tokens, forced_ids=None, tie_eps: float = 1e-2,
             dumps: Sequence[str] = ()) -> Dict[str, np.ndarray]:
        d = self.dims
        B, L, k, E = self.B, d.n_layers, d.top_k, d.n_experts
        D, Hq, Hkv, dm = d.head_dim, d.n_q_heads, d.n_kv_heads, d.d_model
        res = {
            "logits": np.empty((B, d.vocab), np.float32),
            "next_tokens": np.empty(B, np.int32),
            "argmax_margin": np.empty(B, np.float32),
            "route_ids": np.empty((L, B, k), np.int32),
            "route_w": np.empty((L, B, k), np.float32),
            "route_margin": np.empty((L, B), np.float32),
        }
        shapes = {"router_logits": ((L, B, E), np.float32), "h": ((L + 1, B, dm), np.uint16),
                  "n": ((L, B, dm), np.uint16), "q": ((L, B, Hq * D), np.uint16),
                  "k": ((L, B, Hkv * D), np.uint16), "v": ((L, B, Hkv * D), np.uint16),
                  "o": ((L, B, Hq * D), np.uint16), "attn": ((L, B, dm), np.uint16),
                  "moe": ((L, B, dm), np.uint16)}
        for name in dumps:
            shp, dt = shapes[name]
            res[name] = np.empty(shp, dt)
        so = StepOut()
        for name, arr in res.items():
            setattr(so, name, arr.ctypes.data)
        tok = _c(tokens, np.int32)
        fid = None if forced_ids is None else _c(forced_ids, np.int32)
        rc = lib().orc_step(self.h, _ptr(tok), _ptr(fid), tie_eps, ctypes.byref(so))
        if rc != 0:
            raise ValueError(f"orc_step failed ({rc})")
        res["route_mismatch"] = so.route_mismatch
        return res

    # ------------------------------------------------ teacher-forced evaluation

    def layer(self, layer: int, h_in, forced_ids=None, tie_eps: float = 1e-2, keep: bool = False,
              dumps: Sequence[str] = ()) -> Dict[str, np.ndarray]:
        """Layer `layer` of the step from the residual h_in (bf16 bits [B][d]),
        e.g. another implementation's; returns the residual entering the next
        layer ("h_out", bf16 bits) plus the routing and the requested one-layer
        dumps ("n", "q", "k", "v", "o", "attn", "moe", "router_logits").  keep:
        keep the new K/V rows (replaying a whole step; call advance() after
        the last layer)."""
        d = self.dims
        B, k, E = self.B, d.top_k, d.n_experts
        D, Hq, Hkv, dm = d.head_dim, d.n_q_heads, d.n_kv_heads, d.d_model
        res = {"h_out": np.empty((B, dm), np.uint16),
               "route_ids": np.empty((B, k), np.int32),
               "route_w": np.empty((B, k), np.float32),
               "route_margin": np.empty(B, np.float32)}
        shapes = {"router_logits": ((B, E), np.float32), "n": ((B, dm), np.uint16),
                  "q": ((B, Hq * D), np.uint16), "k": ((B, Hkv * D), np.uint16),
                  "v": ((B, Hkv * D), np.uint16), "o": ((B, Hq * D), np.uint16),
                  "attn": ((B, dm), np.uint16), "moe": ((B, dm), np.uint16)}
        for name in dumps:
            shp, dt = shapes[name]
            res[name] = np.empty(shp, dt)
        so = StepOut()
        for name, arr in res.items():
            if name != "h_out":
                setattr(so, name, arr.ctypes.data)
        h = _c(h_in, np.uint16)
        fid = None if forced_ids is None else _c(forced_ids, np.int32)
        rc = lib().orc_layer_step(self.h, layer, _ptr(h), _ptr(fid), tie_eps, int(keep),
                                  _ptr(res["h_out"]), ctypes.byref(so))
        if rc != 0:
            raise ValueError(f"orc_layer_step failed ({rc})")
        res["route_mismatch"] = so.route_mismatch
        return res

    def head(self, h_final) -> Dict[str, np.ndarray]:
        """Final norm, LM head and argmax of the final residual h_final (bf16
        bits [B][d])."""
        B, V = self.B, self.dims.vocab
        res = {"logits": np.empty((B, V), np.float32), "next_tokens": np.empty(B, np.int32),
               "argmax_margin": np.empty(B, np.float32)}
        so = StepOut()
        for name, arr in res.items():
            setattr(so, name, arr.ctypes.data)
        h = _c(h_final, np.uint16)
        if lib().orc_head(self.h, _ptr(h), ctypes.byref(so)) != 0:
            raise ValueError("orc_head failed")
        return res

    def advance(self) -> None:
        """Every sequence's length advances by one (the end of a replayed step)."""
        if lib().orc_advance(self.h) != 0:
            raise ValueError("orc_advance failed")

    def reset_seq(self, b: int, new_len: int, page_row) -> None:
        """Slot b gets a new sequence of new_len cached tokens in the pages of
        page_row (continuous batching); the other slots keep their state."""
        pr = _c(page_row, np.int32)
        if pr.size != self.pt.shape[1]:
            raise ValueError("page_row must have max_pages entries")
        if lib().orc_reset_seq(self.h, b, new_len, _ptr(pr)) != 0:
            raise ValueError("orc_reset_seq failed")
        self.pt[b] = pr
