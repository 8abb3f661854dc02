"""Seeded synthetic inputs for the MoE decode step (shared by oracle and GPU side).

This module holds the input generator only: model shapes, tensor ids, the
counter-based generator (``synth_rng.h``) exposed to Python, page tables and
token streams.  It contains none of the decode step's arithmetic.  Both the
CPU oracle and the GPU harness draw their inputs from here, so the two sides
see identical bytes without sharing any code of the method itself.

Input recipe (every workload): matrices bf16 ~ N(0, 0.02^2) (Irwin-Hall(12)
approximation, see ``synth_rng.h``), norm gains 1.0, cached K/V bf16 ~ N(0, 1),
token ids uniform over the vocabulary, page tables a seeded permutation of
the KV pool's physical pages, seed 0.  The pages' model (a 30B-total /
3.3B-active MoE, "Cohere speeds up North Mini Code with new megakernel",
paragraph 1) has no public weights here; these shapes stand in for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Tuple, Dict, List, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
HOST_LIB = os.path.join(BUILD, "libsynth_host.so")
DEV_LIB = os.path.join(BUILD, "libsynth_dev.so")

BF16_ONE = 0x3F80


# --------------------------------------------------------------------------- build


def build_commands() -> List[List[str]]:
    os.makedirs(BUILD, exist_ok=True)
    host = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
            os.path.join(HERE, "synth_host.c"), "-o", HOST_LIB]
    dev = ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
           "-Xcompiler", "-fPIC", "-fmad=false", os.path.join(HERE, "synth_dev.cu"),
           "-o", DEV_LIB]
    return [host, dev]


def build() -> None:
    procs = [subprocess.Popen(c) for c in build_commands()]
    for p, c in zip(procs, build_commands()):
        if p.wait() != 0:
            raise RuntimeError("synth build failed: " + " ".join(c))


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(HOST_LIB)
        u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.syn_host_key.argtypes = [u64, u64]
        lib.syn_host_key.restype = u64
        lib.syn_host_fill_normal_bf16.argtypes = [u64, u64, dbl, vp, i64, i64]
        lib.syn_host_fill_normal_f64.argtypes = [u64, u64, vp, i64, i64]
        lib.syn_host_fill_uniform_int.argtypes = [u64, u64, ctypes.c_uint32, vp, i64, i64]
        lib.syn_host_permutation.argtypes = [u64, u64, vp, i64]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"{DEV_LIB} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_LIB)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.syn_dev_fill_normal_bf16.argtypes = [u64, u64, dbl, vp, i64, i64, vp]
        lib.syn_dev_fill_normal_bf16.restype = ctypes.c_int
        lib.syn_dev_fill_const_bf16.argtypes = [ctypes.c_uint16, vp, i64, vp]
        lib.syn_dev_fill_const_bf16.restype = ctypes.c_int
        _dev = lib
    return _dev


# ----------------------------------------------------------------------- generator


def normal_bf16(seed: int, tid: int, sigma: float, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _host_lib().syn_host_fill_normal_bf16(seed, tid, sigma, out.ctypes.data, n, offset)
    return out


def normal_f64(seed: int, tid: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _host_lib().syn_host_fill_normal_f64(seed, tid, out.ctypes.data, n, offset)
    return out


def uniform_int(seed: int, tid: int, m: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _host_lib().syn_host_fill_uniform_int(seed, tid, m, out.ctypes.data, n, offset)
    return out


def permutation(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _host_lib().syn_host_permutation(seed, tid, out.ctypes.data, n)
    return out


def fill_normal_bf16_device(seed: int, tid: int, sigma: float, ptr: int, n: int,
                            offset: int = 0, stream: int = 0) -> None:
    rc = _dev_lib().syn_dev_fill_normal_bf16(seed, tid, sigma, ptr, n, offset, stream)
    if rc != 0:
        raise RuntimeError(f"syn_dev_fill_normal_bf16 failed: cuda error {rc}")


def fill_const_bf16_device(bits: int, ptr: int, n: int, stream: int = 0) -> None:
    rc = _dev_lib().syn_dev_fill_const_bf16(bits, ptr, n, stream)
    if rc != 0:
        raise RuntimeError(f"syn_dev_fill_const_bf16 failed: cuda error {rc}")


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ tensor identity

K_EMBED, K_LM_HEAD, K_FINAL_NORM = 1, 2, 3
K_WQ, K_WK, K_WV, K_WO, K_WR, K_WG, K_WU, K_WD, K_NORM = 16, 17, 18, 19, 20, 21, 22, 23, 24
K_KPOOL, K_VPOOL = 32, 33
K_TOKENS, K_PAGEPERM, K_ZIPF, K_CTX, K_BUDGET = 48, 49, 50, 51, 52


def tensor_id(kind: int, layer: int = -1, gen: int = 0) -> int:
    """64-bit tensor id: generation (for refreshed KV), layer + 1, kind."""
    return (gen << 40) | ((layer + 1) << 16) | kind


# ------------------------------------------------------------------------ workloads


@dataclass(frozen=True)
class Dims:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    d_ffn: int
    vocab: int
    page_size: int = 16
    rope_base: float = 10000.0
    rms_eps: float = 1e-6


TINY = Dims(2, 256, 4, 2, 64, 8, 2, 256, 1024)
MID = Dims(8, 1024, 16, 4, 64, 32, 4, 512, 32000)
FULL = Dims(48, 2048, 32, 4, 128, 128, 8, 768, 152064)


@dataclass
class Workload:
    name: str
    dims: Dims
    batch: int
    seq_lens: List[int]
    steps: int
    zipf_s: Optional[float] = None
    seed: int = 0
    note: str = ""


def ragged_lens(seed: int, batch: int, lo: int, hi: int, gen: int = 0) -> List[int]:
    u = uniform_int(seed, tensor_id(K_CTX, gen=gen), hi - lo + 1, batch)
    return [int(lo + x) for x in u]


def replacement_events(seed: int, batch: int, steps: int, lo: int = 16,
                       hi: int = 128) -> List[Tuple[int, int]]:
    """Continuous batching: every slot's sequence gets a generation budget
    ~U[lo, hi] (seeded per slot and generation); when it is spent the slot
    takes a fresh sequence.  Returns the (step, slot) replacements within
    `steps` steps, in order (step k: before the k-th step)."""
    ev = []
    for b in range(batch):
        t, g = 0, 0
        while True:
            t += lo + int(uniform_int(seed, tensor_id(K_BUDGET, layer=b, gen=g), hi - lo + 1, 1)[0])
            if t >= steps:
                break
            ev.append((t, b))
            g += 1
    return sorted(ev)


def workloads() -> Dict[str, Workload]:
    """The five workloads: tiny, mid, full-scale (B=1 at 8K), full-scale B=8
    ragged with Zipf router skew, and long context."""
    return {
        "tiny": Workload("tiny", TINY, 1, [64], 9,
                         note="2 layers, d 256, 8 experts top-2; 1 step + 8 greedy"),
        "mid": Workload("mid", MID, 1, [2048], 128),
        "full": Workload("full", FULL, 1, [8192], 256),
        "full_b8": Workload("full_b8", FULL, 8, ragged_lens(0, 8, 1024, 16384), 256,
                            zipf_s=1.1),
        "long_b1": Workload("long_b1", FULL, 1, [262144], 64),
        "long_b2": Workload("long_b2", FULL, 2, [131072, 131072], 64),
    }


# ----------------------------------------------------------------- tensor catalogue


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    tid: int
    sigma: float = 0.02
    const_bits: Optional[int] = None  # set: every element equals these bf16 bits

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape))


def weight_specs(dims: Dims) -> Dict[str, TensorSpec]:
    """Every weight tensor of the model, in the library's layouts:
    W[out][in] row-major (K-contiguous), experts [E][F][d] / [E][d][F]."""
    d, D, Hq, Hkv = dims.d_model, dims.head_dim, dims.n_q_heads, dims.n_kv_heads
    E, F, V = dims.n_experts, dims.d_ffn, dims.vocab
    s: Dict[str, TensorSpec] = {}
    s["embed"] = TensorSpec("embed", (V, d), tensor_id(K_EMBED))
    s["lm_head"] = TensorSpec("lm_head", (V, d), tensor_id(K_LM_HEAD))
    s["final_norm"] = TensorSpec("final_norm", (d,), tensor_id(K_FINAL_NORM), const_bits=BF16_ONE)
    for l in range(dims.n_layers):
        p = f"l{l}."
        s[p + "norm"] = TensorSpec(p + "norm", (d,), tensor_id(K_NORM, l), const_bits=BF16_ONE)
        s[p + "wq"] = TensorSpec(p + "wq", (Hq * D, d), tensor_id(K_WQ, l))
        s[p + "wk"] = TensorSpec(p + "wk", (Hkv * D, d), tensor_id(K_WK, l))
        s[p + "wv"] = TensorSpec(p + "wv", (Hkv * D, d), tensor_id(K_WV, l))
        s[p + "wo"] = TensorSpec(p + "wo", (d, Hq * D), tensor_id(K_WO, l))
        s[p + "wr"] = TensorSpec(p + "wr", (E, d), tensor_id(K_WR, l))
        s[p + "wg"] = TensorSpec(p + "wg", (E, F, d), tensor_id(K_WG, l))
        s[p + "wu"] = TensorSpec(p + "wu", (E, F, d), tensor_id(K_WU, l))
        s[p + "wd"] = TensorSpec(p + "wd", (E, d, F), tensor_id(K_WD, l))
    return s


def kv_specs(dims: Dims, num_pages: int, gen: int = 0) -> Dict[str, TensorSpec]:
    """Per-layer K and V pools [num_pages][Hkv][P][D], bf16 ~ N(0, 1)."""
    shape = (num_pages, dims.n_kv_heads, dims.page_size, dims.head_dim)
    s = {}
    for l in range(dims.n_layers):
        s[f"l{l}.kpool"] = TensorSpec(f"l{l}.kpool", shape, tensor_id(K_KPOOL, l, gen), 1.0)
        s[f"l{l}.vpool"] = TensorSpec(f"l{l}.vpool", shape, tensor_id(K_VPOOL, l, gen), 1.0)
    return s


def router_bias(dims: Dims, layer: int, zipf_s: Optional[float], seed: int = 0):
    """Zipf(s) router skew, read as a per-expert fp32 logit bias
    b_e = -s * ln(rank_e), rank a seeded per-layer permutation of 1..E.
    Returns None when there is no skew."""
    if zipf_s is None:
        return None
    rank = permutation(seed, tensor_id(K_ZIPF, layer), dims.n_experts) + 1
    return (-zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)


def host_tensor(spec: TensorSpec, seed: int = 0) -> np.ndarray:
    """The tensor's bf16 bits on the host, shape spec.shape."""
    if spec.const_bits is not None:
        return np.full(spec.shape, spec.const_bits, dtype=np.uint16)
    return normal_bf16(seed, spec.tid, spec.sigma, spec.numel).reshape(spec.shape)


def device_tensor(spec: TensorSpec, seed: int = 0, device="cuda"):
    """The same tensor generated directly in device memory (torch bf16)."""
    import torch

    t = torch.empty(spec.shape, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(t.device).cuda_stream
    if spec.const_bits is not None:
        fill_const_bf16_device(spec.const_bits, t.data_ptr(), spec.numel, stream)
    else:
        fill_normal_bf16_device(seed, spec.tid, spec.sigma, t.data_ptr(), spec.numel, 0, stream)
    return t


# ---------------------------------------------------------------- paging and tokens


@dataclass
class PageLayout:
    num_pages: int
    max_pages: int
    page_tables: np.ndarray  # int32 [B][max_pages], -1 = unallocated


def page_layout(dims: Dims, seq_lens: Sequence[int], reserve_steps: int, seed: int = 0,
                gen: int = 0, shuffle: bool = True) -> PageLayout:
    """Pages for positions 0 .. L_b + reserve_steps - 1 of every sequence, drawn
    from a seeded permutation of the pool (identity order if not shuffle)."""
    P = dims.page_size
    need = [max(1, -(-(L + reserve_steps) // P)) for L in seq_lens]
    total = int(sum(need))
    order = (permutation(seed, tensor_id(K_PAGEPERM, gen=gen), total) if shuffle
             else np.arange(total, dtype=np.int32))
    maxp = max(need)
    pt = np.full((len(seq_lens), maxp), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        pt[b, :n] = order[at:at + n]
        at += n
    return PageLayout(total, maxp, pt)


def first_tokens(dims: Dims, batch: int, seed: int = 0, gen: int = 0) -> np.ndarray:
    return uniform_int(seed, tensor_id(K_TOKENS, gen=gen), dims.vocab, batch)


def weight_bytes_total(dims: Dims) -> int:
    return sum(s.numel * 2 for s in weight_specs(dims).values())


def fmt_bytes(n: float) -> str:
    for unit in ("B", "KB", "MB", "GB", "TB"):
        if abs(n) < 1000:
            return f"{n:.1f} {unit}"
        n /= 1000.0
    return f"{n:.1f} PB"


# ------------------------------------------------------------- device-side inputs


@dataclass
class DeviceInputs:
    """Every input of a workload, generated in device memory."""
    dims: Dims
    tensors: Dict[str, object]      # name -> torch bf16 tensor (weights and KV pools)
    layout: PageLayout
    biases: List[Optional[np.ndarray]]
    bias_tensors: List[object]      # torch fp32 [E] or None per layer
    seed: int


def device_inputs(dims: Dims, seq_lens: Sequence[int], reserve_steps: int,
                  zipf_s: Optional[float] = None, seed: int = 0, gen: int = 0,
                  shuffle: bool = True, device="cuda", weights=None) -> DeviceInputs:
    """Weights, KV pools (laid out for seq_lens plus reserve_steps tokens)
    and router biases on the device.  weights: the weight tensors of an
    earlier DeviceInputs of the same dims and seed, reused as they are."""
    import torch

    layout = page_layout(dims, seq_lens, reserve_steps, seed, gen, shuffle)
    specs = {} if weights is not None else dict(weight_specs(dims))
    specs.update(kv_specs(dims, layout.num_pages, gen))
    tensors = {n: device_tensor(s, seed, device) for n, s in specs.items()}
    if weights is not None:
        tensors.update({n: weights[n] for n in weight_specs(dims)})
    biases = [router_bias(dims, l, zipf_s, seed) for l in range(dims.n_layers)]
    bias_t = [None if b is None else torch.from_numpy(b).to(device) for b in biases]
    return DeviceInputs(dims, tensors, layout, biases, bias_t, seed)


def host_inputs(dims: Dims, layout: PageLayout, seed: int = 0, gen: int = 0,
                materialise: bool = True) -> Dict[str, object]:
    """The same inputs for the oracle: host arrays, or (materialise=False)
    the TensorSpecs from which the oracle regenerates every value."""
    specs = dict(weight_specs(dims))
    specs.update(kv_specs(dims, layout.num_pages, gen))
    if not materialise:
        return specs
    return {n: host_tensor(s, seed) for n, s in specs.items()}


__all__ = [n for n in dir() if not n.startswith("_")]
