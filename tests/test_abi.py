"""The C ABI library loads and exports every function include/mk.h declares;
host-side argument checks that need no GPU (CPU)."""
import ctypes
import os
import re

import numpy as np

import persistent_moe_decode_sm_gb300 as mk
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(mk.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(mk.EXPORTS) <= set(names)


def test_status_strings():
    for code in range(12):
        assert mk.status_string(code) not in ("", "unknown status")
        assert code in mk.STATUS_NAMES
    assert mk.status_string(99) == "unknown status"


def full_dims(max_batch=8, num_pages=5000, max_pages=1040, **over):
    d = synth.FULL
    args = dict(n_layers=d.n_layers, d_model=d.d_model, n_q_heads=d.n_q_heads,
                n_kv_heads=d.n_kv_heads, head_dim=d.head_dim, n_experts=d.n_experts,
                top_k=d.top_k, d_ffn=d.d_ffn, vocab=d.vocab, page_size=16, max_batch=max_batch,
                num_pages=num_pages, max_pages_per_seq=max_pages)
    args.update(over)
    return mk.make_dims(**args)


def plan_rc(dims, n_sm=152, batch=1, lens=(8192,)):
    info = mk.mk_plan_info()
    sl = np.asarray(lens if len(lens) else [0], np.int32)
    return mk.lib().mk_plan(ctypes.byref(dims), n_sm, batch, sl.ctypes.data, ctypes.byref(info),
                            None, 0)


def test_plan_rejects_bad_arguments():
    assert plan_rc(full_dims()) == mk.MK_OK
    assert plan_rc(full_dims(head_dim=96)) == mk.MK_ERR_UNSUPPORTED
    assert plan_rc(full_dims(n_q_heads=30)) == mk.MK_ERR_INVALID_ARG      # 30 % 4
    assert plan_rc(full_dims(top_k=200)) == mk.MK_ERR_INVALID_ARG         # > E
    assert plan_rc(full_dims(d_model=2000)) == mk.MK_ERR_UNSUPPORTED      # not a multiple of 64
    assert plan_rc(full_dims(max_batch=9)) == mk.MK_ERR_BATCH
    assert plan_rc(full_dims(), batch=0, lens=()) == mk.MK_ERR_BATCH
    assert plan_rc(full_dims(max_batch=2), batch=3, lens=(1, 2, 3)) == mk.MK_ERR_BATCH
    assert plan_rc(full_dims(max_pages=512), lens=(8192,)) == mk.MK_ERR_PAGE_OOB  # no room for L+1
    assert plan_rc(full_dims(), lens=(-1,)) == mk.MK_ERR_PAGE_OOB
    assert plan_rc(full_dims(), n_sm=0) == mk.MK_ERR_INVALID_ARG


def test_create_rejects_null_and_misaligned_pointers_without_a_gpu():
    dims = full_dims()
    w = mk.Weights(0, [{}] * dims.n_layers, 0, 0)
    ctx = ctypes.c_void_p()
    assert mk.lib().mk_create(ctypes.byref(dims), ctypes.byref(w.c), None,
                              ctypes.byref(ctx)) == mk.MK_ERR_INVALID_ARG
    layer = {f[0]: 0x10000 for f in mk.mk_layer_ptrs._fields_}
    layer["router_bias"] = None
    layer["wq"] = 0x10008  # misaligned
    w = mk.Weights(0x10000, [layer] * dims.n_layers, 0x10000, 0x10000)
    assert mk.lib().mk_create(ctypes.byref(dims), ctypes.byref(w.c), None,
                              ctypes.byref(ctx)) == mk.MK_ERR_INVALID_ARG
    assert mk.lib().mk_create(ctypes.byref(full_dims(head_dim=48)), ctypes.byref(w.c), None,
                              ctypes.byref(ctx)) == mk.MK_ERR_UNSUPPORTED


def test_calls_on_null_context():
    L = mk.lib()
    assert L.mk_decode_step(None, None, None, None) == mk.MK_ERR_INVALID_ARG
    assert L.mk_build_schedule(None, 1, None, None) == mk.MK_ERR_INVALID_ARG
    assert L.mk_sync(None) == mk.MK_ERR_INVALID_ARG
    assert L.mk_set_wait_limit_ns(None, 5) == mk.MK_ERR_INVALID_ARG
    L.mk_destroy(None)
