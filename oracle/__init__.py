"""Oracle for paged GQA attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls anything here, and nothing here imports the CUDA library: the two share only
the seeded input generator (``paged_kv_attention_gqa_gb300.workloads``), which holds
no attention arithmetic.

Contents
  ref_attn.c   plain single-threaded fp32 C: gather pages, textbook softmax
               attention + LSE, last-page append, dense varlen attention over
               contiguous K/V runs (see its header for the definitions and the page
               passages they follow).
  plan_ref.py  the index work in plain Python: append slots, visible ranges, the
               mixed-step classification, permutation and sink routing.

Pins (tests/test_oracle_pins.py): hand-worked 2-token examples stored under
tests/golden/, torch's scaled_dot_product_attention in float64 on unpaged K/V,
invariance under page-pool permutation and page_size 1 vs 16, an all-ones V
channel (softmax rows sum to 1), the window_left = 0 / single-key special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_attn.c")
_SO = os.path.join(_HERE, "_ref_attn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ref_attn.c with gcc into oracle/_ref_attn.so (plain -O2, no fast-math,
    no FMA contraction, so x86 and Arm hosts round identically)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def load(path: str | None = None):
    """Open the oracle's shared object (``path`` lets the mutation tests open a
    deliberately broken copy); the default one is built on first use."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        if path is None:
            build()
        lib = ctypes.CDLL(path or _SO)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_attention.argtypes = [p, p, ctypes.c_int64, p, p, p, p, i, i, i, i, i,
                                         i, i, ctypes.c_float, p, p, p]
        lib.oracle_attention.restype = i
        lib.oracle_kv_append.argtypes = [p, ctypes.c_int64, p, p, p, p, p, p, i, i, i, i]
        lib.oracle_kv_append.restype = i
        lib.oracle_dense_attention.argtypes = [p, p, p, p, p, i, i, i, i, i, i, ctypes.c_float, p, p]
        lib.oracle_dense_attention.restype = i
        if path is None:
            _lib = lib
    return lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16, "bf16 data is passed as its uint16 bit pattern"
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q_bits, kv_layer_bits, qo_indptr, kv_indptr, kv_indices, last_page_len, *,
              num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
              causal: bool = True, window_left: int = -1, sm_scale: float | None = None,
              rows=None, threads: int = 1, lib=None):
    """Ragged paged attention over one layer slice.

    q_bits        uint16 [T, num_qo_heads, head_dim]   (bf16 bit patterns)
    kv_layer_bits uint16 [max_pages, 2, page_size, num_kv_heads, head_dim]
    rows          optional iterable of row ids to compute (others stay NaN)
    threads       rows are split over this many Python threads; each calls the
                  single-threaded C routine on its own rows (ctypes drops the GIL).
    Returns (out float32 [T, Hq, D], lse float32 [T, Hq]).
    """
    lib = lib or load()
    q_bits = _u16(q_bits)
    kv = _u16(kv_layer_bits)
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    batch = len(kvp) - 1
    T = int(qo[-1])
    max_pages = kv.shape[0]
    assert kv.shape[1:] == (2, page_size, num_kv_heads, head_dim), kv.shape
    assert q_bits.shape == (T, num_qo_heads, head_dim), q_bits.shape
    if sm_scale is None:
        sm_scale = 1.0 / float(np.sqrt(head_dim))
    out = np.full((T, num_qo_heads, head_dim), np.nan, dtype=np.float32)
    lse = np.full((T, num_qo_heads), np.nan, dtype=np.float32)
    row_list = list(range(batch)) if rows is None else [int(r) for r in rows]
    threads = max(1, min(int(threads), len(row_list) or 1))
    chunks = [row_list[k::threads] for k in range(threads)]
    errors = []

    def work(chunk):
        mask = np.zeros(batch, dtype=np.uint8)
        mask[chunk] = 1
        rc = lib.oracle_attention(_ptr(q_bits), _ptr(kv), max_pages, _ptr(qo), _ptr(kvp), _ptr(kvi),
                                  _ptr(lpl), batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                                  int(causal if causal == 2 else bool(causal)), int(window_left), float(sm_scale),
                                  _ptr(mask),
                                  _ptr(out), _ptr(lse))
        if rc != 0:
            errors.append(rc)

    if threads == 1:
        work(chunks[0])
    else:
        ts = [threading.Thread(target=work, args=(c,)) for c in chunks]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    if errors:
        raise ValueError(f"oracle_attention rejected its input (code {errors[0]})")
    return out, lse


def kv_append(kv_layer_bits, k_new_bits, v_new_bits, qo_indptr, kv_indptr, kv_indices,
              last_page_len, *, num_kv_heads: int, head_dim: int, page_size: int, lib=None):
    """Return a copy of the layer slice with this step's new K/V stored in place."""
    lib = lib or load()
    kv = np.array(_u16(kv_layer_bits), copy=True)
    k = _u16(k_new_bits)
    v = _u16(v_new_bits)
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    rc = lib.oracle_kv_append(_ptr(kv), kv.shape[0], _ptr(k), _ptr(v), _ptr(qo), _ptr(kvp), _ptr(kvi),
                              _ptr(lpl), len(kvp) - 1, num_kv_heads, head_dim, page_size)
    if rc != 0:
        raise ValueError(f"oracle_kv_append rejected its input (code {rc})")
    return kv


def dense_attention(q_bits, k_bits, v_bits, cu_q, cu_k, *, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                    causal: bool = True, window_left: int = -1, sm_scale: float | None = None, lib=None):
    """Dense varlen attention over contiguous per-segment K/V runs (DenseAttentionManager).
    q_bits [Tq, Hq, D], k_bits / v_bits [Tk, Hkv, D] uint16; returns (out, lse) float32."""
    lib = lib or load()
    q, k, v = _u16(q_bits), _u16(k_bits), _u16(v_bits)
    cq, ck = _i32(cu_q), _i32(cu_k)
    if sm_scale is None:
        sm_scale = 1.0 / float(np.sqrt(head_dim))
    T = int(cq[-1])
    out = np.full((T, num_qo_heads, head_dim), np.nan, dtype=np.float32)
    lse = np.full((T, num_qo_heads), np.nan, dtype=np.float32)
    rc = lib.oracle_dense_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck), len(cq) - 1, num_qo_heads,
                                    num_kv_heads, head_dim, int(bool(causal)), int(window_left), float(sm_scale),
                                    _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_dense_attention rejected its input (code {rc})")
    return out, lse
