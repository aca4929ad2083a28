"""ctypes binding of libpkv (include/pkv.h).  Argument marshalling only: every step of
the attention path runs in the library's CUDA kernels.  torch tensors are passed as
device pointers; the stream is torch's current CUDA stream unless one is given.

``load()`` raises if libpkv.so has not been built; nothing here falls back to another
implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_TOO_MANY_PREFILL_ROWS, ERR_NOT_PLANNED, ERR_CUDA, ERR_DEVICE = range(8)
MODE_DECODE, MODE_PREFILL, MODE_MIXED, MODE_DENSE = 0, 1, 2, 3
NON_CAUSAL, CAUSAL, CONTEXT_ONLY = 0, 1, 2
STATUS_NAMES = ["OK", "INVALID", "UNSUPPORTED", "WORKSPACE", "TOO_MANY_PREFILL_ROWS", "NOT_PLANNED", "CUDA", "DEVICE"]

# every symbol include/pkv.h declares
EXPORTS = ["pkv_create", "pkv_destroy", "pkv_last_error", "pkv_workspace_size", "pkv_plan", "pkv_kv_append", "pkv_kv_append_planned",
           "pkv_run_decode", "pkv_run_prefill", "pkv_run_mixed", "pkv_check_device_error", "pkv_append_slots",
           "pkv_mixed_layout", "pkv_decode_split", "pkv_decode_head_rows", "pkv_run_decode_static", "pkv_context_only_views",
           "pkv_plan_dense", "pkv_run_dense", "pkv_gather_kv", "pkv_run_decode_append", "pkv_selftest_wait_timeout"]


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"pkv status {name}: {message}")


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_qo_heads", "num_kv_heads", "head_dim", "page_size", "max_batch", "max_total_tokens",
        "max_num_pages", "num_cache_pages", "max_prefill_rows", "sm_count", "sink_page", "graph_static",
        "enable_nvtx")]


_lib = None


def load(path: str = LIB_PATH):
    """Open libpkv.so (built by paged_kv_attention_gqa_gb300.build); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with `python -m paged_kv_attention_gqa_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i, i32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    sig = {
        "pkv_create": ([ctypes.POINTER(Config), ctypes.POINTER(vp)], i),
        "pkv_destroy": ([vp], None),
        "pkv_last_error": ([vp], ctypes.c_char_p),
        "pkv_workspace_size": ([vp, i, ctypes.POINTER(ctypes.c_size_t)], i),
        "pkv_plan": ([vp, i, i32p, i32p, i32p, i32p, i, i, i, ctypes.c_float, vp, ctypes.c_size_t, vp], i),
        "pkv_kv_append": ([vp, vp, vp, i, vp, vp, vp, vp, vp, i, vp], i),
        "pkv_kv_append_planned": ([vp, vp, vp, vp, vp, vp], i),
        "pkv_run_decode": ([vp, vp, vp, vp, vp, vp, vp], i),
        "pkv_run_decode_append": ([vp, vp, vp, vp, vp, vp, vp, vp, vp], i),
        "pkv_selftest_wait_timeout": ([vp, vp, i, vp], i),
        "pkv_run_prefill": ([vp, vp, vp, vp, vp, vp, vp], i),
        "pkv_run_mixed": ([vp, vp, vp, vp, vp, vp, vp], i),
        "pkv_check_device_error": ([vp, vp, vp, ctypes.POINTER(i)], i),
        "pkv_append_slots": ([i, i32p, i32p, i32p, i32p, i, i32p, i32p], i),
        "pkv_mixed_layout": ([i32p, i32p, i32p, i32p, i, i, i] + [i32p] * 9 + [ctypes.POINTER(i)], i),
        "pkv_decode_split": ([vp, i32p, i32p, i, i, i32p, ctypes.POINTER(i), ctypes.POINTER(i)], i),
        "pkv_decode_head_rows": ([vp, i32p, i32p, i32p, i, i, i32p, ctypes.POINTER(i)], i),
        "pkv_run_decode_static": ([vp, vp, vp, vp, vp, i32p, i32p, i32p, i, i, ctypes.c_float, vp], i),
        "pkv_context_only_views": ([i, i32p, i32p, i32p, i32p, i, i32p, i32p, i32p, ctypes.POINTER(i)], i),
        "pkv_plan_dense": ([vp, i32p, i32p, i, i, i, ctypes.c_float, vp, ctypes.c_size_t, vp], i),
        "pkv_run_dense": ([vp, vp, vp, vp, vp, vp, vp, vp], i),
        "pkv_gather_kv": ([vp, vp, vp, i, vp, vp, vp], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dptr(t):
    """Device pointer of a torch tensor (or None)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class Handle:
    """One pkv handle: static shape and the last plan (see include/pkv.h)."""

    def __init__(self, *, num_qo_heads, num_kv_heads, head_dim, page_size, max_batch, max_total_tokens=0,
                 max_num_pages, num_cache_pages, max_prefill_rows=0, sm_count=0, sink_page=-1, graph_static=0,
                 enable_nvtx=False):
        self.lib = load()
        self.cfg = Config(num_qo_heads, num_kv_heads, head_dim, page_size, max_batch, max_total_tokens,
                          max_num_pages, num_cache_pages, max_prefill_rows, sm_count, sink_page, int(graph_static),
                          int(enable_nvtx))
        h = ctypes.c_void_p()
        st = self.lib.pkv_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != OK:
            raise PkvError(st, self.lib.pkv_last_error(None).decode())
        self.h = h
        self._keep = []

    def close(self):
        if getattr(self, "h", None):
            self.lib.pkv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st):
        if st != OK:
            raise PkvError(st, self.lib.pkv_last_error(self.h).decode())

    def workspace_size(self, mode: int) -> int:
        n = ctypes.c_size_t()
        self._check(self.lib.pkv_workspace_size(self.h, mode, ctypes.byref(n)))
        return n.value

    def plan(self, mode, qo_indptr, kv_indptr, kv_indices, last_page_len, *, workspace, causal=True,
             window_left=-1, sm_scale=0.0, stream=None):
        arrs = [_i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)]
        batch = len(arrs[1]) - 1
        self._keep = arrs  # host arrays are read synchronously; kept only for symmetry
        st = self.lib.pkv_plan(self.h, mode, *(_p(a) for a in arrs), batch,
                               int(causal) if causal == CONTEXT_ONLY else int(bool(causal)), int(window_left),
                               float(sm_scale), _dptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
        self._check(st)

    def kv_append(self, k, v, num_new_tokens, kv_layer, qo_indptr, kv_indptr, kv_indices, last_page_len, batch,
                  stream=None):
        """pkv_kv_append: k / v, the layer slice and the four index arrays are device
        tensors (qo_indptr may be None: one new token per row)."""
        self._check(self.lib.pkv_kv_append(self.h, _dptr(k), _dptr(v), int(num_new_tokens), _dptr(kv_layer),
                                           _dptr(qo_indptr), _dptr(kv_indptr), _dptr(kv_indices),
                                           _dptr(last_page_len), int(batch), _stream(stream)))

    def kv_append_planned(self, k, v, kv_layer, *, workspace, stream=None):
        """pkv_kv_append_planned: at the write locations of the last plan on `workspace`."""
        self._check(self.lib.pkv_kv_append_planned(self.h, _dptr(k), _dptr(v), _dptr(kv_layer), _dptr(workspace),
                                                   _stream(stream)))

    def _run(self, fn, q, kv_layer, out, lse, workspace, stream):
        self._check(fn(self.h, _dptr(q), _dptr(kv_layer), _dptr(out), _dptr(lse), _dptr(workspace), _stream(stream)))

    def run_decode(self, q, kv_layer, out, lse=None, *, workspace, stream=None):
        self._run(self.lib.pkv_run_decode, q, kv_layer, out, lse, workspace, stream)

    def run_decode_append(self, q, k, v, kv_layer, out, lse=None, *, workspace, stream=None):
        """kv_append + run_decode in one launch (decode plans)."""
        self._check(self.lib.pkv_run_decode_append(self.h, _dptr(q), _dptr(k), _dptr(v), _dptr(kv_layer), _dptr(out),
                                                    _dptr(lse), _dptr(workspace), _stream(stream)))

    def run_prefill(self, q, kv_layer, out, lse=None, *, workspace, stream=None):
        self._run(self.lib.pkv_run_prefill, q, kv_layer, out, lse, workspace, stream)

    def run_mixed(self, q, kv_layer, out, lse=None, *, workspace, stream=None):
        self._run(self.lib.pkv_run_mixed, q, kv_layer, out, lse, workspace, stream)

    def plan_dense(self, cu_q, cu_k, *, workspace, causal=True, window_left=-1, sm_scale=0.0, stream=None):
        cq, ck = _i32(cu_q), _i32(cu_k)
        self._check(self.lib.pkv_plan_dense(self.h, _p(cq), _p(ck), len(cq) - 1, int(bool(causal)), int(window_left),
                                            float(sm_scale), _dptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream)))

    def run_dense(self, q, k, v, out, lse=None, *, workspace, stream=None):
        self._check(self.lib.pkv_run_dense(self.h, _dptr(q), _dptr(k), _dptr(v), _dptr(out), _dptr(lse),
                                           _dptr(workspace), _stream(stream)))

    def gather_kv(self, kv_layer, pages, num_tokens, k_out, v_out, stream=None):
        """pages: a device int32 tensor of page ids."""
        self._check(self.lib.pkv_gather_kv(self.h, _dptr(kv_layer), _dptr(pages), int(num_tokens), _dptr(k_out),
                                           _dptr(v_out), _stream(stream)))

    def selftest_wait_timeout(self, workspace, polls=1000, stream=None):
        """Make one device wait give up (see pkv.h); check_device_error then reports code 4."""
        self._check(self.lib.pkv_selftest_wait_timeout(self.h, _dptr(workspace), int(polls), _stream(stream)))

    def check_device_error(self, workspace, stream=None) -> int:
        code = ctypes.c_int()
        st = self.lib.pkv_check_device_error(self.h, _dptr(workspace), _stream(stream), ctypes.byref(code))
        if st not in (OK, ERR_DEVICE):
            self._check(st)
        return code.value

    def decode_split(self, kv_indptr, last_page_len, window_left=-1):
        kvp, lpl = _i32(kv_indptr), _i32(last_page_len)
        batch = len(kvp) - 1
        cap = batch + 16 * max(1, self.cfg.sm_count or 256) + 8  # up to 8 decode CTAs per SM
        tiles = np.zeros(5 * cap, np.int32)
        nt, nc = ctypes.c_int(cap), ctypes.c_int()
        self._check(self.lib.pkv_decode_split(self.h, _p(kvp), _p(lpl), batch, int(window_left), _p(tiles),
                                              ctypes.byref(nt), ctypes.byref(nc)))
        return tiles[: 5 * nt.value].reshape(-1, 5), nc.value

    def decode_head_rows(self, kv_indptr, kv_indices, last_page_len, window_left=-1):
        """Cache rows of each decode CTA's first 4 chunks ([CTAs, 4], -1 past its end)."""
        kvp, kvi, lpl = _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
        batch = len(kvp) - 1
        cap = batch + 16 * max(1, self.cfg.sm_count or 256) + 8  # up to 8 decode CTAs per SM
        rows = np.zeros(4 * cap, np.int32)
        nc = ctypes.c_int(cap)
        self._check(self.lib.pkv_decode_head_rows(self.h, _p(kvp), _p(kvi), _p(lpl), batch, int(window_left),
                                                  _p(rows), ctypes.byref(nc)))
        return rows[: 4 * nc.value].reshape(-1, 4)


def append_slots(page_size, qo_indptr, kv_indptr, kv_indices, last_page_len):
    lib = load()
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    T = int(qo[-1])
    pages, slots = np.zeros(T, np.int32), np.zeros(T, np.int32)
    st = lib.pkv_append_slots(page_size, _p(qo), _p(kvp), _p(kvi), _p(lpl), len(kvp) - 1, _p(pages), _p(slots))
    if st != OK:
        raise PkvError(st, "append_slots")
    return pages, slots


def context_only_views(page_size, qo_indptr, kv_indptr, kv_indices, last_page_len):
    lib = load()
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    B = len(kvp) - 1
    okvp, okvi, olpl = np.zeros(B + 1, np.int32), np.zeros(max(len(kvi), 1), np.int32), np.zeros(B, np.int32)
    nnz = ctypes.c_int()
    st = lib.pkv_context_only_views(page_size, _p(qo), _p(kvp), _p(kvi), _p(lpl), B, _p(okvp), _p(okvi), _p(olpl),
                                    ctypes.byref(nnz))
    if st != OK:
        raise PkvError(st, "context_only_views")
    return okvp, okvi[: nnz.value], olpl


def mixed_layout(qo_indptr, kv_indptr, kv_indices, last_page_len, *, max_prefill_rows, sink_page):
    lib = load()
    qo, kvp, kvi, lpl = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(last_page_len)
    B, T = len(kvp) - 1, int(qo[-1])
    out = dict(is_decode=np.zeros(B, np.int32), prompt_rows=np.zeros(max_prefill_rows, np.int32),
               perm=np.zeros(T, np.int32), pf_qo_indptr=np.zeros(max_prefill_rows + 1, np.int32),
               dec_kv_indptr=np.zeros(B + 1, np.int32), dec_kv_indices=np.zeros(len(kvi) + B, np.int32),
               dec_last_page_len=np.zeros(B, np.int32), dec_q_token=np.zeros(B, np.int32),
               dec_out_token=np.zeros(B, np.int32))
    nnz = ctypes.c_int()
    keys = ["is_decode", "prompt_rows", "perm", "pf_qo_indptr", "dec_kv_indptr", "dec_kv_indices",
            "dec_last_page_len", "dec_q_token", "dec_out_token"]
    st = lib.pkv_mixed_layout(_p(qo), _p(kvp), _p(kvi), _p(lpl), B, max_prefill_rows, sink_page,
                              *(_p(out[k]) for k in keys), ctypes.byref(nnz))
    if st != OK:
        raise PkvError(st, "mixed_layout")
    out["dec_kv_indices"] = out["dec_kv_indices"][: nnz.value]
    return out
