"""Python handle on the fp64 CPU oracle (pa_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline
leg may call this; the product path never does.  It shares no code with the CUDA
library.  The oracle is built with the host C compiler into oracle/_build/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_E4M3, KV_BF16 = 0, 1
SCALE_NONE, SCALE_SCALAR, SCALE_PER_TOKEN = 0, 1, 2


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("group_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32), ("num_pages", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("k_scale_scalar", ctypes.c_double), ("v_scale_scalar", ctypes.c_double),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int32),
        ("context_lens", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("selected", ctypes.c_void_p), ("sel_stride", ctypes.c_int32),
        ("num_selected", ctypes.c_void_p), ("sm_scale", ctypes.c_double),
    ]


class _IndexProblem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("index_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int32),
        ("context_lens", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("sm_scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile pa_oracle.c (plain C, -O2, pthreads) if it is missing or stale."""
    with _lock:
        os.makedirs(_BUILD, exist_ok=True)
        if force or not os.path.exists(_LIB_PATH) or \
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-pthread", "-shared",
                                   "-fPIC", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """One loaded build of the oracle (the default one, or a test's mutated copy)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_decode.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_dec_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_dec_e4m3.restype = ctypes.c_double
        lib.oracle_dec_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_dec_bf16.restype = ctypes.c_double
        lib.oracle_key_positions.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_key_positions.restype = ctypes.c_int64
        lib.oracle_enc_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_enc_e4m3.restype = ctypes.c_uint8
        lib.oracle_kv_quantize_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_kv_quantize_write.restype = ctypes.c_int64
        lib.oracle_lse_merge.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_void_p]
        lib.oracle_lse_merge.restype = None
        lib.oracle_index_topk.argtypes = [ctypes.POINTER(_IndexProblem), ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        lib.oracle_index_topk.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def decode(self, p, threads: int | None = None):
        """fp64 attention output [rows, Hq, D] and natural-log LSE [rows, Hq]."""
        keep = []
        st = _problem(p, keep)
        rows = int(p.cu_seqlens_q[-1])
        Hq = p.num_kv_heads * p.group_size
        out = np.zeros((rows, Hq, p.head_dim), dtype=np.float64)
        lse = np.zeros((rows, Hq), dtype=np.float64)
        n = threads if threads is not None else (os.cpu_count() or 1)
        rc = self.lib.oracle_decode(ctypes.byref(st), out.ctypes.data, lse.ctypes.data, int(n))
        if rc != 0:
            raise RuntimeError("oracle_decode failed")
        return out, lse

    def key_positions(self, p, r: int, tok: int) -> np.ndarray:
        """Attended positions of (request r, query token tok) in key-set order."""
        keep = []
        st = _problem(p, keep)
        cap = int(p.context_lens[r])
        if p.selected is not None:
            cap = max(cap, int(p.num_selected[r]) * p.page_size)
        buf = np.zeros(max(cap, 1), dtype=np.int64)
        n = self.lib.oracle_key_positions(ctypes.byref(st), int(r), int(tok), buf.ctypes.data,
                                          buf.size)
        if n < 0:
            raise RuntimeError("key buffer too small")
        return buf[:n].copy()

    def dec_e4m3(self, code: int) -> float:
        return float(self.lib.oracle_dec_e4m3(int(code)))

    def dec_bf16(self, bits: int) -> float:
        return float(self.lib.oracle_dec_bf16(int(bits)))

    def enc_e4m3(self, x: float) -> int:
        return int(self.lib.oracle_enc_e4m3(float(x)))

    def index_topk(self, ip):
        """Indexer block scores and top-k pages of an index problem (synth.IndexProblem):
        (selected int32 [rows, topk], num_selected int32 [rows], scores fp64
        [rows, max pages], -inf where a page is not a candidate)."""
        R = int(ip.cu_seqlens_q[-1])
        stride = max(int(ip.block_table.shape[1]), 1)
        arrs = dict(q=np.ascontiguousarray(ip.q, dtype=np.uint16),
                    k=np.ascontiguousarray(ip.k_cache, dtype=np.uint8),
                    ks=None if ip.k_scale is None else np.ascontiguousarray(ip.k_scale, dtype=np.float32),
                    bt=np.ascontiguousarray(ip.block_table, dtype=np.int32),
                    L=np.ascontiguousarray(ip.context_lens, dtype=np.int32),
                    cu=np.ascontiguousarray(ip.cu_seqlens_q, dtype=np.int32))
        st = _IndexProblem(num_seqs=len(arrs["L"]), index_heads=ip.q.shape[1],
                           head_dim=ip.q.shape[2], page_size=ip.k_cache.shape[1],
                           topk=ip.topk, num_pages=ip.k_cache.shape[0],
                           q=arrs["q"].ctypes.data, k_cache=arrs["k"].ctypes.data,
                           k_scale=None if arrs["ks"] is None else arrs["ks"].ctypes.data,
                           block_table=arrs["bt"].ctypes.data, bt_stride=stride,
                           context_lens=arrs["L"].ctypes.data, cu_seqlens_q=arrs["cu"].ctypes.data,
                           sm_scale=float(ip.sm_scale))
        sel = np.zeros((R, max(ip.topk, 1)), dtype=np.int32)
        nsel = np.zeros(R, dtype=np.int32)
        scores = np.zeros((R, stride), dtype=np.float64)
        rc = self.lib.oracle_index_topk(ctypes.byref(st), sel.ctypes.data, nsel.ctypes.data,
                                        scores.ctypes.data, stride)
        if rc != 0:
            raise RuntimeError("oracle_index_topk failed")
        return sel[:, :ip.topk], nsel, scores

    def lse_merge(self, part_out, part_lse):
        """fp64 log-sum-exp merge of partials: part_out [P, rows, heads, D], part_lse
        [P, rows, heads] (natural log, -inf for an empty part) -> (out [rows, heads, D],
        lse [rows, heads])."""
        po = np.ascontiguousarray(part_out, dtype=np.float64)
        pl = np.ascontiguousarray(part_lse, dtype=np.float64)
        P, D = po.shape[0], po.shape[-1]
        nv = int(np.prod(po.shape[1:-1]))
        assert pl.shape == po.shape[:-1]
        out = np.zeros(po.shape[1:], dtype=np.float64)
        lse = np.zeros(pl.shape[1:], dtype=np.float64)
        self.lib.oracle_lse_merge(po.ctypes.data, pl.ctypes.data, int(P), nv, int(D),
                                  out.ctypes.data, lse.ctypes.data)
        return out, lse

    def kv_quantize_write(self, k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale):
        """Per-token e4m3 quantisation of new K/V rows (bf16 bit patterns [T, Hkv, D]) into
        the paged cache arrays, in place; returns the number of out-of-range slots."""
        T, Hkv, D = k_new.shape
        P, _, ps, _ = k_cache.shape
        for a, dt in ((k_new, np.uint16), (v_new, np.uint16), (k_cache, np.uint8),
                      (v_cache, np.uint8), (k_scale, np.float32), (v_scale, np.float32)):
            assert a.dtype == dt and a.flags.c_contiguous
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        return int(self.lib.oracle_kv_quantize_write(
            k_new.ctypes.data, v_new.ctypes.data, sm.ctypes.data, T, Hkv, D, ps, P,
            k_cache.ctypes.data, v_cache.ctypes.data, k_scale.ctypes.data, v_scale.ctypes.data))


def build_variant(source_text: str, out_path: str) -> str:
    """Compile a given oracle source text (used by the pin tests' mutation checks)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-w", "-pthread", "-shared", "-fPIC",
                           "-o", out_path, src, "-lm"])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def default() -> OracleLib:
    global _lib
    if _lib is None:
        _lib = OracleLib(build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _problem(p, keep):
    """Marshal a synth.Problem (or any object with the same fields) into the C struct."""
    def c(a, dt):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dt)
        keep.append(a)
        return a
    kv = KV_E4M3 if p.kv_dtype == "fp8" else KV_BF16
    sm = {"none": SCALE_NONE, "scalar": SCALE_SCALAR, "per_token": SCALE_PER_TOKEN}[p.scale_mode]
    cdt = np.uint8 if kv == KV_E4M3 else np.uint16
    st = _Problem()
    st.num_seqs, st.num_kv_heads = p.num_seqs, p.num_kv_heads
    st.group_size, st.head_dim, st.page_size = p.group_size, p.head_dim, p.page_size
    st.kv_dtype, st.scale_mode = kv, sm
    st.num_pages = p.k_cache.shape[0]
    st.q = _ptr(c(p.q, np.uint16))
    st.k_cache = _ptr(c(p.k_cache, cdt))
    st.v_cache = _ptr(c(p.v_cache, cdt))
    st.k_scale = _ptr(c(p.k_scale, np.float32)) if sm == SCALE_PER_TOKEN else None
    st.v_scale = _ptr(c(p.v_scale, np.float32)) if sm == SCALE_PER_TOKEN else None
    st.k_scale_scalar = float(p.k_scale_scalar)
    st.v_scale_scalar = float(p.v_scale_scalar)
    bt = c(p.block_table, np.int32)
    st.block_table, st.bt_stride = _ptr(bt), bt.shape[1]
    st.context_lens = _ptr(c(p.context_lens, np.int32))
    st.cu_seqlens_q = _ptr(c(p.cu_seqlens_q, np.int32))
    if p.selected is not None:
        sel = c(p.selected, np.int32)
        st.selected, st.sel_stride = _ptr(sel), sel.shape[1]
        st.num_selected = _ptr(c(p.num_selected, np.int32))
    else:
        st.selected, st.sel_stride, st.num_selected = None, 0, None
    st.sm_scale = float(p.sm_scale)
    return st


def decode(p, threads: int | None = None):
    return default().decode(p, threads)


def key_positions(p, r: int, tok: int) -> np.ndarray:
    return default().key_positions(p, r, tok)


def dec_e4m3(code: int) -> float:
    return default().dec_e4m3(code)


def dec_bf16(bits: int) -> float:
    return default().dec_bf16(bits)


def enc_e4m3(x: float) -> int:
    return default().enc_e4m3(x)


def index_topk(ip):
    return default().index_topk(ip)


def kv_quantize_write(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    return default().kv_quantize_write(k_new, v_new, slot_mapping, k_cache, v_cache,
                                       k_scale, v_scale)


def lse_merge(part_out, part_lse):
    return default().lse_merge(part_out, part_lse)


def row_map(cu_seqlens_q, context_lens):
    """(request, query token, causal cutoff) for every flat query row, from cu_seqlens_q."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    L = np.asarray(context_lens, dtype=np.int64)
    rows = int(cu[-1])
    out = np.zeros((rows, 3), dtype=np.int64)
    for r in range(len(L)):
        ql = cu[r + 1] - cu[r]
        for tok in range(ql):
            out[cu[r] + tok] = (r, tok, L[r] - ql + tok + 1)
    return out
