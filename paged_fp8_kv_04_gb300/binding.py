"""Thin Python binding of libpagedfp8 (include/pa.h): argument marshalling only.

Every step of the attention runs in the library's CUDA kernels; this module checks
tensor dtypes and devices, passes data pointers and the current torch stream, and
raises on a non-OK status.  It fails loudly when the shared library is missing.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import numpy as np

from . import build as _build

KV_FP8_E4M3, KV_BF16 = 0, 1
SCALE_NONE, SCALE_SCALAR, SCALE_PER_TOKEN = 0, 1, 2
Q_UNIFORM, Q_RAGGED = 0, 1
OUT_BF16, OUT_F32 = 0, 1
PLAN_NO_PDL = 0x1
PLAN_TCGEN05 = 0x2

STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CAPACITY",
          4: "PA_ERR_RAGGED", 5: "PA_ERR_ALIGN", 6: "PA_ERR_CUDA", 7: "PA_ERR_DEVICE_DATA",
          8: "PA_ERR_WORKSPACE"}
DEV_FLAGS = {0x01: "BAD_PAGE", 0x02: "BAD_CONTEXT", 0x04: "BAD_QLEN", 0x08: "NOT_UNIFORM",
             0x10: "BAD_SELECTED", 0x20: "Q_RANGE", 0x40: "TIMEOUT", 0x80: "DUMP_RANGE"}


class PaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class PlanDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_kv_heads", "group_size", "head_dim", "page_size", "kv_dtype", "scale_mode",
        "q_mode", "q_len", "max_batch", "max_rows", "max_context_len", "max_selected_pages",
        "partition_tokens", "out_dtype", "num_sms", "flags")] + [("reserved", ctypes.c_int32 * 2)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("k_scale_scalar", ctypes.c_float), ("v_scale_scalar", ctypes.c_float),
        ("num_pages", ctypes.c_int64), ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
        ("context_lens", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_q_host", ctypes.c_void_p), ("selected_pages", ctypes.c_void_p),
        ("num_selected", ctypes.c_void_p), ("selected_stride", ctypes.c_int32),
        ("num_rows", ctypes.c_int32), ("sm_scale", ctypes.c_float),
        ("reserved0", ctypes.c_int32), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [("grid_ctas", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("threads_per_cta", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("partial_slots", ctypes.c_int64), ("kernel", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class KvWriteArgs(ctypes.Structure):
    _fields_ = [("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("slot_mapping", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("num_tokens", ctypes.c_int64), ("num_pages", ctypes.c_int64),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("reserved", ctypes.c_int32)]


DEV_BAD_SLOT = 0x100
DEV_BAD_INDEX_ROW = 0x200


class IndexArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
                ("cu_seqlens_q", ctypes.c_void_p), ("selected", ctypes.c_void_p),
                ("num_selected", ctypes.c_void_p), ("scores", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("num_seqs", ctypes.c_int32), ("num_rows", ctypes.c_int32),
                ("index_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("block_table_stride", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("reserved", ctypes.c_int32)]

class LseMergeArgs(ctypes.Structure):
    _fields_ = [("part_out", ctypes.c_void_p), ("part_lse", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("num_parts", ctypes.c_int32), ("num_rows", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None
P = ctypes.c_void_p


def header_functions() -> list:
    """Names of every function include/pa.h declares."""
    with open(os.path.join(_build.INCLUDE, "pa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def lib(path: Optional[str] = None):
    """Loads libpagedfp8.so (built in-tree by __graft_entry__.build()); raises if missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libpagedfp8.so is not built ({p}); run __graft_entry__.build()")
    L = ctypes.CDLL(p)
    L.pa_plan_validate.argtypes = [ctypes.POINTER(PlanDesc)]
    L.pa_plan_validate.restype = ctypes.c_int
    L.pa_plan_workspace_size.argtypes = [ctypes.POINTER(PlanDesc)]
    L.pa_plan_workspace_size.restype = ctypes.c_size_t
    L.pa_plan_create.argtypes = [ctypes.POINTER(PlanDesc), P, ctypes.c_size_t, ctypes.POINTER(P)]
    L.pa_plan_create.restype = ctypes.c_int
    L.pa_decode_check.argtypes = [P, ctypes.POINTER(DecodeArgs)]
    L.pa_decode_check.restype = ctypes.c_int
    L.pa_decode.argtypes = [P, ctypes.POINTER(DecodeArgs), P]
    L.pa_decode.restype = ctypes.c_int
    L.pa_plan_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    L.pa_plan_get_device_status.restype = ctypes.c_int
    L.pa_plan_get_info.argtypes = [P, ctypes.POINTER(PlanInfo)]
    L.pa_plan_get_info.restype = ctypes.c_int
    L.pa_plan_destroy.argtypes = [P]
    L.pa_plan_destroy.restype = None
    L.pa_status_string.argtypes = [ctypes.c_int]
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_debug_row_map.argtypes = [P, ctypes.POINTER(DecodeArgs), P, P]
    L.pa_debug_row_map.restype = ctypes.c_int
    L.pa_debug_gather_tile_bytes.argtypes = [P]
    L.pa_debug_gather_tile_bytes.restype = ctypes.c_size_t
    L.pa_debug_gather.argtypes = [P, ctypes.POINTER(DecodeArgs), P, ctypes.c_size_t, P]
    L.pa_debug_gather.restype = ctypes.c_int
    L.pa_decode_noalloc.argtypes = [ctypes.POINTER(PlanDesc), ctypes.POINTER(DecodeArgs), P]
    L.pa_decode_noalloc.restype = ctypes.c_int
    L.pa_kv_quantize_write.argtypes = [ctypes.POINTER(KvWriteArgs), P]
    L.pa_kv_quantize_write.restype = ctypes.c_int
    L.pa_index_topk.argtypes = [ctypes.POINTER(IndexArgs), P]
    L.pa_index_topk.restype = ctypes.c_int
    L.pa_lse_merge.argtypes = [ctypes.POINTER(LseMergeArgs), P]
    L.pa_lse_merge.restype = ctypes.c_int
    L.pa_debug_trace.argtypes = [P, ctypes.c_size_t]
    L.pa_debug_trace.restype = ctypes.c_int
    if path is None:
        _lib = L
    return L


def make_desc(*, num_kv_heads=1, group_size=16, head_dim=128, page_size=128, kv_dtype="fp8",
              scale_mode="per_token", q_mode="uniform", q_len=1, max_batch=1, max_rows=None,
              max_context_len=1, max_selected_pages=0, partition_tokens=0, out_dtype="bf16",
              num_sms=0, pdl=True, tcgen05=False) -> PlanDesc:
    d = PlanDesc()
    d.num_kv_heads, d.group_size, d.head_dim, d.page_size = num_kv_heads, group_size, head_dim, page_size
    d.kv_dtype = {"fp8": KV_FP8_E4M3, "bf16": KV_BF16}[kv_dtype] if isinstance(kv_dtype, str) else kv_dtype
    d.scale_mode = ({"none": SCALE_NONE, "scalar": SCALE_SCALAR, "per_token": SCALE_PER_TOKEN}[scale_mode]
                    if isinstance(scale_mode, str) else scale_mode)
    d.q_mode = {"uniform": Q_UNIFORM, "ragged": Q_RAGGED}[q_mode] if isinstance(q_mode, str) else q_mode
    d.q_len, d.max_batch = q_len, max_batch
    d.max_rows = max_rows if max_rows is not None else max_batch * q_len
    d.max_context_len, d.max_selected_pages = max_context_len, max_selected_pages
    d.partition_tokens = partition_tokens
    d.out_dtype = {"bf16": OUT_BF16, "f32": OUT_F32}[out_dtype] if isinstance(out_dtype, str) else out_dtype
    d.num_sms = num_sms
    d.flags = (0 if pdl else PLAN_NO_PDL) | (PLAN_TCGEN05 if tcgen05 else 0)
    return d


def _ptr(t):
    return None if t is None else t.data_ptr()


class Plan:
    """A plan over a capacity bucket, owning its device workspace (a torch uint8 tensor)."""

    def __init__(self, device=None, check_only: bool = False, **desc_kw):
        import torch
        self._lib = lib()
        self.desc = make_desc(**desc_kw)
        self.kv_dtype = desc_kw.get("kv_dtype", "fp8")
        self.scale_mode = desc_kw.get("scale_mode", "per_token")
        self.out_dtype = desc_kw.get("out_dtype", "bf16")
        self._plan = P()
        self.workspace = None
        if check_only:
            st = self._lib.pa_plan_create(ctypes.byref(self.desc), None, 0, ctypes.byref(self._plan))
        else:
            self.device = torch.device(device if device is not None else "cuda")
            nbytes = self._lib.pa_plan_workspace_size(ctypes.byref(self.desc))
            if nbytes == 0:
                raise PaError(self._lib.pa_plan_validate(ctypes.byref(self.desc)) or 2,
                              "pa_plan_workspace_size")
            with torch.cuda.device(self.device):
                self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
                st = self._lib.pa_plan_create(ctypes.byref(self.desc), self.workspace.data_ptr(),
                                              nbytes, ctypes.byref(self._plan))
        if st != 0:
            raise PaError(st, "pa_plan_create")

    def __del__(self):
        try:
            if getattr(self, "_plan", None):
                self._lib.pa_plan_destroy(self._plan)
                self._plan = P()
        except Exception:
            pass

    def info(self) -> dict:
        inf = PlanInfo()
        st = self._lib.pa_plan_get_info(self._plan, ctypes.byref(inf))
        if st != 0:
            raise PaError(st, "pa_plan_get_info")
        return {n: getattr(inf, n) for n, _ in PlanInfo._fields_}

    # ------------------------------------------------------------------ argument building
    def args(self, q, k_cache, v_cache, block_table, context_lens, *, k_scale=None, v_scale=None,
             k_scale_scalar=1.0, v_scale_scalar=1.0, cu_seqlens_q=None, cu_seqlens_q_host=None,
             selected_pages=None, num_selected=None, sm_scale=None, out=None, lse=None,
             num_pages=None, keep=None):
        a = DecodeArgs()
        a.q, a.k_cache, a.v_cache = _ptr(q), _ptr(k_cache), _ptr(v_cache)
        a.k_scale, a.v_scale = _ptr(k_scale), _ptr(v_scale)
        a.k_scale_scalar, a.v_scale_scalar = float(k_scale_scalar), float(v_scale_scalar)
        a.num_pages = int(num_pages if num_pages is not None else k_cache.shape[0])
        a.block_table = _ptr(block_table)
        a.block_table_stride = int(block_table.shape[1]) if block_table is not None else 0
        a.num_seqs = int(context_lens.shape[0]) if context_lens is not None else 0
        a.context_lens = _ptr(context_lens)
        a.cu_seqlens_q = _ptr(cu_seqlens_q)
        if cu_seqlens_q_host is not None:
            h = np.ascontiguousarray(cu_seqlens_q_host, dtype=np.int32)
            if keep is not None:
                keep.append(h)
            a.cu_seqlens_q_host = h.ctypes.data
        a.selected_pages = _ptr(selected_pages)
        a.selected_stride = int(selected_pages.shape[1]) if selected_pages is not None else 0
        a.num_selected = _ptr(num_selected)
        a.num_rows = int(q.shape[0]) if q is not None else 0
        hd = self.desc.head_dim
        a.sm_scale = float(sm_scale if sm_scale is not None else 1.0 / np.sqrt(hd))
        a.out = _ptr(out)
        a.lse = _ptr(lse)
        return a

    def check(self, a: DecodeArgs) -> int:
        return self._lib.pa_decode_check(self._plan, ctypes.byref(a))

    def _stream(self, stream):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return ctypes.c_void_p(s.cuda_stream)

    def decode(self, q, k_cache, v_cache, block_table, context_lens, *, out=None, lse=None,
               stream=None, **kw):
        """Enqueues one decode; returns `out` ([rows, Hq, D], bf16 or fp32 per the plan)."""
        import torch
        if out is None:
            dt = torch.float32 if self.out_dtype == "f32" else torch.bfloat16
            out = torch.empty(q.shape, dtype=dt, device=q.device)
        keep = []
        a = self.args(q, k_cache, v_cache, block_table, context_lens, out=out, lse=lse,
                      keep=keep, **kw)
        st = self._lib.pa_decode(self._plan, ctypes.byref(a), self._stream(stream))
        if st != 0:
            raise PaError(st, "pa_decode")
        return out

    def decode_args(self, a: DecodeArgs, stream=None) -> None:
        """Enqueues a decode from prepared arguments (for timing loops and graph capture)."""
        st = self._lib.pa_decode(self._plan, ctypes.byref(a), self._stream(stream))
        if st != 0:
            raise PaError(st, "pa_decode")

    def device_status(self, clear: bool = True) -> int:
        v = ctypes.c_uint32(0)
        st = self._lib.pa_plan_get_device_status(self._plan, ctypes.byref(v), int(clear))
        if st != 0:
            raise PaError(st, "pa_plan_get_device_status")
        return int(v.value)

    def _scratch_out(self, q, kw):
        import torch
        out = kw.pop("out", None)
        if out is None:
            dt = torch.float32 if self.out_dtype == "f32" else torch.bfloat16
            out = torch.empty(q.shape, dtype=dt, device=q.device)
        return out

    def row_map(self, q, k_cache, v_cache, block_table, context_lens, **kw):
        import torch
        keep = []
        a = self.args(q, k_cache, v_cache, block_table, context_lens, keep=keep,
                      out=self._scratch_out(q, kw), **kw)
        rm = torch.full((a.num_rows, 3), -1, dtype=torch.int32, device=q.device)
        st = self._lib.pa_debug_row_map(self._plan, ctypes.byref(a), rm.data_ptr(),
                                        self._stream(None))
        if st != 0:
            raise PaError(st, "pa_debug_row_map")
        return rm

    def gather(self, q, k_cache, v_cache, block_table, context_lens, num_tiles, **kw):
        import torch
        keep = []
        a = self.args(q, k_cache, v_cache, block_table, context_lens, keep=keep,
                      out=self._scratch_out(q, kw), **kw)
        tb = self._lib.pa_debug_gather_tile_bytes(self._plan)
        dump = torch.zeros(max(num_tiles, 1) * tb, dtype=torch.uint8, device=q.device)
        st = self._lib.pa_debug_gather(self._plan, ctypes.byref(a), dump.data_ptr(),
                                       num_tiles * tb, self._stream(None))
        if st != 0:
            raise PaError(st, "pa_debug_gather")
        return dump, tb


def kv_write_args(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, status=None,
                  num_tokens=None) -> KvWriteArgs:
    """pa_kv_write_args_t over torch tensors: k_new / v_new bf16 [T, Hkv, D], slot_mapping
    int64 [T], caches uint8 [num_pages, Hkv, page_size, D], scales fp32
    [num_pages, Hkv, page_size], status an optional int32/uint32 device word."""
    a = KvWriteArgs()
    a.k_new, a.v_new, a.slot_mapping = _ptr(k_new), _ptr(v_new), _ptr(slot_mapping)
    a.k_cache, a.v_cache, a.k_scale, a.v_scale = (_ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                                  _ptr(v_scale))
    a.status = _ptr(status)
    a.num_tokens = int(num_tokens if num_tokens is not None else k_new.shape[0])
    a.num_pages = int(k_cache.shape[0])
    a.num_kv_heads = int(k_cache.shape[1])
    a.page_size = int(k_cache.shape[2])
    a.head_dim = int(k_cache.shape[3])
    a.reserved = 0
    return a


def kv_quantize_write(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                      status=None, stream=None, args: Optional[KvWriteArgs] = None) -> None:
    """Enqueues pa_kv_quantize_write on `stream` (default: torch's current stream)."""
    import torch
    a = args if args is not None else kv_write_args(k_new, v_new, slot_mapping, k_cache, v_cache,
                                                    k_scale, v_scale, status)
    s = stream if stream is not None else torch.cuda.current_stream(k_cache.device)
    st = lib().pa_kv_quantize_write(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    if st != 0:
        raise PaError(st, "pa_kv_quantize_write")


def index_args(q, k_cache, k_scale, block_table, context_lens, cu_seqlens_q, selected,
               num_selected, scores, *, topk, max_q_len, sm_scale, status=None) -> IndexArgs:
    """pa_index_args_t over torch tensors: q bf16 [rows, heads, 128], k_cache uint8
    [num_pages, page_size, 128], k_scale fp32 [num_pages, page_size] or None, int32 block
    table / context lens / cu_seqlens_q, outputs selected int32 [rows, topk], num_selected
    int32 [rows], scores fp32 [rows, stride]."""
    a = IndexArgs()
    a.q, a.k_cache, a.k_scale = _ptr(q), _ptr(k_cache), _ptr(k_scale)
    a.block_table, a.context_lens, a.cu_seqlens_q = _ptr(block_table), _ptr(context_lens), _ptr(cu_seqlens_q)
    a.selected, a.num_selected, a.scores, a.status = (_ptr(selected), _ptr(num_selected),
                                                      _ptr(scores), _ptr(status))
    a.num_pages = int(k_cache.shape[0])
    a.num_seqs = int(context_lens.shape[0])
    a.num_rows = int(q.shape[0])
    a.index_heads = int(q.shape[1])
    a.head_dim = int(q.shape[2])
    a.page_size = int(k_cache.shape[1])
    a.topk = int(topk)
    a.block_table_stride = int(block_table.shape[1])
    a.max_q_len = int(max_q_len)
    a.sm_scale = float(sm_scale)
    a.reserved = 0
    return a


def index_topk(args: IndexArgs, device=None, stream=None) -> None:
    """Enqueues pa_index_topk on `stream` (default: torch's current stream)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    st = lib().pa_index_topk(ctypes.byref(args), ctypes.c_void_p(s.cuda_stream))
    if st != 0:
        raise PaError(st, "pa_index_topk")


def lse_merge_args(part_out, part_lse, out, lse=None) -> LseMergeArgs:
    """pa_lse_merge_args_t over torch tensors: part_out fp32 [parts, rows, heads, D],
    part_lse fp32 [parts, rows, heads], out bf16 or fp32 [rows, heads, D], lse fp32
    [rows, heads] or None."""
    import torch
    a = LseMergeArgs()
    a.part_out, a.part_lse, a.out, a.lse = _ptr(part_out), _ptr(part_lse), _ptr(out), _ptr(lse)
    a.num_parts, a.num_rows, a.num_heads, a.head_dim = (int(x) for x in part_out.shape)
    a.out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    a.reserved = 0
    return a


def lse_merge(part_out, part_lse, out, lse=None, stream=None, args: Optional[LseMergeArgs] = None):
    """Enqueues pa_lse_merge on `stream` (default: torch's current stream); returns out."""
    import torch
    a = args if args is not None else lse_merge_args(part_out, part_lse, out, lse)
    s = stream if stream is not None else torch.cuda.current_stream(out.device)
    st = lib().pa_lse_merge(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    if st != 0:
        raise PaError(st, "pa_lse_merge")
    return out
