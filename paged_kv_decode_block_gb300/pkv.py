"""Python binding of libpkv (include/pkv.h): argument marshalling only.

Every call forwards device pointers (``tensor.data_ptr()``), sizes and the CUDA
stream handle to the C ABI; all of the decode path runs in the library's CUDA
kernels.  PyTorch is used for device memory and streams.  If the library has
not been built, every entry point raises -- there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

MODE_AUTO, MODE_DIRECT, MODE_SPLIT_QUEUE, MODE_SPLIT_PADDED, MODE_PERSISTENT = range(5)
MODE_NAMES = {MODE_AUTO: "auto", MODE_DIRECT: "direct", MODE_SPLIT_QUEUE: "split_queue",
              MODE_SPLIT_PADDED: "split_padded", MODE_PERSISTENT: "persistent"}
MODES = {v: k for k, v in MODE_NAMES.items()}
MATH = {"auto": 0, "fma": 1, "mma": 2}
COPY = {"auto": 0, "lsu": 1, "tma": 2}
COPY_NAMES = {v: k for k, v in COPY.items()}
MERGE = {"auto": 0, "last": 1, "all": 2}
MERGE_NAMES = {0: "none", 1: "last", 2: "all", 3: "separate"}

OK, EINVAL, ENOMEM, ECUDA, EUNSUPPORTED, EDEVICE, ENOSPACE = range(7)
DEV_PAGE_OOB, DEV_PLAN_MISMATCH, DEV_TIMEOUT, DEV_ROW_FULL = 1, 2, 4, 8
# per-CTA timeline rows (pkv_trace_read): word index of each field
TRACE_WORDS = 12
(TR_TILES, TR_SM, TR_ENTRY, TR_WAIT_DONE, TR_FIRST_BLOCK, TR_STREAM_END, TR_COMBINE_END, TR_ARRIVED,
 TR_MERGE_END, TR_EXIT, TR_LAST_TILE) = range(11)


class Geom(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


class PlanOpts(ctypes.Structure):
    _fields_ = [("force_mode", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("direct_units_per_sm", ctypes.c_int32), ("target_ctas_per_sm", ctypes.c_int32),
                ("min_chunk_pages", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("separate_merge", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("math", ctypes.c_int32), ("copy", ctypes.c_int32), ("merge", ctypes.c_int32)]


class WorkItem(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int32), ("kvh", ctypes.c_int32), ("split", ctypes.c_int32),
                ("page_begin", ctypes.c_int32), ("page_end", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("chunk_pages", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
                ("num_work_items", ctypes.c_int32), ("empty_tiles", ctypes.c_int32),
                ("launches_per_step", ctypes.c_int32), ("grid_ctas", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("merge", ctypes.c_int32),
                ("kv_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("table_bytes", ctypes.c_int64), ("copy", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["mode_name"] = MODE_NAMES.get(self.mode, "?")
        d["merge_name"] = MERGE_NAMES.get(self.merge, "?")
        d["copy_name"] = COPY_NAMES.get(self.copy, "?")
        return d


# symbol -> (restype, argtypes); the full C ABI of include/pkv.h
_P, _I32, _I64, _U32P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint32)
_I32P = ctypes.POINTER(ctypes.c_int32)
SIGNATURES = {
    "pkv_plan": (ctypes.c_int, [_I32P, _I32P, _I32, ctypes.POINTER(Geom), ctypes.POINTER(PlanOpts),
                                ctypes.POINTER(ctypes.c_void_p)]),
    "pkv_plan_dry_run": (ctypes.c_int, [_I32P, _I32P, _I32, ctypes.POINTER(Geom), ctypes.POINTER(PlanOpts),
                                        ctypes.POINTER(PlanInfo), ctypes.POINTER(WorkItem), _I32, _I32P]),
    "pkv_plan_update": (ctypes.c_int, [_P, _P, _P]),
    "pkv_plan_destroy": (None, [_P]),
    "pkv_plan_get_info": (ctypes.c_int, [_P, ctypes.POINTER(PlanInfo)]),
    "pkv_plan_queue": (ctypes.c_int, [_P, ctypes.POINTER(WorkItem), _I32, _I32P]),
    "pkv_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pkv_decode_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pkv_append": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "pkv_status": (ctypes.c_int, [_P, _P, _U32P]),
    "pkv_read_workspace": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32P]),
    "pkv_profile_enable": (ctypes.c_int, [_P, _I32]),
    "pkv_profile_read": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_float), _I32, _I32P]),
    "pkv_trace_enable": (ctypes.c_int, [_P, _I32]),
    "pkv_trace_read": (ctypes.c_int, [_P, _P, _I32, _I32P]),
    "pkv_pool_create": (ctypes.c_int, [_I32P, _I32, _I32, ctypes.POINTER(ctypes.c_void_p)]),
    "pkv_pool_reserve": (ctypes.c_int, [_P, _I32P, _I32P, _I32, _I32, _I32, _I32P, _I32P]),
    "pkv_pool_release": (ctypes.c_int, [_P, _I32P, _I32]),
    "pkv_pool_free_count": (ctypes.c_int32, [_P]),
    "pkv_pool_destroy": (None, [_P]),
    "pkv_decode_static": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, ctypes.POINTER(Geom), _I32, _I32, _P, _P, _P]),
    "pkv_session_create": (ctypes.c_int, [_P, _P, _I32P, _I32P, _P, _P, ctypes.POINTER(ctypes.c_void_p)]),
    "pkv_session_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pkv_session_lengths": (ctypes.c_int, [_P, _I32P]),
    "pkv_session_table": (ctypes.c_int, [_P, _I32P]),
    "pkv_session_destroy": (None, [_P]),
    "pkv_session_device_plan": (ctypes.c_int, [_P, _P]),
    "pkv_session_device_queue": (ctypes.c_int, [_P, ctypes.POINTER(WorkItem), _I32P, _I32, _I32P]),
    "pkv_selftest_wait": (ctypes.c_int, [_I64, _U32P, _I32P]),
    "pkv_resident_start": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I32, _I32,
                                          ctypes.POINTER(ctypes.c_void_p)]),
    "pkv_resident_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64]),
    "pkv_resident_stop": (ctypes.c_int, [_P]),
    "pkv_resident_times": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint64), _I32, _I32P]),
    "pkv_resident_destroy": (None, [_P]),
    "pkv_resident_launches": (ctypes.c_int, [_P, _I32P]),
    "pkv_session_evict": (ctypes.c_int, [_P, _I32P, _I32, _P]),
    "pkv_session_admit": (ctypes.c_int, [_P, _I32P, _I32P, _I32, _P, _P, _P, _P, _P]),
    "pkv_session_free_pages": (ctypes.c_int, [_P, _I32P, _I32, _I32P, _I32P]),
    "pkv_resident_evict": (ctypes.c_int, [_P, _I32P, _I32]),
    "pkv_resident_admit": (ctypes.c_int, [_P, _I32P, _I32P, _I32, _P, _P]),
    "pkv_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_last_cuda_error": (ctypes.c_int, []),
}

_lib = None


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = load().pkv_strerror(code).decode()
        if code == ECUDA:
            msg += f" (cudaError {load().pkv_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [code {code}]" if what else f"{msg} [code {code}]")


def load(path: str = LIB_PATH):
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libpkv is not built ({path} missing); run __graft_entry__.build() "
                               "or python -m paged_kv_decode_block_gb300.csrc.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != OK:
        raise PkvError(rc, what)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr_i32(a):
    return a.ctypes.data_as(_I32P) if a is not None else None


def _opts(force_mode=MODE_AUTO, num_splits=0, direct_units_per_sm=0, target_ctas_per_sm=0,
          min_chunk_pages=0, ctas_per_sm=0, separate_merge=False, num_sms=0, math="auto",
          copy="auto", merge="auto") -> PlanOpts:
    if isinstance(force_mode, str):
        force_mode = MODES[force_mode]
    if isinstance(math, str):
        math = MATH[math]
    if isinstance(copy, str):
        copy = COPY[copy]
    if isinstance(merge, str):
        merge = MERGE[merge]
    return PlanOpts(int(force_mode), int(num_splits), int(direct_units_per_sm),
                    int(target_ctas_per_sm), int(min_chunk_pages), int(ctas_per_sm),
                    int(bool(separate_merge)), int(num_sms), int(math), int(copy), int(merge))


def _geom(B, Hq, Hkv, D, max_pages, num_pages) -> Geom:
    return Geom(int(B), int(Hq), int(Hkv), int(D), int(max_pages), int(num_pages))


def dry_run(seq_lens, block_table, page_size, *, B, Hq, Hkv, D, max_pages, num_pages, **opts):
    """Planner only (no device): returns (info dict, tiles int32 [n][5])."""
    lib = load()
    lens = _i32(seq_lens)
    table = _i32(block_table) if block_table is not None else None
    g = _geom(B, Hq, Hkv, D, max_pages, num_pages)
    o = _opts(**opts)
    info = PlanInfo()
    n = ctypes.c_int32(0)
    _check(lib.pkv_plan_dry_run(_ptr_i32(lens), _ptr_i32(table), int(page_size), ctypes.byref(g),
                                ctypes.byref(o), ctypes.byref(info), None, 0, ctypes.byref(n)), "pkv_plan_dry_run")
    items = (WorkItem * max(n.value, 1))()
    _check(lib.pkv_plan_dry_run(_ptr_i32(lens), _ptr_i32(table), int(page_size), ctypes.byref(g),
                                ctypes.byref(o), None, items, n.value, ctypes.byref(n)), "pkv_plan_dry_run")
    arr = np.ctypeslib.as_array(ctypes.cast(items, _I32P), shape=(max(n.value, 1) * 5,))
    return info.as_dict(), arr[: n.value * 5].reshape(-1, 5).copy()


def _stream_handle(stream):
    """cudaStream_t of `stream` (a torch.cuda.Stream or a raw handle); None means
    torch's current stream on the current device."""
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:   # the handle alone, without building a Stream object
            return raw(torch._C._cuda_getDevice())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Plan:
    """An opaque pkv plan (see pkv_plan in include/pkv.h)."""

    def __init__(self, seq_lens, block_table, page_size, *, B, Hq, Hkv, D, max_pages, num_pages, **opts):
        lib = load()
        lens = _i32(seq_lens)
        table = _i32(block_table) if block_table is not None else None
        self.geom = _geom(B, Hq, Hkv, D, max_pages, num_pages)
        self.page_size = int(page_size)
        self.G = Hq // Hkv
        self.D = D
        o = _opts(**opts)
        h = ctypes.c_void_p()
        _check(lib.pkv_plan(_ptr_i32(lens), _ptr_i32(table), self.page_size, ctypes.byref(self.geom),
                            ctypes.byref(o), ctypes.byref(h)), "pkv_plan")
        self._h = h

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan destroyed")
        return self._h

    def update(self, seq_lens, block_table=None):
        lens = _i32(seq_lens)
        table = _i32(block_table) if block_table is not None else None
        rc = (_lib or load()).pkv_plan_update(self.handle, lens.ctypes.data,
                                              table.ctypes.data if table is not None else None)
        if rc:
            _check(rc, "pkv_plan_update")

    def info(self) -> dict:
        info = PlanInfo()
        _check(load().pkv_plan_get_info(self.handle, ctypes.byref(info)), "pkv_plan_get_info")
        return info.as_dict()

    def queue(self) -> np.ndarray:
        n = ctypes.c_int32(0)
        _check(load().pkv_plan_queue(self.handle, None, 0, ctypes.byref(n)), "pkv_plan_queue")
        items = (WorkItem * max(n.value, 1))()
        _check(load().pkv_plan_queue(self.handle, items, n.value, ctypes.byref(n)), "pkv_plan_queue")
        arr = np.ctypeslib.as_array(ctypes.cast(items, _I32P), shape=(max(n.value, 1) * 5,))
        return arr[: n.value * 5].reshape(-1, 5).copy()

    def status(self, stream=None) -> int:
        st = ctypes.c_uint32(0)
        _check(load().pkv_status(self.handle, _stream_handle(stream), ctypes.byref(st)), "pkv_status")
        return st.value

    def read_workspace(self, stream=None):
        n = ctypes.c_int32(0)
        _check(load().pkv_read_workspace(self.handle, _stream_handle(stream), None, None, 0, ctypes.byref(n)),
               "pkv_read_workspace")
        o = np.zeros((max(n.value, 1), self.G, self.D), np.float32)
        lse = np.zeros((max(n.value, 1), self.G), np.float32)
        _check(load().pkv_read_workspace(self.handle, _stream_handle(stream), o.ctypes.data, lse.ctypes.data,
                                         n.value, ctypes.byref(n)), "pkv_read_workspace")
        return o[: n.value], lse[: n.value]

    def profile(self, enable: bool = True):
        _check(load().pkv_profile_enable(self.handle, int(enable)), "pkv_profile_enable")

    def profile_read(self) -> list:
        ms = (ctypes.c_float * 4)()
        n = ctypes.c_int32(0)
        _check(load().pkv_profile_read(self.handle, ms, 4, ctypes.byref(n)), "pkv_profile_read")
        return [ms[i] for i in range(n.value)]

    def trace(self, enable: bool = True):
        """Per-CTA timeline of the attention launches (pkv_trace_enable)."""
        _check(load().pkv_trace_enable(self.handle, int(enable)), "pkv_trace_enable")

    def read_trace(self) -> np.ndarray:
        """uint64 [CTAs][TRACE_WORDS] rows of the last traced launch (pkv_trace_read)."""
        n = ctypes.c_int32(0)
        _check(load().pkv_trace_read(self.handle, None, 0, ctypes.byref(n)), "pkv_trace_read")
        rows = np.zeros((n.value, TRACE_WORDS), np.uint64)
        if n.value:
            _check(load().pkv_trace_read(self.handle, rows.ctypes.data, n.value, ctypes.byref(n)), "pkv_trace_read")
        return rows

    def close(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.pkv_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan(seq_lens, block_table, page_size, **kw) -> Plan:
    return Plan(seq_lens, block_table, page_size, **kw)


def _dev_ptr(t, name, dtypes=None):
    """Device address of a contiguous CUDA tensor (checked), as an int."""
    try:
        ok = t.is_cuda and t.is_contiguous()
    except AttributeError:
        ok = False
    if not ok:
        raise TypeError(f"{name} must be a contiguous CUDA tensor")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    return t.data_ptr()


_BF16 = None
_I32T = None
_F32T = None


def _bf16_types():
    global _BF16, _I32T, _F32T
    if _BF16 is None:
        import torch
        _BF16 = (torch.bfloat16, torch.int16, getattr(torch, "uint16", torch.int16))
        _I32T = (torch.int32,)
        _F32T = (torch.float32,)
    return _BF16


def decode(q, k_pages, v_pages, block_table, seq_lens, plan: Plan, out, lse, stream=None):
    """pkv_decode: out[b][h] / lse[b][h] for every row and query head."""
    bf = _bf16_types()
    rc = (_lib or load()).pkv_decode(_dev_ptr(q, "q", bf), _dev_ptr(k_pages, "k_pages", bf),
                                     _dev_ptr(v_pages, "v_pages", bf), _dev_ptr(block_table, "block_table", _I32T),
                                     _dev_ptr(seq_lens, "seq_lens", _I32T), plan.handle,
                                     _dev_ptr(out, "out", _F32T), _dev_ptr(lse, "lse", _F32T), _stream_handle(stream))
    if rc:
        _check(rc, "pkv_decode")


def decode_host(q_h, k_pages, v_pages, block_table, seq_lens, plan: Plan, out_h, lse_h, stream=None):
    """pkv_decode_host: q from host memory, out / lse back to host memory (synchronises).
    Pinned buffers (torch ``pin_memory()``) are used in place by the kernel; pageable
    ones are staged through the plan's pinned buffer."""
    bf = _bf16_types()
    rows = plan.geom.batch * plan.geom.num_q_heads
    for buf, what, nbytes in ((q_h, "q_h", rows * plan.D * 2), (out_h, "out_h", rows * plan.D * 4),
                              (lse_h, "lse_h", rows * 4)):
        size = buf.nbytes if isinstance(buf, np.ndarray) else buf.numel() * buf.element_size()
        if size != nbytes:
            raise ValueError(f"{what}: {size} bytes, expected {nbytes}")
    rc = (_lib or load()).pkv_decode_host(_host_ptr(q_h, "q_h"), _dev_ptr(k_pages, "k_pages", bf),
                                          _dev_ptr(v_pages, "v_pages", bf),
                                          _dev_ptr(block_table, "block_table", _I32T),
                                          _dev_ptr(seq_lens, "seq_lens", _I32T), plan.handle,
                                          _host_ptr(out_h, "out_h"), _host_ptr(lse_h, "lse_h"), _stream_handle(stream))
    if rc:
        _check(rc, "pkv_decode_host")


STATIC_SCRATCH_BYTES = 8 * 1024 * 1024


def decode_static(q, k_pages, v_pages, block_table, seq_lens, out, lse, *, page_size, max_seq_len,
                  num_splits, num_pages, stream=None):
    """pkv_decode_static: decode attention that allocates nothing (see include/pkv.h)."""
    import torch
    bf = _bf16_types()
    B, Hq, D = q.shape
    g = _geom(B, Hq, k_pages.shape[2], D, block_table.shape[1], num_pages)
    rc = load().pkv_decode_static(_dev_ptr(q, "q", bf), _dev_ptr(k_pages, "k_pages", bf),
                                  _dev_ptr(v_pages, "v_pages", bf),
                                  _dev_ptr(block_table, "block_table", (torch.int32,)),
                                  _dev_ptr(seq_lens, "seq_lens", (torch.int32,)), int(page_size), ctypes.byref(g),
                                  int(max_seq_len), int(num_splits), _dev_ptr(out, "out", (torch.float32,)),
                                  _dev_ptr(lse, "lse", (torch.float32,)), _stream_handle(stream))
    _check(rc, "pkv_decode_static")


def append(k_new, v_new, k_pages, v_pages, block_table, seq_lens, plan: Plan, stream=None):
    """pkv_append: one new K/V token per row at position seq_lens[b]; seq_lens[b] += 1."""
    import torch
    bf = _bf16_types()
    rc = load().pkv_append(_dev_ptr(k_new, "k_new", bf), _dev_ptr(v_new, "v_new", bf),
                           _dev_ptr(k_pages, "k_pages", bf), _dev_ptr(v_pages, "v_pages", bf),
                           _dev_ptr(block_table, "block_table", (torch.int32,)),
                           _dev_ptr(seq_lens, "seq_lens", (torch.int32,)), plan.handle, _stream_handle(stream))
    _check(rc, "pkv_append")


class Pool:
    """Host FIFO page pool (pkv_pool_*)."""

    def __init__(self, free_pages, num_pages: int):
        pages = _i32(free_pages)
        h = ctypes.c_void_p()
        _check(load().pkv_pool_create(_ptr_i32(pages), len(pages), int(num_pages), ctypes.byref(h)),
               "pkv_pool_create")
        self._h = h

    def reserve(self, seq_lens, block_table: np.ndarray, page_size: int) -> np.ndarray:
        """Assigns pages in place in `block_table` (int32, C-contiguous); returns touched rows."""
        lens = _i32(seq_lens)
        if block_table.dtype != np.int32 or not block_table.flags.c_contiguous:
            raise TypeError("block_table must be a C-contiguous int32 array")
        B, max_pages = block_table.shape
        rows = np.zeros(max(B, 1), np.int32)
        n = ctypes.c_int32(0)
        _check(load().pkv_pool_reserve(self._h, _ptr_i32(lens), _ptr_i32(block_table), B, max_pages,
                                       int(page_size), _ptr_i32(rows), ctypes.byref(n)), "pkv_pool_reserve")
        return rows[: n.value].copy()

    def release(self, pages):
        p = _i32(pages)
        _check(load().pkv_pool_release(self._h, _ptr_i32(p), len(p)), "pkv_pool_release")

    def free_count(self) -> int:
        return int(load().pkv_pool_free_count(self._h))

    def close(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.pkv_pool_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Session:
    """Continuous sessions (pkv_session_*): every step appends one token per row and
    decodes.  The plan, pool and device tensors must outlive the session."""

    def __init__(self, plan: Plan, pool: Pool, seq_lens, block_table, block_table_d, seq_lens_d):
        lens = _i32(seq_lens)
        table = _i32(block_table)
        self.B, self.max_pages = table.shape
        self._keep = (plan, pool, block_table_d, seq_lens_d)
        h = ctypes.c_void_p()
        _check(load().pkv_session_create(plan.handle, pool._h, _ptr_i32(lens), _ptr_i32(table),
                                         _dev_ptr(block_table_d, "block_table_d"),
                                         _dev_ptr(seq_lens_d, "seq_lens_d"), ctypes.byref(h)),
               "pkv_session_create")
        self._h = h

    def step(self, k_new, v_new, k_pages, v_pages, q, out, lse, stream=None):
        bf = _bf16_types()
        import torch
        rc = load().pkv_session_step(self._h, _dev_ptr(k_new, "k_new", bf), _dev_ptr(v_new, "v_new", bf),
                                     _dev_ptr(k_pages, "k_pages", bf), _dev_ptr(v_pages, "v_pages", bf),
                                     _dev_ptr(q, "q", bf), _dev_ptr(out, "out", (torch.float32,)),
                                     _dev_ptr(lse, "lse", (torch.float32,)), _stream_handle(stream))
        _check(rc, "pkv_session_step")

    def lengths(self) -> np.ndarray:
        out = np.zeros(self.B, np.int32)
        _check(load().pkv_session_lengths(self._h, _ptr_i32(out)), "pkv_session_lengths")
        return out

    def table(self) -> np.ndarray:
        out = np.zeros((self.B, self.max_pages), np.int32)
        _check(load().pkv_session_table(self._h, _ptr_i32(out)), "pkv_session_table")
        return out

    def device_plan(self, stream=None):
        """Switch to device-planned (graph-capturable) steps."""
        _check(load().pkv_session_device_plan(self._h, _stream_handle(stream)), "pkv_session_device_plan")

    def device_queue(self):
        """(tiles int32 [n][5], hand-out order int32 [n]) of the last device-built plan."""
        n = ctypes.c_int32(0)
        _check(load().pkv_session_device_queue(self._h, None, None, 0, ctypes.byref(n)), "pkv_session_device_queue")
        items = (WorkItem * max(n.value, 1))()
        order = np.zeros(max(n.value, 1), np.int32)
        _check(load().pkv_session_device_queue(self._h, items, _ptr_i32(order), n.value, ctypes.byref(n)),
               "pkv_session_device_queue")
        arr = np.ctypeslib.as_array(ctypes.cast(items, _I32P), shape=(max(n.value, 1) * 5,))
        return arr[: n.value * 5].reshape(-1, 5).copy(), order[: n.value].copy()

    def evict(self, rows, stream=None):
        """pkv_session_evict: the rows become idle; their pages go back to the free list."""
        r = _i32(rows)
        _check(load().pkv_session_evict(self._h, _ptr_i32(r), len(r), _stream_handle(stream)), "pkv_session_evict")

    def admit(self, rows, lens, k_src, v_src, k_pages, v_pages, stream=None):
        """pkv_session_admit: idle rows take new sessions of `lens` tokens whose K/V
        (device bf16 [sum(lens)][Hkv][D], rows one after another) is copied into fresh pages."""
        bf = _bf16_types()
        r, n = _i32(rows), _i32(lens)
        if len(r) != len(n):
            raise ValueError("rows and lens differ in length")
        _check(load().pkv_session_admit(self._h, _ptr_i32(r), _ptr_i32(n), len(r),
                                        _dev_ptr(k_src, "k_src", bf) if k_src is not None else None,
                                        _dev_ptr(v_src, "v_src", bf) if v_src is not None else None,
                                        _dev_ptr(k_pages, "k_pages", bf), _dev_ptr(v_pages, "v_pages", bf),
                                        _stream_handle(stream)), "pkv_session_admit")

    def free_pages(self):
        """(free list front first, active flags [B]) -- pkv_session_free_pages."""
        n = ctypes.c_int32(0)
        active = np.zeros(max(self.B, 1), np.int32)
        _check(load().pkv_session_free_pages(self._h, None, 0, ctypes.byref(n), _ptr_i32(active)),
               "pkv_session_free_pages")
        pages = np.zeros(max(n.value, 1), np.int32)
        _check(load().pkv_session_free_pages(self._h, _ptr_i32(pages), n.value, ctypes.byref(n), None),
               "pkv_session_free_pages")
        return pages[: n.value].copy(), active[: self.B].copy()

    def close(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.pkv_session_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _host_ptr(t, what):
    """Address (int) of a contiguous host buffer (torch CPU tensor or numpy array), or None."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{what}: host array must be contiguous")
        return t.ctypes.data
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what}: must be a contiguous host tensor")
    return t.data_ptr()


class Resident:
    """Resident steps (pkv_resident_*): one cooperative kernel stays on the GPU and
    runs a continuous-decoding step (plan, append, decode) each time step() is
    called.  The session must be in device-plan mode; the device tensors are bound
    for the kernel's life."""

    def __init__(self, session: "Session", k_pages, v_pages, q, k_new, v_new, out, lse,
                 idle_limit_ns: int = 2_000_000_000, times_cap: int = 4096, yield_every: int = 0):
        import torch
        bf = _bf16_types()
        self._keep = (session, k_pages, v_pages, q, k_new, v_new, out, lse)
        h = ctypes.c_void_p()
        _check(load().pkv_resident_start(session._h, _dev_ptr(k_pages, "k_pages", bf), _dev_ptr(v_pages, "v_pages", bf),
                                         _dev_ptr(q, "q", bf), _dev_ptr(k_new, "k_new", bf),
                                         _dev_ptr(v_new, "v_new", bf), _dev_ptr(out, "out", (torch.float32,)),
                                         _dev_ptr(lse, "lse", (torch.float32,)), int(idle_limit_ns), int(times_cap),
                                         int(yield_every), ctypes.byref(h)), "pkv_resident_start")
        self._h = h

    def step(self, q_h=None, k_new_h=None, v_new_h=None, out_h=None, lse_h=None,
             wait_limit_ns: int = 5_000_000_000):
        """One step: host inputs (None keeps the bound device buffer) in, outputs to the
        host buffers given."""
        _check(load().pkv_resident_step(self._h, _host_ptr(q_h, "q_h"), _host_ptr(k_new_h, "k_new_h"),
                                        _host_ptr(v_new_h, "v_new_h"), _host_ptr(out_h, "out_h"),
                                        _host_ptr(lse_h, "lse_h"), int(wait_limit_ns)), "pkv_resident_step")

    def stop(self):
        _check(load().pkv_resident_stop(self._h), "pkv_resident_stop")

    def launches(self) -> int:
        """Launches of the resident kernel so far (1 + relaunches after yields)."""
        n = ctypes.c_int32(0)
        _check(load().pkv_resident_launches(self._h, ctypes.byref(n)), "pkv_resident_launches")
        return n.value

    def evict(self, rows):
        """pkv_resident_evict: applied at the start of the next step."""
        r = _i32(rows)
        _check(load().pkv_resident_evict(self._h, _ptr_i32(r), len(r)), "pkv_resident_evict")

    def admit(self, rows, lens, k_src, v_src):
        """pkv_resident_admit: applied at the start of the next step (k_src / v_src device
        bf16 [sum(lens)][Hkv][D], kept alive until that step returns)."""
        bf = _bf16_types()
        r, n = _i32(rows), _i32(lens)
        if len(r) != len(n):
            raise ValueError("rows and lens differ in length")
        self._admit_src = (k_src, v_src)
        _check(load().pkv_resident_admit(self._h, _ptr_i32(r), _ptr_i32(n), len(r),
                                         _dev_ptr(k_src, "k_src", bf) if k_src is not None else None,
                                         _dev_ptr(v_src, "v_src", bf) if v_src is not None else None),
               "pkv_resident_admit")

    def times(self) -> np.ndarray:
        """[steps][4] globaltimer ns of each step (after stop): seen, planned, appended,
        published."""
        n = ctypes.c_int32(0)
        _check(load().pkv_resident_times(self._h, None, 0, ctypes.byref(n)), "pkv_resident_times")
        buf = (ctypes.c_uint64 * max(4 * n.value, 1))()
        _check(load().pkv_resident_times(self._h, buf, n.value, ctypes.byref(n)), "pkv_resident_times")
        return np.ctypeslib.as_array(buf)[: 4 * n.value].reshape(-1, 4).copy()

    def close(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.pkv_resident_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def selftest_wait(limit_ns: int = 50_000_000):
    """pkv_selftest_wait: returns (status bits, [first wait ok, abort raised, second wait ok])."""
    st = ctypes.c_uint32(0)
    res = (ctypes.c_int32 * 3)()
    _check(load().pkv_selftest_wait(int(limit_ns), ctypes.byref(st), res), "pkv_selftest_wait")
    return st.value, list(res)
