"""Thin Python binding of the kvq C ABI (``include/kvq.h``).

Argument marshalling only: every step of packing and attention runs in the
CUDA kernels of ``libkvq.so``. PyTorch provides device memory and the current
stream. There is no CPU fallback: if the library is missing or a call fails,
these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

F32, BF16, MXFP8 = 0, 1, 2
DTYPES = {"f32": F32, "bf16": BF16, "mxfp8": MXFP8}
TORCH_OF = {F32: torch.float32, BF16: torch.bfloat16}

STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_ARG", 2: "KVQ_ERR_ALIGN", 3: "KVQ_ERR_UNSUPPORTED",
          4: "KVQ_ERR_WORKSPACE", 5: "KVQ_ERR_CUDA"}
DEV_INDEX, DEV_DUP, DEV_TIMEOUT, DEV_BOUNDS = 1, 2, 4, 8
# columns of kv_attend_stats (include/kvq.h, KVQ_STAT_*)
STATS = ("entropy", "support", "top1", "top5", "top10", "zero", "p_zero", "p_tv", "p_sum",
         "qk_tv", "qk_agree")

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")
# the same library built with every kernel's access ranges checked (KVQ_DEBUG)
DEBUG_LIB_PATH = os.path.join(_HERE, "libkvq_debug.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kvq.h")


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class KvqCacheStruct(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("kv_heads", ctypes.c_int32), ("n_tokens", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("recent", ctypes.c_int32),
        ("kwin_dtype", ctypes.c_int32), ("vwin_dtype", ctypes.c_int32),
        ("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
        ("k_window", ctypes.c_void_p), ("v_window", ctypes.c_void_p),
        ("k_window_e8m0", ctypes.c_void_p),
        ("header", ctypes.c_uint32 * 4),
        ("cap_groups", ctypes.c_int32), ("cap_window", ctypes.c_int32),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so (built in-tree by ``quantized_sparse_kv_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with quantized_sparse_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    cp = ctypes.POINTER(KvqCacheStruct)
    lib.kvq_cache_sizes.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.kvq_cache_sizes.restype = i32
    lib.kvq_cache_sizes_reserved.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                             ctypes.POINTER(sz)]
    lib.kvq_cache_sizes_reserved.restype = i32
    lib.kv_append.argtypes = [cp, vp, vp, i32, i32, i32, vp, vp]
    lib.kv_append.restype = i32
    lib.kv_attend_stats.argtypes = [cp, vp, i32, i32, i32, f32, vp, vp, vp, ctypes.POINTER(sz),
                                    vp, vp]
    lib.kv_attend_stats.restype = i32
    lib.kv_attend_candidates_topk.argtypes = [cp, vp, i32, i32, i32, vp, i32, i32, f32, vp, i32,
                                              vp, vp, vp]
    lib.kv_attend_candidates_topk.restype = i32
    lib.kv_attend_candidates_block.argtypes = [cp, vp, i32, i32, i32, vp, i32, i32, f32, vp, i32,
                                               vp, ctypes.POINTER(sz), vp, vp]
    lib.kv_attend_candidates_block.restype = i32
    lib.kv_attend_region_drop.argtypes = [cp, vp, i32, i32, i32, f32, ctypes.POINTER(i32), i32,
                                          ctypes.c_uint32, vp, i32, vp, ctypes.POINTER(sz), vp,
                                          vp]
    lib.kv_attend_region_drop.restype = i32
    lib.kvq_cache_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.kvq_cache_bytes.restype = sz
    lib.kv_pack.argtypes = [vp, vp, i32, cp, vp, vp]
    lib.kv_pack.restype = i32
    lib.kv_attend.argtypes = [cp, vp, i32, i32, i32, f32, vp, i32, ctypes.POINTER(i32), i32, vp,
                              vp, ctypes.POINTER(sz), vp, vp]
    lib.kv_attend.restype = i32
    lib.kv_attend_candidates.argtypes = [cp, vp, i32, i32, i32, vp, i32, i32, f32, vp, i32, vp,
                                         ctypes.POINTER(sz), vp, vp]
    lib.kv_attend_candidates.restype = i32
    lib.kvq_last_launch_count.argtypes = []
    lib.kvq_last_launch_count.restype = i32
    lib.kvq_last_path.argtypes = []
    lib.kvq_last_path.restype = ctypes.c_char_p
    lib.kvq_debug_set.argtypes = [ctypes.c_uint32, i32]
    lib.kvq_debug_set.restype = None
    lib.kvq_debug_checks.argtypes = []
    lib.kvq_debug_checks.restype = i32
    _lib = lib
    return lib


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions include/kvq.h declares."""
    text = open(path, encoding="utf-8").read()
    return re.findall(r"KVQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def _check(status: int, what: str):
    if status != 0:
        raise KvqError(status, what)


def cache_sizes(batch, kv_heads, n_tokens, head_dim, recent, kwin=F32, vwin=F32) -> list[int]:
    lib = load_library()
    out = (ctypes.c_size_t * 8)()
    _check(lib.kvq_cache_sizes(batch, kv_heads, n_tokens, head_dim, recent, kwin, vwin, out),
           "kvq_cache_sizes")
    return list(out)


def cache_sizes_reserved(batch, kv_heads, head_dim, kwin, vwin, cap_groups, cap_window) -> list[int]:
    lib = load_library()
    out = (ctypes.c_size_t * 8)()
    _check(lib.kvq_cache_sizes_reserved(batch, kv_heads, head_dim, kwin, vwin, cap_groups,
                                        cap_window, out), "kvq_cache_sizes_reserved")
    return list(out)


def cache_bytes(batch, kv_heads, n_tokens, head_dim, recent, kwin=F32, vwin=F32) -> int:
    return int(load_library().kvq_cache_bytes(batch, kv_heads, n_tokens, head_dim, recent, kwin,
                                              vwin))


def _dtype(x) -> int:
    return DTYPES[x] if isinstance(x, str) else int(x)


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t is not None and t.numel() else None)


class PackedCache:
    """Device arrays of one packed cache plus the C descriptor pointing at them.

    ``reserve=(cap_groups, cap_window)`` lays the arrays out with room for
    kv_append: cap_groups K groups (32 per group V rows) and cap_window window
    rows per (sequence, head)."""

    def __init__(self, batch, kv_heads, n_tokens, head_dim, recent, kwin="f32", vwin="f32",
                 device="cuda", reserve=None):
        self.batch, self.kv_heads, self.n_tokens = batch, kv_heads, n_tokens
        self.head_dim, self.recent = head_dim, recent
        self.kwin, self.vwin = _dtype(kwin), _dtype(vwin)
        self.cut = n_tokens - recent
        self.gk = -(-self.cut // 32)
        self.reserve = tuple(reserve) if reserve else (0, 0)
        if reserve:
            cap_g, cap_w = self.reserve
            if cap_g < self.gk or cap_w < recent:
                raise ValueError("reserve is smaller than the cache")
            rows_g, rows_v, rows_w = cap_g, 32 * cap_g, cap_w
        else:
            rows_g, rows_v, rows_w = self.gk, self.cut, recent
        self.sizes = cache_sizes(batch, kv_heads, n_tokens, head_dim, recent, self.kwin, self.vwin)
        u8 = torch.uint8
        b, h, d = batch, kv_heads, head_dim
        self.k_codes = torch.empty((b, h, rows_g, 32, d // 2), dtype=u8, device=device)
        self.k_scales = torch.empty((b, h, rows_g, d), dtype=torch.float32, device=device)
        self.v_codes = torch.empty((b, h, rows_v, d // 2), dtype=u8, device=device)
        self.v_scales = torch.empty((b, h, rows_v, d // 32), dtype=torch.float32, device=device)
        kdt = u8 if self.kwin == MXFP8 else TORCH_OF[self.kwin]
        self.k_window = torch.empty((b, h, rows_w, d), dtype=kdt, device=device)
        self.v_window = torch.empty((b, h, rows_w, d), dtype=TORCH_OF[self.vwin], device=device)
        self.k_window_e8m0 = torch.empty((b, h, rows_w, d // 32) if self.kwin == MXFP8 else (0,),
                                         dtype=u8, device=device)
        self.struct = KvqCacheStruct(
            batch, kv_heads, n_tokens, head_dim, recent, self.kwin, self.vwin,
            _ptr(self.k_codes), _ptr(self.k_scales), _ptr(self.v_codes), _ptr(self.v_scales),
            _ptr(self.k_window), _ptr(self.v_window), _ptr(self.k_window_e8m0),
            (ctypes.c_uint32 * 4)(0, 0, 0, 0), self.reserve[0], self.reserve[1])
        self.ref = ctypes.byref(self.struct)

    def _sync_shape(self):
        """Take n_tokens and recent back from the descriptor (kv_append moves them)."""
        self.n_tokens, self.recent = int(self.struct.n_tokens), int(self.struct.recent)
        self.cut = self.n_tokens - self.recent
        self.gk = -(-self.cut // 32)
        self.sizes = cache_sizes(self.batch, self.kv_heads, self.n_tokens, self.head_dim,
                                 self.recent, self.kwin, self.vwin)

    def used(self) -> dict:
        """Views of the filled part of every array (the tight layout's content)."""
        return {"k_codes": self.k_codes[:, :, :self.gk], "k_scales": self.k_scales[:, :, :self.gk],
                "v_codes": self.v_codes[:, :, :self.cut], "v_scales": self.v_scales[:, :, :self.cut],
                "k_window": self.k_window[:, :, :self.recent],
                "v_window": self.v_window[:, :, :self.recent]}

    @property
    def header(self):
        return list(self.struct.header)

    def payload_bytes(self) -> int:
        return int(sum(self.sizes))


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(4, dtype=torch.int32, device=device)


def read_status(status: torch.Tensor) -> int:
    """Synchronise on the current stream and return the device status word."""
    torch.cuda.current_stream().synchronize()
    return int(status[0].item())


def pack(k: torch.Tensor, v: torch.Tensor, recent: int, kwin="f32", vwin=None,
         status: torch.Tensor | None = None, out: PackedCache | None = None,
         reserve=None) -> PackedCache:
    """kv_pack: k, v (batch, kv_heads, N, D) fp32 or bf16 on the GPU.

    ``out`` reuses the arrays of an existing cache of the same shape;
    ``reserve=(cap_groups, cap_window)`` leaves room for kv_append."""
    if k.dtype not in (torch.float32, torch.bfloat16) or v.dtype != k.dtype:
        raise TypeError("k and v must both be float32 or bfloat16")
    k = k.contiguous()
    v = v.contiguous()
    b, h, n, d = k.shape
    if out is None:
        vw = vwin if vwin is not None else ("f32" if _dtype(kwin) == F32 else "bf16")
        out = PackedCache(b, h, n, d, recent, kwin, vw, device=k.device, reserve=reserve)
    in_dt = F32 if k.dtype == torch.float32 else BF16
    lib = load_library()
    _check(lib.kv_pack(_ptr(k), _ptr(v), in_dt, out.ref,
                       _ptr(status) if status is not None else None, _stream()), "kv_pack")
    return out


class Attend:
    """A prepared kv_attend call: output, region-mass, workspace and status
    buffers are allocated once; ``run()`` only re-issues the C call."""

    def __init__(self, cache: PackedCache, q: torch.Tensor, sm_scale: float = 0.0,
                 out_dtype=None, region_bounds=None, out=None):
        self.lib = load_library()
        self.cache = cache
        self.q = q.contiguous()
        if self.q.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("q must be float32 or bfloat16")
        b, hq, nq, d = self.q.shape
        if b != cache.batch or d != cache.head_dim:
            raise ValueError("q does not match the cache")
        self.q_dt = F32 if self.q.dtype == torch.float32 else BF16
        self.out_dt = _dtype(out_dtype) if out_dtype is not None else self.q_dt
        self.out = out if out is not None else torch.empty(
            (b, hq, nq, d), dtype=TORCH_OF[self.out_dt], device=self.q.device)
        self.hq, self.nq, self.sm_scale = hq, nq, float(sm_scale or 0.0)
        if region_bounds is not None:
            rb = [int(x) for x in region_bounds]
            self.n_regions = len(rb) - 1
            self.bounds = (ctypes.c_int32 * len(rb))(*rb)
            self.mass = torch.empty((b, hq, nq, self.n_regions), dtype=torch.float32,
                                    device=self.q.device)
        else:
            self.n_regions, self.bounds, self.mass = 0, None, None
        self.status = new_status(self.q.device)
        need = ctypes.c_size_t(0)
        self._call(None, need)
        self.ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=self.q.device)
        self.ws_bytes = ctypes.c_size_t(self.ws.numel())
        self.path = None

    def _call(self, ws, ws_bytes):
        st = self.lib.kv_attend(self.cache.ref, _ptr(self.q), self.q_dt, self.hq, self.nq,
                                self.sm_scale, _ptr(self.out), self.out_dt, self.bounds,
                                self.n_regions, _ptr(self.mass), ws, ctypes.byref(ws_bytes),
                                _ptr(self.status), _stream())
        _check(st, "kv_attend")

    def run(self):
        self._call(_ptr(self.ws), self.ws_bytes)
        self.path = self.lib.kvq_last_path().decode()
        return self.out

    def launches(self) -> int:
        return int(self.lib.kvq_last_launch_count())


def attend(cache: PackedCache, q: torch.Tensor, sm_scale: float = 0.0, out_dtype=None,
           region_bounds=None):
    """kv_attend; returns (out, region_mass or None, path)."""
    a = Attend(cache, q, sm_scale, out_dtype, region_bounds)
    a.run()
    return a.out, a.mass, a.path


class AttendCandidates:
    """A prepared kv_attend_candidates call (see Attend)."""

    def __init__(self, cache: PackedCache, q: torch.Tensor, idx: torch.Tensor,
                 sm_scale: float = 0.0, out_dtype=None, validate: bool = False, out=None):
        self.lib = load_library()
        self.cache = cache
        self.q = q.contiguous()
        self.idx = idx.to(torch.int32).contiguous()
        b, hq, nq, d = self.q.shape
        if tuple(self.idx.shape[:3]) != (b, hq, nq):
            raise ValueError("idx must be (batch, q_heads, n_q, C)")
        self.q_dt = F32 if self.q.dtype == torch.float32 else BF16
        self.out_dt = _dtype(out_dtype) if out_dtype is not None else self.q_dt
        self.out = out if out is not None else torch.empty(
            (b, hq, nq, d), dtype=TORCH_OF[self.out_dt], device=self.q.device)
        self.hq, self.nq, self.c = hq, nq, int(self.idx.shape[3])
        self.sm_scale, self.validate = float(sm_scale or 0.0), int(bool(validate))
        self.status = new_status(self.q.device)
        need = ctypes.c_size_t(0)
        self._call(None, need)
        self.ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=self.q.device)
        self.ws_bytes = ctypes.c_size_t(self.ws.numel())

    def _call(self, ws, ws_bytes):
        st = self.lib.kv_attend_candidates(self.cache.ref, _ptr(self.q), self.q_dt, self.hq,
                                           self.nq, _ptr(self.idx), self.c, self.validate,
                                           self.sm_scale, _ptr(self.out), self.out_dt, ws,
                                           ctypes.byref(ws_bytes), _ptr(self.status), _stream())
        _check(st, "kv_attend_candidates")

    def run(self):
        self._call(_ptr(self.ws), self.ws_bytes)
        return self.out

    def launches(self) -> int:
        return int(self.lib.kvq_last_launch_count())


def attend_candidates(cache: PackedCache, q: torch.Tensor, idx: torch.Tensor,
                      sm_scale: float = 0.0, out_dtype=None, validate: bool = False):
    """kv_attend_candidates; returns (out, status tensor)."""
    a = AttendCandidates(cache, q, idx, sm_scale, out_dtype, validate)
    a.run()
    return a.out, a.status


def debug_set(wait_limit_ns: int = 0, drop_item: int = -1):
    """Failure-test hook (see kvq_debug_set in include/kvq.h)."""
    load_library().kvq_debug_set(int(wait_limit_ns), int(drop_item))


def append(cache: PackedCache, k_new: torch.Tensor, v_new: torch.Tensor, window: int,
           status: torch.Tensor | None = None) -> PackedCache:
    """kv_append: k_new, v_new (batch, kv_heads, T, D) fp32 or bf16 on the GPU,
    added after the cache's tokens; the window keeps at least ``window`` tokens
    and whole 32-token groups move from its oldest end into int4."""
    if k_new.dtype not in (torch.float32, torch.bfloat16) or v_new.dtype != k_new.dtype:
        raise TypeError("k_new and v_new must both be float32 or bfloat16")
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    b, h, t, d = k_new.shape
    if (b, h, d) != (cache.batch, cache.kv_heads, cache.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("new tokens do not match the cache")
    in_dt = F32 if k_new.dtype == torch.float32 else BF16
    lib = load_library()
    _check(lib.kv_append(cache.ref, _ptr(k_new), _ptr(v_new), in_dt, t, window,
                         _ptr(status) if status is not None else None, _stream()), "kv_append")
    cache._sync_shape()
    return cache


def attend_stats(cache: PackedCache, q: torch.Tensor, signs: torch.Tensor | None = None,
                 sm_scale: float = 0.0, status: torch.Tensor | None = None) -> torch.Tensor:
    """kv_attend_stats: observer statistics of the softmax rows of q over the
    cache; returns float32 (batch, q_heads, n_q, len(STATS)), columns STATS.
    ``signs`` (D,) of +-1 turns on the signed Hadamard rotation of the MXFP8
    Q/K path."""
    q = q.contiguous()
    if q.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("q must be float32 or bfloat16")
    b, hq, nq, d = q.shape
    out = torch.empty((b, hq, nq, len(STATS)), dtype=torch.float32, device=q.device)
    sg = None
    if signs is not None:
        sg = signs.to(device=q.device, dtype=torch.float32).contiguous()
        if sg.shape != (d,):
            raise ValueError("signs must have head_dim entries")
    lib = load_library()
    q_dt = F32 if q.dtype == torch.float32 else BF16
    need = ctypes.c_size_t(0)
    _check(lib.kv_attend_stats(cache.ref, _ptr(q), q_dt, hq, nq, float(sm_scale or 0.0), _ptr(sg),
                               _ptr(out), None, ctypes.byref(need), None, _stream()),
           "kv_attend_stats")
    ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=q.device)
    ws_bytes = ctypes.c_size_t(ws.numel())
    _check(lib.kv_attend_stats(cache.ref, _ptr(q), q_dt, hq, nq, float(sm_scale or 0.0), _ptr(sg),
                               _ptr(out), _ptr(ws), ctypes.byref(ws_bytes),
                               _ptr(status) if status is not None else None, _stream()),
           "kv_attend_stats")
    return out


def attend_candidates_topk(cache: PackedCache, q: torch.Tensor, idx: torch.Tensor, top_k: int,
                           sm_scale: float = 0.0, out_dtype=None):
    """kv_attend_candidates_topk: attend only the top_k of each row's listed
    keys by exact score. Returns (out, selected positions, status tensor)."""
    q = q.contiguous()
    if q.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("q must be float32 or bfloat16")
    idx = idx.to(torch.int32).contiguous()
    b, hq, nq, d = q.shape
    if tuple(idx.shape[:3]) != (b, hq, nq):
        raise ValueError("idx must be (batch, q_heads, n_q, C)")
    q_dt = F32 if q.dtype == torch.float32 else BF16
    out_dt = _dtype(out_dtype) if out_dtype is not None else q_dt
    out = torch.empty((b, hq, nq, d), dtype=TORCH_OF[out_dt], device=q.device)
    selected = torch.empty((b, hq, nq, top_k), dtype=torch.int32, device=q.device)
    status = new_status(q.device)
    lib = load_library()
    _check(lib.kv_attend_candidates_topk(cache.ref, _ptr(q), q_dt, hq, nq, _ptr(idx),
                                         idx.shape[3], top_k, float(sm_scale or 0.0), _ptr(out),
                                         out_dt, _ptr(selected), _ptr(status), _stream()),
           "kv_attend_candidates_topk")
    return out, selected, status


class AttendCandidatesBlock:
    """A prepared kv_attend_candidates_block call: rows [k*block_q, (k+1)*block_q)
    of a head attend over list k of idx (batch, q_heads, ceil(n_q / block_q), C)."""

    def __init__(self, cache: PackedCache, q: torch.Tensor, idx: torch.Tensor, block_q: int,
                 sm_scale: float = 0.0, out_dtype=None):
        self.lib = load_library()
        self.cache = cache
        self.q = q.contiguous()
        if self.q.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("q must be float32 or bfloat16")
        self.idx = idx.to(torch.int32).contiguous()
        b, hq, nq, d = self.q.shape
        if tuple(self.idx.shape[:3]) != (b, hq, -(-nq // block_q)):
            raise ValueError("idx must be (batch, q_heads, ceil(n_q / block_q), C)")
        self.block_q = block_q
        self.q_dt = F32 if self.q.dtype == torch.float32 else BF16
        self.out_dt = _dtype(out_dtype) if out_dtype is not None else self.q_dt
        self.out = torch.empty((b, hq, nq, d), dtype=TORCH_OF[self.out_dt], device=self.q.device)
        self.hq, self.nq, self.sm_scale = hq, nq, float(sm_scale or 0.0)
        self.status = new_status(self.q.device)
        need = ctypes.c_size_t(0)
        self._call(None, need)
        self.ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=self.q.device)
        self.ws_bytes = ctypes.c_size_t(self.ws.numel())
        self.path = None

    def _call(self, ws, ws_bytes):
        st = self.lib.kv_attend_candidates_block(
            self.cache.ref, _ptr(self.q), self.q_dt, self.hq, self.nq, _ptr(self.idx),
            self.idx.shape[3], self.block_q, self.sm_scale, _ptr(self.out), self.out_dt, ws,
            ctypes.byref(ws_bytes), _ptr(self.status), _stream())
        _check(st, "kv_attend_candidates_block")

    def run(self) -> torch.Tensor:
        self._call(_ptr(self.ws), self.ws_bytes)
        self.path = self.lib.kvq_last_path().decode()
        return self.out


class AttendRegionDrop:
    """A prepared kv_attend_region_drop call: attention over the keys of the
    regions not listed in ``drop`` (region r = [bounds[r], bounds[r + 1]))."""

    def __init__(self, cache: PackedCache, q: torch.Tensor, region_bounds, drop,
                 sm_scale: float = 0.0, out_dtype=None):
        self.lib = load_library()
        self.cache = cache
        self.q = q.contiguous()
        if self.q.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("q must be float32 or bfloat16")
        rb = [int(x) for x in region_bounds]
        self.n_regions = len(rb) - 1
        self.bounds = (ctypes.c_int32 * len(rb))(*rb)
        self.mask = 0
        for r in drop:
            self.mask |= 1 << int(r)
        b, hq, nq, d = self.q.shape
        self.q_dt = F32 if self.q.dtype == torch.float32 else BF16
        self.out_dt = _dtype(out_dtype) if out_dtype is not None else self.q_dt
        self.out = torch.empty((b, hq, nq, d), dtype=TORCH_OF[self.out_dt], device=self.q.device)
        self.hq, self.nq, self.sm_scale = hq, nq, float(sm_scale or 0.0)
        self.status = new_status(self.q.device)
        need = ctypes.c_size_t(0)
        self._call(None, need)
        self.ws = torch.empty(max(int(need.value), 256), dtype=torch.uint8, device=self.q.device)
        self.ws_bytes = ctypes.c_size_t(self.ws.numel())

    def _call(self, ws, ws_bytes):
        st = self.lib.kv_attend_region_drop(
            self.cache.ref, _ptr(self.q), self.q_dt, self.hq, self.nq, self.sm_scale, self.bounds,
            self.n_regions, self.mask, _ptr(self.out), self.out_dt, ws, ctypes.byref(ws_bytes),
            _ptr(self.status), _stream())
        _check(st, "kv_attend_region_drop")

    def run(self) -> torch.Tensor:
        self._call(_ptr(self.ws), self.ws_bytes)
        return self.out
