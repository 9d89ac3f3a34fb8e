"""ctypes binding of libcpattn.so (argument marshalling only).

Every function here passes device pointers, sizes and the current CUDA stream
of PyTorch to the C ABI declared in ``include/cpattn.h``; all arithmetic runs
in the library's kernels.  PyTorch only provides device memory and streams.
If the library is missing the import of any entry point raises: there is no
fallback.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcpattn.so")

CP_F32, CP_BF16 = 0, 1
CP_ORDER_ORIGINAL, CP_ORDER_RANK_LOCAL = 0, 1
CP_PARTITION_ZIGZAG, CP_PARTITION_STRIPED = 0, 1
STATUS = {0: "CP_OK", -1: "CP_ERR_INVALID_ARG", -2: "CP_ERR_ALIGNMENT", -3: "CP_ERR_UNSUPPORTED",
          -4: "CP_ERR_WORKSPACE", -5: "CP_ERR_CUDA", -6: "CP_ERR_TIMEOUT"}

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ("cp_status_string", "cp_validate_desc", "cp_partition_indices", "cp_permute_tokens",
           "cp_tile_attn_fwd", "cp_merge_partials", "cp_ring_attn_workspace_bytes",
           "cp_ring_attn_fwd", "cp_ring_attn_bwd", "cp_get_device_error", "cp_ring_plan_stats",
           "cp_profile_enable", "cp_profile_read", "cp_ring_attn_fwd_static_ws",
           "cp_static_ws_capacity", "cp_ring_bwd_schedule", "cp_permute_rope", "cp_hybrid_schedule",
           "cp_ring_plan_tables", "cp_token_seq_pos", "cp_debug_set_wait_limit")
KERNEL_CLASSES = ("partition", "permute", "tile_fwd", "merge", "delta", "tile_bwd", "convert", "tables", "rope")


class CpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class CpAttnDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("heads_q", ctypes.c_int32),
        ("heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("cp", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("seqlen", ctypes.c_int64),
        ("cu_seqlens_host", ctypes.c_void_p),
        ("cu_seqlens_dev", ctypes.c_void_p),
        ("n_seqs", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("order", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("partition", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("seq_cp_host", ctypes.c_void_p),
        ("seq_rank0_host", ctypes.c_void_p),
        ("seq_cp_dev", ctypes.c_void_p),
        ("seq_rank0_dev", ctypes.c_void_p),
    ]


_lib = None


def lib():
    """Loads the library once; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libcpattn.so not built ({_LIB_PATH}); run "
                              "python -m tile_attention_lse_gb300.build")
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(CpAttnDesc)
        sig = {
            "cp_status_string": ([I32], ctypes.c_char_p),
            "cp_validate_desc": ([D], I32),
            "cp_partition_indices": ([D, P, P, P], I32),
            "cp_permute_tokens": ([D, P, I32, P, P, I32, P], I32),
            "cp_permute_rope": ([D, P, I32, ctypes.c_float, P, P, I32, P], I32),
            "cp_tile_attn_fwd": ([D, P, P, P, I64, I64, I64, I64, I64, I64, P, P, P], I32),
            "cp_merge_partials": ([I32, I64, I32, I32, P, P, P, I32, P, P], I32),
            "cp_ring_attn_workspace_bytes": ([D, I32], SZ),
            "cp_ring_attn_fwd": ([D, P, P, P, P, P, P, SZ, P], I32),
            "cp_ring_attn_bwd": ([D, P, P, P, P, P, P, P, P, P, P, SZ, P], I32),
            "cp_get_device_error": ([P], I32),
            "cp_ring_plan_stats": ([D, P], I32),
            "cp_ring_bwd_schedule": ([D, P, P, P, P, P], I32),
            "cp_profile_enable": ([I32], I32),
            "cp_profile_read": ([P, P], I32),
            "cp_ring_attn_fwd_static_ws": ([D, P, P, P, P, P, P], I32),
            "cp_static_ws_capacity": ([], SZ),
            "cp_hybrid_schedule": ([P, I32, I32, I64, P, P, P, P], I32),
            "cp_ring_plan_tables": ([D, I32, P, P, P, P], I32),
            "cp_token_seq_pos": ([D, P, P, P], I32),
            "cp_debug_set_wait_limit": ([I64], I32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise CpError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return CP_BF16
    if dt == torch.float32:
        return CP_F32
    raise ValueError(f"unsupported dtype {dt}")


@dataclass
class Problem:
    """A descriptor plus the arrays it points to (kept alive here)."""
    batch: int
    heads_q: int
    heads_kv: int
    head_dim: int
    cp: int
    seqlen: int
    dtype: torch.dtype = torch.bfloat16
    cu_seqlens: object = None          # host sequence of int (THD) or None (BSHD)
    order: int = CP_ORDER_ORIGINAL
    causal: bool = True
    softmax_scale: float = 0.0
    device: str = "cuda"
    partition: int = CP_PARTITION_ZIGZAG
    window: int = 0                    # sliding-window width (0: none)
    seq_cp: object = None              # hybrid CP: per sub-sequence CP size (host ints) or None
    seq_rank0: object = None           # hybrid CP: first rank of each sub-sequence's group
    _cu_host: np.ndarray = field(default=None, repr=False)
    _cu_dev: torch.Tensor = field(default=None, repr=False)
    _grp_host: list = field(default=None, repr=False)   # hybrid CP arrays kept alive (host)
    _grp_dev: list = field(default=None, repr=False)    # and their device copies
    _desc: CpAttnDesc = field(default=None, repr=False)

    def __post_init__(self):
        d = CpAttnDesc()
        d.batch, d.heads_q, d.heads_kv, d.head_dim = self.batch, self.heads_q, self.heads_kv, self.head_dim
        d.cp, d.causal, d.seqlen = self.cp, int(bool(self.causal)), self.seqlen
        d.dtype, d.order, d.softmax_scale = _dtype_code(self.dtype), self.order, float(self.softmax_scale)
        d.partition = int(self.partition)
        d.window = int(self.window)
        if self.seq_cp is not None:
            self._grp_host = [np.ascontiguousarray(np.asarray(x, dtype=np.int32)) for x in (self.seq_cp, self.seq_rank0)]
            d.seq_cp_host, d.seq_rank0_host = (a.ctypes.data for a in self._grp_host)
            if self.device != "cpu" and torch.cuda.is_available():
                self._grp_dev = [torch.from_numpy(a).to(self.device) for a in self._grp_host]
                d.seq_cp_dev, d.seq_rank0_dev = (t.data_ptr() for t in self._grp_dev)
        if self.cu_seqlens is not None:
            self._cu_host = np.ascontiguousarray(np.asarray(self.cu_seqlens, dtype=np.int32))
            d.cu_seqlens_host = self._cu_host.ctypes.data
            d.n_seqs = len(self._cu_host) - 1
            if self.device != "cpu" and torch.cuda.is_available():
                self._cu_dev = torch.from_numpy(self._cu_host).to(self.device)
                d.cu_seqlens_dev = self._cu_dev.data_ptr()
        self._desc = d

    @property
    def desc(self):
        return ctypes.byref(self._desc)

    @property
    def thd(self) -> bool:
        return self.cu_seqlens is not None


def status_string(code: int) -> str:
    return lib().cp_status_string(code).decode()


def validate(p: Problem) -> int:
    return int(lib().cp_validate_desc(p.desc))


def plan_stats(p: Problem) -> dict:
    out = (ctypes.c_int64 * 6)()
    _check(lib().cp_ring_plan_stats(p.desc, ctypes.cast(out, ctypes.c_void_p)), "cp_ring_plan_stats")
    keys = ("fwd_items", "partial_rows", "merge_segments", "bwd_items", "pairs", "fwd_key_tiles")
    return dict(zip(keys, list(out)))


PLAN_TABLES = {"fwd": 0, "fwd_wide": 1, "bwd": 2, "dq": 3, "merge": 4}


def plan_tables(p: Problem, which: str):
    """The planner's items [n, 8] and segments [m, 4] (int32 numpy, host only)."""
    import numpy as np
    n, m = ctypes.c_int64(0), ctypes.c_int64(0)
    w = PLAN_TABLES[which]
    _check(lib().cp_ring_plan_tables(p.desc, w, ctypes.byref(n), ctypes.byref(m), None, None),
           "cp_ring_plan_tables")
    items = np.zeros((n.value, 8), dtype=np.int32)
    segs = np.zeros((m.value, 4), dtype=np.int32)
    _check(lib().cp_ring_plan_tables(p.desc, w, None, None, items.ctypes.data if n.value else None,
                                     segs.ctypes.data if m.value else None), "cp_ring_plan_tables")
    return items, segs


def bwd_schedule(p: Problem) -> dict:
    """The tensor-core backward's per-CTA work lists (host only): grid, cta
    offsets [grid + 1], work indices and per-CTA planned loads (numpy)."""
    import numpy as np
    grid, n = ctypes.c_int32(0), ctypes.c_int64(0)
    _check(lib().cp_ring_bwd_schedule(p.desc, ctypes.byref(grid), ctypes.byref(n), None, None, None),
           "cp_ring_bwd_schedule")
    cta = np.zeros(grid.value + 1, dtype=np.int32)
    work = np.zeros(n.value, dtype=np.int32)
    load = np.zeros(grid.value, dtype=np.int64)
    _check(lib().cp_ring_bwd_schedule(p.desc, None, None, cta.ctypes.data, work.ctypes.data, load.ctypes.data),
           "cp_ring_bwd_schedule")
    return {"grid": grid.value, "cta": cta, "work": work, "load": load}


def workspace_bytes(p: Problem, backward: bool = False) -> int:
    return int(lib().cp_ring_attn_workspace_bytes(p.desc, int(backward)))


def workspace(p: Problem, backward: bool = False) -> torch.Tensor:
    n = workspace_bytes(p, backward)
    if n == 0:
        raise CpError(-1, "cp_ring_attn_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=p.device)


def partition_indices(p: Problem, out: torch.Tensor | None = None):
    """idx [cp, seqlen/cp] int32 (device) and, for THD, local cu_seqlens.

    Hybrid CP: idx [seqlen] (ranks of different lengths) and local_cu
    [cp, n_seqs + 1], the slot where each rank's slice of each sub-sequence
    starts."""
    if p.seq_cp is not None:
        idx = torch.empty(p.seqlen, dtype=torch.int32, device=p.device) if out is None else out
        local_cu = torch.empty((p.cp, len(p._cu_host)), dtype=torch.int32, device=p.device)
    else:
        idx = torch.empty((p.cp, p.seqlen // p.cp), dtype=torch.int32, device=p.device) if out is None else out
        local_cu = (torch.empty(len(p._cu_host), dtype=torch.int32, device=p.device) if p.thd else None)
    _check(lib().cp_partition_indices(p.desc, _ptr(idx), _ptr(local_cu), _stream()),
           "cp_partition_indices")
    return idx, local_cu


def hybrid_schedule(lens, world: int, capacity: int):
    """Hybrid CP schedule (host only): per sequence (round, cp, rank0) and the round count."""
    L = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    n = len(L)
    rnd, cp, r0 = (np.zeros(n, dtype=np.int32) for _ in range(3))
    nr = ctypes.c_int32(0)
    _check(lib().cp_hybrid_schedule(L.ctypes.data if n else None, n, int(world), int(capacity),
                                    rnd.ctypes.data if n else None, cp.ctypes.data if n else None,
                                    r0.ctypes.data if n else None, ctypes.byref(nr)), "cp_hybrid_schedule")
    return rnd, cp, r0, nr.value


def token_seq_pos(p: Problem, idx: torch.Tensor) -> torch.Tensor:
    """[seqlen, 2] int32: sub-sequence index and in-sequence position of every rank-local slot."""
    out = torch.empty((p.seqlen, 2), dtype=torch.int32, device=p.device)
    _check(lib().cp_token_seq_pos(p.desc, _ptr(idx), _ptr(out), _stream()), "cp_token_seq_pos")
    return out


def permute_tokens(p: Problem, idx: torch.Tensor, x: torch.Tensor, inverse: bool = False,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    assert x.is_contiguous() and x.dtype == p.dtype
    heads = x.shape[-2]
    out = torch.empty_like(x) if out is None else out
    _check(lib().cp_permute_tokens(p.desc, _ptr(idx), heads, _ptr(x), _ptr(out), int(inverse),
                                   _stream()), "cp_permute_tokens")
    return out


def permute_rope(p: Problem, idx: torch.Tensor, x: torch.Tensor, rope_base: float = 10000.0,
                 inverse: bool = False, out: torch.Tensor | None = None) -> torch.Tensor:
    """Token gather with the rotary position embedding fused in (cp_permute_rope)."""
    assert x.is_contiguous() and x.dtype == p.dtype
    heads = x.shape[-2]
    out = torch.empty_like(x) if out is None else out
    _check(lib().cp_permute_rope(p.desc, _ptr(idx), heads, float(rope_base), _ptr(x), _ptr(out), int(inverse),
                                 _stream()), "cp_permute_rope")
    return out


def tile_attn_fwd(p: Problem, q, k, v, q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len):
    """One TileAttention edge -> (o_part [b, q_len, H, d] f32, lse_part [b, q_len, H] f32)."""
    o = torch.empty((p.batch, q_len, p.heads_q, p.head_dim), dtype=torch.float32, device=q.device)
    l = torch.empty((p.batch, q_len, p.heads_q), dtype=torch.float32, device=q.device)
    _check(lib().cp_tile_attn_fwd(p.desc, _ptr(q), _ptr(k), _ptr(v), q_row0, q_pos0, q_len,
                                  kv_row0, kv_pos0, kv_len, _ptr(o), _ptr(l), _stream()),
           "cp_tile_attn_fwd")
    return o, l


def merge_partials(o_parts: torch.Tensor, lse_parts: torch.Tensor, out_dtype=torch.float32):
    """o_parts [P, rows, H, d] f32, lse_parts [P, rows, H] f32 -> (o, lse)."""
    n, rows, H, d = o_parts.shape
    o = torch.empty((rows, H, d), dtype=out_dtype, device=o_parts.device)
    l = torch.empty((rows, H), dtype=torch.float32, device=o_parts.device)
    _check(lib().cp_merge_partials(n, rows, H, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o),
                                   _dtype_code(out_dtype), _ptr(l), _stream()), "cp_merge_partials")
    return o, l


def ring_attn_fwd(p: Problem, q, k, v, ws: torch.Tensor | None = None, out=None, lse=None):
    ws = workspace(p, False) if ws is None else ws
    o = torch.empty_like(q) if out is None else out
    l = (torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if lse is None else lse)
    _check(lib().cp_ring_attn_fwd(p.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(ws),
                                  ws.numel(), _stream()), "cp_ring_attn_fwd")
    return o, l


def ring_attn_bwd(p: Problem, q, k, v, o, lse, dout, ws: torch.Tensor | None = None,
                  dq=None, dk=None, dv=None):
    ws = workspace(p, True) if ws is None else ws
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().cp_ring_attn_bwd(p.desc, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream()),
           "cp_ring_attn_bwd")
    return dq, dk, dv


def device_error() -> int:
    """Synchronises the current stream and returns the library's device status."""
    return int(lib().cp_get_device_error(_stream()))


def set_wait_limit(cycles: int) -> None:
    """Cycle budget of the tcgen05 kernels' main-loop waits (0: the default)."""
    _check(lib().cp_debug_set_wait_limit(int(cycles)), "cp_debug_set_wait_limit")


def profile_enable(on: bool = True) -> None:
    _check(lib().cp_profile_enable(int(on)), "cp_profile_enable")


def profile_read() -> dict:
    """{class: (total_ms, launches)} since the last read (waits for the events)."""
    ms = (ctypes.c_double * len(KERNEL_CLASSES))()
    n = (ctypes.c_int64 * len(KERNEL_CLASSES))()
    _check(lib().cp_profile_read(ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(n, ctypes.c_void_p)),
           "cp_profile_read")
    return {name: (ms[i], n[i]) for i, name in enumerate(KERNEL_CLASSES)}
