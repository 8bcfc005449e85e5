"""Gated DeltaNet recurrent-state engine for GB300 (sm_103a).

This package is a thin binding of the C ABI declared in ``include/gdn.h``:
every function below has the C entry point's name and only marshals
arguments (torch tensors -> device pointers, the current CUDA stream).  All
arithmetic of the path runs in the CUDA kernels of ``libgdn.so``; there is no
CPU or PyTorch fallback, and every call raises if the library cannot be
loaded.

PyTorch provides device memory and streams: ``StatePool`` allocates a pool of
state pages as one uint8 tensor and exposes views of a page's state and conv
window for tests and tools.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import inputs
from .inputs import BF16, F32, LayerShape

__all__ = [
    "GdnError", "LayerShape", "StatePool", "load_library", "library_path", "make_desc",
    "gdn_status_string", "gdn_version", "gdn_conv_dim", "gdn_mamba_page_bytes",
    "gdn_block_size_for", "gdn_mamba_pages_per_request", "gdn_pool_blocks_for_pages",
    "gdn_chunk_end", "gdn_cached_tokens", "gdn_resume_block", "gdn_replay_boundary_rows", "gdn_spec_copy_bytes",
    "gdn_replay_bytes_per_request", "gdn_prefill_workspace_size", "gdn_prefill_plan_for",
    "gdn_replay_workspace_size",
    "gdn_prefill_chunked", "gdn_prefill_chunked_noalloc", "workspace_for", "NOALLOC_SCRATCH_BYTES",
    "gdn_mixed_workspace_size", "gdn_mixed_step",
    "gdn_core_prefill_workspace_size", "gdn_core_prefill", "gdn_core_decode",
    "gdn_decode_step", "gdn_checkpoint_resume", "gdn_checkpoint_save", "gdn_replay_append",
    "gdn_replay_rollback", "gdn_replay_flush", "REPLAY_LOG_SLOTS", "PREFILL_AUTO", "PREFILL_FUSED", "PREFILL_TWO_KERNELS", "STATUS",
]

REPLAY_LOG_SLOTS = 32
PREFILL_AUTO, PREFILL_FUSED, PREFILL_TWO_KERNELS = 0, 1, 2   # gdn_prefill_args.path
NOALLOC_SCRATCH_BYTES = 64 << 20   # GDN_NOALLOC_SCRATCH_BYTES
STATUS = {
    0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED_SHAPE",
    3: "GDN_ERR_NOT_BLOCK_ALIGNED", 4: "GDN_ERR_PARTIAL_BLOCK", 5: "GDN_ERR_LOG_OVERFLOW",
    6: "GDN_ERR_ROLLBACK_RANGE", 7: "GDN_ERR_WORKSPACE", 8: "GDN_ERR_CUDA",
    9: "GDN_ERR_PAGE_RANGE", 10: "GDN_ERR_TIMEOUT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgdn.so")
_lib = None


class GdnError(RuntimeError):
    """A gdn_status other than GDN_OK."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)}")


# --------------------------------------------------------------------------- ABI structs

class _Desc(ctypes.Structure):
    _fields_ = [("num_qk_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_dim_k", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
                ("conv_kernel", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("reserved", ctypes.c_int32)]


class _Pool(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("page_bytes", ctypes.c_int64),
                ("num_pages", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_P = ctypes.c_void_p


class _PrefillArgs(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("max_seq_len", ctypes.c_int64),
                ("cu_seqlens", _P), ("start_pos", _P),
                ("start_pos_host", _P), ("init_page_host", _P), ("x", _P), ("g", _P),
                ("beta", _P), ("conv_w", _P), ("init_page", _P), ("block_table", _P),
                ("out_slot", _P), ("o", _P), ("dev_error", _P), ("wait_cycles", ctypes.c_int64),
                ("path", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _DecodeArgs(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("reserved", ctypes.c_int32), ("x", _P),
                ("g", _P), ("beta", _P), ("conv_w", _P), ("slot", _P), ("o", _P),
                ("dev_error", _P)]


class _CoreArgs(ctypes.Structure):
    _fields_ = [("ba", _P), ("A_log", _P), ("dt_bias", _P), ("norm_w", _P), ("norm_eps", ctypes.c_float),
                ("reserved", ctypes.c_int32)]


class _MixedArgs(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("max_seq_len", ctypes.c_int64),
                ("cu_seqlens", _P), ("cu_seqlens_host", _P), ("is_decode", _P), ("is_decode_host", _P),
                ("start_pos", _P), ("start_pos_host", _P), ("init_page", _P), ("init_page_host", _P),
                ("block_table", _P), ("slot", _P), ("x", _P), ("g", _P), ("beta", _P), ("conv_w", _P),
                ("o", _P), ("dev_error", _P)]


class _ReplayArgs(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_new", ctypes.c_int32), ("ckpt_slot", _P),
                ("log_x", _P), ("log_g", _P), ("log_beta", _P), ("log_len", _P), ("x_new", _P),
                ("g_new", _P), ("beta_new", _P), ("conv_w", _P), ("o", _P), ("dev_error", _P),
                ("workspace", _P), ("workspace_bytes", ctypes.c_size_t), ("boundary_rows", _P),
                ("boundary_page", _P)]


class _PrefillPlan(ctypes.Structure):
    _fields_ = [("chains", ctypes.c_int64), ("piece_chunks", ctypes.c_int64), ("levels", ctypes.c_int64),
                ("ctas_per_launch", ctypes.c_int64), ("launches", ctypes.c_int64), ("two_kernels", ctypes.c_int64),
                ("chunk_launches", ctypes.c_int64)]


# --------------------------------------------------------------------------- loading

def library_path() -> str:
    return _LIB_PATH


def load_library(build_if_missing: bool = True):
    """Load libgdn.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        from . import _build
        _build.build()
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"GDN engine library missing: {_LIB_PATH} (build it with "
                           "python -m gated_deltanet_state_gb300._build)")
    lib = ctypes.CDLL(_LIB_PATH)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D, PL = ctypes.POINTER(_Desc), ctypes.POINTER(_Pool)
    sig = {
        "gdn_status_string": ([i32], ctypes.c_char_p),
        "gdn_version": ([], i32),
        "gdn_conv_dim": ([D], i64),
        "gdn_mamba_page_bytes": ([D], i64),
        "gdn_block_size_for": ([i64, i64, i32], i64),
        "gdn_mamba_pages_per_request": ([i32, i32, i32], i64),
        "gdn_pool_blocks_for_pages": ([i64, i32], i64),
        "gdn_chunk_end": ([i64, i64, i64, i32], i64),
        "gdn_cached_tokens": ([i64, i32], i64),
        "gdn_resume_block": ([i64, i32, ctypes.POINTER(i32)], i32),
        "gdn_replay_boundary_rows": ([i64, i32, i32], i32),
        "gdn_spec_copy_bytes": ([i32, i32, i64], i64),
        "gdn_replay_bytes_per_request": ([i32, i64, i32, i64], i64),
        "gdn_prefill_workspace_size": ([D, i32, i64], sz),
        "gdn_prefill_plan_for": ([D, i32, i64, i32, i32, ctypes.POINTER(_PrefillPlan)], i32),
        "gdn_replay_workspace_size": ([D, i32], sz),
        "gdn_prefill_chunked": ([D, PL, ctypes.POINTER(_PrefillArgs), _P, sz, _P], i32),
        "gdn_prefill_chunked_noalloc": ([D, PL, ctypes.POINTER(_PrefillArgs), _P], i32),
        "gdn_decode_step": ([D, PL, ctypes.POINTER(_DecodeArgs), _P], i32),
        "gdn_mixed_workspace_size": ([D, i32, i64], sz),
        "gdn_core_prefill_workspace_size": ([D, i32, i64], sz),
        "gdn_core_prefill": ([D, PL, ctypes.POINTER(_PrefillArgs), ctypes.POINTER(_CoreArgs), _P, sz, _P], i32),
        "gdn_core_decode": ([D, PL, ctypes.POINTER(_DecodeArgs), ctypes.POINTER(_CoreArgs), _P], i32),
        "gdn_mixed_step": ([D, PL, ctypes.POINTER(_MixedArgs), _P, sz, _P], i32),
        "gdn_checkpoint_resume": ([D, PL, _P, _P, _P, i32, _P, _P], i32),
        "gdn_checkpoint_save": ([D, PL, _P, _P, _P, i32, _P, _P], i32),
        "gdn_replay_append": ([D, PL, ctypes.POINTER(_ReplayArgs), _P], i32),
        "gdn_replay_rollback": ([_P, _P, i32, i32, _P, _P], i32),
        "gdn_replay_flush": ([D, PL, ctypes.POINTER(_ReplayArgs), _P], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# --------------------------------------------------------------------------- helpers

def make_desc(shape: LayerShape) -> _Desc:
    return _Desc(shape.num_qk_heads, shape.num_v_heads, shape.head_dim_k, shape.head_dim_v, 4,
                 shape.block_size, shape.chunk_size, shape.in_dtype, shape.out_dtype,
                 float(shape.q_scale), float(shape.norm_eps), 0)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _host(t, dtype, name: str):
    """(ctypes array, keep-alive) for a host-side integer array."""
    if t is None:
        return None, None
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().to(dtype).contiguous()
    else:
        t = torch.as_tensor(list(t), dtype=dtype)
    return t.data_ptr(), t


def _check(status: int, where: str) -> int:
    if status != 0:
        raise GdnError(status, where)
    return 0


class StatePool:
    """A pool of state pages in one device tensor (PyTorch owns the memory)."""

    def __init__(self, shape: LayerShape, num_pages: int, device="cuda", fill: Optional[int] = None):
        self.shape = shape
        self.page_bytes = shape.page
        self.num_pages = int(num_pages)
        alloc = torch.empty if fill is None else torch.full
        args = ((self.num_pages * self.page_bytes + 256,),) if fill is None else \
            ((self.num_pages * self.page_bytes + 256,), fill)
        self.storage = alloc(*args, dtype=torch.uint8, device=device)
        off = (-self.storage.data_ptr()) % 256
        self.buf = self.storage[off:off + self.num_pages * self.page_bytes]

    def abi(self) -> _Pool:
        return _Pool(self.buf.data_ptr(), self.page_bytes, self.num_pages, 0)

    def _page(self, p: int) -> torch.Tensor:
        return self.buf[p * self.page_bytes:(p + 1) * self.page_bytes]

    def state(self, p: int) -> torch.Tensor:
        sh = self.shape
        return self._page(p)[:sh.state_bytes].view(torch.float32).view(
            sh.num_v_heads, sh.head_dim_v, sh.head_dim_k)

    def window(self, p: int) -> torch.Tensor:
        sh = self.shape
        return self._page(p)[sh.state_bytes:sh.state_bytes + sh.window_bytes].view(
            sh.torch_in()).view(3, sh.conv_dim)

    def payload(self, p: int) -> torch.Tensor:
        return self._page(p)[:self.shape.payload_bytes]


# --------------------------------------------------------------------------- host arithmetic

def gdn_status_string(status: int) -> str:
    return load_library().gdn_status_string(int(status)).decode()


def gdn_version() -> int:
    return int(load_library().gdn_version())


def gdn_conv_dim(shape: LayerShape) -> int:
    return int(load_library().gdn_conv_dim(ctypes.byref(make_desc(shape))))


def gdn_mamba_page_bytes(shape: LayerShape) -> int:
    return int(load_library().gdn_mamba_page_bytes(ctypes.byref(make_desc(shape))))


def gdn_block_size_for(mamba_page_bytes: int, attn_bytes_per_token: int, alignment: int) -> int:
    return int(load_library().gdn_block_size_for(mamba_page_bytes, attn_bytes_per_token, alignment))


def gdn_mamba_pages_per_request(num_gdn_layers: int, prefix_caching: int, num_spec_tokens: int) -> int:
    return int(load_library().gdn_mamba_pages_per_request(num_gdn_layers, int(prefix_caching), num_spec_tokens))


def gdn_pool_blocks_for_pages(pages: int, layers_per_block: int) -> int:
    return int(load_library().gdn_pool_blocks_for_pages(pages, layers_per_block))


def gdn_chunk_end(num_computed: int, num_tokens: int, token_budget: int, block_size: int) -> int:
    return int(load_library().gdn_chunk_end(num_computed, num_tokens, token_budget, block_size))


def gdn_cached_tokens(shared_tokens: int, block_size: int) -> int:
    return int(load_library().gdn_cached_tokens(shared_tokens, block_size))


def gdn_resume_block(hit_tokens: int, block_size: int) -> int:
    out = ctypes.c_int32(0)
    _check(load_library().gdn_resume_block(hit_tokens, block_size, ctypes.byref(out)), "gdn_resume_block")
    return int(out.value)


def gdn_replay_boundary_rows(absorbed: int, kept: int, block_size: int) -> int:
    return int(load_library().gdn_replay_boundary_rows(absorbed, kept, block_size))


def gdn_spec_copy_bytes(draft_tokens: int, num_gdn_layers: int, page_bytes: int) -> int:
    return int(load_library().gdn_spec_copy_bytes(draft_tokens, num_gdn_layers, page_bytes))


def gdn_replay_bytes_per_request(num_gdn_layers: int, page_bytes: int, log_slots: int, slot_bytes: int) -> int:
    return int(load_library().gdn_replay_bytes_per_request(num_gdn_layers, page_bytes, log_slots, slot_bytes))


def gdn_prefill_workspace_size(shape: LayerShape, num_seqs: int, total_tokens: int) -> int:
    return int(load_library().gdn_prefill_workspace_size(ctypes.byref(make_desc(shape)), num_seqs, total_tokens))


def gdn_prefill_plan_for(shape: LayerShape, num_seqs: int, max_seq_len: int, num_sms: int = 0,
                         path: int = 0) -> dict:
    """The path and chain plan of one prefill call (num_sms <= 0: the current
    device's SM count; path: PREFILL_AUTO as a call with a workspace resolves
    it, or one of the two paths)."""
    out = _PrefillPlan()
    _check(load_library().gdn_prefill_plan_for(ctypes.byref(make_desc(shape)), num_seqs, max_seq_len, num_sms,
                                               int(path), ctypes.byref(out)), "gdn_prefill_plan_for")
    return {f: int(getattr(out, f)) for f, _ in _PrefillPlan._fields_}


def gdn_replay_workspace_size(shape: LayerShape, num_reqs: int) -> int:
    return int(load_library().gdn_replay_workspace_size(ctypes.byref(make_desc(shape)), num_reqs))


def workspace_for(nbytes: int, device="cuda") -> torch.Tensor:
    """A device scratch buffer of at least nbytes (PyTorch owns the memory)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------- device entry points

def _prefill_args(shape, *, cu_seqlens, start_pos, init_page, block_table, out_slot, x, g, beta, conv_w,
                  o, dev_error, start_pos_host, init_page_host, max_seq_len, wait_cycles=0, path=0):
    n = int(cu_seqlens.numel()) - 1
    sph, keep1 = _host(start_pos_host, torch.int64, "start_pos_host")
    iph, keep2 = _host(init_page_host, torch.int32, "init_page_host")
    bt = block_table
    a = _PrefillArgs(n, int(bt.shape[1]) if bt is not None and bt.dim() == 2 else 0,
                     int(x.shape[0]), int(max_seq_len), _dev(cu_seqlens, torch.int32, "cu_seqlens"),
                     _dev(start_pos, torch.int64, "start_pos"), sph, iph,
                     _dev(x, shape.torch_in(), "x"), _dev(g, torch.float32, "g"),
                     _dev(beta, torch.float32, "beta"), _dev(conv_w, torch.float32, "conv_w"),
                     _dev(init_page, torch.int32, "init_page"),
                     _dev(bt, torch.int32, "block_table") if bt is not None and bt.numel() else None,
                     _dev(out_slot, torch.int32, "out_slot"), _dev(o, shape.torch_out(), "o"),
                     _dev(dev_error, torch.int32, "dev_error"), int(wait_cycles), int(path), 0)
    return a, (keep1, keep2)


def gdn_prefill_chunked(shape: LayerShape, pool: StatePool, *, cu_seqlens, start_pos, init_page,
                        block_table, out_slot, x, g, beta, conv_w, o, dev_error,
                        start_pos_host=None, init_page_host=None, workspace=None, max_seq_len: int = 0,
                        wait_cycles: int = 0, path: int = 0, stream=None, raise_on_error: bool = True) -> int:
    """Chunked prefill with block checkpoints (see gdn.h for the contract).
    Without `workspace` a scratch tensor of gdn_prefill_workspace_size bytes is
    taken from PyTorch's allocator for the call; `workspace=False` passes none
    (a tensor-core layer then takes the fused kernel).  `max_seq_len` (the
    longest sequence; 0: the call's total tokens) sizes the launch plan
    (gdn_prefill_plan_for): a batch of several sequences runs best with the
    exact value.  `wait_cycles` bounds the device-side waits; `path` picks the
    tensor-core path (PREFILL_AUTO, PREFILL_FUSED, PREFILL_TWO_KERNELS; gdn.h)."""
    lib = load_library()
    n = int(cu_seqlens.numel()) - 1
    if workspace is None:
        workspace = workspace_for(gdn_prefill_workspace_size(shape, n, int(x.shape[0])), x.device)
    a, keep = _prefill_args(shape, cu_seqlens=cu_seqlens, start_pos=start_pos, init_page=init_page,
                            block_table=block_table, out_slot=out_slot, x=x, g=g, beta=beta, conv_w=conv_w,
                            o=o, dev_error=dev_error, start_pos_host=start_pos_host,
                            init_page_host=init_page_host, max_seq_len=max_seq_len, wait_cycles=wait_cycles,
                            path=path)
    if workspace is False:
        ws, wsb = None, 0
    else:
        ws = _dev(workspace, None, "workspace")
        wsb = workspace.numel() * workspace.element_size()
    st = lib.gdn_prefill_chunked(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()),
                                 ctypes.byref(a), ws, wsb, _stream(stream))
    return _check(st, "gdn_prefill_chunked") if raise_on_error else st


def gdn_prefill_chunked_noalloc(shape: LayerShape, pool: StatePool, *, cu_seqlens, start_pos, init_page,
                                block_table, out_slot, x, g, beta, conv_w, o, dev_error,
                                start_pos_host=None, init_page_host=None, max_seq_len: int = 0,
                                stream=None, raise_on_error: bool = True) -> int:
    """The prefill with the library's fixed device scratch instead of a
    workspace (gdn.h: gdn_prefill_chunked_noalloc); nothing is allocated."""
    lib = load_library()
    a, keep = _prefill_args(shape, cu_seqlens=cu_seqlens, start_pos=start_pos, init_page=init_page,
                            block_table=block_table, out_slot=out_slot, x=x, g=g, beta=beta, conv_w=conv_w,
                            o=o, dev_error=dev_error, start_pos_host=start_pos_host,
                            init_page_host=init_page_host, max_seq_len=max_seq_len)
    st = lib.gdn_prefill_chunked_noalloc(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()),
                                         ctypes.byref(a), _stream(stream))
    return _check(st, "gdn_prefill_chunked_noalloc") if raise_on_error else st


def _core_args(shape, ba, A_log, dt_bias, norm_w, norm_eps):
    return _CoreArgs(_dev(ba, shape.torch_in(), "ba"), _dev(A_log, torch.float32, "A_log"),
                     _dev(dt_bias, torch.float32, "dt_bias"), _dev(norm_w, torch.float32, "norm_w"),
                     float(norm_eps), 0)


def gdn_core_prefill_workspace_size(shape: LayerShape, num_seqs: int, total_tokens: int) -> int:
    return int(load_library().gdn_core_prefill_workspace_size(ctypes.byref(make_desc(shape)), num_seqs,
                                                              total_tokens))


def gdn_core_prefill(shape: LayerShape, pool: StatePool, *, cu_seqlens, start_pos, init_page, block_table,
                     out_slot, qkvz, ba, conv_w, A_log, dt_bias, norm_w, norm_eps: float, o, dev_error,
                     start_pos_host=None, init_page_host=None, workspace=None, max_seq_len: int = 0,
                     stream=None, raise_on_error: bool = True, path: int = PREFILL_AUTO) -> int:
    """The prefill on packed q | k | v | z and b | a rows, gated-normalised
    outputs (gdn.h: gdn_core_prefill).  Without `workspace` one of
    gdn_core_prefill_workspace_size bytes is taken from PyTorch's allocator."""
    lib = load_library()
    n = int(cu_seqlens.numel()) - 1
    T = int(qkvz.shape[0])
    if workspace is None:
        workspace = workspace_for(gdn_core_prefill_workspace_size(shape, n, T), qkvz.device)
    sph, keep1 = _host(start_pos_host, torch.int64, "start_pos_host")
    iph, keep2 = _host(init_page_host, torch.int32, "init_page_host")
    bt = block_table
    a = _PrefillArgs(n, int(bt.shape[1]) if bt is not None and bt.dim() == 2 else 0, T, int(max_seq_len),
                     _dev(cu_seqlens, torch.int32, "cu_seqlens"), _dev(start_pos, torch.int64, "start_pos"),
                     sph, iph, _dev(qkvz, shape.torch_in(), "qkvz"), None, None,
                     _dev(conv_w, torch.float32, "conv_w"), _dev(init_page, torch.int32, "init_page"),
                     _dev(bt, torch.int32, "block_table") if bt is not None and bt.numel() else None,
                     _dev(out_slot, torch.int32, "out_slot"), _dev(o, shape.torch_out(), "o"),
                     _dev(dev_error, torch.int32, "dev_error"))
    a.path = int(path)
    c = _core_args(shape, ba, A_log, dt_bias, norm_w, norm_eps)
    st = lib.gdn_core_prefill(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()), ctypes.byref(a),
                              ctypes.byref(c), _dev(workspace, None, "workspace"),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(st, "gdn_core_prefill") if raise_on_error else st


def gdn_core_decode(shape: LayerShape, pool: StatePool, *, qkvz, ba, conv_w, A_log, dt_bias, norm_w,
                    norm_eps: float, slot, o, dev_error, stream=None, raise_on_error: bool = True) -> int:
    """One packed token per sequence; gated-normalised outputs (gdn.h:
    gdn_core_decode)."""
    lib = load_library()
    a = _DecodeArgs(int(qkvz.shape[0]), 0, _dev(qkvz, shape.torch_in(), "qkvz"), None, None,
                    _dev(conv_w, torch.float32, "conv_w"), _dev(slot, torch.int32, "slot"),
                    _dev(o, shape.torch_out(), "o"), _dev(dev_error, torch.int32, "dev_error"))
    c = _core_args(shape, ba, A_log, dt_bias, norm_w, norm_eps)
    st = lib.gdn_core_decode(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()), ctypes.byref(a),
                             ctypes.byref(c), _stream(stream))
    return _check(st, "gdn_core_decode") if raise_on_error else st


def gdn_mixed_workspace_size(shape: LayerShape, num_seqs: int, total_tokens: int) -> int:
    return int(load_library().gdn_mixed_workspace_size(ctypes.byref(make_desc(shape)), num_seqs, total_tokens))


def gdn_mixed_step(shape: LayerShape, pool: StatePool, *, cu_seqlens, is_decode, start_pos, init_page,
                   block_table, slot, x, g, beta, conv_w, o, dev_error, start_pos_host=None,
                   init_page_host=None, workspace=None, max_seq_len: int = 0, stream=None,
                   raise_on_error: bool = True) -> int:
    """A packed batch of prefill sequences and single decode tokens (gdn.h:
    gdn_mixed_step).  The host copies of cu_seqlens and is_decode are taken
    from the device tensors."""
    lib = load_library()
    n = int(cu_seqlens.numel()) - 1
    T = int(x.shape[0])
    if workspace is None:
        workspace = workspace_for(gdn_mixed_workspace_size(shape, n, T), x.device)
    cuh, k1 = _host(cu_seqlens, torch.int32, "cu_seqlens_host")
    dh, k2 = _host(is_decode, torch.int8, "is_decode_host")
    sph, k3 = _host(start_pos_host, torch.int64, "start_pos_host")
    iph, k4 = _host(init_page_host, torch.int32, "init_page_host")
    bt = block_table
    a = _MixedArgs(n, int(bt.shape[1]) if bt is not None and bt.dim() == 2 else 0, T, int(max_seq_len),
                   _dev(cu_seqlens, torch.int32, "cu_seqlens"), cuh, _dev(is_decode, torch.int8, "is_decode"), dh,
                   _dev(start_pos, torch.int64, "start_pos"), sph, _dev(init_page, torch.int32, "init_page"), iph,
                   _dev(bt, torch.int32, "block_table") if bt is not None and bt.numel() else None,
                   _dev(slot, torch.int32, "slot"), _dev(x, shape.torch_in(), "x"), _dev(g, torch.float32, "g"),
                   _dev(beta, torch.float32, "beta"), _dev(conv_w, torch.float32, "conv_w"),
                   _dev(o, shape.torch_out(), "o"), _dev(dev_error, torch.int32, "dev_error"))
    ws = _dev(workspace, None, "workspace")
    wsb = workspace.numel() * workspace.element_size()
    st = lib.gdn_mixed_step(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()), ctypes.byref(a), ws, wsb,
                            _stream(stream))
    return _check(st, "gdn_mixed_step") if raise_on_error else st


def gdn_decode_step(shape: LayerShape, pool: StatePool, *, x, g, beta, conv_w, slot, o, dev_error,
                    stream=None, raise_on_error: bool = True) -> int:
    """One token per sequence; the slot pages advance in place."""
    lib = load_library()
    a = _DecodeArgs(int(x.shape[0]), 0, _dev(x, shape.torch_in(), "x"), _dev(g, torch.float32, "g"),
                    _dev(beta, torch.float32, "beta"), _dev(conv_w, torch.float32, "conv_w"),
                    _dev(slot, torch.int32, "slot"), _dev(o, shape.torch_out(), "o"),
                    _dev(dev_error, torch.int32, "dev_error"))
    st = lib.gdn_decode_step(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()), ctypes.byref(a),
                             _stream(stream))
    return _check(st, "gdn_decode_step") if raise_on_error else st


def _copy(fn_name, shape, pool, src_page, dst_page, num_computed_host, dev_error, stream, raise_on_error):
    lib = load_library()
    nch, keep = _host(num_computed_host, torch.int64, "num_computed_host")
    st = getattr(lib, fn_name)(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()),
                               _dev(src_page, torch.int32, "src_page"), _dev(dst_page, torch.int32, "dst_page"),
                               nch, int(src_page.numel()), _dev(dev_error, torch.int32, "dev_error"),
                               _stream(stream))
    return _check(st, fn_name) if raise_on_error else st


def gdn_checkpoint_resume(shape: LayerShape, pool: StatePool, src_page, dst_page, num_computed_host,
                          dev_error, stream=None, raise_on_error: bool = True) -> int:
    """Bit-exact copy block page -> working slot at a block boundary."""
    return _copy("gdn_checkpoint_resume", shape, pool, src_page, dst_page, num_computed_host, dev_error,
                 stream, raise_on_error)


def gdn_checkpoint_save(shape: LayerShape, pool: StatePool, src_page, dst_page, num_computed_host,
                        dev_error, stream=None, raise_on_error: bool = True) -> int:
    """Bit-exact copy working slot -> block page at a block boundary."""
    return _copy("gdn_checkpoint_save", shape, pool, src_page, dst_page, num_computed_host, dev_error,
                 stream, raise_on_error)


def _replay_args(shape, *, ckpt_slot, log_x, log_g, log_beta, log_len, conv_w, dev_error,
                 x_new=None, g_new=None, beta_new=None, o=None, num_new=0, workspace=None,
                 boundary_rows=None, boundary_page=None):
    if workspace is None:
        workspace = workspace_for(gdn_replay_workspace_size(shape, int(ckpt_slot.numel())), log_x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    return workspace, _ReplayArgs(int(ckpt_slot.numel()), int(num_new), _dev(ckpt_slot, torch.int32, "ckpt_slot"),
                       _dev(log_x, shape.torch_in(), "log_x"), _dev(log_g, torch.float32, "log_g"),
                       _dev(log_beta, torch.float32, "log_beta"), _dev(log_len, torch.int32, "log_len"),
                       _dev(x_new, shape.torch_in(), "x_new"), _dev(g_new, torch.float32, "g_new"),
                       _dev(beta_new, torch.float32, "beta_new"), _dev(conv_w, torch.float32, "conv_w"),
                       _dev(o, shape.torch_out(), "o"), _dev(dev_error, torch.int32, "dev_error"),
                       _dev(workspace, None, "workspace"), ws_bytes,
                       _dev(boundary_rows, torch.int32, "boundary_rows"),
                       _dev(boundary_page, torch.int32, "boundary_page"))


def gdn_replay_append(shape: LayerShape, pool: StatePool, *, ckpt_slot, log_x, log_g, log_beta, log_len,
                      x_new, g_new, beta_new, conv_w, o, dev_error, workspace=None, stream=None,
                      raise_on_error: bool = True) -> int:
    """Outputs of the new rows from checkpoint + log; the rows join the log."""
    lib = load_library()
    keep, a = _replay_args(shape, ckpt_slot=ckpt_slot, log_x=log_x, log_g=log_g, log_beta=log_beta,
                           log_len=log_len, conv_w=conv_w, dev_error=dev_error, x_new=x_new, g_new=g_new,
                           beta_new=beta_new, o=o, num_new=int(x_new.shape[1]), workspace=workspace)
    st = lib.gdn_replay_append(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()), ctypes.byref(a),
                               _stream(stream))
    return _check(st, "gdn_replay_append") if raise_on_error else st


def gdn_replay_rollback(log_len, accepted, num_appended: int, dev_error, stream=None,
                        raise_on_error: bool = True) -> int:
    """Drop the rejected rows of the last append from each log."""
    lib = load_library()
    st = lib.gdn_replay_rollback(_dev(log_len, torch.int32, "log_len"), _dev(accepted, torch.int32, "accepted"),
                                 int(num_appended), int(log_len.numel()),
                                 _dev(dev_error, torch.int32, "dev_error"), _stream(stream))
    return _check(st, "gdn_replay_rollback") if raise_on_error else st


def gdn_replay_flush(shape: LayerShape, pool: StatePool, *, ckpt_slot, log_x, log_g, log_beta, log_len,
                     conv_w, dev_error, workspace=None, boundary_rows=None, boundary_page=None, stream=None,
                     raise_on_error: bool = True) -> int:
    """Apply the logged rows to the checkpoint page in place; empties the log.
    With boundary_rows / boundary_page, the state after the first j kept rows
    is also written to a block-boundary page."""
    lib = load_library()
    keep, a = _replay_args(shape, ckpt_slot=ckpt_slot, log_x=log_x, log_g=log_g, log_beta=log_beta,
                           log_len=log_len, conv_w=conv_w, dev_error=dev_error, workspace=workspace,
                           boundary_rows=boundary_rows, boundary_page=boundary_page)
    st = lib.gdn_replay_flush(ctypes.byref(make_desc(shape)), ctypes.byref(pool.abi()), ctypes.byref(a),
                              _stream(stream))
    return _check(st, "gdn_replay_flush") if raise_on_error else st
