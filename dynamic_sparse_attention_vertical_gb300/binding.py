"""ctypes binding of libmi.so: the C ABI of ``include/mi.h`` under the same names.

Argument marshalling only: torch tensors are checked (device, dtype, layout)
and passed as raw device pointers with the current CUDA stream; outputs and
workspaces are allocated here with torch when the caller does not pass them.
Every step of the computation runs in the library's CUDA kernels.  There is no
fallback: if ``libmi.so`` is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmi.so")

MI_OK = 0
MI_ERR_ARG = -1
MI_ERR_SHAPE = -2
MI_ERR_WORKSPACE = -3
MI_ERR_CUDA = -4
MI_ERR_INDEX = -5
MI_ERR_TIMEOUT = -6
MI_ERR_UNIMPLEMENTED = -7
MI_ERR_DEVICE = -8

MI_OP_VS_ESTIMATE = 1
MI_OP_VS_SPARSE_ATTN = 2
MI_OP_BLOCK_SPARSE_ATTN = 3
MI_OP_ASHAPE_ATTN = 4
MI_OP_DENSE_CAUSAL_ATTN = 5
MI_OP_GRID_ESTIMATE = 6
MI_OP_GRID_ATTN = 7
MI_OP_QBOUNDARY_ESTIMATE = 8
MI_OP_QBOUNDARY_ATTN = 9
MI_OP_BOUNDARY2D_ATTN = 10
MI_MAX_RUNS = 64
MI_MAX_MODALITIES = 8
MI_GRID_MAX_SIGMA = 4096
MI_IDX_GIVEN = 1
MI_VS_BLOCK_EXPANDED = 1
MI_MAX_KV = 2048  # largest vertical budget; block-sparse top-k is at most half of it

# every entry point of include/mi.h
SYMBOLS = (
    "mi_workspace_bytes",
    "mi_vs_estimate",
    "mi_vs_estimate_noalloc",
    "mi_vs_sparse_attn",
    "mi_block_sparse_attn",
    "mi_ashape_attn",
    "mi_dense_causal_attn",
    "mi_layer_workspace_bytes",
    "mi_layer_attn",
    "mi_layer_workspace_bytes_varlen",
    "mi_layer_attn_varlen",
    "mi_grid_estimate",
    "mi_grid_attn",
    "mi_qboundary_estimate",
    "mi_qboundary_attn",
    "mi_boundary2d_attn",
    "mi_read_status",
    "mi_strerror",
    "mi_debug_inject",
)
MI_FAULT_NONE = 0
MI_FAULT_SKIP_Q_LOAD = 1

MI_PAT_SKIP = -1
MI_PAT_DENSE = 0
MI_PAT_VS = 1
MI_PAT_BLOCK = 2
MI_PAT_ASHAPE = 3


class HeadCfg(ctypes.Structure):
    """One q-head of a layer call (mi_head_cfg in include/mi.h)."""
    _fields_ = [("pattern", ctypes.c_int32), ("k_v", ctypes.c_int32), ("k_s", ctypes.c_int32),
                ("vs_flags", ctypes.c_int32), ("topk", ctypes.c_int32), ("n_init", ctypes.c_int32),
                ("window", ctypes.c_int32)]

    @staticmethod
    def vs(k_v: int = 1000, k_s: int = 6096, expanded: bool = False) -> "HeadCfg":
        return HeadCfg(MI_PAT_VS, k_v, k_s, MI_VS_BLOCK_EXPANDED if expanded else 0, 0, 0, 0)

    @staticmethod
    def block(topk: int = 100) -> "HeadCfg":
        return HeadCfg(MI_PAT_BLOCK, 0, 0, 0, topk, 0, 0)

    @staticmethod
    def ashape(n_init: int = 128, window: int = 4096) -> "HeadCfg":
        return HeadCfg(MI_PAT_ASHAPE, 0, 0, 0, 0, n_init, window)

    @staticmethod
    def dense() -> "HeadCfg":
        return HeadCfg(MI_PAT_DENSE, 0, 0, 0, 0, 0, 0)

    @staticmethod
    def skip() -> "HeadCfg":
        return HeadCfg(MI_PAT_SKIP, 0, 0, 0, 0, 0, 0)


class MIError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mi_strerror(code)} (code {code})")


_lib = None


def load() -> ctypes.CDLL:
    """Load libmi.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.mi_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.mi_workspace_bytes.restype = S
    lib.mi_vs_estimate.argtypes = [P, P, I, I, I, I, P, I, I, I, I, P, P, P, S, P]
    lib.mi_vs_estimate.restype = I
    lib.mi_vs_estimate_noalloc.argtypes = [P, P, I, I, I, I, P, I, I, I, I, P, P, P]
    lib.mi_vs_estimate_noalloc.restype = I
    lib.mi_vs_sparse_attn.argtypes = [P, P, P, I, I, I, I, P, I, P, I, P, I, I, P, P, P, S, P]
    lib.mi_vs_sparse_attn.restype = I
    lib.mi_block_sparse_attn.argtypes = [P, P, P, I, I, I, I, P, I, I, I, P, I, P, P, P, S, P]
    lib.mi_block_sparse_attn.restype = I
    lib.mi_ashape_attn.argtypes = [P, P, P, I, I, I, I, P, I, I, I, P, P, P, S, P]
    lib.mi_ashape_attn.restype = I
    lib.mi_dense_causal_attn.argtypes = [P, P, P, I, I, I, I, P, I, P, P, P, S, P]
    lib.mi_dense_causal_attn.restype = I
    lib.mi_layer_workspace_bytes.argtypes = [I, I, I, P]
    lib.mi_layer_workspace_bytes.restype = S
    lib.mi_layer_attn.argtypes = [P, P, P, I, I, I, I, P, P, P, P, S, P]
    lib.mi_layer_attn.restype = I
    lib.mi_layer_workspace_bytes_varlen.argtypes = [I, I, P, I, P]
    lib.mi_layer_workspace_bytes_varlen.restype = S
    lib.mi_layer_attn_varlen.argtypes = [P, P, P, I, I, I, I, P, I, P, P, P, P, S, P]
    lib.mi_layer_attn_varlen.restype = I
    lib.mi_grid_estimate.argtypes = [P, P, I, I, I, I, P, I, I, I, I, P, P, S, P]
    lib.mi_grid_estimate.restype = I
    lib.mi_grid_attn.argtypes = [P, P, P, I, I, I, I, P, I, P, I, P, P, P, S, P]
    lib.mi_grid_attn.restype = I
    lib.mi_qboundary_estimate.argtypes = [P, P, I, I, I, I, P, I, P, I, I, I, I, P, P, P, S, P]
    lib.mi_qboundary_estimate.restype = I
    lib.mi_qboundary_attn.argtypes = [P, P, P, I, I, I, I, P, I, P, I, P, I, P, I, P, P, P, S, P]
    lib.mi_qboundary_attn.restype = I
    lib.mi_boundary2d_attn.argtypes = [P, P, P, I, I, I, I, P, I, I, I, P, P, I, P, P, P, S, P]
    lib.mi_boundary2d_attn.restype = I
    lib.mi_read_status.argtypes = [P, P]
    lib.mi_read_status.restype = I
    lib.mi_debug_inject.argtypes = [I, ctypes.c_uint64]
    lib.mi_debug_inject.restype = I
    lib.mi_strerror.argtypes = [I]
    lib.mi_strerror.restype = ctypes.c_char_p
    _lib = lib
    return lib


# ------------------------------------------------------------- helpers ----

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_qkv(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 3:
            raise ValueError("q/k/v/out must be contiguous CUDA bf16 tensors of shape [heads, N, d]")


def _check_idx(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous()):
            raise ValueError("index arrays must be contiguous CUDA int32 tensors")


def _heads(heads: Optional[Sequence[int]], Hq: int):
    if heads is None:
        return None, Hq
    hs = [int(h) for h in heads]
    return (ctypes.c_int32 * len(hs))(*hs), len(hs)


def _workspace(op: int, n_heads: int, Hkv: int, N: int, k_v=0, k_s=0, topk=0, ws=None,
               device=None):
    need = mi_workspace_bytes(op, n_heads, Hkv, N, k_v, k_s, topk)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    if ws.numel() < need:
        raise ValueError(f"workspace too small: {ws.numel()} < {need} bytes")
    return ws


def _raise(rc: int, where: str):
    if rc != MI_OK:
        raise MIError(rc, where)


# ----------------------------------------------------------------- ABI ----

def mi_workspace_bytes(op: int, n_heads: int, Hkv: int, N: int, k_v: int = 0, k_s: int = 0,
                       topk: int = 0) -> int:
    return int(load().mi_workspace_bytes(op, n_heads, Hkv, N, k_v, k_s, topk))


def mi_strerror(code: int) -> str:
    return load().mi_strerror(int(code)).decode()


def mi_debug_inject(mode: int, wait_limit_ns: int = 0) -> int:
    """Test-only: make the attention kernels' first wait expire (see include/mi.h)."""
    return int(load().mi_debug_inject(int(mode), int(wait_limit_ns)))


def mi_read_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load().mi_read_status(_ptr(workspace), _stream(stream)))


def mi_vs_estimate(q, k, heads=None, last_q: int = 64, k_v: int = 1000, k_s: int = 6096,
                   v_idx=None, s_idx=None, workspace=None, stream=None):
    """Top-k vertical columns and slash offsets of each listed head -> (v_idx, s_idx)."""
    _check_qkv(q, k)
    _check_idx(v_idx, s_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if v_idx is None:
        v_idx = torch.empty((n, k_v), dtype=torch.int32, device=q.device)
    if s_idx is None:
        s_idx = torch.empty((n, k_s), dtype=torch.int32, device=q.device)
    ws = _workspace(MI_OP_VS_ESTIMATE, n, Hkv, N, k_v, k_s, 0, workspace, q.device)
    rc = load().mi_vs_estimate(_ptr(q), _ptr(k), Hq, Hkv, N, d, harr, n, last_q, k_v, k_s,
                               _ptr(v_idx), _ptr(s_idx), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_vs_estimate")
    return v_idx, s_idx


def mi_vs_estimate_noalloc(q, k, heads=None, last_q: int = 64, k_v: int = 1000, k_s: int = 6096,
                           v_idx=None, s_idx=None, stream=None):
    """mi_vs_estimate with the library's own fixed scratch array instead of a workspace.

    For callers that cannot allocate device memory at call time; the index outputs
    are allocated here only when not passed in.
    """
    _check_qkv(q, k)
    _check_idx(v_idx, s_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if v_idx is None:
        v_idx = torch.empty((n, k_v), dtype=torch.int32, device=q.device)
    if s_idx is None:
        s_idx = torch.empty((n, k_s), dtype=torch.int32, device=q.device)
    rc = load().mi_vs_estimate_noalloc(_ptr(q), _ptr(k), Hq, Hkv, N, d, harr, n, last_q, k_v, k_s,
                                       _ptr(v_idx), _ptr(s_idx), _stream(stream))
    _raise(rc, "mi_vs_estimate_noalloc")
    return v_idx, s_idx


def mi_vs_sparse_attn(q, k, v, v_idx, s_idx, heads=None, out=None, lse=None, workspace=None,
                      stream=None, expanded: bool = False):
    """Vertical-slash sparse attention of the listed heads into ``out`` ([Hq, N, d]).

    ``expanded`` selects the 64x64 block cover of the diagonals
    (MI_VS_BLOCK_EXPANDED) instead of exact diagonals."""
    _check_qkv(q, k, v, out)
    _check_idx(v_idx, s_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if out is None:
        out = torch.zeros_like(q)
    k_v = v_idx.shape[1] if v_idx is not None else 0
    k_s = s_idx.shape[1] if s_idx is not None else 0
    ws = _workspace(MI_OP_VS_SPARSE_ATTN, n, Hkv, N, k_v, k_s, 0, workspace, q.device)
    rc = load().mi_vs_sparse_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, harr, n,
                                  _ptr(v_idx), k_v, _ptr(s_idx), k_s,
                                  MI_VS_BLOCK_EXPANDED if expanded else 0, _ptr(out), _ptr(lse),
                                  _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_vs_sparse_attn")
    return out


def mi_block_sparse_attn(q, k, v, topk: int = 100, heads=None, blk_idx=None, given: bool = False,
                         out=None, lse=None, workspace=None, stream=None, block: int = 64):
    """Block-sparse attention; returns (out, blk_idx)."""
    _check_qkv(q, k, v, out)
    _check_idx(blk_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if out is None:
        out = torch.zeros_like(q)
    if blk_idx is None:
        blk_idx = torch.empty((n, (N + 63) // 64, topk), dtype=torch.int32, device=q.device)
    ws = _workspace(MI_OP_BLOCK_SPARSE_ATTN, n, Hkv, N, 0, 0, topk, workspace, q.device)
    rc = load().mi_block_sparse_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, harr, n, block,
                                     topk, _ptr(blk_idx), MI_IDX_GIVEN if given else 0,
                                     _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_block_sparse_attn")
    return out, blk_idx


def mi_ashape_attn(q, k, v, n_init: int = 128, window: int = 4096, heads=None, out=None,
                   lse=None, workspace=None, stream=None):
    """A-shape (sink + local window) attention of the listed heads."""
    _check_qkv(q, k, v, out)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if out is None:
        out = torch.zeros_like(q)
    ws = _workspace(MI_OP_ASHAPE_ATTN, n, Hkv, N, ws=workspace, device=q.device)
    rc = load().mi_ashape_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, harr, n, n_init, window,
                               _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_ashape_attn")
    return out


def mi_dense_causal_attn(q, k, v, heads=None, out=None, lse=None, workspace=None, stream=None):
    """Dense causal attention of the listed heads."""
    _check_qkv(q, k, v, out)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if out is None:
        out = torch.zeros_like(q)
    ws = _workspace(MI_OP_DENSE_CAUSAL_ATTN, n, Hkv, N, ws=workspace, device=q.device)
    rc = load().mi_dense_causal_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, harr, n,
                                     _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_dense_causal_attn")
    return out


def _cfg_array(cfg, Hq: int):
    if len(cfg) != Hq:
        raise ValueError(f"one configuration per q-head: got {len(cfg)} for {Hq} heads")
    arr = (HeadCfg * Hq)()
    for i, c in enumerate(cfg):
        arr[i] = c
    return arr


def mi_layer_workspace_bytes(Hq: int, Hkv: int, N: int, cfg) -> int:
    arr = _cfg_array(cfg, Hq)
    return int(load().mi_layer_workspace_bytes(Hq, Hkv, N, ctypes.cast(arr, ctypes.c_void_p)))


def mi_layer_attn(q, k, v, cfg, out=None, lse=None, workspace=None, stream=None):
    """A whole layer in one call: ``cfg[h]`` (a ``HeadCfg``) gives q-head h its pattern and budgets."""
    _check_qkv(q, k, v, out)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    arr = _cfg_array(cfg, Hq)
    if out is None:
        out = torch.zeros_like(q)
    need = int(load().mi_layer_workspace_bytes(Hq, Hkv, N, ctypes.cast(arr, ctypes.c_void_p)))
    if need == 0:
        raise MIError(MI_ERR_ARG, "mi_layer_workspace_bytes")
    ws = torch.empty(need, dtype=torch.uint8, device=q.device) if workspace is None else workspace
    if ws.numel() < need:
        raise ValueError(f"workspace too small: {ws.numel()} < {need} bytes")
    rc = load().mi_layer_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, ctypes.cast(arr, ctypes.c_void_p),
                              _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_layer_attn")
    return out


def _cu_array(cu_seqlens):
    vals = [int(c) for c in cu_seqlens]
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, len(vals) - 1


def mi_layer_workspace_bytes_varlen(Hq: int, Hkv: int, cu_seqlens, cfg) -> int:
    arr = _cfg_array(cfg, Hq)
    cu, n = _cu_array(cu_seqlens)
    return int(load().mi_layer_workspace_bytes_varlen(Hq, Hkv, ctypes.cast(cu, ctypes.c_void_p), n,
                                                      ctypes.cast(arr, ctypes.c_void_p)))


def mi_layer_attn_varlen(q, k, v, cu_seqlens, cfg, out=None, lse=None, workspace=None, stream=None):
    """A packed batch: sequence b holds tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 of every head."""
    _check_qkv(q, k, v, out)
    Hq, total, d = q.shape
    Hkv = k.shape[0]
    arr = _cfg_array(cfg, Hq)
    cu, n = _cu_array(cu_seqlens)
    if out is None:
        out = torch.zeros_like(q)
    need = int(load().mi_layer_workspace_bytes_varlen(Hq, Hkv, ctypes.cast(cu, ctypes.c_void_p), n,
                                                      ctypes.cast(arr, ctypes.c_void_p)))
    if need == 0:
        raise MIError(MI_ERR_ARG, "mi_layer_workspace_bytes_varlen")
    ws = torch.empty(need, dtype=torch.uint8, device=q.device) if workspace is None else workspace
    if ws.numel() < need:
        raise ValueError(f"workspace too small: {ws.numel()} < {need} bytes")
    rc = load().mi_layer_attn_varlen(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, total, d,
                                     ctypes.cast(cu, ctypes.c_void_p), n, ctypes.cast(arr, ctypes.c_void_p),
                                     _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_layer_attn_varlen")
    return out


# -------------------------------------------------------- multi-modal heads ----

def mi_grid_estimate(q, k, sigma_min: int, sigma_max: int, heads=None, last_q: int = 64, grid=None,
                     workspace=None, stream=None):
    """(sigma, phi) of each listed grid head -> int32 [n_heads, 2] on the device."""
    _check_qkv(q, k)
    _check_idx(grid)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if grid is None:
        grid = torch.empty((n, 2), dtype=torch.int32, device=q.device)
    ws = _workspace(MI_OP_GRID_ESTIMATE, n, Hkv, N, 0, 0, 0, workspace, q.device)
    rc = load().mi_grid_estimate(_ptr(q), _ptr(k), Hq, Hkv, N, d, harr, n, last_q, sigma_min, sigma_max,
                                 _ptr(grid), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_grid_estimate")
    return grid


def mi_grid_attn(q, k, v, grid, sigma_min: int, heads=None, out=None, lse=None, workspace=None, stream=None):
    """Grid attention of the listed heads with (sigma, phi) from ``grid`` (int32 [n_heads, 2])."""
    _check_qkv(q, k, v, out)
    _check_idx(grid)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if out is None:
        out = torch.zeros_like(q)
    ws = _workspace(MI_OP_GRID_ATTN, n, Hkv, N, 0, 0, 0, workspace, q.device)
    rc = load().mi_grid_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, harr, n, _ptr(grid), sigma_min,
                             _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_grid_attn")
    return out


def mi_qboundary_estimate(q, k, modality, n_mod: int, heads=None, last_q: int = 64, k_v: int = 1000,
                          k_s: int = 6096, v_idx=None, s_idx=None, workspace=None, stream=None):
    """Per modality, the vertical-slash index sets of each listed head from the 64 query rows
    ending at that modality's last token -> (v_idx [n_mod, n, k_v], s_idx [n_mod, n, k_s])."""
    _check_qkv(q, k)
    _check_idx(modality, v_idx, s_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if v_idx is None:
        v_idx = torch.empty((n_mod, n, k_v), dtype=torch.int32, device=q.device)
    if s_idx is None:
        s_idx = torch.empty((n_mod, n, k_s), dtype=torch.int32, device=q.device)
    ws = _workspace(MI_OP_QBOUNDARY_ESTIMATE, n, Hkv, N, 0, 0, 0, workspace, q.device)
    rc = load().mi_qboundary_estimate(_ptr(q), _ptr(k), Hq, Hkv, N, d, harr, n, _ptr(modality), n_mod,
                                      last_q, k_v, k_s, _ptr(v_idx), _ptr(s_idx), _ptr(ws), ws.numel(),
                                      _stream(stream))
    _raise(rc, "mi_qboundary_estimate")
    return v_idx, s_idx


def mi_qboundary_attn(q, k, v, modality, n_mod: int, v_idx, s_idx, heads=None, out=None, lse=None,
                      workspace=None, stream=None):
    """Q-boundary attention: each row with its modality's index sets (layouts as returned above)."""
    _check_qkv(q, k, v, out)
    _check_idx(modality, v_idx, s_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    harr, n = _heads(heads, Hq)
    if out is None:
        out = torch.zeros_like(q)
    k_v, k_s = int(v_idx.shape[-1]), int(s_idx.shape[-1])
    ws = _workspace(MI_OP_QBOUNDARY_ATTN, n, Hkv, N, 0, 0, 0, workspace, q.device)
    rc = load().mi_qboundary_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, harr, n, _ptr(modality), n_mod,
                                  _ptr(v_idx), k_v, _ptr(s_idx), k_s, _ptr(out), _ptr(lse), _ptr(ws),
                                  ws.numel(), _stream(stream))
    _raise(rc, "mi_qboundary_attn")
    return out


def mi_boundary2d_attn(q, k, v, runs, k_v: int = 1000, k_s: int = 6096, v_idx=None, s_idx=None,
                       given: bool = False, out=None, lse=None, workspace=None, stream=None):
    """2D-boundary attention of every q-head over two modalities given as ``runs``
    [(modality 0|1, length), ...] in token order -> (out, v_idx [2, Hq, k_v], s_idx [2, Hq, k_s]);
    with ``given`` the index sets (sub-sequence positions) are read instead of estimated."""
    _check_qkv(q, k, v, out)
    _check_idx(v_idx, s_idx)
    Hq, N, d = q.shape
    Hkv = k.shape[0]
    flat = [int(x) for r in runs for x in r]
    rarr = (ctypes.c_int32 * len(flat))(*flat)
    if out is None:
        out = torch.zeros_like(q)
    if v_idx is None:
        v_idx = torch.full((2, Hq, k_v), -1, dtype=torch.int32, device=q.device)
    if s_idx is None:
        s_idx = torch.full((2, Hq, k_s), -1, dtype=torch.int32, device=q.device)
    k_v, k_s = int(v_idx.shape[-1]), int(s_idx.shape[-1])
    ws = _workspace(MI_OP_BOUNDARY2D_ATTN, Hq, Hkv, N, 0, 0, 0, workspace, q.device)
    rc = load().mi_boundary2d_attn(_ptr(q), _ptr(k), _ptr(v), Hq, Hkv, N, d, rarr, len(runs), k_v, k_s,
                                   _ptr(v_idx), _ptr(s_idx), MI_IDX_GIVEN if given else 0, _ptr(out), _ptr(lse),
                                   _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "mi_boundary2d_attn")
    return out, v_idx, s_idx
