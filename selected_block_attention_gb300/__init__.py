"""selected_block_attention_gb300 -- Python binding of libsba (GB300, sm_103a).

Thin ctypes marshalling over the C ABI declared in ``include/sba.h``: every
function below checks tensor placement/dtypes, allocates outputs with torch (device
memory is torch's job here), and passes raw device pointers plus the current CUDA
stream to the library.  No step of the computation runs in Python, and there is no
fallback: if ``libsba.so`` is missing or a tensor is not on a CUDA device the call
raises.

Entry points (same names as the C ABI without the ``sba_`` prefix):
  nsa_select_fwd, sparse_mask_bounds (forward and dK/dV bounds), blocksparse_attn_fwd,
  ragged_decode_fwd,
  ragged_decode_fwd_noalloc, ragged_decode_workspace_size, ragged_flash_attention_fwd,
  ragged_flash_attention_workspace_size, check_error.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "SBAError", "load_library", "library_path", "nsa_select_fwd", "nsa_select_fwd_host",
    "nsa_select_host_workspace_size", "sparse_mask_bounds",
    "blocksparse_attn_fwd", "ragged_decode_fwd", "ragged_decode_fwd_noalloc",
    "ragged_decode_workspace_size", "ragged_flash_attention_fwd",
    "ragged_flash_attention_workspace_size", "l2_read_probe", "check_error",
    "set_wait_timeout_cycles", "get_wait_timeout_cycles", "nsa_select_bwd",
    "nsa_select_bwd_workspace_size", "EXPORTED_SYMBOLS",
]

EXPORTED_SYMBOLS = (
    "sba_version", "sba_last_error", "sba_nsa_select_fwd", "sba_sparse_mask_bounds",
    "sba_sparse_mask_dkdv_bounds",
    "sba_blocksparse_attn_fwd", "sba_ragged_decode_workspace_size", "sba_ragged_decode_fwd",
    "sba_ragged_decode_fwd_noalloc", "sba_ragged_flash_attention_workspace_size",
    "sba_ragged_flash_attention_fwd", "sba_l2_read_probe", "sba_check_error",
    "sba_nsa_select_host_workspace_size", "sba_nsa_select_fwd_host",
    "sba_set_wait_timeout_cycles", "sba_get_wait_timeout_cycles",
    "sba_nsa_select_bwd", "sba_nsa_select_bwd_workspace_size",
)

SBA_BF16, SBA_F32 = 0, 1
_ERRORS = {-1: "invalid argument", -2: "unsupported", -3: "CUDA error", -4: "timeout",
           -5: "malformed device input"}

_lib = None


class SBAError(RuntimeError):
    def __init__(self, code, message):
        super().__init__(f"{_ERRORS.get(code, code)}: {message}")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libsba.so (built in-tree by ``_build.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libsba.so not found at {path}; build it with "
                           "selected_block_attention_gb300._build.build()")
    lib = ctypes.CDLL(path)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    ci, cf, csz = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.sba_version.restype = ctypes.c_char_p
    lib.sba_last_error.restype = ctypes.c_char_p
    lib.sba_nsa_select_host_workspace_size.argtypes = [ci] * 10
    lib.sba_nsa_select_host_workspace_size.restype = csz
    lib.sba_nsa_select_fwd_host.argtypes = [vp, vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, ci, ci,
                                            ci, ci, cf, ci, vp, f32p, vp, csz, vp]
    lib.sba_nsa_select_fwd_host.restype = ci
    lib.sba_nsa_select_fwd.argtypes = [vp, vp, vp, vp, i32p, i32p, ci, ci, i32p, ci, ci, ci, ci, ci,
                                       ci, ci, ci, cf, ci, vp, f32p, vp]
    lib.sba_nsa_select_fwd.restype = ci
    lib.sba_sparse_mask_bounds.argtypes = [i32p, i32p, i32p, i32p, ci, ci, ci, ci, ci, ci, ci, ci,
                                           ci, i32p, i32p, i32p, i32p, vp]
    lib.sba_sparse_mask_bounds.restype = ci
    lib.sba_sparse_mask_dkdv_bounds.argtypes = [i32p, i32p, i32p, i32p, ci, ci, ci, ci, ci, ci, ci,
                                                ci, ci, i32p, i32p, i32p, i32p, vp]
    lib.sba_sparse_mask_dkdv_bounds.restype = ci
    lib.sba_blocksparse_attn_fwd.argtypes = [vp, vp, vp, i32p, i32p, i32p, i32p, i32p, i32p, i32p,
                                             i32p, ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, cf,
                                             vp, f32p, vp]
    lib.sba_blocksparse_attn_fwd.restype = ci
    lib.sba_ragged_decode_workspace_size.argtypes = [ci, ci, ci, ci, ci]
    lib.sba_ragged_decode_workspace_size.restype = csz
    lib.sba_ragged_decode_fwd.argtypes = [vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, cf, ci, ci,
                                          cf, f32p, ci, ci, vp, f32p, vp, csz, vp]
    lib.sba_ragged_decode_fwd.restype = ci
    lib.sba_ragged_decode_fwd_noalloc.argtypes = [vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, cf,
                                                  ci, ci, cf, f32p, ci, ci, vp, f32p, vp]
    lib.sba_ragged_decode_fwd_noalloc.restype = ci
    lib.sba_ragged_flash_attention_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci, ci]
    lib.sba_ragged_flash_attention_workspace_size.restype = csz
    lib.sba_ragged_flash_attention_fwd.argtypes = [vp, vp, vp, i32p, i32p, ci, ci, ci, ci, ci, ci,
                                                   cf, ci, ci, cf, f32p, ci, ci, vp, f32p, vp,
                                                   csz, vp]
    lib.sba_ragged_flash_attention_fwd.restype = ci
    lib.sba_l2_read_probe.argtypes = [vp, csz, ci, vp, vp]
    lib.sba_l2_read_probe.restype = ci
    lib.sba_check_error.argtypes = [vp]
    lib.sba_check_error.restype = ci
    lib.sba_nsa_select_bwd_workspace_size.argtypes = [ci] * 6
    lib.sba_nsa_select_bwd_workspace_size.restype = csz
    lib.sba_nsa_select_bwd.argtypes = [vp, vp, vp, vp, f32p, vp, i32p, i32p, ci, ci, i32p, ci, ci, ci,
                                       ci, ci, ci, ci, ci, cf, ci, vp, vp, vp, vp, csz, vp]
    lib.sba_nsa_select_bwd.restype = ci
    lib.sba_set_wait_timeout_cycles.argtypes = [ctypes.c_longlong]
    lib.sba_set_wait_timeout_cycles.restype = ci
    lib.sba_get_wait_timeout_cycles.argtypes = []
    lib.sba_get_wait_timeout_cycles.restype = ctypes.c_longlong
    if path == _build.LIB_PATH:
        _lib = lib
    return lib


def _check(code):
    if code != 0:
        raise SBAError(code, load_library().sba_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*tensors):
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libsba works on CUDA tensors only (no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _call(dev, fn, *args):
    """Call a library entry point with ``dev`` current: the library launches on the
    current device (and looks up per-device state there), so the stream's device must
    be the current one."""
    with torch.cuda.device(dev):
        _check(fn(*args))


def _i32(t, name):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return t


def nsa_select_fwd(q, k, v, block_indices, block_counts, block_size, *, cu_seqlens=None,
                   causal=True, softmax_scale=None, g_slc=None, out=None, lse=None,
                   return_lse=True):
    """Selection-branch NSA forward.  q [B,T,Hq,D], k/v [B,T,Hkv,D] (bf16 or fp32),
    block_indices int32 [B,T,Hkv,S], block_counts int or int32 [B,T,Hkv], cu_seqlens
    int32 [N+1] or None, g_slc [B,T,Hq] (q's dtype) gate of the output rows or None.
    Returns (out, lse)."""
    lib = load_library()
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    S = block_indices.shape[-1]
    counts_t = None if isinstance(block_counts, int) else _i32(block_counts, "block_counts")
    dev = _dev(q, k, v, block_indices, counts_t, cu_seqlens)
    _i32(block_indices, "block_indices")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    dtype = {torch.bfloat16: SBA_BF16, torch.float32: SBA_F32}.get(q.dtype)
    if dtype is None:
        raise TypeError("q must be bfloat16 or float32")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=dev)
    num_seqs = 0
    if cu_seqlens is not None:
        _i32(cu_seqlens, "cu_seqlens")
        num_seqs = cu_seqlens.numel() - 1
    if g_slc is not None:
        if g_slc.dtype != q.dtype or tuple(g_slc.shape) != (B, T, Hq) or not g_slc.is_contiguous():
            raise ValueError("g_slc must be a contiguous [B, T, Hq] tensor of q's dtype")
        _dev(q, g_slc)
    _call(dev, lib.sba_nsa_select_fwd,
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_slc), _ptr(block_indices), _ptr(counts_t),
        int(block_counts) if counts_t is None else 0, S, _ptr(cu_seqlens), num_seqs,
        B, T, Hq, Hkv, D, int(block_size), int(bool(causal)),
        float(softmax_scale or 0.0), dtype, _ptr(out), _ptr(lse), _stream(dev))
    return out, lse


def nsa_select_bwd_workspace_size(B, T, Hq, Hkv, S, num_seqs=0) -> int:
    return int(load_library().sba_nsa_select_bwd_workspace_size(B, T, Hq, Hkv, S, num_seqs))


def nsa_select_bwd(q, k, v, out, lse, d_out, block_indices, block_counts, block_size, *,
                   cu_seqlens=None, causal=True, softmax_scale=None, dq=None, dk=None, dv=None,
                   workspace=None):
    """Gradients (dq, dk, dv) of the selection forward (bf16): ``out`` and ``lse`` are
    the forward's results for the same arguments, ``d_out`` the gradient of the loss
    with respect to ``out``."""
    lib = load_library()
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    S = block_indices.shape[-1]
    counts_t = None if isinstance(block_counts, int) else _i32(block_counts, "block_counts")
    dev = _dev(q, k, v, out, lse, d_out, block_indices, counts_t, cu_seqlens, dq, dk, dv, workspace)
    _i32(block_indices, "block_indices")
    if any(t.dtype != q.dtype for t in (k, v, out, d_out)):
        raise TypeError("q, k, v, out and d_out must share a dtype")
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    dtype = {torch.bfloat16: SBA_BF16, torch.float32: SBA_F32}.get(q.dtype)
    if dtype is None:
        raise TypeError("q must be bfloat16 or float32")
    num_seqs = 0
    if cu_seqlens is not None:
        _i32(cu_seqlens, "cu_seqlens")
        num_seqs = cu_seqlens.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        need = nsa_select_bwd_workspace_size(B, T, Hq, Hkv, S, num_seqs)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _call(dev, lib.sba_nsa_select_bwd,
          _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(d_out), _ptr(block_indices),
          _ptr(counts_t), int(block_counts) if counts_t is None else 0, S, _ptr(cu_seqlens),
          num_seqs, B, T, Hq, Hkv, D, int(block_size), int(bool(causal)),
          float(softmax_scale or 0.0), dtype, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(dev))
    return dq, dk, dv


def nsa_select_host_workspace_size(B, T, Hq, Hkv, D, S, dtype=SBA_BF16, has_counts=True,
                                   has_gate=False, has_lse=True) -> int:
    return int(load_library().sba_nsa_select_host_workspace_size(
        B, T, Hq, Hkv, D, S, dtype, int(bool(has_counts)), int(bool(has_gate)), int(bool(has_lse))))


def nsa_select_fwd_host(q, k, v, block_indices, block_counts, block_size, *, causal=True,
                        softmax_scale=None, g_slc=None, out=None, lse=None, return_lse=True,
                        workspace=None, device=None):
    """Selection-branch NSA forward on CPU tensors (pinned for asynchronous copies):
    the library stages them in a device workspace, overlapping the copies of batch-row
    chunks with the computation.  Fixed-length rows only.  Returns (out, lse) as CPU
    tensors; they are complete when the current stream of ``device`` is."""
    lib = load_library()
    for t in (q, k, v, block_indices, g_slc, out, lse,
              None if isinstance(block_counts, int) else block_counts):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("host entry point: tensors must be contiguous CPU tensors")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    S = block_indices.shape[-1]
    counts_t = None if isinstance(block_counts, int) else block_counts
    if block_indices.dtype != torch.int32 or (counts_t is not None and counts_t.dtype != torch.int32):
        raise TypeError("block_indices / block_counts must be int32")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    dtype = {torch.bfloat16: SBA_BF16, torch.float32: SBA_F32}.get(q.dtype)
    if dtype is None:
        raise TypeError("q must be bfloat16 or float32")
    if g_slc is not None and (g_slc.dtype != q.dtype or tuple(g_slc.shape) != (B, T, Hq)):
        raise ValueError("g_slc must be a [B, T, Hq] tensor of q's dtype")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if lse is None and return_lse:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, pin_memory=pin)
    need = nsa_select_host_workspace_size(B, T, Hq, Hkv, D, S, dtype, counts_t is not None,
                                          g_slc is not None, lse is not None)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _call(dev, lib.sba_nsa_select_fwd_host,
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_slc), _ptr(block_indices), _ptr(counts_t),
        int(block_counts) if counts_t is None else 0, S, B, T, Hq, Hkv, D, int(block_size),
        int(bool(causal)), float(softmax_scale or 0.0), dtype, _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(dev))
    return out, lse


def sparse_mask_bounds(q_positions, q_segment_ids, kv_positions, kv_segment_ids, q_blocksize,
                       kv_blocksize, *, causal=True, window_left=-1, window_right=-1,
                       padding_segment_id=-1, calculate_dkdv_mask=False):
    """SparseMask bounds: returns (lower, upper, lower_full, upper_full), each int32
    [B, 1, ceil(Tq / q_blocksize)] (forward / dQ: key/value block ranges per query
    block), or with ``calculate_dkdv_mask`` [B, 1, ceil(Tkv / kv_blocksize)] (dK/dV:
    query block ranges per key/value block)."""
    lib = load_library()
    for name, t in (("q_positions", q_positions), ("q_segment_ids", q_segment_ids),
                    ("kv_positions", kv_positions), ("kv_segment_ids", kv_segment_ids)):
        _i32(t, name)
    dev = _dev(q_positions, q_segment_ids, kv_positions, kv_segment_ids)
    B, Tq = q_positions.shape
    Tkv = kv_positions.shape[1]
    nb = -(-Tkv // kv_blocksize) if calculate_dkdv_mask else -(-Tq // q_blocksize)
    outs = [torch.empty((B, 1, nb), dtype=torch.int32, device=dev) for _ in range(4)]
    fn = lib.sba_sparse_mask_dkdv_bounds if calculate_dkdv_mask else lib.sba_sparse_mask_bounds
    _call(dev, fn,
        _ptr(q_positions), _ptr(q_segment_ids), _ptr(kv_positions), _ptr(kv_segment_ids),
        B, Tq, Tkv, int(q_blocksize), int(kv_blocksize), int(bool(causal)), int(window_left),
        int(window_right), int(padding_segment_id), *[_ptr(o) for o in outs], _stream(dev))
    return tuple(outs)


def blocksparse_attn_fwd(q, k, v, q_positions, q_segment_ids, kv_positions, kv_segment_ids,
                         lower, upper, lower_full, upper_full, q_blocksize, kv_blocksize, *,
                         causal=True, window_left=-1, window_right=-1, padding_segment_id=-1,
                         softmax_scale=None, out=None, lse=None, return_lse=True):
    """Attention restricted by SparseMask bounds (bf16).  Returns (out, lse)."""
    lib = load_library()
    ints = (q_positions, q_segment_ids, kv_positions, kv_segment_ids, lower, upper, lower_full,
            upper_full)
    for t in ints:
        _i32(t, "positions/segments/bounds")
    dev = _dev(q, k, v, *ints)
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bfloat16")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=dev)
    _call(dev, lib.sba_blocksparse_attn_fwd,
        _ptr(q), _ptr(k), _ptr(v), *[_ptr(t) for t in ints], B, T, Hq, Hkv, D,
        int(q_blocksize), int(kv_blocksize), int(bool(causal)), int(window_left),
        int(window_right), int(padding_segment_id), float(softmax_scale or 0.0), _ptr(out),
        _ptr(lse), _stream(dev))
    return out, lse


def ragged_decode_workspace_size(B, Hq, S, D, window_left=-1) -> int:
    return int(load_library().sba_ragged_decode_workspace_size(B, Hq, S, D, window_left))


def ragged_decode_fwd(q, k, v, sequence_start, sequence_end, *, softmax_scale=None,
                      window_left=-1, window_right=-1, logits_soft_cap=None, sink_bias=None,
                      out=None, lse=None, workspace=None, return_lse=True):
    """Ragged single-token decode (bf16).  q [B,Hq,D], k/v [B,S,Hkv,D], sequence_start /
    sequence_end int32 [B], sink_bias fp32 [Hq, num_sinks] or [num_sinks].
    Returns (out, lse)."""
    lib = load_library()
    _i32(sequence_start, "sequence_start")
    _i32(sequence_end, "sequence_end")
    dev = _dev(q, k, v, sequence_start, sequence_end, sink_bias, workspace)
    B, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    num_sinks, per_head = 0, 0
    if sink_bias is not None:
        if sink_bias.dtype != torch.float32:
            raise TypeError("sink_bias must be float32")
        num_sinks = sink_bias.shape[-1]
        per_head = int(sink_bias.dim() == 2)
    need = ragged_decode_workspace_size(B, Hq, S, D, window_left)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _call(dev, lib.sba_ragged_decode_fwd,
        _ptr(q), _ptr(k), _ptr(v), _ptr(sequence_start), _ptr(sequence_end), B, Hq, Hkv, S, D,
        float(softmax_scale or 0.0), int(window_left), int(window_right),
        float(logits_soft_cap or 0.0), _ptr(sink_bias), num_sinks, per_head, _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(dev))
    return out, lse


def ragged_decode_fwd_noalloc(q, k, v, sequence_start, sequence_end, *, softmax_scale=None,
                              window_left=-1, window_right=-1, logits_soft_cap=None,
                              sink_bias=None, out=None, lse=None, return_lse=True):
    """ragged_decode_fwd for callers that cannot allocate device scratch: the split
    partials use a fixed 16 MiB array inside the library (shared by every call on a
    device, so calls that overlap on the GPU race).  Outputs may be passed in."""
    lib = load_library()
    _i32(sequence_start, "sequence_start")
    _i32(sequence_end, "sequence_end")
    dev = _dev(q, k, v, sequence_start, sequence_end, sink_bias, out, lse)
    B, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    num_sinks, per_head = 0, 0
    if sink_bias is not None:
        if sink_bias.dtype != torch.float32:
            raise TypeError("sink_bias must be float32")
        num_sinks = sink_bias.shape[-1]
        per_head = int(sink_bias.dim() == 2)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _call(dev, lib.sba_ragged_decode_fwd_noalloc,
        _ptr(q), _ptr(k), _ptr(v), _ptr(sequence_start), _ptr(sequence_end), B, Hq, Hkv, S, D,
        float(softmax_scale or 0.0), int(window_left), int(window_right),
        float(logits_soft_cap or 0.0), _ptr(sink_bias), num_sinks, per_head, _ptr(out), _ptr(lse),
        _stream(dev))
    return out, lse


def ragged_flash_attention_workspace_size(B, Q, Hq, S, D, window_left=-1, window_right=-1) -> int:
    return int(load_library().sba_ragged_flash_attention_workspace_size(
        B, Q, Hq, S, D, window_left, window_right))


def ragged_flash_attention_fwd(q, k, v, sequence_start, sequence_end, *, softmax_scale=None,
                               window_left=-1, window_right=-1, logits_soft_cap=None,
                               sink_bias=None, out=None, lse=None, workspace=None,
                               return_lse=True):
    """Ragged multi-query attention (bf16).  q [B,Q,Hq,D], k/v [B,S,Hkv,D],
    sequence_start / sequence_end int32 [B] (query i of a row sits at end - Q + i),
    sink_bias fp32 [Hq, num_sinks] or [num_sinks].  Returns (out [B,Q,Hq,D],
    lse [B,Q,Hq])."""
    lib = load_library()
    _i32(sequence_start, "sequence_start")
    _i32(sequence_end, "sequence_end")
    dev = _dev(q, k, v, sequence_start, sequence_end, sink_bias, workspace, out, lse)
    B, Q, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    num_sinks, per_head = 0, 0
    if sink_bias is not None:
        if sink_bias.dtype != torch.float32:
            raise TypeError("sink_bias must be float32")
        num_sinks = sink_bias.shape[-1]
        per_head = int(sink_bias.dim() == 2)
    need = ragged_flash_attention_workspace_size(B, Q, Hq, S, D, window_left, window_right)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=dev)
    _call(dev, lib.sba_ragged_flash_attention_fwd,
        _ptr(q), _ptr(k), _ptr(v), _ptr(sequence_start), _ptr(sequence_end), B, Q, Hq, Hkv, S, D,
        float(softmax_scale or 0.0), int(window_left), int(window_right),
        float(logits_soft_cap or 0.0), _ptr(sink_bias), num_sinks, per_head, _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(dev))
    return out, lse


def l2_read_probe(buf, reps, sink):
    """Measurement helper (not part of the method): read ``buf`` (a CUDA tensor) ``reps``
    times with 16-byte L1-bypassing loads on every SM; XOR of the data into ``sink``
    (an int32 CUDA tensor of one element)."""
    _dev(buf, sink)
    _check(load_library().sba_l2_read_probe(_ptr(buf), buf.numel() * buf.element_size(), int(reps),
                                            _ptr(sink), _stream(buf.device)))


def check_error(device=None):
    """Synchronise the current stream and raise if a kernel flagged an error."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(load_library().sba_check_error(_stream(dev)))


def set_wait_timeout_cycles(cycles):
    """Limit (SM cycles) on every internal wait of the warp-specialised kernels launched
    from now on; 0 restores the default (about two seconds).  A launch whose wait runs
    past it returns early and check_error() raises SBAError with code -4 (timeout)."""
    _check(load_library().sba_set_wait_timeout_cycles(int(cycles)))


def get_wait_timeout_cycles() -> int:
    return int(load_library().sba_get_wait_timeout_cycles())
