"""Python binding of libpa.so: paged-KV GQA attention for one GB300 (sm_103a).

This module only marshals arguments: it takes torch CUDA tensors, checks their dtype,
device and layout, and passes raw pointers, sizes and the current CUDA stream to the
C ABI declared in include/pa.h.  Every step of the computation runs in the library's
CUDA kernels.  There is no CPU or PyTorch fallback: if libpa.so is missing or cannot be
loaded, every call raises.

Functions (names follow the C ABI):
    slot_mapping(positions, block_table, block_size, seq_idx=None)    -> int64 slots
    decode_input_prep(positions, block_tables, block_sizes, sampled_ids=None)
                                                                      -> step inputs
    reshape_and_cache(key, value, k_cache, v_cache, slot_mapping)     (in place)
    decode_workspace_size(...), decode(q, k_cache, v_cache, block_table, seq_lens, ...)
    prefill_workspace_size(...), prefill_chunk(q, k_cache, v_cache, block_table, q_start,
                                               causal, scale, workspace=None)
    prefill_varlen_workspace_size(...), prefill_varlen(q, k_cache, v_cache, block_table,
                                               cu_seqlens_q, seq_lens_k, causal, scale)
    prefill_plan(q_len, q_start, causal, num_q_heads, block_size, num_ctas)  (host only)
    device_errors(clear=True)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = ["load", "build", "slot_mapping", "decode_input_prep", "reshape_and_cache",
           "decode_workspace_size",
           "decode", "decode_append", "prefill_chunk", "prefill_varlen", "prefill_plan",
           "prefill_workspace_size", "prefill_varlen_workspace_size", "prefill_plan_pieces", "device_errors", "set_kernel_events", "build_info", "PAError",
           "DEVERR_PAGE", "DEVERR_SEQLEN", "DEVERR_SLOT", "DEVERR_TIMEOUT", "DEVERR_POSITION", "DEVERR_LAYOUT",
           "LIB_PATH"]

LIB_PATH = _build.LIB
DEVERR_PAGE, DEVERR_SEQLEN, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_POSITION = 1, 2, 4, 8, 16
DEVERR_LAYOUT = 32
ERR_TIMEOUT = 4  # PA_ERR_TIMEOUT

_lib = None
_lock = threading.Lock()


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = _lib.pa_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {name}")


def build(force: bool = False) -> str:
    """Compile libpa.so (nvcc, sm_103a) in-tree."""
    return _build.build(force=force)


def load():
    """Load libpa.so and declare the C signatures.  Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        sig = {
            "pa_slot_mapping": ([P, P, P, i32, i64, i32, i32, i32, P, P], i32),
            "pa_reshape_and_cache": ([P, P, P, P, i64, i64, P, i32, i32, i32, i32, P], i32),
            "pa_decode_input_prep": ([P, P, P, P, P, i32, i32, P, P, P, P, P, P], i32),
            "pa_decode_workspace_size": ([i32, i32, i32, i32, i32, i32], sz),
            "pa_decode": ([P, P, P, i64, i64, P, i64, P, i32, i32, i32, i32, i32, i32, f32, P, P,
                           sz, P, P, P, P], i32),
            "pa_decode_append": ([P, P, P, i64, i64, P, i64, P, i32, i32, i32, i32, i32, i32, f32,
                                  P, P, sz, P, P, P, P], i32),
            "pa_prefill_workspace_size": ([i32, i32, i32, i32, i32, i32, i32], sz),
            "pa_prefill_chunk": ([P, P, P, i64, i64, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                  P, P, sz, P], i32),
            "pa_prefill_varlen_workspace_size": ([P, P, i32, i32, i32, i32, i32, i32], sz),
            "pa_prefill_plan": ([i32, i32, i32, i32, i32, i32, i32, P, P, P], i32),
            "pa_prefill_plan_pieces": ([i32, i32, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P,
                                        P,
                                        P], i32),
            "pa_prefill_varlen": ([P, P, P, i64, i64, P, i64, P, P, i32, i32, i32, i32, i32,
                                   i32, f32, P, P, sz, P], i32),
            "pa_copy": ([P, P, sz, P], i32),
            "pa_get_device_errors": ([ctypes.POINTER(ctypes.c_uint), i32, P], i32),
            "pa_set_kernel_events": ([P, P], i32),
            "pa_status_string": ([i32], ctypes.c_char_p),
            "pa_build_info": ([], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _check_out(out, like):
    """A caller's decode output: BF16, contiguous, shaped like q, on the GPU or in
    page-locked host memory (which the combine kernel writes directly)."""
    if not isinstance(out, torch.Tensor) or not (out.is_cuda or out.is_pinned()):
        raise TypeError("out must be a CUDA tensor or a pinned host tensor")
    if out.dtype != torch.bfloat16 or out.shape != like.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous BF16 tensor shaped like q")


def _check_cache(k_cache, v_cache):
    for n, c in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(c, n, torch.bfloat16, 4)
        if c.stride(3) != 1 or c.stride(2) != c.shape[3] or c.stride(1) != c.shape[2] * c.shape[3]:
            raise ValueError(f"{n}: each page must be a contiguous [BS, Hkv, D] block")
    if k_cache.shape != v_cache.shape or k_cache.stride(0) != v_cache.stride(0):
        raise ValueError("k_cache and v_cache must have the same shape and page stride")
    return k_cache.stride(0)


def _raise(rc, where):
    if rc != 0:
        raise PAError(rc, where)


def build_info() -> str:
    return load().pa_build_info().decode()


def slot_mapping(positions, block_table, block_size, seq_idx=None, max_blocks=None, out=None):
    """int64 slot of each position (see pa_slot_mapping)."""
    lib = load()
    _check(positions, "positions", torch.int32, 1)
    _check(block_table, "block_table", torch.int32)
    bt = block_table if block_table.dim() == 2 else block_table.view(1, -1)
    if bt.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    if seq_idx is not None:
        _check(seq_idx, "seq_idx", torch.int32, 1)
    n = positions.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.int64, device=positions.device)
    mb = bt.shape[1] if max_blocks is None else int(max_blocks)
    _raise(lib.pa_slot_mapping(_ptr(positions.contiguous()), _ptr(seq_idx), _ptr(bt),
                               bt.shape[0], bt.stride(0), mb, n, int(block_size), _ptr(out),
                               _stream()), "pa_slot_mapping")
    return out


def decode_input_prep(positions, block_tables, block_sizes, sampled_ids=None, max_blocks=None,
                      out=None):
    """One decode step's inputs for several KV-cache groups in one launch (see
    pa_decode_input_prep).  block_tables / block_sizes: one int32 [S, n] table and one
    block size per group.  Returns a dict with seq_lens, query_start_loc, input_ids (when
    sampled_ids is given) and slot_mappings (a list, one int64 [S] tensor per group);
    `out` may pass that dict back in to reuse its tensors."""
    lib = load()
    _check(positions, "positions", torch.int32, 1)
    S, G = positions.shape[0], len(block_tables)
    if len(block_sizes) != G or not 1 <= G <= 8:
        raise ValueError("one block size per group, 1..8 groups")
    dev = positions.device
    if out is None:
        out = {"seq_lens": torch.empty(S, dtype=torch.int32, device=dev),
               "query_start_loc": torch.empty(S + 1, dtype=torch.int32, device=dev),
               "slot_mappings": [torch.empty(S, dtype=torch.int64, device=dev) for _ in range(G)]}
        if sampled_ids is not None:
            out["input_ids"] = torch.empty(S, dtype=torch.int32, device=dev)
    tables = []
    for t in block_tables:
        _check(t, "block_table", torch.int32, 2)
        if t.shape[0] < S or t.stride(1) != 1:
            raise ValueError("block tables: one row per sequence, contiguous rows")
        tables.append(t)
    mb = max_blocks if max_blocks is not None else [t.shape[1] for t in tables]
    arr = lambda ctype, vals: (ctype * G)(*vals)
    bt_ptrs = arr(ctypes.c_void_p, [t.data_ptr() for t in tables])
    sm_ptrs = arr(ctypes.c_void_p, [m.data_ptr() for m in out["slot_mappings"]])
    strides = arr(ctypes.c_int64, [t.stride(0) for t in tables])
    mbs = arr(ctypes.c_int, [int(x) for x in mb])
    bss = arr(ctypes.c_int, [int(x) for x in block_sizes])
    sid = None
    if sampled_ids is not None:
        _check(sampled_ids, "sampled_ids", torch.int32, 1)
        sid = sampled_ids.contiguous()
    _raise(lib.pa_decode_input_prep(_ptr(positions.contiguous()), _ptr(sid),
                                    _ptr(out.get("input_ids")), _ptr(out["seq_lens"]),
                                    _ptr(out["query_start_loc"]), S, G, bt_ptrs, strides, mbs,
                                    bss, sm_ptrs, _stream()), "pa_decode_input_prep")
    return out


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping_):
    """Write key/value [T, Hkv, D] into the caches at slot_mapping_ (in place)."""
    lib = load()
    _check(key, "key", torch.bfloat16, 3)
    _check(value, "value", torch.bfloat16, 3)
    _check(slot_mapping_, "slot_mapping", torch.int64, 1)
    ps = _check_cache(k_cache, v_cache)
    key, value = key.contiguous(), value.contiguous()
    T, hkv, d = key.shape
    _raise(lib.pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), ps,
                                    k_cache.shape[0], _ptr(slot_mapping_), T, hkv, d,
                                    k_cache.shape[1], _stream()), "pa_reshape_and_cache")


def copy(dst, src):
    """Copy src into dst (same byte size, both contiguous) with a kernel on the current
    stream (see pa_copy).  Each tensor may live on the GPU or in pinned host memory."""
    lib = load()
    for t, nm in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{nm} must be a CUDA tensor or pinned host memory")
    nb = dst.numel() * dst.element_size()
    if nb != src.numel() * src.element_size():
        raise ValueError("dst and src differ in size")
    _raise(lib.pa_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nb,
                       _stream()), "pa_copy")
    return dst


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                          max_seq_len) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               block_size, max_seq_len))


def decode(q, k_cache, v_cache, block_table, seq_lens, scale, max_seq_len, out=None,
           workspace=None, new_k=None, new_v=None, new_slots=None):
    """q=1 paged decode (see pa_decode).  Returns out [S, Hq, D] BF16."""
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    ps = _check_cache(k_cache, v_cache)
    q = q.contiguous()
    S, hq, d = q.shape
    _, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_out(out, q)
    need = decode_workspace_size(S, hq, hkv, d, bs, max_seq_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if new_k is not None:
        new_k, new_v = new_k.contiguous(), new_v.contiguous()
    _raise(lib.pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), ps, k_cache.shape[0],
                         _ptr(block_table), block_table.stride(0), _ptr(seq_lens), S,
                         int(max_seq_len), hq, hkv, d, bs, float(scale), _ptr(out),
                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _ptr(new_k), _ptr(new_v), _ptr(new_slots), _stream()), "pa_decode")
    return out


def decode_append(q, k_cache, v_cache, block_table, seq_lens, scale, max_seq_len, new_k, new_v,
                  out=None, workspace=None, slot_mapping=None):
    """Decode step that appends each sequence's newest token (position seq_lens[s] - 1)
    from new_k / new_v at the slot the kernel derives from the block table, then attends
    (see pa_decode_append).  slot_mapping, if given (int64 [S]), receives those slots.
    Returns out [S, Hq, D] BF16."""
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(new_k, "new_k", torch.bfloat16, 3)
    _check(new_v, "new_v", torch.bfloat16, 3)
    if slot_mapping is not None:
        _check(slot_mapping, "slot_mapping", torch.int64, 1)
        if not slot_mapping.is_contiguous() or slot_mapping.numel() < q.shape[0]:
            raise ValueError("slot_mapping must be a contiguous int64 tensor of num_seqs entries")
    ps = _check_cache(k_cache, v_cache)
    q = q.contiguous()
    new_k, new_v = new_k.contiguous(), new_v.contiguous()
    S, hq, d = q.shape
    _, bs, hkv, _ = k_cache.shape
    if new_k.shape != (S, hkv, d) or new_v.shape != (S, hkv, d):
        raise ValueError("new_k / new_v must be [num_seqs, num_kv_heads, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_out(out, q)
    need = decode_workspace_size(S, hq, hkv, d, bs, max_seq_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _raise(lib.pa_decode_append(_ptr(q), _ptr(k_cache), _ptr(v_cache), ps, k_cache.shape[0],
                                _ptr(block_table), block_table.stride(0), _ptr(seq_lens), S,
                                int(max_seq_len), hq, hkv, d, bs, float(scale), _ptr(out),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(new_k), _ptr(new_v), _ptr(slot_mapping), _stream()),
           "pa_decode_append")
    return out


def prefill_workspace_size(q_len, q_start, causal, num_q_heads, num_kv_heads, head_dim,
                           block_size):
    """Bytes of workspace with which pa_prefill_chunk may split items (0: none would pay)."""
    return int(load().pa_prefill_workspace_size(int(q_len), int(q_start), int(bool(causal)),
                                                num_q_heads, num_kv_heads, head_dim,
                                                block_size))


def _workspace_arg(workspace, need, device):
    """(pointer, bytes) of a caller's workspace, or of a fresh one of `need` bytes."""
    if workspace is None:
        if need == 0:
            return None, 0
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    return workspace, workspace.numel() * workspace.element_size()


def prefill_chunk(q, k_cache, v_cache, block_table, q_start, causal, scale, out=None,
                  workspace=None):
    """Causal (or full) chunk attention of one sequence (see pa_prefill_chunk).  Without a
    workspace, one of pa_prefill_workspace_size bytes is allocated for the call."""
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(block_table, "block_table", torch.int32)
    ps = _check_cache(k_cache, v_cache)
    q = q.contiguous()
    bt = block_table.reshape(-1).contiguous()
    q_len, hq, d = q.shape
    _, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        need = prefill_workspace_size(q_len, q_start, causal, hq, hkv, d, bs)
    ws, ws_bytes = _workspace_arg(workspace, need if workspace is None else 0, q.device)
    _raise(lib.pa_prefill_chunk(_ptr(q), _ptr(k_cache), _ptr(v_cache), ps, k_cache.shape[0],
                                _ptr(bt), q_len, int(q_start), int(bool(causal)), hq, hkv, d,
                                bs, float(scale), _ptr(out), _ptr(ws), ws_bytes, _stream()),
           "pa_prefill_chunk")
    return out


def prefill_varlen_workspace_size(cu_seqlens_q, seq_lens_k, causal, num_q_heads, num_kv_heads,
                                  head_dim, block_size):
    """Bytes of workspace with which pa_prefill_varlen may split items."""
    B = len(seq_lens_k)
    cu = (ctypes.c_int32 * (B + 1))(*[int(x) for x in cu_seqlens_q])
    sk = (ctypes.c_int32 * max(B, 1))(*[int(x) for x in seq_lens_k])
    return int(load().pa_prefill_varlen_workspace_size(cu, sk, B, int(bool(causal)),
                                                       num_q_heads, num_kv_heads, head_dim,
                                                       block_size))


def prefill_varlen(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, causal, scale,
                   out=None, workspace=None):
    """Chunks of several sequences stacked row-wise in q (see pa_prefill_varlen).
    cu_seqlens_q and seq_lens_k are host sequences of ints (lists or arrays).  Without a
    workspace, one of pa_prefill_varlen_workspace_size bytes is allocated for the call."""
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(block_table, "block_table", torch.int32, 2)
    ps = _check_cache(k_cache, v_cache)
    q = q.contiguous()
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    B = len(seq_lens_k)
    if len(cu_seqlens_q) != B + 1 or int(cu_seqlens_q[-1]) != q.shape[0]:
        raise ValueError("cu_seqlens_q: num_seqs + 1 offsets ending at q's row count")
    cu = (ctypes.c_int32 * (B + 1))(*[int(x) for x in cu_seqlens_q])
    sk = (ctypes.c_int32 * max(B, 1))(*[int(x) for x in seq_lens_k])
    _, hq, d = q.shape
    _, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    need = 0
    if workspace is None:
        need = int(lib.pa_prefill_varlen_workspace_size(cu, sk, B, int(bool(causal)), hq, hkv,
                                                        d, bs))
    ws, ws_bytes = _workspace_arg(workspace, need, q.device)
    _raise(lib.pa_prefill_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), ps, k_cache.shape[0],
                                 _ptr(block_table), block_table.stride(0), cu, sk, B,
                                 int(bool(causal)), hq, hkv, d, bs, float(scale), _ptr(out),
                                 _ptr(ws), ws_bytes, _stream()), "pa_prefill_varlen")
    return out


def prefill_plan(q_len, q_start, causal, num_q_heads, num_kv_heads, block_size, num_ctas):
    """The static work assignment of prefill_chunk (see pa_prefill_plan): returns
    (cta_of_item, max_cost) with cta_of_item a list indexed by work item."""
    lib = load()
    n = ctypes.c_int(0)
    mc = ctypes.c_int(0)
    args = (int(q_len), int(q_start), int(bool(causal)), int(num_q_heads), int(num_kv_heads),
            int(block_size), int(num_ctas))
    _raise(lib.pa_prefill_plan(*args, None, ctypes.byref(n), None), "pa_prefill_plan")
    cta = (ctypes.c_int32 * n.value)()
    _raise(lib.pa_prefill_plan(*args, cta, ctypes.byref(n), ctypes.byref(mc)), "pa_prefill_plan")
    return list(cta), mc.value


def prefill_plan_pieces(q_len, q_start, causal, num_q_heads, num_kv_heads, block_size,
                        num_ctas, max_pieces=480):
    """The plan used with a workspace (host only, see pa_prefill_plan_pieces): returns
    (cta_of_item with -1 for split items, [(item, tile_begin, tile_end, cta), ...], max_cost)."""
    lib = load()
    ni, npc, mc = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    items = (ctypes.c_int32 * (-(-int(q_len) // 128) * num_q_heads))()  # an upper bound
    arrs = [(ctypes.c_int32 * max(1, max_pieces))() for _ in range(4)]
    _raise(lib.pa_prefill_plan_pieces(int(q_len), int(q_start), int(bool(causal)), num_q_heads,
                                      num_kv_heads, block_size, num_ctas, max_pieces, items,
                                      *arrs, ctypes.byref(ni), ctypes.byref(npc),
                                      ctypes.byref(mc)),
           "pa_prefill_plan_pieces")
    pieces = [(arrs[0][p], arrs[1][p], arrs[2][p], arrs[3][p]) for p in range(npc.value)]
    return list(items)[:ni.value], pieces, mc.value


def set_kernel_events(start, stop):
    """Measurement hook: the next decode / prefill_chunk call records these
    torch.cuda.Event objects around its main kernel (see pa_set_kernel_events)."""
    lib = load()
    for e in (start, stop):
        if not e.cuda_event:          # torch creates the CUDA event on first record
            e.record()
    _raise(lib.pa_set_kernel_events(ctypes.c_void_p(start.cuda_event),
                                    ctypes.c_void_p(stop.cuda_event)), "pa_set_kernel_events")


def device_errors(clear: bool = True) -> int:
    """Waits for the current stream and returns (and by default clears) the error bits.
    A bounded wait that ran out shows as DEVERR_TIMEOUT among them (the C call then
    returns PA_ERR_TIMEOUT, which is not raised here)."""
    lib = load()
    v = ctypes.c_uint(0)
    rc = lib.pa_get_device_errors(ctypes.byref(v), int(clear), _stream())
    if rc != ERR_TIMEOUT:
        _raise(rc, "pa_get_device_errors")
    return int(v.value)
