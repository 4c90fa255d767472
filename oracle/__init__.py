"""fp64 CPU oracle for paged GQA attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The product library never calls it and shares
no code with it: the arithmetic lives in ``pa_oracle.c`` (plain loops in fp64), and this
module only compiles that file with gcc and marshals numpy arrays into it.

BF16 tensors cross this boundary as their raw 16-bit patterns (``numpy.uint16``); the
C code decodes them to their exact values itself.

Function -> passage it follows (pages cited by post and section):
  slot_mapping       -- input-prep post §3.2 (slot = block_table[pos // bs] * bs + pos % bs)
  decode_input_prep  -- input-prep post §2, §4, §5: seq_lens = position + 1 (0 for padding),
                        query_start_loc = running count of query rows (none for padding),
                        input_ids from the sampled tokens, one slot mapping per KV group
  reshape_and_cache  -- page832 post §4 (cache layout [pages, BS, Hkv, D]) and the slot above
  attend_row         -- page832 post §1 (address translation) and §5 (score = q.k * scale,
                        softmax, weighted V), written as the exact, non-online definition
  decode             -- attend_row over seq_lens[i] keys per sequence, head h -> kv head h // G
  prefill_rows       -- page832 post §6: causal chunk, row i at position q_start + i sees
                        keys 0..q_start+i
  prefill_varlen     -- page832 post §6 (cu_seqlens_q interface): `prefill` per sequence
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
_LIB_PATH = os.path.join(_BUILD, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into a shared library (OpenMP if the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.pa_oracle_threads.restype = i32
            lib.pa_oracle_slot_mapping.argtypes = [P, P, P, i64, i32, i32, P]
            lib.pa_oracle_slot_mapping.restype = i32
            lib.pa_oracle_decode_input_prep.argtypes = [P, P, P, P, P, i32, i32, P, P, P, P]
            lib.pa_oracle_decode_input_prep.restype = i32
            lib.pa_oracle_reshape_and_cache.argtypes = [P, P, P, P, i64, P, i32, i32, i32, i32]
            lib.pa_oracle_reshape_and_cache.restype = None
            lib.pa_oracle_attend_row.argtypes = [P, P, P, i64, i64, P, i32, i32, i32, i32, i64,
                                                 f64, P, P]
            lib.pa_oracle_attend_row.restype = i32
            lib.pa_oracle_decode.argtypes = [P, P, P, i64, i64, P, i64, P, i32, i32, i32, i32,
                                             i32, f64, P, i32]
            lib.pa_oracle_decode.restype = i32
            lib.pa_oracle_prefill_rows.argtypes = [P, P, P, i64, i64, P, i32, i32, i32, i32, i32,
                                                   i32, i32, f64, P, P, i64, P, i32]
            lib.pa_oracle_prefill_rows.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def max_threads() -> int:
    """Threads the oracle's parallel loops may use (OpenMP default, 1 without OpenMP)."""
    return int(_load().pa_oracle_threads())


def slot_mapping(positions, block_table, block_size, seq_idx=None) -> np.ndarray:
    """slot[i] = block_table[seq_idx[i], pos // bs] * bs + pos % bs  (int64)."""
    lib = _load()
    pos = _c(positions, np.int32)
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt[None, :]
    sidx = None if seq_idx is None else _c(seq_idx, np.int32)
    out = np.empty(pos.shape[0], dtype=np.int64)
    rc = lib.pa_oracle_slot_mapping(_ptr(pos), _ptr(sidx), _ptr(bt), bt.shape[1], pos.shape[0],
                                    block_size, _ptr(out))
    if rc != 0:
        raise ValueError("oracle slot_mapping failed")
    return out


def decode_input_prep(positions, block_tables, block_sizes, sampled_ids=None):
    """One decode step's inputs: dict of seq_lens, query_start_loc, input_ids (or None)
    and slot_mappings (one int64 array per KV-cache group)."""
    lib = _load()
    pos = _c(positions, np.int32)
    S, G = pos.shape[0], len(block_tables)
    tables = [_c(t, np.int32) for t in block_tables]
    sid = None if sampled_ids is None else _c(sampled_ids, np.int32)
    seq_lens = np.empty(S, np.int32)
    qsl = np.empty(S + 1, np.int32)
    ids = None if sid is None else np.empty(S, np.int32)
    slots = [np.empty(S, np.int64) for _ in range(G)]
    tp = (ctypes.c_void_p * G)(*[t.ctypes.data for t in tables])
    sp = (ctypes.c_void_p * G)(*[x.ctypes.data for x in slots])
    strides = (ctypes.c_int64 * G)(*[t.shape[1] for t in tables])
    bss = (ctypes.c_int * G)(*[int(b) for b in block_sizes])
    rc = lib.pa_oracle_decode_input_prep(_ptr(pos), _ptr(sid), _ptr(ids), _ptr(seq_lens),
                                         _ptr(qsl), S, G, tp, strides, bss, sp)
    if rc != 0:
        raise ValueError("oracle decode_input_prep failed")
    return {"seq_lens": seq_lens, "query_start_loc": qsl, "input_ids": ids, "slot_mappings": slots}


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping_, block_size,
                      page_stride=None):
    """Write [T, Hkv, D] key/value rows into the uint16 caches in place."""
    lib = _load()
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    sm = _c(slot_mapping_, np.int64)
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    T, hkv, d = key.shape
    if page_stride is None:
        page_stride = block_size * hkv * d
    lib.pa_oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                    page_stride, _ptr(sm), T, hkv, d, block_size)


def _num_pages(cache, page_stride):
    return cache.size // page_stride


def attend_row(q_row, k_cache, v_cache, block_table_row, block_size, kv_head, num_keys,
               scale, page_stride=None, return_weights=False):
    """Exact softmax attention of one BF16 query row over keys 0..num_keys-1."""
    lib = _load()
    q = _c(q_row, np.uint16)
    _, bs, hkv, d = k_cache.shape
    assert bs == block_size
    if page_stride is None:
        page_stride = bs * hkv * d
    bt = _c(block_table_row, np.int32)
    out = np.empty(d, dtype=np.float64)
    w = np.empty(num_keys, dtype=np.float64) if return_weights else None
    rc = lib.pa_oracle_attend_row(_ptr(q), _ptr(k_cache), _ptr(v_cache), page_stride,
                                  _num_pages(k_cache, page_stride), _ptr(bt), block_size, hkv, d,
                                  kv_head, num_keys, float(scale), _ptr(out), _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle attend_row failed ({rc})")
    return (out, w) if return_weights else out


def decode(q, k_cache, v_cache, block_table, seq_lens, scale, num_threads=None):
    """q: uint16 [S, Hq, D]; caches uint16 [pages, BS, Hkv, D]; returns fp64 [S, Hq, D]."""
    lib = _load()
    q = _c(q, np.uint16)
    S, hq, d = q.shape
    _, bs, hkv, _ = k_cache.shape
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt[None, :]
    sl = _c(seq_lens, np.int32)
    out = np.empty((S, hq, d), dtype=np.float64)
    page_stride = bs * hkv * d
    nt = max_threads() if num_threads is None else int(num_threads)
    rc = lib.pa_oracle_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), page_stride,
                              _num_pages(k_cache, page_stride), _ptr(bt), bt.shape[1], _ptr(sl),
                              S, hq, hkv, d, bs, float(scale), _ptr(out), nt)
    if rc != 0:
        raise ValueError(f"oracle decode failed ({rc})")
    return out


def prefill_rows(q, k_cache, v_cache, block_table_row, q_start, causal, scale, rows, heads,
                 num_threads=None):
    """Outputs of the listed (row, head) pairs of a chunk; q: uint16 [q_len, Hq, D]."""
    lib = _load()
    q = _c(q, np.uint16)
    q_len, hq, d = q.shape
    _, bs, hkv, _ = k_cache.shape
    bt = _c(block_table_row, np.int32)
    r = _c(rows, np.int32)
    h = _c(heads, np.int32)
    assert r.shape == h.shape
    out = np.empty((r.shape[0], d), dtype=np.float64)
    page_stride = bs * hkv * d
    nt = max_threads() if num_threads is None else int(num_threads)
    rc = lib.pa_oracle_prefill_rows(_ptr(q), _ptr(k_cache), _ptr(v_cache), page_stride,
                                    _num_pages(k_cache, page_stride), _ptr(bt), q_len, q_start,
                                    int(bool(causal)), hq, hkv, d, bs, float(scale), _ptr(r),
                                    _ptr(h), r.shape[0], _ptr(out), nt)
    if rc != 0:
        raise ValueError(f"oracle prefill failed ({rc})")
    return out


def prefill(q, k_cache, v_cache, block_table_row, q_start, causal, scale, num_threads=None):
    """All rows and heads of a chunk: fp64 [q_len, Hq, D]."""
    q_len, hq, d = np.asarray(q).shape
    rows = np.repeat(np.arange(q_len, dtype=np.int32), hq)
    heads = np.tile(np.arange(hq, dtype=np.int32), q_len)
    out = prefill_rows(q, k_cache, v_cache, block_table_row, q_start, causal, scale, rows, heads,
                       num_threads)
    return out.reshape(q_len, hq, d)


def prefill_varlen(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, causal, scale,
                   num_threads=None):
    """Chunks of several sequences stacked row-wise (page832 post §6's varlen interface):
    chunk b = rows cu[b]..cu[b+1]-1, the last rows of sequence b's seq_lens_k[b] keys, each
    computed by `prefill` over row b of the block table."""
    q = np.ascontiguousarray(q)
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(len(seq_lens_k)):
        r0, r1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        if r1 > r0:
            out[r0:r1] = prefill(q[r0:r1], k_cache, v_cache, block_table[b],
                                 int(seq_lens_k[b]) - (r1 - r0), causal, scale, num_threads)
    return out
