"""ctypes binding of the C ABI in ``include/pa.h`` (argument marshalling only).

Every function keeps the C name and argument order.  Tensors are passed as raw device
pointers (``tensor.data_ptr()``); plain ints are accepted as pointers too.  A non-OK status
raises :class:`PaError` (its ``status`` attribute holds the code).  There is no fallback: if
the shared library has not been built, loading it raises.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE_TOO_SMALL = 3
PA_ERR_CUDA = 4
PA_ERR_OUT_OF_BLOCKS = 5

PA_BF16 = 0
PA_FP8_E4M3 = 1
PA_INT8 = 2
PA_INT4 = 3
PA_FP8_E4M3_TOKEN = 4

PA_EFLAG_BAD_BLOCK_ID = 1
PA_EFLAG_CTX_OVERFLOW = 2
PA_EFLAG_BAD_SEQ = 4
PA_EFLAG_TIMEOUT = 8

BLOCK_SIZE = 16

_DTYPES = {"bf16": PA_BF16, "fp8_e4m3": PA_FP8_E4M3, "e4m3": PA_FP8_E4M3, "int8": PA_INT8, "int4": PA_INT4,
           "e4m3_tok": PA_FP8_E4M3_TOKEN}

# Every symbol the header declares, for load checks.
EXPORTED = [
    "pa_status_string", "pa_kv_append", "pa_kv_append_tokens", "pa_block_copy",
    "pa_decode_workspace_size", "pa_decode_attention", "pa_decode_attention_noalloc", "pa_decode_step",
    "pa_decode_shared_workspace_size", "pa_decode_attention_shared",
    "pa_prefill_attention", "pa_prefill_step", "pa_prefill_workspace_size", "pa_prefill_attention_ws",
    "pa_prefill_step_ws",
    "pa_bm_create", "pa_bm_destroy", "pa_bm_alloc", "pa_bm_claim", "pa_bm_incref", "pa_bm_decref",
    "pa_bm_refcount", "pa_bm_num_free", "pa_bm_fork", "pa_bm_release", "pa_bm_prepare_step",
    "pa_bm_slide_window",
    "pa_pc_block_hashes", "pa_pc_create", "pa_pc_destroy", "pa_pc_match", "pa_pc_insert", "pa_pc_evict",
    "pa_pc_size", "pa_pc_clear",
]

DIGEST_BYTES = 32


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class CacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("block_size", ctypes.c_int),
        ("num_blocks", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("k_dtype", ctypes.c_int),
        ("v_dtype", ctypes.c_int),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("k_sink", ctypes.c_void_p),
        ("v_sink", ctypes.c_void_p),
        ("num_sink", ctypes.c_int),
        ("sliding_window", ctypes.c_int),
    ]


_LIB = None
_LIB_PATH = LIB_PATH


def use_library(path: str) -> None:
    """Bind to another build of the same library (e.g. one compiled with tuning defines).
    Must be called before the first call into the library."""
    global _LIB_PATH
    if _LIB is not None:
        raise RuntimeError("the library is already loaded")
    _LIB_PATH = path


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises if it was never built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with paged_kv_cache_table_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32p, c_int = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int
        dp = ctypes.POINTER(CacheDesc)
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_status_string.argtypes = [c_int]
        L.pa_kv_append.restype = c_int
        L.pa_kv_append.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.pa_kv_append_tokens.restype = c_int
        L.pa_kv_append_tokens.argtypes = [dp, vp, vp, vp, vp, c_int, vp, vp, vp, vp, vp]
        L.pa_block_copy.restype = c_int
        L.pa_block_copy.argtypes = [dp, vp, vp, vp, c_int, vp, vp]
        L.pa_decode_workspace_size.restype = ctypes.c_size_t
        L.pa_decode_workspace_size.argtypes = [dp, c_int, c_int]
        L.pa_decode_attention.restype = c_int
        L.pa_decode_attention.argtypes = [dp, vp, vp, vp, vp, vp, vp, c_int, ctypes.c_float, c_int, vp,
                                          ctypes.c_size_t, vp, vp]
        L.pa_decode_shared_workspace_size.restype = ctypes.c_size_t
        L.pa_decode_shared_workspace_size.argtypes = [dp, c_int, c_int, c_int]
        L.pa_decode_attention_shared.restype = c_int
        L.pa_decode_attention_shared.argtypes = [dp, vp, vp, vp, vp, vp, vp, c_int, ctypes.c_float, c_int, vp,
                                                 c_int, c_int, vp, ctypes.c_size_t, vp, vp]
        L.pa_prefill_attention.restype = c_int
        L.pa_prefill_attention.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, c_int, ctypes.c_float, vp, vp]
        L.pa_prefill_workspace_size.restype = ctypes.c_size_t
        L.pa_prefill_workspace_size.argtypes = [dp, c_int]
        L.pa_prefill_attention_ws.restype = c_int
        L.pa_prefill_attention_ws.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, ctypes.c_float, vp,
                                              ctypes.c_size_t, vp, vp]
        L.pa_prefill_step_ws.restype = c_int
        L.pa_prefill_step_ws.argtypes = [dp, vp, vp, vp, vp, vp, vp, c_int, vp, vp, vp, vp, vp, c_int, c_int,
                                         ctypes.c_float, vp, ctypes.c_size_t, vp, vp]
        L.pa_prefill_step.restype = c_int
        L.pa_prefill_step.argtypes = [dp, vp, vp, vp, vp, vp, vp, c_int, vp, vp, vp, vp, vp, c_int,
                                      ctypes.c_float, vp, vp]
        L.pa_decode_attention_noalloc.restype = c_int
        L.pa_decode_attention_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, vp, c_int, ctypes.c_float, c_int, vp, vp]
        L.pa_decode_step.restype = c_int
        L.pa_decode_step.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int, ctypes.c_float, c_int, vp,
                                     ctypes.c_size_t, vp, vp]
        L.pa_bm_create.restype = vp
        L.pa_bm_create.argtypes = [c_int, c_int]
        L.pa_bm_destroy.restype = None
        L.pa_bm_destroy.argtypes = [vp]
        for name in ("pa_bm_alloc", "pa_bm_num_free"):
            getattr(L, name).restype = c_int
        L.pa_bm_alloc.argtypes = [vp]
        L.pa_bm_num_free.argtypes = [vp]
        for name in ("pa_bm_claim", "pa_bm_incref", "pa_bm_decref", "pa_bm_refcount"):
            getattr(L, name).restype = c_int
            getattr(L, name).argtypes = [vp, c_int]
        L.pa_bm_fork.restype = c_int
        L.pa_bm_fork.argtypes = [vp, i32p, i32p, c_int]
        L.pa_bm_release.restype = c_int
        L.pa_bm_release.argtypes = [vp, i32p, c_int]
        L.pa_bm_prepare_step.restype = c_int
        # (array arguments of the per-step calls as plain addresses: ctypes pointer objects cost
        # microseconds each to build)
        L.pa_bm_prepare_step.argtypes = [vp, vp, c_int, c_int, vp, vp, ctypes.POINTER(c_int),
                                         ctypes.POINTER(c_int)]
        L.pa_bm_slide_window.restype = c_int
        L.pa_bm_slide_window.argtypes = [vp, vp, c_int, c_int, vp, c_int, ctypes.POINTER(c_int)]
        u64, u8p = ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint8)
        L.pa_pc_block_hashes.restype = c_int
        L.pa_pc_block_hashes.argtypes = [i32p, c_int, u64, u64, u8p]
        L.pa_pc_create.restype = vp
        L.pa_pc_create.argtypes = [vp, c_int]
        L.pa_pc_destroy.restype = None
        L.pa_pc_destroy.argtypes = [vp]
        L.pa_pc_match.restype = c_int
        L.pa_pc_match.argtypes = [vp, u8p, c_int, i32p]
        L.pa_pc_insert.restype = c_int
        L.pa_pc_insert.argtypes = [vp, u8p, i32p, c_int]
        L.pa_pc_evict.restype = c_int
        L.pa_pc_evict.argtypes = [vp, c_int]
        for name in ("pa_pc_size", "pa_pc_clear"):
            getattr(L, name).restype = c_int
            getattr(L, name).argtypes = [vp]
        _LIB = L
    return _LIB


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


pa_status_string = status_string


def _check(status: int, where: str):
    if status != PA_OK:
        raise PaError(status, where)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq,
              k_dtype="bf16", v_dtype="bf16", k_scales=None, v_scales=None,
              k_sink=None, v_sink=None, num_sink=0, block_size=BLOCK_SIZE, sliding_window=0) -> CacheDesc:
    """Fill a pa_cache_desc.  Tensors passed here must outlive every call that uses it."""
    return CacheDesc(int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                     int(num_blocks), int(max_blocks_per_seq), _DTYPES.get(k_dtype, k_dtype),
                     _DTYPES.get(v_dtype, v_dtype), _ptr(k_scales), _ptr(v_scales), _ptr(k_sink),
                     _ptr(v_sink), int(num_sink), int(sliding_window))


def pa_kv_append(desc, k_cache, v_cache, k_new, v_new, block_tables, positions, err_flag=None, stream=None):
    _check(lib().pa_kv_append(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                              _ptr(block_tables), _ptr(positions), _ptr(err_flag), _stream(stream)),
           "pa_kv_append")


def pa_kv_append_tokens(desc, k_cache, v_cache, k_new, v_new, num_tokens, token_seq, token_pos,
                        block_tables, err_flag=None, stream=None):
    _check(lib().pa_kv_append_tokens(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(k_new),
                                     _ptr(v_new), int(num_tokens), _ptr(token_seq), _ptr(token_pos),
                                     _ptr(block_tables), _ptr(err_flag), _stream(stream)),
           "pa_kv_append_tokens")


def pa_block_copy(desc, k_cache, v_cache, src_dst_pairs, n_pairs, err_flag=None, stream=None):
    _check(lib().pa_block_copy(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs),
                               int(n_pairs), _ptr(err_flag), _stream(stream)), "pa_block_copy")


def pa_decode_workspace_size(desc, max_context_len, partition_size=0) -> int:
    return int(lib().pa_decode_workspace_size(ctypes.byref(desc), int(max_context_len), int(partition_size)))


def pa_decode_attention(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                        scale, partition_size, workspace, workspace_bytes=None, err_flag=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_attention(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_tables), _ptr(context_lens), int(max_context_len),
                                     float(scale), int(partition_size), _ptr(workspace),
                                     int(workspace_bytes), _ptr(err_flag), _stream(stream)),
           "pa_decode_attention")


def pa_decode_shared_workspace_size(desc, max_context_len, partition_size=0, shared_len=0) -> int:
    return int(lib().pa_decode_shared_workspace_size(ctypes.byref(desc), int(max_context_len),
                                                     int(partition_size), int(shared_len)))


def pa_decode_attention_shared(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                               scale, partition_size, shared_seqs, n_shared, shared_len, workspace,
                               workspace_bytes=None, err_flag=None, stream=None):
    """pa_decode_attention with a prefix shared by the listed sequences attended once (see pa.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_attention_shared(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
                                            int(max_context_len), float(scale), int(partition_size),
                                            _ptr(shared_seqs), int(n_shared), int(shared_len), _ptr(workspace),
                                            int(workspace_bytes), _ptr(err_flag), _stream(stream)),
           "pa_decode_attention_shared")


def pa_decode_step(desc, out, q, k_cache, v_cache, k_new, v_new, block_tables, positions, context_lens,
                   max_context_len, scale, partition_size, workspace, workspace_bytes=None, err_flag=None,
                   stream=None):
    """pa_kv_append of one token per sequence, then pa_decode_attention, as one step (see pa.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_step(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                _ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(positions),
                                _ptr(context_lens), int(max_context_len), float(scale), int(partition_size),
                                _ptr(workspace), int(workspace_bytes), _ptr(err_flag), _stream(stream)),
           "pa_decode_step")


def pa_prefill_attention(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                         scale, err_flag=None, stream=None):
    _check(lib().pa_prefill_attention(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(block_tables), _ptr(q_start), _ptr(context_lens), int(max_query_len),
                                      float(scale), _ptr(err_flag), _stream(stream)),
           "pa_prefill_attention")


def pa_prefill_workspace_size(desc, max_context_len) -> int:
    return int(lib().pa_prefill_workspace_size(ctypes.byref(desc), int(max_context_len)))


def pa_prefill_attention_ws(desc, out, q, k_cache, v_cache, block_tables, q_start, context_lens, max_query_len,
                            max_context_len, scale, workspace, workspace_bytes=None, err_flag=None, stream=None):
    """pa_prefill_attention with each attended block decoded once into the workspace (see pa.h)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_prefill_attention_ws(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(block_tables), _ptr(q_start), _ptr(context_lens),
                                         int(max_query_len), int(max_context_len), float(scale), _ptr(workspace),
                                         int(workspace_bytes), _ptr(err_flag), _stream(stream)),
           "pa_prefill_attention_ws")


def pa_prefill_step_ws(desc, out, q, k_cache, v_cache, k_new, v_new, num_tokens, token_seq, token_pos, block_tables,
                       q_start, context_lens, max_query_len, max_context_len, scale, workspace, workspace_bytes=None,
                       err_flag=None, stream=None):
    """pa_kv_append_tokens of a chunk, then pa_prefill_attention_ws, as one step (see pa.h)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_prefill_step_ws(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(k_new), _ptr(v_new), int(num_tokens), _ptr(token_seq), _ptr(token_pos),
                                    _ptr(block_tables), _ptr(q_start), _ptr(context_lens), int(max_query_len),
                                    int(max_context_len), float(scale), _ptr(workspace), int(workspace_bytes),
                                    _ptr(err_flag), _stream(stream)),
           "pa_prefill_step_ws")


def pa_prefill_step(desc, out, q, k_cache, v_cache, k_new, v_new, num_tokens, token_seq, token_pos, block_tables,
                    q_start, context_lens, max_query_len, scale, err_flag=None, stream=None):
    """pa_kv_append_tokens of a chunk, then pa_prefill_attention, as one step (see pa.h)."""
    _check(lib().pa_prefill_step(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(k_new), _ptr(v_new), int(num_tokens), _ptr(token_seq), _ptr(token_pos),
                                 _ptr(block_tables), _ptr(q_start), _ptr(context_lens), int(max_query_len),
                                 float(scale), _ptr(err_flag), _stream(stream)),
           "pa_prefill_step")


def pa_decode_attention_noalloc(desc, out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                                scale, partition_size, err_flag=None, stream=None):
    """pa_decode_attention with its scratch in the library's static device array (see pa.h)."""
    _check(lib().pa_decode_attention_noalloc(ctypes.byref(desc), _ptr(out), _ptr(q), _ptr(k_cache),
                                             _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
                                             int(max_context_len), float(scale), int(partition_size),
                                             _ptr(err_flag), _stream(stream)),
           "pa_decode_attention_noalloc")


def _i32(a) -> np.ndarray:
    if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
        raise TypeError("expected a C-contiguous int32 numpy array (it is modified in place)")
    return a


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class BlockManager:
    """The host block pool (pa_bm_*): free list, reference counts, copy-on-write decisions."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        h = lib().pa_bm_create(int(num_blocks), int(block_size))
        if not h:
            raise PaError(PA_ERR_INVALID_ARG, "pa_bm_create")
        self._h = ctypes.c_void_p(h)
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self) -> int:
        return lib().pa_bm_alloc(self._h)

    def claim(self, blk: int) -> bool:
        return lib().pa_bm_claim(self._h, int(blk)) == 0

    def incref(self, blk: int) -> int:
        return lib().pa_bm_incref(self._h, int(blk))

    def decref(self, blk: int) -> int:
        return lib().pa_bm_decref(self._h, int(blk))

    def refcount(self, blk: int) -> int:
        return lib().pa_bm_refcount(self._h, int(blk))

    def num_free(self) -> int:
        return lib().pa_bm_num_free(self._h)

    def fork(self, src_row: np.ndarray, n_blocks: int, dst_row: np.ndarray | None = None) -> np.ndarray:
        src = _i32(np.ascontiguousarray(src_row, dtype=np.int32))
        dst = np.full(len(src), -1, dtype=np.int32) if dst_row is None else _i32(dst_row)
        _check(lib().pa_bm_fork(self._h, _p32(src), _p32(dst), int(n_blocks)), "pa_bm_fork")
        return dst

    def release(self, row: np.ndarray, n_blocks: int) -> int:
        r = lib().pa_bm_release(self._h, _p32(_i32(row)), int(n_blocks))
        if r < 0:
            raise PaError(PA_ERR_INVALID_ARG, "pa_bm_release")
        return r

    def prepare_step(self, block_tables: np.ndarray, positions: np.ndarray):
        """Make every sequence's append slot writable; returns (pairs [n][2], n_changed).
        ``block_tables`` (int32 [B][max_blocks]) is updated in place."""
        bt = _i32(block_tables)
        pos = _i32(np.ascontiguousarray(positions, dtype=np.int32))
        B, M = bt.shape
        pairs = np.empty((max(B, 1), 2), dtype=np.int32)
        n_pairs = ctypes.c_int(0)
        n_changed = ctypes.c_int(0)
        st = lib().pa_bm_prepare_step(self._h, bt.ctypes.data, B, M, pos.ctypes.data, pairs.ctypes.data,
                                      ctypes.byref(n_pairs), ctypes.byref(n_changed))
        _check(st, "pa_bm_prepare_step")
        return pairs[:n_pairs.value].copy(), n_changed.value

    def slide_window(self, block_tables: np.ndarray, context_lens: np.ndarray, window: int):
        """Release every block wholly before each sequence's window; returns (entries released,
        blocks freed).  ``block_tables`` (int32 [B][max_blocks]) is updated in place."""
        bt = _i32(block_tables)
        ctx = _i32(np.ascontiguousarray(context_lens, dtype=np.int32))
        B, M = bt.shape
        n_freed = ctypes.c_int(0)
        r = lib().pa_bm_slide_window(self._h, bt.ctypes.data, B, M, ctx.ctypes.data, int(window), ctypes.byref(n_freed))
        if r < 0:
            raise PaError(PA_ERR_INVALID_ARG, "pa_bm_slide_window")
        return r, n_freed.value


def _p8(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def block_hashes(tokens, salt: int = 0, extra_key: int = 0) -> np.ndarray:
    """Digests uint8 [n_tokens // 16][32] of a token sequence's full blocks (pa_pc_block_hashes)."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.zeros((len(t) // BLOCK_SIZE, DIGEST_BYTES), dtype=np.uint8)
    n = lib().pa_pc_block_hashes(_p32(t), len(t), int(salt) & (2 ** 64 - 1), int(extra_key) & (2 ** 64 - 1),
                                 _p8(out))
    if n < 0:
        raise PaError(PA_ERR_INVALID_ARG, "pa_pc_block_hashes")
    return out


class PrefixCache:
    """The host prefix cache over a BlockManager's pool (pa_pc_*)."""

    def __init__(self, bm: "BlockManager", capacity: int = 0):
        h = lib().pa_pc_create(bm._h, int(capacity))
        if not h:
            raise PaError(PA_ERR_INVALID_ARG, "pa_pc_create")
        self._h = ctypes.c_void_p(h)
        self.bm = bm  # the pool must outlive the cache

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_pc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __len__(self):
        return lib().pa_pc_size(self._h)

    def match(self, digests: np.ndarray, n_blocks: int, table_row: np.ndarray) -> int:
        """Longest cached leading run of digests[:n_blocks] into table_row (int32, in place)."""
        d = np.ascontiguousarray(digests, dtype=np.uint8)
        n = min(int(n_blocks), len(d))
        r = lib().pa_pc_match(self._h, _p8(d), max(0, n), _p32(_i32(table_row)))
        if r < 0:
            raise PaError(PA_ERR_INVALID_ARG, "pa_pc_match")
        return r

    def insert(self, digests: np.ndarray, table_row: np.ndarray, n_blocks: int) -> int:
        d = np.ascontiguousarray(digests, dtype=np.uint8)
        r = lib().pa_pc_insert(self._h, _p8(d), _p32(_i32(np.ascontiguousarray(table_row, dtype=np.int32))),
                               min(int(n_blocks), len(d)))
        if r < 0:
            raise PaError(PA_ERR_INVALID_ARG, "pa_pc_insert")
        return r

    def evict(self, n: int) -> int:
        return lib().pa_pc_evict(self._h, int(n))

    def clear(self) -> int:
        return lib().pa_pc_clear(self._h)
