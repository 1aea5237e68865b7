"""Paged attention for GB300: Python binding of libtvl.so.

Thin argument marshalling over the C ABI declared in ``include/tvl.h``:
torch CUDA tensors are checked (dtype, device, shape, contiguity) and passed as
raw pointers with the current CUDA stream.  Every step of the computation runs
in the library's CUDA kernels; there is no fallback.  If ``libtvl.so`` has not
been built, every call raises ``TvlError``.

Functions (same names as the C entry points, without the ``tvl_`` prefix):
  paged_kv_write, paged_attention_decode, paged_attention_decode_workspace_size,
  paged_decode_step, paged_attention_prefill, rope_paged_kv_write,
  copy_blocks, get_device_status, version.

Bound calls (``bind_paged_decode_step``, ``bind_paged_attention_decode``,
``bind_paged_attention_prefill``, ``bind_paged_kv_write``) check their
tensors once and return a callable that re-issues the same C call -- same
pointers, sizes and stream -- with one ctypes call and no further checks.
They are for loops that call the library with the same buffers every step
(a serving loop, a benchmark): the tensors must keep their storage, and the
device that was current at bind time must be current when the call is made.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "TvlError", "paged_kv_write", "paged_attention_decode", "copy_blocks", "BlockAllocator",
    "rope_paged_kv_write",
    "paged_attention_decode_workspace_size", "paged_attention_prefill", "get_device_status",
    "version", "library_path", "DEV_BAD_SLOT", "DEV_BAD_BLOCK_ID", "DEV_BAD_CONTEXT_LEN",
    "DEV_BAD_QUERY_LEN", "DEV_TIMEOUT", "DEV_NONFINITE", "selftest_bounded_wait",
    "paged_decode_step", "BoundCall", "bind_paged_decode_step", "bind_paged_attention_decode",
    "bind_paged_attention_prefill", "bind_paged_kv_write",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtvl.so")

(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_CHECK,
 ERR_OUT_OF_BLOCKS) = range(7)
DEV_BAD_SLOT, DEV_BAD_BLOCK_ID, DEV_BAD_CONTEXT_LEN, DEV_BAD_QUERY_LEN, DEV_TIMEOUT = (
    0x1, 0x2, 0x4, 0x8, 0x10)
DEV_NONFINITE = 0x20

_lock = threading.Lock()
_lib = None


class TvlError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"tvl status {status}: {detail}")
        self.status = status
        self.detail = detail


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise TvlError(ERR_CUDA, f"{_LIB_PATH} is missing: build it with "
                                         "paged_kv_cache_198_gb300._build.build()")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.tvl_paged_kv_write.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
            lib.tvl_paged_attention_decode_workspace_size.argtypes = [
                I, I, I, I, I, I, I, ctypes.POINTER(SZ)]
            lib.tvl_paged_attention_decode.argtypes = [
                P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, SZ, P]
            lib.tvl_paged_attention_prefill.argtypes = [
                P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P]
            lib.tvl_paged_decode_step.argtypes = [
                P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, SZ, P]
            lib.tvl_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            lib.tvl_selftest_bounded_wait.argtypes = [P]
            lib.tvl_selftest_bounded_wait.restype = I
            for name in ("tvl_paged_kv_write", "tvl_paged_attention_decode_workspace_size",
                         "tvl_paged_attention_decode", "tvl_paged_attention_prefill",
                         "tvl_paged_decode_step", "tvl_get_device_status"):
                getattr(lib, name).restype = I
            lib.tvl_status_string.argtypes = [I]
            lib.tvl_status_string.restype = ctypes.c_char_p
            lib.tvl_last_error.argtypes = []
            lib.tvl_last_error.restype = ctypes.c_char_p
            lib.tvl_version.argtypes = []
            lib.tvl_version.restype = I
            lib.tvl_rope_paged_kv_write.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
            lib.tvl_rope_paged_kv_write.restype = I
            lib.tvl_copy_blocks.argtypes = [P, P, P, P, I, I, I, I, I, P]
            lib.tvl_copy_blocks.restype = I
            I32P = ctypes.POINTER(ctypes.c_int32)
            IP = ctypes.POINTER(ctypes.c_int)
            lib.tvl_allocator_create.argtypes = [I, I, ctypes.POINTER(P)]
            lib.tvl_allocator_destroy.argtypes = [P]
            lib.tvl_allocator_destroy.restype = None
            lib.tvl_allocator_new_sequence.argtypes = [P, IP]
            lib.tvl_allocator_fork.argtypes = [P, I, IP]
            lib.tvl_allocator_append.argtypes = [P, I, I, I32P]
            lib.tvl_allocator_free_sequence.argtypes = [P, I]
            lib.tvl_allocator_context_len.argtypes = [P, I, ctypes.POINTER(ctypes.c_longlong)]
            lib.tvl_allocator_build_tables.argtypes = [P, IP, I, I, I32P, I32P]
            lib.tvl_allocator_take_copies.argtypes = [P, I32P, I32P, I, IP]
            lib.tvl_allocator_stats.argtypes = [P, ctypes.c_void_p]
            for name in ("tvl_allocator_create", "tvl_allocator_new_sequence", "tvl_allocator_fork",
                         "tvl_allocator_append", "tvl_allocator_free_sequence",
                         "tvl_allocator_context_len", "tvl_allocator_build_tables",
                         "tvl_allocator_take_copies", "tvl_allocator_stats"):
                getattr(lib, name).restype = I
            _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc != OK:
        lib = _load()
        raise TvlError(rc, (lib.tvl_last_error() or b"").decode() or
                       lib.tvl_status_string(rc).decode())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t: torch.Tensor, name: str, dtype, ndim=None, device=None):
    """Checks one argument; `device` is a torch.device or a CUDA device index.
    Cheap on the common path (it runs for every tensor of every call)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    idx = t.get_device()                                # -1 on the CPU
    if idx < 0:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None:
        want = device if isinstance(device, int) else device.index
        if idx != want:
            raise ValueError(f"{name} is on cuda:{idx}, expected cuda:{want}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


class _on_device:
    """Makes CUDA device `idx` current for the call (a no-op when it already
    is, which is the common case)."""

    __slots__ = ("idx", "prev")

    def __init__(self, idx):
        self.idx = idx if isinstance(idx, int) else idx.index
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)


def version() -> int:
    return int(_load().tvl_version())


def _prep_kv_write(k_new, v_new, k_cache, v_cache, slot_mapping, stream):
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.get_device()
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(k_new, "k_new", torch.bfloat16, 3, dev)
    _need(v_new, "v_new", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    nb, bs, hkv, d = k_cache.shape
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    t = slot_mapping.shape[0]
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d):
        raise ValueError(f"k_new/v_new must be [{t}, {hkv}, {d}]")
    with _on_device(dev):
        args = (_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                t, hkv, d, bs, nb, _stream(stream))
    return dev, _load().tvl_paged_kv_write, args, (k_new, v_new, k_cache, v_cache, slot_mapping)


def paged_kv_write(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """k_cache/v_cache bf16 [NB, bs, Hkv, D] (in place) <- k_new/v_new bf16
    [T, Hkv, D] at rows slot_mapping int32 [T] (negative = skip)."""
    dev, fn, args, _ = _prep_kv_write(k_new, v_new, k_cache, v_cache, slot_mapping, stream)
    with _on_device(dev):
        _check(fn(*args))


def bind_paged_kv_write(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None):
    """paged_kv_write, checked once; returns a BoundCall."""
    return BoundCall(*_prep_kv_write(k_new, v_new, k_cache, v_cache, slot_mapping, stream))


def rope_paged_kv_write(q, k_new, v_new, k_cache, v_cache, slot_mapping, positions,
                        rope_theta=500000.0, stream=None) -> None:
    """RoPE of q (in place; may be None) and of k_new at `positions` (int32
    [T]), then the paged write of the rotated K rows and the V rows."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.get_device()
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(k_new, "k_new", torch.bfloat16, 3, dev)
    _need(v_new, "v_new", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    _need(positions, "positions", torch.int32, 1, dev)
    nb, bs, hkv, d = k_cache.shape
    t = slot_mapping.shape[0]
    hq = 0
    if q is not None:
        _need(q, "q", torch.bfloat16, 3, dev)
        if q.shape[0] != t or q.shape[2] != d:
            raise ValueError("q must be [T, Hq, D]")
        hq = q.shape[1]
    if k_new.shape != (t, hkv, d) or v_new.shape != (t, hkv, d) or positions.shape[0] != t:
        raise ValueError("k_new/v_new must be [T, Hkv, D] and positions [T]")
    with _on_device(dev):
        _check(_load().tvl_rope_paged_kv_write(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                               _ptr(v_cache), _ptr(slot_mapping),
                                               _ptr(positions), t, hq, hkv, d, bs, nb,
                                               float(rope_theta), _stream(stream)))


def paged_attention_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                          max_blocks_per_seq, block_size,
                                          partition_size=0) -> int:
    """Bytes of workspace the decode needs (tvl_paged_attention_decode_workspace_size)
    on the current device; the answer is remembered per device and shape."""
    key = (torch.cuda.current_device() if torch.cuda.is_available() else -1, num_seqs,
           num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, partition_size)
    hit = _ws_sizes.get(key)
    if hit is not None:
        return hit
    out = ctypes.c_size_t(0)
    _check(_load().tvl_paged_attention_decode_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
        partition_size, ctypes.byref(out)))
    _ws_sizes[key] = int(out.value)
    return int(out.value)


_ws_sizes = {}


def _workspace_for(dev, s, hq, hkv, d, mb, bs, partition_size, workspace):
    need = paged_attention_decode_workspace_size(s, hq, hkv, d, mb, bs, partition_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1, dev)
    return workspace, (workspace.numel() if workspace is not None else 0)


def _prep_decode(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                 partition_size, workspace, stream):
    """Checks of a decode (k_new is None) or decode-step call; returns the
    device, the C function, its arguments and the tensors they point into."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.get_device()
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(out, "out", torch.float32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    nb, bs, hkv, d = k_cache.shape
    s, hq, d2 = q.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent q / out / cache shapes")
    if block_tables.shape[0] != s or context_lens.shape[0] != s:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    step = k_new is not None
    if step:
        _need(k_new, "k_new", torch.bfloat16, 3, dev)
        _need(v_new, "v_new", torch.bfloat16, 3, dev)
        if tuple(k_new.shape) != (s, hkv, d) or v_new.shape != k_new.shape:
            raise ValueError("k_new / v_new must be [num_seqs, num_kv_heads, head_dim]")
    mb = block_tables.shape[1]
    with _on_device(dev):
        workspace, ws_bytes = _workspace_for(dev, s, hq, hkv, d, mb, bs, int(partition_size),
                                             workspace)
        tail = (_ptr(block_tables), _ptr(context_lens), s, hq, hkv, d, bs, nb, mb,
                float(scale), int(partition_size), _ptr(workspace), ws_bytes, _stream(stream))
    lib = _load()
    keep = (out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, workspace)
    if step:
        return dev, lib.tvl_paged_decode_step, (
            _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache)) + tail, keep
    return dev, lib.tvl_paged_attention_decode, (
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache)) + tail, keep


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           partition_size=0, workspace=None, stream=None):
    """out fp32 [S, Hq, D] <- paged decode attention of q bf16 [S, Hq, D].
    workspace: uint8 CUDA tensor (allocated here when None and needed)."""
    dev, fn, args, _ = _prep_decode(out, q, None, None, k_cache, v_cache, block_tables,
                                    context_lens, scale, partition_size, workspace, stream)
    with _on_device(dev):
        _check(fn(*args))
    return out


def bind_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                partition_size=0, workspace=None, stream=None):
    """paged_attention_decode, checked once (the workspace, when None and
    needed, is allocated here once); returns a BoundCall."""
    return BoundCall(*_prep_decode(out, q, None, None, k_cache, v_cache, block_tables,
                                   context_lens, scale, partition_size, workspace, stream))


def paged_decode_step(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                      partition_size=0, workspace=None, stream=None):
    """One decode step (tvl_paged_decode_step): writes k_new / v_new bf16
    [S, Hkv, D] at position context_lens[s] - 1 of each sequence, then
    out fp32 [S, Hq, D] <- paged decode attention of q bf16 [S, Hq, D] over
    the updated cache."""
    if k_new is None or v_new is None:
        raise TypeError("k_new and v_new are required")
    dev, fn, args, _ = _prep_decode(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                    context_lens, scale, partition_size, workspace, stream)
    with _on_device(dev):
        _check(fn(*args))
    return out


def bind_paged_decode_step(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                           scale, partition_size=0, workspace=None, stream=None):
    """paged_decode_step, checked once; returns a BoundCall."""
    if k_new is None or v_new is None:
        raise TypeError("k_new and v_new are required")
    return BoundCall(*_prep_decode(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                   context_lens, scale, partition_size, workspace, stream))


def _prep_prefill(out, q, query_start_loc, k_cache, v_cache, block_tables, context_lens, scale,
                  max_q_len, stream):
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.get_device()
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(q, "q", torch.bfloat16, 3, dev)
    _need(out, "out", torch.float32, 3, dev)
    _need(query_start_loc, "query_start_loc", torch.int32, 1, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    nb, bs, hkv, d = k_cache.shape
    tq, hq, d2 = q.shape
    s = context_lens.shape[0]
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent q / out / cache shapes")
    if query_start_loc.shape[0] != s + 1 or block_tables.shape[0] != s:
        raise ValueError("query_start_loc must be [S+1] and block_tables [S, MB]")
    mb = block_tables.shape[1]
    with _on_device(dev):
        args = (_ptr(out), _ptr(q), _ptr(query_start_loc), _ptr(k_cache), _ptr(v_cache),
                _ptr(block_tables), _ptr(context_lens), s, tq, int(max_q_len), hq, hkv, d, bs,
                nb, mb, float(scale), _stream(stream))
    keep = (out, q, query_start_loc, k_cache, v_cache, block_tables, context_lens)
    return dev, _load().tvl_paged_attention_prefill, args, keep


def paged_attention_prefill(out, q, query_start_loc, k_cache, v_cache, block_tables,
                            context_lens, scale, max_q_len, stream=None):
    """out fp32 [Tq, Hq, D] <- causal attention of the last Lq tokens of each
    sequence (q bf16 [Tq, Hq, D], packed by query_start_loc int32 [S+1])."""
    dev, fn, args, _ = _prep_prefill(out, q, query_start_loc, k_cache, v_cache, block_tables,
                                     context_lens, scale, max_q_len, stream)
    with _on_device(dev):
        _check(fn(*args))
    return out


def bind_paged_attention_prefill(out, q, query_start_loc, k_cache, v_cache, block_tables,
                                 context_lens, scale, max_q_len, stream=None):
    """paged_attention_prefill, checked once; returns a BoundCall."""
    return BoundCall(*_prep_prefill(out, q, query_start_loc, k_cache, v_cache, block_tables,
                                    context_lens, scale, max_q_len, stream))


class BoundCall:
    """One C-ABI call whose arguments were checked and converted once.
    Calling it re-issues the call (same pointers, sizes and stream); a non-OK
    status raises TvlError.  It keeps references to the tensors it points
    into; they must keep their storage, and the bind-time device must be
    current when it is called."""

    __slots__ = ("device", "_fn", "_args", "_keep")

    def __init__(self, device, fn, args, keep):
        self.device = device
        self._fn = fn
        self._args = args
        self._keep = keep

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc:
            _check(rc)


def selftest_bounded_wait(stream=None) -> None:
    """Launches one CTA whose bounded wait is never satisfied: it gives up
    after about a second and sets DEV_TIMEOUT (tvl_selftest_bounded_wait)."""
    _check(_load().tvl_selftest_bounded_wait(_stream(stream)))


def get_device_status(stream=None) -> int:
    """Reads and clears the device status word; returns its bits (0 = clean).
    Synchronises the stream."""
    bits = ctypes.c_uint32(0)
    rc = _load().tvl_get_device_status(_stream(stream), ctypes.byref(bits))
    if rc not in (OK, ERR_DEVICE_CHECK):
        _check(rc)
    return int(bits.value)


def copy_blocks(k_cache, v_cache, src, dst, stream=None) -> None:
    """Physical block dst[i] of both caches <- block src[i] (int32 CUDA
    tensors [n]); bit-exact; the pairs must not overlap."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    dev = k_cache.get_device()
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(src, "src", torch.int32, 1, dev)
    _need(dst, "dst", torch.int32, 1, dev)
    if src.shape != dst.shape:
        raise ValueError("src and dst differ in length")
    nb, bs, hkv, d = k_cache.shape
    with _on_device(dev):
        _check(_load().tvl_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src), _ptr(dst),
                                       src.numel(), hkv, d, bs, nb, _stream(stream)))


class _Stats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("free_blocks", ctypes.c_int),
                ("live_sequences", ctypes.c_int), ("shared_blocks", ctypes.c_int),
                ("tokens", ctypes.c_longlong), ("slack_slots", ctypes.c_longlong)]


class BlockAllocator:
    """Host block allocator of libtvl (tvl_allocator_*): hands out physical
    blocks and cache slots, shares blocks between forked sequences and queues
    copy-on-write block copies.  Host memory only."""

    def __init__(self, num_blocks: int, block_size: int):
        import numpy as np  # noqa: F401

        self._lib = _load()
        self._h = ctypes.c_void_p()
        _check(self._lib.tvl_allocator_create(num_blocks, block_size, ctypes.byref(self._h)))
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            self._lib.tvl_allocator_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_sequence(self) -> int:
        out = ctypes.c_int(0)
        _check(self._lib.tvl_allocator_new_sequence(self._h, ctypes.byref(out)))
        return out.value

    def fork(self, parent: int) -> int:
        out = ctypes.c_int(0)
        _check(self._lib.tvl_allocator_fork(self._h, parent, ctypes.byref(out)))
        return out.value

    def append(self, seq: int, num_tokens: int):
        import numpy as np

        slots = np.zeros(max(num_tokens, 1), dtype=np.int32)
        _check(self._lib.tvl_allocator_append(
            self._h, seq, num_tokens, slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return slots[:num_tokens]

    def free(self, seq: int) -> None:
        _check(self._lib.tvl_allocator_free_sequence(self._h, seq))

    def context_len(self, seq: int) -> int:
        out = ctypes.c_longlong(0)
        _check(self._lib.tvl_allocator_context_len(self._h, seq, ctypes.byref(out)))
        return int(out.value)

    def build_tables(self, seqs, max_blocks_per_seq: int):
        import numpy as np

        ids = np.ascontiguousarray(seqs, dtype=np.intc)
        n = ids.shape[0]
        tables = np.zeros((max(n, 1), max_blocks_per_seq), dtype=np.int32)
        ctx = np.zeros(max(n, 1), dtype=np.int32)
        _check(self._lib.tvl_allocator_build_tables(
            self._h, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n, max_blocks_per_seq,
            tables.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            ctx.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return tables[:n], ctx[:n]

    def take_copies(self):
        import numpy as np

        count = ctypes.c_int(0)
        rc = self._lib.tvl_allocator_take_copies(self._h, None, None, 0, ctypes.byref(count))
        if rc == OK and count.value == 0:
            return np.zeros(0, np.int32), np.zeros(0, np.int32)
        src = np.zeros(count.value, dtype=np.int32)
        dst = np.zeros(count.value, dtype=np.int32)
        _check(self._lib.tvl_allocator_take_copies(
            self._h, src.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            dst.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), count.value,
            ctypes.byref(count)))
        return src[:count.value], dst[:count.value]

    def stats(self) -> dict:
        st = _Stats()
        _check(self._lib.tvl_allocator_stats(self._h, ctypes.byref(st)))
        return {name: getattr(st, name) for name, _ in _Stats._fields_}
