"""GB300 (sm_103a) Kamera reuse operator: thin Python binding of the C ABI.

The operator ("Kamera: Unified Position-Invariant Multimodal KV Cache for
Training-Free Reuse", gist.science technical summary, section 2) relocates a
position-free canonical chunk to a new position and restores its cross-chunk
conditioning:  KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T, written into a
paged KV pool.  Every step runs in the CUDA kernels of ``libkamera.so``
(``include/kamera.h``); this module only marshals torch tensors into the C
structs and calls the entry points of the same names.  There is no CPU path:
without the compiled library (or without a GPU) every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

__all__ = [
    "KameraError", "Rope", "ChunkSpec", "load_library", "pack_chunks",
    "kamera_relocate_patch", "kamera_slide_inplace", "kamera_mla_relocate_patch",
    "kamera_ingest_canonical", "kamera_mla_ingest_canonical", "kamera_form_patch", "kamera_attend_reused",
    "kamera_prefill_attend_reused",
    "kamera_validate_chunks", "kamera_status_string", "kamera_abi_version",
    "ROTATE_HALF", "INTERLEAVED", "DEVERR",
]

ROTATE_HALF = 0
INTERLEAVED = 1
MAX_RANK = 128

DEVERR = {
    1: "slot out of range",
    2: "source rows out of range",
    4: "malformed descriptor",
    8: "len > max_len",
    16: "rank > max_rank",
    32: "pipeline wait timed out",
}


class KameraError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {kamera_status_string(status)} (status {status})")
        self.status = status


# ----------------------------------------------------------------- C structs
class _Chunk(C.Structure):
    _fields_ = [("src_offset", C.c_int64), ("len", C.c_int32), ("rank", C.c_int32),
                ("delta", C.c_int64), ("patch_ptrs", C.c_void_p * 4),
                ("dst_slot_mapping", C.c_void_p)]


class _Rope(C.Structure):
    _fields_ = [("base", C.c_double), ("rot_dim", C.c_int32), ("rot_offset", C.c_int32),
                ("pairing", C.c_int32), ("n_axes", C.c_int32),
                ("inv_freq_override", C.POINTER(C.c_double)),
                ("freq_axis", C.POINTER(C.c_uint8)), ("d_axis_delta", C.c_void_p)]


class _GqaPool(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("reserved", C.c_int32), ("k", C.c_void_p), ("v", C.c_void_p),
                ("num_slots", C.c_int64), ("layer_stride", C.c_int64), ("slot_stride", C.c_int64)]


class _GqaStore(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("num_rows", C.c_int64),
                ("layer_stride", C.c_int64), ("row_stride", C.c_int64)]


class _SlidePool(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("reserved", C.c_int32), ("k", C.c_void_p), ("num_slots", C.c_int64),
                ("layer_stride", C.c_int64), ("slot_stride", C.c_int64)]


class _MlaPool(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("kv_lora_rank", C.c_int32), ("rope_dim", C.c_int32),
                ("reserved", C.c_int32), ("kv", C.c_void_p), ("num_slots", C.c_int64),
                ("layer_stride", C.c_int64), ("slot_stride", C.c_int64)]


class _Deficit(C.Structure):
    _fields_ = [("x", C.c_void_p), ("n_outer", C.c_int64), ("n_inner", C.c_int64),
                ("outer_stride", C.c_int64), ("inner_stride", C.c_int64), ("row_stride", C.c_int64),
                ("term_stride", C.c_int64), ("n_terms", C.c_int32), ("rows", C.c_int32), ("cols", C.c_int32),
                ("reserved", C.c_int32)]


class _AttnKV(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("num_rows", C.c_int64), ("row_stride", C.c_int64),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("layer", C.c_int32),
                ("reserved", C.c_int32)]


class _AttnQuery(C.Structure):
    _fields_ = [("q", C.c_void_p), ("out", C.c_void_p), ("n_seqs", C.c_int32), ("num_q_heads", C.c_int32),
                ("scale", C.c_float), ("reserved", C.c_int32)]


class _PrefillQuery(C.Structure):
    _fields_ = [("q", C.c_void_p), ("out", C.c_void_p), ("lse", C.c_void_p), ("n_seqs", C.c_int32),
                ("q_tokens", C.c_int32), ("num_q_heads", C.c_int32), ("scale", C.c_float)]


class _AttnMlaKV(C.Structure):
    _fields_ = [("kv", C.c_void_p), ("num_rows", C.c_int64), ("row_stride", C.c_int64),
                ("kv_lora_rank", C.c_int32), ("rope_dim", C.c_int32), ("layer", C.c_int32),
                ("reserved", C.c_int32)]


class _MlaStore(C.Structure):
    _fields_ = [("kv", C.c_void_p), ("num_rows", C.c_int64), ("layer_stride", C.c_int64),
                ("row_stride", C.c_int64)]


assert C.sizeof(_Chunk) == 64

_LIB: Optional[C.CDLL] = None


def load_library(path: Optional[str] = None, build_if_missing: bool = True) -> C.CDLL:
    """Load ``libkamera.so`` (building it in-tree with nvcc if absent or stale)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    if path is None:
        path = _build.LIB_PATH
        if build_if_missing:
            _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"Kamera CUDA library not found at {path}; run build()")
    lib = C.CDLL(path)
    P = C.POINTER
    lib.kamera_relocate_patch.restype = C.c_int
    lib.kamera_relocate_patch.argtypes = [P(_GqaPool), P(_GqaStore), P(_Rope), C.c_void_p, C.c_void_p,
                                          C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
    lib.kamera_slide_inplace.restype = C.c_int
    lib.kamera_slide_inplace.argtypes = [P(_SlidePool), P(_Rope), C.c_void_p, C.c_int32, C.c_int32,
                                         C.c_void_p, C.c_void_p]
    lib.kamera_mla_relocate_patch.restype = C.c_int
    lib.kamera_mla_relocate_patch.argtypes = [P(_MlaPool), P(_MlaStore), P(_Rope), C.c_void_p, C.c_void_p,
                                              C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
    lib.kamera_ingest_canonical.restype = C.c_int
    lib.kamera_ingest_canonical.argtypes = [P(_GqaPool), P(_GqaStore), P(_Rope), C.c_void_p, C.c_int32,
                                            C.c_int32, C.c_void_p, C.c_void_p]
    lib.kamera_mla_ingest_canonical.restype = C.c_int
    lib.kamera_mla_ingest_canonical.argtypes = [P(_MlaPool), P(_MlaStore), P(_Rope), C.c_void_p, C.c_int32,
                                                C.c_int32, C.c_void_p, C.c_void_p]
    lib.kamera_form_patch.restype = C.c_int
    lib.kamera_form_patch.argtypes = [P(_Deficit), C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p]
    lib.kamera_attend_reused.restype = C.c_int
    lib.kamera_attend_reused.argtypes = [P(_AttnKV), P(_AttnQuery), P(_Rope), C.c_void_p, C.c_void_p, C.c_int32,
                                         C.c_int32, C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p]
    lib.kamera_mla_attend_reused.restype = C.c_int
    lib.kamera_mla_attend_reused.argtypes = [P(_AttnMlaKV), P(_AttnQuery), P(_Rope), C.c_void_p, C.c_void_p,
                                             C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_size_t, C.c_void_p,
                                             C.c_void_p]
    lib.kamera_prefill_attend_reused.restype = C.c_int
    lib.kamera_prefill_attend_reused.argtypes = [P(_AttnKV), P(_PrefillQuery), P(_Rope), C.c_void_p, C.c_void_p,
                                                 C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
    lib.kamera_attend_reused_static.restype = C.c_int
    lib.kamera_attend_reused_static.argtypes = [P(_AttnKV), P(_AttnQuery), P(_Rope), C.c_void_p, C.c_void_p,
                                                C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]
    lib.kamera_attend_workspace_bytes.restype = C.c_size_t
    lib.kamera_attend_workspace_bytes.argtypes = [C.c_int32, C.c_int32, C.c_int32]
    lib.kamera_mla_attend_workspace_bytes.restype = C.c_size_t
    lib.kamera_mla_attend_workspace_bytes.argtypes = [C.c_int32, C.c_int32]
    lib.kamera_validate_chunks.restype = C.c_int
    lib.kamera_validate_chunks.argtypes = [P(_Chunk), C.c_int32, C.c_int64, C.c_int64, C.c_int32,
                                           C.c_int32, P(C.c_int32), P(C.c_int32)]
    lib.kamera_status_string.restype = C.c_char_p
    lib.kamera_status_string.argtypes = [C.c_int]
    lib.kamera_abi_version.restype = C.c_int
    lib.kamera_abi_version.argtypes = []
    if lib.kamera_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{path} implements Kamera ABI {lib.kamera_abi_version()}, these bindings "
                           f"expect {ABI_VERSION}; rebuild it with build()")
    if path == _build.LIB_PATH:
        _LIB = lib
    return lib


def kamera_status_string(status: int) -> str:
    return load_library().kamera_status_string(int(status)).decode()


ABI_VERSION = 9   # the KAMERA_ABI_VERSION these bindings marshal for


def kamera_abi_version() -> int:
    return int(load_library().kamera_abi_version())


# ------------------------------------------------------------------ helpers
@dataclass
class Rope:
    """RoPE layout (see ``KameraRope``): theta_i = base^(-2i/rot_dim) unless
    ``inv_freq`` is given.

    Multi-axis RoPE: ``freq_axis`` gives, per frequency, the axis it follows
    (0..n_axes-1) and ``axis_delta`` is a device int64 tensor [n_chunks, n_axes]
    of each chunk's move along each axis; the chunks' own deltas are then not
    used for the phases."""
    base: float
    rot_dim: int
    rot_offset: int = 0
    pairing: int = ROTATE_HALF
    inv_freq: Optional[Sequence[float]] = None
    freq_axis: Optional[Sequence[int]] = None
    axis_delta: Optional[torch.Tensor] = None

    def _c(self, n_chunks: int = 0):
        keep = []
        ptr = None
        if self.inv_freq is not None:
            keep.append(np.ascontiguousarray(self.inv_freq, dtype=np.float64))
            ptr = keep[-1].ctypes.data_as(C.POINTER(C.c_double))
        n_axes, axes, dptr = 0, None, None
        if self.axis_delta is not None:
            if (self.freq_axis is None or self.axis_delta.dtype != torch.int64 or self.axis_delta.dim() != 2
                    or not self.axis_delta.is_cuda):
                raise ValueError("axis_delta needs freq_axis and a device int64 [n_chunks, n_axes] tensor")
            if self.axis_delta.shape[0] < int(n_chunks) or len(self.freq_axis) != int(self.rot_dim) // 2:
                raise ValueError("axis_delta needs a row per chunk and freq_axis an entry per frequency")
            n_axes = int(self.axis_delta.shape[1])
            keep.append(self.axis_delta.contiguous())
            dptr = keep[-1].data_ptr()
            keep.append(np.ascontiguousarray(self.freq_axis, dtype=np.uint8))
            axes = keep[-1].ctypes.data_as(C.POINTER(C.c_uint8))
        elif self.freq_axis is not None:
            raise ValueError("freq_axis without axis_delta")
        return _Rope(float(self.base), int(self.rot_dim), int(self.rot_offset), int(self.pairing), n_axes,
                     ptr, axes, dptr), keep


@dataclass
class ChunkSpec:
    """One chunk descriptor before packing.  ``patches`` holds the four bf16
    factor tensors (GQA: Uk, Vk, Uv, Vv; MLA: Uc, Vc, Ur, Vr) or is empty."""
    src_offset: int
    length: int
    delta: int
    rank: int
    slots: torch.Tensor
    patches: Sequence[torch.Tensor] = ()


def _addr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else int(t.data_ptr())


def pack_chunks(chunks: Sequence, device=None) -> torch.Tensor:
    """Marshal chunk descriptors into the 64-byte ``KameraChunk`` layout.

    Accepts ``ChunkSpec``-like objects (attributes src_offset, length, delta,
    rank, slots, patches).  Returns a uint8 tensor on ``device`` (default: the
    slot tensors' device) holding ``len(chunks)`` packed descriptors; the
    referenced tensors must stay alive while the call runs.  The host bytes
    ride along as the attribute ``kamera_host`` (passed to the relocate entry
    points as their ``h_chunks`` copy).
    """
    n = len(chunks)
    arr = (_Chunk * max(n, 1))()
    for i, c in enumerate(chunks):
        ptrs = [0, 0, 0, 0]
        if c.rank > 0:
            for k in range(4):
                ptrs[k] = _addr(c.patches[k])
        arr[i] = _Chunk(int(c.src_offset), int(c.length), int(c.rank), int(c.delta),
                        (C.c_void_p * 4)(*ptrs), _addr(c.slots) if c.length > 0 else 0)
    raw = bytes(arr)[: 64 * n]
    if device is None:
        device = chunks[0].slots.device if n else "cpu"
    host = torch.frombuffer(bytearray(raw), dtype=torch.uint8) if n else torch.empty(0, dtype=torch.uint8)
    out = host.to(device)
    out.kamera_host = host if out.device.type != "cpu" else out
    return out


def _host_copy(chunks: torch.Tensor, host_chunks) -> int:
    """Address of the host descriptor copy: ``host_chunks`` if given (False: none),
    else the copy ``pack_chunks`` attached."""
    if host_chunks is False:
        return 0
    if host_chunks is None:
        host_chunks = getattr(chunks, "kamera_host", None)
    if host_chunks is None:
        return 0
    if host_chunks.device.type != "cpu" or host_chunks.numel() != chunks.numel():
        raise ValueError("host_chunks must be a CPU copy of the packed descriptors")
    return _addr(host_chunks)


def _stream_handle(stream) -> int:
    if stream is None:
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return int(stream.cuda_stream)
    return int(stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise KameraError(rc, where)


def _on_device(where: str, **tensors):
    """Every tensor a compute entry point reads or writes must live in device
    memory: a host address handed to a kernel is not a valid device address.
    Checked wherever CUDA is present (without it no call reaches a kernel, and
    the library's own argument checks can be exercised with host tensors)."""
    if not torch.cuda.is_available():
        return
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{where}: {name} must be a CUDA tensor")


def _bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")


# -------------------------------------------------------------- entry points
def kamera_relocate_patch(pool_k: torch.Tensor, pool_v: torch.Tensor, store_k: torch.Tensor,
                          store_v: torch.Tensor, rope: Rope, chunks: torch.Tensor, n_chunks: int,
                          max_len: int, max_rank: int, err: Optional[torch.Tensor] = None,
                          stream=None, host_chunks=None) -> None:
    """GQA/MHA relocate + patch + paged scatter.

    pool_*: bf16 ``[L, S, H, d]`` (layer/slot strides free, head/dim packed);
    store_*: bf16 ``[L, N, H, d]``; chunks: packed descriptors (``pack_chunks``)
    on the device; err: optional device int32 error word; host_chunks: the
    host copy of ``chunks`` (default: the one ``pack_chunks`` attached; False:
    none, every U tile then moves by per-thread copies).
    """
    _on_device("kamera_relocate_patch", pool_k=pool_k, pool_v=pool_v, store_k=store_k, store_v=store_v,
               chunks=chunks, err=err)
    for t, nm in ((pool_k, "pool_k"), (pool_v, "pool_v"), (store_k, "store_k"), (store_v, "store_v")):
        _bf16(t, nm)
        if t.dim() != 4 or t.stride(3) != 1 or t.stride(2) != t.shape[3]:
            raise ValueError(f"{nm} must be [L, rows, H, d] with packed heads")
    L, S, H, d = pool_k.shape
    pool = _GqaPool(L, H, d, 0, _addr(pool_k), _addr(pool_v), S, pool_k.stride(0), pool_k.stride(1))
    if pool_v.stride() != pool_k.stride() or pool_v.shape != pool_k.shape:
        raise ValueError("pool_k and pool_v must share shape and strides")
    if store_v.stride() != store_k.stride() or store_v.shape != store_k.shape:
        raise ValueError("store_k and store_v must share shape and strides")
    if store_k.shape[0] != L or store_k.shape[2] != H or store_k.shape[3] != d:
        raise ValueError("store and pool disagree on L, H or d")
    store = _GqaStore(_addr(store_k), _addr(store_v), store_k.shape[1], store_k.stride(0), store_k.stride(1))
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_relocate_patch(C.byref(pool), C.byref(store), C.byref(r), _addr(chunks),
                                              _host_copy(chunks, host_chunks), int(n_chunks), int(max_len),
                                              int(max_rank), _addr(err), _stream_handle(stream))
    del keep
    _check(rc, "kamera_relocate_patch")


def kamera_slide_inplace(pool_k: torch.Tensor, rope: Rope, chunks: torch.Tensor, n_chunks: int,
                         max_len: int, err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Sliding-window survival: rotate the key rows at the chunks' slots in place.

    pool_k: bf16 ``[L, S, H, d]`` (for MLA k_rope: ``[L, S, 1, kv_lora + rope]``
    with ``rope.rot_offset = kv_lora``)."""
    _on_device("kamera_slide_inplace", pool_k=pool_k, chunks=chunks, err=err)
    _bf16(pool_k, "pool_k")
    if pool_k.dim() != 4 or pool_k.stride(3) != 1 or pool_k.stride(2) != pool_k.shape[3]:
        raise ValueError("pool_k must be [L, S, H, d] with packed heads")
    L, S, H, d = pool_k.shape
    pool = _SlidePool(L, H, d, 0, _addr(pool_k), S, pool_k.stride(0), pool_k.stride(1))
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_slide_inplace(C.byref(pool), C.byref(r), _addr(chunks), int(n_chunks),
                                             int(max_len), _addr(err), _stream_handle(stream))
    del keep
    _check(rc, "kamera_slide_inplace")


def kamera_mla_relocate_patch(pool: torch.Tensor, store: torch.Tensor, kv_lora: int, rope: Rope,
                              chunks: torch.Tensor, n_chunks: int, max_len: int, max_rank: int,
                              err: Optional[torch.Tensor] = None, stream=None, host_chunks=None) -> None:
    """MLA relocate + patch + paged scatter.  pool: bf16 ``[L, S, kv_lora + rope]``;
    store: bf16 ``[L, N, kv_lora + rope]``; rope offsets relative to k_rope;
    host_chunks as for ``kamera_relocate_patch``."""
    _on_device("kamera_mla_relocate_patch", pool=pool, store=store, chunks=chunks, err=err)
    _bf16(pool, "pool")
    _bf16(store, "store")
    for t, nm in ((pool, "pool"), (store, "store")):
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError(f"{nm} must be [L, rows, width] with packed rows")
    L, S, W = pool.shape
    if store.shape[0] != L or store.shape[2] != W:
        raise ValueError("store and pool disagree on L or row width")
    p = _MlaPool(L, int(kv_lora), W - int(kv_lora), 0, _addr(pool), S, pool.stride(0), pool.stride(1))
    s = _MlaStore(_addr(store), store.shape[1], store.stride(0), store.stride(1))
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_mla_relocate_patch(C.byref(p), C.byref(s), C.byref(r), _addr(chunks),
                                                  _host_copy(chunks, host_chunks), int(n_chunks), int(max_len),
                                                  int(max_rank), _addr(err), _stream_handle(stream))
    del keep
    _check(rc, "kamera_mla_relocate_patch")


def kamera_ingest_canonical(pool_k: torch.Tensor, pool_v: torch.Tensor, store_k: torch.Tensor,
                            store_v: torch.Tensor, rope: Rope, chunks: torch.Tensor, n_chunks: int,
                            max_len: int, err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Canonical ingest (the inverse of relocation): gather each chunk's rows from the
    pool at its slots (``slots`` of the descriptor), turn the keys by R(delta)
    (delta = minus the chunk's start position in the live cache), copy the values,
    and write store rows ``src_offset``.. .  pool_*: bf16 ``[L, S, H, d]``;
    store_*: bf16 ``[L, N, H, d]`` (written); rank 0 descriptors."""
    _on_device("kamera_ingest_canonical", pool_k=pool_k, pool_v=pool_v, store_k=store_k, store_v=store_v,
               chunks=chunks, err=err)
    for t, nm in ((pool_k, "pool_k"), (pool_v, "pool_v"), (store_k, "store_k"), (store_v, "store_v")):
        _bf16(t, nm)
        if t.dim() != 4 or t.stride(3) != 1 or t.stride(2) != t.shape[3]:
            raise ValueError(f"{nm} must be [L, rows, H, d] with packed heads")
    L, S, H, d = pool_k.shape
    if pool_v.stride() != pool_k.stride() or pool_v.shape != pool_k.shape:
        raise ValueError("pool_k and pool_v must share shape and strides")
    if store_v.stride() != store_k.stride() or store_v.shape != store_k.shape:
        raise ValueError("store_k and store_v must share shape and strides")
    if store_k.shape[0] != L or store_k.shape[2] != H or store_k.shape[3] != d:
        raise ValueError("store and pool disagree on L, H or d")
    pool = _GqaPool(L, H, d, 0, _addr(pool_k), _addr(pool_v), S, pool_k.stride(0), pool_k.stride(1))
    store = _GqaStore(_addr(store_k), _addr(store_v), store_k.shape[1], store_k.stride(0), store_k.stride(1))
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_ingest_canonical(C.byref(pool), C.byref(store), C.byref(r), _addr(chunks),
                                                int(n_chunks), int(max_len), _addr(err), _stream_handle(stream))
    del keep
    _check(rc, "kamera_ingest_canonical")


def kamera_mla_ingest_canonical(pool: torch.Tensor, store: torch.Tensor, kv_lora: int, rope: Rope,
                                chunks: torch.Tensor, n_chunks: int, max_len: int,
                                err: Optional[torch.Tensor] = None, stream=None) -> None:
    """MLA canonical ingest: c_KV copied, k_rope turned by R(delta).  pool: bf16
    ``[L, S, kv_lora + rope]``; store: bf16 ``[L, N, kv_lora + rope]`` (written);
    rope offsets relative to k_rope."""
    _on_device("kamera_mla_ingest_canonical", pool=pool, store=store, chunks=chunks, err=err)
    _bf16(pool, "pool")
    _bf16(store, "store")
    for t, nm in ((pool, "pool"), (store, "store")):
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError(f"{nm} must be [L, rows, width] with packed rows")
    L, S, Wd = pool.shape
    if store.shape[0] != L or store.shape[2] != Wd:
        raise ValueError("store and pool disagree on L or row width")
    p = _MlaPool(L, int(kv_lora), Wd - int(kv_lora), 0, _addr(pool), S, pool.stride(0), pool.stride(1))
    s = _MlaStore(_addr(store), store.shape[1], store.stride(0), store.stride(1))
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_mla_ingest_canonical(C.byref(p), C.byref(s), C.byref(r), _addr(chunks),
                                                    int(n_chunks), int(max_len), _addr(err),
                                                    _stream_handle(stream))
    del keep
    _check(rc, "kamera_mla_ingest_canonical")


def _aligned_i64(a) -> np.ndarray:
    """Copy into a 16-byte aligned int64 array (the ABI wants aligned slot maps)."""
    a = np.asarray(a, dtype=np.int64).reshape(-1)
    buf = np.empty(a.size + 2, dtype=np.int64)
    off = (-buf.ctypes.data % 16) // 8
    out = buf[off:off + a.size]
    out[:] = a
    return out


def kamera_validate_chunks(chunks: Sequence, num_store_rows: int, num_slots: int, max_len: int,
                           max_rank: int):
    """Host-side check of descriptors (slot tensors read on the host).

    Returns ``(status, bad_chunk, bad_bits)``; status 0 means valid."""
    n = len(chunks)
    arr = (_Chunk * max(n, 1))()
    keep = []
    for i, c in enumerate(chunks):
        s = _aligned_i64(c.slots.detach().cpu().numpy() if isinstance(c.slots, torch.Tensor) else c.slots)
        keep.append(s)
        ptrs = [0, 0, 0, 0]
        if c.rank > 0:
            ptrs = [_addr(p) if isinstance(p, torch.Tensor) else int(p) for p in c.patches]
        arr[i] = _Chunk(int(c.src_offset), int(c.length), int(c.rank), int(c.delta),
                        (C.c_void_p * 4)(*ptrs), s.ctypes.data if c.length > 0 else 0)
    bad = C.c_int32(-1)
    bits = C.c_int32(0)
    rc = load_library().kamera_validate_chunks(arr, n, int(num_store_rows), int(num_slots), int(max_len),
                                               int(max_rank), C.byref(bad), C.byref(bits))
    del keep
    return int(rc), int(bad.value), int(bits.value)


def kamera_form_patch(delta: torch.Tensor, m: int, u: Optional[torch.Tensor] = None,
                      v: Optional[torch.Tensor] = None, sigma: Optional[torch.Tensor] = None,
                      err: Optional[torch.Tensor] = None, stream=None):
    """Rank-m patch factors of deficit blocks: U V^T is the best rank-m
    approximation of each block, V with orthonormal columns, the singular values
    in U (and in ``sigma`` when given).

    delta: bf16 ``[O, I, rows, cols]`` (any strides with packed columns, e.g. a
    ``[L, len, H, d]`` deficit permuted to ``[L, H, len, d]``), or
    ``[T, O, I, rows, cols]`` to factor the mean over T (the orbit patch).
    u: bf16 ``[O, I, rows, m]``, v: bf16 ``[O, I, cols, m]`` (allocated when
    None), sigma: optional fp32 ``[O, I, m]``.  Returns ``(u, v)``."""
    _on_device("kamera_form_patch", delta=delta, u=u, v=v, sigma=sigma, err=err)
    _bf16(delta, "delta")
    if delta.dim() == 4:
        delta5, t_stride = delta.unsqueeze(0), 0
    elif delta.dim() == 5:
        delta5, t_stride = delta, delta.stride(0)
    else:
        raise ValueError("delta must be [O, I, rows, cols] or [T, O, I, rows, cols]")
    T, O, I, rows, cols = delta5.shape
    if delta5.stride(4) != 1:
        raise ValueError("delta's columns must be packed")
    if u is None:
        u = torch.empty(O, I, rows, m, dtype=torch.bfloat16, device=delta.device)
    if v is None:
        v = torch.empty(O, I, cols, m, dtype=torch.bfloat16, device=delta.device)
    for t, nm, shape in ((u, "u", (O, I, rows, m)), (v, "v", (O, I, cols, m))):
        _bf16(t, nm)
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous {shape} tensor")
    if sigma is not None and (sigma.dtype != torch.float32 or tuple(sigma.shape) != (O, I, m)
                              or not sigma.is_contiguous()):
        raise ValueError(f"sigma must be a contiguous float32 {(O, I, m)} tensor")
    df = _Deficit(_addr(delta5), O, I, delta5.stride(1), delta5.stride(2), delta5.stride(3),
                  t_stride if T > 1 else 0, T, rows, cols, 0)
    rc = load_library().kamera_form_patch(C.byref(df), int(m), _addr(u), _addr(v), _addr(sigma), _addr(err),
                                          _stream_handle(stream))
    _check(rc, "kamera_form_patch")
    return u, v


# Attention workspaces the binding keeps, per (device, stream): a call's
# partial softmax states live there until its merge launch has read them, so
# calls on one stream (which run in order) may share one, and calls on
# different streams get their own.
_WORKSPACES = {}


def _workspace(workspace, need: int, device, stream):
    """(address, bytes) of the attention workspace: the caller's tensor, none
    (workspace=False or nothing needed), or the binding's cached buffer for this
    device and stream, grown to `need` bytes."""
    if workspace is False or (workspace is None and need == 0):
        return None, 0
    if isinstance(workspace, torch.Tensor):
        _on_device("attention workspace", workspace=workspace)
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    key = (torch.device(device).index, _stream_handle(stream))
    buf = _WORKSPACES.get(key)
    if buf is None or buf.numel() < need:
        buf = torch.empty(need, dtype=torch.uint8, device=device)
        _WORKSPACES[key] = buf
    return buf.data_ptr(), buf.numel()


def kamera_attend_reused(store_k: torch.Tensor, store_v: torch.Tensor, q: torch.Tensor, rope: Rope,
                         chunks: torch.Tensor, seq_start: torch.Tensor, n_chunks: int, max_len: int,
                         max_rank: int, layer: int = 0, scale: Optional[float] = None,
                         out: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                         stream=None, workspace=None) -> torch.Tensor:
    """Decode attention of one query token per sequence over its reused chunks,
    never writing a relocated row (see ``kamera_attend_reused`` in kamera.h).

    store_k/v: bf16 ``[N, H_kv, d]`` (one layer; packed heads, any row stride);
    q: bf16 ``[S, H_q, d]`` contiguous; seq_start: device int32 ``[S + 1]``;
    chunks: packed descriptors; layer: the factors' layer index; scale:
    default 1/sqrt(d); workspace: None (a buffer this module keeps per device
    and stream, sized by ``kamera_attend_workspace_bytes``), False (none: the
    cluster path) or a CUDA tensor of the caller's.  Returns ``out`` (bf16
    ``[S, H_q, d]``)."""
    _on_device("kamera_attend_reused", store_k=store_k, store_v=store_v, q=q, chunks=chunks, seq_start=seq_start,
               out=out, err=err)
    for t, nm in ((store_k, "store_k"), (store_v, "store_v"), (q, "q")):
        _bf16(t, nm)
    if store_k.dim() != 3 or store_k.stride(2) != 1 or store_k.stride(1) != store_k.shape[2]:
        raise ValueError("store_k must be [N, H_kv, d] with packed heads")
    if store_v.shape != store_k.shape or store_v.stride() != store_k.stride():
        raise ValueError("store_k and store_v must share shape and strides")
    N, H, d = store_k.shape
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous():
        raise ValueError("q must be a contiguous [S, H_q, d] tensor")
    S, Hq, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if seq_start.dtype != torch.int32 or seq_start.numel() != S + 1:
        raise ValueError("seq_start must hold S + 1 int32 values")
    kv = _AttnKV(_addr(store_k), _addr(store_v), N, store_k.stride(0), H, d, int(layer), 0)
    qq = _AttnQuery(_addr(q), _addr(out), S, Hq, float(d ** -0.5 if scale is None else scale), 0)
    lib = load_library()
    need = lib.kamera_attend_workspace_bytes(S, H, d) if workspace is None and S > 0 else 0
    ws, ws_bytes = _workspace(workspace, need, q.device, stream)
    r, keep = rope._c(n_chunks)
    rc = lib.kamera_attend_reused(C.byref(kv), C.byref(qq), C.byref(r), _addr(chunks), _addr(seq_start),
                                  int(n_chunks), int(max_len), int(max_rank), ws, ws_bytes, _addr(err),
                                  _stream_handle(stream))
    del keep
    _check(rc, "kamera_attend_reused")
    return out


def kamera_attend_reused_static(store_k: torch.Tensor, store_v: torch.Tensor, q: torch.Tensor, rope: Rope,
                                chunks: torch.Tensor, seq_start: torch.Tensor, n_chunks: int, max_len: int,
                                max_rank: int, out: torch.Tensor, layer: int = 0, scale: Optional[float] = None,
                                err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """``kamera_attend_reused`` for callers that cannot allocate device memory
    (see ``kamera_attend_reused_static`` in kamera.h): the library's fixed
    scratch serves as the workspace, and this binding allocates nothing either,
    so the caller passes ``out`` (bf16, shaped like ``q``).  Returns ``out``."""
    _on_device("kamera_attend_reused_static", store_k=store_k, store_v=store_v, q=q, chunks=chunks,
               seq_start=seq_start, out=out, err=err)
    for t, nm in ((store_k, "store_k"), (store_v, "store_v"), (q, "q"), (out, "out")):
        _bf16(t, nm)
    if store_k.dim() != 3 or store_k.stride(2) != 1 or store_k.stride(1) != store_k.shape[2]:
        raise ValueError("store_k must be [N, H_kv, d] with packed heads")
    if store_v.shape != store_k.shape or store_v.stride() != store_k.stride():
        raise ValueError("store_k and store_v must share shape and strides")
    N, H, d = store_k.shape
    if q.dim() != 3 or q.shape[2] != d or not q.is_contiguous():
        raise ValueError("q must be a contiguous [S, H_q, d] tensor")
    S, Hq, _ = q.shape
    if out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if seq_start.dtype != torch.int32 or seq_start.numel() != S + 1:
        raise ValueError("seq_start must hold S + 1 int32 values")
    kv = _AttnKV(_addr(store_k), _addr(store_v), N, store_k.stride(0), H, d, int(layer), 0)
    qq = _AttnQuery(_addr(q), _addr(out), S, Hq, float(d ** -0.5 if scale is None else scale), 0)
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_attend_reused_static(C.byref(kv), C.byref(qq), C.byref(r), _addr(chunks),
                                                    _addr(seq_start), int(n_chunks), int(max_len), int(max_rank),
                                                    _addr(err), _stream_handle(stream))
    del keep
    _check(rc, "kamera_attend_reused_static")
    return out


def kamera_prefill_attend_reused(store_k: torch.Tensor, store_v: torch.Tensor, q: torch.Tensor, rope: Rope,
                                 chunks: torch.Tensor, seq_start: torch.Tensor, n_chunks: int, max_len: int,
                                 max_rank: int, layer: int = 0, scale: Optional[float] = None,
                                 out: Optional[torch.Tensor] = None, lse=None, err: Optional[torch.Tensor] = None,
                                 stream=None):
    """Prefill attention of T new query tokens per sequence over its reused
    chunks (see ``kamera_prefill_attend_reused`` in kamera.h).

    store_k/v: bf16 ``[N, H_kv, d]`` (one layer; packed heads, any row stride);
    q: bf16 ``[S, T, H_q, d]`` contiguous; seq_start: device int32 ``[S + 1]``;
    lse: None (allocated: fp32 ``[S, T, H_q]``), False (not computed) or a
    contiguous fp32 tensor of that shape.  Returns ``(out, lse)`` (lse None
    when not computed)."""
    _on_device("kamera_prefill_attend_reused", store_k=store_k, store_v=store_v, q=q, chunks=chunks,
               seq_start=seq_start, out=out, err=err, lse=lse if isinstance(lse, torch.Tensor) else None)
    for t, nm in ((store_k, "store_k"), (store_v, "store_v"), (q, "q")):
        _bf16(t, nm)
    if store_k.dim() != 3 or store_k.stride(2) != 1 or store_k.stride(1) != store_k.shape[2]:
        raise ValueError("store_k must be [N, H_kv, d] with packed heads")
    if store_v.shape != store_k.shape or store_v.stride() != store_k.stride():
        raise ValueError("store_k and store_v must share shape and strides")
    N, H, d = store_k.shape
    if q.dim() != 4 or q.shape[3] != d or not q.is_contiguous():
        raise ValueError("q must be a contiguous [S, T, H_q, d] tensor")
    S, T, Hq, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse is None:
        lse = torch.empty(S, T, Hq, dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    if lse is not None and (tuple(lse.shape) != (S, T, Hq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [S, T, H_q] tensor")
    if seq_start.dtype != torch.int32 or seq_start.numel() != S + 1:
        raise ValueError("seq_start must hold S + 1 int32 values")
    kv = _AttnKV(_addr(store_k), _addr(store_v), N, store_k.stride(0), H, d, int(layer), 0)
    qq = _PrefillQuery(_addr(q), _addr(out), _addr(lse), S, T, Hq, float(d ** -0.5 if scale is None else scale))
    r, keep = rope._c(n_chunks)
    rc = load_library().kamera_prefill_attend_reused(C.byref(kv), C.byref(qq), C.byref(r), _addr(chunks),
                                                     _addr(seq_start), int(n_chunks), int(max_len), int(max_rank),
                                                     _addr(err), _stream_handle(stream))
    del keep
    _check(rc, "kamera_prefill_attend_reused")
    return out, lse


def kamera_mla_attend_reused(store: torch.Tensor, kv_lora: int, q: torch.Tensor, rope: Rope, chunks: torch.Tensor,
                             seq_start: torch.Tensor, n_chunks: int, max_len: int, max_rank: int, layer: int = 0,
                             scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                             err: Optional[torch.Tensor] = None, stream=None, workspace=None) -> torch.Tensor:
    """MLA decode attention (absorbed form) of one query token per sequence over
    its reused chunks (see ``kamera_mla_attend_reused`` in kamera.h).

    store: bf16 ``[N, kv_lora + rope_dim]`` (one layer, any row stride);
    q: bf16 ``[S, H_q, kv_lora + rope_dim]`` contiguous (latent query, then
    rope query); seq_start: device int32 ``[S + 1]``; rope: rot_offset
    relative to k_rope; scale: default 1/sqrt(kv_lora + rope_dim); workspace:
    as for ``kamera_attend_reused``.  Returns ``out`` (bf16 ``[S, H_q, kv_lora]``)."""
    _on_device("kamera_mla_attend_reused", store=store, q=q, chunks=chunks, seq_start=seq_start, out=out, err=err)
    for t, nm in ((store, "store"), (q, "q")):
        _bf16(t, nm)
    if store.dim() != 2 or store.stride(1) != 1:
        raise ValueError("store must be [N, kv_lora + rope_dim] with packed rows")
    N, W = store.shape
    if q.dim() != 3 or q.shape[2] != W or not q.is_contiguous():
        raise ValueError("q must be a contiguous [S, H_q, kv_lora + rope_dim] tensor")
    S, Hq, _ = q.shape
    if out is None:
        out = torch.empty(S, Hq, kv_lora, dtype=torch.bfloat16, device=q.device)
    if tuple(out.shape) != (S, Hq, kv_lora) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 [S, H_q, kv_lora] tensor")
    if seq_start.dtype != torch.int32 or seq_start.numel() != S + 1:
        raise ValueError("seq_start must hold S + 1 int32 values")
    kv = _AttnMlaKV(_addr(store), N, store.stride(0), int(kv_lora), int(W - kv_lora), int(layer), 0)
    qq = _AttnQuery(_addr(q), _addr(out), S, Hq, float(W ** -0.5 if scale is None else scale), 0)
    lib = load_library()
    need = lib.kamera_mla_attend_workspace_bytes(S, Hq) if workspace is None and S > 0 else 0
    ws, ws_bytes = _workspace(workspace, need, q.device, stream)
    r, keep = rope._c(n_chunks)
    rc = lib.kamera_mla_attend_reused(C.byref(kv), C.byref(qq), C.byref(r), _addr(chunks), _addr(seq_start),
                                      int(n_chunks), int(max_len), int(max_rank), ws, ws_bytes, _addr(err),
                                      _stream_handle(stream))
    del keep
    _check(rc, "kamera_mla_attend_reused")
    return out
