"""fp64 CPU oracle of the Kamera reuse operator -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The CUDA product path
(``position_invariant_kv_chunk_gb300``) never imports it and shares no code
with it; the two meet only in the seeded input generators (``workloads``).

The arithmetic lives in ``kamera_oracle.c`` (plain loops, fp64, one direct
fp64 -> bf16 round-to-nearest-even).  This module builds it with gcc, loads it
with ctypes and adds numpy conveniences.  What it follows ("Kamera: Unified
Position-Invariant Multimodal KV Cache for Training-Free Reuse", gist.science
technical summary):

* section 2, reuse equation  KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T   -> ``row``,
  ``gqa``, ``mla``
* section 2, patch formation (one conditioned forward, then an SVD keeping the
  top-m factors)                                                      -> ``form_patch``
* section 3.2, sliding-window survival by rotation only               -> ``slide``
* attention over reused chunks (the pages' attention-kernel hook, section 3):
  softmax attention of a decode query over the reuse equation's rows -> ``attend``,
  and its MLA form over the latent rows (absorbed query)                 -> ``attend_mla``;
  many new query tokens at once (prefill), with each row's log-sum-exp -> ``attend_prefill``

Pinned by ``tests/test_oracle_pins.py`` (closed forms, group laws of R, an
independent complex-number RoPE, brute-force bf16 rounding, Eckart-Young by
eigen-decomposition, bit-exact copies) and ``tests/test_oracle_mutants.py``
(planted mistakes in this oracle's source must fail a pin).  The pages'
accuracy and KL figures need trained weights and datasets: parity unpinned.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import tempfile
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "kamera_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libkamera_oracle.so")

ROTATE_HALF = 0
INTERLEAVED = 1

_u16p = C.POINTER(C.c_uint16)
_f64p = C.POINTER(C.c_double)
_i64p = C.POINTER(C.c_int64)
_i32p = C.POINTER(C.c_int32)


def build(out_path: str = LIB_PATH, source: str = SOURCE, openmp: bool = True) -> str:
    """Compile the oracle into a shared library (gcc, fp64, no FMA contraction).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded on
    both x86-64 and aarch64, so the oracle gives the same bits on either host.
    """
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
            source, "-o", out_path + ".tmp", "-lm"]
    cmds = [base[:1] + ["-fopenmp"] + base[1:]] if openmp else []
    cmds.append(base)
    last = None
    for cmd in cmds:
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(out_path + ".tmp", out_path)
            return out_path
        last = r
    raise RuntimeError(f"oracle build failed:\n{last.stderr}")


def _declare(lib: C.CDLL) -> C.CDLL:
    lib.kamera_oracle_bf16_rne.restype = C.c_uint16
    lib.kamera_oracle_bf16_rne.argtypes = [C.c_double]
    lib.kamera_oracle_bf16_to_f64.restype = C.c_double
    lib.kamera_oracle_bf16_to_f64.argtypes = [C.c_uint16]
    lib.kamera_oracle_bf16_rne_array.argtypes = [_f64p, C.c_int64, _u16p]
    lib.kamera_oracle_bf16_to_f64_array.argtypes = [_u16p, C.c_int64, _f64p]
    lib.kamera_oracle_inv_freq.argtypes = [C.c_double, C.c_int, _f64p]
    lib.kamera_oracle_rotate.argtypes = [_f64p, C.c_int, C.c_int64, _f64p, C.c_int, C.c_int,
                                         C.c_int, _f64p]
    lib.kamera_oracle_row.argtypes = [_u16p, C.c_int, C.c_int, C.c_int64, _f64p, C.c_int,
                                      C.c_int, C.c_int, _u16p, _u16p, C.c_int, _u16p, _f64p,
                                      _f64p]
    P = C.POINTER(_u16p)
    S = C.POINTER(_i64p)
    lib.kamera_oracle_gqa.restype = C.c_int
    lib.kamera_oracle_gqa.argtypes = [
        C.c_int, C.c_int, C.c_int,
        _u16p, _u16p, C.c_int64, C.c_int64, C.c_int64,
        _u16p, _u16p, C.c_int64, C.c_int64, C.c_int64,
        _f64p, C.c_int, C.c_int, C.c_int,
        C.c_int, _i64p, _i32p, _i64p, _i32p, P, P, P, P, S, _f64p, _f64p]
    lib.kamera_oracle_mla.restype = C.c_int
    lib.kamera_oracle_mla.argtypes = [
        C.c_int, C.c_int, C.c_int,
        _u16p, C.c_int64, C.c_int64, C.c_int64,
        _u16p, C.c_int64, C.c_int64, C.c_int64,
        _f64p, C.c_int,
        C.c_int, _i64p, _i32p, _i64p, _i32p, P, P, P, P, S, _f64p]
    lib.kamera_oracle_slide.restype = C.c_int
    lib.kamera_oracle_slide.argtypes = [
        C.c_int, C.c_int, C.c_int, _u16p, C.c_int64, C.c_int64, C.c_int64,
        _f64p, C.c_int, C.c_int, C.c_int,
        C.c_int, _i32p, _i64p, S, _f64p]
    lib.kamera_oracle_ingest.restype = C.c_int
    lib.kamera_oracle_ingest.argtypes = [
        C.c_int, C.c_int, C.c_int, _u16p, _u16p, C.c_int64, C.c_int64, C.c_int64,
        _u16p, _u16p, C.c_int64, C.c_int64, C.c_int64,
        _f64p, C.c_int, C.c_int, C.c_int,
        C.c_int, _i64p, _i32p, _i64p, S, _f64p]
    lib.kamera_oracle_num_threads.restype = C.c_int
    lib.kamera_oracle_num_threads.argtypes = []
    return lib


def _ptr(a: Optional[np.ndarray], t):
    if a is None:
        return None
    return a.ctypes.data_as(t)


def _c_u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 bit patterns must be uint16, got {a.dtype}")
    return a


@dataclass
class Chunk:
    """One chunk of work as the oracle sees it (its own description, host arrays).

    ``patches`` holds the four bf16 factor arrays (uint16 bit patterns) or is
    empty when ``rank == 0``; their meaning depends on the problem (GQA:
    Uk, Vk, Uv, Vv; MLA: Uc, Vc, Ur, Vr).
    """
    src_offset: int
    length: int
    delta: int
    rank: int
    slots: np.ndarray
    patches: Sequence[np.ndarray] = field(default_factory=tuple)


class Oracle:
    """ctypes front end to one build of ``kamera_oracle.c``."""

    def __init__(self, lib_path: Optional[str] = None):
        if lib_path is None:
            lib_path = LIB_PATH
            if not os.path.exists(lib_path) or os.path.getmtime(lib_path) < os.path.getmtime(SOURCE):
                build(lib_path)
        self.lib = _declare(C.CDLL(lib_path))

    # -------------------------------------------------------------- bf16
    def bf16_rne(self, x) -> np.ndarray:
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.kamera_oracle_bf16_rne_array(_ptr(x, _f64p), x.size, _ptr(out, _u16p))
        return out

    def bf16_to_f64(self, bits) -> np.ndarray:
        bits = _c_u16(np.asarray(bits))
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.kamera_oracle_bf16_to_f64_array(_ptr(bits, _u16p), bits.size, _ptr(out, _f64p))
        return out

    # -------------------------------------------------------------- RoPE
    def inv_freq(self, base: float, rot_dim: int) -> np.ndarray:
        out = np.empty(rot_dim // 2, dtype=np.float64)
        self.lib.kamera_oracle_inv_freq(float(base), int(rot_dim), _ptr(out, _f64p))
        return out

    def rotate(self, x, delta: int, inv_freq, rot_dim: int, rot_offset: int = 0,
               pairing: int = ROTATE_HALF, want_scale: bool = False):
        """R(delta) on every row of ``x`` (fp64, ``[..., width]``); returns a new array."""
        y = np.array(x, dtype=np.float64, copy=True, order="C")
        f = np.ascontiguousarray(inv_freq, dtype=np.float64)
        width = y.shape[-1]
        rows = y.reshape(-1, width)
        sc = np.empty_like(rows) if want_scale else None
        for i in range(rows.shape[0]):
            r = rows[i]
            self.lib.kamera_oracle_rotate(
                r.ctypes.data_as(_f64p), width, int(delta), _ptr(f, _f64p), rot_dim, rot_offset,
                pairing, sc[i].ctypes.data_as(_f64p) if sc is not None else None)
        if want_scale:
            return y, sc.reshape(y.shape)
        return y

    def row(self, x_bits, rotate: bool, delta: int, inv_freq, rot_dim: int, rot_offset: int = 0,
            pairing: int = ROTATE_HALF, u=None, vm=None):
        """One output row.  Returns (bf16 bits, fp64 value, magnitude scale)."""
        x_bits = _c_u16(np.asarray(x_bits))
        width = x_bits.shape[-1]
        f = np.ascontiguousarray(inv_freq, dtype=np.float64)
        m = 0
        if u is not None:
            u = _c_u16(np.asarray(u))
            vm = _c_u16(np.asarray(vm))
            m = u.shape[-1]
            if vm.shape != (width, m):
                raise ValueError("vm must be [width, m]")
        ob = np.empty(width, dtype=np.uint16)
        of = np.empty(width, dtype=np.float64)
        osc = np.empty(width, dtype=np.float64)
        self.lib.kamera_oracle_row(_ptr(x_bits, _u16p), width, int(bool(rotate)), int(delta),
                                   _ptr(f, _f64p), rot_dim, rot_offset, pairing,
                                   _ptr(u, _u16p), _ptr(vm, _u16p), m,
                                   _ptr(ob, _u16p), _ptr(of, _f64p), _ptr(osc, _f64p))
        return ob, of, osc

    # ---------------------------------------------------- whole problems
    @staticmethod
    def _chunk_arrays(chunks: Sequence[Chunk]):
        n = len(chunks)
        src = np.array([c.src_offset for c in chunks], dtype=np.int64)
        ln = np.array([c.length for c in chunks], dtype=np.int32)
        de = np.array([c.delta for c in chunks], dtype=np.int64)
        rk = np.array([c.rank for c in chunks], dtype=np.int32)
        keep = []
        slots = []
        for c in chunks:
            s = np.ascontiguousarray(c.slots, dtype=np.int64)
            if s.shape != (c.length,):
                raise ValueError("slots must have one entry per token")
            keep.append(s)
            slots.append(s.ctypes.data_as(_i64p))
        pp = [(_u16p * max(n, 1))() for _ in range(4)]
        for i, c in enumerate(chunks):
            if c.rank > 0:
                if len(c.patches) != 4:
                    raise ValueError("rank > 0 needs four patch factors")
                for k in range(4):
                    a = _c_u16(c.patches[k])
                    keep.append(a)
                    pp[k][i] = a.ctypes.data_as(_u16p)
        sp = (_i64p * max(n, 1))(*slots)
        return n, src, ln, de, rk, pp, sp, keep

    def gqa(self, store_k, store_v, pool_k, pool_v, chunks: Sequence[Chunk], inv_freq,
            rot_dim: int, rot_offset: int = 0, pairing: int = ROTATE_HALF,
            want_scale: bool = False):
        """GQA/MHA relocate + patch + scatter into ``pool_k``/``pool_v`` (in place).

        ``store_*``: uint16 ``[L, N_store, H, d]``; ``pool_*``: uint16 ``[L, S, H, d]``
        (C-contiguous).  Patch factors per chunk: Uk, Vk, Uv, Vv with U
        ``[L, H, len, m]`` and V_m ``[L, H, d, m]``.  Returns the scale arrays
        (pool-shaped, fp64) when ``want_scale``.
        """
        for a in (store_k, store_v, pool_k, pool_v):
            if a.dtype != np.uint16 or not a.flags.c_contiguous:
                raise TypeError("store/pool must be C-contiguous uint16")
        L, N, H, d = store_k.shape
        S = pool_k.shape[1]
        f = np.ascontiguousarray(inv_freq, dtype=np.float64)
        n, src, ln, de, rk, pp, sp, keep = self._chunk_arrays(chunks)
        sk = np.zeros(pool_k.shape) if want_scale else None
        sv = np.zeros(pool_v.shape) if want_scale else None
        rc = self.lib.kamera_oracle_gqa(
            L, H, d, _ptr(store_k, _u16p), _ptr(store_v, _u16p), N, N * H * d, H * d,
            _ptr(pool_k, _u16p), _ptr(pool_v, _u16p), S, S * H * d, H * d,
            _ptr(f, _f64p), rot_dim, rot_offset, pairing,
            n, _ptr(src, _i64p), _ptr(ln, _i32p), _ptr(de, _i64p), _ptr(rk, _i32p),
            pp[0], pp[1], pp[2], pp[3], sp, _ptr(sk, _f64p), _ptr(sv, _f64p))
        if rc != 0:
            raise ValueError("oracle: index out of range in the chunk list")
        del keep
        return (sk, sv) if want_scale else None

    def mla(self, store, pool, chunks: Sequence[Chunk], kv_lora: int, inv_freq,
            pairing: int = INTERLEAVED, want_scale: bool = False):
        """MLA relocate + patch + scatter into ``pool`` (in place).

        ``store``: uint16 ``[L, N_store, kv_lora + rope]``; ``pool``: uint16
        ``[L, S, kv_lora + rope]``.  Factors per chunk: Uc ``[L, len, m]``, Vc
        ``[L, kv_lora, m]``, Ur ``[L, len, m]``, Vr ``[L, rope, m]``.
        """
        for a in (store, pool):
            if a.dtype != np.uint16 or not a.flags.c_contiguous:
                raise TypeError("store/pool must be C-contiguous uint16")
        L, N, W = store.shape
        S = pool.shape[1]
        rope = W - kv_lora
        f = np.ascontiguousarray(inv_freq, dtype=np.float64)
        n, src, ln, de, rk, pp, sp, keep = self._chunk_arrays(chunks)
        sc = np.zeros(pool.shape) if want_scale else None
        rc = self.lib.kamera_oracle_mla(
            L, kv_lora, rope, _ptr(store, _u16p), N, N * W, W,
            _ptr(pool, _u16p), S, S * W, W, _ptr(f, _f64p), pairing,
            n, _ptr(src, _i64p), _ptr(ln, _i32p), _ptr(de, _i64p), _ptr(rk, _i32p),
            pp[0], pp[1], pp[2], pp[3], sp, _ptr(sc, _f64p))
        if rc != 0:
            raise ValueError("oracle: index out of range in the chunk list")
        del keep
        return sc if want_scale else None

    def slide(self, pool_k, chunks: Sequence[Chunk], inv_freq, rot_dim: int, rot_offset: int = 0,
              pairing: int = ROTATE_HALF, want_scale: bool = False):
        """Rotation-only in-place relocation of the key rows at each chunk's slots.

        ``pool_k``: uint16 ``[L, S, H, d]``.  ``src_offset`` and ``rank`` of
        the chunks are ignored.
        """
        if pool_k.dtype != np.uint16 or not pool_k.flags.c_contiguous:
            raise TypeError("pool must be C-contiguous uint16")
        L, S, H, d = pool_k.shape
        f = np.ascontiguousarray(inv_freq, dtype=np.float64)
        n, src, ln, de, rk, pp, sp, keep = self._chunk_arrays(
            [Chunk(0, c.length, c.delta, 0, c.slots) for c in chunks])
        sc = np.zeros(pool_k.shape) if want_scale else None
        rc = self.lib.kamera_oracle_slide(
            L, H, d, _ptr(pool_k, _u16p), S, S * H * d, H * d, _ptr(f, _f64p), rot_dim,
            rot_offset, pairing, n, _ptr(ln, _i32p), _ptr(de, _i64p), sp, _ptr(sc, _f64p))
        if rc != 0:
            raise ValueError("oracle: index out of range in the chunk list")
        del keep
        return sc if want_scale else None

    def ingest(self, pool_k, pool_v, store_k, store_v, chunks: Sequence[Chunk], inv_freq, rot_dim: int,
               rot_offset: int = 0, pairing: int = ROTATE_HALF, want_scale: bool = False):
        """Canonical ingest: gather each chunk's rows from its slots, turn the keys by
        R(delta) (delta = minus the chunk's start position in the live cache) and
        write them to the store rows src_offset.. (``src_offset`` names the first
        store row written; ``rank`` is ignored).  ``pool_*``: uint16 ``[L, S, H, d]``,
        ``store_*``: uint16 ``[L, N, H, d]`` (``*_v`` may be None: MLA rows or keys only).
        """
        for t in (pool_k, store_k) + tuple(x for x in (pool_v, store_v) if x is not None):
            if t.dtype != np.uint16 or not t.flags.c_contiguous:
                raise TypeError("arrays must be C-contiguous uint16")
        if (pool_v is None) != (store_v is None):
            raise ValueError("pool_v and store_v go together")
        L, S, H, d = pool_k.shape
        N = store_k.shape[1]
        f = np.ascontiguousarray(inv_freq, dtype=np.float64)
        n, src, ln, de, rk, pp, sp, keep = self._chunk_arrays(
            [Chunk(c.src_offset, c.length, c.delta, 0, c.slots) for c in chunks])
        sc = np.zeros(store_k.shape) if want_scale else None
        rc = self.lib.kamera_oracle_ingest(
            L, H, d, _ptr(pool_k, _u16p), _ptr(pool_v, _u16p), S, S * H * d, H * d,
            _ptr(store_k, _u16p), _ptr(store_v, _u16p), N, N * H * d, H * d,
            _ptr(f, _f64p), rot_dim, rot_offset, pairing, n, _ptr(src, _i64p), _ptr(ln, _i32p),
            _ptr(de, _i64p), sp, _ptr(sc, _f64p))
        if rc != 0:
            raise ValueError("oracle: index out of range in the chunk list")
        del keep
        return sc if want_scale else None

    def attend(self, store_k, store_v, chunks: Sequence[Chunk], seq_starts, q, layer: int, inv_freq,
               rot_dim: int, rot_offset: int = 0, pairing: int = ROTATE_HALF, scale: float = None):
        """Decode attention of one query token per sequence over its reused chunks,
        each chunk's keys and values being the reuse equation's rows (technical
        summary section 2: K = R(delta) K_canonical + U_k V_k^T, V = V_canonical +
        U_v V_v^T), exact and unrounded (fp64), then softmax(scale q K^T) V.

        ``store_*``: uint16 ``[N, H_kv, d]`` (one layer); ``q``: uint16
        ``[S, H_q, d]`` (RoPE already applied at the query's position); sequence
        s attends over chunks ``seq_starts[s] .. seq_starts[s+1]-1`` in order;
        factors ``[L, H_kv, len, m]`` / ``[L, H_kv, d, m]`` read at ``layer``.
        Returns (bf16 bits ``[S, H_q, d]``, fp64 output, magnitude scale
        sum_j p_j |V_j| per element).  ``q`` and the factors may also be given
        as fp64 values (for the pins).  ``inv_freq`` is one table, or one row
        per chunk (chunks whose multi-axis moves differ: each chunk's phases
        are its own per-frequency products delta_f * theta_f)."""
        N, H, d = store_k.shape
        S, Hq, _ = q.shape
        G = Hq // H
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        f64 = lambda a: a if np.asarray(a).dtype == np.float64 else self.bf16_to_f64(a)
        kf, vf, qf = self.bf16_to_f64(store_k), self.bf16_to_f64(store_v), f64(q)
        out = np.zeros((S, Hq, d))
        mag = np.zeros((S, Hq, d))
        for s in range(S):
            for g in range(H):
                Ks, Vs = [], []
                for ci in range(seq_starts[s], seq_starts[s + 1]):
                    c = chunks[ci]
                    th = inv_freq[ci] if np.ndim(inv_freq) == 2 else inv_freq
                    rows = slice(c.src_offset, c.src_offset + c.length)
                    kk = self.rotate(kf[rows, g, :], c.delta, th, rot_dim, rot_offset, pairing)
                    vv = vf[rows, g, :].copy()
                    if c.rank > 0:
                        uk, vk, uv, vvm = (f64(a)[layer, g] for a in c.patches)
                        kk = kk + uk @ vk.T
                        vv = vv + uv @ vvm.T
                    Ks.append(kk)
                    Vs.append(vv)
                K = np.concatenate(Ks) if Ks else np.zeros((0, d))
                V = np.concatenate(Vs) if Vs else np.zeros((0, d))
                for h in range(g * G, (g + 1) * G):
                    if K.shape[0] == 0:
                        continue
                    sc = scale * (K @ qf[s, h])
                    w = np.exp(sc - sc.max())
                    pr = w / w.sum()
                    out[s, h] = pr @ V
                    mag[s, h] = pr @ np.abs(V)
        return self.bf16_rne(out), out, mag

    def attend_prefill(self, store_k, store_v, chunks: Sequence[Chunk], seq_starts, q, layer: int, inv_freq,
                       rot_dim: int, rot_offset: int = 0, pairing: int = ROTATE_HALF, scale: float = None):
        """Prefill attention of T new query tokens per sequence over its reused
        chunks: every token attends, in one softmax and with no mask (the chunks
        precede the new tokens), over the reuse equation's rows of the sequence's
        chunks (technical summary section 2; served by the attention-kernel hook
        of section 3), exact and unrounded (fp64), and also gets the
        log-sum-exp of its scores, lse = log sum_j exp(scale q . K_j).

        ``q``: uint16 ``[S, T, H_q, d]`` (or fp64); the rest as for ``attend``.
        Returns (bf16 bits ``[S, T, H_q, d]``, fp64 output, magnitude scale
        sum_j p_j |V_j| per element, lse ``[S, T, H_q]``; -inf and zeros for a
        sequence with no token)."""
        N, H, d = store_k.shape
        S, T, Hq, _ = q.shape
        G = Hq // H
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        f64 = lambda a: a if np.asarray(a).dtype == np.float64 else self.bf16_to_f64(a)
        kf, vf, qf = self.bf16_to_f64(store_k), self.bf16_to_f64(store_v), f64(q)
        out = np.zeros((S, T, Hq, d))
        mag = np.zeros((S, T, Hq, d))
        lse = np.full((S, T, Hq), -np.inf)
        for s in range(S):
            for g in range(H):
                # the rows of this KV head over the sequence's chunks, in order
                Ks, Vs = [], []
                for ci in range(seq_starts[s], seq_starts[s + 1]):
                    c = chunks[ci]
                    th = inv_freq[ci] if np.ndim(inv_freq) == 2 else inv_freq
                    rows = slice(c.src_offset, c.src_offset + c.length)
                    kk = self.rotate(kf[rows, g, :], c.delta, th, rot_dim, rot_offset, pairing)
                    vv = vf[rows, g, :].copy()
                    if c.rank > 0:
                        uk, vk, uv, vvm = (f64(a)[layer, g] for a in c.patches)
                        kk = kk + uk @ vk.T
                        vv = vv + uv @ vvm.T
                    Ks.append(kk)
                    Vs.append(vv)
                if not Ks or sum(k.shape[0] for k in Ks) == 0:
                    continue
                K, V = np.concatenate(Ks), np.concatenate(Vs)
                for t in range(T):
                    for h in range(g * G, (g + 1) * G):
                        sc = scale * (K @ qf[s, t, h])
                        mx = sc.max()
                        w = np.exp(sc - mx)
                        den = w.sum()
                        pr = w / den
                        out[s, t, h] = pr @ V
                        mag[s, t, h] = pr @ np.abs(V)
                        lse[s, t, h] = mx + np.log(den)
        return self.bf16_rne(out), out, mag, lse

    def attend_mla(self, store, chunks: Sequence[Chunk], seq_starts, q, layer: int, kv_lora: int, inv_freq,
                   rot_dim: int, rot_offset: int = 0, pairing: int = INTERLEAVED, scale: float = None):
        """MLA decode attention (absorbed form) of one query token per sequence over
        its reused chunks.  Each chunk's rows are the MLA reuse rows (technical
        summary section 2, with section 3's MLA rule: c_KV carried over, the
        decoupled k_rope turned), exact and unrounded (fp64):
            c' = c + U_c V_c^T,   kr' = R(delta) kr + U_r V_r^T
        and query head h (latent part q_lat, rope part q_rope) attends with
        softmax_j(scale (q_lat . c'_j + q_rope . kr'_j)) over c'_j.

        ``store``: uint16 ``[N, kv_lora + rope]`` (one layer); ``q``: uint16
        ``[S, H_q, kv_lora + rope]``; factors Uc ``[L, len, m]``, Vc ``[L, kv_lora,
        m]``, Ur ``[L, len, m]``, Vr ``[L, rope, m]`` read at ``layer``;
        ``rot_offset`` is relative to k_rope; ``inv_freq`` one table or one row per
        chunk.  Returns (bf16 bits ``[S, H_q, kv_lora]``, fp64 output, magnitude
        sum_j p_j |c'_j| per element).  ``q`` and the factors may be fp64."""
        N, Wd = store.shape
        S, Hq, _ = q.shape
        scale = 1.0 / np.sqrt(Wd) if scale is None else float(scale)
        f64 = lambda a: a if np.asarray(a).dtype == np.float64 else self.bf16_to_f64(a)
        sf, qf = self.bf16_to_f64(store), f64(q)
        out = np.zeros((S, Hq, kv_lora))
        mag = np.zeros((S, Hq, kv_lora))
        for s in range(S):
            lat, keys = [], []
            for ci in range(seq_starts[s], seq_starts[s + 1]):
                c = chunks[ci]
                th = inv_freq[ci] if np.ndim(inv_freq) == 2 else inv_freq
                rows = slice(c.src_offset, c.src_offset + c.length)
                cl = sf[rows, :kv_lora].copy()
                kr = self.rotate(sf[rows, kv_lora:], c.delta, th, rot_dim, rot_offset, pairing)
                if c.rank > 0:
                    uc, vc, ur, vr = (f64(a)[layer] for a in c.patches)
                    cl = cl + uc @ vc.T
                    kr = kr + ur @ vr.T
                lat.append(cl)
                keys.append(np.concatenate([cl, kr], axis=1))
            if not keys or sum(k.shape[0] for k in keys) == 0:
                continue
            K, V = np.concatenate(keys), np.concatenate(lat)
            for h in range(Hq):
                sc = scale * (K @ qf[s, h])
                w = np.exp(sc - sc.max())
                pr = w / w.sum()
                out[s, h] = pr @ V
                mag[s, h] = pr @ np.abs(V)
        return self.bf16_rne(out), out, mag

    def num_threads(self) -> int:
        return int(self.lib.kamera_oracle_num_threads())


def form_patch(delta: np.ndarray, m: int):
    """Rank-m conditioning patch from a deficit matrix (technical summary section 2).

    The pages form the patch once per chunk from Delta = KV(B|A) - KV(B|empty)
    by an SVD and keep the top-m factors.  With Delta = W diag(s) Z^T
    (singular values descending), the singular values are absorbed into U:
    ``U = W[:, :m] * s[:m]`` (``[T, m]``) and ``V = Z[:, :m]`` (``[d, m]``),
    so that ``U @ V.T`` is the best rank-m approximation of Delta.
    """
    delta = np.asarray(delta, dtype=np.float64)
    w, s, zt = np.linalg.svd(delta, full_matrices=False)
    m = int(m)
    return w[:, :m] * s[:m], zt[:m, :].T.copy()


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
