"""Shared test plumbing: run a workload through the C ABI on the GPU, run the
same seeded inputs through the fp64 oracle on the host, and compare.

Tolerances (stated for the operator: within 1 bf16 ulp per element of the
fp64 result rounded to bf16; relative Frobenius error <= 4e-3 per (layer,
head) block; bit-exact for copies and indexing):

* every element: |ord(gpu) - ord(oracle)| <= 1 in the ordered bf16 encoding
  (adjacent representable values, across binade boundaries and +-0);
* elements beyond 1 ulp are accepted only as cancellation: the true value is
  small against the terms that made it, so fp32 rounding of those terms moves
  it by more than a bf16 ulp of the result.  They must satisfy
  |gpu - oracle| <= 2^-8 * scale, scale = |x cos| + |y sin| + sum |u_r v_r|
  (the oracle's per-element magnitude), and be rare (<= 1e-4 of the elements
  compared, plus 2);
* per (layer, head) block: ||gpu - oracle||_F <= 4e-3 ||oracle||_F.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass

import numpy as np
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy array of its bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _ordered_table() -> np.ndarray:
    b = np.arange(65536, dtype=np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b).astype(np.int32)


_ORDERED = _ordered_table()


def ordered(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers whose differences count representable steps
    (+0 and -0 both map to 0)."""
    return _ORDERED[np.asarray(bits, dtype=np.uint16)]


def to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Stats:
    """Outcome of one comparison (or of several, summed with +): elements
    compared, elements beyond 1 ulp (every one accepted as cancellation, see
    above; compare raises otherwise), the largest ulp distance and the worst
    relative Frobenius error of a (layer, head) block."""
    n: int = 0
    cancellation: int = 0
    max_ulp: int = 0
    worst_frob: float = 0.0

    def __add__(self, o: "Stats") -> "Stats":
        return Stats(self.n + o.n, self.cancellation + o.cancellation, max(self.max_ulp, o.max_ulp),
                     max(self.worst_frob, o.worst_frob))

    def line(self, what: str) -> str:
        return (f"{what}: {self.n} elements, {self.cancellation} beyond 1 ulp (cancellation, scale-relative "
                f"pass), max {self.max_ulp} ulp, worst block Frobenius {self.worst_frob:.2e}")


# Lines the GPU parity tests record; tests/conftest.py prints them at the end of
# the session (the count of elements beyond 1 ulp per case).
REPORT = []


def report(what: str, stats) -> None:
    if isinstance(stats, Stats):
        stats = [stats]
    tot = Stats()
    for st in stats:
        tot = tot + st
    REPORT.append(tot.line(what))


def compare(gpu: np.ndarray, ref: np.ndarray, scale: np.ndarray, block_axes=None, what="") -> Stats:
    """Element-wise comparison under the tolerances above; raises AssertionError."""
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    d = np.abs(ordered(gpu) - ordered(ref))
    over = d > 1
    n_over = int(over.sum())
    if n_over:
        g = to_f64(gpu[over])
        r = to_f64(ref[over])
        lim = 2.0 ** -8 * scale[over]
        bad = np.abs(g - r) > lim
        assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1 ulp and the cancellation bound; " \
                              f"first gpu={g[bad][:4]} oracle={r[bad][:4]} scale={scale[over][bad][:4]}"
        assert n_over <= 1e-4 * gpu.size + 2, f"{what}: {n_over} of {gpu.size} elements beyond 1 ulp"
    worst = 0.0
    if block_axes is not None:
        # bf16 -> fp32 is exact, and so is the difference of two bf16 values in
        # fp32 (their exponents differ by far less than 16 here); squares and
        # sums in fp64
        g = to_f32(gpu)
        r = to_f32(ref)
        num = np.sqrt(np.square(g - r, dtype=np.float64).sum(axis=block_axes))
        den = np.sqrt(np.square(r, dtype=np.float64).sum(axis=block_axes))
        rel = np.where(den > 0, num / np.where(den > 0, den, 1), num)
        worst = float(rel.max()) if rel.size else 0.0
        assert worst <= 4e-3, f"{what}: relative Frobenius error {worst:.3g} > 4e-3"
    return Stats(gpu.size, n_over, int(d.max()) if d.size else 0, worst)


# ------------------------------------------------------------- execution
def rope_of(wl: W.Workload) -> K.Rope:
    axes = {}
    if wl.axis_delta is not None:
        axes = dict(freq_axis=wl.freq_axis,
                    axis_delta=torch.as_tensor(wl.axis_delta, dtype=torch.int64, device=wl.pool_k.device))
    off = 0 if wl.kind in ("mla", "mla_ingest") else wl.rot_offset   # the ABI's MLA range is relative to k_rope
    return K.Rope(wl.base, wl.rot_dim, off, wl.pairing, inv_freq=wl.inv_freq, **axes)


def theta_of(wl: W.Workload, orc: O.Oracle) -> np.ndarray:
    """The frequency table both sides use: the workload's own, else base^(-2i/r)."""
    if wl.inv_freq is not None:
        return np.asarray(wl.inv_freq, dtype=np.float64)
    return orc.inv_freq(wl.base, wl.rot_dim)


def max_rank(wl: W.Workload) -> int:
    return max((c.rank for c in wl.chunks), default=0)


# False: relocate calls withhold the host copy of the descriptors, so every
# factor tile moves by per-thread copies instead of tensor-map loads
USE_HOST_COPY = True


def run_gpu(wl: W.Workload, chunks_dev=None, err=None, max_len=None, mrank=None, stream=None):
    """One call of the workload's entry point through the C ABI."""
    if chunks_dev is None:
        chunks_dev = K.pack_chunks(wl.chunks, device=wl.pool_k.device)
    n = len(wl.chunks)
    ml = wl.max_len if max_len is None else max_len
    mr = max_rank(wl) if mrank is None else mrank
    hc = None if USE_HOST_COPY else False
    if wl.kind == "gqa":
        K.kamera_relocate_patch(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, rope_of(wl), chunks_dev, n,
                                ml, mr, err, stream, host_chunks=hc)
    elif wl.kind == "mla":
        K.kamera_mla_relocate_patch(wl.pool_k, wl.store_k, wl.kv_lora, rope_of(wl), chunks_dev, n, ml, mr,
                                    err, stream, host_chunks=hc)
    elif wl.kind == "ingest":
        K.kamera_ingest_canonical(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, rope_of(wl), chunks_dev, n, ml,
                                  err, stream)
    elif wl.kind == "mla_ingest":
        K.kamera_mla_ingest_canonical(wl.pool_k, wl.store_k, wl.kv_lora, rope_of(wl), chunks_dev, n, ml, err,
                                      stream)
    else:
        K.kamera_slide_inplace(wl.pool_k, rope_of(wl), chunks_dev, n, ml, err, stream)
    return chunks_dev


def oracle_chunks(wl: W.Workload):
    out = []
    for c in wl.chunks:
        out.append(O.Chunk(c.src_offset, c.length, c.delta, c.rank,
                           c.slots.detach().cpu().numpy().astype(np.int64),
                           [u16(p) for p in c.patches] if c.rank else []))
    return out


@dataclass
class HostCopy:
    store_k: np.ndarray = None
    store_v: np.ndarray = None
    pool_k: np.ndarray = None
    pool_v: np.ndarray = None
    chunks: list = None


def snapshot(wl: W.Workload) -> HostCopy:
    """Host copies of every input, taken before the GPU call."""
    h = HostCopy()
    h.store_k = u16(wl.store_k) if wl.store_k is not None else None
    h.store_v = u16(wl.store_v) if wl.store_v is not None else None
    h.pool_k = u16(wl.pool_k)
    h.pool_v = u16(wl.pool_v) if wl.pool_v is not None else None
    h.chunks = oracle_chunks(wl)
    return h


def axis_tables(wl: W.Workload, th: np.ndarray):
    """Multi-axis RoPE, chunk by chunk: frequency f of chunk c turns by the
    chunk's move along f's axis, which is R(1) over the table
    theta'_f = move_c[axis_f] * theta_f (the same fp64 products, so the same
    phases).  Returns (per-chunk tables, the delta each chunk then takes: 1,
    or 0 for a chunk that does not move)."""
    moves = np.asarray(wl.axis_delta, dtype=np.int64)
    axis = np.asarray(wl.freq_axis, dtype=np.int64)
    tabs = [moves[c][axis].astype(np.float64) * th for c in range(len(moves))]
    return tabs, [1 if np.any(moves[c] != 0) else 0 for c in range(len(moves))]


def run_oracle(wl: W.Workload, h: HostCopy, orc: O.Oracle = None):
    """Oracle result on host copies: returns (pool_k, pool_v, scale_k, scale_v)."""
    orc = orc or O.default()
    if wl.axis_delta is not None:   # per-chunk tables: one oracle call per chunk, results merged
        tabs, deltas = axis_tables(wl, theta_of(wl, orc))
        acc = None
        for c, (tab, de) in enumerate(zip(tabs, deltas)):
            one = copy.copy(wl)
            one.axis_delta, one.freq_axis, one.inv_freq = None, None, tab
            hc = copy.copy(h)
            ch = h.chunks[c]
            hc.chunks = [O.Chunk(ch.src_offset, ch.length, de, ch.rank, ch.slots, ch.patches)]
            if acc is not None:   # chunks write disjoint rows: chain the arrays through the calls
                if wl.kind in ("ingest", "mla_ingest"):
                    hc.store_k, hc.store_v = acc[0], acc[1]
                else:
                    hc.pool_k, hc.pool_v = acc[0], acc[1]
            r = run_oracle(one, hc, orc)
            acc = r if acc is None else (r[0], r[1], acc[2] + r[2], None if r[3] is None else acc[3] + r[3])
        return acc
    pk = h.pool_k.copy()
    pv = h.pool_v.copy() if h.pool_v is not None else None
    if wl.kind == "gqa":
        th = theta_of(wl, orc)
        sk, sv = orc.gqa(h.store_k, h.store_v, pk, pv, h.chunks, th, wl.rot_dim, wl.rot_offset, wl.pairing,
                         want_scale=True)
        return pk, pv, sk, sv
    if wl.kind == "mla":
        th = theta_of(wl, orc)
        sk = orc.mla(h.store_k, pk, h.chunks, wl.kv_lora, th, wl.pairing, want_scale=True)
        return pk, None, sk, None
    if wl.kind in ("ingest", "mla_ingest"):   # returns the store arrays instead of the pool's
        th = theta_of(wl, orc)
        st_k = h.store_k.copy()
        st_v = h.store_v.copy() if h.store_v is not None else None
        if wl.kind == "ingest":
            sk = orc.ingest(h.pool_k, h.pool_v, st_k, st_v, h.chunks, th, wl.rot_dim, wl.rot_offset, wl.pairing,
                            want_scale=True)
        else:
            L, S, Wd = h.pool_k.shape
            sk = orc.ingest(h.pool_k.reshape(L, S, 1, Wd), None, st_k.reshape(L, -1, 1, Wd), None, h.chunks, th,
                            wl.rot_dim, wl.rot_offset, wl.pairing, want_scale=True)
            sk = sk.reshape(st_k.shape)
        return st_k, st_v, sk, None
    th = theta_of(wl, orc)
    sk = orc.slide(pk, h.chunks, th, wl.rot_dim, wl.rot_offset, wl.pairing, want_scale=True)
    return pk, None, sk, None


def touched_slots(wl: W.Workload) -> np.ndarray:
    if not wl.chunks:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([c.slots.detach().cpu().numpy() for c in wl.chunks]).astype(np.int64)


def written_rows(wl: W.Workload) -> np.ndarray:
    """Store rows an ingest call writes."""
    return np.concatenate([np.arange(c.src_offset, c.src_offset + c.length) for c in wl.chunks]
                          or [np.zeros(0, np.int64)]).astype(np.int64)


def check_ingest_parity(wl: W.Workload, h: HostCopy, what: str):
    torch.cuda.synchronize()
    ok, ov, sk, _ = run_oracle(wl, h)
    gk = u16(wl.store_k)
    rows = np.zeros(gk.shape[1], dtype=bool)
    rows[written_rows(wl)] = True
    assert np.array_equal(gk[:, ~rows], h.store_k[:, ~rows]), f"{what}: unwritten store rows changed"
    assert np.array_equal(u16(wl.pool_k), h.pool_k), f"{what}: the pool changed"
    stats = []
    if wl.kind == "mla_ingest":
        kv = wl.kv_lora
        g, r, s = gk[:, rows], ok[:, rows], sk[:, rows]
        assert np.array_equal(g[..., :kv], r[..., :kv]), f"{what}: c_KV not a bit copy"
        stats.append(compare(g[..., kv:], r[..., kv:], s[..., kv:], block_axes=(1, 2), what=what + " k_rope"))
        return stats
    stats.append(compare(gk[:, rows], ok[:, rows], sk[:, rows], block_axes=(1, 3), what=what + " K"))
    gv = u16(wl.store_v)
    assert np.array_equal(gv, ov), f"{what}: values not a bit copy (or unwritten rows changed)"
    assert np.array_equal(u16(wl.pool_v), h.pool_v), f"{what}: the value pool changed"
    if all(c.delta == 0 for c in wl.chunks):
        assert np.array_equal(gk, ok), f"{what}: delta 0 is not a bit copy"
    return stats


def check_parity(wl: W.Workload, h: HostCopy, what: str):
    """Full comparison of the GPU pool (or, for ingest, the store) against the oracle."""
    if wl.kind in ("ingest", "mla_ingest"):
        return check_ingest_parity(wl, h, what)
    torch.cuda.synchronize()
    ok, ov, sk, sv = run_oracle(wl, h)
    gk = u16(wl.pool_k)
    touched = np.zeros(gk.shape[1], dtype=bool)
    touched[touched_slots(wl)] = True
    # untouched slots keep their bytes exactly (canary)
    assert np.array_equal(gk[:, ~touched], h.pool_k[:, ~touched]), f"{what}: untouched K slots changed"
    stats = []
    if wl.kind == "mla":
        kv = wl.kv_lora
        g = gk[:, touched]
        r = ok[:, touched]
        s = sk[:, touched]
        stats.append(compare(g[..., :kv], r[..., :kv], s[..., :kv], block_axes=(1, 2), what=what + " c_KV"))
        stats.append(compare(g[..., kv:], r[..., kv:], s[..., kv:], block_axes=(1, 2), what=what + " k_rope"))
        if all(c.rank == 0 for c in wl.chunks):
            assert np.array_equal(g[..., :kv], r[..., :kv]), f"{what}: c_KV not a bit copy"
        return stats
    stats.append(compare(gk[:, touched], ok[:, touched], sk[:, touched], block_axes=(1, 3), what=what + " K"))
    if wl.kind == "gqa":
        gv = u16(wl.pool_v)
        assert np.array_equal(gv[:, ~touched], h.pool_v[:, ~touched]), f"{what}: untouched V slots changed"
        stats.append(compare(gv[:, touched], ov[:, touched], sv[:, touched], block_axes=(1, 3), what=what + " V"))
    return stats


# ------------------------------------------------ whole outputs, layer by layer
def _layer_chunks(wl: W.Workload, l: int, slots):
    """The chunks with their factors cut to layer l (host copies)."""
    out = []
    for c, s in zip(wl.chunks, slots):
        out.append(O.Chunk(c.src_offset, c.length, c.delta, c.rank, s,
                           [u16(p[l:l + 1]) for p in c.patches] if c.rank else []))
    return out


def check_layers(wl: W.Workload, layers, what: str, pool_before: torch.Tensor = None, workers: int = 8):
    """Every output row of the given layers against the oracle, after one GPU
    call over the whole workload (the launch under test).  Layer by layer: the
    layer's store rows, factors and pool are copied to the host, the oracle
    computes the layer (the pools start as canary, or as ``pool_before`` for
    the in-place slide), and every targeted slot is compared element by
    element, with the Frobenius bound per (layer, head) block, while every
    other slot must keep its bytes.  Comparisons run in worker threads while
    the oracle computes the next layer.  Returns the summed Stats per array."""
    from concurrent.futures import ThreadPoolExecutor
    if wl.pool_k.is_cuda:
        torch.cuda.synchronize()
    orc = O.default()
    th = theta_of(wl, orc)
    slots = [c.slots.detach().cpu().numpy().astype(np.int64) for c in wl.chunks]
    S = wl.pool_k.shape[1]
    touched = np.zeros(S, dtype=bool)
    if slots:
        touched[np.concatenate(slots)] = True
    canary = np.uint16(W.CANARY_BITS)

    def cmp(tag, l, got, want, scale, before, axes, split=None):
        assert np.array_equal(got[:, ~touched], before[:, ~touched]), f"{what} {tag} layer {l}: untouched slots changed"
        g, r, s = got[:, touched], want[:, touched], scale[:, touched]
        if split is None:
            return {tag: compare(g, r, s, block_axes=axes, what=f"{what} {tag} layer {l}")}
        return {f"{tag} c_KV": compare(g[..., :split], r[..., :split], s[..., :split], block_axes=axes,
                                       what=f"{what} c_KV layer {l}"),
                f"{tag} k_rope": compare(g[..., split:], r[..., split:], s[..., split:], block_axes=axes,
                                         what=f"{what} k_rope layer {l}")}

    totals = {}
    pending = []

    def collect(block):
        while len(pending) > block:
            for k, st in pending.pop(0).result().items():
                totals[k] = totals.get(k, Stats()) + st

    with ThreadPoolExecutor(max_workers=workers) as ex:
        for l in layers:
            ch = _layer_chunks(wl, l, slots)
            if wl.kind == "gqa":
                pk = np.full((1,) + tuple(wl.pool_k.shape[1:]), canary, dtype=np.uint16)
                pv = pk.copy()
                sk, sv = orc.gqa(u16(wl.store_k[l:l + 1]), u16(wl.store_v[l:l + 1]), pk, pv, ch, th, wl.rot_dim,
                                 wl.rot_offset, wl.pairing, want_scale=True)
                canaries = np.full_like(pk, canary)
                pending.append(ex.submit(cmp, "K", l, u16(wl.pool_k[l:l + 1]), pk, sk, canaries, (1, 3)))
                pending.append(ex.submit(cmp, "V", l, u16(wl.pool_v[l:l + 1]), pv, sv, canaries, (1, 3)))
            elif wl.kind == "mla":
                pk = np.full((1,) + tuple(wl.pool_k.shape[1:]), canary, dtype=np.uint16)
                sk = orc.mla(u16(wl.store_k[l:l + 1]), pk, ch, wl.kv_lora, th, wl.pairing, want_scale=True)
                pending.append(ex.submit(cmp, "row", l, u16(wl.pool_k[l:l + 1]), pk, sk, np.full_like(pk, canary),
                                         (1, 2), wl.kv_lora))
            elif wl.kind == "slide":
                before = u16(pool_before[l:l + 1])
                pk = before.copy()
                sk = orc.slide(pk, ch, th, wl.rot_dim, wl.rot_offset, wl.pairing, want_scale=True)
                pending.append(ex.submit(cmp, "K", l, u16(wl.pool_k[l:l + 1]), pk, sk, before, (1, 3)))
            else:
                raise ValueError(f"check_layers: {wl.kind} not handled")
            collect(workers)
        collect(0)
    return totals
