"""Seeded synthetic workloads for the Kamera relocate + patch + scatter operator.

This module only draws inputs: canonical K/V stores, patch factors, chunk
lengths, phase shifts, page permutations and canary-filled pools.  It holds
none of the operator's arithmetic, and both sides use it: the CUDA path (the
tensors go to the GPU through the C-ABI binding) and the fp64 oracle (the same
tensors, copied to host memory).

The shapes follow the workloads named for the method ("Kamera: Unified
Position-Invariant Multimodal KV Cache for Training-Free Reuse"): Qwen2.5-VL-7B
shaped GQA caches with image-sized chunks, a DeepSeek-V2-Lite shaped MLA cache,
sliding-window survival and an MHA reorder + recall batch.  The pages' own
benchmarks (MM-NIAH, MileBench, two-page doc-QA) measure accuracy with trained
weights; these synthetic inputs stand in for them as shapes only.

Recipe (the pages give none; readings):
  * K/V ~ N(0, 1) drawn in fp32, rounded to bf16; config "qwen_recall" scales
    each (layer, head, dim) channel by exp(U(ln 0.1, ln 10)), K and V independently.
  * patch factors U, V_m ~ N(0, 0.05^2) (std 0.05), bf16.
  * pools are paged (P tokens per page); a chunk's tokens fill pages in order and
    the pages are a random permutation of the pool's pages; unused slots hold a
    canary bit pattern.
  * tensors are drawn with torch.Generator seeded from (SEED, workload, tensor);
    lengths, deltas and page permutations with numpy PCG64 SeedSequence([SEED, ...]).
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

SEED = 20260623
CANARY_BITS = 0x5A5A  # bf16 pattern left in slots that no chunk targets

ROTATE_HALF = 0
INTERLEAVED = 1


# ---------------------------------------------------------------- specs ----
@dataclass(frozen=True)
class GqaSpec:
    """GQA/MHA relocate + patch (kind 'gqa'), rotate-only slide (kind 'slide') or
    canonical ingest (kind 'ingest': the chunks sit in the pool at live positions,
    delta = minus each chunk's start, and are written to the store)."""
    name: str
    kind: str                      # "gqa" | "slide" | "ingest"
    L: int
    H: int
    d: int
    base: float
    lens: Sequence[int]
    deltas: Sequence[int]
    m: int
    page: int
    pairing: int = ROTATE_HALF
    rot_dim: Optional[int] = None  # default: whole head (d)
    rot_offset: int = 0
    channel_scale: bool = False
    pool_pages: Optional[int] = None
    window: int = 0                # slide: tokens held in the window (pool)
    evicted: int = 0               # slide: oldest tokens evicted


@dataclass(frozen=True)
class MlaSpec:
    name: str
    L: int
    kv_lora: int
    rope: int
    base: float
    lens: Sequence[int]
    deltas: Sequence[int]
    m: int
    page: int
    pairing: int = INTERLEAVED
    pool_pages: Optional[int] = None

    kind: str = "mla"             # "mla" | "mla_ingest"


def _np_rng(*tags) -> np.random.Generator:
    key = [SEED] + [zlib.crc32(str(t).encode()) for t in tags]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def _torch_seed(*tags) -> int:
    return int(_np_rng("torch", *tags).integers(0, 2**62))


# ------------------------------------------------------------ the configs --
def tiny_gqa() -> GqaSpec:
    """1 layer, 2 KV heads, d=64, one 128-token chunk, delta=+37, rank 4, base 1e4, P=16."""
    return GqaSpec("tiny_gqa", "gqa", L=1, H=2, d=64, base=1e4, lens=(128,), deltas=(37,),
                   m=4, page=16, pool_pages=16)


def qwen_recall() -> GqaSpec:
    """Qwen2.5-VL-7B shaped recall batch: 28 L, 4 KV heads, d=128, base 1e6,
    8 chunks of 1296 tokens, delta ~ U{-32768..32768}, rank 32, P=16."""
    r = _np_rng("qwen_recall", "delta")
    deltas = tuple(int(x) for x in r.integers(-32768, 32769, size=8))
    return GqaSpec("qwen_recall", "gqa", L=28, H=4, d=128, base=1e6, lens=(1296,) * 8,
                   deltas=deltas, m=32, page=16, channel_scale=True)


def dsv2_mla() -> MlaSpec:
    """DeepSeek-V2-Lite shaped MLA: 27 L, c_KV 512 + k_rope 64, base 1e4 on k_rope,
    16 chunks of 4096 tokens, delta ~ U{-16384..16384}, rank 16 on both channels, P=64."""
    r = _np_rng("dsv2_mla", "delta")
    deltas = tuple(int(x) for x in r.integers(-16384, 16385, size=16))
    return MlaSpec("dsv2_mla", L=27, kv_lora=512, rope=64, base=1e4, lens=(4096,) * 16,
                   deltas=deltas, m=16, page=64)


def qwen_slide() -> GqaSpec:
    """Sliding-window survival: 131072-token window of a Qwen2.5-VL-7B shaped cache;
    the oldest 32768 are evicted and the 98304 survivors (75 x 1296 + 1104) turn by -32768."""
    survivors = 131072 - 32768
    lens = [1296] * (survivors // 1296)
    if survivors % 1296:
        lens.append(survivors % 1296)
    return GqaSpec("qwen_slide", "slide", L=28, H=4, d=128, base=1e6, lens=tuple(lens),
                   deltas=(-32768,) * len(lens), m=0, page=16, window=131072, evicted=32768)


def mha_reorder_recall() -> GqaSpec:
    """MHA reorder + recall: 32 L, 32 heads, d=128, base 1e4, 64 chunks of U{256..2048}
    tokens permuted (delta = new start - old start) plus 8 recall chunks placed after them
    (canonical at position 0, delta = target start), rank 64 on K and V, P=16."""
    r = _np_rng("mha_reorder_recall", "lens")
    lens = [int(x) for x in r.integers(256, 2049, size=64)]
    rec = [int(x) for x in r.integers(256, 2049, size=8)]
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    perm = _np_rng("mha_reorder_recall", "perm").permutation(64)
    new_starts = np.empty(64, dtype=np.int64)
    pos = 0
    for c in perm:                       # chunk c now sits at position pos
        new_starts[c] = pos
        pos += lens[c]
    deltas = [int(new_starts[c] - starts[c]) for c in range(64)]
    for t in rec:                        # recalled chunks follow the reordered set
        deltas.append(int(pos))
        pos += t
    return GqaSpec("mha_reorder_recall", "gqa", L=32, H=32, d=128, base=1e4,
                   lens=tuple(lens + rec), deltas=tuple(deltas), m=64, page=16)


def qwen_ingest() -> GqaSpec:
    """Canonical ingest of a Qwen2.5-VL-7B shaped recall batch's chunks from a live
    cache: 28 L, 4 KV heads, d=128, base 1e6, 8 chunks of 1296 tokens whose first
    tokens sit at positions s ~ U{0..32767} (delta = -s), P=16."""
    r = _np_rng("qwen_ingest", "start")
    deltas = tuple(-int(x) for x in r.integers(0, 32768, size=8))
    return GqaSpec("qwen_ingest", "ingest", L=28, H=4, d=128, base=1e6, lens=(1296,) * 8,
                   deltas=deltas, m=0, page=16)


def dsv2_mla_ingest() -> MlaSpec:
    """Canonical ingest on the DeepSeek-V2-Lite shaped MLA cache: 27 L, c_KV 512
    (copied) + k_rope 64 (interleaved, base 1e4, turned), 16 chunks of 4096 tokens
    starting at s ~ U{0..16383} (delta = -s), P=64."""
    r = _np_rng("dsv2_mla_ingest", "start")
    deltas = tuple(-int(x) for x in r.integers(0, 16384, size=16))
    return MlaSpec("dsv2_mla_ingest", L=27, kv_lora=512, rope=64, base=1e4, lens=(4096,) * 16,
                   deltas=deltas, m=0, page=64, kind="mla_ingest")


def tiny_gqa_x(n: int = 4096) -> GqaSpec:
    """The tiny GQA chunk replicated n times in one call (n chunks of 128 tokens)."""
    r = _np_rng("tiny_gqa_x", n)
    deltas = tuple(int(x) for x in r.integers(-32768, 32769, size=n))
    return GqaSpec(f"tiny_gqa_x{n}", "gqa", L=1, H=2, d=64, base=1e4, lens=(128,) * n,
                   deltas=deltas, m=4, page=16, pool_pages=2 * 8 * n)


CONFIGS = {
    "tiny_gqa": tiny_gqa,
    "qwen_recall": qwen_recall,
    "dsv2_mla": dsv2_mla,
    "qwen_slide": qwen_slide,
    "mha_reorder_recall": mha_reorder_recall,
    "qwen_ingest": qwen_ingest,
    "dsv2_mla_ingest": dsv2_mla_ingest,
}


def scaled(spec, L: Optional[int] = None, lens: Optional[Sequence[int]] = None,
           H: Optional[int] = None, m: Optional[int] = None, name: Optional[str] = None):
    """A smaller copy of a spec (fewer layers / tokens / heads) with the same structure."""
    kw = dict(spec.__dict__)
    if L is not None:
        kw["L"] = L
    if H is not None:
        kw["H"] = H
    if m is not None:
        kw["m"] = m
    if lens is not None:
        n = len(lens)
        kw["lens"] = tuple(lens)
        kw["deltas"] = tuple(spec.deltas[i % len(spec.deltas)] for i in range(n))
        kw["pool_pages"] = None
        if spec.kind == "slide":
            kw["evicted"] = sum(lens) // 3
            kw["window"] = sum(lens) + kw["evicted"]
    kw["name"] = name or (spec.name + "_small")
    return type(spec)(**kw)


# ----------------------------------------------------- frequency tables --
def mrope_sections(n_freq: int):
    """Frequency index ranges of a three-axis (time, height, width) rotary
    layout: a quarter of the frequencies follow time, the rest split evenly
    between height and width (16/24/24 of the 64 frequencies of a 128-wide
    head, the split of Qwen2.5-VL's multimodal RoPE)."""
    t = n_freq // 4
    hgt = (n_freq - t) // 2
    return [(0, t), (t, t + hgt), (t + hgt, n_freq)]


def freq_axes(n_freq: int, layout: str = "sections") -> np.ndarray:
    """The axis (0 time, 1 height, 2 width) each frequency follows:
    'sections'     contiguous ranges (``mrope_sections``)
    'interleaved'  frequency f follows axis f mod 3 (an interleaved layout)"""
    out = np.empty(n_freq, dtype=np.uint8)
    if layout == "sections":
        for a, (lo, hi) in enumerate(mrope_sections(n_freq)):
            out[lo:hi] = a
    else:
        out[:] = np.arange(n_freq) % 3
    return out


def axis_moves(n_chunks: int, *tags) -> np.ndarray:
    """Seeded per-chunk (time, height, width) moves, int64 [n_chunks, 3],
    cycling through the kinds a multimodal prompt produces: a text or whole-
    segment move (d, d, d), a move along time only (d, 0, 0), independent
    axis moves, and no move (0, 0, 0)."""
    rng = _np_rng("axis_moves", n_chunks, *tags)
    out = np.zeros((n_chunks, 3), dtype=np.int64)
    for c in range(n_chunks):
        d = int(rng.integers(-5000, 30000))
        kind = c % 4
        if kind == 0:
            out[c] = (d, d, d)
        elif kind == 1:
            out[c] = (d, 0, 0)
        elif kind == 2:
            out[c] = rng.integers(-2000, 2000, size=3)
    return out


def model_inv_freq(kind: str, base: float, rot_dim: int) -> np.ndarray:
    """A model's own rotary frequency table, passed to the operator as an input.

    'standard'  base^(-2i/r)
    'extended'  a context-extension rescale of the standard table by s = 8:
                wavelengths longer than the 4096-token original context are
                interpolated (theta/s), those shorter than 1/32 of it keep
                theta, a linear ramp in between
    'temporal'  multi-axis RoPE moved along time only: the height and width
                sections' frequencies are 0, so R(delta) turns the time section
                and leaves the spatial ones as they are
    'axes'      multi-axis RoPE moved by (delta, delta/2, delta/4) along (time,
                height, width): each section's frequencies scaled by its axis's
                share of delta"""
    n = rot_dim // 2
    th = base ** (-2.0 * np.arange(n, dtype=np.float64) / rot_dim)
    if kind == "standard":
        return th
    if kind == "extended":
        s, ctx, lo, hi = 8.0, 4096.0, 1.0, 32.0
        wavelengths = 2.0 * math.pi / th
        ramp = np.clip((ctx / wavelengths - lo) / (hi - lo), 0.0, 1.0)   # 0: interpolate, 1: keep
        return th * (ramp + (1.0 - ramp) / s)
    sec = mrope_sections(n)
    if kind == "temporal":
        share = (1.0, 0.0, 0.0)
    elif kind == "axes":
        share = (1.0, 0.5, 0.25)
    else:
        raise ValueError(kind)
    out = th.copy()
    for (a, b), w in zip(sec, share):
        out[a:b] *= w
    return out


# -------------------------------------------------------------- deficits --
@dataclass(frozen=True)
class DeficitSpec:
    """Deficits Delta = KV(B|A) - KV(B|empty) of one chunk's keys and values for
    patch formation, synthetic: each (kv, layer, head) block is a planted
    low-rank matrix (``planted`` orthonormal directions on both sides with
    singular values geometric from s_max to s_min: the deficit's energy sits in
    about 32 feature directions) plus i.i.d. N(0, noise^2) entries; bf16
    ``[kv, L, len, H, d]`` (kv = 2: keys and values), rank-m factors asked for."""
    name: str
    L: int
    length: int
    H: int
    d: int
    m: int = 32
    kv: int = 2
    planted: int = 32
    s_max: float = 1.0
    s_min: float = 0.05
    noise: float = 1e-4
    terms: int = 1          # > 1: that many deficits per block, factored as their mean (orbit patch)
    kind: str = "patch_form"


def qwen_patch_form() -> DeficitSpec:
    """Rank-32 patch formation for one Qwen2.5-VL-7B shaped 1296-token frame chunk:
    keys and values of 28 layers x 4 KV heads, d = 128 (224 blocks)."""
    return DeficitSpec("qwen_patch_form", L=28, length=1296, H=4, d=128, m=32)


def make_deficit(spec: DeficitSpec, device="cpu") -> torch.Tensor:
    """Materialise a DeficitSpec (seeded): bf16 [terms, kv, L, len, H, d], or
    [kv, L, len, H, d] when terms == 1."""
    rng = _np_rng("deficit", spec.name, spec.L, spec.length, spec.H, spec.d, spec.terms)
    T, n = spec.terms, spec.kv * spec.L * spec.H
    k = min(spec.planted, spec.length, spec.d)
    s = np.geomspace(spec.s_max, spec.s_min, k) if k > 1 else np.array([spec.s_max])
    out = np.empty((T, spec.kv, spec.L, spec.H, spec.length, spec.d), dtype=np.float32)
    flat = out.reshape(T, n, spec.length, spec.d)
    for t in range(T):
        for b in range(n):
            a, _ = np.linalg.qr(rng.standard_normal((spec.length, k)))
            z, _ = np.linalg.qr(rng.standard_normal((spec.d, k)))
            flat[t, b] = (a * s) @ z.T + spec.noise * rng.standard_normal((spec.length, spec.d))
    x = torch.from_numpy(out).to(torch.bfloat16).permute(0, 1, 2, 4, 3, 5).contiguous()
    x = x.to(device)
    return x[0] if T == 1 else x


def dsv2_patch_form() -> DeficitSpec:
    """Rank-16 patch formation for one DeepSeek-V2-Lite shaped 4096-token chunk's
    c_KV deficits: 27 layers, one 4096 x 512 block each (the wide-block path)."""
    return DeficitSpec("dsv2_patch_form", L=27, length=4096, H=1, d=512, m=16, kv=1)


def dsv2_joint_patch_form() -> DeficitSpec:
    """Rank-16 patch formation for the same chunk with one joint factor over the
    whole 576-wide latent row (c_KV 512 | k_rope 64): 27 blocks of 4096 x 576."""
    return DeficitSpec("dsv2_joint_patch_form", L=27, length=4096, H=1, d=576, m=16, kv=1)


FORMATION = {"qwen_patch_form": qwen_patch_form, "dsv2_patch_form": dsv2_patch_form,
             "dsv2_joint_patch_form": dsv2_joint_patch_form}


# ------------------------------------------------------ attention inputs --
@dataclass(frozen=True)
class AttendSpec:
    """Decode attention over reused chunks: ``seqs`` lists each sequence's chunk
    lengths; every chunk has its own canonical rows in one layer's store
    (K, V ~ N(0, 1)), a delta drawn from U{-dmax..dmax} and, when m > 0, factors
    ~ N(0, 0.1^2) for ``L`` layers (read at ``layer``); one query token per
    sequence and query head, N(0, 1)."""
    name: str
    H: int
    G: int
    d: int
    seqs: tuple
    m: int = 32
    L: int = 2
    layer: int = 1
    base: float = 1e6
    rot_dim: int = -1          # -1: the whole head
    rot_offset: int = 0
    pairing: int = ROTATE_HALF
    dmax: int = 32768
    zero_rank_every: int = 0   # > 0: every n-th chunk carries no patch
    kind: str = "attend"
    T: int = 0                 # > 0: prefill, T query tokens per sequence (q [S, T, H * G, d])


@dataclass
class AttendData:
    spec: AttendSpec
    store_k: torch.Tensor      # [N, H, d]
    store_v: torch.Tensor
    chunks: List["ChunkData"]
    seq_start: List[int]
    q: torch.Tensor            # [S, H * G, d]

    @property
    def rot_dim(self) -> int:
        return self.spec.d if self.spec.rot_dim < 0 else self.spec.rot_dim


def qwen_attend_reused() -> AttendSpec:
    """A decode step over reused chunks, Qwen2.5-VL-7B shaped (4 KV heads, 28 query
    heads, d = 128, base 1e6): 38 sequences, each the 8-chunk recall batch
    (8 x 1296 tokens), rank 32 on K and V -- one CTA per (sequence, KV head),
    152 in all."""
    return AttendSpec("qwen_attend_reused", H=4, G=7, d=128, seqs=tuple((1296,) * 8 for _ in range(38)), m=32)


def make_attend(spec: AttendSpec, device="cpu") -> AttendData:
    rng = _np_rng("attend", spec.name, spec.H, spec.G, spec.d)
    lens = [t for seq in spec.seqs for t in seq]
    N = max(1, sum(lens))
    gen = _gen(device, "attend", spec.name)
    store_k = _randn_bf16((N, spec.H, spec.d), 1.0, gen, device)
    store_v = _randn_bf16((N, spec.H, spec.d), 1.0, gen, device)
    chunks, seq_start, off, idx = [], [0], 0, 0
    for seq in spec.seqs:
        for t in seq:
            m = 0 if (spec.zero_rank_every and idx % spec.zero_rank_every == spec.zero_rank_every - 1) else spec.m
            pat = []
            if m > 0 and t > 0:
                pat = [_randn_bf16((spec.L, spec.H, t, m), 0.1, gen, device),
                       _randn_bf16((spec.L, spec.H, spec.d, m), 0.1, gen, device),
                       _randn_bf16((spec.L, spec.H, t, m), 0.1, gen, device),
                       _randn_bf16((spec.L, spec.H, spec.d, m), 0.1, gen, device)]
            else:
                m = 0
            delta = int(rng.integers(-spec.dmax, spec.dmax + 1))
            slots = torch.arange(max(t, 1), dtype=torch.int64, device=device)[:t]
            chunks.append(ChunkData(off, t, delta, m, slots, pat))
            off += t
            idx += 1
        seq_start.append(len(chunks))
    qshape = (len(spec.seqs),) + ((spec.T,) if spec.T > 0 else ()) + (spec.H * spec.G, spec.d)
    q = _randn_bf16(qshape, 1.0, gen, device)
    return AttendData(spec, store_k, store_v, chunks, seq_start, q)


def qwen_prefill_reused() -> AttendSpec:
    """A prefill over reused chunks, Qwen2.5-VL-7B shaped (4 KV heads, 28 query
    heads, d = 128, base 1e6): 38 sequences, each recalling the 8-chunk batch
    (8 x 1296 tokens, rank 32 on K and V) and bringing 256 new query tokens
    that attend over it -- 256 x 7 = 1792 query rows per (sequence, KV head),
    14 CTAs of 128 rows each."""
    return AttendSpec("qwen_prefill_reused", H=4, G=7, d=128, seqs=tuple((1296,) * 8 for _ in range(38)), m=32,
                      kind="prefill", T=256)


def prefill_flops(spec: AttendSpec) -> int:
    """Floating-point operations of prefill attention in the folded form (the
    rows are never formed): per query row and token, 2 (d + m) for the score
    (q'.k + x.u) and 2 (d + m) for the weighted sums (p v and p u'); per query
    row and patched chunk, 2 d m for V_k^T q and 2 d m for the V_v fold."""
    rows = spec.T * spec.H * spec.G * len(spec.seqs)
    per_seq_tok = [sum(seq) for seq in spec.seqs]
    per_seq_ch = [sum(1 for t in seq if t > 0) for seq in spec.seqs]
    rows_per_seq = spec.T * spec.H * spec.G
    tok = sum(rows_per_seq * t for t in per_seq_tok)
    ch = sum(rows_per_seq * c for c in per_seq_ch)
    assert rows == rows_per_seq * len(spec.seqs)
    return 4 * tok * (spec.d + spec.m) + 4 * ch * spec.d * spec.m


def attend_bytes(spec: AttendSpec) -> int:
    """Bytes a decode step must move: each token's canonical K and V rows of each
    KV head, its U rows (2m per head), each patched chunk's V factors (2 d m per
    head), the queries read and the outputs written."""
    B = 2
    tok = sum(t for seq in spec.seqs for t in seq)
    nch = sum(1 for seq in spec.seqs for t in seq if t > 0)
    q = len(spec.seqs) * spec.H * spec.G * spec.d * B
    return tok * spec.H * (2 * spec.d + 2 * spec.m) * B + nch * spec.H * 2 * spec.d * spec.m * B + 2 * q


@dataclass
class MlaAttendSpec:
    """MLA decode attention over reused chunks (absorbed form): ``seqs`` lists
    each sequence's chunk lengths; every chunk has its own canonical rows
    (c_KV | k_rope ~ N(0, 1)) in one layer's store, a delta drawn from
    U{-dmax..dmax} and, when m > 0, factors Uc, Vc, Ur, Vr ~ N(0, 0.1^2) for ``L``
    layers (read at ``layer``); one query token per sequence and query head
    (latent part | rope part ~ N(0, 1)).  DeepSeek's plain RoPE pairs
    interleaved components."""
    name: str
    Hq: int
    seqs: tuple
    m: int = 16
    kv_lora: int = 512
    rope: int = 64
    L: int = 2
    layer: int = 1
    base: float = 1e4
    rot_dim: int = -1          # -1: all of k_rope
    rot_offset: int = 0
    pairing: int = INTERLEAVED
    dmax: int = 16384
    zero_rank_every: int = 0   # > 0: every n-th chunk carries no patch
    kind: str = "mla_attend"


@dataclass
class MlaAttendData:
    spec: MlaAttendSpec
    store: torch.Tensor        # [N, kv_lora + rope]
    chunks: List["ChunkData"]
    seq_start: List[int]
    q: torch.Tensor            # [S, Hq, kv_lora + rope]

    @property
    def rot_dim(self) -> int:
        return self.spec.rope if self.spec.rot_dim < 0 else self.spec.rot_dim


def make_mla_attend(spec: MlaAttendSpec, device="cpu") -> MlaAttendData:
    rng = _np_rng("mla_attend", spec.name, spec.Hq)
    lens = [t for seq in spec.seqs for t in seq]
    W = spec.kv_lora + spec.rope
    gen = _gen(device, "mla_attend", spec.name)
    store = _randn_bf16((max(1, sum(lens)), W), 1.0, gen, device)
    chunks, seq_start, off, idx = [], [0], 0, 0
    for seq in spec.seqs:
        for t in seq:
            m = 0 if (spec.zero_rank_every and idx % spec.zero_rank_every == spec.zero_rank_every - 1) else spec.m
            pat = []
            if m > 0 and t > 0:
                pat = [_randn_bf16((spec.L, t, m), 0.1, gen, device),
                       _randn_bf16((spec.L, spec.kv_lora, m), 0.1, gen, device),
                       _randn_bf16((spec.L, t, m), 0.1, gen, device),
                       _randn_bf16((spec.L, spec.rope, m), 0.1, gen, device)]
            else:
                m = 0
            delta = int(rng.integers(-spec.dmax, spec.dmax + 1))
            slots = torch.arange(max(t, 1), dtype=torch.int64, device=device)[:t]
            chunks.append(ChunkData(off, t, delta, m, slots, pat))
            off += t
            idx += 1
        seq_start.append(len(chunks))
    q = _randn_bf16((len(spec.seqs), spec.Hq, W), 1.0, gen, device)
    return MlaAttendData(spec, store, chunks, seq_start, q)


def dsv2_attend_reused() -> MlaAttendSpec:
    """A decode step over reused chunks, DeepSeek-V2-Lite shaped (16 query heads on
    one 512 + 64 latent row, base 1e4): 38 sequences, each four of the MLA
    workload's 4096-token chunks, rank 16 on both channels."""
    return MlaAttendSpec("dsv2_attend_reused", Hq=16, seqs=tuple((4096,) * 4 for _ in range(38)), m=16)


def mla_attend_bytes(spec: MlaAttendSpec) -> int:
    """Bytes an MLA decode step must move: each token's canonical row and its two
    U rows (2m), each patched chunk's V factors ((kv_lora + rope) m), the queries
    read and the latent outputs written."""
    B = 2
    W = spec.kv_lora + spec.rope
    tok = sum(t for seq in spec.seqs for t in seq)
    nch = sum(1 for seq in spec.seqs for t in seq if t > 0)
    S = len(spec.seqs)
    return (tok * (W + 2 * spec.m) + nch * W * spec.m + S * spec.Hq * (W + spec.kv_lora)) * B


ATTENTION = {"qwen_attend_reused": qwen_attend_reused, "dsv2_attend_reused": dsv2_attend_reused,
             "qwen_prefill_reused": qwen_prefill_reused}


# ------------------------------------------------------------- workloads --
@dataclass
class ChunkData:
    src_offset: int
    length: int
    delta: int
    rank: int
    slots: torch.Tensor                       # int64 [length]
    patches: List[torch.Tensor] = field(default_factory=list)   # 4 bf16 tensors or empty


@dataclass
class Workload:
    spec: object
    kind: str
    chunks: List[ChunkData]
    store_k: Optional[torch.Tensor] = None    # gqa: [L, N, H, d]; mla: store [L, N, W]
    store_v: Optional[torch.Tensor] = None
    pool_k: Optional[torch.Tensor] = None     # gqa/slide: [L, S, H, d]; mla: pool [L, S, W]
    pool_v: Optional[torch.Tensor] = None
    rot_dim: int = 0
    rot_offset: int = 0
    pairing: int = ROTATE_HALF
    base: float = 1e4
    kv_lora: int = 0
    inv_freq: Optional[np.ndarray] = None      # a model's own rotary frequency table (default: base^(-2i/r))
    freq_axis: Optional[np.ndarray] = None     # multi-axis RoPE: the axis each frequency follows
    axis_delta: Optional[np.ndarray] = None    # multi-axis RoPE: int64 [n_chunks, n_axes] per-chunk moves

    @property
    def tokens(self) -> int:
        return sum(c.length for c in self.chunks)

    @property
    def max_len(self) -> int:
        return max((c.length for c in self.chunks), default=0)

    @property
    def num_slots(self) -> int:
        return self.pool_k.shape[1]


def _randn_bf16(shape, std, gen, device, scale=None) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws, generated one leading slice at a time."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for i in range(shape[0]):
        x = torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32)
        if scale is not None:
            x.mul_(scale[i])
        if std != 1.0:
            x.mul_(std)
        out[i].copy_(x)
    return out


def _canary(shape, device) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.int16, device=device)
    t.fill_(CANARY_BITS if CANARY_BITS < 0x8000 else CANARY_BITS - 0x10000)
    return t.view(torch.bfloat16)


def _page_slots(name: str, lens: Sequence[int], page: int, pool_pages: Optional[int],
                first_page_gap: int = 0):
    """Slots for chunks laid end to end over randomly permuted pages.

    Chunk tokens occupy consecutive positions of one logical sequence; position p
    lives in slot perm[p // page] * page + p % page.  Returns (per-chunk slots,
    number of pool pages).
    """
    total = sum(lens) + first_page_gap
    need = -(-total // page)
    if pool_pages is None:
        pool_pages = need + max(1, need // 8)
    if pool_pages < need:
        raise ValueError("pool too small")
    perm = _np_rng(name, "pages").permutation(pool_pages)[:need].astype(np.int64)
    out = []
    pos = first_page_gap
    for t in lens:
        p = np.arange(pos, pos + t, dtype=np.int64)
        out.append(perm[p // page] * page + p % page)
        pos += t
    return out, pool_pages


def make(spec, device="cpu", with_patches: bool = True) -> Workload:
    """Materialise a spec on ``device`` (seeded; the same spec gives the same draws
    on the same device type)."""
    device = torch.device(device)
    if isinstance(spec, MlaSpec):
        return _make_mla_ingest(spec, device) if spec.kind == "mla_ingest" else _make_mla(spec, device)
    if spec.kind == "slide":
        return _make_slide(spec, device)
    if spec.kind == "ingest":
        return _make_ingest(spec, device)
    return _make_gqa(spec, device, with_patches)


def _gen(device, *tags) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_torch_seed(*tags))
    return g


def _make_gqa(spec: GqaSpec, device, with_patches: bool) -> Workload:
    L, H, d, m = spec.L, spec.H, spec.d, spec.m
    N = sum(spec.lens)
    scale_k = scale_v = None
    if spec.channel_scale:
        gs = _gen(device, spec.name, "scale")
        lo, hi = math.log(0.1), math.log(10.0)
        scale_k = torch.exp(torch.rand((L, 1, H, d), generator=gs, device=device) * (hi - lo) + lo)
        scale_v = torch.exp(torch.rand((L, 1, H, d), generator=gs, device=device) * (hi - lo) + lo)
        scale_k = scale_k[:, 0]
        scale_v = scale_v[:, 0]
    store_k = _randn_bf16((L, N, H, d), 1.0, _gen(device, spec.name, "store_k"), device, scale_k)
    store_v = _randn_bf16((L, N, H, d), 1.0, _gen(device, spec.name, "store_v"), device, scale_v)
    slots, pages = _page_slots(spec.name, spec.lens, spec.page, spec.pool_pages)
    S = pages * spec.page
    pool_k = _canary((L, S, H, d), device)
    pool_v = _canary((L, S, H, d), device)
    chunks = []
    gp = _gen(device, spec.name, "patch")
    off = 0
    for c, t in enumerate(spec.lens):
        patches = []
        if m > 0 and with_patches:
            patches = [
                _randn_bf16((L, H, t, m), 0.05, gp, device),
                _randn_bf16((L, H, d, m), 0.05, gp, device),
                _randn_bf16((L, H, t, m), 0.05, gp, device),
                _randn_bf16((L, H, d, m), 0.05, gp, device),
            ]
        chunks.append(ChunkData(off, t, int(spec.deltas[c]), m if with_patches else 0,
                                torch.from_numpy(slots[c]).to(device), patches))
        off += t
    return Workload(spec, "gqa", chunks, store_k, store_v, pool_k, pool_v,
                    rot_dim=spec.rot_dim or d, rot_offset=spec.rot_offset,
                    pairing=spec.pairing, base=spec.base)


def _make_slide(spec: GqaSpec, device) -> Workload:
    L, H, d = spec.L, spec.H, spec.d
    window = spec.window or (sum(spec.lens) + spec.evicted)
    if window != spec.evicted + sum(spec.lens):
        raise ValueError("window must equal evicted + survivors")
    # the whole window sits in the pool; the survivors are its last tokens
    win_slots, pages = _page_slots(spec.name, [window], spec.page,
                                   spec.pool_pages or -(-window // spec.page))
    S = pages * spec.page
    pool_k = _randn_bf16((L, S, H, d), 1.0, _gen(device, spec.name, "pool_k"), device)
    ws = win_slots[0]
    chunks = []
    pos = spec.evicted
    for c, t in enumerate(spec.lens):
        chunks.append(ChunkData(0, t, int(spec.deltas[c]), 0,
                                torch.from_numpy(ws[pos:pos + t].copy()).to(device), []))
        pos += t
    return Workload(spec, "slide", chunks, pool_k=pool_k, rot_dim=spec.rot_dim or d,
                    rot_offset=spec.rot_offset, pairing=spec.pairing, base=spec.base)


def _make_mla(spec: MlaSpec, device) -> Workload:
    L, W, m = spec.L, spec.kv_lora + spec.rope, spec.m
    N = sum(spec.lens)
    store = _randn_bf16((L, N, W), 1.0, _gen(device, spec.name, "store"), device)
    slots, pages = _page_slots(spec.name, spec.lens, spec.page, spec.pool_pages)
    S = pages * spec.page
    pool = _canary((L, S, W), device)
    gp = _gen(device, spec.name, "patch")
    chunks = []
    off = 0
    for c, t in enumerate(spec.lens):
        patches = []
        if m > 0:
            patches = [
                _randn_bf16((L, t, m), 0.05, gp, device),
                _randn_bf16((L, spec.kv_lora, m), 0.05, gp, device),
                _randn_bf16((L, t, m), 0.05, gp, device),
                _randn_bf16((L, spec.rope, m), 0.05, gp, device),
            ]
        chunks.append(ChunkData(off, t, int(spec.deltas[c]), m,
                                torch.from_numpy(slots[c]).to(device), patches))
        off += t
    return Workload(spec, "mla", chunks, store_k=store, pool_k=pool, rot_dim=spec.rope,
                    rot_offset=spec.kv_lora, pairing=spec.pairing, base=spec.base,
                    kv_lora=spec.kv_lora)


def _make_ingest(spec: GqaSpec, device) -> Workload:
    """Live paged cache (K, V ~ N(0,1) at the chunks' slots and elsewhere) -> canonical
    store (canary-filled); chunk c's store rows follow chunk c-1's."""
    L, H, d = spec.L, spec.H, spec.d
    N = sum(spec.lens)
    slots, pages = _page_slots(spec.name, spec.lens, spec.page, spec.pool_pages)
    S = pages * spec.page
    pool_k = _randn_bf16((L, S, H, d), 1.0, _gen(device, spec.name, "pool_k"), device)
    pool_v = _randn_bf16((L, S, H, d), 1.0, _gen(device, spec.name, "pool_v"), device)
    store_k = _canary((L, N, H, d), device)
    store_v = _canary((L, N, H, d), device)
    chunks = []
    off = 0
    for c, t in enumerate(spec.lens):
        chunks.append(ChunkData(off, t, int(spec.deltas[c]), 0, torch.from_numpy(slots[c]).to(device), []))
        off += t
    return Workload(spec, "ingest", chunks, store_k, store_v, pool_k, pool_v, rot_dim=spec.rot_dim or d,
                    rot_offset=spec.rot_offset, pairing=spec.pairing, base=spec.base)


def _make_mla_ingest(spec: MlaSpec, device) -> Workload:
    L, W = spec.L, spec.kv_lora + spec.rope
    N = sum(spec.lens)
    slots, pages = _page_slots(spec.name, spec.lens, spec.page, spec.pool_pages)
    S = pages * spec.page
    pool = _randn_bf16((L, S, W), 1.0, _gen(device, spec.name, "pool"), device)
    store = _canary((L, N, W), device)
    chunks = []
    off = 0
    for c, t in enumerate(spec.lens):
        chunks.append(ChunkData(off, t, int(spec.deltas[c]), 0, torch.from_numpy(slots[c]).to(device), []))
        off += t
    return Workload(spec, "mla_ingest", chunks, store_k=store, pool_k=pool, rot_dim=spec.rope,
                    rot_offset=spec.kv_lora, pairing=spec.pairing, base=spec.base, kv_lora=spec.kv_lora)


# ------------------------------------------------------------- accounting --
def algorithmic_bytes(spec) -> int:
    """Bytes the operator must move at minimum: canonical rows read, patch factors
    read (U: len x m and V_m: width x m per factor), rows written, int64 slot map."""
    B = 2
    T = sum(spec.lens)
    if isinstance(spec, MlaSpec):
        W = spec.kv_lora + spec.rope
        kv = T * spec.L * W * B
        patch = 0
        if spec.m:
            patch = sum((t + spec.kv_lora) * spec.m + (t + spec.rope) * spec.m
                        for t in spec.lens) * spec.L * B
        return 2 * kv + patch + T * 8
    if spec.kind == "slide":
        kv = T * spec.L * spec.H * spec.d * B
        return 2 * kv + T * 8
    if spec.kind == "ingest":
        kv = 2 * T * spec.L * spec.H * spec.d * B                  # K and V
        return 2 * kv + T * 8
    kv = 2 * T * spec.L * spec.H * spec.d * B                      # K and V
    patch = sum((t + spec.d) * spec.m for t in spec.lens) * spec.L * spec.H * 2 * B if spec.m else 0
    return 2 * kv + patch + T * 8


def tokens(spec) -> int:
    return sum(spec.lens)


def deficit_blocks(spec: DeficitSpec) -> int:
    return spec.kv * spec.L * spec.H


def deficit_bytes(spec: DeficitSpec) -> int:
    """Bytes patch formation must move at minimum: every deficit block read once
    (each of its terms), U (len x m) and V (d x m) written in bf16, fp32 sigma."""
    n = deficit_blocks(spec)
    return n * (spec.terms * spec.length * spec.d * 2 + (spec.length + spec.d) * spec.m * 2 + spec.m * 4)


def deficit_flops(spec: DeficitSpec) -> int:
    """Multiply-adds x 2 of the two contractions every method needs: the Gram
    matrix X^T X (len d^2) and U = X V (len d m), per block."""
    return deficit_blocks(spec) * 2 * (spec.length * spec.d * spec.d + spec.length * spec.d * spec.m)
