"""GPU parity of MLA decode attention over reused chunks (kamera_mla_attend_reused)
against the oracle's fp64 attention over the MLA reuse rows.

Tolerance: the kernel accumulates in fp32 on bf16 MMA operands; the canonical
rows, U rows and latent queries are bf16 already and the rest (the turned rope
query, the per-chunk folds, the softmax weights) enter as a bf16 hi + lo pair
(about 16 significant bits), and the output is rounded once to bf16.  So every
element must lie within one bf16 ulp of the fp64 result, plus 2^-16 of
sum_j p_j |c'_j| (the scale of the terms the weighted sum is made of), as for
GQA attention."""
import functools

import numpy as np
import pytest
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["workspace", "clusters"])
def attend_path(request, monkeypatch):
    """Every case twice: with the binding's workspace (the call spreads the
    units' tiles over all SMs and merges the partial states in a second
    launch) and without one (the units' tiles split within clusters)."""
    if request.param == "clusters":
        monkeypatch.setattr(K, "kamera_mla_attend_reused", functools.partial(K.kamera_mla_attend_reused, workspace=False))
    return request.param

DEV = "cuda"


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def run_mla(a: W.MlaAttendData, err=None, seq_start=None, freq_axis=None, axis_delta=None, max_rank=None):
    spec = a.spec
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start if seq_start is None else seq_start, dtype=torch.int32, device=DEV)
    axes = {}
    if axis_delta is not None:
        axes = dict(freq_axis=freq_axis, axis_delta=torch.as_tensor(axis_delta, dtype=torch.int64, device=DEV))
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing, **axes)
    ml = max([c.length for c in a.chunks], default=0)
    mr = max([c.rank for c in a.chunks], default=0) if max_rank is None else max_rank
    out = K.kamera_mla_attend_reused(a.store, spec.kv_lora, a.q, rope, chunks, seq, len(a.chunks), ml, mr,
                                     layer=spec.layer, err=err)
    torch.cuda.synchronize()
    return out


def oracle_mla(a: W.MlaAttendData, freq_axis=None, axis_delta=None, seqs=None):
    """The oracle on the same inputs (optionally only sequences ``seqs``); with
    multi-axis moves, one table per chunk, theta'_f = move_c[axis_f] * theta_f,
    at delta 1 (0 for a chunk that does not move)."""
    spec = a.spec
    orc = O.default()
    th = orc.inv_freq(spec.base, a.rot_dim)
    deltas = [c.delta for c in a.chunks]
    if axis_delta is not None:
        ax = np.asarray(freq_axis, dtype=np.int64)
        th = np.stack([mv[ax].astype(np.float64) * th for mv in axis_delta])
        deltas = [int(np.any(mv != 0)) for mv in axis_delta]
    oc = [O.Chunk(c.src_offset, c.length, de, c.rank, c.slots.cpu().numpy(), [_bits(t) for t in c.patches])
          for c, de in zip(a.chunks, deltas)]
    q = _bits(a.q)
    starts = a.seq_start
    if seqs is not None:   # the chosen sequences only, with their own chunk ranges
        q = q[list(seqs)]
        ranges = [(a.seq_start[s], a.seq_start[s + 1]) for s in seqs]
        sub, starts = [], [0]
        for lo, hi in ranges:
            sub += oc[lo:hi]
            starts.append(len(sub))
        if np.ndim(th) == 2:
            th = np.concatenate([th[lo:hi] for lo, hi in ranges]) if sub else th[:0]
        oc = sub
    W_ = spec.kv_lora + spec.rope
    return orc.attend_mla(_bits(a.store), oc, starts, q, spec.layer, spec.kv_lora, th, a.rot_dim, spec.rot_offset,
                          spec.pairing, scale=W_ ** -0.5)


def check(a: W.MlaAttendData, out: torch.Tensor, what: str, seqs=None, **axes):
    _, ref, mag = oracle_mla(a, seqs=seqs, **axes)
    got = out.float().cpu().numpy().astype(np.float64)
    if seqs is not None:
        got = got[list(seqs)]
    err = np.abs(got - ref)
    allowed = _ulp_bf16(ref) + 2.0 ** -16 * mag
    bad = err > allowed
    assert not bad.any(), (what, int(bad.sum()), float(err[bad].max()), float(allowed[bad].min()))


CASES = {
    "dsv2_ragged": W.MlaAttendSpec("mla_dsv2", Hq=16, seqs=((300, 129), (64,), (200, 1, 77)), m=16),
    "rank32": W.MlaAttendSpec("mla_m32", Hq=16, seqs=((150, 65),), m=32),
    "rank0": W.MlaAttendSpec("mla_r0", Hq=16, seqs=((129,), (1, 2, 3)), m=0),
    "few_heads_rotate_half_partial": W.MlaAttendSpec("mla_h5", Hq=5, seqs=((90, 33), (17,)), m=8,
                                                     pairing=K.ROTATE_HALF, rot_dim=32, rot_offset=16),
    "mixed_ranks": W.MlaAttendSpec("mla_mix", Hq=16, seqs=((100, 50, 20), (64, 64)), m=6, zero_rank_every=2),
    "one_sequence_ten_chunks": W.MlaAttendSpec("mla_10", Hq=16, seqs=((70,) * 10,), m=16),
    "one_head": W.MlaAttendSpec("mla_h1", Hq=1, seqs=((65, 64),), m=16, base=1e6),
    "one_long_chunk_cut_across_the_cluster": W.MlaAttendSpec("mla_long", Hq=16, seqs=((1000,),), m=32),
    # more than 16 query heads per latent row: groups of 16, the last one partial
    "heads_17": W.MlaAttendSpec("mla_h17", Hq=17, seqs=((130, 40), (64,)), m=16),
    "heads_40_ragged": W.MlaAttendSpec("mla_h40", Hq=40, seqs=((300, 7), (1,), (129, 64, 65)), m=8),
    "deepseek_v3_128_heads": W.MlaAttendSpec("mla_h128", Hq=128, seqs=((500, 77), (256,)), m=32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_mla_attend_parity(name):
    a = W.make_mla_attend(CASES[name], DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_mla(a, err=err)
    assert int(err.item()) == 0
    check(a, out, name)


def test_mla_attend_rank_instantiations():
    """A rank-8 call run through the rank-16 and rank-32 kernels (max_rank 16 and
    32) gives the same bits: the padded U columns contribute exact zeros."""
    a = W.make_mla_attend(W.MlaAttendSpec("mla_pad", Hq=16, seqs=((130, 40),), m=8), DEV)
    o16 = run_mla(a, max_rank=16).clone()
    o32 = run_mla(a, max_rank=32)
    assert torch.equal(o16, o32)
    check(a, o16, "pad")


@pytest.mark.parametrize("layout", ["sections", "interleaved"])
def test_mla_attend_multi_axis_moves(layout):
    a = W.make_mla_attend(CASES["dsv2_ragged"], DEV)
    axes = dict(freq_axis=W.freq_axes(a.rot_dim // 2, layout),
                axis_delta=W.axis_moves(len(a.chunks), "mla_attend", layout))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_mla(a, err=err, **axes)
    assert int(err.item()) == 0
    check(a, out, layout, **axes)


def test_mla_attend_empty_sequences_give_zeros():
    a = W.make_mla_attend(W.MlaAttendSpec("mla_empty", Hq=16, seqs=((40,), (), (0,)), m=8), DEV)
    out = run_mla(a)
    assert torch.count_nonzero(out[1:]).item() == 0
    check(a, out, "empty")


def test_mla_attend_matches_attention_over_the_materialised_pool():
    """The fused path and MLA relocation followed by plain attention over the
    pool rows agree within the bf16 rounding the materialised pool adds."""
    spec = W.MlaAttendSpec("mla_pool", Hq=16, seqs=((257, 100),), m=16, L=1, layer=0)
    a = W.make_mla_attend(spec, DEV)
    out = run_mla(a)
    n = sum(c.length for c in a.chunks)
    Wd = spec.kv_lora + spec.rope
    pool = torch.zeros(1, n, Wd, dtype=torch.bfloat16, device=DEV)
    specs = [K.ChunkSpec(c.src_offset, c.length, c.delta, c.rank,
                         torch.arange(c.src_offset, c.src_offset + c.length, dtype=torch.int64, device=DEV),
                         c.patches) for c in a.chunks]
    ch = K.pack_chunks(specs, device=DEV)
    K.kamera_mla_relocate_patch(pool, a.store[None], spec.kv_lora, K.Rope(spec.base, spec.rope, 0, spec.pairing), ch,
                                len(specs), max(c.length for c in a.chunks), spec.m)
    rows = pool[0].float()                                   # [n, W]
    q = a.q[0].float()                                       # [Hq, W]
    sc = (q @ rows.T) * Wd ** -0.5
    ref = torch.softmax(sc, dim=-1) @ rows[:, :spec.kv_lora]
    rel = (out[0].float() - ref).norm() / ref.norm()
    assert rel < 1e-2, float(rel)


def test_mla_attend_device_errors():
    a = W.make_mla_attend(W.MlaAttendSpec("mla_err", Hq=16, seqs=((40,), (30,)), m=8), DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_mla(a, err=err, seq_start=[0, 2, 1])   # second sequence's range runs backwards
    assert int(err.item()) & 4
    a.chunks[1].src_offset = 10 ** 6              # source rows past the store
    err.zero_()
    out = run_mla(a, err=err)
    assert int(err.item()) & 2
    assert torch.count_nonzero(out[1]).item() == 0
    b = W.make_mla_attend(W.MlaAttendSpec("mla_odd", Hq=16, seqs=((40,), (30,)), m=8), DEV)
    b.chunks[0].rank = 7                          # an odd rank is a descriptor error
    err.zero_()
    out = run_mla(b, err=err, max_rank=8)
    assert int(err.item()) & 4
    assert torch.count_nonzero(out[0]).item() == 0
    check_b = W.MlaAttendData(b.spec, b.store, [b.chunks[1]], [0, 0, 1], b.q)
    check(check_b, out, "odd rank: the other sequence")


def test_mla_attend_host_errors():
    a = W.make_mla_attend(W.MlaAttendSpec("mla_h129", Hq=129, seqs=((10,),), m=8), DEV)
    with pytest.raises(K.KameraError) as e:        # more than 128 query heads
        run_mla(a)
    assert e.value.status == 3
    a = W.make_mla_attend(W.MlaAttendSpec("mla_m34", Hq=16, seqs=((10,),), m=34), DEV)
    with pytest.raises(K.KameraError) as e:        # rank above 32
        run_mla(a)
    assert e.value.status == 3
    a = W.make_mla_attend(W.MlaAttendSpec("mla_c256", Hq=16, seqs=((10,),), m=8, kv_lora=256), DEV)
    with pytest.raises(K.KameraError) as e:        # a latent width other than 512
        run_mla(a)
    assert e.value.status == 3
