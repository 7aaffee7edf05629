"""GPU parity of decode attention over reused chunks (kamera_attend_reused)
against the oracle's fp64 attention over the reuse equation's unrounded rows.

Tolerance: the kernel accumulates in fp32 on bf16 MMA operands (the canonical
rows and U rows are bf16 already; the turned query, V_k^T q and the softmax
weights enter as bf16 hi + lo pairs, about 16 significant bits) and rounds the
output once to bf16, so every element must lie within one bf16 ulp of the fp64
result, plus 2^-16 of sum_j p_j |V_j| (the magnitude the sums are made of:
where the output is a small difference of large terms, rounding of the terms
is what moves it)."""
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
        monkeypatch.setattr(K, "kamera_attend_reused", functools.partial(K.kamera_attend_reused, workspace=False))
    return request.param

DEV = "cuda"


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def run_attend(a: W.AttendData, err=None, seq_start=None, freq_axis=None, axis_delta=None):
    spec = a.spec
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start if seq_start is None else seq_start, dtype=torch.int32, device=DEV)
    axes = {}
    if axis_delta is not None:
        axes = dict(freq_axis=freq_axis, axis_delta=torch.as_tensor(axis_delta, dtype=torch.int64, device=DEV))
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing, **axes)
    max_len = max([c.length for c in a.chunks], default=0)
    max_rank = max([c.rank for c in a.chunks], default=0)
    out = K.kamera_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), max_len, max_rank,
                                 layer=spec.layer, err=err)
    torch.cuda.synchronize()
    return out


def oracle_attend(a: W.AttendData, freq_axis=None, axis_delta=None):
    """The oracle on the same inputs; with multi-axis moves, one table per
    chunk, theta'_f = move_c[axis_f] * theta_f, at delta 1 (0 for a chunk
    that does not move)."""
    spec = a.spec
    orc = O.default()
    th = orc.inv_freq(spec.base, a.rot_dim)
    deltas = [c.delta for c in a.chunks]
    if axis_delta is not None:
        ax = np.asarray(freq_axis, dtype=np.int64)
        th = np.stack([mv[ax].astype(np.float64) * th for mv in axis_delta]) if len(axis_delta) else th
        deltas = [int(np.any(mv != 0)) for mv in axis_delta]
    oc = [O.Chunk(c.src_offset, c.length, de, c.rank, c.slots.cpu().numpy(), [_bits(t) for t in c.patches])
          for c, de in zip(a.chunks, deltas)]
    return orc.attend(_bits(a.store_k), _bits(a.store_v), oc, a.seq_start, _bits(a.q), spec.layer, th, a.rot_dim,
                      spec.rot_offset, spec.pairing, scale=spec.d ** -0.5)


def check(a: W.AttendData, out: torch.Tensor, what: str, **axes):
    _, ref, mag = oracle_attend(a, **axes)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    allowed = _ulp_bf16(ref) + 2.0 ** -16 * mag
    bad = err > allowed
    assert not bad.any(), (what, int(bad.sum()), float(err[bad].max()), float(allowed[bad].min()))


CASES = {
    "qwen_gqa": W.AttendSpec("at_qwen", H=4, G=7, d=128, seqs=((300, 129), (64,), (200, 1, 77)), m=32),
    "mha": W.AttendSpec("at_mha", H=3, G=1, d=128, seqs=((130, 70), (65,)), m=16, base=1e4),
    "d64_interleaved_partial": W.AttendSpec("at_d64", H=2, G=2, d=64, seqs=((90, 33), (17,)), m=8, base=1e4,
                                            rot_dim=32, rot_offset=16, pairing=K.INTERLEAVED),
    "odd_rank_and_rank0": W.AttendSpec("at_odd", H=2, G=4, d=128, seqs=((100, 50, 20), (64, 64)), m=3,
                                       zero_rank_every=2),
    "rank0_only": W.AttendSpec("at_r0", H=1, G=8, d=64, seqs=((129,), (1, 2, 3)), m=0),
    "rank64": W.AttendSpec("at_m64", H=2, G=3, d=128, seqs=((150,),), m=64),
}


@pytest.mark.parametrize("name", list(CASES))
def test_attend_parity(name):
    a = W.make_attend(CASES[name], DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_attend(a, err=err)
    assert int(err.item()) == 0
    check(a, out, name)


@pytest.mark.parametrize("layout", ["sections", "interleaved"])
@pytest.mark.parametrize("name", ["qwen_gqa", "d64_interleaved_partial", "rank64"])
def test_attend_multi_axis_moves(name, layout):
    """Chunks of one sequence moved by different (time, height, width)
    amounts; the descriptors' own deltas are not used."""
    a = W.make_attend(CASES[name], DEV)
    axes = dict(freq_axis=W.freq_axes(a.rot_dim // 2, layout), axis_delta=W.axis_moves(len(a.chunks), name, layout))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_attend(a, err=err, **axes)
    assert int(err.item()) == 0
    check(a, out, f"{name} {layout}", **axes)


def test_attend_axis_move_out_of_range():
    a = W.make_attend(W.AttendSpec("at_axerr", H=2, G=2, d=64, seqs=((40,), (30,)), m=8), DEV)
    moves = np.array([[1, 2, 3], [0, -2 ** 40, 0]], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_attend(a, err=err, freq_axis=W.freq_axes(32), axis_delta=moves)
    assert int(err.item()) & 4
    assert torch.count_nonzero(out[1]).item() == 0   # the only chunk of sequence 1 was skipped


def test_empty_sequences_give_zeros():
    """A sequence without chunks, and one whose only chunk has no token."""
    a = W.make_attend(W.AttendSpec("at_empty", H=2, G=2, d=64, seqs=((40,), (), (0,)), m=8), DEV)
    out = run_attend(a)
    assert torch.count_nonzero(out[1:]).item() == 0
    check(a, out, "empty")


def test_matches_attention_over_the_materialised_pool():
    """The fused path and relocation followed by plain attention agree within the
    bf16 rounding the materialised pool adds (the pool rows are rounded, the
    fused kernel's are not)."""
    spec = W.AttendSpec("at_pool", H=4, G=7, d=128, seqs=((257, 100),), m=32, L=1, layer=0)
    a = W.make_attend(spec, DEV)
    out = run_attend(a)
    n = sum(c.length for c in a.chunks)
    pool_k = torch.zeros(1, n, spec.H, spec.d, dtype=torch.bfloat16, device=DEV)
    pool_v = torch.zeros_like(pool_k)
    specs = [K.ChunkSpec(c.src_offset, c.length, c.delta, c.rank,
                         torch.arange(c.src_offset, c.src_offset + c.length, dtype=torch.int64, device=DEV),
                         c.patches) for c in a.chunks]
    ch = K.pack_chunks(specs, device=DEV)
    K.kamera_relocate_patch(pool_k, pool_v, a.store_k[None], a.store_v[None], K.Rope(spec.base, spec.d), ch,
                            len(specs), max(c.length for c in a.chunks), spec.m)
    kf, vf = pool_k[0].float(), pool_v[0].float()               # [n, H, d]
    q = a.q[0].float().view(spec.H, spec.G, spec.d)             # [H, G, d]
    sc = torch.einsum("hgd,nhd->hgn", q, kf) * spec.d ** -0.5
    ref = torch.einsum("hgn,nhd->hgd", torch.softmax(sc, dim=-1), vf).reshape(spec.H * spec.G, spec.d)
    rel = (out[0].float() - ref).norm() / ref.norm()
    assert rel < 1e-2, float(rel)


def test_device_errors():
    a = W.make_attend(W.AttendSpec("at_err", H=2, G=2, d=64, seqs=((40,), (30,)), m=8), DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_attend(a, err=err, seq_start=[0, 2, 1])   # second sequence's range runs backwards
    assert int(err.item()) & 4
    a.chunks[1].src_offset = 10 ** 6              # source rows past the store
    err.zero_()
    run_attend(a, err=err)
    assert int(err.item()) & 2


def test_host_errors():
    a = W.make_attend(W.AttendSpec("at_host", H=2, G=3, d=96, seqs=((10,),), m=8), DEV)
    with pytest.raises(K.KameraError) as e:        # head_dim 96 is not handled
        run_attend(a)
    assert e.value.status == 3
    a = W.make_attend(W.AttendSpec("at_host9", H=1, G=9, d=64, seqs=((10,),), m=8), DEV)
    with pytest.raises(K.KameraError) as e:        # more than 8 query heads per KV head
        run_attend(a)
    assert e.value.status == 3


def test_one_unit_over_every_sm():
    """One sequence of one KV head: with a workspace its 11 tiles spread over
    every CTA that fits, so most CTAs hold an empty share and leave an empty
    partial state, which the merge must skip."""
    a = W.make_attend(W.AttendSpec("at_one", H=1, G=2, d=128, seqs=((1000, 300),), m=16), DEV)
    check(a, run_attend(a), "one unit")


def test_workspace_errors():
    """A workspace that is too small or misaligned is refused before any launch."""
    a = W.make_attend(W.AttendSpec("at_ws", H=2, G=2, d=64, seqs=((40,), (30,)), m=8), DEV)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    rope = K.Rope(a.spec.base, a.rot_dim, a.spec.rot_offset, a.spec.pairing)
    need = K.load_library().kamera_attend_workspace_bytes(2, 2, 64)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(K.KameraError) as e:
        K.kamera_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, 2, 40, 8, workspace=small)
    assert e.value.status == 1
    odd = torch.empty(need + 16, dtype=torch.uint8, device=DEV)[8:]
    with pytest.raises(K.KameraError) as e:
        K.kamera_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, 2, 40, 8, workspace=odd)
    assert e.value.status == 2
    exact = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = K.kamera_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, 2, 40, 8, layer=a.spec.layer,
                                 workspace=exact)
    torch.cuda.synchronize()
    check(a, out, "caller's workspace")
