"""The algorithmic byte counts behind every roofline figure, checked against
the tensors the seeded generators actually build (small copies of each
workload, on the CPU): the rows a call reads and writes, the factors it reads
(one layer's for attention), the slot map, the queries and outputs."""
import pytest
import torch

import workloads as W


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


@pytest.mark.parametrize("name", ["qwen_recall", "dsv2_mla", "qwen_slide", "qwen_ingest", "dsv2_mla_ingest",
                                  "mha_reorder_recall"])
def test_relocation_bytes_match_the_generated_tensors(name):
    spec = W.scaled(W.CONFIGS[name](), L=2, lens=(130, 64, 7))
    wl = W.make(spec, "cpu")
    L = spec.L
    total = 0
    for c in wl.chunks:
        if wl.kind in ("mla", "mla_ingest"):
            row = wl.pool_k.shape[2] * 2                              # c_KV | k_rope
        elif wl.kind == "slide":
            row = spec.H * spec.d * 2                                 # K only
        else:
            row = 2 * spec.H * spec.d * 2                             # K and V
        total += 2 * c.length * L * row                              # read once, written once
        total += sum(_nbytes(p) for p in c.patches)                   # every layer's factors
        total += c.length * 8                                         # int64 slot map
    assert W.algorithmic_bytes(spec) == total


def test_attention_bytes_match_the_generated_tensors():
    spec = W.AttendSpec("bytes_at", H=4, G=7, d=128, seqs=((130, 64), (7,)), m=16, L=3, layer=1)
    a = W.make_attend(spec, "cpu")
    total = 0
    for c in a.chunks:
        total += c.length * spec.H * 2 * spec.d * 2                   # canonical K and V rows
        if c.rank:
            total += sum(_nbytes(p[spec.layer]) for p in c.patches)   # one layer's factors
    total += 2 * _nbytes(a.q)                                         # queries read, outputs written
    assert W.attend_bytes(spec) == total


def test_mla_attention_bytes_match_the_generated_tensors():
    spec = W.MlaAttendSpec("bytes_mla", Hq=16, seqs=((130, 64), (7,)), m=16, L=3, layer=1)
    a = W.make_mla_attend(spec, "cpu")
    total = 0
    for c in a.chunks:
        total += c.length * (spec.kv_lora + spec.rope) * 2           # canonical c_KV | k_rope rows
        if c.rank:
            total += sum(_nbytes(p[spec.layer]) for p in c.patches)   # one layer's factors
    total += _nbytes(a.q) + a.q.shape[0] * spec.Hq * spec.kv_lora * 2   # queries read, latent outputs written
    assert W.mla_attend_bytes(spec) == total


def test_deficit_bytes_match_the_generated_tensors():
    spec = W.DeficitSpec("bytes_pf", L=2, length=96, H=4, d=128, m=32, kv=2, terms=1)
    x = W.make_deficit(spec, "cpu")
    n = W.deficit_blocks(spec)
    want = _nbytes(x) + n * ((spec.length + spec.d) * spec.m * 2 + spec.m * 4)   # deficit in, U, V, sigma out
    assert W.deficit_bytes(spec) == want


def test_multi_axis_generators():
    """The axis map covers every frequency with axes 0..2 (contiguous: 1/4, 3/8,
    3/8 of the frequencies; interleaved: f mod 3) and the per-chunk moves cycle
    through whole-segment, time-only, independent and no moves."""
    sec = W.freq_axes(64, "sections")
    assert sec.tolist() == [0] * 16 + [1] * 24 + [2] * 24
    assert W.freq_axes(32, "interleaved").tolist() == [f % 3 for f in range(32)]
    mv = W.axis_moves(8, "tag")
    assert mv.shape == (8, 3)
    for c in range(8):
        kind = c % 4
        if kind == 0:
            assert mv[c, 0] == mv[c, 1] == mv[c, 2]
        elif kind == 1:
            assert mv[c, 1] == 0 and mv[c, 2] == 0
        elif kind == 3:
            assert not mv[c].any()
    assert (W.axis_moves(8, "tag") == mv).all()   # seeded


def test_prefill_flops_and_query_shape():
    """The prefill flop count against a hand count for a small case (query rows
    x tokens x 4(d + m), plus 4 d m per query row and patched chunk; every chunk
    here carries a patch), and the generated query's [S, T, H * G, d] shape."""
    spec = W.AttendSpec("pf_count", H=2, G=3, d=64, seqs=((10, 20), (5,)), m=8, kind="prefill", T=4)
    rows = 4 * 2 * 3                               # per sequence
    want = 4 * (rows * 30 + rows * 5) * (64 + 8) + 4 * (rows * 2 + rows * 1) * 64 * 8
    assert W.prefill_flops(spec) == want
    a = W.make_attend(spec, "cpu")
    assert tuple(a.q.shape) == (2, 4, 6, 64)
    full = W.qwen_prefill_reused()
    assert W.prefill_flops(full) == 1843111395328   # the figure the design notes quote
