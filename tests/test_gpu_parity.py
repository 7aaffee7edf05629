"""GPU parity: every entry point through the C ABI against the fp64 oracle,
element by element, at sizes that span several token tiles, ragged tails and
page boundaries, plus the degenerate cases of the method."""
import numpy as np
import pytest
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(params=["auto", "copies", "simt", "umma"])
def path(request, monkeypatch):
    """Run the case on the default kernel choice (tensor-core path for patched
    GQA/MHA/MLA calls but short chunks with tiny ranks; factor tiles by
    tensor-map loads where the host copy of the descriptors allows), on the same
    choice without the host copy (every factor tile by per-thread copies),
    pinned to the CUDA-core path, and on the tensor-core path wherever it
    applies."""
    monkeypatch.setenv("KAMERA_PATH", request.param if request.param in ("simt", "umma") else "auto")
    monkeypatch.setattr(Hn, "USE_HOST_COPY", request.param != "copies")
    return request.param


def _cases():
    return {
        "tiny_gqa": W.tiny_gqa(),
        "qwen_recall_small": W.scaled(W.qwen_recall(), L=3, lens=(1296, 200, 65, 1)),
        "dsv2_mla_small": W.scaled(W.dsv2_mla(), L=2, lens=(300, 129, 64, 7)),
        "qwen_slide_small": W.scaled(W.qwen_slide(), L=2, lens=(1296, 77, 128)),
        "mha_reorder_recall_small": W.scaled(W.mha_reorder_recall(), L=2, H=4, lens=(513, 256, 1000, 2048, 300)),
        "tiny_gqa_x64": W.tiny_gqa_x(64),
        "qwen_ingest_small": W.scaled(W.qwen_ingest(), L=2, lens=(1296, 200, 65, 1)),
        "dsv2_mla_ingest_small": W.scaled(W.dsv2_mla_ingest(), L=2, lens=(300, 129, 7)),
    }


@pytest.mark.parametrize("name", list(_cases()))
def test_parity(name, path):
    spec = _cases()[name]
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, name)
    assert int(err.item()) == 0


@pytest.mark.parametrize("pairing,rot_dim,rot_offset", [(K.INTERLEAVED, 128, 0), (K.ROTATE_HALF, 64, 32),
                                                        (K.INTERLEAVED, 32, 96), (K.ROTATE_HALF, 16, 0),
                                                        (K.ROTATE_HALF, 0, 0)])
def test_gqa_rope_layouts(pairing, rot_dim, rot_offset, path):
    spec = W.scaled(W.qwen_recall(), L=2, lens=(150, 64), m=16)
    spec = W.GqaSpec(**{**spec.__dict__, "pairing": pairing, "rot_dim": rot_dim, "rot_offset": rot_offset})
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, f"rope {pairing}/{rot_dim}/{rot_offset}")


@pytest.mark.parametrize("table", ["extended", "temporal", "axes"])
@pytest.mark.parametrize("name", ["qwen_recall", "dsv2_mla", "qwen_slide", "qwen_ingest", "dsv2_mla_ingest"])
def test_model_frequency_tables(name, table, path):
    """A model's own frequency table passed through the RoPE override: a
    context-extension rescale, and multi-axis RoPE moved along time only or by
    per-axis shares of delta.  Every kind of call, against the oracle given
    the same table."""
    spec = W.scaled(W.CONFIGS[name](), L=2, lens=(300, 129, 7))
    wl = W.make(spec, DEV)
    wl.inv_freq = W.model_inv_freq(table, wl.base, wl.rot_dim)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, f"{name} {table}")
    assert int(err.item()) == 0


@pytest.mark.parametrize("layout", ["sections", "interleaved"])
@pytest.mark.parametrize("name", ["qwen_recall", "dsv2_mla", "qwen_slide", "qwen_ingest", "dsv2_mla_ingest",
                                  "mha_reorder_recall"])
def test_multi_axis_moves(name, layout, path):
    """Multi-axis RoPE with per-chunk moves along (time, height, width): a
    whole-segment move, a move along time only, independent axis moves and no
    move, in one call, the frequencies following their axes in contiguous
    sections or interleaved.  The descriptors' own deltas are not used.
    Against the oracle run chunk by chunk over each chunk's table
    theta'_f = move[axis_f] * theta_f."""
    spec = W.scaled(W.CONFIGS[name](), L=2, lens=(300, 129, 7, 64, 33))
    wl = W.make(spec, DEV)
    wl.freq_axis = W.freq_axes(wl.rot_dim // 2, layout)
    wl.axis_delta = W.axis_moves(len(wl.chunks), name, layout)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, f"{name} {layout}")
    assert int(err.item()) == 0
    if wl.kind == "slide":   # a chunk that does not move is left as it was, bit for bit
        for c, mv in zip(wl.chunks, wl.axis_delta):
            if not mv.any():
                sl = c.slots.cpu().numpy()
                assert np.array_equal(Hn.u16(wl.pool_k)[:, sl], h.pool_k[:, sl])


@pytest.mark.parametrize("kind", ["qwen_recall", "qwen_slide"])
def test_device_error_axis_move_out_of_range(kind, path):
    """A chunk with an axis move beyond 2^31 - 1 is skipped whole with the
    descriptor bit; the other chunk is still right."""
    spec = W.scaled(W.CONFIGS[kind](), L=2, lens=(70, 50))
    wl = W.make(spec, DEV)
    wl.freq_axis = W.freq_axes(wl.rot_dim // 2)
    wl.axis_delta = np.array([[5, -3, 9], [0, 2 ** 40, 0]], dtype=np.int64)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 4
    gk = Hn.u16(wl.pool_k)
    s1 = wl.chunks[1].slots.cpu().numpy()
    assert np.array_equal(gk[:, s1], h.pool_k[:, s1])
    good = W.Workload(wl.spec, wl.kind, [wl.chunks[0]], wl.store_k, wl.store_v, wl.pool_k, wl.pool_v,
                      wl.rot_dim, wl.rot_offset, wl.pairing, wl.base, freq_axis=wl.freq_axis,
                      axis_delta=wl.axis_delta[:1])
    hg = Hn.HostCopy(h.store_k, h.store_v, h.pool_k, h.pool_v, [h.chunks[0]])
    ok, ov, sk, sv = Hn.run_oracle(good, hg)
    s0 = h.chunks[0].slots
    Hn.compare(gk[:, s0], ok[:, s0], sk[:, s0], what="good chunk")


@pytest.mark.parametrize("m", [1, 3, 8, 16, 17, 32, 48, 64, 96, 128])
def test_gqa_ranks(m, path):
    spec = W.scaled(W.qwen_recall(), L=1, H=2, lens=(130, 5), m=m)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, f"rank {m}")


@pytest.mark.parametrize("m", [16, 32, 64, 128])
def test_mla_ranks(m, path):
    """Every rank whose factor tiles a tensor map can carry, on both MLA channels."""
    spec = W.scaled(W.dsv2_mla(), L=2, lens=(300, 128, 9), m=m)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, f"mla rank {m}")


def test_more_chunks_than_map_table(path):
    """A call with more chunks than the tensor-map table: the chunks past it
    move their factor tiles by per-thread copies within the same launch."""
    spec = W.scaled(W.qwen_recall(), L=1, H=2, lens=tuple([37, 130, 64, 1, 200] * 24), m=32)
    wl = W.make(spec, DEV)
    assert len(wl.chunks) == 120
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, "120 chunks")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_gqa_head_dims(d, path):
    spec = W.GqaSpec("hd", "gqa", L=2, H=2, d=d, base=1e4, lens=(140, 33), deltas=(999, -5), m=16, page=16)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, f"head_dim {d}")


def test_zero_delta_zero_rank_is_bit_exact_permutation(path):
    spec = W.scaled(W.qwen_recall(), L=2, lens=(300, 41), m=0)
    spec = W.GqaSpec(**{**spec.__dict__, "deltas": (0, 0)})
    wl = W.make(spec, DEV)
    wl.store_k.view(torch.int16)[0, :5] = -32768          # -0.0 survives a copy
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    torch.cuda.synchronize()
    gk, gv = Hn.u16(wl.pool_k), Hn.u16(wl.pool_v)
    for c in h.chunks:
        src = slice(c.src_offset, c.src_offset + c.length)
        assert np.array_equal(gk[:, c.slots], h.store_k[:, src])
        assert np.array_equal(gv[:, c.slots], h.store_v[:, src])


def test_rank0_values_are_bit_copies():
    spec = W.scaled(W.qwen_recall(), L=2, lens=(200,), m=0)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    torch.cuda.synchronize()
    gv = Hn.u16(wl.pool_v)
    c = h.chunks[0]
    assert np.array_equal(gv[:, c.slots], h.store_v[:, c.src_offset:c.src_offset + c.length])
    Hn.check_parity(wl, h, "rank0")


def test_mla_rank0_c_kv_bit_exact(path):
    spec = W.scaled(W.dsv2_mla(), L=2, lens=(257, 64), m=0)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, "mla rank0")   # includes the bit-exact c_KV check


def test_slide_mla_rope_subrange(path):
    """Slide on an MLA pool: only k_rope (offset 512, 64 wide, interleaved) turns."""
    spec = W.GqaSpec("mla_slide", "slide", L=2, H=1, d=576, base=1e4, lens=(200, 64), deltas=(-4096, 17),
                     m=0, page=64, pairing=K.INTERLEAVED, rot_dim=64, rot_offset=512, evicted=100, window=364)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    Hn.check_parity(wl, h, "mla slide")
    gk = Hn.u16(wl.pool_k)
    sl = Hn.touched_slots(wl)
    assert np.array_equal(gk[:, sl, :, :512], h.pool_k[:, sl, :, :512])


def test_slide_zero_delta_is_noop(path):
    spec = W.scaled(W.qwen_slide(), L=1, lens=(100,))
    spec = W.GqaSpec(**{**spec.__dict__, "deltas": (0,)})
    wl = W.make(spec, DEV)
    before = Hn.u16(wl.pool_k)
    Hn.run_gpu(wl)
    torch.cuda.synchronize()
    assert np.array_equal(Hn.u16(wl.pool_k), before)


@pytest.mark.parametrize("H,d,rot_dim,rot_offset,pairing", [
    (3, 128, 128, 0, K.ROTATE_HALF),     # 24 units per row: the CUDA-core path
    (8, 64, 32, 16, K.ROTATE_HALF),      # rotary sub-range inside each head
    (2, 256, 256, 0, K.ROTATE_HALF),
    (32, 128, 128, 0, K.ROTATE_HALF),    # 256 units per row: one row per pass
    (64, 64, 64, 0, K.INTERLEAVED),      # 512 units per row: the CUDA-core path
    (4, 128, 64, 64, K.INTERLEAVED)])
def test_slide_shapes(H, d, rot_dim, rot_offset, pairing, path):
    """In-place rotation over head counts, head dims, rotary sub-ranges and
    pairings, with ragged chunk tails and page boundaries."""
    spec = W.GqaSpec("slide_shape", "slide", L=2, H=H, d=d, base=1e4, lens=(300, 129, 1), deltas=(-32768, 5, 999),
                     m=0, page=16, pairing=pairing, rot_dim=rot_dim, rot_offset=rot_offset, evicted=100, window=530)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, f"slide H{H} d{d} r{rot_dim}+{rot_offset}")
    assert int(err.item()) == 0


def test_empty_and_zero_length():
    spec = W.scaled(W.qwen_recall(), L=1, lens=(40,), m=4)
    wl = W.make(spec, DEV)
    before_k = Hn.u16(wl.pool_k)
    # no chunks: a no-op
    K.kamera_relocate_patch(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, Hn.rope_of(wl),
                            torch.empty(0, dtype=torch.uint8, device=DEV), 0, 40, 4)
    # a zero-length chunk: nothing written, no error
    z = W.ChunkData(0, 0, 5, 0, torch.empty(0, dtype=torch.int64, device=DEV), [])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    K.kamera_relocate_patch(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, Hn.rope_of(wl),
                            K.pack_chunks([z], device=DEV), 1, 40, 4, err)
    torch.cuda.synchronize()
    assert np.array_equal(Hn.u16(wl.pool_k), before_k)
    assert int(err.item()) == 0


def _bad_case(mutate, expect_bits, skip_whole_chunk=True):
    spec = W.scaled(W.qwen_recall(), L=2, lens=(70, 50), m=8)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    bad = wl.chunks[1]
    mutate(wl, bad)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err, max_len=70, mrank=8)
    torch.cuda.synchronize()
    assert int(err.item()) & expect_bits == expect_bits
    # the good chunk is still right
    good = W.Workload(wl.spec, wl.kind, [wl.chunks[0]], wl.store_k, wl.store_v, wl.pool_k, wl.pool_v,
                      wl.rot_dim, wl.rot_offset, wl.pairing, wl.base)
    hg = Hn.HostCopy(h.store_k, h.store_v, h.pool_k, h.pool_v, [h.chunks[0]])
    ok, ov, sk, sv = Hn.run_oracle(good, hg)
    gk = Hn.u16(wl.pool_k)
    s0 = h.chunks[0].slots
    Hn.compare(gk[:, s0], ok[:, s0], sk[:, s0], what="good chunk")
    return wl, h, gk


def test_device_error_slot_out_of_range(path):
    def mut(wl, c):
        c.slots = c.slots.clone()
        c.slots[7] = wl.num_slots + 3
    wl, h, gk = _bad_case(mut, 1)
    # only that row was skipped: the others of the chunk were written
    sl = wl.chunks[1].slots.cpu().numpy()
    written = [s for i, s in enumerate(sl) if i != 7]
    assert not np.array_equal(gk[:, written], h.pool_k[:, written])


def test_device_error_source_range(path):
    def mut(wl, c):
        c.src_offset = wl.store_k.shape[1] - 10
    wl, h, gk = _bad_case(mut, 2)
    sl = wl.chunks[1].slots.cpu().numpy()
    assert np.array_equal(gk[:, sl], h.pool_k[:, sl])   # whole chunk skipped


def test_device_error_len_and_rank(path):
    def mut(wl, c):
        c.rank = 8
    spec = W.scaled(W.qwen_recall(), L=1, lens=(70, 90), m=8)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err, max_len=80, mrank=8)        # chunk 1 is longer than max_len
    torch.cuda.synchronize()
    assert int(err.item()) == 8
    gk = Hn.u16(wl.pool_k)
    sl = wl.chunks[1].slots.cpu().numpy()
    assert np.array_equal(gk[:, sl], h.pool_k[:, sl])
    err.zero_()
    Hn.run_gpu(wl, err=err, max_len=90, mrank=4)        # rank 8 > max_rank 4
    torch.cuda.synchronize()
    assert int(err.item()) == 16


def test_device_error_null_factor(path):
    def mut(wl, c):
        c.patches = [c.patches[0], None, c.patches[2], c.patches[3]]
    wl, h, gk = _bad_case(mut, 4)


def test_host_errors():
    """Argument errors are reported synchronously and enqueue nothing."""
    spec = W.scaled(W.qwen_recall(), L=1, lens=(16,), m=4)
    wl = W.make(spec, DEV)
    before = Hn.u16(wl.pool_k)
    ch = K.pack_chunks(wl.chunks, device=DEV)
    r = Hn.rope_of(wl)
    args = (wl.pool_k, wl.pool_v, wl.store_k, wl.store_v)
    cases = [
        ((*args, K.Rope(1e6, 12), ch, 1, 16, 4), 3),          # rot_dim not a multiple of 16
        ((*args, K.Rope(1e6, 128, 8), ch, 1, 16, 4), 1),      # rotary range past head_dim
        ((*args, r, ch, 1, 16, 999), 3),                      # max_rank beyond the build limit
        ((*args, r, ch, -1, 16, 4), 1),                       # negative chunk count
        ((*args, K.Rope(-1.0, 128), ch, 1, 16, 4), 1),        # base must be positive
    ]
    L, S, H, d = wl.pool_k.shape
    mis_k = torch.as_strided(wl.pool_k.view(-1)[1:], (L, S - 1, H, d), (S * H * d, H * d, d, 1))
    mis_v = torch.as_strided(wl.pool_v.view(-1)[1:], (L, S - 1, H, d), (S * H * d, H * d, d, 1))
    cases.append(((mis_k, mis_v, wl.store_k, wl.store_v, r, ch, 1, 16, 4), 2))     # misaligned base
    over = torch.as_strided(wl.pool_k, wl.store_k.shape, wl.store_k.stride())
    cases.append(((wl.pool_k, wl.pool_v, over, wl.store_v, r, ch, 1, 16, 4), 1))  # store overlaps pool
    for a, status in cases:
        with pytest.raises(K.KameraError) as e:
            K.kamera_relocate_patch(*a)
        assert e.value.status == status, (status, e.value)
    torch.cuda.synchronize()
    assert np.array_equal(Hn.u16(wl.pool_k), before)


def test_mixed_ranks_in_one_call(path):
    """Chunks of rank 32, 0 and 16 in one call (the tensor-core path skips the
    MMA for rank-0 chunks and pads rank 16 inside its operand tiles)."""
    spec = W.scaled(W.qwen_recall(), L=2, lens=(300, 200, 129, 64, 260), m=32)
    wl = W.make(spec, DEV)
    for i in (1, 3):
        wl.chunks[i].rank = 0
        wl.chunks[i].patches = []
    c = wl.chunks[2]
    c.rank = 16
    c.patches = [p[..., :16].contiguous() for p in c.patches]
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, "mixed ranks")
    assert int(err.item()) == 0


def test_many_tiles_per_cta_boundaries(path):
    """More tiles than CTAs with uneven chunk lengths: contiguous tile ranges of
    the persistent grid start and end inside chunks and segments."""
    lens = tuple(int(x) for x in np.random.default_rng(5).integers(1, 700, size=23))
    spec = W.scaled(W.mha_reorder_recall(), L=3, H=3, lens=lens, m=24)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, "many tiles")
    assert int(err.item()) == 0


# ------------------------------------------------------------ canonical ingest
@pytest.mark.parametrize("H,d,rot_dim,rot_offset,pairing", [
    (4, 128, 128, 0, K.ROTATE_HALF),
    (3, 128, 128, 0, K.ROTATE_HALF),     # units per row do not divide the block: strided items
    (8, 64, 32, 16, K.ROTATE_HALF),      # copied columns on both sides of the rotary range
    (2, 256, 256, 0, K.ROTATE_HALF),
    (4, 128, 24, 8, K.INTERLEAVED),      # interleaved range that is not a multiple of 16
    (32, 128, 128, 0, K.INTERLEAVED),
    (2, 64, 0, 0, K.ROTATE_HALF)])       # no rotary range: a pure gather
def test_ingest_shapes(H, d, rot_dim, rot_offset, pairing):
    spec = W.GqaSpec("ingest_shape", "ingest", L=2, H=H, d=d, base=1e4, lens=(300, 129, 1),
                     deltas=(-32768, -5, 0), m=0, page=16, pairing=pairing, rot_dim=rot_dim, rot_offset=rot_offset)
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    Hn.check_parity(wl, h, f"ingest H{H} d{d} r{rot_dim}+{rot_offset}")
    assert int(err.item()) == 0


def test_ingest_zero_delta_is_a_bit_exact_gather():
    spec = W.scaled(W.qwen_ingest(), L=2, lens=(257, 3))
    spec = W.GqaSpec(**{**spec.__dict__, "deltas": (0, 0)})
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    Hn.run_gpu(wl)
    torch.cuda.synchronize()
    for c in wl.chunks:
        sl = c.slots.cpu().numpy()
        rows = np.arange(c.src_offset, c.src_offset + c.length)
        assert np.array_equal(Hn.u16(wl.store_k)[:, rows], h.pool_k[:, sl])
        assert np.array_equal(Hn.u16(wl.store_v)[:, rows], h.pool_v[:, sl])


def test_ingest_then_relocate_round_trip():
    """Ingest by -s, then relocate (rank 0) by +s into an empty pool at the same
    slots: the live rows come back within two bf16 roundings."""
    spec = W.scaled(W.qwen_ingest(), L=2, lens=(300, 77))
    wl = W.make(spec, DEV)
    Hn.run_gpu(wl)
    pool_k2 = torch.zeros_like(wl.pool_k)
    pool_v2 = torch.zeros_like(wl.pool_v)
    back = [W.ChunkData(c.src_offset, c.length, -c.delta, 0, c.slots, []) for c in wl.chunks]
    K.kamera_relocate_patch(pool_k2, pool_v2, wl.store_k, wl.store_v, Hn.rope_of(wl),
                            K.pack_chunks(back, device=DEV), len(back), wl.max_len, 0)
    torch.cuda.synchronize()
    sl = Hn.touched_slots(wl)
    a = wl.pool_k[:, sl].float()
    b = pool_k2[:, sl].float()
    assert torch.equal(pool_v2[:, sl], wl.pool_v[:, sl])
    assert float((a - b).abs().max()) <= 2.0 ** -6 * float(a.abs().max())


@pytest.mark.parametrize("bad", ["slot", "store_row", "rank"])
def test_ingest_device_errors(bad):
    spec = W.scaled(W.qwen_ingest(), L=1, lens=(100, 50))
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    c = wl.chunks[1]
    if bad == "slot":
        c.slots = c.slots.clone()
        c.slots[7] = wl.pool_k.shape[1] + 3
    elif bad == "store_row":
        c.src_offset = wl.store_k.shape[1] - 10
    else:
        c.rank = 1
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    chunks = K.pack_chunks(wl.chunks, device=DEV) if bad != "rank" else None
    if bad == "rank":   # a rank-1 descriptor with no factors: pack by hand through the ChunkSpec path
        specs = [K.ChunkSpec(x.src_offset, x.length, x.delta, 0, x.slots) for x in wl.chunks]
        chunks = K.pack_chunks(specs, device=DEV)
        raw = chunks.cpu().numpy().copy()
        raw[64 + 12:64 + 16] = np.frombuffer(np.int32(1).tobytes(), np.uint8)   # rank field of chunk 1
        chunks = torch.from_numpy(raw).to(DEV)
    Hn.run_gpu(wl, chunks_dev=chunks, err=err)
    torch.cuda.synchronize()
    bits = {"slot": 1, "store_row": 2, "rank": 4}[bad]   # KAMERA_DEVERR_SLOT, _SOURCE, _DESCRIPTOR
    assert int(err.item()) & bits
    # chunk 0 was ingested regardless
    rows0 = np.arange(0, 100)
    assert not np.array_equal(Hn.u16(wl.store_k)[:, rows0], h.store_k[:, rows0])


@pytest.mark.parametrize("family,stale", [("gqa", "pointers"), ("gqa", "len"), ("mla", "pointers")])
def test_stale_host_copy_takes_the_copy_path(family, stale):
    """A host descriptor copy that disagrees with the device array: its U
    pointers name other live tensors of the same shape (or its len differs).
    The device descriptors decide: the output matches the oracle on them, the
    mismatched chunks' factor tiles move by per-thread copies, and the call
    reports KAMERA_DEVERR_DESCRIPTOR.  Every address involved stays valid."""
    base = W.qwen_recall() if family == "gqa" else W.dsv2_mla()
    spec = W.scaled(base, L=2, lens=(300, 129, 200))
    wl = W.make(spec, DEV)
    h = Hn.snapshot(wl)
    chunks = K.pack_chunks(wl.chunks, device=DEV)
    decoys = []
    host = []
    for i, c in enumerate(wl.chunks):
        if i == 1:   # the middle chunk is described differently on the host
            if stale == "pointers":
                d = [torch.randn_like(c.patches[0], dtype=torch.float32).to(torch.bfloat16), c.patches[1],
                     torch.randn_like(c.patches[2], dtype=torch.float32).to(torch.bfloat16), c.patches[3]]
                decoys.append(d)
                host.append(W.ChunkData(c.src_offset, c.length, c.delta, c.rank, c.slots, d))
            else:
                host.append(W.ChunkData(c.src_offset, c.length - 64, c.delta, c.rank, c.slots[:c.length - 64],
                                        c.patches))
        else:
            host.append(c)
    hc = K.pack_chunks(host, device="cpu")
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    n, ml, mr = len(wl.chunks), wl.max_len, Hn.max_rank(wl)
    if family == "gqa":
        K.kamera_relocate_patch(wl.pool_k, wl.pool_v, wl.store_k, wl.store_v, Hn.rope_of(wl), chunks, n, ml, mr,
                                err, host_chunks=hc)
    else:
        K.kamera_mla_relocate_patch(wl.pool_k, wl.store_k, wl.kv_lora, Hn.rope_of(wl), chunks, n, ml, mr, err,
                                    host_chunks=hc)
    torch.cuda.synchronize()
    assert int(err.item()) == 4, int(err.item())   # KAMERA_DEVERR_DESCRIPTOR alone
    Hn.check_parity(wl, h, f"stale host copy ({family}, {stale})")
    del decoys
