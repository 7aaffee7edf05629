"""GPU parity of prefill attention over reused chunks
(kamera_prefill_attend_reused) against the oracle's fp64 attention of every
query token over the reuse equation's unrounded rows, with its log-sum-exp.

Tolerance: the kernel accumulates in fp32 on the tensor cores from bf16
operands (the canonical rows and U rows are bf16 already; the turned query,
V_k^T q and the softmax weights enter as bf16 hi + lo pairs, about 16
significant bits) and rounds the output once to bf16, so every element must lie
within one bf16 ulp of the fp64 result plus 2^-16 of sum_j p_j |V_j| (the
magnitude the sums are made of).  The log-sum-exp is a float: its error is
that of the scores (about 2^-16 of their size) plus the fp32 rounding of the
sum of weights, so it must lie within 1e-4 + 2^-16 |lse| of the oracle's."""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def run_prefill(a: W.AttendData, err=None, seq_start=None, lse=None):
    spec = a.spec
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start if seq_start is None else seq_start, dtype=torch.int32, device=DEV)
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing)
    max_len = max([c.length for c in a.chunks], default=0)
    max_rank = max([c.rank for c in a.chunks], default=0)
    out, lse = K.kamera_prefill_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), max_len,
                                              max_rank, layer=spec.layer, err=err, lse=lse)
    torch.cuda.synchronize()
    return out, lse


def oracle_prefill(a: W.AttendData, seqs=None):
    """The oracle on the same inputs (optionally on a subset of the sequences)."""
    spec = a.spec
    orc = O.default()
    th = orc.inv_freq(spec.base, a.rot_dim)
    seqs = range(len(a.seq_start) - 1) if seqs is None else seqs
    chunks, starts = [], [0]
    for s in seqs:
        for c in a.chunks[a.seq_start[s]:a.seq_start[s + 1]]:
            chunks.append(O.Chunk(c.src_offset, c.length, c.delta, c.rank, c.slots.cpu().numpy(),
                                  [_bits(t) for t in c.patches]))
        starts.append(len(chunks))
    q = _bits(a.q)[list(seqs)]
    return orc.attend_prefill(_bits(a.store_k), _bits(a.store_v), chunks, starts, q, spec.layer, th, a.rot_dim,
                              spec.rot_offset, spec.pairing, scale=spec.d ** -0.5)


def check(a: W.AttendData, out: torch.Tensor, lse: torch.Tensor, what: str, seqs=None):
    _, ref, mag, ref_lse = oracle_prefill(a, seqs)
    idx = list(range(out.shape[0])) if seqs is None else list(seqs)
    got = out[idx].float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    allowed = _ulp_bf16(ref) + 2.0 ** -16 * mag
    bad = err > allowed
    assert not bad.any(), (what, int(bad.sum()), float(err[bad].max()), float(allowed[bad].min()))
    if lse is not None:
        gl = lse[idx].cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin), what
        assert np.all(gl[~fin] == -np.inf), what
        le = np.abs(gl[fin] - ref_lse[fin])
        assert np.all(le <= 1e-4 + 2.0 ** -16 * np.abs(ref_lse[fin])), (what, float(le.max()))


def spec(name, T, **kw):
    return W.AttendSpec(name, kind="prefill", T=T, **kw)


CASES = {
    # 140 query rows per (sequence, KV head): a full block of 128 and a ragged one
    "qwen_gqa": spec("pf_qwen", 20, H=4, G=7, d=128, seqs=((300, 129), (64,), (200, 1, 77)), m=32),
    "mha": spec("pf_mha", 130, H=3, G=1, d=128, seqs=((130, 70), (65,)), m=16, base=1e4),
    "d64_interleaved_partial": spec("pf_d64", 70, H=2, G=2, d=64, seqs=((90, 33), (17,)), m=8, base=1e4,
                                    rot_dim=32, rot_offset=16, pairing=K.INTERLEAVED),
    "odd_rank_and_rank0": spec("pf_odd", 33, H=2, G=4, d=128, seqs=((100, 50, 20), (64, 64)), m=3,
                               zero_rank_every=2),
    "rank0_only": spec("pf_r0", 16, H=1, G=8, d=64, seqs=((129,), (1, 2, 3)), m=0),
    "rank64": spec("pf_m64", 50, H=2, G=3, d=128, seqs=((150,),), m=64),
    "rank12_d64": spec("pf_m12", 40, H=2, G=5, d=64, seqs=((70, 200),), m=12),
    # partial rotary ranges: rotate-half with a half of three 16-byte pieces, interleaved pairs over
    # five pieces, both starting past the first piece
    "rope_half_48_at_8": spec("pf_r48", 30, H=2, G=2, d=64, seqs=((90, 40),), m=8, base=1e4, rot_dim=48,
                              rot_offset=8),
    "rope_interleaved_40_at_8": spec("pf_i40", 30, H=1, G=4, d=128, seqs=((100,),), m=16, base=1e4, rot_dim=40,
                                     rot_offset=8, pairing=K.INTERLEAVED),
    # two 1296-token chunks: 41 tiles, several laps of the tile ring, lazy rescales
    "long_chunks": spec("pf_long", 64, H=1, G=4, d=128, seqs=((1296, 1296),), m=32),
    "one_token": spec("pf_t1", 1, H=2, G=2, d=128, seqs=((100,), (5,)), m=16),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_parity(name):
    a = W.make_attend(CASES[name], DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_prefill(a, err=err)
    assert int(err.item()) == 0
    check(a, out, lse, name)


def test_prefill_without_lse():
    a = W.make_attend(CASES["qwen_gqa"], DEV)
    out, lse = run_prefill(a, lse=False)
    assert lse is None
    check(a, out, None, "no lse")


def test_prefill_large_scores_rescale():
    """Queries scaled up so the running max grows by far more than the lazy
    threshold from tile to tile: every rescale path of O (and of the value
    patch accumulator inside a chunk) runs."""
    a = W.make_attend(spec("pf_big", 24, H=2, G=4, d=128, seqs=((300, 200),), m=16), DEV)
    a.q = (a.q.float() * 6.0).to(torch.bfloat16)
    out, lse = run_prefill(a)
    check(a, out, lse, "large scores")


def test_prefill_empty_sequences():
    """A sequence without chunks and one whose only chunk has no token: zeros
    and lse = -inf."""
    a = W.make_attend(spec("pf_empty", 9, H=2, G=2, d=64, seqs=((40,), (), (0,)), m=8), DEV)
    out, lse = run_prefill(a)
    assert torch.count_nonzero(out[1:]).item() == 0
    assert bool(torch.all(lse[1:] == -float("inf")))
    check(a, out, lse, "empty")


def test_prefill_matches_decode_per_token():
    """Each query token of a prefill gets what the decode kernel gives that
    token alone (both within the same bound of the oracle)."""
    a = W.make_attend(CASES["qwen_gqa"], DEV)
    out, _ = run_prefill(a)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    rope = K.Rope(a.spec.base, a.rot_dim, a.spec.rot_offset, a.spec.pairing)
    for t in (0, 7, a.spec.T - 1):
        dec = K.kamera_attend_reused(a.store_k, a.store_v, a.q[:, t].contiguous(), rope, chunks, seq,
                                     len(a.chunks), 300, a.spec.m, layer=a.spec.layer)
        torch.cuda.synchronize()
        diff = (dec.float() - out[:, t].float()).abs()
        ulp = torch.from_numpy(_ulp_bf16(dec.float().cpu().numpy().astype(np.float64))).to(DEV)
        assert bool(torch.all(diff <= 2 * ulp + 1e-3 * dec.float().abs().amax())), t


def test_prefill_device_errors():
    a = W.make_attend(spec("pf_err", 5, H=2, G=2, d=64, seqs=((40,), (30,)), m=8), DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_prefill(a, err=err, seq_start=[0, 2, 1])   # second sequence's range runs backwards
    assert int(err.item()) & 4
    a.chunks[1].src_offset = 10 ** 6              # source rows past the store
    err.zero_()
    out, lse = run_prefill(a, err=err)
    assert int(err.item()) & 2
    assert torch.count_nonzero(out[1]).item() == 0
    assert bool(torch.all(lse[1] == -float("inf")))


def test_prefill_host_errors():
    a = W.make_attend(spec("pf_host", 3, H=2, G=3, d=96, seqs=((10,),), m=8), DEV)
    with pytest.raises(K.KameraError) as e:        # head_dim 96 is not handled
        run_prefill(a)
    assert e.value.status == 3
    a = W.make_attend(spec("pf_host2", 3, H=2, G=3, d=64, seqs=((10,),), m=8), DEV)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    rope = K.Rope(a.spec.base, a.rot_dim)
    with pytest.raises(K.KameraError) as e:        # max_rank above 64
        K.kamera_prefill_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, 1, 10, 65)
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:        # out overlapping q
        K.kamera_prefill_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, 1, 10, 8, out=a.q)
    assert e.value.status == 1


def test_prefill_timeout_expiry():
    """The producer withholds every tile load (test hook) under a 1 ms bound:
    the MMA warp's first wait runs out, the call returns with TIMEOUT set, and
    the next call on the same device (a fresh process state is not needed)
    still matches the oracle, so TMEM was freed and nothing is left in flight."""
    code = textwrap.dedent("""
        import os, sys, torch
        sys.path.insert(0, os.getcwd())
        import workloads as W
        from tests import test_gpu_prefill as T
        a = W.make_attend(T.CASES["qwen_gqa"], "cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        os.environ["KAMERA_WAIT_LIMIT_NS"] = "1000000"
        os.environ["KAMERA_TEST_WITHHOLD_LOADS"] = "1"
        T.run_prefill(a, err=err)
        assert int(err.item()) & 32, int(err.item())
        del os.environ["KAMERA_WAIT_LIMIT_NS"], os.environ["KAMERA_TEST_WITHHOLD_LOADS"]
        err.zero_()
        out, lse = T.run_prefill(a, err=err)
        assert int(err.item()) == 0
        T.check(a, out, lse, "after timeout")
        print("ok")
    """)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_prefill_fullsize_sampled():
    """The bench's workload (38 sequences of 8 x 1296 reused tokens, 256 new
    query tokens, Qwen2.5-VL-7B heads) in the launch the bench times: every
    query row of the last sequence against the oracle, every row of the rest
    finite, and the lse of every row at least the largest score's lower bound
    log(1) (so no row lost its softmax state)."""
    a = W.make_attend(W.qwen_prefill_reused(), DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_prefill(a, err=err)
    assert int(err.item()) == 0
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
    check(a, out, lse, "qwen_prefill_reused, last sequence", seqs=[len(a.seq_start) - 2])
