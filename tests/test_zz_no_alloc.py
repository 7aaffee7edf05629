"""kamera_attend_reused_static -- decode attention for callers that cannot
allocate device memory -- against the ordinary entry point.

Such a caller (a plug-in inside a process whose device memory belongs to
another allocator, or a serving loop that may not call cudaMalloc while it
runs) passes only its inputs and outputs; the library supplies the workspace
from a fixed scratch array of its own.  The test calls the new entry point
through the C ABI twice in a row (the second call finds the scratch holding
the first call's partial states) and compares each output with the ordinary
entry point's, element by element, to one bf16 ulp: the tolerance the
attention tests allow against the oracle, here between two runs of the same
kernels."""
import numpy as np
import pytest
import torch

import position_invariant_kv_chunk_gb300 as K
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def test_static_scratch_matches_the_ordinary_entry_point():
    spec = W.AttendSpec("noalloc", H=4, G=7, d=128, seqs=((300, 129), (64,), (200, 1, 77)), m=32)
    a = W.make_attend(spec, DEV)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing)
    max_len = max(c.length for c in a.chunks)
    max_rank = max(c.rank for c in a.chunks)
    ref = K.kamera_attend_reused(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), max_len, max_rank,
                                 layer=spec.layer)
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(a.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        K.kamera_attend_reused_static(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), max_len,
                                      max_rank, out, layer=spec.layer, err=err)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        assert int(err.item()) == 0
        assert np.isfinite(got).all(), f"call {call}: unwritten outputs"
        bad = np.abs(got - want) > _ulp_bf16(want)
        assert not bad.any(), (call, int(bad.sum()))


def test_static_scratch_refuses_batches_it_cannot_hold():
    """A batch whose partial states exceed the fixed scratch gets
    KAMERA_ERR_UNSUPPORTED before anything is launched."""
    spec = W.AttendSpec("noalloc_big", H=8, G=1, d=128, seqs=((4,),) * 64, m=0)
    a = W.make_attend(spec, DEV)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    rope = K.Rope(spec.base, a.rot_dim, spec.rot_offset, spec.pairing)
    out = torch.empty_like(a.q)
    with pytest.raises(K.KameraError) as e:
        K.kamera_attend_reused_static(a.store_k, a.store_v, a.q, rope, chunks, seq, len(a.chunks), 4, 0, out,
                                      layer=spec.layer)
    assert e.value.status == 3
