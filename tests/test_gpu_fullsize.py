"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (same entry point, descriptors, max_len and max_rank as the benchmark
call).

Every output row of the Qwen2.5-VL recall batch, the DeepSeek-V2-Lite MLA
batch, the sliding-window survival and the tiny chunk x 4096 is compared with
the fp64 oracle, layer by layer (``harness.check_layers``: the layer's inputs
copied to the host after the one GPU call, the oracle run on them, every
targeted slot compared element by element with the per-(layer, head)
Frobenius bound, every other slot checked for its bytes).  The MHA
reorder + recall batch (107 GB moved) is compared the same way on its first
and last layers, and on a seeded sample of rows of every layer.  Each case
records the count of elements beyond 1 ulp (all of them cancellation
within the scale-relative bound) in the session summary.
"""
import numpy as np
import pytest
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_SAMPLES = 96     # sampled (chunk, layer) groups
TOK_PER = 3        # sampled tokens per group


def _targeted_mask(wl):
    mask = torch.zeros(wl.num_slots, dtype=torch.bool, device=DEV)
    for c in wl.chunks:
        mask[c.slots] = True
    return mask


def _samples(wl, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(N_SAMPLES):
        ci = int(rng.integers(len(wl.chunks)))
        c = wl.chunks[ci]
        l = int(rng.integers(wl.spec.L))
        toks = sorted(set(int(t) for t in rng.integers(0, c.length, TOK_PER)))
        out.append((ci, l, toks))
    return out


def _u16(t):
    return Hn.u16(t)


def _check_rows(got, want, scale, what):
    return Hn.compare(np.stack(got), np.stack(want), np.stack(scale), block_axes=(1,), what=what)


FULL = {
    "qwen_recall": W.qwen_recall,
    "dsv2_mla": W.dsv2_mla,
    "qwen_slide": W.qwen_slide,
    "tiny_gqa_x4096": lambda: W.tiny_gqa_x(4096),
    "mha_reorder_recall": W.mha_reorder_recall,
}
PARTIAL_LAYERS = {"mha_reorder_recall": (0, 31)}   # every row of these layers; the rest sampled below


@pytest.mark.parametrize("name", list(FULL))
def test_fullsize_every_row(name):
    spec = FULL[name]()
    wl = W.make(spec, DEV)
    before = wl.pool_k.clone() if wl.kind == "slide" else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    layers = PARTIAL_LAYERS.get(name, range(spec.L))
    workers = 2 if name == "mha_reorder_recall" else 8
    st = Hn.check_layers(wl, layers, name, pool_before=before, workers=workers)
    which = "every row" if name not in PARTIAL_LAYERS else f"every row of layers {list(layers)}"
    for tag, s in st.items():
        Hn.report(f"{name} {tag} (full size, {which})", s)
    assert sum(s.n for s in st.values()) > 0


def test_mha_fullsize_sampled():
    """The MHA reorder + recall batch's layers not compared whole above: a
    seeded sample of rows of every layer, from the same kind of call."""
    name = "mha_reorder_recall"
    spec = W.CONFIGS[name]()
    wl = W.make(spec, DEV)
    orc = O.default()
    th = orc.inv_freq(wl.base, wl.rot_dim)
    samples = _samples(wl, 11)
    snap = []
    for ci, l, toks in samples:   # host copies of every input the sampled rows need
        c = wl.chunks[ci]
        rows = torch.tensor([c.src_offset + j for j in toks], device=DEV)
        item = {"k": _u16(wl.store_k[l, rows]), "v": _u16(wl.store_v[l, rows]),
                "slots": c.slots[toks].cpu().numpy()}
        if c.rank:
            item["uk"] = _u16(c.patches[0][l][:, toks])
            item["vk"] = _u16(c.patches[1][l])
            item["uv"] = _u16(c.patches[2][l][:, toks])
            item["vv"] = _u16(c.patches[3][l])
        snap.append(item)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H = wl.spec.H
    gk, wk, sk, gv, wv, sv = [], [], [], [], [], []
    for (ci, l, toks), item in zip(samples, snap):
        c = wl.chunks[ci]
        pk = _u16(wl.pool_k[l, torch.as_tensor(item["slots"], device=DEV)])
        pv = _u16(wl.pool_v[l, torch.as_tensor(item["slots"], device=DEV)])
        for a in range(len(toks)):
            for h in range(H):
                kw = dict(u=item["uk"][h, a], vm=item["vk"][h]) if c.rank else {}
                vw = dict(u=item["uv"][h, a], vm=item["vv"][h]) if c.rank else {}
                b, _, s = orc.row(item["k"][a, h], True, c.delta, th, wl.rot_dim, wl.rot_offset, wl.pairing, **kw)
                gk.append(pk[a, h]); wk.append(b); sk.append(s)
                b, _, s = orc.row(item["v"][a, h], False, 0, th, wl.rot_dim, wl.rot_offset, wl.pairing, **vw)
                gv.append(pv[a, h]); wv.append(b); sv.append(s)
    Hn.report(f"{name} K (full size, sampled rows of every layer)", _check_rows(gk, wk, sk, f"{name} K (sampled)"))
    Hn.report(f"{name} V (full size, sampled rows of every layer)", _check_rows(gv, wv, sv, f"{name} V (sampled)"))
    untouched = ~_targeted_mask(wl)
    canary = torch.tensor(W.CANARY_BITS - 0x10000 if W.CANARY_BITS >= 0x8000 else W.CANARY_BITS,
                          dtype=torch.int16, device=DEV)
    for pool in (wl.pool_k, wl.pool_v):
        assert bool((pool.view(torch.int16)[:, untouched] == canary).all()), f"{name}: untouched slots changed"


# ----------------------------------------------------- the NEXT rows, full size
def test_patch_form_fullsize_every_block():
    """qwen_patch_form as bench.py times it (224 blocks of 1296 x 128, rank 32, one
    call): every block against the oracle's truncated SVD."""
    from tests.test_gpu_patchform import check_factors
    spec = W.qwen_patch_form()
    x = W.make_deficit(spec, DEV)
    xb = x.reshape(spec.kv * spec.L, spec.length, spec.H, spec.d).permute(0, 2, 1, 3)
    sig = torch.empty(spec.kv * spec.L, spec.H, spec.m, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    u, v = K.kamera_form_patch(xb, spec.m, sigma=sig, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    vt = v.float()
    gram = torch.einsum("oicm,oicn->oimn", vt, vt)
    assert float((gram - torch.eye(spec.m, device=DEV)).abs().max()) <= 8e-3
    xh = xb.float().cpu().numpy().astype(np.float64)
    uh, vh = u.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64)
    sh = sig.cpu().numpy().astype(np.float64)
    for o in range(spec.kv * spec.L):
        for i in range(spec.H):
            check_factors(xh[o, i], uh[o, i], vh[o, i], sh[o, i], spec.m, f"block ({o},{i})")


@pytest.mark.parametrize("name", ["dsv2_patch_form", "dsv2_joint_patch_form"])
def test_wide_patch_form_fullsize_every_block(name):
    """dsv2_patch_form and dsv2_joint_patch_form as bench.py times them (27
    blocks of 4096 x 512, or x 576 for the joint latent-row factor, rank 16: the
    wide path, one call): every block against the oracle's truncated SVD."""
    from tests.test_gpu_patchform import check_factors
    spec = W.FORMATION[name]()
    x = W.make_deficit(spec, DEV)
    xb = x.reshape(spec.kv * spec.L, spec.length, spec.H, spec.d).permute(0, 2, 1, 3)
    sig = torch.empty(spec.kv * spec.L, spec.H, spec.m, dtype=torch.float32, device=DEV)
    u, v = K.kamera_form_patch(xb, spec.m, sigma=sig)
    torch.cuda.synchronize()
    for o in range(spec.kv * spec.L):
        blk = xb[o, 0].float().cpu().numpy().astype(np.float64)
        check_factors(blk, u[o, 0].float().cpu().numpy().astype(np.float64),
                      v[o, 0].float().cpu().numpy().astype(np.float64),
                      sig[o, 0].cpu().numpy().astype(np.float64), spec.m, f"block {o}")


def test_attend_fullsize_every_sequence():
    """qwen_attend_reused as bench.py times it (38 sequences x 8 chunks of 1296
    tokens, one call): every sequence against the oracle."""
    from tests.test_gpu_attend import _bits, _ulp_bf16
    spec = W.qwen_attend_reused()
    a = W.make_attend(spec, DEV)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = K.kamera_attend_reused(a.store_k, a.store_v, a.q, K.Rope(spec.base, spec.d), chunks, seq, len(a.chunks),
                                 max(c.length for c in a.chunks), spec.m, layer=spec.layer, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    orc = O.default()
    th = orc.inv_freq(spec.base, spec.d)
    for s in range(len(spec.seqs)):
        cs = a.chunks[a.seq_start[s]:a.seq_start[s + 1]]
        lo, hi = cs[0].src_offset, cs[-1].src_offset + cs[-1].length
        oc = [O.Chunk(c.src_offset - lo, c.length, c.delta, c.rank, c.slots.cpu().numpy(),
                      [_bits(t) for t in c.patches]) for c in cs]
        _, ref, mag = orc.attend(_bits(a.store_k[lo:hi]), _bits(a.store_v[lo:hi]), oc, [0, len(cs)],
                                 _bits(a.q[s:s + 1]), spec.layer, th, spec.d, scale=spec.d ** -0.5)
        got = out[s:s + 1].float().cpu().numpy().astype(np.float64)
        bad = np.abs(got - ref) > _ulp_bf16(ref) + 2.0 ** -16 * mag
        assert not bad.any(), (s, int(bad.sum()))


def test_mla_attend_fullsize_every_sequence():
    """dsv2_attend_reused as bench.py times it (38 sequences x 4 chunks of 4096
    tokens, one call, the cluster split it launches with): every sequence against
    the oracle."""
    from tests.test_gpu_attend_mla import _bits, _ulp_bf16
    spec = W.dsv2_attend_reused()
    a = W.make_mla_attend(spec, DEV)
    chunks = K.pack_chunks(a.chunks, device=DEV)
    seq = torch.tensor(a.seq_start, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = K.kamera_mla_attend_reused(a.store, spec.kv_lora, a.q, K.Rope(spec.base, spec.rope, 0, spec.pairing), chunks,
                                     seq, len(a.chunks), max(c.length for c in a.chunks), spec.m, layer=spec.layer,
                                     err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    orc = O.default()
    th = orc.inv_freq(spec.base, spec.rope)
    Wd = spec.kv_lora + spec.rope
    for s in range(len(spec.seqs)):
        cs = a.chunks[a.seq_start[s]:a.seq_start[s + 1]]
        lo, hi = cs[0].src_offset, cs[-1].src_offset + cs[-1].length
        oc = [O.Chunk(c.src_offset - lo, c.length, c.delta, c.rank, c.slots.cpu().numpy(),
                      [_bits(t) for t in c.patches]) for c in cs]
        _, ref, mag = orc.attend_mla(_bits(a.store[lo:hi]), oc, [0, len(cs)], _bits(a.q[s:s + 1]), spec.layer,
                                     spec.kv_lora, th, spec.rope, 0, spec.pairing, scale=Wd ** -0.5)
        got = out[s:s + 1].float().cpu().numpy().astype(np.float64)
        bad = np.abs(got - ref) > _ulp_bf16(ref) + 2.0 ** -16 * mag
        assert not bad.any(), (s, int(bad.sum()))
