"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (same entry point, max_len and max_rank as the benchmark call).

The fp64 oracle cannot compute whole workloads of 1-100 GB in a test, so it
computes a seeded sample of output rows one by one (``oracle.row`` on the
sampled canonical rows and patch factors, copied to the host before the
call), and properties that hold at any size are checked on the whole pool:
every slot no chunk targets keeps its canary bits, and no device error bit
is raised.
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
    Hn.compare(np.stack(got), np.stack(want), np.stack(scale), what=what)


@pytest.mark.parametrize("name", ["qwen_recall", "mha_reorder_recall", "tiny_gqa_x4096"])
def test_gqa_fullsize_sampled(name):
    spec = W.tiny_gqa_x(4096) if name == "tiny_gqa_x4096" else W.CONFIGS[name]()
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
    _check_rows(gk, wk, sk, f"{name} K (sampled)")
    _check_rows(gv, wv, sv, f"{name} V (sampled)")
    untouched = ~_targeted_mask(wl)
    canary = torch.tensor(W.CANARY_BITS - 0x10000 if W.CANARY_BITS >= 0x8000 else W.CANARY_BITS,
                          dtype=torch.int16, device=DEV)
    for pool in (wl.pool_k, wl.pool_v):
        assert bool((pool.view(torch.int16)[:, untouched] == canary).all()), f"{name}: untouched slots changed"


def test_mla_fullsize_sampled():
    wl = W.make(W.dsv2_mla(), DEV)
    orc = O.default()
    th = orc.inv_freq(wl.base, wl.rot_dim)
    kv = wl.kv_lora
    samples = _samples(wl, 12)
    snap = []
    for ci, l, toks in samples:
        c = wl.chunks[ci]
        rows = torch.tensor([c.src_offset + j for j in toks], device=DEV)
        snap.append({"x": _u16(wl.store_k[l, rows]), "slots": c.slots[toks].cpu().numpy(),
                     "uc": _u16(c.patches[0][l][toks]), "vc": _u16(c.patches[1][l]),
                     "ur": _u16(c.patches[2][l][toks]), "vr": _u16(c.patches[3][l])})
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    gc, wc, sc, gr, wr, sr = [], [], [], [], [], []
    for (ci, l, toks), item in zip(samples, snap):
        c = wl.chunks[ci]
        pool = _u16(wl.pool_k[l, torch.as_tensor(item["slots"], device=DEV)])
        for a in range(len(toks)):
            b, _, s = orc.row(item["x"][a, :kv], False, 0, th, wl.rot_dim, 0, wl.pairing, u=item["uc"][a], vm=item["vc"])
            gc.append(pool[a, :kv]); wc.append(b); sc.append(s)
            b, _, s = orc.row(item["x"][a, kv:], True, c.delta, th, wl.rot_dim, 0, wl.pairing, u=item["ur"][a],
                              vm=item["vr"])
            gr.append(pool[a, kv:]); wr.append(b); sr.append(s)
    _check_rows(gc, wc, sc, "dsv2_mla c_KV (sampled)")
    _check_rows(gr, wr, sr, "dsv2_mla k_rope (sampled)")
    untouched = ~_targeted_mask(wl)
    canary = torch.tensor(W.CANARY_BITS, dtype=torch.int16, device=DEV)
    assert bool((wl.pool_k.view(torch.int16)[:, untouched] == canary).all())


def test_slide_fullsize_sampled():
    wl = W.make(W.qwen_slide(), DEV)
    orc = O.default()
    th = orc.inv_freq(wl.base, wl.rot_dim)
    samples = _samples(wl, 13)
    before = []
    for ci, l, toks in samples:
        c = wl.chunks[ci]
        before.append(_u16(wl.pool_k[l, c.slots[toks]]))
    targeted = _targeted_mask(wl)
    # a sample of evicted (untouched) slots, copied before the call
    ev = torch.nonzero(~targeted).flatten()
    ev = ev[torch.randperm(ev.numel(), generator=torch.Generator().manual_seed(3))[:4096].to(DEV)]
    ev_before = _u16(wl.pool_k[:, ev])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got, want, scale = [], [], []
    for (ci, l, toks), x in zip(samples, before):
        c = wl.chunks[ci]
        after = _u16(wl.pool_k[l, c.slots[toks]])
        for a in range(len(toks)):
            for h in range(wl.spec.H):
                b, _, s = orc.row(x[a, h], True, c.delta, th, wl.rot_dim, wl.rot_offset, wl.pairing)
                got.append(after[a, h]); want.append(b); scale.append(s)
    _check_rows(got, want, scale, "qwen_slide (sampled)")
    assert np.array_equal(_u16(wl.pool_k[:, ev]), ev_before), "evicted slots changed"


# ----------------------------------------------------- the NEXT rows, full size
def test_patch_form_fullsize_sampled():
    """qwen_patch_form as bench.py times it (224 blocks of 1296 x 128, rank 32, one
    call): a seeded sample of blocks against the oracle's truncated SVD, the rest
    checked for V^T V = I."""
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
    rng = np.random.default_rng(21)
    for _ in range(12):
        o, i = int(rng.integers(spec.kv * spec.L)), int(rng.integers(spec.H))
        blk = xb[o, i].float().cpu().numpy().astype(np.float64)
        check_factors(blk, u[o, i].float().cpu().numpy().astype(np.float64),
                      v[o, i].float().cpu().numpy().astype(np.float64),
                      sig[o, i].cpu().numpy().astype(np.float64), spec.m, f"block ({o},{i})")


def test_wide_patch_form_fullsize_sampled():
    """dsv2_patch_form (27 blocks of 4096 x 512, rank 16: the wide path), sampled blocks."""
    from tests.test_gpu_patchform import check_factors
    spec = W.dsv2_patch_form()
    x = W.make_deficit(spec, DEV)
    xb = x.reshape(spec.kv * spec.L, spec.length, spec.H, spec.d).permute(0, 2, 1, 3)
    sig = torch.empty(spec.kv * spec.L, spec.H, spec.m, dtype=torch.float32, device=DEV)
    u, v = K.kamera_form_patch(xb, spec.m, sigma=sig)
    torch.cuda.synchronize()
    for o in (0, 13, 26):
        blk = xb[o, 0].float().cpu().numpy().astype(np.float64)
        check_factors(blk, u[o, 0].float().cpu().numpy().astype(np.float64),
                      v[o, 0].float().cpu().numpy().astype(np.float64),
                      sig[o, 0].cpu().numpy().astype(np.float64), spec.m, f"block {o}")


def test_attend_fullsize_sampled():
    """qwen_attend_reused as bench.py times it (38 sequences x 8 chunks of 1296
    tokens, one call): a seeded sample of sequences against the oracle."""
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
    rng = np.random.default_rng(22)
    for s in sorted(set(int(x) for x in rng.integers(0, len(spec.seqs), 3))):
        cs = a.chunks[a.seq_start[s]:a.seq_start[s + 1]]
        lo, hi = cs[0].src_offset, cs[-1].src_offset + cs[-1].length
        oc = [O.Chunk(c.src_offset - lo, c.length, c.delta, c.rank, c.slots.cpu().numpy(),
                      [_bits(t) for t in c.patches]) for c in cs]
        _, ref, mag = orc.attend(_bits(a.store_k[lo:hi]), _bits(a.store_v[lo:hi]), oc, [0, len(cs)],
                                 _bits(a.q[s:s + 1]), spec.layer, th, spec.d, scale=spec.d ** -0.5)
        got = out[s:s + 1].float().cpu().numpy().astype(np.float64)
        bad = np.abs(got - ref) > _ulp_bf16(ref) + 2.0 ** -16 * mag
        assert not bad.any(), (s, int(bad.sum()))


def test_mla_attend_fullsize_sampled():
    """dsv2_attend_reused as bench.py times it (38 sequences x 4 chunks of 4096
    tokens, one call, the cluster split it launches with): a seeded sample of
    sequences against the oracle."""
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
    rng = np.random.default_rng(23)
    for s in sorted(set(int(x) for x in rng.integers(0, len(spec.seqs), 2))):
        cs = a.chunks[a.seq_start[s]:a.seq_start[s + 1]]
        lo, hi = cs[0].src_offset, cs[-1].src_offset + cs[-1].length
        oc = [O.Chunk(c.src_offset - lo, c.length, c.delta, c.rank, c.slots.cpu().numpy(),
                      [_bits(t) for t in c.patches]) for c in cs]
        _, ref, mag = orc.attend_mla(_bits(a.store[lo:hi]), oc, [0, len(cs)], _bits(a.q[s:s + 1]), spec.layer,
                                     spec.kv_lora, th, spec.rope, 0, spec.pairing, scale=Wd ** -0.5)
        got = out[s:s + 1].float().cpu().numpy().astype(np.float64)
        bad = np.abs(got - ref) > _ulp_bf16(ref) + 2.0 ** -16 * mag
        assert not bad.any(), (s, int(bad.sum()))
