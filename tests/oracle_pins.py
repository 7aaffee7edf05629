"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch.  ``test_oracle_pins.py`` runs them against the oracle as built;
``test_oracle_mutants.py`` runs them against copies of the oracle with planted
mistakes (a flipped sign, a wrong pair index, a transposed factor, a dropped
term, a wrong rounding step) and requires every mutant to fail at least one.

What they pin against (never the oracle's own formula retyped):
  * closed forms: theta_0 = 1, theta_{r/4} = base^-1/2, theta_i theta_{r/2-i} = 1/base,
    a quarter turn per position maps (a, b) -> (-b, a);
  * group laws of R: R(d1) R(d2) = R(d1 + d2), R(d) R(-d) = I, per-pair norms;
  * independent formulations: complex multiplication (x_a + i x_b) e^{i phi},
    the concatenated cos/sin-table RoPE used by common model code, the relative
    position property <R(p) q, R(p') k> = <R(p - p') q, k>;
  * library routines: numpy matmul / einsum for the patch, torch's fp32 -> bf16
    conversion, numpy eigh for singular values;
  * brute force: nearest bf16 by search over every finite bf16 value;
  * bit-exact copies (delta = 0, rank 0; MLA c_KV with rank 0) and canary slots.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import workloads as W

RH, IL = O.ROTATE_HALF, O.INTERLEAVED


# ------------------------------------------------------------------ helpers
def _all_finite_bf16():
    bits = np.arange(0x10000, dtype=np.uint32)
    f32 = (bits << 16).astype(np.uint32).view(np.float32)
    keep = np.isfinite(f32)
    f = np.where(keep, f32, 0).astype(np.float64)
    return bits[keep].astype(np.uint16), f[keep]


_TABLE = None


def _bf16_table():
    global _TABLE
    if _TABLE is None:
        bits, vals = _all_finite_bf16()
        order = np.lexsort((bits, vals))        # by value; -0 before +0
        _TABLE = (bits[order], vals[order])
    return _TABLE


def brute_bf16(x: float) -> int:
    """Nearest finite bf16 to x by exhaustive search; ties to the even pattern;
    beyond the largest finite value by half an ulp or more: infinity."""
    if math.isnan(x):
        raise ValueError("nan")
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    bits, vals = _bf16_table()
    if abs(x) >= float(vals.max()) + 2.0 ** (127 - 8):
        return 0xFF80 if x < 0 else 0x7F80
    same_sign = (bits >= 0x8000) == (x < 0)     # a tiny x rounds to the zero of its sign
    bits, vals = bits[same_sign], vals[same_sign]
    err = np.abs(vals - x)
    cand = [int(c) for c in bits[err == err.min()]]
    even = [c for c in cand if c & 1 == 0]
    return even[0] if even else cand[0]


def complex_rotate(x, delta, theta, rot_dim, rot_offset, pairing):
    """R(delta) by complex multiplication, vectorised over leading dims."""
    x = np.array(x, dtype=np.float64, copy=True)
    o, r = rot_offset, rot_dim
    if pairing == RH:
        z = x[..., o:o + r // 2] + 1j * x[..., o + r // 2:o + r]
    else:
        z = x[..., o:o + r:2] + 1j * x[..., o + 1:o + r:2]
    z = z * np.exp(1j * (float(delta) * theta))
    if pairing == RH:
        x[..., o:o + r // 2] = z.real
        x[..., o + r // 2:o + r] = z.imag
    else:
        x[..., o:o + r:2] = z.real
        x[..., o + 1:o + r:2] = z.imag
    return x


def table_rope(x, pos, theta, pairing):
    """RoPE at position ``pos`` the way common model code writes it: x*cos + rot(x)*sin
    with a cos/sin table over the whole head (rotate-half: [freqs, freqs];
    interleaved: each frequency repeated twice)."""
    x = np.asarray(x, dtype=np.float64)
    ang = pos * theta
    if pairing == RH:
        emb = np.concatenate([ang, ang])
        h = x.shape[-1] // 2
        rot = np.concatenate([-x[..., h:], x[..., :h]], axis=-1)
    else:
        emb = np.repeat(ang, 2)
        rot = np.empty_like(x)
        rot[..., 0::2] = -x[..., 1::2]
        rot[..., 1::2] = x[..., 0::2]
    return x * np.cos(emb) + rot * np.sin(emb)


def rand_bf16(rng, shape, std=1.0):
    f = (rng.standard_normal(shape) * std).astype(np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------- bf16
def pin_bf16_bruteforce(orc: O.Oracle):
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-40, 38, 300))
    xs += list(rng.standard_normal(100) * 1e-39)           # bf16 subnormal range
    xs += [3.3895313892515355e38, 3.40e38, -3.39e38, 1e-45, 0.0, -0.0, 1.0, -1.0]
    got = orc.bf16_rne(np.array(xs))
    for x, g in zip(xs, got):
        assert int(g) == brute_bf16(float(x)), (x, hex(int(g)), hex(brute_bf16(float(x))))


def pin_bf16_ties(orc: O.Oracle):
    bits, vals = _bf16_table()
    pos = vals > 0
    b, v = bits[pos], vals[pos]
    idx = np.random.default_rng(2).integers(0, len(v) - 1, 400)
    mids = (v[idx] + v[idx + 1]) / 2            # exact in fp64
    got = orc.bf16_rne(mids)
    for i, m, g in zip(idx, mids, got):
        lo, hi = int(b[i]), int(b[i + 1])
        want = lo if lo % 2 == 0 else hi
        assert int(g) == want, (m, hex(int(g)), hex(want))
    got_neg = orc.bf16_rne(-mids)
    assert np.all(got_neg == (got | 0x8000))


def pin_bf16_vs_torch(orc: O.Oracle):
    rng = np.random.default_rng(3)
    f32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    want = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_rne(f32.astype(np.float64))
    assert np.array_equal(got, want)


def pin_bf16_specials(orc: O.Oracle):
    mid = 2.0 ** 128 - 2.0 ** 119     # halfway between the largest bf16 and 2^128
    got = orc.bf16_rne(np.array([np.inf, -np.inf, 0.0, -0.0, mid, np.nextafter(mid, 0.0), 1e39]))
    # the tie goes to the even neighbour, which is the overflow (infinity)
    assert list(got[:4]) == [0x7F80, 0xFF80, 0x0000, 0x8000]
    assert got[4] == 0x7F80 and got[6] == 0x7F80
    assert got[5] == 0x7F7F
    assert orc.bf16_rne(np.array([np.nan]))[0] & 0x7F80 == 0x7F80
    allbits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    f = orc.bf16_to_f64(allbits)
    want = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(want)
    assert np.array_equal(f[fin], want[fin])
    assert np.array_equal(np.signbit(f[fin]), np.signbit(want[fin]))
    assert np.array_equal(orc.bf16_rne(f[fin]), allbits[fin])


# ------------------------------------------------------------------- theta
def pin_inv_freq_closed_forms(orc: O.Oracle):
    for base, r, quarter in ((1e4, 64, 0.01), (1e4, 128, 0.01), (1e6, 128, 0.001),
                             (1e6, 64, 0.001), (1e4, 16, 0.01)):
        th = orc.inv_freq(base, r)
        assert th.shape == (r // 2,)
        assert th[0] == 1.0
        assert abs(th[r // 4] - quarter) <= 1e-15 * quarter
        for i in range(1, r // 2):
            assert abs(th[i] * th[r // 2 - i] - 1.0 / base) <= 1e-14 / base
        assert np.all(np.diff(th) < 0)


# ---------------------------------------------------------------- rotation
def pin_rotation_quarter_turn(orc: O.Oracle):
    """theta = pi/2 for every pair: one position turns (a, b) into (-b, a)."""
    rng = np.random.default_rng(4)
    for pairing in (RH, IL):
        for (width, r, o) in ((64, 64, 0), (96, 32, 16), (576, 64, 512)):
            x = rng.standard_normal(width)
            theta = np.full(r // 2, math.pi / 2)
            if pairing == RH:
                a = np.arange(o, o + r // 2)
                b = a + r // 2
            else:
                a = np.arange(o, o + r, 2)
                b = a + 1
            rest = np.setdiff1d(np.arange(width), np.concatenate([a, b]))
            for delta, fa, fb in ((1, lambda xa, xb: -xb, lambda xa, xb: xa),
                                  (2, lambda xa, xb: -xa, lambda xa, xb: -xb),
                                  (-1, lambda xa, xb: xb, lambda xa, xb: -xa),
                                  (4, lambda xa, xb: xa, lambda xa, xb: xb)):
                y = orc.rotate(x, delta, theta, r, o, pairing)
                assert np.allclose(y[a], fa(x[a], x[b]), atol=1e-14, rtol=0), (pairing, delta)
                assert np.allclose(y[b], fb(x[a], x[b]), atol=1e-14, rtol=0), (pairing, delta)
                assert np.array_equal(y[rest], x[rest])


def pin_rotation_group_laws(orc: O.Oracle):
    rng = np.random.default_rng(5)
    for pairing in (RH, IL):
        for base, r in ((1e4, 64), (1e6, 128)):
            th = orc.inv_freq(base, r)
            x = rng.standard_normal((3, r))
            for _ in range(6):
                d1, d2 = (int(v) for v in rng.integers(-32768, 32769, 2))
                y12 = orc.rotate(orc.rotate(x, d2, th, r, 0, pairing), d1, th, r, 0, pairing)
                ys = orc.rotate(x, d1 + d2, th, r, 0, pairing)
                assert np.max(np.abs(y12 - ys)) < 1e-10
                back = orc.rotate(orc.rotate(x, d1, th, r, 0, pairing), -d1, th, r, 0, pairing)
                assert np.max(np.abs(back - x)) < 1e-12
                y = orc.rotate(x, d1, th, r, 0, pairing)
                if pairing == RH:
                    n0 = x[:, :r // 2] ** 2 + x[:, r // 2:] ** 2
                    n1 = y[:, :r // 2] ** 2 + y[:, r // 2:] ** 2
                else:
                    n0 = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
                    n1 = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
                assert np.max(np.abs(n0 - n1)) < 1e-12


def pin_rotation_complex(orc: O.Oracle):
    rng = np.random.default_rng(6)
    for pairing in (RH, IL):
        for (width, r, o, base) in ((128, 128, 0, 1e6), (64, 64, 0, 1e4), (576, 64, 512, 1e4),
                                    (128, 64, 32, 1e4)):
            th = orc.inv_freq(base, r)
            x = rng.standard_normal((4, width))
            for delta in (37, -32768, 32768, 1, -5, 123456):
                y = orc.rotate(x, delta, th, r, o, pairing)
                z = complex_rotate(x, delta, th, r, o, pairing)
                assert np.max(np.abs(y - z)) < 1e-12, (pairing, delta)


def pin_rotation_relocates_keys(orc: O.Oracle):
    """Keys made at position p (model-style RoPE table) equal R(p) applied to the
    same keys made at position 0; and q.k after RoPE depends only on p - p'."""
    rng = np.random.default_rng(7)
    for pairing in (RH, IL):
        for base, d in ((1e4, 64), (1e6, 128)):
            th = orc.inv_freq(base, d)
            W = rng.standard_normal((d, 32)) / 6
            h = rng.standard_normal((5, 32))
            k0 = h @ W.T                          # keys at position 0: RoPE(., 0) = identity
            for p in (0, 1, 37, 1000, 32767):
                kp = table_rope(k0, p, th, pairing)
                assert np.max(np.abs(orc.rotate(k0, p, th, d, 0, pairing) - kp)) < 1e-10
            q = rng.standard_normal(d)
            k = rng.standard_normal(d)
            for p, pp in ((10, 3), (5000, 4000), (-7, 20)):
                lhs = orc.rotate(q, p, th, d, 0, pairing) @ orc.rotate(k, pp, th, d, 0, pairing)
                rhs = orc.rotate(q, p - pp, th, d, 0, pairing) @ k
                assert abs(lhs - rhs) < 1e-10


# ------------------------------------------------------------------- patch
def pin_rotation_model_tables(orc: O.Oracle):
    """R(delta) with a model's own frequency table.  A context-extension table:
    keys made at position p with that table equal R(p) of the keys made at 0.
    Multi-axis RoPE (per-frequency positions: time, height, width sections):
    keys made at axis positions (t, h, w) and moved by (dt, dh, dw) equal
    R(dt) with each section's frequencies scaled by its axis's share of dt --
    the tables 'temporal' (dt, 0, 0) and 'axes' (dt, dt/2, dt/4) of the input
    generator."""
    rng = np.random.default_rng(21)
    for pairing in (RH, IL):
        for base, d in ((1e6, 128), (1e4, 64), (1e4, 16)):
            th = base ** (-2.0 * np.arange(d // 2) / d)
            k0 = rng.standard_normal((3, d))
            ext = W.model_inv_freq("extended", base, d)
            assert not np.allclose(ext, th) or d < 64
            for p in (1, 37, 4096, 32767, -900):
                assert np.max(np.abs(orc.rotate(k0, p, ext, d, 0, pairing) - table_rope(k0, p, ext, pairing))) < 1e-9
            axis = np.empty(d // 2, dtype=np.int64)
            for a, (lo, hi) in enumerate(W.mrope_sections(d // 2)):
                axis[lo:hi] = a
            start = np.array([40.0, 3.0, 11.0])   # a frame's (t, h, w) position
            kt = table_rope(k0, start[axis], th, pairing)
            for kind, move in (("temporal", lambda dt: (dt, 0, 0)), ("axes", lambda dt: (dt, dt // 2, dt // 4)),
                               ("standard", lambda dt: (dt, dt, dt))):
                tab = W.model_inv_freq(kind, base, d)
                for dt in (4, 1000, -40, 32764):
                    want = table_rope(k0, (start + np.array(move(dt), dtype=np.float64))[axis], th, pairing)
                    got = orc.rotate(kt, dt, tab, d, 0, pairing)
                    assert np.max(np.abs(got - want)) < 1e-8, (kind, dt, pairing, d)
            # independent per-axis moves, contiguous or interleaved sections: R(1)
            # over the table theta'_f = move[axis_f] * theta_f
            for layout in ("sections", "interleaved"):
                ax = W.freq_axes(d // 2, layout).astype(np.int64)
                kt = table_rope(k0, start[ax], th, pairing)
                for move in ((7, -3, 250), (0, 5, 0), (-30000, 12, 29999)):
                    mv = np.array(move, dtype=np.int64)
                    want = table_rope(k0, (start + mv)[ax], th, pairing)
                    got = orc.rotate(kt, 1, mv[ax].astype(np.float64) * th, d, 0, pairing)
                    assert np.max(np.abs(got - want)) < 1e-8, (layout, move, pairing, d)


def pin_row_patch_is_matmul(orc: O.Oracle):
    """delta = 0 reduces the row operator to x + U V^T (numpy matmul, fp64)."""
    rng = np.random.default_rng(8)
    for width, m in ((64, 4), (128, 32), (512, 16), (64, 1)):
        x = rand_bf16(rng, (width,))
        u = rand_bf16(rng, (m,), 0.05)
        vm = rand_bf16(rng, (width, m), 0.05)
        for rotate in (0, 1):
            b, f, sc = orc.row(x, rotate, 0, np.ones(width // 2), width, 0, RH, u, vm)
            want = to_f64(x) + to_f64(vm) @ to_f64(u)
            assert np.allclose(f, want, rtol=1e-14, atol=1e-15)
            assert np.array_equal(b, np.array([brute_bf16(v) for v in want], dtype=np.uint16))
            assert np.all(sc + 1e-15 >= np.abs(f))


def pin_row_rotate_plus_patch(orc: O.Oracle):
    rng = np.random.default_rng(9)
    for pairing in (RH, IL):
        for width, r, o, m, delta in ((128, 128, 0, 32, -23452), (576, 64, 512, 16, 1847),
                                      (64, 64, 0, 4, 37), (128, 64, 64, 8, 9)):
            th = orc.inv_freq(1e4, r)
            x = rand_bf16(rng, (width,))
            u = rand_bf16(rng, (m,), 0.05)
            vm = rand_bf16(rng, (width, m), 0.05)
            b, f, sc = orc.row(x, 1, delta, th, r, o, pairing, u, vm)
            want = complex_rotate(to_f64(x), delta, th, r, o, pairing) + to_f64(vm) @ to_f64(u)
            assert np.max(np.abs(f - want)) < 1e-12
            assert np.all(sc + 1e-12 >= np.abs(f))
            # value rows (rotate = 0) ignore delta
            b0, f0, _ = orc.row(x, 0, delta, th, r, o, pairing, u, vm)
            assert np.allclose(f0, to_f64(x) + to_f64(vm) @ to_f64(u), rtol=1e-14, atol=1e-15)


def pin_patch_frame_identity(orc: O.Oracle):
    """R(delta)(K + U V^T) = R(delta) K + U (R(delta) V)^T: the patch may be given in
    the canonical frame by rotating the columns of V_m."""
    rng = np.random.default_rng(10)
    for pairing in (RH, IL):
        d, T, m, delta = 64, 12, 5, -777
        th = orc.inv_freq(1e4, d)
        K = rng.standard_normal((T, d))
        U = rng.standard_normal((T, m))
        V = rng.standard_normal((d, m))
        lhs = orc.rotate(K + U @ V.T, delta, th, d, 0, pairing)
        RV = orc.rotate(V.T, delta, th, d, 0, pairing).T
        rhs = orc.rotate(K, delta, th, d, 0, pairing) + U @ RV.T
        assert np.max(np.abs(lhs - rhs)) < 1e-12


def pin_bit_exact_identity(orc: O.Oracle):
    """delta = 0 with no patch copies bits, signed zeros included."""
    x = np.array([0x8000, 0x0000, 0x3F80, 0xBF80, 0x0001, 0x8001, 0x7F7F, 0x1234] * 8,
                 dtype=np.uint16)
    for rotate in (0, 1):
        b, _, _ = orc.row(x, rotate, 0, np.ones(32), 64, 0, RH)
        assert np.array_equal(b, x)


# ------------------------------------------------------------ patch (SVD)
def pin_form_patch_full_rank(orc: O.Oracle):
    rng = np.random.default_rng(11)
    for T, d in ((32, 16), (16, 32), (20, 20)):
        D = rng.standard_normal((T, d))
        U, V = O.form_patch(D, min(T, d))
        assert np.max(np.abs(U @ V.T - D)) < 1e-12


def pin_eckart_young(orc: O.Oracle):
    rng = np.random.default_rng(12)
    for T, d in ((32, 16), (24, 12), (16, 16)):
        D = rng.standard_normal((T, d)) @ np.diag(np.geomspace(3, 0.01, d))
        # singular values by a different route: eigenvalues of D^T D
        ev = np.sort(np.linalg.eigh(D.T @ D)[0])[::-1]
        for m in (1, 4, 8):
            U, V = O.form_patch(D, m)
            assert np.allclose(V.T @ V, np.eye(m), atol=1e-12)
            resid = np.linalg.norm(D - U @ V.T) ** 2
            assert abs(resid - ev[m:].sum()) <= 1e-9 * max(1.0, ev.sum())
            for _ in range(30):
                A = rng.standard_normal((T, m))
                B = rng.standard_normal((d, m))
                P = (U + 0.05 * A) @ (V + 0.05 * B).T
                assert np.linalg.norm(D - P) ** 2 >= resid - 1e-12
                assert np.linalg.norm(D - A @ B.T) ** 2 >= resid


# ----------------------------------------------------------- whole problems
def _gqa_numpy(store_k, store_v, pool_k, pool_v, chunks, th, r, o, pairing):
    """Vectorised restatement (complex rotation, einsum patch, brute-force-pinned
    rounding through torch) used to pin the oracle's indexing."""
    pk = pool_k.copy()
    pv = pool_v.copy()
    K = to_f64(store_k)
    V = to_f64(store_v)
    for c in chunks:
        sl = slice(c.src_offset, c.src_offset + c.length)
        k = complex_rotate(K[:, sl], c.delta, th, r, o, pairing) if c.delta else K[:, sl].copy()
        v = V[:, sl].copy()
        if c.rank:
            Uk, Vk, Uv, Vv = (to_f64(p) for p in c.patches)
            k += np.einsum("lhtm,lhdm->lthd", Uk, Vk)
            v += np.einsum("lhtm,lhdm->lthd", Uv, Vv)
        pk[:, c.slots] = _round(k)
        pv[:, c.slots] = _round(v)
    return pk, pv


def _round(x):
    """fp64 -> bf16 round-to-nearest-even.  Through torch's fp32 -> bf16 where the
    two-step rounding provably agrees with one step (the fp32 value is not exactly
    a bf16 midpoint); the remaining elements by brute force."""
    x = np.asarray(x, dtype=np.float64)
    f32 = x.astype(np.float32)
    out = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    low = f32.view(np.uint32) & 0xFFFF
    ambiguous = (f32.astype(np.float64) != x) & (low == 0x8000)
    flat_out = out.reshape(-1)
    flat_x = x.reshape(-1)
    for i in np.flatnonzero(ambiguous.reshape(-1)):
        flat_out[i] = brute_bf16(float(flat_x[i]))
    return out


def _small_gqa(rng, L=2, H=3, d=32, lens=(20, 16, 7), m=4, deltas=(5, -300, 0), page=4,
               zero_rank=False):
    N = sum(lens)
    store_k = rand_bf16(rng, (L, N, H, d))
    store_v = rand_bf16(rng, (L, N, H, d))
    need = -(-N // page)
    S = (need + 3) * page
    perm = rng.permutation(S // page)
    pool_k = np.full((L, S, H, d), 0x5A5A, dtype=np.uint16)
    pool_v = pool_k.copy()
    chunks = []
    pos = 0
    off = 0
    for t, dl in zip(lens, deltas):
        p = np.arange(pos, pos + t)
        slots = perm[p // page] * page + p % page
        mm = 0 if zero_rank else m
        pat = []
        if mm:
            pat = [rand_bf16(rng, (L, H, t, mm), .05), rand_bf16(rng, (L, H, d, mm), .05),
                   rand_bf16(rng, (L, H, t, mm), .05), rand_bf16(rng, (L, H, d, mm), .05)]
        chunks.append(O.Chunk(off, t, dl, mm, slots.astype(np.int64), pat))
        pos += t
        off += t
    return store_k, store_v, pool_k, pool_v, chunks


def pin_gqa_problem(orc: O.Oracle):
    rng = np.random.default_rng(13)
    for pairing, r, o in ((RH, 32, 0), (IL, 32, 0), (RH, 16, 8)):
        sk, sv, pk, pv, chunks = _small_gqa(rng)
        th = orc.inv_freq(1e4, r)
        want_k, want_v = _gqa_numpy(sk, sv, pk, pv, chunks, th, r, o, pairing)
        orc.gqa(sk, sv, pk, pv, chunks, th, r, o, pairing)
        assert np.array_equal(pk, want_k)
        assert np.array_equal(pv, want_v)


def pin_gqa_permutation_bit_exact(orc: O.Oracle):
    rng = np.random.default_rng(14)
    sk, sv, pk, pv, chunks = _small_gqa(rng, deltas=(0, 0, 0), zero_rank=True)
    sk[0, 0, 0, :4] = [0x8000, 0x8000, 0x0000, 0x8001]
    before = pk.copy()
    orc.gqa(sk, sv, pk, pv, chunks, orc.inv_freq(1e4, 32), 32, 0, RH)
    touched = np.zeros(pk.shape[1], dtype=bool)
    for c in chunks:
        assert np.array_equal(pk[:, c.slots], sk[:, c.src_offset:c.src_offset + c.length])
        assert np.array_equal(pv[:, c.slots], sv[:, c.src_offset:c.src_offset + c.length])
        touched[c.slots] = True
    assert np.array_equal(pk[:, ~touched], before[:, ~touched])
    assert np.array_equal(pv[:, ~touched], before[:, ~touched])


def pin_mla_problem(orc: O.Oracle):
    rng = np.random.default_rng(15)
    L, kv, rope, lens, m = 2, 64, 16, (9, 12), 3
    W = kv + rope
    N = sum(lens)
    store = rand_bf16(rng, (L, N, W))
    S = 32
    for rank in (0, m):
        pool = np.full((L, S, W), 0x5A5A, dtype=np.uint16)
        slots = rng.permutation(S)[:N].astype(np.int64)
        chunks = []
        off = 0
        for i, t in enumerate(lens):
            pat = []
            if rank:
                pat = [rand_bf16(rng, (L, t, rank), .05), rand_bf16(rng, (L, kv, rank), .05),
                       rand_bf16(rng, (L, t, rank), .05), rand_bf16(rng, (L, rope, rank), .05)]
            chunks.append(O.Chunk(off, t, (-1000, 77)[i], rank, slots[off:off + t], pat))
            off += t
        th = orc.inv_freq(1e4, rope)
        before = pool.copy()
        orc.mla(store, pool, chunks, kv, th, IL)
        X = to_f64(store)
        for c in chunks:
            src = X[:, c.src_offset:c.src_offset + c.length]
            ckv = src[..., :kv].copy()
            kr = complex_rotate(src[..., kv:], c.delta, th, rope, 0, IL)
            if rank:
                Uc, Vc, Ur, Vr = (to_f64(p) for p in c.patches)
                ckv += np.einsum("ltm,ldm->ltd", Uc, Vc)
                kr += np.einsum("ltm,ldm->ltd", Ur, Vr)
            got = pool[:, c.slots]
            if rank == 0:   # c_KV reused byte for byte
                assert np.array_equal(got[..., :kv], store[:, c.src_offset:c.src_offset + c.length, :kv])
            else:
                assert np.array_equal(got[..., :kv], _round(ckv))
            assert np.array_equal(got[..., kv:], _round(kr))
        untouched = np.setdiff1d(np.arange(S), slots)
        assert np.array_equal(pool[:, untouched], before[:, untouched])


def pin_slide_problem(orc: O.Oracle):
    rng = np.random.default_rng(16)
    L, S, H, d = 2, 40, 2, 32
    for pairing, r, o in ((RH, 32, 0), (IL, 16, 16)):
        pool = rand_bf16(rng, (L, S, H, d))
        before = pool.copy()
        slots = rng.permutation(S)[:25].astype(np.int64)
        chunks = [O.Chunk(0, 15, -4096, 0, slots[:15]), O.Chunk(0, 10, 0, 0, slots[15:])]
        th = orc.inv_freq(1e6, r)
        orc.slide(pool, chunks, th, r, o, pairing)
        want = complex_rotate(to_f64(before[:, slots[:15]]), -4096, th, r, o, pairing)
        assert np.array_equal(pool[:, slots[:15]], _round(want))
        assert np.array_equal(pool[:, slots[15:]], before[:, slots[15:]])   # delta 0: no-op
        rest = np.setdiff1d(np.arange(S), slots)
        assert np.array_equal(pool[:, rest], before[:, rest])


def pin_ingest_problem(orc: O.Oracle):
    """Ingest = gather by slot, turn the keys by R(delta) (complex formulation,
    exact rounding), copy the values, write store rows src_offset..; other
    store rows untouched; delta 0 is a bit-exact gather."""
    rng = np.random.default_rng(18)
    L, S, H, d, N = 2, 48, 2, 32, 40
    for pairing, r, o in ((RH, 32, 0), (IL, 16, 16)):
        pool_k, pool_v = rand_bf16(rng, (L, S, H, d)), rand_bf16(rng, (L, S, H, d))
        store_k = np.full((L, N, H, d), 0x5A5A, np.uint16)
        store_v = store_k.copy()
        slots = rng.permutation(S)[:30].astype(np.int64)
        chunks = [O.Chunk(3, 18, -5000, 0, slots[:18]), O.Chunk(25, 12, 0, 0, slots[18:])]
        th = orc.inv_freq(1e4, r)
        orc.ingest(pool_k, pool_v, store_k, store_v, chunks, th, r, o, pairing)
        want = complex_rotate(to_f64(pool_k[:, slots[:18]]), -5000, th, r, o, pairing)
        assert np.array_equal(store_k[:, 3:21], _round(want))
        assert np.array_equal(store_k[:, 25:37], pool_k[:, slots[18:]])      # delta 0: exact gather
        assert np.array_equal(store_v[:, 3:21], pool_v[:, slots[:18]])
        assert np.array_equal(store_v[:, 25:37], pool_v[:, slots[18:]])
        rest = np.r_[0:3, 21:25, 37:N]
        assert np.all(store_k[:, rest] == 0x5A5A) and np.all(store_v[:, rest] == 0x5A5A)


def pin_ingest_recovers_canonical_keys(orc: O.Oracle):
    """A chunk prefilled at positions s..s+T-1 (model-style RoPE table, rounded
    to bf16 in the cache) and ingested with delta = -s equals the same keys made
    at positions 0..T-1, to within the cache's own bf16 rounding; relocating the
    ingested chunk back by +s returns the cache rows within that rounding too."""
    rng = np.random.default_rng(19)
    for pairing in (RH, IL):
        d, T, s0, S = 64, 24, 4242, 64
        th = orc.inv_freq(1e4, d)
        k_raw = rng.standard_normal((T, d))
        pos = s0 + np.arange(T)
        live = np.stack([table_rope(k_raw[j], pos[j], th, pairing) for j in range(T)])
        canon = np.stack([table_rope(k_raw[j], j, th, pairing) for j in range(T)])
        pool = np.zeros((1, S, 1, d), np.uint16)
        slots = rng.permutation(S)[:T].astype(np.int64)
        pool[0, slots, 0] = _round(live)
        store = np.zeros((1, T, 1, d), np.uint16)
        orc.ingest(pool, None, store, None, [O.Chunk(0, T, -s0, 0, slots)], th, d, 0, pairing)
        got = to_f64(store[0, :, 0])
        tol = 2.0 ** -7 * np.max(np.abs(canon), axis=1, keepdims=True)   # two bf16 roundings of the row
        assert np.all(np.abs(got - canon) <= tol)
        assert np.abs(got - canon).max() > 0                               # the rounding is really there
        rows = orc.rotate(got, s0, th, d, 0, pairing)
        assert np.all(np.abs(rows - to_f64(pool[0, slots, 0])) <= tol)


# --------------------------------------------------- attention over chunks
def _attend_problem(rng, H=2, G=3, d=32, lens=(9, 5, 12, 3), deltas=(40, -7, 0, 1000), m=4, seqs=(0, 2, 4),
                    L=2, layer=1, zero_rank=False):
    N = sum(lens)
    store_k = rand_bf16(rng, (L, N, H, d))
    store_v = rand_bf16(rng, (L, N, H, d))
    chunks, off = [], 0
    for t, dl in zip(lens, deltas):
        mm = 0 if zero_rank else m
        pat = []
        if mm:
            pat = [rand_bf16(rng, (L, H, t, mm), .3), rand_bf16(rng, (L, H, d, mm), .3),
                   rand_bf16(rng, (L, H, t, mm), .3), rand_bf16(rng, (L, H, d, mm), .3)]
        chunks.append(O.Chunk(off, t, dl, mm, np.arange(t, dtype=np.int64), pat))
        off += t
    q = rand_bf16(rng, (len(seqs) - 1, H * G, d))
    return store_k[layer], store_v[layer], chunks, list(seqs), q, layer


def pin_attend_single_token(orc: O.Oracle):
    """One token: the softmax weight is 1, so the output is that token's value row."""
    rng = np.random.default_rng(31)
    sk, sv, chunks, seqs, q, layer = _attend_problem(rng, lens=(1,), deltas=(77,), seqs=(0, 1), zero_rank=True)
    th = orc.inv_freq(1e4, 32)
    bits, out, _ = orc.attend(sk, sv, chunks, seqs, q, layer, th, 32)
    for h in range(q.shape[1]):
        assert np.array_equal(bits[0, h], sv[0, h // 3])


def pin_attend_uniform_keys(orc: O.Oracle):
    """Identical keys (delta 0, no patch): uniform weights, the mean of the values."""
    rng = np.random.default_rng(32)
    sk, sv, chunks, seqs, q, layer = _attend_problem(rng, lens=(6, 4), deltas=(0, 0), seqs=(0, 2), zero_rank=True)
    sk[:] = sk[0]
    th = orc.inv_freq(1e4, 32)
    _, out, _ = orc.attend(sk, sv, chunks, seqs, q, layer, th, 32)
    vmean = to_f64(sv).mean(axis=0)
    for h in range(q.shape[1]):
        assert np.max(np.abs(out[0, h] - vmean[h // 3])) < 1e-12


def _attend_fused(orc, sk, sv, chunks, seqs, q, layer, th, r, o, pairing, scale):
    """The same attention by the identity a fused kernel uses: the query turned by
    -delta per chunk against the canonical keys, the patch as (V_k^T q) . u, and
    the value patch folded in per chunk as V_v (sum_j p_j u_v,j); rotation by
    complex multiplication (not the oracle's routine)."""
    kf, vf, qf = to_f64(sk), to_f64(sv), to_f64(q)
    S, Hq, d = qf.shape
    H = kf.shape[1]
    G = Hq // H
    out = np.zeros((S, Hq, d))
    for s in range(S):
        cs = chunks[seqs[s]:seqs[s + 1]]
        for h in range(Hq):
            g = h // G
            scores, parts = [], []
            for c in cs:
                rows = slice(c.src_offset, c.src_offset + c.length)
                qr = complex_rotate(qf[s, h], -c.delta, th, r, o, pairing)
                sc = kf[rows, g, :] @ qr
                if c.rank:
                    uk, vk, uv, vv = (to_f64(a)[layer, g] for a in c.patches)
                    sc = sc + uk @ (vk.T @ qf[s, h])
                scores.append(scale * sc)
                parts.append(c)
            allsc = np.concatenate(scores)
            w = np.exp(allsc - allsc.max())
            w /= w.sum()
            acc, at = np.zeros(d), 0
            for c, sc in zip(parts, scores):
                pw = w[at:at + len(sc)]
                at += len(sc)
                rows = slice(c.src_offset, c.src_offset + c.length)
                acc += pw @ vf[rows, g, :]
                if c.rank:
                    uk, vk, uv, vv = (to_f64(a)[layer, g] for a in c.patches)
                    acc += vv @ (pw @ uv)
            out[s, h] = acc
    return out


def pin_attend_fused_identity(orc: O.Oracle):
    """The oracle's attention over the reuse equation's rows equals the fused
    formulation (query turned per chunk, rank-m score and value corrections)."""
    rng = np.random.default_rng(33)
    for pairing, r, o in ((RH, 32, 0), (IL, 16, 8)):
        sk, sv, chunks, seqs, q, layer = _attend_problem(rng)
        th = orc.inv_freq(1e4, r)
        _, out, _ = orc.attend(sk, sv, chunks, seqs, q, layer, th, r, o, pairing, scale=0.2)
        ref = _attend_fused(orc, sk, sv, chunks, seqs, q, layer, th, r, o, pairing, 0.2)
        assert np.max(np.abs(out - ref)) < 1e-10, (pairing, np.max(np.abs(out - ref)))


def pin_attend_relative_position(orc: O.Oracle):
    """Moving every chunk and the query by the same D changes nothing (RoPE
    depends on relative position); with patches, V_k turned by R(D) as well (the
    patch-frame identity R(D)(K + U V^T) = R(D) K + U (R(D) V)^T)."""
    rng = np.random.default_rng(34)
    for zero_rank in (True, False):
        sk, sv, chunks, seqs, q, layer = _attend_problem(rng, zero_rank=zero_rank)
        th = orc.inv_freq(1e4, 32)
        _, out, _ = orc.attend(sk, sv, chunks, seqs, q, layer, th, 32)
        D = 123
        moved = []
        for c in chunks:
            pat = c.patches
            if c.rank:
                vk = to_f64(pat[1])
                vk_t = np.swapaxes(complex_rotate(np.swapaxes(vk, -1, -2), D, th, 32, 0, RH), -1, -2)
                pat = [to_f64(pat[0]), vk_t, to_f64(pat[2]), to_f64(pat[3])]
            moved.append(O.Chunk(c.src_offset, c.length, c.delta + D, c.rank, c.slots, pat))
        qm = complex_rotate(to_f64(q), D, th, 32, 0, RH)
        _, out2, _ = orc.attend(sk, sv, moved, seqs, qm, layer, th, 32)
        assert np.max(np.abs(out2 - out)) < 1e-9, (zero_rank, np.max(np.abs(out2 - out)))


def pin_attend_per_chunk_tables(orc: O.Oracle):
    """Chunks of one sequence moved by different multi-axis amounts: attention
    over keys built independently at per-axis positions (table RoPE at
    move_c[axis_f] per frequency, plus the key patch) equals the oracle given
    one table per chunk, theta'_f = move_c[axis_f] * theta_f, at delta 1 (0
    for a chunk that does not move)."""
    rng = np.random.default_rng(35)
    d, G = 32, 3
    sk, sv, chunks, seqs, q, layer = _attend_problem(rng, d=d, G=G)
    th = orc.inv_freq(1e4, d)
    for layout in ("sections", "interleaved"):
        axis = W.freq_axes(d // 2, layout).astype(np.int64)
        moves = np.array([[40, 40, 40], [-7, 0, 0], [0, 0, 0], [900, -13, 250]], dtype=np.int64)
        tabs = np.stack([mv[axis].astype(np.float64) * th for mv in moves])
        run = [O.Chunk(c.src_offset, c.length, int(np.any(mv != 0)), c.rank, c.slots, c.patches)
               for c, mv in zip(chunks, moves)]
        _, out, _ = orc.attend(sk, sv, run, seqs, q, layer, tabs, d)
        kf, vf, qf = to_f64(sk), to_f64(sv), to_f64(q)
        for s in range(len(seqs) - 1):
            for h in range(q.shape[1]):
                g = h // G
                Ks, Vs = [], []
                for ci in range(seqs[s], seqs[s + 1]):
                    c = chunks[ci]
                    rows = slice(c.src_offset, c.src_offset + c.length)
                    kk = table_rope(kf[rows, g], moves[ci][axis].astype(np.float64), th, RH)
                    vv = vf[rows, g]
                    if c.rank:
                        uk, vk, uv, vvm = (to_f64(a)[layer, g] for a in c.patches)
                        kk, vv = kk + uk @ vk.T, vv + uv @ vvm.T
                    Ks.append(kk)
                    Vs.append(vv)
                K, V = np.concatenate(Ks), np.concatenate(Vs)
                sc = (K @ qf[s, h]) / np.sqrt(d)
                pr = np.exp(sc - sc.max())
                want = (pr / pr.sum()) @ V
                assert np.max(np.abs(out[s, h] - want)) < 1e-9, (layout, s, h)


def _mla_attend_problem(rng, C=32, R=16, Hq=5, lens=(9, 5, 12, 3), deltas=(40, -7, 0, 1000), m=4, seqs=(0, 2, 4),
                        L=2, layer=1, zero_rank=False):
    store = rand_bf16(rng, (sum(lens), C + R))
    chunks, off = [], 0
    for t, dl in zip(lens, deltas):
        mm = 0 if zero_rank else m
        pat = []
        if mm:
            pat = [rand_bf16(rng, (L, t, mm), .3), rand_bf16(rng, (L, C, mm), .3),
                   rand_bf16(rng, (L, t, mm), .3), rand_bf16(rng, (L, R, mm), .3)]
        chunks.append(O.Chunk(off, t, dl, mm, np.arange(t, dtype=np.int64), pat))
        off += t
    q = rand_bf16(rng, (len(seqs) - 1, Hq, C + R))
    return store, chunks, list(seqs), q, layer


def pin_attend_mla_is_gqa_attention(orc: O.Oracle):
    """MLA attention is GQA attention with one KV head whose key is the whole
    row [c_KV | k_rope] turned on k_rope only, and whose value is the same row:
    the first kv_lora output columns agree.  The MLA factors become the key and
    value factors [U_c | U_r] and blockdiag(V_c, V_r) of rank 2m."""
    rng = np.random.default_rng(36)
    C, R = 32, 16
    for pairing in (IL, RH):
        for zero_rank in (False, True):
            store, chunks, seqs, q, layer = _mla_attend_problem(rng, C, R, zero_rank=zero_rank)
            th = orc.inv_freq(1e4, R)
            _, out, _ = orc.attend_mla(store, chunks, seqs, q, layer, C, th, R, 0, pairing)
            gch = []
            for c in chunks:
                pat = []
                if c.rank:
                    uc, vc, ur, vr = (to_f64(a) for a in c.patches)
                    u = np.concatenate([uc, ur], axis=2)[:, None]
                    v = np.zeros((uc.shape[0], 1, C + R, 2 * c.rank))
                    v[:, 0, :C, :c.rank] = vc
                    v[:, 0, C:, c.rank:] = vr
                    pat = [u, v, u, v]
                gch.append(O.Chunk(c.src_offset, c.length, c.delta, 2 * c.rank, c.slots, pat))
            rows = store[:, None, :]
            _, gout, _ = orc.attend(rows, rows, gch, seqs, q, layer, th, R, C, pairing, scale=(C + R) ** -0.5)
            assert np.max(np.abs(gout[..., :C] - out)) < 1e-10, (pairing, zero_rank)


def pin_attend_mla_single_token(orc: O.Oracle):
    """One token, no patch: every head's output is that token's c_KV row, bit for bit."""
    rng = np.random.default_rng(37)
    store, chunks, seqs, q, layer = _mla_attend_problem(rng, lens=(1,), deltas=(77,), seqs=(0, 1), zero_rank=True)
    bits, _, _ = orc.attend_mla(store, chunks, seqs, q, layer, 32, orc.inv_freq(1e4, 16), 16)
    for h in range(q.shape[1]):
        assert np.array_equal(bits[0, h], store[0, :32])


def pin_attend_mla_relative_position(orc: O.Oracle):
    """Moving every chunk and the rope query by the same D changes nothing; with
    patches, V_r turned by R(D) as well (the patch-frame identity on k_rope)."""
    rng = np.random.default_rng(38)
    C, R = 32, 16
    for zero_rank in (True, False):
        store, chunks, seqs, q, layer = _mla_attend_problem(rng, C, R, zero_rank=zero_rank)
        th = orc.inv_freq(1e4, R)
        _, out, _ = orc.attend_mla(store, chunks, seqs, q, layer, C, th, R, 0, IL)
        D = 321
        moved = []
        for c in chunks:
            pat = c.patches
            if c.rank:
                vr = to_f64(pat[3])
                vr_t = np.swapaxes(complex_rotate(np.swapaxes(vr, -1, -2), D, th, R, 0, IL), -1, -2)
                pat = [to_f64(pat[0]), to_f64(pat[1]), to_f64(pat[2]), vr_t]
            moved.append(O.Chunk(c.src_offset, c.length, c.delta + D, c.rank, c.slots, pat))
        qm = to_f64(q)
        qm[..., C:] = complex_rotate(qm[..., C:], D, th, R, 0, IL)
        _, out2, _ = orc.attend_mla(store, moved, seqs, qm, layer, C, th, R, 0, IL)
        assert np.max(np.abs(out2 - out)) < 1e-9, (zero_rank, np.max(np.abs(out2 - out)))


def pin_attend_mla_per_chunk_tables(orc: O.Oracle):
    """MLA chunks of one sequence moved by different multi-axis amounts: attention
    over latent rows whose k_rope is built independently at per-axis positions
    (table RoPE at move_c[axis_f] per frequency, plus the patches) equals the
    oracle given one table per chunk at delta 1 (0 for a chunk that does not move)."""
    rng = np.random.default_rng(39)
    C, R = 32, 16
    store, chunks, seqs, q, layer = _mla_attend_problem(rng, C, R)
    th = orc.inv_freq(1e4, R)
    for layout in ("sections", "interleaved"):
        axis = W.freq_axes(R // 2, layout).astype(np.int64)
        moves = np.array([[40, 40, 40], [-7, 0, 0], [0, 0, 0], [900, -13, 250]], dtype=np.int64)
        tabs = np.stack([mv[axis].astype(np.float64) * th for mv in moves])
        run = [O.Chunk(c.src_offset, c.length, int(np.any(mv != 0)), c.rank, c.slots, c.patches)
               for c, mv in zip(chunks, moves)]
        _, out, _ = orc.attend_mla(store, run, seqs, q, layer, C, tabs, R, 0, IL)
        sf, qf = to_f64(store), to_f64(q)
        for s in range(len(seqs) - 1):
            lat, keys = [], []
            for ci in range(seqs[s], seqs[s + 1]):
                c = chunks[ci]
                rows = slice(c.src_offset, c.src_offset + c.length)
                cl = sf[rows, :C]
                kr = table_rope(sf[rows, C:], moves[ci][axis].astype(np.float64), th, IL)
                if c.rank:
                    uc, vc, ur, vr = (to_f64(a)[layer] for a in c.patches)
                    cl, kr = cl + uc @ vc.T, kr + ur @ vr.T
                lat.append(cl)
                keys.append(np.concatenate([cl, kr], axis=1))
            K, V = np.concatenate(keys), np.concatenate(lat)
            for h in range(q.shape[1]):
                sc = (K @ qf[s, h]) / np.sqrt(C + R)
                pr = np.exp(sc - sc.max())
                want = (pr / pr.sum()) @ V
                assert np.max(np.abs(out[s, h] - want)) < 1e-9, (layout, s, h)


def _softmax_attend(K, V, q, scale):
    sc = scale * (K @ q)
    w = np.exp(sc - sc.max())
    return (w / w.sum()) @ V


def pin_attend_rows_are_the_row_oracle(orc: O.Oracle):
    """The attention oracles build each chunk's rows (numpy rotation and factor
    products) exactly as the C row oracle defines one output row of the reuse
    equation: attention over rows taken from ``row`` (fp64 values) agrees with
    ``attend`` (GQA) and ``attend_mla`` to 1e-10, both pairings."""
    rng = np.random.default_rng(40)
    for pairing in (RH, IL):
        sk, sv, chunks, seqs, q, layer = _attend_problem(rng)
        H, d = sk.shape[1], sk.shape[2]
        G = q.shape[1] // H
        th = orc.inv_freq(1e4, d)
        _, out, _ = orc.attend(sk, sv, chunks, seqs, q, layer, th, d, 0, pairing)
        qf = to_f64(q)
        for s in range(len(seqs) - 1):
            for g in range(H):
                K, V = [], []
                for c in chunks[seqs[s]:seqs[s + 1]]:
                    for j in range(c.length):
                        r = c.src_offset + j
                        pk = pv = {}
                        if c.rank:
                            pk = dict(u=c.patches[0][layer, g, j], vm=c.patches[1][layer, g])
                            pv = dict(u=c.patches[2][layer, g, j], vm=c.patches[3][layer, g])
                        K.append(orc.row(sk[r, g], True, c.delta, th, d, 0, pairing, **pk)[1])
                        V.append(orc.row(sv[r, g], False, 0, th, d, 0, pairing, **pv)[1])
                for h in range(g * G, (g + 1) * G):
                    want = _softmax_attend(np.array(K), np.array(V), qf[s, h], d ** -0.5)
                    assert np.max(np.abs(out[s, h] - want)) < 1e-10, ("gqa", pairing, s, h)
        C, R = 32, 16
        store, chunks, seqs, q, layer = _mla_attend_problem(rng, C, R)
        th = orc.inv_freq(1e4, R)
        _, out, _ = orc.attend_mla(store, chunks, seqs, q, layer, C, th, R, 0, pairing)
        qf = to_f64(q)
        for s in range(len(seqs) - 1):
            K, V = [], []
            for c in chunks[seqs[s]:seqs[s + 1]]:
                for j in range(c.length):
                    r = c.src_offset + j
                    pc = pr = {}
                    if c.rank:
                        pc = dict(u=c.patches[0][layer, j], vm=c.patches[1][layer])
                        pr = dict(u=c.patches[2][layer, j], vm=c.patches[3][layer])
                    cl = orc.row(store[r, :C], False, 0, th, R, 0, pairing, **pc)[1]
                    kr = orc.row(store[r, C:], True, c.delta, th, R, 0, pairing, **pr)[1]
                    K.append(np.concatenate([cl, kr]))
                    V.append(cl)
            for h in range(q.shape[1]):
                want = _softmax_attend(np.array(K), np.array(V), qf[s, h], (C + R) ** -0.5)
                assert np.max(np.abs(out[s, h] - want)) < 1e-10, ("mla", pairing, s, h)


def pin_rejects_bad_indices(orc: O.Oracle):
    rng = np.random.default_rng(17)
    sk, sv, pk, pv, chunks = _small_gqa(rng)
    chunks[1].slots = chunks[1].slots.copy()
    chunks[1].slots[3] = pk.shape[1]
    try:
        orc.gqa(sk, sv, pk, pv, chunks, orc.inv_freq(1e4, 32), 32, 0, RH)
    except ValueError:
        return
    raise AssertionError("out-of-range slot accepted")


def _prefill_q(rng, seqs, T, Hq, d):
    return rand_bf16(rng, (len(seqs) - 1, T, Hq, d))


def pin_attend_prefill_is_per_token_decode(orc: O.Oracle):
    """No mask applies among the chunk tokens, so prefill attention of T tokens
    is T independent decode attentions (the pinned decode oracle, ``attend``),
    one per token, both pairings, with patches, to 1e-12."""
    rng = np.random.default_rng(41)
    for pairing, r, o in ((RH, 32, 0), (IL, 16, 8)):
        sk, sv, chunks, seqs, _, layer = _attend_problem(rng)
        H, d = sk.shape[1], sk.shape[2]
        q = _prefill_q(rng, seqs, 5, 3 * H, d)
        th = orc.inv_freq(1e4, r)
        _, out, _, lse = orc.attend_prefill(sk, sv, chunks, seqs, q, layer, th, r, o, pairing, scale=0.3)
        for t in range(q.shape[1]):
            _, want, _ = orc.attend(sk, sv, chunks, seqs, q[:, t], layer, th, r, o, pairing, scale=0.3)
            assert np.max(np.abs(out[:, t] - want)) < 1e-12, (pairing, t)
        assert np.all(np.isfinite(lse))


def pin_attend_prefill_lse_closed_form(orc: O.Oracle):
    """Closed forms of the log-sum-exp: with every key the same row k (delta 0,
    no patch) over L tokens, lse = log L + scale q . k; with q = 0, lse = log L
    for any keys; a sequence with no token gets lse = -inf and zeros."""
    rng = np.random.default_rng(42)
    sk, sv, chunks, seqs, _, layer = _attend_problem(rng, lens=(6, 4), deltas=(0, 0), seqs=(0, 2, 2),
                                                     zero_rank=True)
    sk[:] = sk[0]
    H, d = sk.shape[1], sk.shape[2]
    q = _prefill_q(rng, seqs, 3, 3 * H, d)
    th = orc.inv_freq(1e4, 32)
    _, out, _, lse = orc.attend_prefill(sk, sv, chunks, seqs, q, layer, th, 32, scale=0.25)
    kf, qf = to_f64(sk), to_f64(q)
    for t in range(3):
        for h in range(3 * H):
            want = math.log(10) + 0.25 * float(kf[0, h // 3] @ qf[0, t, h])
            assert abs(lse[0, t, h] - want) < 1e-12, (t, h, lse[0, t, h], want)
    assert np.all(lse[1] == -np.inf) and not np.any(out[1])
    sk2, sv2, chunks2, seqs2, _, layer2 = _attend_problem(rng)
    q0 = np.zeros((len(seqs2) - 1, 2, 3 * H, d))
    _, _, _, lse0 = orc.attend_prefill(sk2, sv2, chunks2, seqs2, q0, layer2, th, 32)
    for s in range(len(seqs2) - 1):
        L = sum(c.length for c in chunks2[seqs2[s]:seqs2[s + 1]])
        assert np.max(np.abs(lse0[s] - math.log(L))) < 1e-12, s


def pin_attend_prefill_lse_merge(orc: O.Oracle):
    """The log-sum-exp merges softmaxes: attention over a sequence's chunks
    equals the two halves' outputs weighted by e^lse (and its lse is
    log(e^lse1 + e^lse2)), which is how a prefill joins the reused chunks'
    softmax with the one over its own new tokens."""
    rng = np.random.default_rng(43)
    sk, sv, chunks, _, _, layer = _attend_problem(rng, seqs=(0, 4))
    H, d = sk.shape[1], sk.shape[2]
    q = _prefill_q(rng, (0, 1), 4, 3 * H, d)
    th = orc.inv_freq(1e4, 32)
    _, out, _, lse = orc.attend_prefill(sk, sv, chunks, [0, 4], q, layer, th, 32, scale=0.4)
    _, o1, _, l1 = orc.attend_prefill(sk, sv, chunks[:1], [0, 1], q, layer, th, 32, scale=0.4)
    _, o2, _, l2 = orc.attend_prefill(sk, sv, chunks[1:], [0, 3], q, layer, th, 32, scale=0.4)
    mx = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - mx)[..., None], np.exp(l2 - mx)[..., None]
    assert np.max(np.abs(out - (w1 * o1 + w2 * o2) / (w1 + w2))) < 1e-12
    assert np.max(np.abs(lse - np.logaddexp(l1, l2))) < 1e-12


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
