"""GPU parity of patch formation (kamera_form_patch) against the oracle's
truncated SVD (LAPACK through numpy, pinned by Eckart-Young).

Singular vectors are unique only up to sign, and only where the singular
value is isolated, so each block is compared on what is unique:
  - singular values: |sigma_g^2 - sigma_o^2| <= 1e-4 sigma_1^2.  The GPU forms
    the Gram matrix in fp32 (relative error of an entry at most rows * 2^-24,
    7.7e-5 at 1296 rows) and the eigen-solve is backward stable to a few
    n * 2^-24 of its norm;
  - V has orthonormal columns: |V^T V - I| <= 8e-3 (bf16 entries carry a
    relative error <= 2^-9, so an inner product of unit vectors moves by at
    most about 2 * 2^-9);
  - Eckart-Young: ||X - U_g V_g^T||_F^2 <= ||X - U_o V_o^T||_F^2 + (8e-3 ||X||_F)^2
    (the bf16 factors add at most ~2 * 2^-9 of ||X_m|| to the error);
  - where sigma_m is separated from sigma_{m+1} by >= 5%: the rank-m
    reconstructions agree, ||U_g V_g^T - U_o V_o^T||_F <= 8e-3 ||U_o V_o^T||_F;
  - every column the Gram route resolves: an eigenvector of X^T X moves by
    about (its fp32 error, ~1e-6 sigma_1^2) / (the eigenvalue gap), so columns
    whose squared singular value is >= 2e-4 sigma_1^2 away from both neighbours
    (and within 5% relative) are compared: after aligning the sign,
    |V_g - V_o| <= 6e-3 and |U_g - U_o| <= 6e-3 max|U_o| elementwise (a bf16
    ulp of a unit-vector entry is at most 2^-8).  Directions far below the
    leading ones (sigma_r ~ 1e-3 sigma_1, noise) are resolved only as a span,
    which the Eckart-Young bound covers.
"""
import numpy as np
import pytest
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def _blocks(x: torch.Tensor) -> torch.Tensor:
    """[kv, L, len, H, d] (or with a leading terms axis) -> [.., kv*L, H, len, d] view."""
    if x.dim() == 5:
        kv, L, n, H, d = x.shape
        return x.reshape(kv * L, n, H, d).permute(0, 2, 1, 3)
    T, kv, L, n, H, d = x.shape
    return x.reshape(T, kv * L, n, H, d).permute(0, 1, 3, 2, 4)


def check_factors(xb: np.ndarray, ug: np.ndarray, vg: np.ndarray, sg: np.ndarray, m: int, what: str):
    """xb [rows, cols] fp64 (the block the GPU factored); ug [rows, m], vg [cols, m],
    sg [m] from the GPU."""
    uo, vo = O.form_patch(xb, m)
    so = np.linalg.svd(xb, compute_uv=False)
    s1 = max(so[0], 1e-30)
    k = min(m, len(so))
    assert np.all(np.abs(sg[:k] ** 2 - so[:k] ** 2) <= 1e-4 * s1 ** 2 + 1e-30), (what, sg[:k], so[:k])
    assert np.all(np.abs(sg[k:]) <= 1e-2 * s1 + 1e-30), what
    gram = vg.T @ vg
    assert np.max(np.abs(gram - np.eye(m))) <= 8e-3, (what, np.max(np.abs(gram - np.eye(m))))
    nx = np.linalg.norm(xb)
    res_g = np.linalg.norm(xb - ug @ vg.T) ** 2
    res_o = np.linalg.norm(xb - uo @ vo.T) ** 2
    assert res_g <= res_o + (8e-3 * nx) ** 2, (what, res_g, res_o, nx)
    nxt = so[m] if m < len(so) else 0.0
    if m <= len(so) and so[m - 1] > 0 and (so[m - 1] - nxt) >= 0.05 * so[m - 1]:
        ro = uo @ vo.T
        d = np.linalg.norm(ug @ vg.T - ro)
        assert d <= 8e-3 * max(np.linalg.norm(ro), 1e-30), (what, d, np.linalg.norm(ro))
    for r in range(k):
        lo = so[r - 1] if r > 0 else np.inf
        hi = so[r + 1] if r + 1 < len(so) else 0.0
        if (lo - so[r]) < 0.05 * so[r] or (so[r] - hi) < 0.05 * so[r]:
            continue
        if min(lo ** 2 - so[r] ** 2, so[r] ** 2 - hi ** 2) < 2e-4 * s1 ** 2:
            continue
        sign = 1.0 if vg[:, r] @ vo[:, r] >= 0 else -1.0
        assert np.max(np.abs(sign * vg[:, r] - vo[:, r])) <= 6e-3, (what, r)
        assert np.max(np.abs(sign * ug[:, r] - uo[:, r])) <= 6e-3 * np.max(np.abs(uo[:, r])), (what, r)


def run_and_check(spec: W.DeficitSpec, m: int = None, contiguous: bool = False):
    m = spec.m if m is None else m
    x = W.make_deficit(spec, DEV)
    xb = _blocks(x)
    if contiguous:
        xb = xb.contiguous()
    O_, I_, rows, cols = xb.shape[-4:]
    sig = torch.empty(O_, I_, m, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    u, v = K.kamera_form_patch(xb, m, sigma=sig, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    xh = _f64(xb)
    if xh.ndim == 5:   # orbit patch: the mean over the terms axis
        xh = xh.mean(axis=0)
    uh, vh, sh = _f64(u), _f64(v), _f64(sig)
    for o in range(O_):
        for i in range(I_):
            check_factors(xh[o, i], uh[o, i], vh[o, i], sh[o, i], m, f"{spec.name} block ({o},{i})")
    return x, u, v, sig


def test_qwen_shaped_chunk():
    run_and_check(W.DeficitSpec("pf_qwen", L=1, length=1296, H=2, d=128, m=32))


@pytest.mark.parametrize("m", [1, 16, 31, 64, 128])
def test_ranks(m):
    run_and_check(W.DeficitSpec("pf_ranks", L=1, length=300, H=1, d=128, m=m))


@pytest.mark.parametrize("d", [8, 16, 40, 64, 96])
def test_widths(d):
    run_and_check(W.DeficitSpec("pf_widths", L=2, length=77, H=1, d=d, m=min(16, d)))


def test_fewer_rows_than_columns():
    """Rank <= rows: the columns past the rank span the null space and carry ~0 in U."""
    run_and_check(W.DeficitSpec("pf_short", L=1, length=20, H=2, d=64, m=32, planted=8))


def test_single_row():
    run_and_check(W.DeficitSpec("pf_row", L=1, length=1, H=2, d=64, m=4, planted=1))


def test_contiguous_blocks():
    run_and_check(W.DeficitSpec("pf_contig", L=2, length=129, H=2, d=64, m=16), contiguous=True)


def test_orbit_patch_of_the_mean_deficit():
    """Section 3.1's orbit patch: one patch from the deficit averaged over orderings."""
    run_and_check(W.DeficitSpec("pf_orbit", L=1, length=200, H=2, d=128, m=32, terms=4))


def test_zero_deficit():
    x = torch.zeros(1, 2, 50, 64, dtype=torch.bfloat16, device=DEV)
    sig = torch.full((1, 2, 8), -1.0, dtype=torch.float32, device=DEV)
    u, v = K.kamera_form_patch(x, 8, sigma=sig)
    torch.cuda.synchronize()
    assert torch.count_nonzero(u).item() == 0
    assert torch.count_nonzero(sig).item() == 0
    vh = _f64(v)
    for i in range(2):
        assert np.max(np.abs(vh[0, i].T @ vh[0, i] - np.eye(8))) <= 8e-3


def test_factors_feed_relocation():
    """Factors formed on the GPU are valid patch factors: relocation with them
    (rank 32, delta 0) adds U V^T, which is within the Eckart-Young bound of the
    planted deficit."""
    spec = W.DeficitSpec("pf_feed", L=2, length=160, H=2, d=128, m=32, kv=2)
    x = W.make_deficit(spec, DEV)
    xb = _blocks(x)
    u, v = K.kamera_form_patch(xb, 32)
    L, H, n, d, m = spec.L, spec.H, spec.length, spec.d, 32
    store_k = torch.zeros(L, n, H, d, dtype=torch.bfloat16, device=DEV)
    store_v = torch.zeros_like(store_k)
    pool_k = torch.zeros(L, n, H, d, dtype=torch.bfloat16, device=DEV)
    pool_v = torch.zeros_like(pool_k)
    uk, vk = u[:L].contiguous(), v[:L].contiguous()
    uv, vv = u[L:].contiguous(), v[L:].contiguous()
    slots = torch.arange(n, dtype=torch.int64, device=DEV)
    ch = K.pack_chunks([K.ChunkSpec(0, n, 0, m, slots, (uk, vk, uv, vv))], device=DEV)
    K.kamera_relocate_patch(pool_k, pool_v, store_k, store_v, K.Rope(1e6, 128), ch, 1, n, m)
    torch.cuda.synchronize()
    xh = _f64(x)   # [kv, L, len, H, d]
    for kv, pool in ((0, pool_k), (1, pool_v)):
        got = _f64(pool)
        for l in range(L):
            for h in range(H):
                blk = xh[kv, l, :, h, :]
                so = np.linalg.svd(blk, compute_uv=False)
                opt = np.sqrt(np.sum(so[m:] ** 2))
                err = np.linalg.norm(got[l, :, h, :] - blk)
                assert err <= opt + 1e-2 * np.linalg.norm(blk), (kv, l, h, err, opt)


@pytest.mark.parametrize("length,d,m", [(300, 512, 16), (4096, 512, 16), (300, 512, 32), (129, 136, 16),
                                        (77, 256, 8), (4096, 576, 16), (300, 576, 32), (1000, 520, 8)])
def test_wide_blocks(length, d, m):
    """Blocks wider than 128 columns (the 512-wide MLA c_KV block, and the
    whole 576-wide latent row c_KV | k_rope as one joint block, whose basis has
    more rows than the CTA has threads): subspace iteration + Rayleigh-Ritz,
    held to the same bounds on the planted deficits, whose spectrum falls off
    past the planted directions."""
    run_and_check(W.DeficitSpec("pf_wide", L=2, length=length, H=1, d=d, m=m, kv=1))


def near_optimal(spec: W.DeficitSpec, m: int):
    """Without a gap after sigma_m the wide path's subspace is not the optimal
    one; its rank-m factor still leaves at most 2% of ||X||^2 beyond the
    Eckart-Young optimum, and V stays orthonormal."""
    x = W.make_deficit(spec, DEV)
    xb = _blocks(x)
    sig = torch.empty(1, 1, m, dtype=torch.float32, device=DEV)
    u, v = K.kamera_form_patch(xb, m, sigma=sig)
    torch.cuda.synchronize()
    xh, uh, vh = _f64(xb), _f64(u)[0, 0], _f64(v)[0, 0]
    xh = xh.mean(axis=0)[0, 0] if xh.ndim == 5 else xh[0, 0]
    so = np.linalg.svd(xh, compute_uv=False)
    opt, tot = np.sum(so[m:] ** 2), np.sum(so ** 2)
    res = np.linalg.norm(xh - uh @ vh.T) ** 2
    assert res <= opt + 0.02 * tot, (res, opt, tot)
    assert np.max(np.abs(vh.T @ vh - np.eye(m))) <= 8e-3
    # sigma holds the Ritz values ||X v_r|| of the returned directions (not the
    # singular values, which they only bound from below without a gap)
    ritz = np.linalg.norm(xh @ vh, axis=0)
    assert np.all(np.abs(sig[0, 0].cpu().numpy() - ritz) <= 1e-2 * so[0]), (sig[0, 0].cpu().numpy(), ritz)
    assert np.all(sig[0, 0].cpu().numpy() <= so[:m] * (1 + 1e-2))


def test_wide_flat_spectrum_is_near_optimal():
    near_optimal(W.DeficitSpec("pf_flat", L=1, length=300, H=1, d=512, m=16, kv=1, planted=1, s_max=0.0,
                               s_min=0.0, noise=1.0), 16)


def test_wide_joint_latent_row_is_near_optimal():
    near_optimal(W.DeficitSpec("pf_flat576", L=1, length=400, H=1, d=576, m=16, kv=1, planted=1, s_max=0.0,
                               s_min=0.0, noise=1.0), 16)


def test_wide_orbit_patch_is_near_optimal():
    """The mean of three independently planted deficits spreads its energy over
    ~96 directions (no gap after sigma_16): the near-optimality bound."""
    near_optimal(W.DeficitSpec("pf_wide_orbit", L=1, length=200, H=1, d=512, m=16, kv=1, terms=3), 16)


def test_host_errors():
    x = torch.zeros(1, 1, 16, 584, dtype=torch.bfloat16, device=DEV)   # wider than the 576-wide latent row
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(x, 8)
    assert e.value.status == 3
    x = torch.zeros(1, 1, 16, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(K.KameraError) as e:   # wide blocks take ranks up to 32
        K.kamera_form_patch(x, 33)
    assert e.value.status == 3
    x = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(x, 65)
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(x[..., 4:60], 8)   # columns not a multiple of 8 / misaligned
    assert e.value.status in (2, 3)
