// kamera_patchform.cu -- rank-m patch factors from deficit blocks on sm_103a.
//
// The one-time step before reuse (gist.science technical summary, section 2,
// "The Kamera Operator": the patch keeps the top-m part of an SVD of the
// deficit Delta = KV(B|A) - KV(B|empty); section 3.1: the orbit patch is the
// same from the deficit averaged over orderings).  For every block
// X (rows x cols: one (layer, head) of a chunk's keys or values, or the mean
// of n_terms such blocks):
//     G = X^T X / trace                 Gram matrix, fp32, scaled to trace 1
//     G = Z diag(lambda) Z^T            top m eigenpairs, lambda descending
//     V = Z[:, :m],  U = X V            (= W Sigma: the singular values sit in U)
// so that U V^T is the best rank-m approximation of X (Eckart-Young) and the
// factors have the layouts the relocation kernels read.
//
// One CTA owns one block; everything between the two passes over X stays in
// shared memory.  The eigen-solve is the textbook route for a few eigenpairs
// of a small dense symmetric matrix (Golub & Van Loan, sections 8.3-8.4; the
// LAPACK tridiagonal-bisection-inverse-iteration path):
//   1. Householder tridiagonalisation T = Q^T G Q, one reflector per column:
//      p = beta G22 v and the rank-2 update G22 -= v w^T + w v^T spread over
//      all warps; the reflectors stay in the zeroed part of G.
//   2. The m largest eigenvalues of T by bisection on Sturm counts (the
//      inertia of T - x I from its LDL^T pivots): S lanes per eigenvalue test
//      S points at once, so each round narrows the interval S + 1 times.
//   3. Their eigenvectors by inverse iteration: (T - lambda I) y = b solved by
//      Gaussian elimination with partial pivoting (U keeps three diagonals),
//      three solves from a fixed pseudo-random start, one lane per vector;
//      then classical Gram-Schmidt applied twice over the m vectors, which
//      also separates vectors of clustered (or repeated) eigenvalues.
//   4. Back-transformation Z = Q Y, reflector by reflector over all columns.
// Shared-memory traffic is O(n^3) words once instead of once per Jacobi sweep.
#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"
#include "kamera_ptx.cuh"

namespace kamera {

namespace {

constexpr int kPfThreads = 512;
constexpr int kPfWarps = kPfThreads / 32;
constexpr int kPfMaxCols = 128;
constexpr int kPfSolves = 3;   // inverse-iteration solves per eigenvector

struct PfShared {
    float* g;      // [n][n+1]: Gram, then its tridiagonal reduction (reflectors below the subdiagonal)
    float* z;      // [n][n+1]: staged rows of X; the elimination work arrays of the solves
    float* y;      // [n][ys]: eigenvectors (row stride ys = m + 1, odd or 1 apart from a bank multiple)
    float* d;      // [n] diagonal of T
    float* e;      // [n] subdiagonal of T
    float* e2;     // [n] its squares
    float* beta;   // [n] reflector scales
    float* vv;     // [n] reflector of the current column
    float* pv;     // [n] beta G22 v; Gram-Schmidt coefficients
    float* lam;    // [m] eigenvalues of the scaled Gram, descending
};

__host__ __device__ inline int pf_round16(int bytes) { return (bytes + 15) & ~15; }

__host__ __device__ inline int pf_mpad(int m) { return (m + 3) & ~3; }

// Row stride of the eigenvector table: m + 1, so that a warp walking down a
// column (Gram-Schmidt, back-transformation) meets 32 different banks
// whenever m is a multiple of 32 (and at most 2-way conflicts otherwise).
__host__ __device__ inline int pf_ystride(int m) { return m + 1; }

// Shared-memory layout (bytes from a 1024-aligned base): the eigenvector
// table first, then G, the staging region, six n-vectors and the eigenvalues.
// The tensor-core operand tiles start at the first 1024-byte boundary after
// the eigenvector table and overlap G and what follows: they live only while
// those are not in use (the Gram pass writes G after its last MMA; the U pass
// runs after the solve).
struct PfLayout {
    int y, g, z, vec, lam, end, tc, tc_end;
};

__host__ __device__ inline int pf_round1024(int bytes) { return (bytes + 1023) & ~1023; }

__host__ __device__ inline int pf_uatoms(int n) { return (n + 63) / 64; }   // 64-column K atoms of X

__host__ __device__ inline int pf_nb(int m) { return (m + 15) & ~15; }     // MMA N of the U pass

__host__ __device__ inline PfLayout pf_layout(int n, int m)
{
    PfLayout L;
    const int ld = n + 1;
    L.y = 0;
    L.g = pf_round16(n * pf_ystride(m) * 4);
    L.z = L.g + pf_round16(n * ld * 4);
    L.vec = L.z + pf_round16(n * ld * 4);
    L.lam = L.vec + 6 * pf_round16(n * 4);
    L.end = L.lam + pf_round16(m * 4);
    L.tc = pf_round1024(L.g);
    const int ua = pf_uatoms(n);
    const int gram_tile = 2 * 128 * 128;                                 // 128 x 128 tokens, bf16
    const int u_tiles = ua * 128 * 128 + 2 * ua * pf_nb(m) * 128;        // X tile, V^T hi and lo
    L.tc_end = L.tc + (gram_tile > u_tiles ? gram_tile : u_tiles);
    return L;
}

__host__ __device__ inline int pf_smem_bytes(int n, int m)
{
    const PfLayout L = pf_layout(n, m);
    return (L.end > L.tc_end ? L.end : L.tc_end) + 1024;   // + room to align the base
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Stage rows [r0, r0 + nr) of the block's (mean) deficit as fp32, row-major with
// stride ld (even).
__device__ __forceinline__ void stage_rows(const PatchFormParams& p, const __nv_bfloat16* x, int r0, int nr,
                                           float* st, int ld)
{
    const int n = p.cols, vpr = n / 8;
    const float inv = 1.0f / (float)p.n_terms;
    for (int it = threadIdx.x; it < nr * vpr; it += kPfThreads) {
        const int r = it / vpr, c8 = (it - r * vpr) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (r0 + r < p.rows) {
            const __nv_bfloat16* src = x + (int64_t)(r0 + r) * p.row_stride + c8;
            for (int k = 0; k < p.n_terms; ++k) {
                float v[8];
                unpack8(*reinterpret_cast<const uint4*>(src + (int64_t)k * p.term_stride), v);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] += v[e];
            }
            if (p.n_terms > 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] *= inv;
            }
        }
        float2* dst = reinterpret_cast<float2*>(st + r * ld + c8);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            dst[e] = make_float2(acc[2 * e], acc[2 * e + 1]);
    }
}

// G = X^T X: every thread owns an 8 x 4 tile of G (rows i0.., columns j0..).
__device__ void gram(const PatchFormParams& p, const __nv_bfloat16* x, const PfShared& s)
{
    const int n = p.cols, ld = n + 1;
    const int tj_n = n / 4, tiles = (n / 8) * tj_n;
    const int ti = threadIdx.x / tj_n, tj = threadIdx.x - ti * tj_n;
    const bool own = threadIdx.x < tiles;
    const int i0 = 8 * ti, j0 = 4 * tj;
    float acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
            acc[a][b] = 0.f;
    const int rt = n;   // rows per staged tile: n x n floats fit the z region
    for (int r0 = 0; r0 < p.rows; r0 += rt) {
        const int nr = min(rt, p.rows - r0);
        __syncthreads();
        stage_rows(p, x, r0, nr, s.z, n);
        __syncthreads();
        if (own) {
            for (int t = 0; t < nr; ++t) {
                const float* row = s.z + t * n;
                const float4 a0 = *reinterpret_cast<const float4*>(row + i0);
                const float4 a1 = *reinterpret_cast<const float4*>(row + i0 + 4);
                const float4 b = *reinterpret_cast<const float4*>(row + j0);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int a = 0; a < 8; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[a][c] = fmaf(av[a], bv[c], acc[a][c]);
            }
        }
    }
    if (own) {
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                s.g[(i0 + a) * ld + j0 + c] = acc[a][c];
    }
    __syncthreads();
}

// ------------------------------------------------------ tensor-core passes --
constexpr uint64_t kPfTimeoutNs = 1000000000ull;   // bound on every MMA completion wait
constexpr uint32_t kPfTmemCols = 128;
constexpr uint32_t kPfAtom = 128 * 128;            // one 64-element K atom of a 128-row operand

struct PfTc {
    uint32_t tile;    // shared address of the operand tiles (1024-aligned)
    uint32_t bar;     // MMA completion barrier
    uint32_t tmem;    // accumulator columns
    uint32_t phase;   // completions waited for so far
};

// Byte offset of the 16-byte piece (row r, K piece kc) of a K-major operand
// with 128-byte swizzle and atoms of atom_bytes.
__device__ __forceinline__ uint32_t pf_piece(int r, int kc, uint32_t atom_bytes)
{
    return (uint32_t)(kc >> 3) * atom_bytes + (uint32_t)r * 128u + ((uint32_t)((kc & 7) ^ (r & 7)) << 4);
}

// Thread 0 waits for the next MMA completion (bounded); the result reaches
// every thread through the barrier that follows.
__device__ __forceinline__ bool pf_wait_mma(PfTc& t, int32_t* err, int* s_abort, uint64_t p_wait_ns)
{
    if (threadIdx.x == 0) {
        // A short bound (the test hook) polls without suspending.  A bound of 0
        // gives up at once, without polling: the wait it stands for is then
        // certainly still pending (every wait here follows an MMA issue), so the
        // exit path must drain that MMA.
        const bool quick = p_wait_ns < 100000u;
        auto poll = [&]() {
            return quick ? ptx::mbar_test_wait(t.bar, t.phase & 1u) : ptx::mbar_try_wait(t.bar, t.phase & 1u);
        };
        if (p_wait_ns == 0 || !poll()) {
            const uint64_t t0 = p_wait_ns == 0 ? 0 : ptx::globaltimer();
            for (;;) {
                if (p_wait_ns == 0 || ptx::globaltimer() - t0 > p_wait_ns) {
                    *s_abort = 1;
                    raise_err(err, KAMERA_DEVERR_TIMEOUT);
                    break;
                }
                if (poll())
                    break;
            }
        }
    }
    ++t.phase;
    __syncthreads();
    ptx::tc_fence_after();
    return *(volatile int*)s_abort == 0;
}

// Eight bf16 rows (one 16-byte vector each) -> eight columns: out[c] holds
// element c of rows 0..7.
__device__ __forceinline__ void transpose8(const uint4 (&in)[8], uint4 (&out)[8])
{
    uint32_t w[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        w[r][0] = in[r].x;
        w[r][1] = in[r].y;
        w[r][2] = in[r].z;
        w[r][3] = in[r].w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = __byte_perm(w[2 * k][c >> 1], w[2 * k + 1][c >> 1], sel);
        out[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// G = X^T X on the tensor cores: per 128-token tile, X^T is written as a
// K-major operand (rows = columns of X, zero rows past n) and multiplied by
// itself; G leaves TMEM into s.g.  Returns false after a timeout.
__device__ bool gram_tc(const PatchFormParams& p, const __nv_bfloat16* x, const PfShared& s, PfTc& t,
                        int* s_abort)
{
    const int n = p.cols, ld = n + 1, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < 2 * (int)kPfAtom / 16; e += kPfThreads)
        ptx::sts128(t.tile + 16u * e, 0u, 0u, 0u, 0u);
    const int nb = n / 8, items = 16 * nb;   // 8 x 8 blocks of a tile: 16 token blocks x n/8 column blocks
    const int tb = threadIdx.x / nb, cb = threadIdx.x - tb * nb;
    const uint32_t idesc = ptx::idesc_bf16_f32(128, 128);
    for (int t0 = 0; t0 < p.rows; t0 += 128) {
        uint4 in[8];
        if (threadIdx.x < items) {
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int tok = t0 + 8 * tb + r;
                in[r] = tok < p.rows ? *reinterpret_cast<const uint4*>(x + (int64_t)tok * p.row_stride + 8 * cb)
                                     : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (t0 > 0 && !pf_wait_mma(t, p.err, s_abort, p.wait_ns))   // the previous tile's MMAs have read the tile
            return false;
        if (threadIdx.x < items) {
            uint4 out[8];
            transpose8(in, out);
#pragma unroll
            for (int c = 0; c < 8; ++c)   // row 8 cb + c, tokens 8 tb .. 8 tb + 7
                ptx::sts128(t.tile + pf_piece(8 * cb + c, tb, kPfAtom), out[c].x, out[c].y, out[c].z, out[c].w);
        }
        ptx::fence_proxy_async();
        __syncthreads();
        if (threadIdx.x == 0) {
            ptx::tc_fence_after();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint64_t d = ptx::desc_k_sw128(t.tile + (q >> 2) * kPfAtom + (q & 3) * 32);
                ptx::umma_bf16(t.tmem, d, d, idesc, (t0 > 0 || q > 0) ? 1u : 0u);
            }
            ptx::umma_commit(t.bar);
        }
    }
    if (!pf_wait_mma(t, p.err, s_abort, p.wait_ns))
        return false;
    {   // TMEM lanes are rows of G; warp w reads lanes 32 (w % 4).., columns 32 (w / 4)..
        const int i = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);
        const uint32_t ta = t.tmem + ((uint32_t)(32 * (warp & 3)) << 16) + c0;
        uint32_t a[8], b[8], c[8], d[8];
        ptx::tmem_ld8x2_issue(ta, ta + 8, a, b);
        ptx::tmem_ld8x2_issue(ta + 16, ta + 24, c, d);
        ptx::tmem_wait8x2(a, b);
        ptx::tmem_wait8x2(c, d);
        if (i < n) {
            float* row = s.g + i * ld + c0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (c0 + k < n) row[k] = __uint_as_float(a[k]);
                if (c0 + 8 + k < n) row[8 + k] = __uint_as_float(b[k]);
                if (c0 + 16 + k < n) row[16 + k] = __uint_as_float(c[k]);
                if (c0 + 24 + k < n) row[24 + k] = __uint_as_float(d[k]);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    return true;
}

// U = X V on the tensor cores: V^T split into bf16 hi + lo parts (B operands,
// rows = ranks, zero past m), X tiles of 128 tokens as A; the two products
// accumulate in TMEM and leave as bf16 rows of U.
__device__ bool u_tc(const PatchFormParams& p, const __nv_bfloat16* x, const PfShared& s, int ys, PfTc& t,
                     __nv_bfloat16* uo, int* s_abort)
{
    const int n = p.cols, m = p.m, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ua = pf_uatoms(n), N = pf_nb(m), kp = 2 * ((n + 15) / 16);   // K pieces the MMAs read
    const uint32_t a_tile = t.tile, b_hi = a_tile + ua * kPfAtom, b_lo = b_hi + ua * N * 128;
    const uint32_t b_atom = (uint32_t)N * 128u;
    for (int e = threadIdx.x; e < N * kp; e += kPfThreads) {   // V^T pieces: rank r, d = 8 kc ..
        const int r = e / kp, kc = e - r * kp;
        float hi[8], lo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = 8 * kc + k;
            const float v = (r < m && c < n) ? s.y[c * ys + r] : 0.f;
            hi[k] = __bfloat162float(__float2bfloat16_rn(v));
            lo[k] = v - hi[k];
        }
        const uint4 h = pack8(hi), l = pack8(lo);
        ptx::sts128(b_hi + pf_piece(r, kc, b_atom), h.x, h.y, h.z, h.w);
        ptx::sts128(b_lo + pf_piece(r, kc, b_atom), l.x, l.y, l.z, l.w);
    }
    const uint32_t idesc = ptx::idesc_bf16_f32(128, N);
    const int ks = (n + 15) / 16;   // 16-element K slices
    for (int t0 = 0; t0 < p.rows; t0 += 128) {
        for (int e = threadIdx.x; e < 128 * kp; e += kPfThreads) {   // X rows t0.. as A, zero past n / rows
            const int r = e / kp, kc = e - r * kp, tok = t0 + r;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (tok < p.rows && 8 * kc < n)
                v = *reinterpret_cast<const uint4*>(x + (int64_t)tok * p.row_stride + 8 * kc);
            ptx::sts128(a_tile + pf_piece(r, kc, kPfAtom), v.x, v.y, v.z, v.w);
        }
        ptx::fence_proxy_async();
        __syncthreads();
        if (threadIdx.x == 0) {
            ptx::tc_fence_after();
            for (int q = 0; q < ks; ++q) {
                const uint32_t ko = (q >> 2), kb = (q & 3) * 32;
                const uint64_t ad = ptx::desc_k_sw128(a_tile + ko * kPfAtom + kb);
                ptx::umma_bf16(t.tmem, ad, ptx::desc_k_sw128(b_hi + ko * b_atom + kb), idesc, q > 0 ? 1u : 0u);
                ptx::umma_bf16(t.tmem, ad, ptx::desc_k_sw128(b_lo + ko * b_atom + kb), idesc, 1u);
            }
            ptx::umma_commit(t.bar);
        }
        if (!pf_wait_mma(t, p.err, s_abort, p.wait_ns))
            return false;
        // TMEM lanes are tokens; warp w reads lanes 32 (w % 4).., 16-column groups g = w / 4, w / 4 + 4, ..
        const int tok = t0 + 32 * (warp & 3) + lane;
        for (int g = warp >> 2; g < N / 16; g += kPfWarps / 4) {
            const uint32_t ta = t.tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * g;
            uint32_t a[8], b[8];
            ptx::tmem_ld8x2_issue(ta, ta + 8, a, b);
            ptx::tmem_wait8x2(a, b);
            if (tok < p.rows) {
                __nv_bfloat16* dst = uo + (int64_t)tok * m + 16 * g;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (16 * g + k < m) dst[k] = __float2bfloat16_rn(__uint_as_float(a[k]));
                    if (16 * g + 8 + k < m) dst[8 + k] = __float2bfloat16_rn(__uint_as_float(b[k]));
                }
            }
        }
        ptx::tc_fence_before();
        __syncthreads();   // TMEM read and the A tile free before the next tile
    }
    return true;
}

// Householder tridiagonalisation of the scaled Gram in s.g (n >= 3 handled;
// n is a multiple of 8 here).  Afterwards d, e hold T and column k of s.g,
// rows k+1.., holds the reflector v_k (v_k[0] = 1) with scale beta_k.
__device__ void tridiagonalise(int n, const PfShared& s)
{
    const int ld = n + 1, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = 0; k < n - 2; ++k) {
        const int L = n - k - 1;
        float* col = s.g + (k + 1) * ld + k;   // x_i = col[i * ld], i < L
        if (warp == 0) {
            float sig = 0.f;
            for (int i = 1 + lane; i < L; i += 32) {
                const float xi = col[i * ld];
                sig = fmaf(xi, xi, sig);
            }
            sig = warp_sum(sig);
            const float x0 = col[0];
            float beta = 0.f, v0 = 1.f, mu = x0;
            if (sig > 0.f) {   // H x = mu e_1 with H = I - beta v v^T, v_0 = 1
                mu = sqrtf(fmaf(x0, x0, sig));
                v0 = x0 <= 0.f ? x0 - mu : -__fdividef(sig, x0 + mu);
                beta = __fdividef(2.f * v0 * v0, fmaf(v0, v0, sig));
            }
            const float inv = __fdividef(1.f, v0);
            for (int i = lane; i < L; i += 32) {
                const float vi = i == 0 ? 1.f : (sig > 0.f ? col[i * ld] * inv : 0.f);
                s.vv[i] = vi;
                col[i * ld] = vi;
            }
            if (lane == 0) {
                s.d[k] = s.g[k * ld + k];
                s.e[k] = mu;
                s.beta[k] = beta;
            }
        }
        __syncthreads();
        const float beta = s.beta[k];
        if (beta == 0.f)
            continue;
        // Four threads per row of G22, each over a quarter of its columns in an
        // order rotated by 8 per quarter: the 32 lanes of a warp (8 rows x 4
        // quarters) touch 32 different banks at every step.
        float* a22 = s.g + (k + 1) * ld + (k + 1);
        const int i = threadIdx.x >> 2, q = threadIdx.x & 3;
        float* row = a22 + i * ld;
        {   // p = beta G22 v
            float acc = 0.f, acc2 = 0.f;
            if (i < L) {
#pragma unroll
                for (int u = 0; u < 32; u += 2) {
                    const int j = 32 * q + ((u + 8 * q) & 31), j2 = 32 * q + ((u + 1 + 8 * q) & 31);
                    if (j < L)
                        acc = fmaf(row[j], s.vv[j], acc);
                    if (j2 < L)
                        acc2 = fmaf(row[j2], s.vv[j2], acc2);
                }
            }
            acc += acc2;
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (q == 0 && i < L)
                s.pv[i] = beta * acc;
        }
        __syncthreads();
        float kk = 0.f;   // w = p - (beta/2)(p.v) v, formed where it is used
        for (int j = lane; j < L; j += 32)
            kk = fmaf(s.pv[j], s.vv[j], kk);
        kk = 0.5f * beta * warp_sum(kk);
        if (i < L) {   // G22 -= v w^T + w v^T, eight columns loaded before any is stored
            const float vi = s.vv[i], wi = fmaf(-kk, vi, s.pv[i]);
            const int jl = min(32, L - 32 * q);   // columns of this quarter
            for (int u0 = 0; u0 < 32; u0 += 8) {
                float a[8], vj[8], pj[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int jj = (u0 + u + 8 * q) & 31, j = 32 * q + jj;
                    const bool ok = jj < jl;
                    a[u] = ok ? row[j] : 0.f;
                    vj[u] = ok ? s.vv[j] : 0.f;
                    pj[u] = ok ? s.pv[j] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int jj = (u0 + u + 8 * q) & 31, j = 32 * q + jj;
                    if (jj < jl)
                        row[j] = a[u] - vi * fmaf(-kk, vj[u], pj[u]) - wi * vj[u];
                }
            }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        s.d[n - 2] = s.g[(n - 2) * ld + n - 2];
        s.d[n - 1] = s.g[(n - 1) * ld + n - 1];
        s.e[n - 2] = s.g[(n - 1) * ld + n - 2];
    }
    __syncthreads();
}

// Eigenvalues of T below x: the negative pivots of the LDL^T factorisation of
// T - x I (Sylvester's law of inertia); tiny pivots are pushed to -piv.
__device__ __forceinline__ int sturm_count(int n, const float* d, const float* e2, float x, float piv)
{
    float q = d[0] - x;
    if (fabsf(q) < piv)
        q = -piv;
    int c = q < 0.f;
    for (int i = 1; i < n; ++i) {
        q = (d[i] - x) - __fdividef(e2[i - 1], q);
        if (fabsf(q) < piv)
            q = -piv;
        c += q < 0.f;
    }
    return c;
}

// The m largest eigenvalues of T into s.lam (descending), by multisection.
__device__ void bisect(int n, int m, const PfShared& s)
{
    __shared__ float s_lo, s_hi, s_piv;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < n - 1; i += kPfThreads)
        s.e2[i] = s.e[i] * s.e[i];
    if (threadIdx.x < 32) {   // Gershgorin interval, pivot floor
        float lo = 3.0e38f, hi = -3.0e38f, emax = 0.f;
        for (int i = lane; i < n; i += 32) {
            const float r = (i > 0 ? fabsf(s.e[i - 1]) : 0.f) + (i < n - 1 ? fabsf(s.e[i]) : 0.f);
            lo = fminf(lo, s.d[i] - r);
            hi = fmaxf(hi, s.d[i] + r);
            if (i < n - 1)
                emax = fmaxf(emax, s.e[i] * s.e[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, o));
        }
        if (lane == 0) {
            const float pad = 1.2e-7f * fmaxf(fabsf(lo), fabsf(hi)) + 1e-30f;
            s_lo = lo - pad;
            s_hi = hi + pad;
            s_piv = fmaxf(1e-30f, 1.2e-7f * emax);
        }
    }
    __syncthreads();
    const int S = m <= 32 ? 16 : (m <= 64 ? 8 : 4);        // lanes per eigenvalue
    const int iters = S == 16 ? 9 : (S == 8 ? 12 : 15);     // (S+1)^iters > 2^32
    const int r = threadIdx.x / S, sl = threadIdx.x - r * S;
    const int k = n - 1 - min(r, m - 1);                    // ascending index of the r-th largest
    const unsigned gmask = (S == 32 ? 0xffffffffu : ((1u << S) - 1u)) << (lane & ~(S - 1));
    float lo = s_lo, hi = s_hi;
    const float piv = s_piv;
    for (int it = 0; it < iters; ++it) {
        const float step = (hi - lo) / (float)(S + 1);
        const int c = sturm_count(n, s.d, s.e2, lo + (float)(sl + 1) * step, piv);
        const int st = __popc(__ballot_sync(0xffffffffu, c <= k) & gmask);   // points left of lambda
        const float nlo = st > 0 ? lo + (float)st * step : lo;
        const float nhi = st < S ? lo + (float)(st + 1) * step : hi;
        lo = nlo;
        hi = nhi;
    }
    if (r < m && sl == 0)
        s.lam[r] = 0.5f * (lo + hi);
    __syncthreads();
}

// A fixed pseudo-random start vector entry in [-1, 1) (integer hash of (i, r)).
__device__ __forceinline__ float start_entry(int i, int r)
{
    uint32_t h = (uint32_t)i * 2654435761u ^ (uint32_t)(r + 1) * 40503u;
    h *= 2246822519u;
    h ^= h >> 15;
    return (float)(h & 0xFFFFFFu) * (1.0f / 8388608.0f) - 1.0f;
}

// (T - lam I) y = b in place (b in y, stride ys), partial pivoting; u0/u1/u2
// (stride ws) hold the three diagonals of U (the first inverted).  Zero pivots become 2^-23
// (T is scaled to trace 1).  The result is scaled to unit length.
__device__ void tridiag_solve(int n, const float* d, const float* e, float lam, float* y, int ys, float* u0,
                              float* u1, float* u2, int ws)
{
    float c0 = d[0] - lam, c1 = n > 1 ? e[0] : 0.f, c2 = 0.f, rc = y[0];
    for (int i = 0; i < n - 1; ++i) {
        float n0 = e[i], n1 = d[i + 1] - lam, n2 = i + 1 < n - 1 ? e[i + 1] : 0.f, rn = y[(i + 1) * ys];
        if (fabsf(n0) > fabsf(c0)) {   // row swap
            float t;
            t = c0; c0 = n0; n0 = t;
            t = c1; c1 = n1; n1 = t;
            t = c2; c2 = n2; n2 = t;
            t = rc; rc = rn; rn = t;
        }
        if (c0 == 0.f)
            c0 = 1.1920929e-7f;
        const float rc0 = __fdividef(1.f, c0);
        const float l = n0 * rc0;
        u0[i * ws] = rc0;   // U's diagonal, stored inverted
        u1[i * ws] = c1;
        u2[i * ws] = c2;
        y[i * ys] = rc;
        c0 = fmaf(-l, c1, n1);
        c1 = fmaf(-l, c2, n2);
        c2 = 0.f;
        rc = fmaf(-l, rc, rn);
    }
    if (c0 == 0.f)
        c0 = 1.1920929e-7f;
    u0[(n - 1) * ws] = __fdividef(1.f, c0);
    y[(n - 1) * ys] = rc;
    float x1 = 0.f, x2 = 0.f, amax = 0.f;
    for (int i = n - 1; i >= 0; --i) {   // back substitution
        const float xi = (y[i * ys] - u1[i * ws] * x1 - u2[i * ws] * x2) * u0[i * ws];
        y[i * ys] = xi;
        amax = fmaxf(amax, fabsf(xi));
        x2 = x1;
        x1 = xi;
    }
    const float inv = amax > 0.f ? 1.f / amax : 1.f;
    float nrm = 0.f;
    for (int i = 0; i < n; ++i) {
        const float v = y[i * ys] * inv;
        nrm = fmaf(v, v, nrm);
    }
    const float sc = inv * rsqrtf(fmaxf(nrm, 1e-30f));
    for (int i = 0; i < n; ++i)
        y[i * ys] *= sc;
}

// Eigenvectors of T for s.lam into s.y (row stride ys).
__device__ void eigenvectors(int n, int m, int ys, const PfShared& s)
{
    const int ld = n + 1, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int q = threadIdx.x; q < n * m; q += kPfThreads) {
        const int i = q / m, r = q - i * m;
        s.y[i * ys + r] = start_entry(i, r);
    }
    __syncthreads();
    // batches of B vectors, one lane each; work arrays [3][n][B] in the z region
    const int B = min(32, (n * ld) / (3 * n));
    if (warp == 0) {
        for (int b0 = 0; b0 < m; b0 += B) {
            const int r = b0 + lane;
            if (lane < B && r < m) {
                for (int it = 0; it < kPfSolves; ++it)
                    tridiag_solve(n, s.d, s.e, s.lam[r], s.y + r, ys, s.z + lane, s.z + n * B + lane,
                                  s.z + 2 * n * B + lane, B);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // classical Gram-Schmidt, twice, vector by vector
    for (int j = 1; j < m; ++j) {
        for (int pass = 0; pass < 2; ++pass) {
            for (int i = warp; i < j; i += kPfWarps) {   // coefficients y_i . y_j
                float acc = 0.f;
                for (int t = lane; t < n; t += 32)
                    acc = fmaf(s.y[t * ys + i], s.y[t * ys + j], acc);
                acc = warp_sum(acc);
                if (lane == 0)
                    s.pv[i] = acc;
            }
            __syncthreads();
            for (int t = threadIdx.x; t < n; t += kPfThreads) {
                float acc = s.y[t * ys + j];
                for (int i = 0; i < j; ++i)
                    acc = fmaf(-s.pv[i], s.y[t * ys + i], acc);
                s.y[t * ys + j] = acc;
            }
            __syncthreads();
        }
        if (warp == 0) {
            float acc = 0.f;
            for (int t = lane; t < n; t += 32)
                acc = fmaf(s.y[t * ys + j], s.y[t * ys + j], acc);
            const float sc = rsqrtf(fmaxf(warp_sum(acc), 1e-30f));
            for (int t = lane; t < n; t += 32)
                s.y[t * ys + j] *= sc;
        }
        __syncthreads();
    }
}

// Z = Q Y = H_0 H_1 ... H_{n-3} Y, one reflector at a time over all columns:
// S threads per column form v^T y_c over interleaved rows, then every thread
// updates its share of the trailing rows.
__device__ void back_transform(int n, int m, int ys, const PfShared& s)
{
    const int ld = n + 1;
    const int S = m <= 16 ? 32 : (m <= 32 ? 16 : (m <= 64 ? 8 : 4));   // S * m <= kPfThreads
    const int c = threadIdx.x / S, sg = threadIdx.x - c * S;
    const int ustep = kPfThreads / m, uc = threadIdx.x % m, ui = threadIdx.x / m;   // update mapping
    for (int k = n - 3; k >= 0; --k) {
        const float beta = s.beta[k];
        if (beta == 0.f)
            continue;
        const float* v = s.g + (k + 1) * ld + k;   // v_i = v[i * ld]
        float* yk = s.y + (k + 1) * ys;            // y_ic = yk[i * ys + c]
        const int L = n - k - 1;
        float acc = 0.f;
        if (c < m)
            for (int i = sg; i < L; i += S)
                acc = fmaf(v[i * ld], yk[i * ys + c], acc);
        for (int o = S >> 1; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (c < m && sg == 0)
            s.pv[c] = beta * acc;
        __syncthreads();
        if (ui < ustep) {   // column uc, rows ui, ui + ustep, ...
            const float sc = s.pv[uc];
            for (int i0 = ui; i0 < L; i0 += 4 * ustep) {
                float yv[4], vv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * ustep;
                    yv[u] = i < L ? yk[i * ys + uc] : 0.f;
                    vv[u] = i < L ? v[i * ld] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * ustep;
                    if (i < L)
                        yk[i * ys + uc] = fmaf(-sc, vv[u], yv[u]);
                }
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kPfThreads, 1) patch_form_kernel(const __grid_constant__ PatchFormParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ float s_trace;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ __align__(8) uint64_t s_bar;
    const int n = p.cols, ld = n + 1, m = p.m, mp = pf_mpad(m), ys = pf_ystride(m);
    const int warp = threadIdx.x >> 5;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const PfLayout lay = pf_layout(n, m);
    PfShared s;
    s.y = reinterpret_cast<float*>(smem + lay.y);
    s.g = reinterpret_cast<float*>(smem + lay.g);
    s.z = reinterpret_cast<float*>(smem + lay.z);
    {
        float** vec[6] = {&s.d, &s.e, &s.e2, &s.beta, &s.vv, &s.pv};
        for (int i = 0; i < 6; ++i)
            *vec[i] = reinterpret_cast<float*>(smem + lay.vec + i * pf_round16(n * 4));
    }
    s.lam = reinterpret_cast<float*>(smem + lay.lam);
    const int64_t blk = blockIdx.x;
    const int64_t bo = blk / p.n_inner, bi = blk - bo * p.n_inner;
    const __nv_bfloat16* x = p.x + bo * p.outer_stride + bi * p.inner_stride;
    __nv_bfloat16* uo = p.u + blk * (int64_t)p.rows * m;

    // The contractions run on the tensor cores when X is a plain bf16 block;
    // the mean of several deficits (not exact in bf16) takes the CUDA cores.
    const bool tc = p.n_terms == 1;
    PfTc t;
    t.tile = ptx::smem_addr(smem) + lay.tc;
    t.bar = ptx::smem_addr(&s_bar);
    t.phase = 0;
    if (tc) {
        if (warp == 0) {
            ptx::tmem_alloc(ptx::smem_addr(&s_tmem), kPfTmemCols);
            ptx::tmem_relinquish();
        }
        if (threadIdx.x == 32) {
            ptx::mbar_init(t.bar, 1);
            ptx::fence_barrier_init();
        }
        if (threadIdx.x == 0)
            s_abort = 0;
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        t.tmem = s_tmem;
    }
    bool ok = true;
    if (tc)
        ok = gram_tc(p, x, s, t, &s_abort);
    else
        gram(p, x, s);

    if (ok) {
        if (threadIdx.x < 32) {   // trace(G) = ||X||_F^2
            float acc = 0.f;
            for (int i = threadIdx.x; i < n; i += 32)
                acc += s.g[i * ld + i];
            acc = warp_sum(acc);
            if (threadIdx.x == 0)
                s_trace = acc;
        }
        __syncthreads();
        const float trace = s_trace;
        if (trace > 0.f) {
            const float inv = 1.f / trace;
            for (int q = threadIdx.x; q < n * n; q += kPfThreads) {
                const int i = q / n, j = q - i * n;
                s.g[i * ld + j] *= inv;
            }
            __syncthreads();
            tridiagonalise(n, s);
            bisect(n, m, s);
            eigenvectors(n, m, ys, s);
            back_transform(n, m, ys, s);
        } else {   // X = 0: any orthonormal V, U = 0, sigma = 0
            for (int q = threadIdx.x; q < n * m; q += kPfThreads) {
                const int i = q / m, r = q - i * m;
                s.y[i * ys + r] = i == r ? 1.f : 0.f;
            }
            for (int r = threadIdx.x; r < m; r += kPfThreads)
                s.lam[r] = 0.f;
            __syncthreads();
        }

        if (p.sigma)
            for (int r = threadIdx.x; r < m; r += kPfThreads)
                p.sigma[blk * m + r] = sqrtf(fmaxf(s.lam[r] * trace, 0.f));
        __nv_bfloat16* vo = p.v + blk * (int64_t)n * m;
        for (int q = threadIdx.x; q < n * m; q += kPfThreads) {
            const int c = q / m, r = q - c * m;
            vo[q] = __float2bfloat16_rn(s.y[c * ys + r]);
        }
        __syncthreads();
        if (tc) {
            u_tc(p, x, s, ys, t, uo, &s_abort);
        } else {
            // fp32 copy of V [n][mp] (16-byte rows, zero-padded) in the g region
            float* vt = s.g;
            for (int q = threadIdx.x; q < n * mp; q += kPfThreads) {
                const int c = q / mp, r = q - c * mp;
                vt[q] = r < m ? s.y[c * ys + r] : 0.f;
            }
            // U = X V: every thread owns 4 rows x 4 ranks of a staged row tile.  The
            // tile's row stride n + 2 puts the rows that the threads of a warp read at
            // once in different banks.
            const int sld = n + 2;
            const int rg = mp / 4, rt = ((n * ld) / sld) & ~3;   // rows that fit the z region
            for (int r0 = 0; r0 < p.rows; r0 += rt) {
                const int nr = min(rt, p.rows - r0);
                __syncthreads();
                stage_rows(p, x, r0, nr, s.z, sld);
                __syncthreads();
                const int items = ((nr + 3) / 4) * rg;
                for (int it = threadIdx.x; it < items; it += kPfThreads) {
                    const int tg = it / rg, k0 = 4 * (it - tg * rg), t0 = 4 * tg;
                    float acc[4][4];
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            acc[a][b] = 0.f;
                    const int tr = min(4, nr - t0);
                    for (int c = 0; c < n; ++c) {
                        const float4 v4 = *reinterpret_cast<const float4*>(vt + c * mp + k0);
#pragma unroll
                        for (int a = 0; a < 4; ++a) {
                            const float xv = a < tr ? s.z[(t0 + a) * sld + c] : 0.f;
                            acc[a][0] = fmaf(xv, v4.x, acc[a][0]);
                            acc[a][1] = fmaf(xv, v4.y, acc[a][1]);
                            acc[a][2] = fmaf(xv, v4.z, acc[a][2]);
                            acc[a][3] = fmaf(xv, v4.w, acc[a][3]);
                        }
                    }
                    for (int a = 0; a < tr; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            if (k0 + b < m)
                                uo[(int64_t)(r0 + t0 + a) * m + k0 + b] = __float2bfloat16_rn(acc[a][b]);
                }
            }
        }
    }
    if (tc) {
        // After a timeout the completion that was waited for last (index
        // t.phase - 1) may still be pending: let that MMA finish before TMEM and
        // the operand tiles are released (no MMA is issued after a timeout).
        if (*(volatile int*)&s_abort && threadIdx.x == 0) {
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(t.bar, (t.phase - 1u) & 1u) && ptx::globaltimer() - t0 < kPfTimeoutNs) {
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(t.tmem, kPfTmemCols);
        }
    }
}

// ------------------------------------------------------------ wide blocks --
// Blocks wider than one SM can hold G for (128 < cols <= 576: the MLA c_KV
// block, or the whole 576-wide latent row as one joint block) take subspace iteration with a Rayleigh-Ritz step (Golub & Van Loan,
// section 8.2.4, orthogonal iteration; the Ritz step of section 8.1): a basis
// Z of k = m + 16 (rounded to 16, at most 48) columns is multiplied by
// G = X^T X kWideIters times, each product streamed over the rows of X as
// X^T (X Z) without forming G, and re-orthonormalised; then C = Z^T G Z
// (k x k) is solved by the routines above, V = Z W[:, :m] and U = X V.  The
// top-m directions converge at the rate (sigma_{k+1} / sigma_m)^2 per
// product.  All on the CUDA cores.  A cluster of CL CTAs shares a block: each
// streams its own share of the rows, and the partial products X^T (X Z) and
// the partial Rayleigh-Ritz sums are added over the cluster through
// distributed shared memory in rank order, so every CTA holds the same basis;
// rank 0 writes V and sigma, every CTA its rows of U.
constexpr int kWideMaxCols = 576;   // rows of Z: one or two per thread
constexpr int kWideMaxRank = 32;
constexpr int kWideIters = 3;
constexpr int kWideT = 32;   // rows of X per staged tile

__host__ __device__ inline int pf_wide_k(int m) { return min(48, (m + 16 + 15) & ~15); }

struct PfWideLayout {
    int z, xt, yt, small, end;
};

// Basis Z (and later V) [c][k+1], X tile [T][c+4], X Z tile [T][k], then the
// small eigenproblem's PfShared for n = k.
__host__ __device__ inline PfWideLayout pf_wide_layout(int c, int m)
{
    const int k = pf_wide_k(m);
    PfWideLayout L;
    L.z = 0;
    L.xt = pf_round16(c * (k + 1) * 4);
    L.yt = L.xt + pf_round16(kWideT * (c + 4) * 4);
    L.small = L.yt + pf_round16(kWideT * k * 4);
    L.end = L.small + pf_round16(k * pf_ystride(m) * 4) + 2 * pf_round16(k * (k + 1) * 4) +
            6 * pf_round16(k * 4) + pf_round16(m * 4);
    return L;
}

// Column-wise classical Gram-Schmidt, twice, on Z [c][zs] (one row per thread;
// rows t and t + 512 when c is above 512),
// every column normalised; coefficients reduced by shuffles and shared atomics
// into coef[0 .. k-1], the squared norm into coef[kWideNormSlot].
constexpr int kWideNormSlot = 63;
template <bool TWO>
__device__ void wide_cgs2_rows(float* z, int zs, int c, int k, float* coef)
{
    const int lane = threadIdx.x & 31, t = threadIdx.x, t2 = TWO ? t + kPfThreads : c;   // rows t and t + 512
    for (int j = 0; j < k; ++j) {
        for (int pass = 0; pass < 2 && j > 0; ++pass) {
            for (int i = t; i < j; i += kPfThreads)
                coef[i] = 0.f;
            __syncthreads();
            const float zj = t < c ? z[t * zs + j] : 0.f, zj2 = t2 < c ? z[t2 * zs + j] : 0.f;
            for (int i = 0; i < j; ++i) {
                float part = (t < c ? z[t * zs + i] * zj : 0.f) + (t2 < c ? z[t2 * zs + i] * zj2 : 0.f);
                part = warp_sum(part);
                if (lane == 0)
                    atomicAdd(&coef[i], part);
            }
            __syncthreads();
            if (t < c) {
                float acc = zj;
                for (int i = 0; i < j; ++i)
                    acc = fmaf(-coef[i], z[t * zs + i], acc);
                z[t * zs + j] = acc;
            }
            if (t2 < c) {
                float acc = zj2;
                for (int i = 0; i < j; ++i)
                    acc = fmaf(-coef[i], z[t2 * zs + i], acc);
                z[t2 * zs + j] = acc;
            }
            __syncthreads();
        }
        if (t == 0)
            coef[kWideNormSlot] = 0.f;
        __syncthreads();
        const float v = t < c ? z[t * zs + j] : 0.f, v2 = t2 < c ? z[t2 * zs + j] : 0.f;
        const float part = warp_sum(v * v + v2 * v2);
        if (lane == 0)
            atomicAdd(&coef[kWideNormSlot], part);
        __syncthreads();
        const float sc = rsqrtf(fmaxf(coef[kWideNormSlot], 1e-30f));
        if (t < c)
            z[t * zs + j] = v * sc;
        if (t2 < c)
            z[t2 * zs + j] = v2 * sc;
        __syncthreads();
    }
}


// Stage rows r0 .. r0 + kWideT - 1 of X (the mean of its terms) as fp32
// [T][c + 4], zero from row r_end on.
__device__ __forceinline__ void wide_stage(const PatchFormParams& p, const __nv_bfloat16* x, int r0, int r_end,
                                           float* xt)
{
    const int c = p.cols, vpr = c / 8, xs = c + 4;
    const float inv = 1.0f / (float)p.n_terms;
    for (int e = threadIdx.x; e < kWideT * vpr; e += kPfThreads) {
        const int r = e / vpr, c8 = (e - r * vpr) * 8;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (r0 + r < r_end) {
            const __nv_bfloat16* src = x + (int64_t)(r0 + r) * p.row_stride + c8;
            for (int tm = 0; tm < p.n_terms; ++tm) {
                float w[8];
                unpack8(*reinterpret_cast<const uint4*>(src + (int64_t)tm * p.term_stride), w);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    v[q] += w[q];
            }
            if (p.n_terms > 1)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    v[q] *= inv;
        }
        float* d = xt + r * xs + c8;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            d[q] = v[q];
    }
}

// out[T][ncol] = Xt[T][c] B[c][ncol] (B row stride bs): each of four adjacent
// threads sums a quarter of c for a 4-row x 4-column block, combined by shuffles.
__device__ void wide_xb(const float* xt, int c, const float* b, int bs, int ncol, float* out, int os)
{
    const int xs = c + 4, cg = (ncol + 3) / 4, blocks = (kWideT / 4) * cg;
    const int q = threadIdx.x & 3, blk = threadIdx.x >> 2;
    float acc[4][4] = {};
    const int t0 = 4 * (blk / cg), j0 = 4 * (blk % cg);
    if (blk < blocks) {
        for (int i = q; i < c; i += 4) {
            float bv[4], xv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                bv[u] = j0 + u < ncol ? b[i * bs + j0 + u] : 0.f;
                xv[u] = xt[(t0 + u) * xs + i];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    acc[a][u] = fmaf(xv[a], bv[u], acc[a][u]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc[a][u] += __shfl_xor_sync(0xffffffffu, acc[a][u], 1);
            acc[a][u] += __shfl_xor_sync(0xffffffffu, acc[a][u], 2);
        }
    if (blk < blocks && q == 0)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + u < ncol)
                    out[(t0 + a) * os + j0 + u] = acc[a][u];
}

// Z <- X^T (X Z) for this CTA's rows of X when Z has more rows than 128 groups
// of four: three column groups, the thread holds rows 4 ig .. 4 ig + 3 of Z and
// columns jg kq .. jg kq + kq - 1 (kq <= 16) in registers.
template <typename TileR0>
__device__ __noinline__ void wide_product3(const PatchFormParams& p, const __nv_bfloat16* x, float* xt, float* yt,
                                             float* z, int zs, int c, int k, int kq, int ig, int jg, bool own,
                                             int n_tiles, int row_hi, const TileR0& tile_r0)
{
    constexpr int KQ = 16;
    float acc[4][KQ] = {};
    for (int q = 0; q < n_tiles; ++q) {
        const int r0 = tile_r0(q);
        wide_stage(p, x, r0, row_hi, xt);
        __syncthreads();
        wide_xb(xt, c, z, zs, k, yt, k);
        __syncthreads();
        if (own) {
            for (int tt = 0; tt < kWideT; ++tt) {
                const float4 xv = *reinterpret_cast<const float4*>(xt + tt * (c + 4) + 4 * ig);
                const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int u = 0; u < KQ; ++u) {
                    if (u < kq && jg * kq + u < k) {
                        const float yv = yt[tt * k + jg * kq + u];
#pragma unroll
                        for (int a = 0; a < 4; ++a)
                            acc[a][u] = fmaf(xa[a], yv, acc[a][u]);
                    }
                }
            }
        }
        __syncthreads();
    }
    if (own)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int u = 0; u < KQ; ++u)
                if (u < kq && jg * kq + u < k)
                    z[(4 * ig + a) * zs + jg * kq + u] = acc[a][u];
}

// TWO: the block is wider than 512 columns, so Z has more rows than the CTA has
// threads (two rows a thread in the per-row steps, three column groups in the
// product).
template <bool TWO>
__global__ void __launch_bounds__(kPfThreads, 1) patch_form_wide_kernel(const __grid_constant__ PatchFormParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float s_coef[kWideNormSlot + 1];
    __shared__ float s_trace;
    const int c = p.cols, m = p.m, k = pf_wide_k(m), zs = k + 1, ys = pf_ystride(m);
    const PfWideLayout lay = pf_wide_layout(c, m);
    float* z = reinterpret_cast<float*>(smem + lay.z);
    float* xt = reinterpret_cast<float*>(smem + lay.xt);
    float* yt = reinterpret_cast<float*>(smem + lay.yt);
    PfShared s;   // the k x k Rayleigh-Ritz problem
    {
        unsigned char* q = smem + lay.small;
        s.y = reinterpret_cast<float*>(q);
        q += pf_round16(k * ys * 4);
        s.g = reinterpret_cast<float*>(q);
        q += pf_round16(k * (k + 1) * 4);
        s.z = reinterpret_cast<float*>(q);
        q += pf_round16(k * (k + 1) * 4);
        float** vec[6] = {&s.d, &s.e, &s.e2, &s.beta, &s.vv, &s.pv};
        for (int i = 0; i < 6; ++i) {
            *vec[i] = reinterpret_cast<float*>(q);
            q += pf_round16(k * 4);
        }
        s.lam = reinterpret_cast<float*>(q);
    }
    // a cluster of CL CTAs shares one block: CTA `crank` streams rows [row_lo, row_hi)
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int CL = p.cluster, crank = (int)(blockIdx.x % (unsigned)CL);
    const int64_t blk = blockIdx.x / CL;
    const int row_lo = (int)((int64_t)p.rows * crank / CL), row_hi = (int)((int64_t)p.rows * (crank + 1) / CL);
    const int64_t bo = blk / p.n_inner, bi = blk - bo * p.n_inner;
    const __nv_bfloat16* x = p.x + bo * p.outer_stride + bi * p.inner_stride;
    const int t = threadIdx.x;

    for (int e = t; e < c * k; e += kPfThreads) {   // fixed pseudo-random start basis
        const int i = e / k, j = e - i * k;
        z[i * zs + j] = start_entry(i, j);
    }
    __syncthreads();
    wide_cgs2_rows<TWO>(z, zs, c, k, s_coef);

    // Z <- orth(X^T (X Z)), kWideIters times; the product accumulates in
    // registers: thread -> rows 4 ig .. 4 ig + 3, columns jg * kq .. + kq, with
    // ncg column groups (4; 3 when the rows of Z outnumber 512 / 4 groups)
    constexpr int ncg = TWO ? 3 : 4;
    const int kq = (k + ncg - 1) / ncg, ig = t / ncg, jg = t - (t / ncg) * ncg;
    const bool own = 4 * ig < c && jg < ncg;
    // The five passes over the rows alternate direction: each pass starts on the
    // rows the one before it read last, which are still in L2 (the 27 blocks of a
    // DeepSeek-V2-Lite chunk stream about as many bytes per pass as L2 holds, so
    // passes that all ran forward found nothing left of the previous one).
    const int n_tiles = (row_hi - row_lo + kWideT - 1) / kWideT;
    int pass = 0;
    auto tile_r0 = [&](int q) { return row_lo + ((pass & 1) ? n_tiles - 1 - q : q) * kWideT; };
    for (int it = 0; it < kWideIters; ++it, ++pass) {
        if constexpr (!TWO) {
            float acc[4][12] = {};
            for (int q = 0; q < n_tiles; ++q) {
                const int r0 = tile_r0(q);
                wide_stage(p, x, r0, row_hi, xt);
                __syncthreads();
                wide_xb(xt, c, z, zs, k, yt, k);
                __syncthreads();
                if (4 * ig < c) {
                    for (int tt = 0; tt < kWideT; ++tt) {
                        const float4 xv = *reinterpret_cast<const float4*>(xt + tt * (c + 4) + 4 * ig);
                        const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int u = 0; u < 12; ++u) {
                            if (u < kq) {
                                const float yv = yt[tt * k + jg * kq + u];
#pragma unroll
                                for (int a = 0; a < 4; ++a)
                                    acc[a][u] = fmaf(xa[a], yv, acc[a][u]);
                            }
                        }
                    }
                }
                __syncthreads();
            }
            if (4 * ig < c)
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int u = 0; u < 12; ++u)
                        if (u < kq)
                            z[(4 * ig + a) * zs + jg * kq + u] = acc[a][u];
        } else {
            wide_product3(p, x, xt, yt, z, zs, c, k, kq, ig, jg, own, n_tiles, row_hi, tile_r0);
        }
        if (CL > 1) {   // add the cluster's partial products, in rank order (the same sum in every CTA)
            cluster.sync();
            float sum[48];
            constexpr int slots = TWO ? 2 : 1;   // rows t, t + 512: the same count in every thread
            for (int sl = 0; sl < slots; ++sl) {
                const int row = t + sl * kPfThreads;
#pragma unroll
                for (int j = 0; j < 48; ++j)
                    sum[j] = 0.f;
                if (row < c)
                    for (int q = 0; q < CL; ++q) {
                        const float* zq = cluster.map_shared_rank(z, q) + row * zs;
#pragma unroll
                        for (int j = 0; j < 48; ++j)
                            if (j < k)
                                sum[j] += zq[j];
                    }
                cluster.sync();   // every CTA has read every partial of this row slot
                if (row < c)
#pragma unroll
                    for (int j = 0; j < 48; ++j)
                        if (j < k)
                            z[row * zs + j] = sum[j];
            }
        }
        __syncthreads();
        wide_cgs2_rows<TWO>(z, zs, c, k, s_coef);
    }

    // Rayleigh-Ritz: C = (X Z)^T (X Z), accumulated per thread over its (a, b) entries
    float cacc[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < n_tiles; ++q) {
        const int r0 = tile_r0(q);
        wide_stage(p, x, r0, row_hi, xt);
        __syncthreads();
        wide_xb(xt, c, z, zs, k, yt, k);
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 5; ++u) {
            const int e = t + u * kPfThreads;
            if (e < k * k) {
                const int a = e / k, b = e - a * k;
                float sum = 0.f;
                for (int tt = 0; tt < kWideT; ++tt)
                    sum = fmaf(yt[tt * k + a], yt[tt * k + b], sum);
                cacc[u] += sum;
            }
        }
        __syncthreads();
    }
    const int ld = k + 1;
#pragma unroll
    for (int u = 0; u < 5; ++u) {
        const int e = t + u * kPfThreads;
        if (e < k * k)
            s.g[(e / k) * ld + e % k] = cacc[u];
    }
    if (CL > 1) {   // the cluster's partial Rayleigh-Ritz sums, in rank order
        cluster.sync();
#pragma unroll
        for (int u = 0; u < 5; ++u) {
            const int e = t + u * kPfThreads;
            cacc[u] = 0.f;
            if (e < k * k)
                for (int q = 0; q < CL; ++q)
                    cacc[u] += cluster.map_shared_rank(s.g, q)[(e / k) * ld + e % k];
        }
        cluster.sync();
#pragma unroll
        for (int u = 0; u < 5; ++u) {
            const int e = t + u * kPfThreads;
            if (e < k * k)
                s.g[(e / k) * ld + e % k] = cacc[u];
        }
    }
    __syncthreads();
    if (t < 32) {
        float acc = 0.f;
        for (int i = t; i < k; i += 32)
            acc += s.g[i * ld + i];
        acc = warp_sum(acc);
        if (t == 0)
            s_trace = acc;
    }
    __syncthreads();
    const float trace = s_trace;
    if (trace > 0.f) {
        const float inv = 1.f / trace;
        for (int q = t; q < k * k; q += kPfThreads)
            s.g[(q / k) * ld + q % k] *= inv;
        __syncthreads();
        tridiagonalise(k, s);
        bisect(k, m, s);
        eigenvectors(k, m, ys, s);
        back_transform(k, m, ys, s);
    } else {
        for (int q = t; q < k * m; q += kPfThreads) {
            const int i = q / m, r = q - i * m;
            s.y[i * ys + r] = i == r ? 1.f : 0.f;
        }
        for (int r = t; r < m; r += kPfThreads)
            s.lam[r] = 0.f;
        __syncthreads();
    }
    if (p.sigma && crank == 0)
        for (int r = t; r < m; r += kPfThreads)
            p.sigma[blk * m + r] = sqrtf(fmaxf(s.lam[r] * trace, 0.f));
    // V = Z W (row t of Z -> row t of V, in place), bf16 out (every CTA of the
    // cluster forms V for its U rows; rank 0 writes it)
    __nv_bfloat16* vo = p.v + blk * (int64_t)c * m;
    for (int row = t; row < c; row += kPfThreads) {
        float zr[48];
#pragma unroll
        for (int j = 0; j < 48; ++j)
            zr[j] = j < k ? z[row * zs + j] : 0.f;
        for (int r = 0; r < m; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 48; ++j)
                if (j < k)
                    acc = fmaf(zr[j], s.y[j * ys + r], acc);
            z[row * zs + r] = acc;
            if (crank == 0)
                vo[(int64_t)row * m + r] = __float2bfloat16_rn(acc);
        }
    }
    __syncthreads();
    // U = X V
    __nv_bfloat16* uo = p.u + blk * (int64_t)p.rows * m;
    ++pass;
    for (int q = 0; q < n_tiles; ++q) {
        const int r0 = tile_r0(q);
        wide_stage(p, x, r0, row_hi, xt);
        __syncthreads();
        wide_xb(xt, c, z, zs, m, yt, m);
        __syncthreads();
        for (int e = t; e < kWideT * m; e += kPfThreads) {
            const int tt = e / m, r = e - tt * m;
            if (r0 + tt < row_hi)
                uo[(int64_t)(r0 + tt) * m + r] = __float2bfloat16_rn(yt[tt * m + r]);
        }
        __syncthreads();
    }
}

}  // namespace

bool patch_form_supported(int cols, int m)
{
    if (cols < 8 || cols % 8 || m < 1 || m > cols)
        return false;
    return cols <= kPfMaxCols || (cols <= kWideMaxCols && m <= kWideMaxRank);
}

cudaError_t launch_patch_form(const PatchFormParams& p, int64_t n_blocks, cudaStream_t stream)
{
    if (p.cols > kPfMaxCols) {
        const int bytes = pf_wide_layout(p.cols, p.m).end;
        const auto kernel = p.cols > kPfThreads ? patch_form_wide_kernel<true> : patch_form_wide_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        // Cluster size: the blocks' rows are split over CL CTAs; each size 1..8
        // is costed as waves / CL (a cluster must sit in one GPC, so the clusters
        // that fit at once can fall short of the blocks), the cheapest taken.
        PatchFormParams q = p;
        q.cluster = 1;
        double best = 1e300;
        for (int cl = 1; cl <= 8; ++cl) {
            const int fit = cluster_fit(reinterpret_cast<const void*>(kernel), kPfThreads, bytes, cl);
            if (fit < 1 || (int64_t)n_blocks * cl > 0x7FFFFFFFll)
                continue;
            const double cost = (double)((n_blocks + fit - 1) / fit) / cl;
            if (cost < best * 0.999) {
                best = cost;
                q.cluster = cl;
            }
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(n_blocks * q.cluster));
        cfg.blockDim = dim3(kPfThreads);
        cfg.dynamicSmemBytes = (size_t)bytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)q.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, q);
    }
    const int bytes = pf_smem_bytes(p.cols, p.m);
    cudaError_t e = cudaFuncSetAttribute(patch_form_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    patch_form_kernel<<<(unsigned)n_blocks, kPfThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kamera
