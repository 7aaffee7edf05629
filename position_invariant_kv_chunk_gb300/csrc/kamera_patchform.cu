// kamera_patchform.cu -- rank-m patch factors from deficit blocks on sm_103a.
//
// The one-time step before reuse (gist.science technical summary, section 2,
// "The Kamera Operator": the patch keeps the top-m part of an SVD of the
// deficit Delta = KV(B|A) - KV(B|empty); section 3.1: the orbit patch is the
// same from the deficit averaged over orderings).  For every block
// X (rows x cols: one (layer, head) of a chunk's keys or values, or the mean
// of n_terms such blocks):
//     G = X^T X                          Gram matrix, fp32
//     G = Z diag(lambda) Z^T             cyclic Jacobi, eigenvalues sorted descending
//     V = Z[:, :m],  U = X V             (= W Sigma: the singular values sit in U)
// so that U V^T is the best rank-m approximation of X (Eckart-Young) and the
// factors have the layouts the relocation kernels read.
//
// One CTA owns one block.  G and Z live in shared memory (row stride cols+1,
// so row- and column-wise accesses of a warp hit distinct banks).  Each Jacobi
// round takes cols/2 disjoint index pairs of the round-robin (circle) ordering,
// so every pair (p, q) is met once per sweep; all rotations of a round come
// from the same G and are applied together: thread-per-2x2-block updates over
// the upper triangle of pair blocks (mirrored to keep G exactly symmetric),
// then the eigenvector columns.  A pair whose off-diagonal entry is already
// below the threshold is skipped, a round with no rotation costs one barrier,
// and the solve ends after a sweep without rotations (KAMERA_DEVERR_NOCONV
// if the sweep limit is reached first).
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"

namespace kamera {

namespace {

constexpr int kPfThreads = 512;
constexpr int kPfMaxCols = 128;
constexpr int kPfMaxSweeps = 30;

struct PfShared {
    float* g;          // [n][n+1] Gram, then the eigenvector table for the U pass
    float* z;          // [n][n+1] eigenvectors; staging of X rows outside the solve
    float4* prm;       // [n/2] pair of the round: (p | q << 16 as bits, c, s, t); t = 0: no turn
    uint32_t* tri;     // (a, b) pair blocks with a <= b, packed a | b << 16
    int* order;        // [n] rank -> eigen index
};

__host__ __device__ inline int pf_round16(int bytes) { return (bytes + 15) & ~15; }

__host__ __device__ inline int pf_smem_bytes(int n)
{
    const int n2 = n / 2;
    return 2 * pf_round16(n * (n + 1) * 4) + pf_round16(n2 * 16) + pf_round16(n2 * (n2 + 1) / 2 * 4) +
           pf_round16(n * 4);
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

// One 2x2 block of G for the pair blocks (a, b), a < b: G <- J_a^T G J_b on
// rows {p_a, q_a} x columns {p_b, q_b}, written to both triangles.
__device__ __forceinline__ void turn_block(float* g, int ld, const float4& A, const float4& B)
{
    const uint32_t ia = __float_as_uint(A.x), ib = __float_as_uint(B.x);
    const int pa = (int)(ia & 0xFFFF), qa = (int)(ia >> 16), pb = (int)(ib & 0xFFFF), qb = (int)(ib >> 16);
    const float ca = A.y, sa = A.z, cb = B.y, sb = B.z;
    const float x00 = g[pa * ld + pb], x01 = g[pa * ld + qb];
    const float x10 = g[qa * ld + pb], x11 = g[qa * ld + qb];
    const float y00 = ca * x00 - sa * x10, y01 = ca * x01 - sa * x11;   // rows of pair a
    const float y10 = sa * x00 + ca * x10, y11 = sa * x01 + ca * x11;
    const float z00 = cb * y00 - sb * y01, z01 = sb * y00 + cb * y01;   // columns of pair b
    const float z10 = cb * y10 - sb * y11, z11 = sb * y10 + cb * y11;
    g[pa * ld + pb] = z00;
    g[pa * ld + qb] = z01;
    g[qa * ld + pb] = z10;
    g[qa * ld + qb] = z11;
    g[pb * ld + pa] = z00;
    g[qb * ld + pa] = z01;
    g[pb * ld + qa] = z10;
    g[qb * ld + qa] = z11;
}

// Diagonal block of pair a: g_pp -= t g_pq, g_qq += t g_pq, g_pq = g_qp = 0.
__device__ __forceinline__ void turn_diag(float* g, int ld, const float4& A)
{
    const uint32_t ia = __float_as_uint(A.x);
    const int p = (int)(ia & 0xFFFF), q = (int)(ia >> 16);
    const float t = A.w, apq = g[p * ld + q];
    g[p * ld + p] -= t * apq;
    g[q * ld + q] += t * apq;
    g[p * ld + q] = 0.f;
    g[q * ld + p] = 0.f;
}

// Z <- Z J on columns p, q of row zr.
__device__ __forceinline__ void turn_z(float* zr, const float4& A)
{
    const uint32_t ia = __float_as_uint(A.x);
    const int p = (int)(ia & 0xFFFF), q = (int)(ia >> 16);
    const float c = A.y, sn = A.z;
    const float zp = zr[p], zq = zr[q];
    zr[p] = c * zp - sn * zq;
    zr[q] = sn * zp + c * zq;
}

// Cyclic Jacobi on s.g (n x n, symmetric); eigenvectors accumulate in s.z.
// Returns true when a sweep ended without a rotation.
__device__ bool jacobi(int n, const PfShared& s, float tol_abs)
{
    const int ld = n + 1, n2 = n / 2, ntri = n2 * (n2 + 1) / 2;
    const float tol_rel = 2.4e-7f;   // ~2 ulp of fp32
    for (int e = threadIdx.x; e < n * n; e += kPfThreads) {
        const int i = e / n, j = e - i * n;
        s.z[i * ld + j] = i == j ? 1.f : 0.f;
    }
    for (int a = threadIdx.x; a < n2; a += kPfThreads) {
        const int base = a * n2 - a * (a - 1) / 2;
        for (int b = a; b < n2; ++b)
            s.tri[base + b - a] = (uint32_t)a | ((uint32_t)b << 16);
    }
    __syncthreads();
    // eigenvector update: a fixed pair per thread when the pairs divide the block
    const bool zfixed = kPfThreads % n2 == 0;
    const int za = threadIdx.x % n2, zi0 = threadIdx.x / n2, zstep = kPfThreads / n2;
    for (int sweep = 0; sweep < kPfMaxSweeps; ++sweep) {
        int swept = 0;
        for (int r = 0; r < n - 1; ++r) {
            int rot = 0;
            if (threadIdx.x < n2) {
                // circle method: position 0 fixed, the others turn by one each round
                const int k = threadIdx.x;
                const int p = k == 0 ? 0 : 1 + (k - 1 + r) % (n - 1);
                const int q = 1 + (n - 2 - k + r) % (n - 1);
                const float apq = s.g[p * ld + q], app = s.g[p * ld + p], aqq = s.g[q * ld + q];
                float c = 1.f, sn = 0.f, t = 0.f;
                if (fabsf(apq) > tol_abs && fabsf(apq) > tol_rel * sqrtf(fabsf(app) * fabsf(aqq))) {
                    // the angle that zeroes g_pq (symmetric 2x2 Schur decomposition)
                    const float tau = (aqq - app) / (2.f * apq);
                    const float at = fabsf(tau);
                    t = at > 1e18f ? 0.5f / tau : copysignf(1.f, tau) / (at + sqrtf(fmaf(tau, tau, 1.f)));
                    if (t != 0.f) {
                        c = rsqrtf(fmaf(t, t, 1.f));
                        sn = t * c;
                        rot = 1;
                    } else {
                        t = 0.f;
                    }
                }
                s.prm[k] = make_float4(__uint_as_float((uint32_t)p | ((uint32_t)q << 16)), c, sn, t);
            }
            if (!__syncthreads_or(rot))
                continue;   // nothing turns this round
            swept = 1;
            // G <- J^T G J over the pair blocks (a <= b), two blocks in flight
            for (int e = threadIdx.x; e < ntri; e += 2 * kPfThreads) {
                const int e2 = e + kPfThreads;
                const uint32_t ab = s.tri[e], ab2 = e2 < ntri ? s.tri[e2] : 0u;
                const int a = (int)(ab & 0xFFFF), b = (int)(ab >> 16);
                const int a2 = (int)(ab2 & 0xFFFF), b2 = (int)(ab2 >> 16);
                const float4 A = s.prm[a], B = s.prm[b];
                const float4 A2 = s.prm[a2], B2 = s.prm[b2];
                if (a == b) {
                    if (A.w != 0.f)
                        turn_diag(s.g, ld, A);
                } else if (A.w != 0.f || B.w != 0.f) {
                    turn_block(s.g, ld, A, B);
                }
                if (e2 < ntri) {
                    if (a2 == b2) {
                        if (A2.w != 0.f)
                            turn_diag(s.g, ld, A2);
                    } else if (A2.w != 0.f || B2.w != 0.f) {
                        turn_block(s.g, ld, A2, B2);
                    }
                }
            }
            // Z <- Z J (columns p, q of every row)
            if (zfixed) {
                const float4 A = s.prm[za];
                if (A.w != 0.f) {
#pragma unroll 4
                    for (int i = zi0; i < n; i += zstep)
                        turn_z(s.z + i * ld, A);
                }
            } else {
                for (int e = threadIdx.x; e < n * n2; e += kPfThreads) {
                    const int i = e / n2, a = e - i * n2;
                    const float4 A = s.prm[a];
                    if (A.w != 0.f)
                        turn_z(s.z + i * ld, A);
                }
            }
            __syncthreads();
        }
        if (!swept)
            return true;
    }
    return false;
}

__global__ void __launch_bounds__(kPfThreads, 1) patch_form_kernel(const __grid_constant__ PatchFormParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int n = p.cols, ld = n + 1, n2 = n / 2, m = p.m;
    PfShared s;
    {
        unsigned char* q = smem;
        s.g = reinterpret_cast<float*>(q);
        q += pf_round16(n * ld * 4);
        s.z = reinterpret_cast<float*>(q);
        q += pf_round16(n * ld * 4);
        s.prm = reinterpret_cast<float4*>(q);
        q += pf_round16(n2 * 16);
        s.tri = reinterpret_cast<uint32_t*>(q);
        q += pf_round16(n2 * (n2 + 1) / 2 * 4);
        s.order = reinterpret_cast<int*>(q);
    }
    const int64_t blk = blockIdx.x;
    const int64_t bo = blk / p.n_inner, bi = blk - bo * p.n_inner;
    const __nv_bfloat16* x = p.x + bo * p.outer_stride + bi * p.inner_stride;

    gram(p, x, s);

    // absolute floor of the threshold: 2^-23 of trace(G) = ||X||_F^2
    __shared__ float trace;
    if (threadIdx.x < 32) {
        float acc = 0.f;
        for (int i = threadIdx.x; i < n; i += 32)
            acc += fabsf(s.g[i * ld + i]);
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (threadIdx.x == 0)
            trace = acc;
    }
    __syncthreads();
    const bool converged = jacobi(n, s, trace * 1.1920929e-7f);
    if (!converged && threadIdx.x == 0)
        raise_err(p.err, KAMERA_DEVERR_NOCONV);

    // eigenvalues in descending order (ties by index); every rank starts at a
    // valid index so that non-finite input still reads in bounds
    for (int i = threadIdx.x; i < n; i += kPfThreads)
        s.order[i] = i;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kPfThreads) {
        const float li = s.g[i * ld + i];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const float lj = s.g[j * ld + j];
            rank += (lj > li) || (lj == li && j < i);
        }
        if (rank < m)
            s.order[rank] = i;
    }
    __syncthreads();
    // V = Z[:, order[:m]] (bf16 out, fp32 copy [n][mp] in the g region), sigma
    const int mp = (m + 3) & ~3;
    float* vt = s.g;   // G is no longer needed
    if (p.sigma)
        for (int r = threadIdx.x; r < m; r += kPfThreads) {
            const float l = s.g[s.order[r] * ld + s.order[r]];
            p.sigma[blk * m + r] = sqrtf(fmaxf(l, 0.f));
        }
    __syncthreads();
    __nv_bfloat16* vo = p.v + blk * (int64_t)n * m;
    for (int e = threadIdx.x; e < n * mp; e += kPfThreads) {
        const int c = e / mp, r = e - c * mp;
        const float z = r < m ? s.z[c * ld + s.order[r]] : 0.f;
        vt[e] = z;
        if (r < m)
            vo[(int64_t)c * m + r] = __float2bfloat16_rn(z);
    }
    // U = X V: every thread owns 4 rows x 4 ranks of a staged row tile.  The
    // tile's row stride n + 2 puts the rows that the threads of a warp read at
    // once in different banks.
    __nv_bfloat16* uo = p.u + blk * (int64_t)p.rows * m;
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

}  // namespace

bool patch_form_supported(int cols, int m)
{
    return cols >= 8 && cols <= kPfMaxCols && cols % 8 == 0 && m >= 1 && m <= cols;
}

cudaError_t launch_patch_form(const PatchFormParams& p, int64_t n_blocks, cudaStream_t stream)
{
    const int bytes = pf_smem_bytes(p.cols);
    cudaError_t e = cudaFuncSetAttribute(patch_form_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    patch_form_kernel<<<(unsigned)n_blocks, kPfThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kamera
