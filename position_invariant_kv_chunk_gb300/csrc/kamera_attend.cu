// kamera_attend.cu -- decode attention over reused chunks, without the pool.
//
// The pages serve reused chunks through a hook in the attention kernel (the
// gist.science technical summary, section 3, "Production Deployment"); the
// rows such a hook attends over are the reuse equation's (section 2):
//     K_j = R(delta_c) k_j + V_k u_j,    V_j = v_j + V_v u'_j
// with k_j, v_j the canonical rows of chunk c, u_j, u'_j the rows of its U
// factors and V_k, V_v its V factors.  For a query q the two terms fold into
// quantities formed once per chunk:
//     q . K_j          = (R(-delta_c) q) . k_j + (V_k^T q) . u_j
//     sum_j p_j V_j    = sum_j p_j v_j + V_v (sum_j p_j u'_j)
// so a decode step streams only the canonical rows and the U rows (d + d + 2m
// elements per token and KV head) and never writes a relocated row.
//
// A cluster of CL CTAs owns (sequence, KV head) and serves its G query heads,
// so each row is read once for all of them.  Per 64-token tile the work is two
// small dense products: S[G x 64] = [R(-delta) q | V_k^T q] [k | u]^T and
// [O | W][G x (d + m)] += P [v | u'], with W = sum_j p_j u'_j folded through V_v
// when the chunk ends.  The G query heads (padded to 16) are the rows of
// warp-level bf16 MMAs (m16n8k16, fp32 accumulate): a decode step has at most
// 8 query rows per KV head, far below the 64-row minimum of the tensor-memory
// MMA.  The per-chunk query part and the softmax weights are not bf16 values,
// so they enter as bf16 hi + lo pairs (about 16 significant bits); the rows and
// U rows are exact bf16.  Warp w computes the scores of tokens 8w .. 8w + 7
// and owns value-side column tiles w, w + 8, ...; the online softmax runs with
// 16 threads per head.  A ring of three or four tile buffers keeps the next
// tiles in flight: the key and value rows arrive as 128B-swizzled TMA boxes
// (one thread issues them; completion on an mbarrier, every wait bounded in
// time), the U rows as 16-byte async copies into rows padded to an odd number
// of 16-byte vectors; both layouts keep the 8x8 matrix loads free of bank
// conflicts.  The CTAs of a cluster split the (sequence, head)'s tiles
// evenly (a chunk cut between CTAs is set up by each, and each folds its own
// share of the value patch), CL chosen from the occupancy query so the grid
// runs in as few waves as possible (a cluster must sit in one GPC); rank 0
// merges the partial softmax states through distributed shared memory.
#include <cooperative_groups.h>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"
#include "kamera_ptx.cuh"
#include "kamera_warpmma.cuh"

namespace kamera {

namespace {

using namespace wmma16;

constexpr int kAtThreads = 256;
constexpr int kAtT = 64;      // tokens per tile
constexpr int kAtH = 16;      // MMA rows: a KV head's query heads, padded
constexpr int kAtMaxG = 8;    // query heads per KV head
constexpr int kAtMaxCL = 8;

// D: head dim (64 or 128); MP: the padded rank the instantiation takes (0, 16, 32, 64).
// The canonical rows of a tile arrive by TMA as 128B-swizzled boxes of 64
// columns x 64 tokens (16-byte piece c of row r at piece c ^ (r & 7)); the U
// rows, narrower and per chunk, by 16-byte async copies into rows padded to an
// odd number of 16-byte vectors.  Both layouts keep the 8x8 matrix loads free
// of bank conflicts.
template <int D, int MP>
struct AtSmem {
    static constexpr int KW = D + MP;    // tile row: k | u (key tile), v | u' (value tile)
    static constexpr int NB = D / 64;    // 64-column boxes of a head row
    static constexpr int RS = KW + 8;    // query-part row stride: an odd number of 16-byte vectors
    static constexpr int NT = KW / 8;    // 8-column tiles of the value side
    static constexpr int MPa = MP > 0 ? MP : 1;
    static constexpr int URS = MP + 8;   // U row stride
    static constexpr int NS = KW > 160 ? 3 : 4;   // tile buffers: NS - 1 tiles in flight while one is used
    static constexpr uint32_t kBoxBytes = kAtT * 128;
    __nv_bfloat16 kt[NS][NB][kAtT][64];  // key rows (TMA boxes); the partial outputs at the end
    __nv_bfloat16 vt[NS][NB][kAtT][64];  // value rows
    __nv_bfloat16 ut[NS][kAtT][URS];     // U rows of the key tiles
    __nv_bfloat16 uv[NS][kAtT][URS];     // U' rows of the value tiles
    __nv_bfloat16 xh[kAtH][RS];          // per-chunk query part R(-delta) q | V_k^T q, bf16 hi
    __nv_bfloat16 xl[kAtH][RS];          // and lo
    __nv_bfloat16 q[kAtH][D];            // the queries (target frame; rows past G zero)
    float sc[kAtH][kAtT + 4];            // scores of the tile
    __nv_bfloat16 ph[kAtH][kAtT + 8];    // softmax weights, hi
    __nv_bfloat16 pl[kAtH][kAtT + 8];    // and lo
    float alpha[kAtH];                   // running-max rescale of the tile
    float2 cs[D / 2];                    // cos/sin of -delta
    static constexpr int VKS = MPa + 8;  // V_k row stride: an odd number of 16-byte vectors
    __nv_bfloat16 vk[D][VKS];            // V_k of this (layer, head), staged per chunk
    float wsum[kAtH][MPa];               // sum_j p_j u'_j of the chunk, at its end
    float cm[kAtH], cl[kAtH];            // this CTA's softmax state, for the merge
    float fac[kAtH][kAtMaxCL];           // merge weights (rank 0)
    uint64_t full[NS];                   // the TMA boxes of buffer b have landed
    int32_t abort;                       // a wait ran out: the rest of the work is skipped
};

// The launch: parameters and the tensor maps of the key and value rows
// ([num_rows][H * d], boxes of 64 columns x 64 rows).
struct AttendLaunch {
    AttendParams p;
    CUtensorMap map_k, map_v;
    uint64_t wait_ns;
};

__device__ __forceinline__ int32_t attend_check(const KameraChunk& ch, int c, const AttendParams& p)
{
    int32_t bits = check_axis_delta(p.rope, c);
    if (ch.len < 0 || ch.rank < 0 || ch.delta > KAMERA_MAX_ABS_DELTA || ch.delta < -KAMERA_MAX_ABS_DELTA)
        bits |= KAMERA_DEVERR_DESCRIPTOR;
    if (ch.src_offset < 0 || ch.src_offset + (int64_t)max(ch.len, 0) > p.num_rows)
        bits |= KAMERA_DEVERR_SOURCE;
    if (ch.len > p.max_len)
        bits |= KAMERA_DEVERR_LEN;
    if (ch.rank > p.max_rank)
        bits |= KAMERA_DEVERR_RANK;
    if (ch.rank > 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(patch_ptr(ch, i));
            if (a == 0 || (a & 15))
                bits |= KAMERA_DEVERR_DESCRIPTOR;
        }
    }
    return bits;
}

// Starts the copies of tile rows j0 .. j0 + n - 1 of chunk `ch` (KV head g)
// into buffer b: one thread issues the TMA boxes of the key and value rows
// (rows past the chunk come from the store or read as zero; the caller clears
// the value rows past n once they land), every thread the async copies of the
// U rows (zero past n and past the rank).  One copy group per call.
template <int D, int MP>
__device__ __forceinline__ void attend_load(const AttendLaunch& P, const KameraChunk& ch, int g, int j0, int n, int b,
                                            AtSmem<D, MP>& s)
{
    using SM = AtSmem<D, MP>;
    const AttendParams& p = P.p;
    if (threadIdx.x == 0) {
        const uint32_t bar = ptx::smem_addr(&s.full[b]);
        const int y = (int)(ch.src_offset + j0);
        ptx::mbar_arrive_expect_tx(bar, 2u * SM::NB * SM::kBoxBytes);
#pragma unroll
        for (int x = 0; x < SM::NB; ++x) {
            ptx::tma_load_2d(ptx::smem_addr(&s.kt[b][x][0][0]), &P.map_k, g * D + 64 * x, y, bar);
            ptx::tma_load_2d(ptx::smem_addr(&s.vt[b][x][0][0]), &P.map_v, g * D + 64 * x, y, bar);
        }
    }
    if constexpr (MP > 0) {
        const int m = ch.rank;
        const int64_t fo = ((int64_t)(p.layer * p.H + g) * ch.len + j0) * m;   // U [L][H][len][m]
        const __nv_bfloat16* uk = patch_ptr(ch, 0);
        const __nv_bfloat16* uv = patch_ptr(ch, 2);
        if ((m & 7) == 0) {   // whole 16-byte vectors (m = 0 too: all zeros)
            constexpr int UV = MP / 8;
            for (int e = threadIdx.x; e < kAtT * UV; e += kAtThreads) {
                const int t = e / UV, v = e - t * UV;
                const uint32_t dk = ptx::smem_addr(&s.ut[b][t][8 * v]);
                const uint32_t dv = ptx::smem_addr(&s.uv[b][t][8 * v]);
                if (t < n && 8 * v < m) {
                    const int64_t off = fo + (int64_t)t * m + 8 * v;
                    ptx::cp_async16(dk, uk + off);
                    ptx::cp_async16(dv, uv + off);
                } else {
                    ptx::st_shared_zero16(dk);
                    ptx::st_shared_zero16(dv);
                }
            }
        } else {   // other ranks: element by element
            for (int e = threadIdx.x; e < kAtT * MP; e += kAtThreads) {
                const int t = e / MP, r = e - t * MP;
                __nv_bfloat16 a = __float2bfloat16_rn(0.f), c = a;
                if (t < n && r < m) {
                    a = uk[fo + (int64_t)t * m + r];
                    c = uv[fo + (int64_t)t * m + r];
                }
                s.ut[b][t][r] = a;
                s.uv[b][t][r] = c;
            }
        }
    }
    ptx::cp_async_commit();
}

// Bounded wait on buffer b's TMA boxes.  On expiry the call reports
// KAMERA_DEVERR_TIMEOUT, every later wait of the CTA returns at once, and the
// kernel runs its barriers to the end (its output is then undefined).
__device__ __forceinline__ bool attend_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort, int32_t* err,
                                            uint64_t limit)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (ptx::globaltimer() - t0 > limit) {
                *abort = 1;
                raise_err(err, KAMERA_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

template <int D, int MP>
__global__ void __launch_bounds__(kAtThreads, 1) attend_kernel(const __grid_constant__ AttendLaunch P)
{
    using SM = AtSmem<D, MP>;
    const AttendParams& p = P.p;
    constexpr int NTW = (SM::NT + 7) / 8;   // value-side column tiles per warp
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // swizzled TMA boxes want 1024-byte alignment (the same offset in every CTA)
    SM& s = *reinterpret_cast<SM*>(smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u));
    namespace cg = cooperative_groups;
    const int CL = p.cluster, rank = (int)(blockIdx.x % (unsigned)CL);
    const int seq = blockIdx.x / CL, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, t4 = lane & 3;
    const int G = p.G, HQ = p.H * G;
    // 8x8 matrix-load addressing: A (row-major 16 x 16) and B^T (token rows)
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;

    int c0 = p.seq_start[seq], c1 = p.seq_start[seq + 1];
    if (c0 < 0 || c1 < c0 || c1 > p.n_chunks) {
        if (g == 0 && rank == 0 && threadIdx.x == 0)
            raise_err(p.err, KAMERA_DEVERR_DESCRIPTOR);
        c0 = c1 = 0;
    }
    // this CTA's share: tiles [lo, hi) of the sequence's valid chunks' tiles, in order
    int64_t total = 0;
    for (int c = c0; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        if (!attend_check(ch, c, p))
            total += (ch.len + kAtT - 1) / kAtT;
    }
    const int64_t lo = total * rank / CL, hi = total * (rank + 1) / CL;

    for (int e = threadIdx.x; e < kAtH * D; e += kAtThreads) {
        const int h = e / D, i = e - h * D;
        s.q[h][i] = h < G ? p.q[((int64_t)seq * HQ + g * G + h) * D + i] : __float2bfloat16_rn(0.f);
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < SM::NS; ++b)
            ptx::mbar_init(ptx::smem_addr(&s.full[b]), 1);
        s.abort = 0;
        ptx::fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        ptx::prefetch_tmap(&P.map_k);
        ptx::prefetch_tmap(&P.map_v);
    }
    uint32_t ph = 0;   // phase parity of each buffer's barrier

    float o[NTW][4];   // value-side tile warp + 8 k: rows gq, gq + 8; columns 2 t4, + 1
#pragma unroll
    for (int k = 0; k < NTW; ++k)
        o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;   // head threadIdx.x / 16
    const RopeParams& rp = p.rope;
    const int ro = rp.rot_offset, rr = rp.rot_dim, half = rr / 2;
    const uint32_t kt0 = ptx::smem_addr(&s.kt[0][0][0][0]), vt0 = ptx::smem_addr(&s.vt[0][0][0][0]);
    const uint32_t ut0 = ptx::smem_addr(&s.ut[0][0][0]), uv0 = ptx::smem_addr(&s.uv[0][0][0]);
    constexpr uint32_t kBuf = SM::NB * SM::kBoxBytes;            // bytes per row buffer
    constexpr uint32_t kUBuf = (uint32_t)(kAtT * SM::URS * 2);   // bytes per U buffer

    int64_t pos = 0;   // tiles of the sequence before chunk c
    for (int c = c0; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        const int32_t bad = attend_check(ch, c, p);
        if (bad) {
            if (rank == 0 && threadIdx.x == 0)
                raise_err(p.err, bad);
            continue;
        }
        const int len = ch.len;
        const int nt = (len + kAtT - 1) / kAtT;
        const int64_t a0 = lo - pos, a1 = hi - pos;
        const int t_lo = a0 > 0 ? (int)a0 : 0, t_hi = a1 < nt ? (int)a1 : nt;
        pos += nt;
        if (t_lo >= t_hi)
            continue;
        const int m = ch.rank;
        __syncthreads();   // the previous chunk (or the query staging) is done with every shared array
        const int64_t fo = (int64_t)(p.layer * p.H + g) * D * m;   // this (layer, head)'s V factors [d][m]
        if constexpr (MP > 0) {   // V_k [d][m], zero past the rank: one copy group, older than the tiles'
            const __nv_bfloat16* vkg = patch_ptr(ch, 1);
            if ((m & 7) == 0) {
                constexpr int VV = MP / 8;
                for (int e = threadIdx.x; e < D * VV; e += kAtThreads) {
                    const int i = e / VV, v = e - i * VV;
                    const uint32_t dst = ptx::smem_addr(&s.vk[i][8 * v]);
                    if (8 * v < m)
                        ptx::cp_async16(dst, vkg + fo + (int64_t)i * m + 8 * v);
                    else
                        ptx::st_shared_zero16(dst);
                }
            } else {
                for (int e = threadIdx.x; e < D * MP; e += kAtThreads) {
                    const int i = e / MP, r = e - i * MP;
                    s.vk[i][r] = r < m ? vkg[fo + (int64_t)i * m + r] : __float2bfloat16_rn(0.f);
                }
            }
        }
        ptx::cp_async_commit();
        for (int j = 0; j < SM::NS - 1; ++j) {   // the first NS - 1 tiles land during set-up
            const int tj = t_lo + j;
            if (tj < t_hi)
                attend_load<D, MP>(P, ch, g, tj * kAtT, min(kAtT, len - tj * kAtT), j, s);
            else
                ptx::cp_async_commit();   // one copy group per tile slot, empty or not
        }
        for (int f = threadIdx.x; f < rp.n_freq; f += kAtThreads) {
            float cc, sn;
            phase_cos_sin(-freq_delta(rp, ch, c, f), rp.inv_freq[f], cc, sn);
            s.cs[f] = make_float2(cc, sn);
        }
        ptx::cp_async_wait<SM::NS - 1>();   // V_k has landed (the tiles may still be in flight)
        __syncthreads();
        for (int e = threadIdx.x; e < kAtH * D; e += kAtThreads) {   // q turned by -delta
            const int h = e / D, i = e - h * D, k = i - ro;
            float v = __bfloat162float(s.q[h][i]);
            if (k >= 0 && k < rr) {
                if (rp.pairing == KAMERA_ROPE_ROTATE_HALF) {
                    const float2 t = s.cs[k < half ? k : k - half];
                    v = k < half ? fmaf(v, t.x, -(__bfloat162float(s.q[h][i + half]) * t.y))
                                 : fmaf(v, t.x, __bfloat162float(s.q[h][i - half]) * t.y);
                } else {
                    const float2 t = s.cs[k >> 1];
                    v = (k & 1) == 0 ? fmaf(v, t.x, -(__bfloat162float(s.q[h][i + 1]) * t.y))
                                     : fmaf(v, t.x, __bfloat162float(s.q[h][i - 1]) * t.y);
                }
            }
            split1(v, s.xh[h][i], s.xl[h][i]);
        }
        if constexpr (MP > 0) {   // V_k^T q (the un-turned query) by warp MMAs: warp w takes ranks 8w .. 8w + 7
            if (warp < MP / 8) {
                float y[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t qa = ptx::smem_addr(&s.q[arow][acol]);
                const uint32_t vka = ptx::smem_addr(&s.vk[lane & 15][8 * warp]);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t a[4], bb[2];
                    ldsm_x4(qa + 32 * ks, a);
                    ldsm_x2_t(vka + (uint32_t)(16 * ks * SM::VKS * 2), bb);
                    mma_bf16(y, a, bb[0], bb[1]);
                }
                const int col = D + 8 * warp + 2 * t4;   // rows gq, gq + 8 (heads); columns col, col + 1
                split1(y[0], s.xh[gq][col], s.xl[gq][col]);
                split1(y[1], s.xh[gq][col + 1], s.xl[gq][col + 1]);
                split1(y[2], s.xh[gq + 8][col], s.xl[gq + 8][col]);
                split1(y[3], s.xh[gq + 8][col + 1], s.xl[gq + 8][col + 1]);
            }
        }

        for (int tl = t_lo; tl < t_hi; ++tl) {
            const int i = tl - t_lo, b = i % SM::NS, ntok = min(kAtT, len - tl * kAtT);
            ptx::cp_async_wait<SM::NS - 2>();   // this thread's copies of tile tl (NS - 2 newer groups may fly)
            attend_wait(ptx::smem_addr(&s.full[b]), (ph >> b) & 1u, &s.abort, p.err, P.wait_ns);
            ph ^= 1u << b;
            const uint32_t kb = kt0 + b * kBuf, vb = vt0 + b * kBuf;
            if (ntok < kAtT) {   // value rows past the chunk: zero, so that their zero weights add nothing
                for (int e = threadIdx.x; e < (kAtT - ntok) * 8 * SM::NB; e += kAtThreads) {
                    const int r = ntok + e / (8 * SM::NB), c = e % (8 * SM::NB);
                    ptx::st_shared_zero16(vb + (c >> 3) * SM::kBoxBytes + r * 128 + (c & 7) * 16);
                }
                ptx::fence_proxy_async();   // before a later TMA load refills the buffer
            }
            __syncthreads();   // tile b (and, first, the chunk's query part) in place; every warp is
                               // done with tile tl - 1, its buffer and its scores and weights
            {   // tile tl + NS - 1 into the buffer tile tl - 1 has left
                const int tn = tl + SM::NS - 1;
                if (tn < t_hi)
                    attend_load<D, MP>(P, ch, g, tn * kAtT, min(kAtT, len - tn * kAtT), (i + SM::NS - 1) % SM::NS, s);
                else
                    ptx::cp_async_commit();
            }
            const uint32_t ub = ut0 + b * kUBuf, uvb = uv0 + b * kUBuf;
            {   // scores of tokens 8 warp .. + 7 against the (padded) 16 heads; k-step ks adds
                // its hi and lo products to sums 2 (ks & 1) and 2 (ks & 1) + 1, so a wider
                // instantiation's padded U columns add exact zeros at the chains' ends
                float sa[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    sa[u][0] = sa[u][1] = sa[u][2] = sa[u][3] = 0.f;
                // key row r = 8 warp + (lane & 7), 16-byte piece 2 ks + hi of the row
                const int kr = 8 * warp + (lane & 7), hi = (lane >> 3) & 1;
                const uint32_t krow = kb + (uint32_t)(kr * 128), lx = (uint32_t)(hi ^ (lane & 7));
                const uint32_t urow = ub + (uint32_t)((kr * SM::URS + 8 * hi) * 2);
                const uint32_t xa = ptx::smem_addr(&s.xh[arow][acol]), xla = ptx::smem_addr(&s.xl[arow][acol]);
#pragma unroll
                for (int ks = 0; ks < SM::KW / 16; ++ks) {
                    uint32_t bb[2], ah[4], al[4];
                    if (ks < D / 16)
                        ldsm_x2(krow + (uint32_t)((2 * ks) >> 3) * SM::kBoxBytes + ((((uint32_t)(2 * ks) & 7u) ^ lx) << 4), bb);
                    else
                        ldsm_x2(urow + 32 * (ks - D / 16), bb);
                    ldsm_x4(xa + 32 * ks, ah);
                    ldsm_x4(xla + 32 * ks, al);
                    mma_bf16(sa[2 * (ks & 1)], ah, bb[0], bb[1]);
                    mma_bf16(sa[2 * (ks & 1) + 1], al, bb[0], bb[1]);
                }
                const int tk = 8 * warp + 2 * t4;
                *reinterpret_cast<float2*>(&s.sc[gq][tk]) =
                    make_float2((sa[0][0] + sa[1][0]) + (sa[2][0] + sa[3][0]), (sa[0][1] + sa[1][1]) + (sa[2][1] + sa[3][1]));
                *reinterpret_cast<float2*>(&s.sc[gq + 8][tk]) =
                    make_float2((sa[0][2] + sa[1][2]) + (sa[2][2] + sa[3][2]), (sa[0][3] + sa[1][3]) + (sa[2][3] + sa[3][3]));
            }
            __syncthreads();
            {   // online softmax: 16 threads per head, 4 tokens each
                const int h = threadIdx.x >> 4, j0 = 4 * (threadIdx.x & 15);
                float sv[4], tmax = -INFINITY;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    sv[u] = j0 + u < ntok ? p.scale * s.sc[h][j0 + u] : -INFINITY;
                    tmax = fmaxf(tmax, sv[u]);
                }
#pragma unroll
                for (int off = 8; off > 0; off >>= 1)
                    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
                const float mnew = fmaxf(m_run, tmax);    // finite: the tile holds a token
                const float alpha = __expf(m_run - mnew);  // 0 while nothing was seen
                float e[4], sum = 0.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    e[u] = __expf(sv[u] - mnew);
                    sum += e[u];
                }
#pragma unroll
                for (int off = 8; off > 0; off >>= 1)
                    sum += __shfl_xor_sync(0xffffffffu, sum, off);
                l_run = fmaf(l_run, alpha, sum);
                m_run = mnew;
                uint32_t h01, l01, h23, l23;
                split_hl(e[0], e[1], h01, l01);
                split_hl(e[2], e[3], h23, l23);
                *reinterpret_cast<uint2*>(&s.ph[h][j0]) = make_uint2(h01, h23);
                *reinterpret_cast<uint2*>(&s.pl[h][j0]) = make_uint2(l01, l23);
                if ((threadIdx.x & 15) == 0)
                    s.alpha[h] = alpha;
            }
            __syncthreads();
            {   // [O | W] += P [v | u']: column tiles warp, warp + 8, ...
                const float r0 = s.alpha[gq], r1 = s.alpha[gq + 8];
                if (!__all_sync(0xffffffffu, r0 == 1.f && r1 == 1.f)) {   // a new running max in some row
#pragma unroll
                    for (int k = 0; k < NTW; ++k) {
                        o[k][0] *= r0;
                        o[k][1] *= r0;
                        o[k][2] *= r1;
                        o[k][3] *= r1;
                    }
                }
                const uint32_t pha = ptx::smem_addr(&s.ph[arow][acol]), pla = ptx::smem_addr(&s.pl[arow][acol]);
                // value row 16 ks + (lane & 15); column tile ntile = 16-byte piece ntile of the row
                const uint32_t vrow = vb + (uint32_t)((lane & 15) * 128) + ((uint32_t)(warp ^ (lane & 7)) << 4);
                const uint32_t uvrow = uvb + (uint32_t)(((lane & 15) * SM::URS + 8 * warp) * 2);
#pragma unroll
                for (int ks = 0; ks < kAtT / 16; ++ks) {
                    uint32_t ah[4], al[4];
                    ldsm_x4(pha + 32 * ks, ah);
                    ldsm_x4(pla + 32 * ks, al);
#pragma unroll
                    for (int k = 0; k < NTW; ++k) {
                        const int ntile = warp + 8 * k;
                        if (ntile < SM::NT) {
                            uint32_t bb[2];
                            if (8 * k < D / 8)   // a canonical column tile: box k, piece warp
                                ldsm_x2_t(vrow + (uint32_t)k * SM::kBoxBytes + (uint32_t)(ks * 16 * 128), bb);
                            else                 // a U' column tile
                                ldsm_x2_t(uvrow + (uint32_t)(((ks * 16) * SM::URS + 8 * (8 * k - D / 8)) * 2), bb);
                            mma_bf16(o[k], ah, bb[0], bb[1]);
                            mma_bf16(o[k], al, bb[0], bb[1]);
                        }
                    }
                }
            }
        }
        if constexpr (MP > 0) {
            if (m > 0) {   // fold W = sum_j p_j u'_j through V_v: O += W V_v^T
#pragma unroll
                for (int k = 0; k < NTW; ++k) {
                    const int ntile = warp + 8 * k;
                    if (ntile >= D / 8 && ntile < SM::NT) {
                        const int col = 8 * ntile - D + 2 * t4;
                        s.wsum[gq][col] = o[k][0];
                        s.wsum[gq][col + 1] = o[k][1];
                        s.wsum[gq + 8][col] = o[k][2];
                        s.wsum[gq + 8][col + 1] = o[k][3];
                        o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
                    }
                }
                __syncthreads();
                const __nv_bfloat16* vvg = patch_ptr(ch, 3) + fo;   // V_v [d][m]
#pragma unroll
                for (int ks = 0; ks < MP / 16; ++ks) {
                    const int q0 = 16 * ks + 2 * t4;
                    uint32_t ah[4], al[4];
                    split_hl(s.wsum[gq][q0], s.wsum[gq][q0 + 1], ah[0], al[0]);
                    split_hl(s.wsum[gq + 8][q0], s.wsum[gq + 8][q0 + 1], ah[1], al[1]);
                    split_hl(s.wsum[gq][q0 + 8], s.wsum[gq][q0 + 9], ah[2], al[2]);
                    split_hl(s.wsum[gq + 8][q0 + 8], s.wsum[gq + 8][q0 + 9], ah[3], al[3]);
#pragma unroll
                    for (int k = 0; k < NTW; ++k) {
                        const int ntile = warp + 8 * k;
                        if (ntile < D / 8) {
                            const int64_t i = 8 * ntile + gq;
                            const uint16_t* vr = reinterpret_cast<const uint16_t*>(vvg + i * m);
                            const uint32_t b0 = (q0 < m ? (uint32_t)vr[q0] : 0u) |
                                                ((q0 + 1 < m ? (uint32_t)vr[q0 + 1] : 0u) << 16);
                            const uint32_t b1 = (q0 + 8 < m ? (uint32_t)vr[q0 + 8] : 0u) |
                                                ((q0 + 9 < m ? (uint32_t)vr[q0 + 9] : 0u) << 16);
                            mma_bf16(o[k], ah, b0, b1);
                            mma_bf16(o[k], al, b0, b1);
                        }
                    }
                }
            }
        }
    }

    // merge: every CTA publishes (max, sum, unnormalised output); rank 0 combines
    ptx::cp_async_wait<0>();
    __syncthreads();   // the tile buffers are free
    float* ob = reinterpret_cast<float*>(&s.kt[0][0][0][0]);   // [kAtH][D]
#pragma unroll
    for (int k = 0; k < NTW; ++k) {
        const int ntile = warp + 8 * k;
        if (ntile < D / 8) {
            const int col = 8 * ntile + 2 * t4;
            *reinterpret_cast<float2*>(&ob[gq * D + col]) = make_float2(o[k][0], o[k][1]);
            *reinterpret_cast<float2*>(&ob[(gq + 8) * D + col]) = make_float2(o[k][2], o[k][3]);
        }
    }
    if ((threadIdx.x & 15) == 0) {
        s.cm[threadIdx.x >> 4] = m_run;
        s.cl[threadIdx.x >> 4] = l_run;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0) {
        if (threadIdx.x < kAtH) {
            const int h = threadIdx.x;
            float mx = -INFINITY;
            for (int r = 0; r < CL; ++r)
                mx = fmaxf(mx, *cluster.map_shared_rank(&s.cm[h], r));
            float l = 0.f;
            for (int r = 0; r < CL; ++r) {
                const float mr = *cluster.map_shared_rank(&s.cm[h], r);
                if (mr != -INFINITY)
                    l = fmaf(*cluster.map_shared_rank(&s.cl[h], r), expf(mr - mx), l);
            }
            for (int r = 0; r < CL; ++r) {
                const float mr = *cluster.map_shared_rank(&s.cm[h], r);
                s.fac[h][r] = (mr == -INFINITY || !(l > 0.f)) ? 0.f : expf(mr - mx) / l;
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < G * (D / 4); e += kAtThreads) {
            const int h = e / (D / 4), i = 4 * (e - h * (D / 4));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < CL; ++r) {
                const float f = s.fac[h][r];
                if (f == 0.f)
                    continue;
                const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(&ob[h * D + i], r));
                acc.x = fmaf(v.x, f, acc.x);
                acc.y = fmaf(v.y, f, acc.y);
                acc.z = fmaf(v.z, f, acc.z);
                acc.w = fmaf(v.w, f, acc.w);
            }
            uint2 w;
            w.x = pack_bf16x2(acc.x, acc.y);
            w.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2*>(p.out + ((int64_t)seq * HQ + g * G + h) * D + i) = w;
        }
    }
    cluster.sync();   // peers stay until rank 0 has read them
}

}  // namespace

bool attend_supported(int head_dim, int G, int max_rank)
{
    return (head_dim == 64 || head_dim == 128) && G >= 1 && G <= kAtMaxG && max_rank >= 0 && max_rank <= 64;
}

// Cluster size.  One CTA fills an SM, and a cluster's CTAs must share a GPC, so
// the clusters that fit at once (the occupancy query) can fall short of the
// grid and push the last ones into another wave.  The CTAs of a cluster split
// the (sequence, head)'s tiles evenly, so each size 1..8 is costed as
// waves / CL and the cheapest taken (ties: the smaller cluster); `fallback` if
// the query is unavailable.  The occupancy answers are cached per kernel and
// device (cluster_fit), so a decode step pays only this arithmetic.
template <int D, int MP>
static int attend_pick_cluster(const AttendParams& p, int bytes, int fallback)
{
    const int64_t units = (int64_t)p.n_seqs * p.H;
    int best = fallback;
    double best_t = 1e300;
    for (int cl = 1; cl <= kAtMaxCL; ++cl) {
        const int fit = cluster_fit(reinterpret_cast<const void*>(attend_kernel<D, MP>), kAtThreads, bytes, cl);
        if (fit < 1)
            continue;
        const double t = (double)((units + fit - 1) / fit) / cl;
        if (t < best_t * 0.999) {
            best_t = t;
            best = cl;
        }
    }
    return best;
}

template <int D, int MP>
static cudaError_t launch_attend_m(const AttendParams& p0, cudaStream_t stream)
{
    AttendLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p = p0;
    AttendParams& p = L.p;
    L.wait_ns = wait_limit_ns();
    // key and value rows: [num_rows][H * d] (an empty store gets a one-row map no tile reads)
    const int64_t rows = p.num_rows > 0 ? p.num_rows : 1, width = (int64_t)p.H * D;
    if (!make_rows_map(&L.map_k, p.k, rows, width, p.row_stride, 64, kAtT) ||
        !make_rows_map(&L.map_v, p.v, rows, width, p.row_stride, 64, kAtT))
        return cudaErrorInvalidValue;
    static_assert(sizeof(AtSmem<D, MP>) + 1024 <= 227 * 1024, "attention tile buffers exceed shared memory");
    const int bytes = (int)sizeof(AtSmem<D, MP>) + 1024;   // + the 1024-byte alignment
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    p.cluster = attend_pick_cluster<D, MP>(p, bytes, p.cluster);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_seqs * p.cluster), (unsigned)p.H);
    cfg.blockDim = dim3(kAtThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attend_kernel<D, MP>, L);
}

template <int D>
static cudaError_t launch_attend_d(const AttendParams& p, cudaStream_t stream)
{
    if (p.max_rank == 0)
        return launch_attend_m<D, 0>(p, stream);
    if (p.max_rank <= 16)
        return launch_attend_m<D, 16>(p, stream);
    if (p.max_rank <= 32)
        return launch_attend_m<D, 32>(p, stream);
    return launch_attend_m<D, 64>(p, stream);
}

// Default cluster size (used when the occupancy query is unavailable): the
// smallest power of two (at most 8) that gives the grid about one CTA per SM.
int attend_cluster(int64_t units)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1)
        sms = 1;
    int cl = 1;
    while (cl < kAtMaxCL && units * cl < sms)
        cl *= 2;
    return cl;
}

cudaError_t launch_attend(const AttendParams& p, cudaStream_t stream)
{
    return p.d == 64 ? launch_attend_d<64>(p, stream) : launch_attend_d<128>(p, stream);
}

}  // namespace kamera
