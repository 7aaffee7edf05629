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
// so each row is read once for all of them.  The G query heads (padded to 16)
// are the rows of warp-level bf16 MMAs (m16n8k16, fp32 accumulate): a decode
// step has at most 8 query rows per KV head, far below the 64-row minimum of
// the tensor-memory MMA.  The per-chunk query part and the softmax weights are
// not bf16 values, so they enter as bf16 hi + lo pairs (about 16 significant
// bits); the rows and U rows are exact bf16.
//
// Tiles hold 128 tokens; warp w owns tokens 16w .. 16w + 15 of every
// tile and runs the whole of attention over them in registers: the scores
// S[16 x 16] = [R(-delta) q | V_k^T q] [k | u]^T, its own online softmax
// (running max and sum per head), and [O | W][16 x (d + m)] += P [v | u'] with
// the weights passed from the score fragments straight into the value MMA's
// A operand; W = sum_j p_j u'_j is folded through V_v when the chunk ends.
// A warp reads only its own 16 rows of a tile, so it also loads them itself,
// NS - 1 tiles ahead into its slice of a ring of NS tile buffers: the key and
// value rows as 128B-swizzled TMA boxes of 16 rows (lane 0 issues them), the U
// rows as 16-byte async copies into rows padded to an odd number of 16-byte
// vectors (both layouts keep the 8x8 matrix loads free of bank conflicts);
// one mbarrier per warp and buffer counts both, and every wait is bounded in
// time.  The warps meet only at chunk boundaries (the chunk's query part) and
// at the end, where their softmax states merge through shared memory.  The CTAs of a
// cluster split the (sequence, head)'s tiles evenly (a chunk cut between CTAs
// is set up by each, and each folds its own share of the value patch), CL
// chosen from the occupancy query so the grid runs in as few waves as
// possible (a cluster must sit in one GPC); rank 0 merges the CTAs' softmax
// states through distributed shared memory.
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

constexpr int kAtCW = 8;                       // warps: each owns 16 tokens of every tile
constexpr int kAtThreads = 32 * kAtCW;
constexpr int kAtT = 16 * kAtCW;               // tokens per tile
constexpr int kAtWR = 16;                      // rows per warp
constexpr int kAtH = 16;                       // MMA rows: a KV head's query heads, padded
constexpr int kAtMaxG = 8;                     // query heads per KV head
constexpr int kAtMaxCL = 8;

// D: head dim (64 or 128); MP: the padded rank the instantiation takes (0, 16, 32, 64).
// The canonical rows of a tile arrive by TMA as 128B-swizzled boxes of 64
// columns x 16 tokens, one per warp (16-byte piece c of row r at piece
// c ^ (r & 7)); the U rows by 16-byte async copies into rows padded to an odd
// number of 16-byte vectors.
template <int D, int MP>
struct AtSmem {
    static constexpr int KW = D + MP;    // tile row: k | u (key side), v | u' (value side)
    static constexpr int NB = D / 64;    // 64-column boxes of a head row
    static constexpr int RS = KW + 8;    // query-part row stride: an odd number of 16-byte vectors
    static constexpr int NT = KW / 8;    // 8-column tiles of the value side
    static constexpr int URS = MP + 8;   // U row stride
    static constexpr int UB = MP > 0 ? 1 : 0;
    static constexpr uint32_t kBoxBytes = kAtT * 128;
    static constexpr uint32_t kBufBytes = 2 * NB * kBoxBytes + UB * 2 * kAtT * URS * 2;
    static constexpr int NS = kBufBytes <= 48 * 1024 ? 4 : kBufBytes <= 64 * 1024 ? 3 : 2;   // tile buffers
    __nv_bfloat16 kt[NS][NB][kAtT][64];  // key rows (TMA boxes); the warps' partial outputs at the end
    __nv_bfloat16 vt[NS][NB][kAtT][64];  // value rows; the CTA's output at the end
    __nv_bfloat16 ut[UB ? NS : 1][kAtT][URS];   // U rows of the key side
    __nv_bfloat16 uv[UB ? NS : 1][kAtT][URS];   // U' rows of the value side
    __nv_bfloat16 xh[kAtH][RS];          // per-chunk query part R(-delta) q | V_k^T q, bf16 hi
    __nv_bfloat16 xl[kAtH][RS];          // and lo
    __nv_bfloat16 q[kAtH][D];            // the queries (target frame; rows past G zero)
    float2 cs[D / 2];                    // cos/sin of -delta
    float wm[kAtCW][kAtH], wl[kAtCW][kAtH];   // the warps' softmax states
    float wf[kAtH][kAtCW];               // their merge weights
    float cm[kAtH], cl[kAtH];            // this CTA's softmax state, for the cluster merge
    float fac[kAtH][kAtMaxCL];           // cluster merge weights (rank 0)
    uint64_t full[kAtCW][NS];            // warp w's rows of buffer b: TMA bytes + its lanes' copies
    int32_t abort;                       // a wait ran out: every later wait returns at once
};

// The launch: parameters and the tensor maps of the key and value rows
// ([num_rows][H * d], boxes of 64 columns x 16 rows).
struct AttendLaunch {
    AttendParams p;
    CUtensorMap map_k, map_v;
    uint64_t wait_ns;
    float* ws;       // split path: the partial softmax states (NULL: the cluster path)
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

// The CTA's share of a sequence: tiles [lo, hi) of its valid chunks' tiles in
// order; for chunk c (nt tiles, pos tiles before it) the tiles [t_lo, t_hi).
__device__ __forceinline__ void share_of_chunk(int64_t lo, int64_t hi, int64_t pos, int nt, int& t_lo, int& t_hi)
{
    const int64_t a0 = lo - pos, a1 = hi - pos;
    t_lo = a0 > 0 ? (int)a0 : 0;
    t_hi = a1 < nt ? (int)a1 : nt;
}

// Moves (c, tl) to the next tile of the CTA's share (t_hi: end of chunk c's
// share, pos: tiles of the sequence before chunk c + 1); false past the last.
__device__ __forceinline__ bool next_tile(const AttendParams& p, int c1, int64_t lo, int64_t hi, int& c, int& tl,
                                          int& t_hi, int64_t& pos)
{
    if (++tl < t_hi)
        return true;
    for (++c; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        if (attend_check(ch, c, p))
            continue;
        const int nt = (ch.len + kAtT - 1) / kAtT;
        int a, b;
        share_of_chunk(lo, hi, pos, nt, a, b);
        pos += nt;
        if (a < b) {
            tl = a;
            t_hi = b;
            return true;
        }
    }
    return false;
}

// Warp w starts the copies of its rows (16w .. 16w + 15) of tile tl of chunk c
// into buffer b: lane 0 the TMA boxes of the key and value rows (rows past the
// chunk come from the store or read as zero: the warp clears the value rows
// past it once they land), every lane the async copies of U rows whose rank
// is a multiple of 8.  Nothing when the chunk ends before the warp's rows.
template <int D, int MP>
__device__ __forceinline__ void warp_load(const AttendLaunch& P, AtSmem<D, MP>& s, int c, int tl, int g, int warp,
                                          int lane, int b)
{
    using SM = AtSmem<D, MP>;
    const AttendParams& p = P.p;
    const KameraChunk& ch = p.chunks[c];
    const int len = ch.len, m = ch.rank, j0 = tl * kAtT, r0 = kAtWR * warp;
    const int n = min(kAtT, len - j0);
    if (r0 >= n)
        return;
    const uint32_t full = ptx::smem_addr(&s.full[warp][b]);
    if (lane == 0) {
        const int y = (int)(ch.src_offset + j0 + r0);
        ptx::mbar_arrive_expect_tx(full, 2u * SM::NB * kAtWR * 128u);
#pragma unroll
        for (int x = 0; x < SM::NB; ++x) {
            ptx::tma_load_2d(ptx::smem_addr(&s.kt[b][x][r0][0]), &P.map_k, g * D + 64 * x, y, full);
            ptx::tma_load_2d(ptx::smem_addr(&s.vt[b][x][r0][0]), &P.map_v, g * D + 64 * x, y, full);
        }
    }
    if constexpr (MP > 0) {
        if (m > 0 && (m & 7) == 0) {
            const int64_t fo = ((int64_t)(p.layer * p.H + g) * len + j0) * m;   // U [L][H][len][m]
            const __nv_bfloat16* uk = patch_ptr(ch, 0) + fo;
            const __nv_bfloat16* uvp = patch_ptr(ch, 2) + fo;
            const int vpr = m >> 3, rows = min(kAtWR, n - r0);
            for (int e = lane; e < rows * vpr; e += 32) {
                const int t = r0 + e / vpr, v = e - (e / vpr) * vpr;
                ptx::cp_async16(ptx::smem_addr(&s.ut[b][t][8 * v]), uk + (int64_t)t * m + 8 * v);
                ptx::cp_async16(ptx::smem_addr(&s.uv[b][t][8 * v]), uvp + (int64_t)t * m + 8 * v);
            }
        }
    }
    ptx::cp_async_mbar_arrive_noinc(full);
}

template <int D, int MP>
__global__ void __launch_bounds__(kAtThreads, 1) attend_kernel(const __grid_constant__ AttendLaunch P)
{
    using SM = AtSmem<D, MP>;
    constexpr int NT = SM::NT, NS = SM::NS;
    const AttendParams& p = P.p;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // swizzled TMA boxes want 1024-byte alignment (the same offset in every CTA)
    SM& s = *reinterpret_cast<SM*>(smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u));
    namespace cg = cooperative_groups;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, t4 = lane & 3;
    const int G = p.G, HQ = p.H * G;
    // 8x8 matrix-load addressing of a row-major 16 x 16 A operand
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
    // The units this CTA serves (unit u: sequence u / H, KV head u % H).  Cluster
    // path: one unit, its tiles split evenly over the cluster's CTAs by rank.  Split
    // path: CTA k of NC takes the unit-fraction range [k U / NC, (k + 1) U / NC) and
    // leaves one partial softmax state per unit it touches in the workspace (slot
    // k + u); a second kernel merges them.
    const bool split = P.ws != nullptr;
    const int CL = split ? 1 : p.cluster, rank = split ? 0 : (int)(blockIdx.x % (unsigned)CL);
    const int64_t U = (int64_t)p.n_seqs * p.H, NC = gridDim.x, kc = blockIdx.x;
    const int64_t u_begin = split ? kc * U / NC : (int64_t)(blockIdx.x / CL) * p.H + blockIdx.y;
    const int64_t u_end = split ? ((kc + 1) * U + NC - 1) / NC : u_begin + 1;

    if (threadIdx.x == 0) {
        for (int w = 0; w < kAtCW; ++w)
            for (int b = 0; b < NS; ++b)
                ptx::mbar_init(ptx::smem_addr(&s.full[w][b]), 1 + 32);   // the TMA issue + the lanes' copies
        s.abort = 0;
        ptx::fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        ptx::prefetch_tmap(&P.map_k);
        ptx::prefetch_tmap(&P.map_v);
    }
    const RopeParams& rp = p.rope;
    uint32_t ph = 0;   // phase parity of this warp's barrier per buffer (kept across units)

    for (int64_t u = u_begin; u < u_end; ++u) {
    const int seq = (int)(u / p.H), g = (int)(u % p.H);
    int c0 = p.seq_start[seq], c1 = p.seq_start[seq + 1];
    if (c0 < 0 || c1 < c0 || c1 > p.n_chunks) {
        if (g == 0 && rank == 0 && threadIdx.x == 0 && (!split || kc * U <= u * NC))
            raise_err(p.err, KAMERA_DEVERR_DESCRIPTOR);
        c0 = c1 = 0;
    }
    int64_t total = 0;
    for (int c = c0; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        if (!attend_check(ch, c, p))
            total += (ch.len + kAtT - 1) / kAtT;
    }
    // this CTA's share of the unit's tiles; `first`: the share that starts the unit
    int64_t lo, hi;
    bool first;
    if (split) {
        const int64_t a = max(kc * U, u * NC), e = min((kc + 1) * U, (u + 1) * NC);
        lo = total * (a - u * NC) / NC;
        hi = total * (e - u * NC) / NC;
        first = a == u * NC;
    } else {
        lo = total * rank / CL;
        hi = total * (rank + 1) / CL;
        first = rank == 0;
    }

    __syncthreads();   // the previous unit is done with every shared array (first: barriers initialised)
    for (int e = threadIdx.x; e < kAtH * D; e += kAtThreads) {
        const int h = e / D, i = e - h * D;
        s.q[h][i] = h < G ? p.q[((int64_t)seq * HQ + g * G + h) * D + i] : __float2bfloat16_rn(0.f);
    }

    {
        // ------------------------------------------------------------ the warps
        float o[NT][4];   // [O | W] of this warp's tokens: column tile j, rows gq and gq + 8
#pragma unroll
        for (int j = 0; j < NT; ++j)
            o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};   // heads gq, gq + 8
        const int ro = rp.rot_offset, rr = rp.rot_dim, half = rr / 2;
        const uint32_t kt0 = ptx::smem_addr(&s.kt[0][0][0][0]), vt0 = ptx::smem_addr(&s.vt[0][0][0][0]);
        const uint32_t ut0 = ptx::smem_addr(&s.ut[0][0][0]), uv0 = ptx::smem_addr(&s.uv[0][0][0]);
        constexpr uint32_t kBuf = SM::NB * SM::kBoxBytes;               // bytes per row buffer
        constexpr uint32_t kUBuf = (uint32_t)(kAtT * SM::URS * 2);      // bytes per U buffer
        const int r0 = 16 * warp;                                       // this warp's first token row
        // score B operand (key rows): matrices (tokens 0-7 | 8-15) x (k 0-7 | 8-15)
        const int kr = r0 + (lane & 7) + 8 * (lane >> 4), khi = (lane >> 3) & 1;
        const uint32_t klx = (uint32_t)(khi ^ (lane & 7));
        // value B operand (value rows, transposed): (tokens 0-7 | 8-15) x (tile j | j + 1)
        const int vr = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const uint32_t vlx = (uint32_t)((lane >> 4) ^ (lane & 7));
        const uint32_t xa = ptx::smem_addr(&s.xh[arow][acol]), xla = ptx::smem_addr(&s.xl[arow][acol]);

        // load cursor: the tile NS - 1 ahead of the one being computed
        int lc = c0 - 1, ltl = 0, lthi = 0;
        int64_t lpos = 0;
        bool lmore = next_tile(p, c1, lo, hi, lc, ltl, lthi, lpos);
        for (int j = 0; j < NS - 1 && lmore; ++j) {
            warp_load<D, MP>(P, s, lc, ltl, g, warp, lane, j);
            lmore = next_tile(p, c1, lo, hi, lc, ltl, lthi, lpos);
        }
        int gi = 0;
        int64_t pos = 0;
        for (int c = c0; c < c1; ++c) {
            const KameraChunk& ch = p.chunks[c];
            const int32_t bad = attend_check(ch, c, p);
            if (bad) {
                if (first && threadIdx.x == 0)
                    raise_err(p.err, bad);
                continue;
            }
            const int len = ch.len, nt = (len + kAtT - 1) / kAtT, m = ch.rank;
            int t_lo, t_hi;
            share_of_chunk(lo, hi, pos, nt, t_lo, t_hi);
            pos += nt;
            if (t_lo >= t_hi)
                continue;
            const int64_t fo = (int64_t)(p.layer * p.H + g) * D * m;   // this (layer, head)'s V factors [d][m]
            // ---- the chunk's query part (every warp is done with the previous one)
            __syncthreads();
            for (int f = threadIdx.x; f < rp.n_freq; f += kAtThreads) {
                float cc, sn;
                phase_cos_sin(-freq_delta(rp, ch, c, f), rp.inv_freq[f], cc, sn);
                s.cs[f] = make_float2(cc, sn);
            }
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
                    const uint16_t* vkg = reinterpret_cast<const uint16_t*>(patch_ptr(ch, 1) + fo);   // V_k [d][m]
                    const int r = 8 * warp + gq;
                    float y[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t qa = ptx::smem_addr(&s.q[arow][acol]);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t a[4];
                        ldsm_x4(qa + 32 * ks, a);
                        const int i0 = 16 * ks + 2 * t4;
                        uint32_t b0 = 0, b1 = 0;
                        if (r < m) {
                            b0 = (uint32_t)vkg[(int64_t)i0 * m + r] | ((uint32_t)vkg[(int64_t)(i0 + 1) * m + r] << 16);
                            b1 = (uint32_t)vkg[(int64_t)(i0 + 8) * m + r] |
                                 ((uint32_t)vkg[(int64_t)(i0 + 9) * m + r] << 16);
                        }
                        mma_bf16(y, a, b0, b1);
                    }
                    const int col = D + 8 * warp + 2 * t4;   // rows gq, gq + 8 (heads); columns col, col + 1
                    split1(y[0], s.xh[gq][col], s.xl[gq][col]);
                    split1(y[1], s.xh[gq][col + 1], s.xl[gq][col + 1]);
                    split1(y[2], s.xh[gq + 8][col], s.xl[gq + 8][col]);
                    split1(y[3], s.xh[gq + 8][col + 1], s.xl[gq + 8][col + 1]);
                }
            }
            __syncthreads();

            for (int tl = t_lo; tl < t_hi; ++tl, ++gi) {
                const int b = gi % NS, j0 = tl * kAtT, ntok = min(kAtT, len - j0);
                if (lmore) {   // tile gi + NS - 1 into the buffer tile gi - 1 has left
                    warp_load<D, MP>(P, s, lc, ltl, g, warp, lane, (gi + NS - 1) % NS);
                    lmore = next_tile(p, c1, lo, hi, lc, ltl, lthi, lpos);
                }
                const uint32_t kb = kt0 + b * kBuf, vb = vt0 + b * kBuf;
                const uint32_t ub = ut0 + (SM::UB ? b : 0) * kUBuf, uvb = uv0 + (SM::UB ? b : 0) * kUBuf;
                const bool active = r0 < ntok;
                if (active) {
                    tile_wait(ptx::smem_addr(&s.full[warp][b]), (ph >> b) & 1u, &s.abort, p.err, P.wait_ns);
                    ph ^= 1u << b;
                    // ---- this warp's rows of the buffer: U rows of ranks that are not whole
                    // 16-byte vectors, U columns past the rank, value rows past the chunk
                    if constexpr (MP > 0) {
                        if ((m & 7) != 0) {   // ranks that are not whole 16-byte vectors: element copies
                            const int64_t fu = ((int64_t)(p.layer * p.H + g) * len + j0) * m;
                            const __nv_bfloat16* uk = patch_ptr(ch, 0) + fu;
                            const __nv_bfloat16* uvp = patch_ptr(ch, 2) + fu;
                            for (int e = lane; e < 16 * MP; e += 32) {
                                const int t = r0 + e / MP, k = e % MP;
                                const bool in = t < ntok && k < m;
                                s.ut[b][t][k] = in ? uk[(int64_t)t * m + k] : __float2bfloat16_rn(0.f);
                                s.uv[b][t][k] = in ? uvp[(int64_t)t * m + k] : __float2bfloat16_rn(0.f);
                            }
                        } else if (m < MP) {
                            const int zv = (MP - m) >> 3;
                            for (int e = lane; e < 16 * zv; e += 32) {
                                const int t = r0 + e / zv, v = (m >> 3) + e % zv;
                                ptx::st_shared_zero16(ptx::smem_addr(&s.ut[b][t][8 * v]));
                                ptx::st_shared_zero16(ptx::smem_addr(&s.uv[b][t][8 * v]));
                            }
                        }
                    }
                    if (ntok < r0 + 16) {   // value rows past the chunk: zero, so zero weights add nothing
                        const int nz = r0 + 16 - ntok;
                        for (int e = lane; e < nz * 8 * SM::NB; e += 32) {
                            const int t = ntok + e / (8 * SM::NB), c8 = e % (8 * SM::NB);
                            ptx::st_shared_zero16(vb + (c8 >> 3) * SM::kBoxBytes + t * 128 + (c8 & 7) * 16);
                        }
                        if constexpr (MP > 0)
                            for (int e = lane; e < nz * (MP / 8); e += 32)
                                ptx::st_shared_zero16(
                                    ptx::smem_addr(&s.uv[b][ntok + e / (MP / 8)][8 * (e % (MP / 8))]));
                    }
                    __syncwarp();

                    // ---- scores S[16 heads x 16 tokens]: two 8-token column tiles, the hi and
                    // lo products in separate chains (padded U columns add exact zeros at
                    // their ends, so every instantiation gives the same scores)
                    float sa[2][2][4];
#pragma unroll
                    for (int nt2 = 0; nt2 < 2; ++nt2)
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            sa[nt2][u][0] = sa[nt2][u][1] = sa[nt2][u][2] = sa[nt2][u][3] = 0.f;
                    const uint32_t krow = kb + (uint32_t)(kr * 128);
                    const uint32_t urow = ub + (uint32_t)((kr * SM::URS + 8 * khi) * 2);
                    auto score_step = [&](uint32_t baddr, int ks) {
                        uint32_t bb[4], ah[4], al[4];
                        ldsm_x4(baddr, bb);
                        ldsm_x4(xa + 32 * ks, ah);
                        ldsm_x4(xla + 32 * ks, al);
                        mma_bf16(sa[0][0], ah, bb[0], bb[1]);
                        mma_bf16(sa[0][1], al, bb[0], bb[1]);
                        mma_bf16(sa[1][0], ah, bb[2], bb[3]);
                        mma_bf16(sa[1][1], al, bb[2], bb[3]);
                    };
#pragma unroll 4
                    for (int ks = 0; ks < D / 16; ++ks)   // key rows
                        score_step(krow + (uint32_t)(ks >> 2) * SM::kBoxBytes + ((((uint32_t)(2 * ks) & 7u) ^ klx) << 4),
                                   ks);
#pragma unroll 4
                    for (int ks = D / 16; ks < SM::KW / 16; ++ks)   // U rows
                        score_step(urow + 32 * (ks - D / 16), ks);

                    // ---- online softmax over this warp's 16 tokens (rows gq, gq + 8)
                    float e[2][4], mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int nt2 = 0; nt2 < 2; ++nt2)
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            const int tok = r0 + 8 * nt2 + 2 * t4 + (f & 1);
                            const float sc = sa[nt2][0][f] + sa[nt2][1][f];
                            e[nt2][f] = tok < ntok ? p.scale * sc : -INFINITY;
                            mx[f >> 1] = fmaxf(mx[f >> 1], e[nt2][f]);
                        }
                    float alpha[2], sum[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                        const float mnew = fmaxf(m_run[r], mx[r]);   // finite: token r0 is in the chunk
                        alpha[r] = __expf(m_run[r] - mnew);         // 0 while nothing was seen
                        m_run[r] = mnew;
                        sum[r] = 0.f;
                    }
#pragma unroll
                    for (int nt2 = 0; nt2 < 2; ++nt2)
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            e[nt2][f] = __expf(e[nt2][f] - m_run[f >> 1]);
                            sum[f >> 1] += e[nt2][f];
                        }
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 1);
                        sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 2);
                        l_run[r] = fmaf(l_run[r], alpha[r], sum[r]);
                    }
                    if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {   // a new running max
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            o[j][0] *= alpha[0];
                            o[j][1] *= alpha[0];
                            o[j][2] *= alpha[1];
                            o[j][3] *= alpha[1];
                        }
                    }
                    // the weights as the A operand (heads x tokens), hi + lo
                    uint32_t ph[4], pl[4];
                    split_hl(e[0][0], e[0][1], ph[0], pl[0]);
                    split_hl(e[0][2], e[0][3], ph[1], pl[1]);
                    split_hl(e[1][0], e[1][1], ph[2], pl[2]);
                    split_hl(e[1][2], e[1][3], ph[3], pl[3]);

                    // ---- [O | W] += P [v | u']: column tiles in pairs
                    const uint32_t vrow = vb + (uint32_t)(vr * 128);
                    const uint32_t uvrow = uvb + (uint32_t)((vr * SM::URS + 8 * (lane >> 4)) * 2);
#pragma unroll
                    for (int j = 0; j < NT; j += 2) {
                        uint32_t bb[4];
                        if (j < D / 8)
                            ldsm_x4_t(vrow + (uint32_t)(j >> 3) * SM::kBoxBytes + ((((uint32_t)j & 7u) ^ vlx) << 4), bb);
                        else
                            ldsm_x4_t(uvrow + 16 * (j - D / 8), bb);
                        mma_bf16(o[j], ph, bb[0], bb[1]);
                        mma_bf16(o[j], pl, bb[0], bb[1]);
                        mma_bf16(o[j + 1], ph, bb[2], bb[3]);
                        mma_bf16(o[j + 1], pl, bb[2], bb[3]);
                    }
                    if (ntok < r0 + 16)
                        ptx::fence_proxy_async();   // zeroed rows precede a later TMA refill of the buffer
                }
                __syncwarp();   // the warp is done with its rows of buffer b before it refills them
            }
            if constexpr (MP > 0) {
                if (m > 0) {   // fold W = sum_j p_j u'_j through V_v: O += W V_v^T (W's fragments -> A operand)
                    const uint16_t* vvg = reinterpret_cast<const uint16_t*>(patch_ptr(ch, 3) + fo);   // V_v [d][m]
#pragma unroll
                    for (int kk = 0; kk < MP / 16; ++kk) {
                        const int j0 = D / 8 + 2 * kk, q0 = 16 * kk + 2 * t4;
                        uint32_t ah[4], al[4];
                        split_hl(o[j0][0], o[j0][1], ah[0], al[0]);
                        split_hl(o[j0][2], o[j0][3], ah[1], al[1]);
                        split_hl(o[j0 + 1][0], o[j0 + 1][1], ah[2], al[2]);
                        split_hl(o[j0 + 1][2], o[j0 + 1][3], ah[3], al[3]);
#pragma unroll
                        for (int j = 0; j < D / 8; ++j) {
                            const uint16_t* vrw = vvg + (int64_t)(8 * j + gq) * m;
                            const uint32_t b0 = (q0 < m ? (uint32_t)vrw[q0] : 0u) |
                                                ((q0 + 1 < m ? (uint32_t)vrw[q0 + 1] : 0u) << 16);
                            const uint32_t b1 = (q0 + 8 < m ? (uint32_t)vrw[q0 + 8] : 0u) |
                                                ((q0 + 9 < m ? (uint32_t)vrw[q0 + 9] : 0u) << 16);
                            mma_bf16(o[j], ah, b0, b1);
                            mma_bf16(o[j], al, b0, b1);
                        }
                    }
#pragma unroll
                    for (int j = D / 8; j < NT; ++j)
                        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
                }
            }
        }
        // ---- publish this warp's state for the CTA merge (after every tile is consumed)
        ptx::cp_async_wait<0>();
        __syncthreads();   // no tile buffer is in use any more
        float* ow = reinterpret_cast<float*>(&s.kt[0][0][0][0]);   // [kAtCW][kAtH][D]
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            const int col = 8 * j + 2 * t4;
            *reinterpret_cast<float2*>(&ow[(warp * kAtH + gq) * D + col]) = make_float2(o[j][0], o[j][1]);
            *reinterpret_cast<float2*>(&ow[(warp * kAtH + gq + 8) * D + col]) = make_float2(o[j][2], o[j][3]);
        }
        if (t4 == 0) {
            s.wm[warp][gq] = m_run[0];
            s.wm[warp][gq + 8] = m_run[1];
            s.wl[warp][gq] = l_run[0];
            s.wl[warp][gq + 8] = l_run[1];
        }
    }
    __syncthreads();   // every warp's state published

    // ---- CTA merge of the warps' softmax states -> (cm, cl, ob)
    float* ow = reinterpret_cast<float*>(&s.kt[0][0][0][0]);
    float* ob = reinterpret_cast<float*>(&s.vt[0][0][0][0]);   // [kAtH][D]
    if (threadIdx.x < kAtH) {
        const int h = threadIdx.x;
        float mx = -INFINITY;
        for (int w = 0; w < kAtCW; ++w)
            mx = fmaxf(mx, s.wm[w][h]);
        float l = 0.f;
        for (int w = 0; w < kAtCW; ++w) {
            const float f = s.wm[w][h] == -INFINITY ? 0.f : expf(s.wm[w][h] - mx);
            s.wf[h][w] = f;
            l = fmaf(s.wl[w][h], f, l);
        }
        s.cm[h] = mx;
        s.cl[h] = l;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kAtH * D; e += kAtThreads) {
        const int h = e / D;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kAtCW; ++w)
            acc = fmaf(ow[(w * kAtH) * D + e], s.wf[h][w], acc);
        ob[e] = acc;
    }

    if (split) {   // ---- this CTA's partial state of unit u -> workspace slot k + u
        float* wp = P.ws + (size_t)(kc + u) * (2 * kAtH + kAtH * D);
        __syncthreads();
        if (threadIdx.x < kAtH) {
            wp[threadIdx.x] = s.cm[threadIdx.x];
            wp[kAtH + threadIdx.x] = s.cl[threadIdx.x];
        }
        for (int e = threadIdx.x; e < kAtH * D / 4; e += kAtThreads)
            reinterpret_cast<float4*>(wp + 2 * kAtH)[e] = reinterpret_cast<const float4*>(ob)[e];
        ptx::fence_proxy_async();   // the merge's shared writes precede the next unit's TMA refills
        continue;
    }
    // ---- cluster merge: every CTA publishes (max, sum, unnormalised output); rank 0 combines
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
}

// Merge of the split path, one CTA per (unit u, head h): the CTAs k that
// overlapped u (k U / NC < u + 1 and (k + 1) U / NC > u) left (max, sum,
// unnormalised output) per head in slot k + u; out = sum_k e^(m_k - M) O_k /
// sum_k e^(m_k - M) l_k, rounded once to bf16.  Unit u's rows start at row
// (u / groups) Hq + (u % groups) 16 of `out` ([*][dout]); `rows` of them.
__global__ void __launch_bounds__(128) attend_merge_kernel(const float* __restrict__ ws, int64_t U, int64_t NC,
                                                           int dout, int groups, int Hq, int rows_max,
                                                           __nv_bfloat16* __restrict__ out)
{
    constexpr int kMaxK = 64;   // overlapping CTAs whose weights are staged (more: computed in place)
    __shared__ float wf[kMaxK];
    __shared__ float stat[2];
    const int64_t u = blockIdx.x;
    const int h = blockIdx.y;
    const int grp = (int)(u % groups), rows = min(rows_max, Hq - grp * kAtH);
    if (h >= rows)
        return;
    const int64_t k_lo = u * NC / U, k_hi = ((u + 1) * NC + U - 1) / U;   // CTAs [k_lo, k_hi)
    const int nk = (int)(k_hi - k_lo);
    const size_t slot = (size_t)(2 * kAtH + kAtH * dout);
    const float* w0 = ws + (size_t)(k_lo + u) * slot;   // slot of CTA k_lo; CTA k_lo + i is i slots on
    if (threadIdx.x == 0) {
        float m = -INFINITY;
        for (int i = 0; i < nk; ++i)
            m = fmaxf(m, w0[(size_t)i * slot + h]);
        float l = 0.f;
        for (int i = 0; i < nk; ++i) {
            const float mk = w0[(size_t)i * slot + h];
            if (mk != -INFINITY)
                l = fmaf(w0[(size_t)i * slot + kAtH + h], expf(mk - m), l);
        }
        stat[0] = m;
        stat[1] = l;
    }
    __syncthreads();
    const float m = stat[0], l = stat[1];
    for (int i = threadIdx.x; i < min(nk, kMaxK); i += blockDim.x) {
        const float mk = w0[(size_t)i * slot + h];
        wf[i] = (mk == -INFINITY || !(l > 0.f)) ? 0.f : expf(mk - m) / l;
    }
    __syncthreads();
    const int64_t row = (u / groups) * Hq + grp * kAtH + h;
    for (int i = 4 * threadIdx.x; i < dout; i += 4 * blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < nk; ++k) {
            float f;
            if (k < kMaxK) {
                f = wf[k];
            } else {
                const float mk = w0[(size_t)k * slot + h];
                f = (mk == -INFINITY || !(l > 0.f)) ? 0.f : expf(mk - m) / l;
            }
            if (f == 0.f)
                continue;
            const float4 v = *reinterpret_cast<const float4*>(w0 + (size_t)k * slot + 2 * kAtH + h * dout + i);
            acc.x = fmaf(v.x, f, acc.x);
            acc.y = fmaf(v.y, f, acc.y);
            acc.z = fmaf(v.z, f, acc.z);
            acc.w = fmaf(v.w, f, acc.w);
        }
        uint2 w;
        w.x = pack_bf16x2(acc.x, acc.y);
        w.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(out + row * dout + i) = w;
    }
}

}  // namespace

cudaError_t launch_attend_merge(const float* ws, int64_t units, int64_t ctas, int dout, int groups, int Hq,
                                int rows, __nv_bfloat16* out, cudaStream_t stream)
{
    if (units < 1)
        return cudaSuccess;
    attend_merge_kernel<<<dim3((unsigned)units, (unsigned)rows), 128, 0, stream>>>(ws, units, ctas, dout, groups, Hq,
                                                                                    rows, out);
    return cudaGetLastError();
}

size_t attend_slot_bytes(int dout) { return sizeof(float) * (size_t)(2 * kAtH + kAtH * dout); }

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
static int attend_pick_cluster(const AttendParams& p, int bytes, int fallback, double& best_t)
{
    const int64_t units = (int64_t)p.n_seqs * p.H;
    int best = fallback;
    best_t = 1e300;
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

// Split path or cluster path.  With a workspace, the split path spreads the
// units' tiles over every CTA that fits at once (NC), evenly to a tile, at the
// cost of a second, small launch that merges the partial states: its time is
// U / NC units against the cluster path's waves / CL; it is taken when that is
// at least 3% less.
template <int D, int MP>
static cudaError_t launch_attend_m(const AttendParams& p0, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    AttendLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p = p0;
    AttendParams& p = L.p;
    L.wait_ns = wait_limit_ns();
    // key and value rows: [num_rows][H * d] (an empty store gets a one-row map no tile reads)
    const int64_t rows = p.num_rows > 0 ? p.num_rows : 1, width = (int64_t)p.H * D;
    if (!make_rows_map(&L.map_k, p.k, rows, width, p.row_stride, 64, kAtWR) ||
        !make_rows_map(&L.map_v, p.v, rows, width, p.row_stride, 64, kAtWR))
        return cudaErrorInvalidValue;
    static_assert(sizeof(AtSmem<D, MP>) + 1024 <= 227 * 1024, "attention tile buffers exceed shared memory");
    const int bytes = (int)sizeof(AtSmem<D, MP>) + 1024;   // + the 1024-byte alignment
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    double t_cluster;
    p.cluster = attend_pick_cluster<D, MP>(p, bytes, p.cluster, t_cluster);
    const int64_t units = (int64_t)p.n_seqs * p.H;
    const int nc = cluster_fit(reinterpret_cast<const void*>(attend_kernel<D, MP>), kAtThreads, bytes, 1);
    if (ws && nc >= 1 && (size_t)(nc + units - 1) * attend_slot_bytes(D) <= ws_bytes &&
        (double)units / nc < 0.97 * t_cluster) {
        L.ws = static_cast<float*>(ws);
        p.cluster = 1;
        attend_kernel<D, MP><<<(unsigned)nc, kAtThreads, bytes, stream>>>(L);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        return launch_attend_merge(L.ws, units, nc, D, 1, p.G, p.G, p.out, stream);
    }
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
static cudaError_t launch_attend_d(const AttendParams& p, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (p.max_rank == 0)
        return launch_attend_m<D, 0>(p, ws, ws_bytes, stream);
    if (p.max_rank <= 16)
        return launch_attend_m<D, 16>(p, ws, ws_bytes, stream);
    if (p.max_rank <= 32)
        return launch_attend_m<D, 32>(p, ws, ws_bytes, stream);
    return launch_attend_m<D, 64>(p, ws, ws_bytes, stream);
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

cudaError_t launch_attend(const AttendParams& p, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    return p.d == 64 ? launch_attend_d<64>(p, ws, ws_bytes, stream) : launch_attend_d<128>(p, ws, ws_bytes, stream);
}

}  // namespace kamera
