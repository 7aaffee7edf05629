// kamera_attend_mla.cu -- MLA decode attention over reused chunks, without the pool.
//
// The MLA rows the reuse equation gives (the gist.science technical summary,
// section 2; the MLA rule of section 3: c_KV is carried over, the decoupled
// k_rope turned) are, for token j of chunk c,
//     c'_j  = c_j + V_c u_j            (latent, kv_lora wide)
//     kr'_j = R(delta_c) kr_j + V_r w_j  (rope_dim wide)
// and absorbed MLA decode attends with the latent query (q_nope taken through
// the key up-projection) and the rope query:
//     score_hj = scale (q_lat_h . c'_j + q_rope_h . kr'_j),  out_h = sum_j p_hj c'_j
// (the caller takes out_h through the value up-projection).  The patch and the
// turn fold into per-chunk quantities, as for GQA attention:
//     q_lat . c'_j  = q_lat . c_j + (V_c^T q_lat) . u_j
//     q_rope . kr'_j = (R(-delta) q_rope) . kr_j + (V_r^T q_rope) . w_j
//     sum_j p_j c'_j = sum_j p_j c_j + V_c (sum_j p_j u_j)
// so a decode step streams the canonical rows and the U rows only.
//
// Every query head shares the one latent row, so the work is a dense
// contraction per 64-token tile: S[16 heads x 64 tokens] over the key width
// (kv_lora + rope_dim + 2 m), then O[16 x kv_lora] += P S-softmax'd x C.  The
// 16 query heads are the rows of warp-level bf16 MMAs (m16n8k16, fp32
// accumulate): a decode step has 16 query rows per latent head, below the
// 64-row minimum of the tensor-memory MMA, and the warp-level form keeps the
// score tile and the output accumulator in registers.  Warp w computes the
// scores of tokens 8w .. 8w + 7 against all 16 heads with the latent query held
// in registers for the whole kernel (loaded once), and owns output columns
// 64w .. 64w + 63.  Operands that are not bf16 already (the turned rope query,
// the folds, the softmax weights) enter as a bf16 hi + lo pair, so products
// keep about 16 bits of their fp32 value; the canonical rows and U rows are
// exact bf16.  Tiles are double-buffered: the 576-wide canonical rows arrive
// as nine 128B-swizzled TMA boxes of 64 columns x 64 tokens (one thread issues
// them; completion on an mbarrier, every wait bounded in time), the u and w
// rows as async copies into rows padded to an odd number of 16-byte vectors;
// both layouts put the eight rows an 8x8 matrix load reads in distinct banks.
// A cluster of CL CTAs serves one sequence, CTA
// r taking the r-th of CL even runs of the sequence's tiles (a chunk cut
// between two CTAs is set up by both, each folding its own share of the value
// patch); rank 0 merges the partial softmax states through distributed shared
// memory.  More than 16 query heads (DeepSeek-V3's 128) are served in groups of
// 16, one CTA row per group (grid y): each group is one more pass over the
// rows, and the clusters of all groups share the GPU in the same waves.
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

constexpr int kMlThreads = 256;
constexpr int kMlT = 64;             // tokens per tile
constexpr int kMlH = 16;             // query heads: the rows of every MMA
constexpr int kMlC = 512;            // kv_lora_rank
constexpr int kMlR = 64;             // rope_dim
constexpr int kMlDK = kMlC + kMlR;   // key width before the U columns
constexpr int kMlQS = kMlC + 8;      // staged latent-query row (elements)
constexpr int kMlMaxCL = 8;
constexpr int kMlMaxHeads = 128;     // query heads per latent row: groups of 16, one pass over the rows each

// MP: the padded rank the instantiation takes (0, 16 or 32).
template <int MP>
struct MlSmem {
    static constexpr int NBX = kMlDK / 64;      // 64-column boxes of a canonical row: c_KV (8) | k_rope (1)
    static constexpr int URS = 2 * MP + 8;      // u (V_c's factor) | w (V_r's) row: an odd number of 16-byte vectors
    static constexpr int XW = kMlR + 2 * MP;    // per-chunk query part: R(-delta) q_rope | V_c^T q_lat | V_r^T q_rope
    static constexpr int XS = XW + 8;
    static constexpr int MPa = MP > 0 ? MP : 1;
    static constexpr uint32_t kBoxBytes = kMlT * 128;
    __nv_bfloat16 kt[2][NBX][kMlT][64];         // canonical rows (TMA boxes); the latent queries at the
                                                // start; the partial outputs at the end
    __nv_bfloat16 ux[2][kMlT][URS];             // u | w rows
    __nv_bfloat16 xh[kMlH][XS];                 // per-chunk query part, bf16 hi
    __nv_bfloat16 xl[kMlH][XS];                 // and lo
    float sc[kMlH][kMlT + 4];                   // scores of the tile
    __nv_bfloat16 ph[kMlH][kMlT + 8];           // softmax weights, hi
    __nv_bfloat16 pl[kMlH][kMlT + 8];           // and lo
    float alpha[kMlH];                          // running-max rescale of the tile
    float qr[kMlH][kMlR];                       // q_rope of the sequence (fp32)
    float vr[kMlR][MPa];                        // V_r of the current chunk
    float wsum[kMlH][MPa];                      // sum_j p_j u_j of the chunk, at its end
    float2 cs[kMlR / 2];                        // cos/sin of -delta
    float cm[kMlH], cl[kMlH];                   // this CTA's softmax state, for the merge
    float fac[kMlH][kMlMaxCL];                  // merge weights (rank 0)
    uint64_t full[2];                           // buffer b's TMA boxes have landed
    int32_t abort;                              // a wait ran out: every later wait returns at once
};

// The launch: parameters and the tensor map of the canonical rows
// ([num_rows][kv_lora + rope_dim], boxes of 64 columns x 64 rows).
struct MlaLaunch {
    MlaAttendParams p;
    CUtensorMap map;
    uint64_t wait_ns;
    float* ws;       // split path: the partial softmax states (NULL: the cluster path)
};

__device__ __forceinline__ void st_shared_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t mla_check(const KameraChunk& ch, int c, const MlaAttendParams& p)
{
    int32_t bits = check_axis_delta(p.rope, c);
    if (ch.len < 0 || ch.rank < 0 || (ch.rank & 1) || ch.delta > KAMERA_MAX_ABS_DELTA ||
        ch.delta < -KAMERA_MAX_ABS_DELTA)
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

// Starts the copies of tile rows j0 .. j0 + n - 1 of chunk `ch` into buffer
// b: thread 0 issues the nine TMA boxes of the canonical rows (rows past the
// chunk come from the store or read as zero; the c_KV rows past n are cleared
// once they land), every thread the async copies of the u and w rows (zero past
// n and past the rank).  One copy group per call.
template <int MP>
__device__ __forceinline__ void mla_load(const MlaLaunch& P, const KameraChunk& ch, int j0, int n, int b,
                                         MlSmem<MP>& s)
{
    using SM = MlSmem<MP>;
    const MlaAttendParams& p = P.p;
    if (threadIdx.x == 0) {
        const uint32_t bar = ptx::smem_addr(&s.full[b]);
        const int y = (int)(ch.src_offset + j0);
        ptx::mbar_arrive_expect_tx(bar, SM::NBX * SM::kBoxBytes);
#pragma unroll
        for (int x = 0; x < SM::NBX; ++x)
            ptx::tma_load_2d(ptx::smem_addr(&s.kt[b][x][0][0]), &P.map, 64 * x, y, bar);
    }
    if constexpr (MP > 0) {   // u and w rows: MP / 2 words each (the rank is even)
        const int m = ch.rank;
        const int64_t fo = ((int64_t)p.layer * ch.len + j0) * m;   // U [L][len][m]
        const __nv_bfloat16* uc = patch_ptr(ch, 0);
        const __nv_bfloat16* ur = patch_ptr(ch, 2);
        for (int e = threadIdx.x; e < kMlT * MP; e += kMlThreads) {
            const int t = e / MP, wd = e - t * MP;
            const int f = wd >= MP / 2 ? 1 : 0, c2 = 2 * (wd - f * (MP / 2));
            const uint32_t dst = ptx::smem_addr(&s.ux[b][t][f * MP + c2]);
            if (t < n && c2 < m)
                ptx::cp_async_small<4>(dst, (f ? ur : uc) + fo + (int64_t)t * m + c2);
            else
                st_shared_u32(dst, 0u);
        }
    }
    ptx::cp_async_commit();
}

template <int MP>
__global__ void __launch_bounds__(kMlThreads, 1) mla_attend_kernel(const __grid_constant__ MlaLaunch P)
{
    using SM = MlSmem<MP>;
    const MlaAttendParams& p = P.p;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // swizzled TMA boxes want 1024-byte alignment (the same offset in every CTA)
    SM& s = *reinterpret_cast<SM*>(smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u));
    namespace cg = cooperative_groups;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int Hq = p.Hq, groups = (Hq + kMlH - 1) / kMlH;
    // 8x8 matrix-load addressing: A (row-major 16 x 16) and B^T (token rows)
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
    // The units this CTA serves (unit u: sequence u / groups, head group u % groups).
    // Cluster path: one unit, its tiles split evenly over the cluster's CTAs by rank.
    // Split path: CTA k of NC takes the unit-fraction range [k U / NC, (k + 1) U / NC)
    // and leaves one partial softmax state per unit it touches in the workspace
    // (slot k + u); a second kernel merges them.
    const bool split = P.ws != nullptr;
    const int CL = split ? 1 : p.cluster, rank = split ? 0 : (int)(blockIdx.x % (unsigned)CL);
    const int64_t U = (int64_t)p.n_seqs * groups, NC = gridDim.x, kc = blockIdx.x;
    const int64_t u_begin = split ? kc * U / NC : (int64_t)(blockIdx.x / CL) * groups + blockIdx.y;
    const int64_t u_end = split ? ((kc + 1) * U + NC - 1) / NC : u_begin + 1;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&s.full[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&s.full[1]), 1);
        s.abort = 0;
        ptx::fence_barrier_init();
    }
    if (threadIdx.x == 32)
        ptx::prefetch_tmap(&P.map);
    uint32_t ph = 0;   // phase parity of each buffer's barrier (kept across units)

    for (int64_t u = u_begin; u < u_end; ++u) {
    const int seq = (int)(u / groups);
    // query heads h0 .. h0 + Hg - 1 (a group of up to 16: the rows of every MMA)
    const int h0 = (int)(u % groups) * kMlH, Hg = min(kMlH, Hq - h0);
    int c0 = p.seq_start[seq], c1 = p.seq_start[seq + 1];
    // this CTA's share of the unit's tiles; `first`: the share that starts the unit
    int64_t lo, hi;
    bool first;
    if (split) {
        const int64_t a = max(kc * U, u * NC), e = min((kc + 1) * U, (u + 1) * NC);
        first = a == u * NC;
        lo = a - u * NC;   // scaled below by the unit's tiles
        hi = e - u * NC;
    } else {
        first = rank == 0;
        lo = rank;
        hi = rank + 1;
    }
    const int64_t den = split ? NC : CL;
    if (c0 < 0 || c1 < c0 || c1 > p.n_chunks) {
        if (first && h0 == 0 && threadIdx.x == 0)
            raise_err(p.err, KAMERA_DEVERR_DESCRIPTOR);
        c0 = c1 = 0;
    }
    int64_t total = 0;
    for (int c = c0; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        if (!mla_check(ch, c, p))
            total += (ch.len + kMlT - 1) / kMlT;
    }
    lo = total * lo / den;
    hi = total * hi / den;

    // the latent queries (rows past Hq zero) staged in the second tile buffer; q_rope as fp32
    __nv_bfloat16* qls = &s.kt[1][0][0][0];
    __syncthreads();   // the previous unit is done with every shared array (first: barriers initialised)
    for (int e = threadIdx.x; e < kMlH * (kMlC / 8); e += kMlThreads) {
        const int h = e / (kMlC / 8), v = e - h * (kMlC / 8);
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (h < Hg)
            w = *reinterpret_cast<const uint4*>(p.q + ((int64_t)seq * Hq + h0 + h) * kMlDK + 8 * v);
        *reinterpret_cast<uint4*>(qls + h * kMlQS + 8 * v) = w;
    }
    for (int e = threadIdx.x; e < kMlH * kMlR; e += kMlThreads) {
        const int h = e / kMlR, i = e - h * kMlR;
        s.qr[h][i] = h < Hg ? __bfloat162float(p.q[((int64_t)seq * Hq + h0 + h) * kMlDK + kMlC + i]) : 0.f;
    }
    ptx::fence_proxy_async();   // the staged queries precede the TMA loads that later refill that buffer
    __syncthreads();
    uint32_t qc[kMlC / 16][4];   // A fragments of the latent query, every k-step
    {
        const uint32_t base = ptx::smem_addr(qls + arow * kMlQS + acol);
#pragma unroll
        for (int ks = 0; ks < kMlC / 16; ++ks)
            ldsm_x4(base + 32 * ks, qc[ks]);
    }

    float o[8][4];   // output rows g, g + 8; columns 64 warp + 8 nt + 2 t4, + 1
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
        o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float wc[4] = {0.f, 0.f, 0.f, 0.f};   // sum_j p_j u_j, columns 8 warp + 2 t4 (warps < MP / 8)
    float m_run = -INFINITY, l_run = 0.f;  // head threadIdx.x / 16
    const RopeParams& rp = p.rope;
    const int ro = rp.rot_offset, rr = rp.rot_dim, half = rr / 2;
    const uint32_t kt0 = ptx::smem_addr(&s.kt[0][0][0][0]), ux0 = ptx::smem_addr(&s.ux[0][0][0]);
    constexpr uint32_t kBuf = SM::NBX * SM::kBoxBytes;          // bytes per row buffer
    constexpr uint32_t kUBuf = (uint32_t)(kMlT * SM::URS * 2);  // bytes per u | w buffer
    // 8x8 matrix-load addressing in the swizzled boxes: score B operand (rows 8 warp + (lane & 7),
    // pieces 4k + lane / 8) and value B operand (rows (lane & 7) + 8 ((lane / 8) & 1), pieces 2np + lane / 16)
    const int kr = 8 * warp + (lane & 7);
    const uint32_t klx = (uint32_t)((lane >> 3) ^ (lane & 7)), vlx = (uint32_t)((lane >> 4) ^ (lane & 7));

    int64_t pos = 0;   // tiles of the sequence before chunk c
    for (int c = c0; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        const int32_t bad = mla_check(ch, c, p);
        if (bad) {
            if (first && h0 == 0 && threadIdx.x == 0)
                raise_err(p.err, bad);
            continue;
        }
        const int len = ch.len;
        const int nt = (len + kMlT - 1) / kMlT;
        const int64_t a0 = lo - pos, a1 = hi - pos;
        const int t_lo = a0 > 0 ? (int)a0 : 0, t_hi = a1 < nt ? (int)a1 : nt;
        pos += nt;
        if (t_lo >= t_hi)
            continue;
        const int m = ch.rank;
        __syncthreads();   // the previous chunk (or the query staging) is done with every shared array
        mla_load<MP>(P, ch, t_lo * kMlT, min(kMlT, len - t_lo * kMlT), 0, s);   // lands while the chunk is set up
        for (int f = threadIdx.x; f < rp.n_freq; f += kMlThreads) {
            float cc, sn;
            phase_cos_sin(-freq_delta(rp, ch, c, f), rp.inv_freq[f], cc, sn);
            s.cs[f] = make_float2(cc, sn);
        }
        if constexpr (MP > 0) {
            const __nv_bfloat16* vrg = patch_ptr(ch, 3) + (int64_t)p.layer * kMlR * m;   // V_r [L][rope][m]
            for (int e = threadIdx.x; e < kMlR * MP; e += kMlThreads) {
                const int i = e / MP, r = e - i * MP;
                s.vr[i][r] = r < m ? __bfloat162float(vrg[i * m + r]) : 0.f;
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kMlH * kMlR; e += kMlThreads) {   // q_rope turned by -delta
            const int h = e / kMlR, i = e - h * kMlR, k = i - ro;
            float v = s.qr[h][i];
            if (k >= 0 && k < rr) {
                if (rp.pairing == KAMERA_ROPE_ROTATE_HALF) {
                    const float2 t = s.cs[k < half ? k : k - half];
                    v = k < half ? fmaf(v, t.x, -(s.qr[h][i + half] * t.y)) : fmaf(v, t.x, s.qr[h][i - half] * t.y);
                } else {
                    const float2 t = s.cs[k >> 1];
                    v = (k & 1) == 0 ? fmaf(v, t.x, -(s.qr[h][i + 1] * t.y)) : fmaf(v, t.x, s.qr[h][i - 1] * t.y);
                }
            }
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            s.xh[h][i] = hi;
            s.xl[h][i] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
        if constexpr (MP > 0) {
            for (int e = threadIdx.x; e < kMlH * MP; e += kMlThreads) {   // V_r^T q_rope (un-turned)
                const int h = e / MP, r = e - h * MP;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
                for (int i = 0; i < kMlR; i += 2) {
                    a0 = fmaf(s.qr[h][i], s.vr[i][r], a0);
                    a1 = fmaf(s.qr[h][i + 1], s.vr[i + 1][r], a1);
                }
                const float v = a0 + a1;
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                s.xh[h][kMlR + MP + r] = hi;
                s.xl[h][kMlR + MP + r] = __float2bfloat16_rn(v - __bfloat162float(hi));
            }
            if (warp < MP / 8) {   // V_c^T q_lat, columns 8 warp .. + 7, by MMA over the latent dimension
                float y[4] = {0.f, 0.f, 0.f, 0.f};
                const int r = 8 * warp + g;   // the B column this lane feeds
                const uint16_t* vc =
                    reinterpret_cast<const uint16_t*>(patch_ptr(ch, 1)) + (int64_t)p.layer * kMlC * m;
#pragma unroll
                for (int ks = 0; ks < kMlC / 16; ++ks) {
                    uint32_t b0 = 0u, b1 = 0u;
                    if (r < m) {
                        const int i0 = 16 * ks + 2 * t4;
                        b0 = (uint32_t)vc[i0 * m + r] | ((uint32_t)vc[(i0 + 1) * m + r] << 16);
                        b1 = (uint32_t)vc[(i0 + 8) * m + r] | ((uint32_t)vc[(i0 + 9) * m + r] << 16);
                    }
                    mma_bf16(y, qc[ks], b0, b1);
                }
                const int col = kMlR + 8 * warp + 2 * t4;
                uint32_t hi, lo;
                split_hl(y[0], y[1], hi, lo);
                *reinterpret_cast<uint32_t*>(&s.xh[g][col]) = hi;
                *reinterpret_cast<uint32_t*>(&s.xl[g][col]) = lo;
                split_hl(y[2], y[3], hi, lo);
                *reinterpret_cast<uint32_t*>(&s.xh[g + 8][col]) = hi;
                *reinterpret_cast<uint32_t*>(&s.xl[g + 8][col]) = lo;
            }
        }

        for (int tl = t_lo; tl < t_hi; ++tl) {
            const int b = (tl - t_lo) & 1, ntok = min(kMlT, len - tl * kMlT);
            tile_wait(ptx::smem_addr(&s.full[b]), (ph >> b) & 1u, &s.abort, p.err, P.wait_ns);
            ph ^= 1u << b;
            ptx::cp_async_wait<0>();   // this thread's copies of tile tl (the only group in flight)
            const uint32_t kb = kt0 + b * kBuf, uxb = ux0 + b * kUBuf;
            if (ntok < kMlT) {   // c_KV rows past the chunk: zero, so that their zero weights add nothing
                for (int e = threadIdx.x; e < (kMlT - ntok) * 64; e += kMlThreads) {
                    const int t = ntok + (e >> 6), c8 = e & 63;
                    ptx::st_shared_zero16(kb + (c8 >> 3) * SM::kBoxBytes + t * 128 + (c8 & 7) * 16);
                }
                ptx::fence_proxy_async();   // before a later TMA load refills the buffer
            }
            __syncthreads();   // tile b (and, first, the chunk's query part) in place; every warp is
                               // done with tile tl - 1, its buffer and its scores and weights
            if (tl + 1 < t_hi)
                mla_load<MP>(P, ch, (tl + 1) * kMlT, min(kMlT, len - (tl + 1) * kMlT), b ^ 1, s);
            {   // scores of tokens 8 warp .. + 7 against the 16 heads (four partial sums: independent MMA chains)
                float sa[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    sa[u][0] = sa[u][1] = sa[u][2] = sa[u][3] = 0.f;
                const uint32_t krow = kb + (uint32_t)(kr * 128);
#pragma unroll
                for (int ks = 0; ks < kMlC / 16; ks += 2) {
                    uint32_t bb[4];
                    ldsm_x4(krow + (uint32_t)(ks >> 2) * SM::kBoxBytes + ((((uint32_t)(2 * ks) & 7u) ^ klx) << 4), bb);
                    mma_bf16(sa[ks & 3], qc[ks], bb[0], bb[1]);
                    mma_bf16(sa[(ks + 1) & 3], qc[ks + 1], bb[2], bb[3]);
                }
                // the per-chunk part, hi and lo: k_rope (4 k-steps), then the u columns into
                // sums 0/1 and the w columns into sums 2/3, so the padded columns of a
                // wider instantiation add exact zeros to the same sums in the same order
                const uint32_t xa = ptx::smem_addr(&s.xh[arow][acol]), xla = ptx::smem_addr(&s.xl[arow][acol]);
                const uint32_t kx = krow + (kMlC / 64) * SM::kBoxBytes;   // the k_rope box
                const uint32_t ukx = uxb + (uint32_t)((kr * SM::URS + 8 * ((lane >> 3) & 1)) * 2);
#pragma unroll
                for (int ks = 0; ks < kMlR / 16; ks += 2) {
                    uint32_t bb[4], ah[4], al[4], ah2[4], al2[4];
                    ldsm_x4(kx + ((((uint32_t)(2 * ks) & 7u) ^ klx) << 4), bb);
                    ldsm_x4(xa + 32 * ks, ah);
                    ldsm_x4(xla + 32 * ks, al);
                    ldsm_x4(xa + 32 * (ks + 1), ah2);
                    ldsm_x4(xla + 32 * (ks + 1), al2);
                    mma_bf16(sa[0], ah, bb[0], bb[1]);
                    mma_bf16(sa[1], al, bb[0], bb[1]);
                    mma_bf16(sa[2], ah2, bb[2], bb[3]);
                    mma_bf16(sa[3], al2, bb[2], bb[3]);
                }
#pragma unroll
                for (int j = 0; j < 2 * (MP / 16); ++j) {
                    const int ks = kMlR / 16 + j, q = j < MP / 16 ? 0 : 2;
                    uint32_t bb[2], ah[4], al[4];
                    ldsm_x2(ukx + 32 * j, bb);
                    ldsm_x4(xa + 32 * ks, ah);
                    ldsm_x4(xla + 32 * ks, al);
                    mma_bf16(sa[q], ah, bb[0], bb[1]);
                    mma_bf16(sa[q + 1], al, bb[0], bb[1]);
                }
                const int tk = 8 * warp + 2 * t4;
                *reinterpret_cast<float2*>(&s.sc[g][tk]) =
                    make_float2((sa[0][0] + sa[1][0]) + (sa[2][0] + sa[3][0]), (sa[0][1] + sa[1][1]) + (sa[2][1] + sa[3][1]));
                *reinterpret_cast<float2*>(&s.sc[g + 8][tk]) =
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
            {   // O[:, 64 warp ..] += P C; sum_j p_j u_j on warps < MP / 8
                const float a0 = s.alpha[g], a1 = s.alpha[g + 8];
                if (!__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {   // a new running max in some row
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        o[nt][0] *= a0;
                        o[nt][1] *= a0;
                        o[nt][2] *= a1;
                        o[nt][3] *= a1;
                    }
                    wc[0] *= a0;
                    wc[1] *= a0;
                    wc[2] *= a1;
                    wc[3] *= a1;
                }
                const uint32_t pha = ptx::smem_addr(&s.ph[arow][acol]), pla = ptx::smem_addr(&s.pl[arow][acol]);
                const uint32_t vb = kb + (uint32_t)warp * SM::kBoxBytes + (uint32_t)(arow * 128);   // box warp: columns 64 warp ..
                const uint32_t ub = uxb + (uint32_t)((arow * SM::URS + 8 * warp) * 2);
#pragma unroll
                for (int ks = 0; ks < kMlT / 16; ++ks) {
                    uint32_t ah[4], al[4];
                    ldsm_x4(pha + 32 * ks, ah);
                    ldsm_x4(pla + 32 * ks, al);
                    const uint32_t vrow = vb + (uint32_t)(ks * 16 * 128);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        uint32_t bb[4];
                        ldsm_x4_t(vrow + ((((uint32_t)(2 * np)) ^ vlx) << 4), bb);
                        mma_bf16(o[2 * np], ah, bb[0], bb[1]);
                        mma_bf16(o[2 * np], al, bb[0], bb[1]);
                        mma_bf16(o[2 * np + 1], ah, bb[2], bb[3]);
                        mma_bf16(o[2 * np + 1], al, bb[2], bb[3]);
                    }
                    if constexpr (MP > 0) {
                        if (warp < MP / 8) {
                            uint32_t bu[2];
                            ldsm_x2_t(ub + (uint32_t)(ks * 16 * SM::URS * 2), bu);
                            mma_bf16(wc, ah, bu[0], bu[1]);
                            mma_bf16(wc, al, bu[0], bu[1]);
                        }
                    }
                }
            }
        }
        if constexpr (MP > 0) {
            if (m > 0) {   // fold sum_j p_j u_j through V_c: O += W V_c^T
                if (warp < MP / 8) {
                    const int col = 8 * warp + 2 * t4;
                    s.wsum[g][col] = wc[0];
                    s.wsum[g][col + 1] = wc[1];
                    s.wsum[g + 8][col] = wc[2];
                    s.wsum[g + 8][col + 1] = wc[3];
                }
                __syncthreads();
                const uint32_t* vcw =
                    reinterpret_cast<const uint32_t*>(patch_ptr(ch, 1) + (int64_t)p.layer * kMlC * m);   // pairs (r, r+1)
#pragma unroll
                for (int ks = 0; ks < MP / 16; ++ks) {
                    const int r0 = 16 * ks + 2 * t4;
                    uint32_t ah[4], al[4];
                    split_hl(s.wsum[g][r0], s.wsum[g][r0 + 1], ah[0], al[0]);
                    split_hl(s.wsum[g + 8][r0], s.wsum[g + 8][r0 + 1], ah[1], al[1]);
                    split_hl(s.wsum[g][r0 + 8], s.wsum[g][r0 + 9], ah[2], al[2]);
                    split_hl(s.wsum[g + 8][r0 + 8], s.wsum[g + 8][r0 + 9], ah[3], al[3]);
                    uint32_t bv[8][2];
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        const int64_t i = 64 * warp + 8 * nt + g;
                        bv[nt][0] = r0 < m ? vcw[(i * m + r0) >> 1] : 0u;
                        bv[nt][1] = r0 + 8 < m ? vcw[(i * m + r0 + 8) >> 1] : 0u;
                    }
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        mma_bf16(o[nt], ah, bv[nt][0], bv[nt][1]);
                        mma_bf16(o[nt], al, bv[nt][0], bv[nt][1]);
                    }
                }
                wc[0] = wc[1] = wc[2] = wc[3] = 0.f;
            }
        }
    }

    // merge: every CTA publishes (max, sum, unnormalised output); rank 0 combines
    __syncthreads();   // all copies have landed (the last wait took every group); the tile buffers are free
    float* ob = reinterpret_cast<float*>(&s.kt[0][0][0][0]);   // [kMlH][kMlC]
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int col = 64 * warp + 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(&ob[g * kMlC + col]) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2*>(&ob[(g + 8) * kMlC + col]) = make_float2(o[nt][2], o[nt][3]);
    }
    if ((threadIdx.x & 15) == 0) {
        s.cm[threadIdx.x >> 4] = m_run;
        s.cl[threadIdx.x >> 4] = l_run;
    }
    if (split) {   // ---- this CTA's partial state of unit u -> workspace slot k + u
        float* wp = P.ws + (size_t)(kc + u) * (2 * kMlH + kMlH * kMlC);
        __syncthreads();
        if (threadIdx.x < kMlH) {
            wp[threadIdx.x] = s.cm[threadIdx.x];
            wp[kMlH + threadIdx.x] = s.cl[threadIdx.x];
        }
        for (int e = threadIdx.x; e < kMlH * kMlC / 4; e += kMlThreads)
            reinterpret_cast<float4*>(wp + 2 * kMlH)[e] = reinterpret_cast<const float4*>(ob)[e];
        ptx::fence_proxy_async();   // the partial outputs' shared writes precede the next unit's TMA refills
        continue;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (rank == 0) {
        if (threadIdx.x < kMlH) {
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
        for (int e = threadIdx.x; e < Hg * (kMlC / 4); e += kMlThreads) {
            const int h = e / (kMlC / 4), i = 4 * (e - h * (kMlC / 4));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < CL; ++r) {
                const float f = s.fac[h][r];
                if (f == 0.f)
                    continue;
                const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(&ob[h * kMlC + i], r));
                acc.x = fmaf(v.x, f, acc.x);
                acc.y = fmaf(v.y, f, acc.y);
                acc.z = fmaf(v.z, f, acc.z);
                acc.w = fmaf(v.w, f, acc.w);
            }
            uint2 w;
            w.x = pack_bf16x2(acc.x, acc.y);
            w.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2*>(p.out + ((int64_t)seq * Hq + h0 + h) * kMlC + i) = w;
        }
    }
    cluster.sync();   // peers stay until rank 0 has read them
    }
}

}  // namespace

bool mla_attend_supported(int kv_lora, int rope_dim, int num_q_heads, int max_rank)
{
    return kv_lora == kMlC && rope_dim == kMlR && num_q_heads >= 1 && num_q_heads <= kMlMaxHeads &&
           max_rank >= 0 && max_rank <= 32;
}

// Cluster size.  One CTA fills an SM, and a cluster's CTAs must share a GPC, so
// clusters of CL can leave SMs of a GPC unused: the number of clusters that fit
// at once (the occupancy query) can fall short of the grid and push the last
// ones into a second wave.  The CTAs of a cluster split the sequence's tiles
// evenly, so each size (1 to 8) is costed as waves / CL and the cheapest taken
// (ties: the smaller cluster).  The occupancy answers are cached per kernel and
// device (cluster_fit).
template <int MP>
static int mla_pick_cluster(int64_t units, int bytes, double& best_t)
{
    int best = 1;
    best_t = 1e300;
    for (int cl = 1; cl <= kMlMaxCL; ++cl) {
        const int fit = cluster_fit(reinterpret_cast<const void*>(mla_attend_kernel<MP>), kMlThreads, bytes, cl);
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

// Split path (with a workspace) or cluster path, chosen as for GQA attention:
// the split path's U / NC against the cluster path's waves / CL, taken when at
// least 3% less (for 38 sequences of 16 heads: 0.26 against CL = 3's 0.33).
template <int MP>
static cudaError_t launch_mla_attend_m(const MlaAttendParams& p0, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    MlaLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p = p0;
    MlaAttendParams& p = L.p;
    L.wait_ns = wait_limit_ns();
    // canonical rows [num_rows][kv_lora + rope_dim] (an empty store gets a one-row map no tile reads)
    if (!make_rows_map(&L.map, p.kv, p.num_rows > 0 ? p.num_rows : 1, kMlDK, p.row_stride, 64, kMlT))
        return cudaErrorInvalidValue;
    static_assert(sizeof(MlSmem<MP>) + 1024 <= 227 * 1024, "MLA tile buffers exceed shared memory");
    const int bytes = (int)sizeof(MlSmem<MP>) + 1024;   // + the 1024-byte alignment
    cudaError_t e = cudaFuncSetAttribute(mla_attend_kernel<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    const int groups = (p.Hq + kMlH - 1) / kMlH;
    const int64_t units = (int64_t)p.n_seqs * groups;
    double t_cluster;
    p.cluster = mla_pick_cluster<MP>(units, bytes, t_cluster);
    const int nc = cluster_fit(reinterpret_cast<const void*>(mla_attend_kernel<MP>), kMlThreads, bytes, 1);
    if (ws && nc >= 1 && (size_t)(nc + units - 1) * attend_slot_bytes(kMlC) <= ws_bytes &&
        (double)units / nc < 0.97 * t_cluster) {
        L.ws = static_cast<float*>(ws);
        p.cluster = 1;
        mla_attend_kernel<MP><<<(unsigned)nc, kMlThreads, bytes, stream>>>(L);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        return launch_attend_merge(L.ws, units, nc, kMlC, groups, p.Hq, kMlH, p.out, stream);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_seqs * p.cluster), (unsigned)groups);
    cfg.blockDim = dim3(kMlThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_attend_kernel<MP>, L);
}

cudaError_t launch_mla_attend(const MlaAttendParams& p, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (p.max_rank == 0)
        return launch_mla_attend_m<0>(p, ws, ws_bytes, stream);
    return p.max_rank <= 16 ? launch_mla_attend_m<16>(p, ws, ws_bytes, stream)
                            : launch_mla_attend_m<32>(p, ws, ws_bytes, stream);
}

}  // namespace kamera
