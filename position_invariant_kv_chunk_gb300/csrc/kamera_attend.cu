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
// so each row is read once for all of them; CTA r of the cluster takes chunks
// r, r + CL, ... of the sequence, and rank 0 merges the CL partial softmax
// states (running max, sum, output accumulator) through distributed shared
// memory.  CL (1 to 8) is chosen from the occupancy query so that the clusters
// fill the GPU in as few waves as possible (a cluster must sit in one GPC).  Per chunk: the cos/sin table of -delta (fp64
// phase), the turned queries and V_k^T q in shared memory.  Per 64-token tile
// (double-buffered 16-byte async copies): the scores of all heads, four lanes
// per token over quarters of the head dimension; then warp h keeps query
// head h's online softmax (running max and sum) and its output accumulator in
// registers (head_dim / 32 columns per lane), and the chunk's sum_j p_j u'_j in
// shared memory, folded through V_v when the chunk ends.  fp32 throughout,
// one rounding to bf16 at the end.
#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"
#include "kamera_ptx.cuh"

namespace kamera {

namespace {

constexpr int kAtThreads = 256;
constexpr int kAtT = 64;                  // tokens per tile
constexpr int kAtMaxG = kAtThreads / 32;  // query heads per KV head (one warp each)
constexpr int kAtMaxD = 128;
constexpr int kAtKS = kAtMaxD + 8;        // tile row stride (elements): 272 bytes, spreads rows over banks
constexpr int kAtQS = kAtMaxD + 16;       // turned-query row: 4 floats of padding per 32 columns

// Column i of a turned query sits at i + 4 (i / 32): the four lanes of a token,
// which read quarter-rows 32 columns apart, then hit four different bank groups.
__device__ __forceinline__ int qpad(int i) { return i + ((i >> 5) << 2); }

// MAXM: the largest rank the instantiation takes (32: two CTAs fit an SM; 64: one).
template <int MAXM>
struct AtSmem {
    float q[kAtMaxG][kAtMaxD];            // the queries (target frame)
    float qr[kAtMaxG][kAtQS];             // turned by -delta (padded); V_v ac at a chunk's end
    float w[kAtMaxG][MAXM];               // V_k^T q
    float ac[kAtMaxG][MAXM];              // sum_j p_j u'_j of the current chunk (running scale)
    float p[kAtMaxG][kAtT];               // scores, then weights, of the current tile
    float2 cs[kAtMaxD / 2];
    __nv_bfloat16 kt[2][kAtT][kAtKS];     // also V_k [d][m] while a chunk starts
    __nv_bfloat16 vt[2][kAtT][kAtKS];     // also V_v^T [m][d] when a chunk ends
    __nv_bfloat16 ukt[2][kAtT * MAXM];
    __nv_bfloat16 uvt[2][kAtT * MAXM];
    float cm[kAtMaxG], cl[kAtMaxG];       // this CTA's running max and sum per query head
};

__device__ __forceinline__ float at_warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float f2_lo(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float f2_hi(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }

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

// Copies tile rows j0 .. j0 + n - 1 of chunk `ch` into buffer b.
template <int MAXM>
__device__ __forceinline__ void attend_load(const AttendParams& p, const KameraChunk& ch, int g, int j0, int n,
                                            int b, AtSmem<MAXM>& s)
{
    const int d = p.d, vpr = d / 8, m = ch.rank;
    const int64_t row0 = ch.src_offset + j0;
    for (int e = threadIdx.x; e < n * vpr; e += kAtThreads) {
        const int t = e / vpr, c8 = (e - t * vpr) * 8;
        const int64_t off = (row0 + t) * p.row_stride + (int64_t)g * d + c8;
        ptx::cp_async16(ptx::smem_addr(&s.kt[b][t][c8]), p.k + off);
        ptx::cp_async16(ptx::smem_addr(&s.vt[b][t][c8]), p.v + off);
    }
    if (m > 0) {
        const int64_t fo = ((int64_t)(p.layer * p.H + g) * ch.len + j0) * m;   // U [L][H][len][m]
        const __nv_bfloat16* uk = patch_ptr(ch, 0) + fo;
        const __nv_bfloat16* uv = patch_ptr(ch, 2) + fo;
        if ((m & 7) == 0) {   // rows of whole 16-byte vectors: the tile is one contiguous run
            for (int e = threadIdx.x; e < n * m / 8; e += kAtThreads) {
                ptx::cp_async16(ptx::smem_addr(&s.ukt[b][8 * e]), uk + 8 * e);
                ptx::cp_async16(ptx::smem_addr(&s.uvt[b][8 * e]), uv + 8 * e);
            }
        } else {
            for (int e = threadIdx.x; e < n * m; e += kAtThreads) {
                s.ukt[b][e] = uk[e];
                s.uvt[b][e] = uv[e];
            }
        }
    }
    ptx::cp_async_commit();
}

template <int MAXM>
__global__ void __launch_bounds__(kAtThreads, MAXM <= 32 ? 2 : 1) attend_kernel(const __grid_constant__ AttendParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AtSmem<MAXM>& s = *reinterpret_cast<AtSmem<MAXM>*>(smem_raw);
    namespace cg = cooperative_groups;
    const int CL = p.cluster, rank = (int)(blockIdx.x % (unsigned)CL);
    const int seq = blockIdx.x / CL, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = p.d, G = p.G, dpl = d / 32, dq = d / 4;
    const int HQ = p.H * G;

    int c0 = p.seq_start[seq], c1 = p.seq_start[seq + 1];
    if (c0 < 0 || c1 < c0 || c1 > p.n_chunks) {
        if (g == 0 && rank == 0 && threadIdx.x == 0)
            raise_err(p.err, KAMERA_DEVERR_DESCRIPTOR);
        c0 = c1 = 0;
    }
    c0 += rank;   // this CTA's chunks: c0, c0 + CL, ...
    for (int e = threadIdx.x; e < G * d; e += kAtThreads) {
        const int h = e / d, i = e - h * d;
        s.q[h][i] = __bfloat162float(p.q[((int64_t)seq * HQ + g * G + h) * d + i]);
    }
    uint64_t acc01 = 0, acc23 = 0;   // output columns dpl*lane .. + 3 as fp32 pairs
    float m_run = -INFINITY, l_run = 0.f;
    const RopeParams& rp = p.rope;
    const int ro = rp.rot_offset, rr = rp.rot_dim, half = rr / 2;

    for (int c = c0; c < c1; c += CL) {
        const KameraChunk ch = p.chunks[c];
        const int32_t bad = attend_check(ch, c, p);
        if (bad) {
            if (threadIdx.x == 0)
                raise_err(p.err, bad);
            continue;
        }
        if (ch.len == 0)
            continue;
        const int m = ch.rank;
        const int64_t fo = (int64_t)(p.layer * p.H + g) * d * m;   // this (layer, head)'s V factors
        __syncthreads();   // the previous chunk is done with every shared array
        for (int f = threadIdx.x; f < rp.n_freq; f += kAtThreads) {
            float cc, sn;
            phase_cos_sin(-freq_delta(rp, ch, c, f), rp.inv_freq[f], cc, sn);
            s.cs[f] = make_float2(cc, sn);
        }
        __nv_bfloat16* vks = &s.kt[1][0][0];   // V_k staged in the second key buffer
        if (m > 0) {
            const __nv_bfloat16* vkg = patch_ptr(ch, 1) + fo;
            for (int e = threadIdx.x; e < d * m; e += kAtThreads)
                vks[e] = vkg[e];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < G * d; e += kAtThreads) {   // q turned by -delta
            const int h = e / d, i = e - h * d, k = i - ro;
            float v = s.q[h][i];
            if (k >= 0 && k < rr) {
                if (rp.pairing == KAMERA_ROPE_ROTATE_HALF) {
                    const float2 t = s.cs[k < half ? k : k - half];
                    v = k < half ? fmaf(v, t.x, -(s.q[h][i + half] * t.y)) : fmaf(v, t.x, s.q[h][i - half] * t.y);
                } else {
                    const float2 t = s.cs[k >> 1];
                    v = (k & 1) == 0 ? fmaf(v, t.x, -(s.q[h][i + 1] * t.y)) : fmaf(v, t.x, s.q[h][i - 1] * t.y);
                }
            }
            s.qr[h][qpad(i)] = v;
        }
        for (int e = threadIdx.x; e < G * m; e += kAtThreads) {   // w = V_k^T q
            const int h = e / m, r = e - h * m;
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int i = 0; i < d; i += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    a[u] = fmaf(__bfloat162float(vks[(i + u) * m + r]), s.q[h][i + u], a[u]);
            }
            s.w[h][r] = (a[0] + a[1]) + (a[2] + a[3]);
            s.ac[h][r] = 0.f;
        }
        __syncthreads();   // the staged V_k is read; buffer 1 may take tile 1
        const int ntile = (ch.len + kAtT - 1) / kAtT;
        attend_load(p, ch, g, 0, min(kAtT, ch.len), 0, s);
        for (int tl = 0; tl < ntile; ++tl) {
            const int b = tl & 1, ntok = min(kAtT, ch.len - tl * kAtT);
            if (tl + 1 < ntile) {
                attend_load(p, ch, g, (tl + 1) * kAtT, min(kAtT, ch.len - (tl + 1) * kAtT), b ^ 1, s);
                ptx::cp_async_wait<1>();
            } else {
                ptx::cp_async_wait<0>();
            }
            __syncthreads();
            {   // scores: warp w takes tokens 8w .. 8w + 7, four lanes per token
                const int t = 8 * warp + (lane >> 2), qd = lane & 3;
                uint64_t part[kAtMaxG];
#pragma unroll
                for (int h = 0; h < kAtMaxG; ++h)
                    part[h] = 0;
                for (int i0 = qd * dq; i0 < (qd + 1) * dq; i0 += 8) {
                    const uint4 kw = *reinterpret_cast<const uint4*>(&s.kt[b][t][i0]);
                    const uint64_t k01 = ptx::f2_from_bf16x2(kw.x), k23 = ptx::f2_from_bf16x2(kw.y);
                    const uint64_t k45 = ptx::f2_from_bf16x2(kw.z), k67 = ptx::f2_from_bf16x2(kw.w);
#pragma unroll
                    for (int h = 0; h < kAtMaxG; ++h) {
                        if (h < G) {
                            const uint4 a = *reinterpret_cast<const uint4*>(&s.qr[h][qpad(i0)]);
                            const uint4 a2 = *reinterpret_cast<const uint4*>(&s.qr[h][qpad(i0) + 4]);
                            part[h] = ptx::f2_fma(ptx::f2_make(a.x, a.y), k01, part[h]);
                            part[h] = ptx::f2_fma(ptx::f2_make(a.z, a.w), k23, part[h]);
                            part[h] = ptx::f2_fma(ptx::f2_make(a2.x, a2.y), k45, part[h]);
                            part[h] = ptx::f2_fma(ptx::f2_make(a2.z, a2.w), k67, part[h]);
                        }
                    }
                }
                float sc[kAtMaxG];
#pragma unroll
                for (int h = 0; h < kAtMaxG; ++h)
                    sc[h] = f2_lo(part[h]) + f2_hi(part[h]);
                if (m > 0 && t < ntok) {
                    for (int r = qd; r < m; r += 4) {
                        const float u = __bfloat162float(s.ukt[b][t * m + r]);
#pragma unroll
                        for (int h = 0; h < kAtMaxG; ++h)
                            if (h < G)
                                sc[h] = fmaf(s.w[h][r], u, sc[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < kAtMaxG; ++h) {
                    sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], 1);
                    sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], 2);
                }
                if (qd == 0)
#pragma unroll
                    for (int h = 0; h < kAtMaxG; ++h)
                        if (h < G)
                            s.p[h][t] = t < ntok ? p.scale * sc[h] : -INFINITY;
            }
            __syncthreads();
            if (warp < G) {   // online softmax and P V for query head `warp`
                const int h = warp;
                const float s0 = s.p[h][lane], s1 = s.p[h][lane + 32];
                float tmax = fmaxf(s0, s1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                const float mnew = fmaxf(m_run, tmax);
                float alpha = 1.f, e0 = 0.f, e1 = 0.f;
                if (mnew != -INFINITY) {
                    alpha = expf(m_run - mnew);
                    e0 = expf(s0 - mnew);
                    e1 = expf(s1 - mnew);
                }
                s.p[h][lane] = e0;
                s.p[h][lane + 32] = e1;
                l_run = fmaf(l_run, alpha, at_warp_sum(e0 + e1));
                m_run = mnew;
                const uint32_t ab = __float_as_uint(alpha);
                acc01 = ptx::f2_mul(acc01, ptx::f2_make(ab, ab));
                acc23 = ptx::f2_mul(acc23, ptx::f2_make(ab, ab));
                for (int r = lane; r < m; r += 32)
                    s.ac[h][r] *= alpha;
                __syncwarp();
                // the weights of tokens past ntok are 0 and their stale rows are not read
                for (int t0 = 0; t0 < ntok; t0 += 8) {
                    float pt[8];
                    uint2 vv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int t = t0 + u;
                        pt[u] = s.p[h][t];
                        vv[u] = make_uint2(0u, 0u);
                        if (t < ntok) {
                            if (dpl == 4)
                                vv[u] = *reinterpret_cast<const uint2*>(&s.vt[b][t][4 * lane]);
                            else
                                vv[u].x = *reinterpret_cast<const uint32_t*>(&s.vt[b][t][2 * lane]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t pb = __float_as_uint(pt[u]);
                        const uint64_t pp = ptx::f2_make(pb, pb);
                        acc01 = ptx::f2_fma(pp, ptx::f2_from_bf16x2(vv[u].x), acc01);
                        acc23 = ptx::f2_fma(pp, ptx::f2_from_bf16x2(vv[u].y), acc23);
                    }
                }
                for (int r = lane; r < m; r += 32) {
                    float a = s.ac[h][r], a2 = 0.f;
                    for (int t0 = 0; t0 < ntok; t0 += 8) {
                        float pt[8], uu[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int t = t0 + u;
                            pt[u] = s.p[h][t];
                            uu[u] = t < ntok ? __bfloat162float(s.uvt[b][t * m + r]) : 0.f;
                        }
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            a = fmaf(pt[u], uu[u], a);
                            a2 = fmaf(pt[u + 1], uu[u + 1], a2);
                        }
                    }
                    s.ac[h][r] = a + a2;
                }
            }
            __syncthreads();   // buffer b is free for the tile after next
        }
        if (m > 0) {   // fold sum_j p_j u'_j through V_v: qr[h][i] <- sum_r V_v[i][r] ac[h][r]
            __nv_bfloat16* vvs = &s.vt[0][0][0];   // V_v^T staged in the first value buffer
            const __nv_bfloat16* vvg = patch_ptr(ch, 3) + fo;
            for (int e = threadIdx.x; e < d * m; e += kAtThreads) {
                const int i = e / m, r = e - i * m;
                vvs[r * d + i] = vvg[e];
            }
            __syncthreads();
            for (int e = threadIdx.x; e < G * d; e += kAtThreads) {
                const int h = e / d, i = e - h * d;
                float a = 0.f;
                for (int r = 0; r < m; ++r)
                    a = fmaf(__bfloat162float(vvs[r * d + i]), s.ac[h][r], a);
                s.qr[h][i] = a;
            }
            __syncthreads();
            if (warp < G) {
                float* f = &s.qr[warp][dpl * lane];
                acc01 = ptx::f2_add(acc01, ptx::f2_make(__float_as_uint(f[0]), __float_as_uint(f[1])));
                if (dpl == 4)
                    acc23 = ptx::f2_add(acc23, ptx::f2_make(__float_as_uint(f[2]), __float_as_uint(f[3])));
            }
        }
    }
    float r4[4] = {f2_lo(acc01), f2_hi(acc01), f2_lo(acc23), f2_hi(acc23)};
    if (CL > 1) {   // publish this CTA's state (acc in qr), then rank 0 merges
        cg::cluster_group cluster = cg::this_cluster();
        __syncthreads();
        if (warp < G) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < dpl)
                    s.qr[warp][dpl * lane + e] = r4[e];
            if (lane == 0) {
                s.cm[warp] = m_run;
                s.cl[warp] = l_run;
            }
        }
        cluster.sync();
        if (rank == 0 && warp < G) {
            float mx = -INFINITY;
            for (int r = 0; r < CL; ++r)
                mx = fmaxf(mx, *cluster.map_shared_rank(&s.cm[warp], r));
            float l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
            for (int r = 0; r < CL; ++r) {
                const float mr = *cluster.map_shared_rank(&s.cm[warp], r);
                if (mr == -INFINITY)
                    continue;
                const float f = expf(mr - mx);
                l = fmaf(*cluster.map_shared_rank(&s.cl[warp], r), f, l);
                const float* ar = cluster.map_shared_rank(&s.qr[warp][dpl * lane], r);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (e < dpl)
                        o[e] = fmaf(ar[e], f, o[e]);
            }
            l_run = l;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                r4[e] = o[e];
        }
        cluster.sync();   // peers stay until rank 0 has read them
    }
    if (rank == 0 && warp < G) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        __nv_bfloat16* o = p.out + ((int64_t)seq * HQ + g * G + warp) * d + dpl * lane;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < dpl)
                o[e] = __float2bfloat16_rn(r4[e] * inv);
    }
}

}  // namespace

bool attend_supported(int head_dim, int G, int max_rank)
{
    return (head_dim == 64 || head_dim == 128) && G >= 1 && G <= kAtMaxG && max_rank >= 0 && max_rank <= 64;
}

// Cluster size.  CTA r of a cluster takes chunks r, r + CL, ... of its (sequence,
// KV head), and a cluster's CTAs must share a GPC, so the clusters that fit at
// once (the occupancy query) can fall short of the grid and leave a last,
// mostly idle wave.  Each size 1..8 is costed as waves x chunks a CTA takes
// (from the chunks a sequence has on average) and the cheapest taken (ties:
// the smaller cluster); `fallback` if the query is unavailable.
template <int MAXM>
static int attend_pick_cluster(const AttendParams& p, int bytes, int fallback)
{
    const int64_t units = (int64_t)p.n_seqs * p.H;
    const int64_t per_seq = p.n_seqs > 0 ? (p.n_chunks + p.n_seqs - 1) / p.n_seqs : 1;
    int best = fallback;
    double best_t = 1e300;
    for (int cl = 1; cl <= 8; ++cl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(p.n_seqs * cl), (unsigned)p.H);
        cfg.blockDim = dim3(kAtThreads);
        cfg.dynamicSmemBytes = bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int fit = 0;
        if (cudaOccupancyMaxActiveClusters(&fit, attend_kernel<MAXM>, &cfg) != cudaSuccess || fit < 1) {
            (void)cudaGetLastError();
            continue;
        }
        const double t = (double)((units + fit - 1) / fit) * (double)((per_seq + cl - 1) / cl);
        if (t < best_t * 0.999) {
            best_t = t;
            best = cl;
        }
    }
    return best;
}

template <int MAXM>
static cudaError_t launch_attend_m(AttendParams p, cudaStream_t stream)
{
    const int bytes = (int)sizeof(AtSmem<MAXM>);
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<MAXM>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    p.cluster = attend_pick_cluster<MAXM>(p, bytes, p.cluster);
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
    return cudaLaunchKernelEx(&cfg, attend_kernel<MAXM>, p);
}

// Default cluster size (used when the occupancy query is unavailable): the
// smallest power of two (at most 8) that gives the grid about four CTAs per SM.
int attend_cluster(int64_t units)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1)
        sms = 1;
    int cl = 1;
    while (cl < 8 && units * cl < 4LL * sms)
        cl *= 2;
    return cl;
}

cudaError_t launch_attend(const AttendParams& p, cudaStream_t stream)
{
    return p.max_rank <= 32 ? launch_attend_m<32>(p, stream) : launch_attend_m<64>(p, stream);
}

}  // namespace kamera
