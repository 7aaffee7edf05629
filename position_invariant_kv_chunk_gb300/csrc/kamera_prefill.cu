// kamera_prefill.cu -- prefill attention over reused chunks, on the tensor cores.
//
// A prefill that reuses chunks attends from its T new query tokens over the
// reuse equation's rows of the chunks (gist.science technical summary, section
// 2), which the pages serve through a hook in the attention kernel (section 3,
// "Production Deployment"):
//     K_j = R(delta_c) k_j + V_k u_j,    V_j = v_j + V_v u'_j
// The chunks precede the new tokens, so no mask applies among them; each query
// row also gets its log-sum-exp, which merges this softmax with the one over
// the new tokens themselves.  As in decode, the turn and the patch fold into
// per-chunk query quantities, so no relocated row is ever formed:
//     q . K_j        = (R(-delta_c) q) . k_j + (V_k^T q) . u_j
//     sum_j p_j V_j  = sum_j p_j v_j + V_v (sum_j p_j u'_j)
//
// A (sequence, KV head) has T x G query rows (token-major: row r is token
// r / G, query head r % G of the KV head); one CTA owns 128 of them, the M of
// the 5th-generation tensor-core MMA (tcgen05.mma, fp32 accumulators in TMEM),
// and streams the sequence's rows in 64-token tiles:
//     S   [128 x 64]   = [Q' | X] [k | u]^T      Q' = R(-delta) q, X = V_k^T q
//     O_v [128 x d]   += P v                     P = the softmax weights
//     O_u [128 x 64]  += P u'                    folded through V_v per chunk
// Q', X and P are not bf16 values: each enters as a bf16 hi + lo pair (two
// MMAs, about 16 significant bits); the rows and U rows are exact bf16.  The
// A operands (Q', X, P) live in TMEM, so the MMAs read only the tile's rows
// from shared memory; P overwrites its S columns.
// Per chunk two more products run on the tensor cores: X = q V_k (the query
// rows, exact bf16, from shared memory) and the fold O_v += W V_v^T of the
// chunk's value patch, W = sum_j p_j u'_j (O_u, as hi + lo).
// Roles (192 threads):
//   warps 0-3  softmax: thread = query row = TMEM lane.  Per tile: the S row,
//              running max with lazy rescaling (O is rescaled in TMEM only when
//              the max grows by more than 2^8, so the weights stay below 256),
//              the weights as hi + lo into TMEM.  Per chunk: V_k, V_v and the
//              cos/sin of -delta into shared memory, Q' (CUDA cores) and X as
//              hi + lo into TMEM, and W from O_u once the chunk's last P u' is
//              done.  At the end: out = O_v / l and lse = m + log l.
//   warp 4     producer: key and value rows of a tile as 128B-swizzled TMA
//              boxes (64 columns x 64 rows), U and U' rows by 16-byte async
//              copies into the same layout; the value rows of a chunk's last,
//              partial tile by async copies too, zero past the chunk.
//   warp 5     MMA: one lane issues S of tile n, then P v and P u' of tile
//              n - 1 (so the softmax of tile n - 1 overlaps the scores of tile
//              n), the per-chunk X and fold, and commits each to an mbarrier;
//              the warp owns TMEM.
// Every wait is bounded in time: on expiry KAMERA_DEVERR_TIMEOUT is raised, the
// waits that follow return at once, the softmax warps run their loops to the
// end without waiting (so their CTA-internal barriers still meet), the MMA
// warp drains what it issued and the producer the copies it started, and TMEM
// is freed.
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

constexpr int kPfRows = 128;          // query rows per CTA = MMA M = TMEM lanes
constexpr int kPfTok = 64;            // tokens per tile
constexpr int kPfMP = 64;             // ranks, padded: the U tiles' width
constexpr int kPfThreads = 192;       // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int kPfProd = 4, kPfMma = 5;
constexpr float kPfLazy = 8.0f;       // log2 of the growth of the running max that forces a rescale
constexpr uint32_t kBox = 8192;       // one TMA box: 64 rows x 128 bytes

// Shared memory from a 1024-byte aligned base: the tile ring (per stage the
// key boxes, U, the value boxes and U'), the CTA's query rows (the A operand
// of X = q V_k), V_k of the current chunk and V_v of the last two ([d][64]
// bf16, ranks padded, 128B-swizzled rows), the cos/sin of -delta, the barriers.
template <int D>
struct PfLayout {
    static constexpr int NB = D / 64;                          // 64-column boxes of a head row
    static constexpr int NS = D == 128 ? 3 : 4;                 // stages
    // per stage: key boxes, U, value boxes, U' -- the value boxes and U' are one
    // MN-major operand of D + 64 columns (64-column atoms kBox apart)
    static constexpr uint32_t kK = 0, kU = NB * kBox, kV = kU + kBox, kU2 = kV + NB * kBox;
    static constexpr uint32_t kStage = kU2 + kBox;
    static constexpr uint32_t kQ = NS * kStage;                 // q [128][D], K-major, NB atoms of 16 KB
    static constexpr uint32_t kVk = kQ + NB * 16384;            // V_k [d][64]
    static constexpr uint32_t kVv = kVk + D * 128;              // V_v [2][d][64]
    static constexpr uint32_t kCs = kVv + 2 * D * 128;          // float2 [64]
    static constexpr uint32_t kBar = kCs + 512;
    static constexpr uint32_t kBytes = kBar + 256 + 1024;       // + alignment slack
    // TMEM columns: S (and P) of tiles 2i and 2i + 1, O_v, O_u, Q' hi and lo, X hi and lo
    static constexpr uint32_t kTmS = 0, kTmOv = 2 * kPfTok, kTmOu = kTmOv + D, kTmQh = kTmOu + kPfMP;
    static constexpr uint32_t kTmQl = kTmQh + D / 2, kTmXh = kTmQl + D / 2, kTmXl = kTmXh + kPfMP / 2;
    static_assert(kTmXl + kPfMP / 2 <= 512, "TMEM columns");
    static_assert(kBytes <= 227 * 1024, "shared memory");
};

struct PfBars {
    uint64_t full[4], empty[4];        // tile ring: loads landed / MMAs done with the stage
    uint64_t s_full[2], p_full[2];     // S of tile n in TMEM / P of tile n in TMEM
    uint64_t pv_done[2];               // P v and P u' of tile n done
    uint64_t vk_ready;                 // per chunk: V_k (and, first, q) in shared memory
    uint64_t x_done;                   // per chunk: q V_k in TMEM
    uint64_t a_ready;                  // per chunk: Q' and X (hi + lo) in TMEM
    uint64_t w_ready;                  // per chunk after the first: the last one's sum p u' as hi + lo
    uint64_t fold_done;                // per chunk after the first: its value patch added to O_v
    uint64_t drained;                  // every MMA of the CTA done
    uint32_t tmem;
    int32_t abort;
};
static_assert(sizeof(PfBars) <= 256, "barrier block");

struct PrefillLaunch {
    PrefillParams p;
    CUtensorMap map_k, map_v;          // [num_rows][H * d], boxes of 64 columns x 64 rows
    uint64_t wait_ns;
    int32_t withhold;                  // test hook: the producer starts no tile copy
};

__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t ta, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t ta, const uint32_t (&r)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(ta), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16-byte piece c of row r of a 128B-swizzled tile of 128-byte rows (the TMA
// and MMA layout): piece c ^ (r & 7).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void bar_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ int32_t prefill_check(const KameraChunk& ch, int c, const PrefillParams& p)
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

// The sequence's chunk range, [c0, c1); empty if d_seq_start is malformed.
__device__ __forceinline__ void seq_chunks(const PrefillParams& p, int seq, int& c0, int& c1)
{
    c0 = p.seq_start[seq];
    c1 = p.seq_start[seq + 1];
    if (c0 < 0 || c1 < c0 || c1 > p.n_chunks)
        c0 = c1 = 0;
}

// Waits for a phase whatever the abort flag says, up to `limit` ns: the drain
// of copies and MMAs a role started before it leaves.
__device__ __forceinline__ void pf_drain_wait(uint32_t bar, uint32_t parity, uint64_t limit)
{
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer() - t0 > limit)
            return;
}

// Rows [0, ntok) of the tile's U and U' blocks (m-wide factor rows, `uk` and
// `uv`: the tile's first row) into 64 x 64-rank tiles (128B-swizzled), by
// 16-byte async copies when m is a multiple of 8, else by element loads.  Only
// what an MMA reads must be finite: U' rows past ntok (zero weights times the
// row) and, in both, the ranks from m up to the next multiple of 16 (zero
// query parts and zero V_v columns times them); those are written as zeros.
// Other padding is left as it is: it reaches only masked scores or O_u columns
// past m, which nothing reads.
__device__ __forceinline__ void pf_load_u(uint32_t du, uint32_t dv, const __nv_bfloat16* uk,
                                          const __nv_bfloat16* uv, int m, int ntok, int lane)
{
    const int vpr = (m + 7) >> 3, vp16 = 2 * ((m + 15) >> 4);   // pieces with data / read by the S MMAs
    if ((m & 7) == 0) {
        const int nv = ntok * vpr;   // the block's rows are contiguous: nv 16-byte pieces
        for (int e = lane; e < nv; e += 32) {
            const int r = e / vpr, c = e - r * vpr;
            ptx::cp_async16(du + sw128(r, c), uk + 8 * e);
            ptx::cp_async16(dv + sw128(r, c), uv + 8 * e);
        }
        if (vp16 > vpr)
            for (int e = lane; e < kPfTok; e += 32) {
                ptx::st_shared_zero16(du + sw128(e, vpr));
                ptx::st_shared_zero16(dv + sw128(e, vpr));
            }
        for (int e = ntok * 8 + lane; e < kPfTok * 8; e += 32)
            ptx::st_shared_zero16(dv + sw128(e >> 3, e & 7));
    } else {   // ranks that are not whole 16-byte pieces
        const uint16_t* k16 = reinterpret_cast<const uint16_t*>(uk);
        const uint16_t* v16 = reinterpret_cast<const uint16_t*>(uv);
        for (int e = lane; e < kPfTok * 8; e += 32) {
            const int r = e >> 3, c = e & 7;
            if (c >= vp16 && r < ntok)
                continue;
            uint32_t a[4] = {0u, 0u, 0u, 0u}, b[4] = {0u, 0u, 0u, 0u};
            if (r < ntok) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 8 * c + k;
                    if (j < m) {
                        a[k >> 1] |= (uint32_t)__ldg(k16 + (int64_t)r * m + j) << (16 * (k & 1));
                        b[k >> 1] |= (uint32_t)__ldg(v16 + (int64_t)r * m + j) << (16 * (k & 1));
                    }
                }
            }
            ptx::sts128(du + sw128(r, c), a[0], a[1], a[2], a[3]);
            ptx::sts128(dv + sw128(r, c), b[0], b[1], b[2], b[3]);
        }
    }
}

// The producer warp: every tile of the unit, in order, into the ring.  The
// key and value rows come by TMA (completion counted in bytes); the U rows
// (and a partial tile's value rows) by async copies, whose landing the warp
// waits for one tile later -- so two tiles' copies are in flight -- before it
// makes them visible to the MMAs and arrives; when the next stage is not free
// yet, it publishes the pending tile at once instead.
template <int D>
__device__ void pf_producer(const PrefillLaunch& P, uint32_t sbase, PfBars& b, int seq, int h, int lane)
{
    using L = PfLayout<D>;
    const PrefillParams& p = P.p;
    int c0, c1;
    seq_chunks(p, seq, c0, c1);
    uint32_t n = 0;   // tiles started
    bool ok = true, pending = false;   // pending: tile n - 1 started but not yet published
    for (int c = c0; c < c1 && ok; ++c) {
        const KameraChunk& ch = p.chunks[c];
        if (prefill_check(ch, c, p))
            continue;
        const int len = ch.len, m = ch.rank, nt = (len + kPfTok - 1) / kPfTok;
        const int64_t fo = (int64_t)(p.layer * p.H + h) * len * m;   // U [L][H][len][m]
        for (int tl = 0; tl < nt; ++tl, ++n) {
            const int st = (int)(n % L::NS);
            if (n >= (uint32_t)L::NS) {   // the MMAs of tile n - NS are done with the stage
                // if the stage is not free yet, publish the previous tile first rather than
                // hold it back while this warp waits
                const uint32_t par = ((n / L::NS) & 1u) ^ 1u;
                if (pending && !__shfl_sync(0xFFFFFFFFu, ptx::mbar_test_wait(ptx::smem_addr(&b.empty[st]), par) ? 1 : 0,
                                            0)) {
                    ptx::cp_async_wait<0>();
                    ptx::fence_proxy_async();
                    ptx::mbar_arrive(ptx::smem_addr(&b.full[(n - 1) % L::NS]));
                    pending = false;
                }
                bool got = true;
                if (lane == 0)
                    got = wmma16::tile_wait(ptx::smem_addr(&b.empty[st]), par, &b.abort, p.err, P.wait_ns);
                if (!__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
            }
            const uint32_t s0 = sbase + st * L::kStage, full = ptx::smem_addr(&b.full[st]);
            const int j0 = tl * kPfTok, ntok = min(kPfTok, len - j0);
            const bool tail = ntok < kPfTok;
            if (lane == 0 && !P.withhold) {
                const int y = (int)(ch.src_offset + j0);
                ptx::mbar_arrive_expect_tx(full, (tail ? 1u : 2u) * L::NB * kBox);
#pragma unroll
                for (int x = 0; x < L::NB; ++x)
                    ptx::tma_load_2d(s0 + L::kK + x * kBox, &P.map_k, h * D + 64 * x, y, full);
                if (!tail) {
#pragma unroll
                    for (int x = 0; x < L::NB; ++x)
                        ptx::tma_load_2d(s0 + L::kV + x * kBox, &P.map_v, h * D + 64 * x, y, full);
                }
            }
            if (m > 0)
                pf_load_u(s0 + L::kU, s0 + L::kU2, patch_ptr(ch, 0) + fo + (int64_t)j0 * m,
                          patch_ptr(ch, 2) + fo + (int64_t)j0 * m, m, ntok, lane);
            if (tail) {   // the chunk's last value rows by async copies, zero past the chunk
                const __nv_bfloat16* vr = p.v + (ch.src_offset + j0) * p.row_stride + (int64_t)h * D;
                for (int e = lane; e < kPfTok * 8 * L::NB; e += 32) {
                    const int r = e / (8 * L::NB), x = (e >> 3) % L::NB, c8 = e & 7;
                    const uint32_t dst = s0 + L::kV + x * kBox + sw128(r, c8);
                    if (r < ntok)
                        ptx::cp_async16(dst, vr + (int64_t)r * p.row_stride + 64 * x + 8 * c8);
                    else
                        ptx::st_shared_zero16(dst);
                }
            }
            ptx::cp_async_commit();
            if (pending) {   // the previous tile's copies have landed: visible to the MMAs
                ptx::cp_async_wait<1>();
                ptx::fence_proxy_async();
                ptx::mbar_arrive(ptx::smem_addr(&b.full[(n - 1) % L::NS]));
            }
            pending = true;
        }
    }
    ptx::cp_async_wait<0>();
    if (pending) {
        ptx::fence_proxy_async();
        ptx::mbar_arrive(ptx::smem_addr(&b.full[(n - 1) % L::NS]));
    }
    // the copies this warp started land before the CTA leaves
    if (lane == 0)
        for (uint32_t k = n > (uint32_t)L::NS ? n - L::NS : 0u; k < n; ++k)
            pf_drain_wait(ptx::smem_addr(&b.full[k % L::NS]), (k / L::NS) & 1u, P.wait_ns);
    __syncwarp();
}

// Shared-memory matrix descriptors as (low word, high word): the low word holds
// the start address (bytes >> 4) and the leading byte offset, so a step inside
// an operand is one 32-bit add.  High word: stride byte offset 1024 (8-row
// groups), descriptor version 1, 128-byte swizzle.  A K-major operand (the key
// and U rows) ignores the leading offset; for an MN-major one (the value and U'
// rows: the rows of a TMA box are K, the N dimension is contiguous) it is the
// distance between 64-element atoms along N.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint64_t pf_desc(uint32_t lo)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(kDescHi));
    return d;
}

// D[tmem] (+)= A[tmem] * B[smem]^T (kind::f16: bf16 in, fp32 accumulate), the
// accumulate flag a compile-time constant.  A's row r sits in TMEM lane r,
// elements 2c and 2c + 1 in the low and high half of column c.
template <bool ACC>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc)
{
    if constexpr (ACC)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.u32 p, 1, 1;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "r"(a_tmem), "l"(pf_desc(b_lo)), "r"(idesc)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, 1, 1;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "r"(a_tmem), "l"(pf_desc(b_lo)), "r"(idesc)
                     : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T (kind::f16), accumulate flag constant.
template <bool ACC>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc)
{
    if constexpr (ACC)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.u32 p, 1, 1;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(pf_desc(a_lo)), "l"(pf_desc(b_lo)), "r"(idesc)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, 1, 1;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                     "l"(pf_desc(a_lo)), "l"(pf_desc(b_lo)), "r"(idesc)
                     : "memory");
}

// The MMA lane.  Per tile n: S(n) = [Q'hi | Q'lo | Xhi | Xlo] [k | k | u | u]^T
// into the S columns of n & 1, then [O_v | O_u] += [Phi | Plo] [v | u'] of tile
// n - 1, one MMA of N = d + 16 ceil(m / 16) per step (on a chunk's first tile
// O_u restarts from zero, so there the two parts are separate MMAs).  Per
// chunk, before its first S: X = q V_k (q and V_k in shared memory) into the S
// columns of that tile, for the softmax warps to split; after the previous
// chunk's last P u': the fold O_v += W V_v^T of that chunk, W = its sum_j p_j
// u'_j as hi + lo in the O_u columns.  MMAs of one thread run in issue order,
// so an MMA never overwrites an operand an earlier one has still to read.
// Everything per MMA is precomputed but one add: the issue rate of this one
// thread bounds the tile rate.
template <int D>
__device__ void pf_mma(const PrefillLaunch& P, uint32_t sbase, PfBars& b, uint32_t tm, int seq)
{
    using L = PfLayout<D>;
    const PrefillParams& p = P.p;
    constexpr uint32_t idS = ptx::idesc_bf16_f32(kPfRows, kPfTok);
    constexpr uint32_t idV = ptx::idesc_bf16_f32(kPfRows, D) | (1u << 16);   // B (value rows) MN-major
    constexpr uint32_t idF = ptx::idesc_bf16_f32(kPfRows, D);                // fold: B = V_v, K-major
    // descriptor low words of stage 0: K-major (LBO field 1, unused), MN-major (LBO = one box)
    const uint32_t k_lo = ((sbase + L::kK) >> 4) | (1u << 16), u_lo = ((sbase + L::kU) >> 4) | (1u << 16);
    const uint32_t v_lo = ((sbase + L::kV) >> 4) | ((kBox >> 4) << 16);
    const uint32_t u2_lo = ((sbase + L::kU2) >> 4) | ((kBox >> 4) << 16);
    const uint32_t q_lo = ((sbase + L::kQ) >> 4) | (1u << 16), vk_lo = ((sbase + L::kVk) >> 4) | ((kBox >> 4) << 16);
    const uint32_t vv_lo = ((sbase + L::kVv) >> 4) | (1u << 16);
    constexpr uint32_t kStep = L::kStage >> 4;
    const uint32_t aQh = tm + L::kTmQh, aQl = tm + L::kTmQl, aXh = tm + L::kTmXh, aXl = tm + L::kTmXl;
    const uint32_t dO = tm + L::kTmOv, dU = tm + L::kTmOu;
    int c0, c1;
    seq_chunks(p, seq, c0, c1);
    // [O_v | O_u] += P [v | u'] of tile i from stage st (m: its chunk's rank; first: its chunk's first tile)
    auto pv = [&](uint32_t i, int st, int m, bool first) -> bool {
        if (!wmma16::tile_wait(ptx::smem_addr(&b.p_full[i & 1]), (i >> 1) & 1u, &b.abort, p.err, P.wait_ns))
            return false;
        ptx::tc_fence_after();
        const uint32_t aP = tm + L::kTmS + (i & 1) * kPfTok, bv = v_lo + st * kStep;
        const int ksu = (m + 15) >> 4;
        if (!first || m == 0) {
            const uint32_t id = ptx::idesc_bf16_f32(kPfRows, D + 16 * ksu) | (1u << 16);
            if (i == 0)
                mma_ts<false>(dO, aP, bv, id);
            else
                mma_ts<true>(dO, aP, bv, id);
#pragma unroll
            for (int ks = 1; ks < kPfTok / 16; ++ks)
                mma_ts<true>(dO, aP + 8 * ks, bv + (2048 >> 4) * ks, id);
#pragma unroll
            for (int ks = 0; ks < kPfTok / 16; ++ks)
                mma_ts<true>(dO, aP + kPfTok / 2 + 8 * ks, bv + (2048 >> 4) * ks, id);
        } else {
            const uint32_t bu = u2_lo + st * kStep, idU = ptx::idesc_bf16_f32(kPfRows, 16 * ksu) | (1u << 16);
            if (i == 0)
                mma_ts<false>(dO, aP, bv, idV);
            else
                mma_ts<true>(dO, aP, bv, idV);
            mma_ts<false>(dU, aP, bu, idU);
#pragma unroll
            for (int ks = 1; ks < kPfTok / 16; ++ks) {
                mma_ts<true>(dO, aP + 8 * ks, bv + (2048 >> 4) * ks, idV);
                mma_ts<true>(dU, aP + 8 * ks, bu + (2048 >> 4) * ks, idU);
            }
#pragma unroll
            for (int ks = 0; ks < kPfTok / 16; ++ks) {
                mma_ts<true>(dO, aP + kPfTok / 2 + 8 * ks, bv + (2048 >> 4) * ks, idV);
                mma_ts<true>(dU, aP + kPfTok / 2 + 8 * ks, bu + (2048 >> 4) * ks, idU);
            }
        }
        ptx::umma_commit(ptx::smem_addr(&b.pv_done[i & 1]));
        ptx::umma_commit(ptx::smem_addr(&b.empty[st]));
        return true;
    };
    uint32_t n = 0, k = 0;   // tiles, chunks
    int pst = 0, pm = 0, prev_chunk_m = -1;
    bool pfirst = false, ok = true;
    for (int c = c0; c < c1 && ok; ++c) {
        const KameraChunk& ch = p.chunks[c];
        if (prefill_check(ch, c, p))
            continue;
        const int m = ch.rank, nt = (ch.len + kPfTok - 1) / kPfTok, ksu = (m + 15) / 16;
        if (nt == 0)
            continue;
        for (int tl = 0; tl < nt; ++tl, ++n) {
            if (tl == 0) {
                // X = q V_k into the S columns of this tile (free: their P was read by an earlier MMA)
                if (!wmma16::tile_wait(ptx::smem_addr(&b.vk_ready), k & 1u, &b.abort, p.err, P.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (m > 0) {
                    const uint32_t dX = tm + L::kTmS + (n & 1) * kPfTok;
                    const uint32_t idX = ptx::idesc_bf16_f32(kPfRows, 16 * ksu) | (1u << 16);   // B MN-major
                    mma_ss<false>(dX, q_lo, vk_lo, idX);
#pragma unroll
                    for (int ks = 1; ks < D / 16; ++ks)
                        mma_ss<true>(dX, q_lo + (ks >> 2) * (16384 >> 4) + 2 * (ks & 3), vk_lo + (2048 >> 4) * ks,
                                     idX);
                }
                ptx::umma_commit(ptx::smem_addr(&b.x_done));
                // the chunk's Q' and X are in TMEM
                if (!wmma16::tile_wait(ptx::smem_addr(&b.a_ready), k & 1u, &b.abort, p.err, P.wait_ns)) {
                    ok = false;
                    break;
                }
            }
            const int st = (int)(n % L::NS);
            if (!wmma16::tile_wait(ptx::smem_addr(&b.full[st]), (n / L::NS) & 1u, &b.abort, p.err, P.wait_ns)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t dS = tm + L::kTmS + (n & 1) * kPfTok;
            const uint32_t bk = k_lo + st * kStep, bu = u_lo + st * kStep;
            mma_ts<false>(dS, aQh, bk, idS);
#pragma unroll
            for (int ks = 1; ks < D / 16; ++ks)
                mma_ts<true>(dS, aQh + 8 * ks, bk + (ks >> 2) * (kBox >> 4) + 2 * (ks & 3), idS);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_ts<true>(dS, aQl + 8 * ks, bk + (ks >> 2) * (kBox >> 4) + 2 * (ks & 3), idS);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                if (ks < ksu) {
                    mma_ts<true>(dS, aXh + 8 * ks, bu + 2 * ks, idS);
                    mma_ts<true>(dS, aXl + 8 * ks, bu + 2 * ks, idS);
                }
            ptx::umma_commit(ptx::smem_addr(&b.s_full[n & 1]));
            if (n > 0 && !pv(n - 1, pst, pm, pfirst)) {
                ok = false;
                break;
            }
            if (tl == 0 && k > 0) {   // the previous chunk's value patch: O_v += W V_v^T
                if (!wmma16::tile_wait(ptx::smem_addr(&b.w_ready), (k - 1) & 1u, &b.abort, p.err, P.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const int pk = (prev_chunk_m + 15) >> 4;
                const uint32_t bvv = vv_lo + ((k - 1) & 1) * ((D * 128) >> 4);
                for (int ks = 0; ks < pk; ++ks) {
                    mma_ts<true>(dO, dU + 8 * ks, bvv + 2 * ks, idF);
                    mma_ts<true>(dO, dU + 32 + 8 * ks, bvv + 2 * ks, idF);
                }
                ptx::umma_commit(ptx::smem_addr(&b.fold_done));
            }
            if (tl == 0)
                ++k;
            pst = st;
            pm = m;
            pfirst = tl == 0;
        }
        prev_chunk_m = m;
    }
    if (ok && n > 0) {
        if (pv(n - 1, pst, pm, pfirst) &&
            wmma16::tile_wait(ptx::smem_addr(&b.w_ready), (k - 1) & 1u, &b.abort, p.err, P.wait_ns)) {
            ptx::tc_fence_after();   // the last chunk's value patch
            const int pk = (prev_chunk_m + 15) >> 4;
            const uint32_t bvv = vv_lo + ((k - 1) & 1) * ((D * 128) >> 4);
            for (int ks = 0; ks < pk; ++ks) {
                mma_ts<true>(dO, dU + 8 * ks, bvv + 2 * ks, idF);
                mma_ts<true>(dO, dU + 32 + 8 * ks, bvv + 2 * ks, idF);
            }
            ptx::umma_commit(ptx::smem_addr(&b.fold_done));
        }
    }
    // every MMA issued here completes before TMEM is freed
    ptx::umma_commit(ptx::smem_addr(&b.drained));
    pf_drain_wait(ptx::smem_addr(&b.drained), 0u, P.wait_ns);
}

// An m-wide V factor block [d][m] (`src`) into a [d][64] bf16 tile of
// 128B-swizzled 128-byte rows (an MMA operand: MN-major for X = q V_k, K-major
// for the fold), the ranks past m up to the next multiple of 16 zero (128
// threads).
template <int D>
__device__ __forceinline__ void pf_stage_v(uint32_t dst, const __nv_bfloat16* src, int m, int r)
{
    const int vpr = (m + 7) >> 3, vp16 = 2 * ((m + 15) >> 4);
    if ((m & 7) == 0) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        for (int e = r; e < D * vpr; e += kPfRows) {
            const uint4 v = __ldg(s4 + e);
            const int i = e / vpr, c = e - i * vpr;
            ptx::sts128(dst + sw128(i, c), v.x, v.y, v.z, v.w);
        }
        if (vp16 > vpr)
            for (int i = r; i < D; i += kPfRows)
                ptx::st_shared_zero16(dst + sw128(i, vpr));
    } else {
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
        for (int e = r; e < D * vp16; e += kPfRows) {
            const int i = e / vp16, c = e - i * vp16;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int j = 8 * c + k;
                if (j < m)
                    w[k >> 1] |= (uint32_t)__ldg(s16 + (int64_t)i * m + j) << (16 * (k & 1));
            }
            ptx::sts128(dst + sw128(i, c), w[0], w[1], w[2], w[3]);
        }
    }
}

// O_u (fp32, the last chunk's sum_j p_j u'_j) -> hi + lo bf16 pairs in place:
// rank pair (2c, 2c + 1) hi in O_u column c, lo in column 32 + c -- the A
// operand of the fold O_v += W V_v^T.
template <int D>
__device__ __forceinline__ void pf_split_w(uint32_t lane_base)
{
    using L = PfLayout<D>;
    uint32_t w0[32], w1[32], hi[32], lo[32];
    tmem_ld32(lane_base + L::kTmOu, w0);
    tmem_ld32(lane_base + L::kTmOu + 32, w1);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const uint32_t* src = c < 16 ? w0 : w1;
        const int k = 2 * (c & 15);
        wmma16::split_hl(__uint_as_float(src[k]), __uint_as_float(src[k + 1]), hi[c], lo[c]);
    }
    tmem_st32(lane_base + L::kTmOu, hi);
    tmem_st32(lane_base + L::kTmOu + 32, lo);
    tmem_wait_st();
}

// 2^x (the MUFU approximation: relative error near 2^-22, subnormal results
// flushed to zero).
__device__ __forceinline__ float pf_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The largest (`neg`: smallest) of the row's first ntok raw scores.
__device__ __forceinline__ float pf_extreme(const uint32_t (&a)[32], const uint32_t (&b)[32], int ntok, bool neg)
{
    float e = neg ? INFINITY : -INFINITY;
    if (ntok >= kPfTok) {
        if (neg) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                e = fminf(e, fminf(__uint_as_float(a[j]), __uint_as_float(b[j])));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                e = fmaxf(e, fmaxf(__uint_as_float(a[j]), __uint_as_float(b[j])));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float x = __uint_as_float(a[j]), y = __uint_as_float(b[j]);
            if (j < ntok)
                e = neg ? fminf(e, x) : fmaxf(e, x);
            if (j + 32 < ntok)
                e = neg ? fminf(e, y) : fmaxf(e, y);
        }
    }
    return e;
}

// O_v (and O_u when `with_u`) times f, in TMEM, for this thread's row.
template <int D>
__device__ __forceinline__ void pf_rescale(uint32_t lane_base, float f, bool with_u)
{
    using L = PfLayout<D>;
#pragma unroll 1
    for (int cb = 0; cb < (D + (with_u ? kPfMP : 0)) / 32; ++cb) {
        uint32_t o[32];
        tmem_ld32(lane_base + L::kTmOv + 32 * cb, o);   // O_u follows O_v
#pragma unroll
        for (int c = 0; c < 32; ++c)
            o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
        tmem_st32(lane_base + L::kTmOv + 32 * cb, o);
    }
    tmem_wait_st();
}

// The softmax warps: thread r holds query row blk * 128 + r (TMEM lane r).
// Waits that run out (abort) make the rest of the loops run without waiting,
// so the four warps still meet at every barrier among them.
template <int D>
__device__ void pf_softmax(const PrefillLaunch& P, uint32_t sbase, PfBars& b, uint32_t tm, int seq, int h, int blk,
                           int r)
{
    using L = PfLayout<D>;
    const PrefillParams& p = P.p;
    const RopeParams& rp = p.rope;
    const int G = p.G, HQ = p.H * G;
    const int row = blk * kPfRows + r;
    const bool valid = row < p.T * G;
    const int tok = valid ? row / G : 0, gq = valid ? row - (row / G) * G : 0;
    const int64_t qoff = (((int64_t)seq * p.T + tok) * HQ + (int64_t)h * G + gq) * D;
    const __nv_bfloat16* qg = p.q + qoff;
    const uint32_t lane_base = tm + ((uint32_t)(r & ~31) << 16);   // this warp's 32 TMEM lanes
    const uint32_t qs = sbase + L::kQ, vk = sbase + L::kVk, vv = sbase + L::kVv;
    float2* cs = reinterpret_cast<float2*>(reinterpret_cast<unsigned char*>(&b) - L::kBar + L::kCs);
    const float sl2 = p.scale * 1.4426950408889634f;   // scores in log2 units
    const int ro = rp.rot_offset, rr = rp.rot_dim, half = rr / 2;
    const bool rot_half = rp.pairing == KAMERA_ROPE_ROTATE_HALF;
    float m_run = -INFINITY, l_run = 0.f;
    int c0, c1;
    seq_chunks(p, seq, c0, c1);
    if (r == 0 && blk == 0 && h == 0 && (p.seq_start[seq] != c0 || p.seq_start[seq + 1] != c1))
        raise_err(p.err, KAMERA_DEVERR_DESCRIPTOR);
    // this thread's query row into the A operand of X = q V_k (K-major, 128B-swizzled; zero past T x G)
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (valid)
            x = __ldg(reinterpret_cast<const uint4*>(qg) + i);
        ptx::sts128(qs + (i >> 3) * 16384 + sw128(r, i & 7), x.x, x.y, x.z, x.w);
    }
    uint32_t n = 0, k = 0;   // tiles, chunks with tiles
    int prev_m = -1;         // rank of the previous chunk (-1: none yet)
    for (int c = c0; c < c1; ++c) {
        const KameraChunk& ch = p.chunks[c];
        const int32_t bad = prefill_check(ch, c, p);
        if (bad) {
            if (r == 0 && blk == 0 && h == 0)
                raise_err(p.err, bad);
            continue;
        }
        const int len = ch.len, m = ch.rank, nt = (len + kPfTok - 1) / kPfTok;
        if (nt == 0)
            continue;
        const int64_t fv = (int64_t)(p.layer * p.H + h) * D * m;   // V factors [L][H][d][m]
        // ---- V_k and the cos/sin of -delta; X = q V_k goes to the MMA lane
        bar_softmax();   // every thread is done with the previous chunk's cos/sin (and X(k-1) read V_k)
        for (int f = r; f < rp.n_freq; f += kPfRows) {
            float cc, sn;
            phase_cos_sin(-freq_delta(rp, ch, c, f), rp.inv_freq[f], cc, sn);
            cs[f] = make_float2(cc, sn);
        }
        if (m > 0)
            pf_stage_v<D>(vk, patch_ptr(ch, 1) + fv, m, r);
        ptx::fence_proxy_async();   // q and V_k, visible to the MMAs
        bar_softmax();
        ptx::mbar_arrive(ptx::smem_addr(&b.vk_ready));
        // ---- Q' = R(-delta) q, hi + lo, into TMEM: a rolled loop over the row's
        // 16-byte pieces (this code runs once a chunk; unrolled in full it would not
        // stay in the instruction cache).  The rotated range starts on a piece and
        // holds whole pieces (rot_offset a multiple of 8, rot_dim of 16 for
        // rotate-half and of 8 for interleaved pairs: the C ABI refuses the rest),
        // so a piece is rotated or not as a whole and its partners are one piece of
        // the row (rotate-half, half a multiple of 8) or inside it (interleaved).
        {
            const float4* cs4 = reinterpret_cast<const float4*>(cs);
#pragma unroll 1
            for (int pc = 0; pc < D / 8; ++pc) {
                float v[8];
                {
                    uint32_t w[4];
                    ptx::lds128(qs + (pc >> 3) * 16384 + sw128(r, pc & 7), w);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        v[2 * k] = bf16lo(w[k]);
                        v[2 * k + 1] = bf16hi(w[k]);
                    }
                }
                const int kk0 = 8 * pc - ro;
                if (kk0 >= 0 && kk0 < rr) {
                    if (rot_half) {
                        const bool neg = kk0 < half;
                        const int f0 = neg ? kk0 : kk0 - half, ppc = neg ? pc + half / 8 : pc - half / 8;
                        uint32_t pw[4];
                        ptx::lds128(qs + (ppc >> 3) * 16384 + sw128(r, ppc & 7), pw);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float4 t = cs4[(f0 >> 1) + k];   // cos/sin of f0 + 2k and f0 + 2k + 1
                            const float p0 = bf16lo(pw[k]), p1 = bf16hi(pw[k]);
                            v[2 * k] = fmaf(v[2 * k], t.x, neg ? -(p0 * t.y) : p0 * t.y);
                            v[2 * k + 1] = fmaf(v[2 * k + 1], t.z, neg ? -(p1 * t.w) : p1 * t.w);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {   // pair (2k, 2k + 1): frequency kk0 / 2 + k
                            const float2 t = cs[(kk0 >> 1) + k];
                            const float a = v[2 * k], bb = v[2 * k + 1];
                            v[2 * k] = fmaf(a, t.x, -(bb * t.y));
                            v[2 * k + 1] = fmaf(bb, t.x, a * t.y);
                        }
                    }
                }
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    wmma16::split_hl(v[2 * k], v[2 * k + 1], hw[k], lw[k]);
                tmem_st4(lane_base + L::kTmQh + 4 * pc, hw);
                tmem_st4(lane_base + L::kTmQl + 4 * pc, lw);
            }
        }
        // ---- X (from the MMA, in the S columns of this chunk's first tile), hi + lo
        {
            wmma16::tile_wait(ptx::smem_addr(&b.x_done), k & 1u, &b.abort, p.err, P.wait_ns);
            ptx::tc_fence_after();
            uint32_t x0[32], x1[32], xh[32], xl[32];
            const uint32_t sx = lane_base + L::kTmS + (n & 1) * kPfTok;
            tmem_ld32(sx, x0);
            tmem_ld32(sx + 32, x1);
            const int mz = m > 0 ? 16 * ((m + 15) >> 4) : 0;   // ranks the MMA wrote
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) {
                const uint32_t* src = cc < 16 ? x0 : x1;
                const int kk = 2 * (cc & 15), rank = 2 * cc;
                const float a0 = rank < mz ? __uint_as_float(src[kk]) : 0.f;
                const float a1 = rank < mz ? __uint_as_float(src[kk + 1]) : 0.f;
                wmma16::split_hl(a0, a1, xh[cc], xl[cc]);
            }
            tmem_st32(lane_base + L::kTmXh, xh);
            tmem_st32(lane_base + L::kTmXl, xl);
        }
        tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&b.a_ready));
        // ---- V_v of this chunk, into the buffer the fold two chunks back has finished with
        if (k >= 2)
            wmma16::tile_wait(ptx::smem_addr(&b.fold_done), (k - 2) & 1u, &b.abort, p.err, P.wait_ns);
        if (m > 0) {
            pf_stage_v<D>(vv + (k & 1) * (D * 128), patch_ptr(ch, 3) + fv, m, r);
            ptx::fence_proxy_async();
        }
        // ---- the previous chunk's sum_j p_j u'_j as hi + lo, for the fold, once its last P u' is done
        if (k > 0) {
            wmma16::tile_wait(ptx::smem_addr(&b.pv_done[(n - 1) & 1]), ((n - 1) >> 1) & 1u, &b.abort, p.err,
                              P.wait_ns);
            ptx::tc_fence_after();
            if (prev_m > 0)
                pf_split_w<D>(lane_base);
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&b.w_ready));
        }
        // ---- the tiles
        for (int tl = 0; tl < nt; ++tl, ++n) {
            const int ntok = min(kPfTok, len - tl * kPfTok);
            const uint32_t sb = L::kTmS + (n & 1) * kPfTok;
            wmma16::tile_wait(ptx::smem_addr(&b.s_full[n & 1]), (n >> 1) & 1u, &b.abort, p.err, P.wait_ns);
            ptx::tc_fence_after();
            uint32_t s0[32], s1[32];   // the S row (raw scores)
            tmem_ld32(lane_base + sb, s0);
            tmem_ld32(lane_base + sb + 32, s1);
            const bool tail = ntok < kPfTok;
            const float mt = sl2 * pf_extreme(s0, s1, ntok, sl2 < 0.f);   // the tile's largest score, log2 units
            const float m_new = fmaxf(m_run, mt);
            if (n == 0) {
                m_run = m_new;   // O is still empty
            } else if (__any_sync(0xFFFFFFFFu, m_new > m_run + kPfLazy)) {
                const float f = pf_ex2(m_run - m_new);
                l_run *= f;
                m_run = m_new;
                // O_v quiescent: the last P v (and, on a chunk's first tile, the previous fold)
                wmma16::tile_wait(ptx::smem_addr(&b.pv_done[(n - 1) & 1]), ((n - 1) >> 1) & 1u, &b.abort, p.err,
                                  P.wait_ns);
                if (tl == 0 && k > 0)
                    wmma16::tile_wait(ptx::smem_addr(&b.fold_done), (k - 1) & 1u, &b.abort, p.err, P.wait_ns);
                ptx::tc_fence_after();
                pf_rescale<D>(lane_base, f, m > 0 && tl > 0);
            }
            // weights p_j = 2^(sl2 s_j - m) as bf16 hi + lo pairs; pairs of fp32 lanes at a time
            uint32_t ph[32], pl[32];
            const uint64_t sl2x2 = ptx::f2_make(__float_as_uint(sl2), __float_as_uint(sl2));
            const uint64_t nmx2 = ptx::f2_make(__float_as_uint(-m_run), __float_as_uint(-m_run));
            const uint64_t neg1 = ptx::f2_make(__float_as_uint(-1.f), __float_as_uint(-1.f));
            uint64_t sum2 = 0ull;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint32_t* src = j < 16 ? s0 : s1;
                const int jj = 2 * (j & 15), col = (j < 16 ? 0 : 32) + jj;
                uint32_t a0, a1;
                asm("mov.b64 {%0, %1}, %2;" : "=r"(a0), "=r"(a1)
                    : "l"(ptx::f2_fma(ptx::f2_make(src[jj], src[jj + 1]), sl2x2, nmx2)));
                float p0 = pf_ex2(__uint_as_float(a0)), p1 = pf_ex2(__uint_as_float(a1));
                if (tail) {
                    p0 = col < ntok ? p0 : 0.f;
                    p1 = col + 1 < ntok ? p1 : 0.f;
                }
                const uint64_t pp = ptx::f2_make(__float_as_uint(p0), __float_as_uint(p1));
                sum2 = ptx::f2_add(sum2, pp);
                ph[j] = pack_bf16x2(p0, p1);
                pl[j] = ptx::f2_to_bf16x2(ptx::f2_fma(ptx::f2_from_bf16x2(ph[j]), neg1, pp));
            }
            {
                uint32_t x0, x1;
                asm("mov.b64 {%0, %1}, %2;" : "=r"(x0), "=r"(x1) : "l"(sum2));
                l_run += __uint_as_float(x0) + __uint_as_float(x1);
            }
            tmem_st32(lane_base + sb, ph);
            tmem_st32(lane_base + sb + kPfTok / 2, pl);
            tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&b.p_full[n & 1]));
        }
        prev_m = m;
        ++k;
    }
    // ---- the end: the last value patch, then out = O_v / l and the log-sum-exp
    if (n > 0) {
        wmma16::tile_wait(ptx::smem_addr(&b.pv_done[(n - 1) & 1]), ((n - 1) >> 1) & 1u, &b.abort, p.err, P.wait_ns);
        ptx::tc_fence_after();
        if (prev_m > 0)
            pf_split_w<D>(lane_base);
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&b.w_ready));
        wmma16::tile_wait(ptx::smem_addr(&b.fold_done), (k - 1) & 1u, &b.abort, p.err, P.wait_ns);
        ptx::tc_fence_after();
    }
    const float inv = n > 0 ? 1.f / l_run : 0.f;
    __nv_bfloat16* og = p.out + qoff;
#pragma unroll 1
    for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t o[32];
        if (n > 0) {
            tmem_ld32(lane_base + L::kTmOv + 32 * cb, o);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
                o[c] = 0u;
        }
        if (valid && !*static_cast<volatile int32_t*>(&b.abort)) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    w[k] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * k]) * inv, __uint_as_float(o[8 * q + 2 * k + 1]) * inv);
                ptx::stg128(og + 32 * cb + 8 * q, w);
            }
        }
    }
    if (valid && p.lse != nullptr)
        p.lse[((int64_t)seq * p.T + tok) * HQ + (int64_t)h * G + gq] =
            n > 0 ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
}

// One CTA per unit u = (sequence, KV head, 128-row block), the block fastest so
// the CTAs that read the same rows run together and share them in L2.
template <int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ PrefillLaunch P)
{
    using L = PfLayout<D>;
    const PrefillParams& p = P.p;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;   // swizzled tiles sit on 1024-byte boundaries
    const uint32_t sbase = raw + pad;
    PfBars& b = *reinterpret_cast<PfBars*>(smem_raw + pad + L::kBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t u = blockIdx.x;
    const int blk = (int)(u % p.blocks), h = (int)((u / p.blocks) % p.H);
    const int seq = (int)(u / ((int64_t)p.blocks * p.H));

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::NS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&b.full[s]), 1 + 32);   // the TMA issue + the warp's stores
            ptx::mbar_init(ptx::smem_addr(&b.empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_addr(&b.s_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&b.p_full[i]), kPfRows);
            ptx::mbar_init(ptx::smem_addr(&b.pv_done[i]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&b.vk_ready), kPfRows);
        ptx::mbar_init(ptx::smem_addr(&b.x_done), 1);
        ptx::mbar_init(ptx::smem_addr(&b.a_ready), kPfRows);
        ptx::mbar_init(ptx::smem_addr(&b.w_ready), kPfRows);
        ptx::mbar_init(ptx::smem_addr(&b.fold_done), 1);
        ptx::mbar_init(ptx::smem_addr(&b.drained), 1);
        b.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kPfProd && lane == 0) {
        ptx::prefetch_tmap(&P.map_k);
        ptx::prefetch_tmap(&P.map_v);
    }
    if (warp == kPfMma) {
        ptx::tmem_alloc(ptx::smem_addr(&b.tmem), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = b.tmem;

    if (warp < 4)
        pf_softmax<D>(P, sbase, b, tm, seq, h, blk, threadIdx.x);
    else if (warp == kPfProd)
        pf_producer<D>(P, sbase, b, seq, h, lane);
    else if (lane == 0)
        pf_mma<D>(P, sbase, b, tm, seq);

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kPfMma) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, 512);
    }
}

template <int D>
cudaError_t launch_prefill_d(const PrefillParams& p, cudaStream_t stream)
{
    using L = PfLayout<D>;
    PrefillLaunch P;
    std::memset(&P, 0, sizeof(P));
    P.p = p;
    P.wait_ns = wait_limit_ns();
    P.withhold = test_withhold_loads() ? 1 : 0;
    const int64_t width = (int64_t)p.H * D;
    if (!make_rows_map(&P.map_k, p.k, p.num_rows, width, p.row_stride, 64, kPfTok) ||
        !make_rows_map(&P.map_v, p.v, p.num_rows, width, p.row_stride, 64, kPfTok))
        return cudaErrorInvalidValue;
    // set at every launch: the attribute belongs to the current device's context
    const cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
    if (e != cudaSuccess)
        return e;
    const int64_t units = (int64_t)p.n_seqs * p.H * p.blocks;
    prefill_kernel<D><<<(unsigned)units, kPfThreads, L::kBytes, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int head_dim, int max_rank)
{
    return (head_dim == 64 || head_dim == 128) && max_rank >= 0 && max_rank <= kPfMP;
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream)
{
    if ((int64_t)p.n_seqs * p.H * p.blocks < 1)
        return cudaSuccess;
    return p.d == 128 ? launch_prefill_d<128>(p, stream) : launch_prefill_d<64>(p, stream);
}

}  // namespace kamera
