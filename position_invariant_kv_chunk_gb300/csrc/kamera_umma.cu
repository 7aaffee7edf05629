// kamera_umma.cu -- tensor-core path of the Kamera operator on sm_103a.
//
// Reuse equation (gist.science technical summary, section 2):
//     KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T
// The rank-m patch U_m V_m^T of one (chunk, layer, row segment) over a tile of
// 128 tokens is a 128 x w x m contraction (w = head_dim for GQA/MHA, 128 for
// an MLA c_KV block, 64 or 128 for k_rope).  It runs on the 5th-generation
// tensor cores: one tcgen05.mma (M=128, N=w, K=16, bf16 in, fp32 out) per 16
// ranks, accumulator in TMEM.  Everything else streams through shared memory:
//
//   warp 0    producer: canonical rows of the tile with tiled TMA loads from a
//             tensor map of the store (128B-swizzled boxes of 64 columns x 128
//             rows; 16-row boxes for the ragged tail), the U tiles of chunks
//             the host mapped (TMA boxes swizzled like the MMA operand), the
//             tile's pool slots, and the per-chunk cos/sin table (phase formed
//             and reduced in fp64).
//   warp 1    operands + MMA: 16-byte async copies build the U tiles the maps
//             do not cover and V_m in the 128B-swizzled K-major layout ahead of
//             use; the copying lanes fence their writes into the async proxy;
//             one lane issues the MMAs and commits them to mbarriers.  Also
//             owns TMEM.
//   warps 4-15 epilogue: three warps per TMEM sub-partition, each owning a
//             third of the columns (whole RoPE pairs) of the same 32 token
//             rows; thread = token row = TMEM lane.  tcgen05.ld the patch, read the canonical
//             row (swizzled, conflict-free), rotate the RoPE pairs in fp32, add,
//             round once to bf16 and write back in place; then each warp stores
//             its columns of its 32 rows to their pool slots with coalesced
//             16-byte stores.
//
// The grid is persistent (one CTA per SM).  The tiles of a call, ordered
// (layer, chunk, segment, tile), are split into equal contiguous ranges:
// consecutive tiles of a CTA share V_m (a job is one chunk, layer and segment)
// and the cos/sin table (one chunk), and every range mixes the segments of its
// chunks (rotated keys and plain values; 128-wide c_KV blocks and the narrower
// k_rope) in the proportion of the whole call, which keeps the CTAs' work even.  Every wait is
// bounded in time: on expiry the CTA records KAMERA_DEVERR_TIMEOUT, drains its
// own copies and MMAs, frees TMEM and returns.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"
#include "kamera_ptx.cuh"

namespace kamera {

namespace {

constexpr int kTileM = 128;                     // tokens per tile = UMMA M = TMEM lanes
constexpr int kWMax = 128;                      // widest segment = UMMA N
constexpr int kHalfBytes = kTileM * 128;        // one 64-column swizzled box of 128 rows
constexpr int kRowsBytes = 2 * kHalfBytes;      // canonical rows of a tile (w <= 128)
constexpr int kTabOff = kRowsBytes;             // cos/sin table of the tile's chunk (1 KB)
constexpr int kSlotOff = kRowsBytes + 1024;      // the tile's 128 destination slots (int64)
constexpr int kStageBytes = kRowsBytes + 2048;  // rows + table + slots, 1024-aligned
constexpr int kAtomBytes = kTileM * 128;        // one 64-rank K atom of a 128-row operand
constexpr int kEpiPerSub = 3;                   // epilogue warps per TMEM sub-partition
constexpr int kEpiWarps = 4 * kEpiPerSub;
constexpr int kEpiWarp0 = 4;                     // warpgroup 0: producer, MMA and two idle warps
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
// Warp w runs on SM sub-partition w % 4, whose register file holds 16384
// registers: the busiest sub-partition bounds the registers per thread at
// launch.  Warpgroup 0 then lowers its budget and the epilogue warpgroups
// take the freed registers (each sub-partition holds one warp of each group).
constexpr int kRegCap = (16384 / (32 * ((kThreads / 32 + 3) / 4))) & ~7;   // allocated in units of 8
constexpr int kRegsLow = 72;                     // producer / MMA warpgroup
constexpr int kRegsEpi = 144;                    // epilogue warpgroups
static_assert(128 * kRegsLow + 32 * kEpiWarps * kRegsEpi <= kThreads * kRegCap, "register split exceeds the launch");
static_assert(32 * (kRegsLow + kEpiPerSub * kRegsEpi) <= 16384, "register split exceeds a sub-partition");
constexpr uint32_t kTmemCols = 2 * kWMax;       // two accumulators
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr int kTailRows = 16;                   // box height of the tail tensor maps
constexpr int kMapChunksFew = 8;                // U map tables: calls of <= 8 chunks ...
constexpr int kMapChunksMany = 104;             // ... and larger ones (the parameter block stays < 32 KB)

struct UmmaParams {
    CUtensorMap map_full[2];   // per array (K|V, or the MLA row): 64 x 128 boxes
    CUtensorMap map_tail[2];   // 64 x 16 boxes
    RowsParams r;
    int32_t family;
    int32_t Z;                 // row segments
    int32_t withhold;          // test hook: the producer issues no loads, so the first waits run out
    uint64_t wait_ns;          // bound of every pipeline wait (drains keep kTimeoutNs)
};

// Per-call U tensor maps (from a host copy of the descriptors): chunk c < MC
// with u_rank[c] > 0 has maps 2c (K or c_KV factor) and 2c+1 (V or k_rope
// factor) over its [L*FH][len][m] U array; boxes of min(m, 64) ranks x 128
// rows, swizzled to match the MMA operand layout.  Beside each map sit the
// host copy's rank, length and the two U base addresses it was encoded from:
// a chunk's tiles move through its maps only when the device descriptor names
// the same four values, so a host copy that disagrees with the device array
// can never point a load at memory the descriptor does not name.
template <int MC>
struct UmmaLaunch {
    UmmaParams core;
    CUtensorMap map_u[2 * MC];
    int32_t u_rank[MC];
    int32_t u_len[MC];
    const void* u_base[MC][2];
};

template <int MC>
__device__ __forceinline__ bool u_map_matches(const UmmaLaunch<MC>& P, int c, const KameraChunk& ch)
{
    return ch.rank > 0 && P.u_rank[c] == ch.rank && P.u_len[c] == ch.len && P.u_base[c][0] == ch.patch_ptrs[0] &&
           P.u_base[c][1] == ch.patch_ptrs[2];
}

// Whether chunk c's U tiles move by its tensor map: bit c of the mask the
// prologue builds from u_map_matches (one check per chunk and CTA).
template <int MC>
__device__ __forceinline__ bool u_mapped(const uint32_t* umask, int c, int rank)
{
    return rank > 0 && c < MC && ((umask[c >> 5] >> (c & 31)) & 1u);
}

template <int KA>
struct Geometry {
    static constexpr int LA = KA == 1 ? 2 : 1;  // operand lookahead (tiles)
    static constexpr int D = LA + 1;            // U operand buffers
    static constexpr int S = KA == 1 ? 4 : 2;   // row stages
    static constexpr int kUBytes = KA * kAtomBytes;
    static constexpr int kVBytes = KA * kWMax * 128;
    static constexpr int kUOff = S * kStageBytes;
    static constexpr int kVOff = kUOff + D * kUBytes;
    static constexpr int kSharedOff = kVOff + 2 * kVBytes;
};

struct Seg {
    int array, e0, w, rot, u_idx, v_idx, fh, FH, vm_row0, vm_rows;
};

__device__ __forceinline__ Seg segment(const UmmaParams& p, int z)
{
    Seg s;
    if (p.family == FAMILY_GQA) {
        const int kv = z & 1, h = z >> 1;
        s.array = kv;
        s.e0 = h * p.r.d;
        s.w = p.r.d;
        s.rot = (kv == 0 && p.r.rope.rot_dim > 0) ? 1 : 0;
        s.u_idx = 2 * kv;
        s.v_idx = 2 * kv + 1;
        s.fh = h;
        s.FH = p.r.H;
        s.vm_row0 = 0;
        s.vm_rows = p.r.d;
    } else {
        const int nb = p.r.kv_lora / kWMax;
        s.array = 0;
        s.fh = 0;
        s.FH = 1;
        if (z < nb) {
            s.e0 = kWMax * z;
            s.w = kWMax;
            s.rot = 0;
            s.u_idx = 0;
            s.v_idx = 1;
            s.vm_row0 = kWMax * z;
            s.vm_rows = p.r.kv_lora;
        } else {
            s.e0 = p.r.kv_lora;
            s.w = p.r.d - p.r.kv_lora;
            s.rot = p.r.rope.rot_dim > 0 ? 1 : 0;
            s.u_idx = 2;
            s.v_idx = 3;
            s.vm_row0 = 0;
            s.vm_rows = p.r.d - p.r.kv_lora;
        }
    }
    return s;
}

__device__ __forceinline__ int chunk_tiles(const KameraChunk& ch, int c, const RowsParams& r)
{
    return check_chunk(ch, c, r, false) ? 0 : (ch.len + kTileM - 1) / kTileM;
}

// Walks the CTA's tiles in (layer, chunk, segment, tile) order; every role
// runs its own copy.  lz = layer * Z + segment.
struct Cursor {
    int lz, c, t, ntile;
    KameraChunk ch;

    __device__ void load(const UmmaParams& p)
    {
        ch = p.r.chunks[c];
        ntile = chunk_tiles(ch, c, p.r);
    }
    __device__ void next(const UmmaParams& p)
    {
        if (++t < ntile)
            return;
        t = 0;
        const int l = lz / p.Z;
        if (++lz < (l + 1) * p.Z)   // the chunk's next segment
            return;
        lz = l * p.Z;               // segment 0 of the next chunk with tiles
        do {
            if (++c == p.r.n_chunks) {
                c = 0;
                lz += p.Z;
            }
            load(p);
        } while (ntile == 0);
    }
};

// What the epilogue needs to know of the tile in a stage (written by the producer).
struct TileInfo {
    int32_t l, z, m, ntok, rot;
};

struct Shared {
    uint64_t full[4], empty[4], tfull[2], tempty[2], uempty[3], ufull[3], vmempty[2], mmadone;
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t start_lz, start_rem, start_c, start_t, count;
    int32_t stage_tag[4];
    TileInfo tinfo[4];
    uint32_t umask[(kMapChunksMany + 31) / 32];
    int64_t part[kThreads];
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* err,
                                         uint64_t limit)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((it & 63) == 0) {
            if (*abort_flag)
                return false;
            if (ptx::globaltimer() - t0 > limit) {
                *abort_flag = 1;
                raise_err(err, KAMERA_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// The whole warp waits; a timeout seen by any lane is seen by all (the abort
// flag reaches every polling lane), so the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* err,
                                          uint64_t limit)
{
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err, limit)) != 0;
}

// time-bounded wait that ignores the abort flag (used while draining)
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer() - t0 > kTimeoutNs)
            return;
}

// Byte offset of the 16-byte piece (row r, piece kc) in a 128B-swizzled
// K-major operand with atoms of `atom_bytes` (64 ranks per atom).
__device__ __forceinline__ uint32_t operand_offset(int r, int kc, uint32_t atom_bytes)
{
    return (kc >> 3) * atom_bytes + r * 128 + ((((kc & 7) ^ (r & 7))) << 4);
}

// Copies `rows` rows of a [*, m] bf16 factor (row stride m) into the
// 128B-swizzled K-major operand layout at `dst`, zero-filling ranks
// m..mpad-1, in async copies of G bytes (G divides the 2m-byte row, so every
// piece stays inside one 16-byte chunk of the swizzled layout).  The 32 lanes
// of the calling warp share the work.
template <int G>
__device__ __forceinline__ void load_operand_g(uint32_t dst, const __nv_bfloat16* src, int rows, int m, int mpad,
                                               uint32_t atom_bytes, int lane)
{
    constexpr int E = G / 2;   // elements per piece
    const int pr = m / E, pp = (mpad - m) / E;
    const bool pow2 = (pr & (pr - 1)) == 0;
    const int sh = 31 - __clz(pr);
    for (int p = lane; p < rows * pr; p += 32) {
        const int r = pow2 ? p >> sh : p / pr;
        const int k = (p - r * pr) * E;
        const uint32_t d = dst + operand_offset(r, k >> 3, atom_bytes) + (k & 7) * 2;
        if constexpr (G == 16)
            ptx::cp_async16(d, src + (size_t)r * m + k);
        else
            ptx::cp_async_small<G>(d, src + (size_t)r * m + k);
    }
    for (int p = lane; p < rows * pp; p += 32) {
        const int r = p / pp, k = m + (p - r * pp) * E;
        const uint32_t d = dst + operand_offset(r, k >> 3, atom_bytes) + (k & 7) * 2;
        if constexpr (G == 16)
            ptx::st_shared_zero16(d);
        else if constexpr (G == 8)
            asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(d), "r"(0) : "memory");
        else
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(d), "r"(0) : "memory");
    }
}

__device__ __forceinline__ void load_operand(uint32_t dst, const __nv_bfloat16* src, int rows, int m, int mpad,
                                             uint32_t atom_bytes, int lane)
{
    if ((m & 7) == 0) {
        load_operand_g<16>(dst, src, rows, m, mpad, atom_bytes, lane);
    } else if ((m & 3) == 0) {
        load_operand_g<8>(dst, src, rows, m, mpad, atom_bytes, lane);
    } else if ((m & 1) == 0) {
        load_operand_g<4>(dst, src, rows, m, mpad, atom_bytes, lane);
    } else {   // odd rank: rows are only 2-byte aligned
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
        for (int p = lane; p < rows * mpad; p += 32) {
            const int r = p / mpad, k = p - r * mpad;
            const uint16_t v = k < m ? s16[(size_t)r * m + k] : (uint16_t)0;
            ptx::st_shared_u16(dst + operand_offset(r, k >> 3, atom_bytes) + (k & 7) * 2, v);
        }
    }
}

// Shared address of the 16-byte piece q of row tt in a stage's canonical rows
// (two 64-column boxes, 128-byte swizzle: piece q of row tt sits at chunk q ^ (tt & 7)).
__device__ __forceinline__ uint32_t piece_addr(uint32_t rows, int tt, int q)
{
    return rows + (q >> 3) * kHalfBytes + tt * 128 + ((((q & 7) ^ (tt & 7))) << 4);
}

// One round of a thread's share of a tile row: 8 columns at a (span A) and
// the 8 at b (span B; RoPE partners for rotate-half), read from the row in
// shared memory, combined with the patch (fp32, from TMEM), rounded once to
// bf16 and written back in place.  MODE: 0 no rotation, 1 rotate-half pairs
// (a+i, b+i), 2 interleaved pairs inside each span; PATCH: a rank-m patch is
// present.  Arithmetic runs on packed fp32 pairs; per element it is the same
// sequence of roundings as x*c + round(y*(-s)) [+ patch].
//   table, rotate-half: cos[64] | sin[64] | -sin[64]      (fp32, by frequency)
//   table, interleaved: (cos, cos)[64] | (-sin, sin)[64]  (fp32 pairs)
template <int MODE, bool PATCH>
__device__ __forceinline__ void epilogue_round(uint32_t rows, int tt, int a, int b, uint32_t tab,
                                               const uint32_t (&pa)[8], const uint32_t (&pb)[8])
{
    uint32_t va[4], vb[4], t0[4], t1[4], t2[4], t3[4], t4[4], t5[4];
    ptx::lds128(piece_addr(rows, tt, a >> 3), va);
    ptx::lds128(piece_addr(rows, tt, b >> 3), vb);
    if constexpr (MODE == 1) {   // 8 frequencies a..a+7: cos, sin, -sin
        const uint32_t f0 = (uint32_t)a * 4u;
        ptx::lds128(tab + f0, t0);
        ptx::lds128(tab + f0 + 16, t1);
        ptx::lds128(tab + 256 + f0, t2);
        ptx::lds128(tab + 256 + f0 + 16, t3);
        ptx::lds128(tab + 512 + f0, t4);
        ptx::lds128(tab + 512 + f0 + 16, t5);
    } else if constexpr (MODE == 2) {   // 4 frequencies per span: (c, c) and (-s, s) pairs
        const uint32_t fa = (uint32_t)(a >> 1) * 8u, fb = (uint32_t)(b >> 1) * 8u;
        ptx::lds128(tab + fa, t0);
        ptx::lds128(tab + fa + 16, t1);
        ptx::lds128(tab + 512 + fa, t2);
        ptx::lds128(tab + 512 + fa + 16, t3);
        ptx::lds128(tab + fb, t4);
        ptx::lds128(tab + fb + 16, t5);
    }
    uint64_t xa[4], xb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xa[i] = ptx::f2_from_bf16x2(va[i]);
        xb[i] = ptx::f2_from_bf16x2(vb[i]);
    }
    if constexpr (MODE == 1) {
        const uint64_t c[4] = {ptx::f2_make(t0[0], t0[1]), ptx::f2_make(t0[2], t0[3]), ptx::f2_make(t1[0], t1[1]),
                               ptx::f2_make(t1[2], t1[3])};
        const uint64_t sn[4] = {ptx::f2_make(t2[0], t2[1]), ptx::f2_make(t2[2], t2[3]), ptx::f2_make(t3[0], t3[1]),
                                ptx::f2_make(t3[2], t3[3])};
        const uint64_t ns[4] = {ptx::f2_make(t4[0], t4[1]), ptx::f2_make(t4[2], t4[3]), ptx::f2_make(t5[0], t5[1]),
                                ptx::f2_make(t5[2], t5[3])};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t oa = ptx::f2_fma(xa[i], c[i], ptx::f2_mul(xb[i], ns[i]));
            const uint64_t ob = ptx::f2_fma(xb[i], c[i], ptx::f2_mul(xa[i], sn[i]));
            xa[i] = oa;
            xb[i] = ob;
        }
    } else if constexpr (MODE == 2) {
        const uint64_t cca[4] = {ptx::f2_make(t0[0], t0[1]), ptx::f2_make(t0[2], t0[3]), ptx::f2_make(t1[0], t1[1]),
                                 ptx::f2_make(t1[2], t1[3])};
        const uint64_t ssa[4] = {ptx::f2_make(t2[0], t2[1]), ptx::f2_make(t2[2], t2[3]), ptx::f2_make(t3[0], t3[1]),
                                 ptx::f2_make(t3[2], t3[3])};
        uint32_t u0[4], u1[4];   // the b span's (-s, s) pairs
        ptx::lds128(tab + 512 + (uint32_t)(b >> 1) * 8u, u0);
        ptx::lds128(tab + 512 + (uint32_t)(b >> 1) * 8u + 16, u1);
        const uint64_t ccb[4] = {ptx::f2_make(t4[0], t4[1]), ptx::f2_make(t4[2], t4[3]), ptx::f2_make(t5[0], t5[1]),
                                 ptx::f2_make(t5[2], t5[3])};
        const uint64_t ssb[4] = {ptx::f2_make(u0[0], u0[1]), ptx::f2_make(u0[2], u0[3]), ptx::f2_make(u1[0], u1[1]),
                                 ptx::f2_make(u1[2], u1[3])};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            xa[i] = ptx::f2_fma(xa[i], cca[i], ptx::f2_mul(ptx::f2_swap(xa[i]), ssa[i]));
            xb[i] = ptx::f2_fma(xb[i], ccb[i], ptx::f2_mul(ptx::f2_swap(xb[i]), ssb[i]));
        }
    }
    if constexpr (PATCH) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            xa[i] = ptx::f2_add(xa[i], ptx::f2_make(pa[2 * i], pa[2 * i + 1]));
            xb[i] = ptx::f2_add(xb[i], ptx::f2_make(pb[2 * i], pb[2 * i + 1]));
        }
    }
    ptx::sts128(piece_addr(rows, tt, a >> 3), ptx::f2_to_bf16x2(xa[0]), ptx::f2_to_bf16x2(xa[1]),
                ptx::f2_to_bf16x2(xa[2]), ptx::f2_to_bf16x2(xa[3]));
    ptx::sts128(piece_addr(rows, tt, b >> 3), ptx::f2_to_bf16x2(xb[0]), ptx::f2_to_bf16x2(xb[1]),
                ptx::f2_to_bf16x2(xb[2]), ptx::f2_to_bf16x2(xb[3]));
}

// A thread's share of a tile row: R rounds over the spans at a0 and b0.  The
// TMEM load of round j+1 is issued before round j's arithmetic, so its
// latency hides behind that work; the rounds go two per loop trip, one per
// TMEM buffer.
template <int MODE, bool PATCH>
__device__ __forceinline__ void epilogue_spans(uint32_t rows, int tt, int a0, int b0, int R, uint32_t tacc,
                                               uint32_t tab, bool valid)
{
    uint32_t p0a[8], p0b[8], p1a[8], p1b[8];
    if constexpr (PATCH)   // warp-collective: every lane loads, valid row or not
        ptx::tmem_ld8x2_issue(tacc + a0, tacc + b0, p0a, p0b);
#pragma unroll 1
    for (int j = 0; j < R; j += 2) {
        const int r0 = 8 * j;
        if constexpr (PATCH) {
            ptx::tmem_wait8x2(p0a, p0b);
            if (j + 1 < R)
                ptx::tmem_ld8x2_issue(tacc + a0 + r0 + 8, tacc + b0 + r0 + 8, p1a, p1b);
        }
        if (valid)
            epilogue_round<MODE, PATCH>(rows, tt, a0 + r0, b0 + r0, tab, p0a, p0b);
        if (j + 1 < R) {
            if constexpr (PATCH) {
                ptx::tmem_wait8x2(p1a, p1b);
                if (j + 2 < R)
                    ptx::tmem_ld8x2_issue(tacc + a0 + r0 + 16, tacc + b0 + r0 + 16, p0a, p0b);
            }
            if (valid)
                epilogue_round<MODE, PATCH>(rows, tt, a0 + r0 + 8, b0 + r0 + 8, tab, p1a, p1b);
        }
    }
}

// The epilogue specialised for the tile's rotation mode and patch: one
// dispatch per tile, branch-free rounds inside.
__device__ __forceinline__ void epilogue_dispatch(int mode, bool patch, uint32_t rows, int tt, int a0, int b0, int R,
                                                  uint32_t tacc, uint32_t tab, bool valid)
{
    switch (mode * 2 + (patch ? 1 : 0)) {
    case 1: epilogue_spans<0, true>(rows, tt, a0, b0, R, tacc, tab, valid); break;
    case 2: epilogue_spans<1, false>(rows, tt, a0, b0, R, tacc, tab, valid); break;
    case 3: epilogue_spans<1, true>(rows, tt, a0, b0, R, tacc, tab, valid); break;
    case 4: epilogue_spans<2, false>(rows, tt, a0, b0, R, tacc, tab, valid); break;
    case 5: epilogue_spans<2, true>(rows, tt, a0, b0, R, tacc, tab, valid); break;
    default: break;   // no rotation and no patch: the row is stored as loaded
    }
}

}  // namespace

template <int KA, int MC>
__global__ void __maxnreg__(kRegCap) relocate_patch_umma_kernel(const __grid_constant__ UmmaLaunch<MC> P)
{
    const UmmaParams& p = P.core;
    using G = Geometry<KA>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // swizzle atoms need 1024-byte alignment
    uint8_t* gbase = smem_raw + (base - raw);
    Shared& sh = *reinterpret_cast<Shared*>(gbase + G::kSharedOff);
    volatile int32_t* abort_flag = &sh.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const RowsParams& r = p.r;

    // ---------------------------------------------------------- prologue
    if (tid == 0) {
        for (int i = 0; i < G::S; ++i) {
            ptx::mbar_init(ptx::smem_addr(&sh.full[i]), 1 + 32);   // TMA issue + the slot copies of 32 lanes
            ptx::mbar_init(ptx::smem_addr(&sh.empty[i]), kEpiWarps);
            sh.stage_tag[i] = -1;
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_addr(&sh.tfull[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.tempty[i]), kEpiWarps);
            ptx::mbar_init(ptx::smem_addr(&sh.vmempty[i]), 1);
        }
        for (int i = 0; i < G::D; ++i) {
            ptx::mbar_init(ptx::smem_addr(&sh.uempty[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.ufull[i]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sh.mmadone), 1);
        sh.abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async();
    }
    if (tid == 32) {
        for (int i = 0; i < 2; ++i) {
            ptx::prefetch_tmap(&p.map_full[i]);
            ptx::prefetch_tmap(&p.map_tail[i]);
        }
    }
    // chunks whose U tiles may move by their tensor maps: the host copy the maps
    // were encoded from must name the device descriptor's rank, length and U
    // factors; a mapped chunk that differs takes the copy path and reports
    // KAMERA_DEVERR_DESCRIPTOR
    if (tid < 32 * ((MC + 31) / 32)) {
        bool ok = false;
        if (tid < MC && tid < r.n_chunks && P.u_rank[tid] > 0) {
            const KameraChunk ch = r.chunks[tid];
            ok = u_map_matches(P, tid, ch);
            if (!ok && blockIdx.x == 0)
                raise_err(r.err, KAMERA_DEVERR_DESCRIPTOR);
        }
        const uint32_t bits = __ballot_sync(0xffffffffu, ok);
        if (lane == 0)
            sh.umask[warp] = bits;
    }
    // tiles per chunk: each thread sums a contiguous block of chunks
    const int n = r.n_chunks;
    const int per = (n + kThreads - 1) / kThreads;
    const int c_lo = min(n, tid * per), c_hi = min(n, c_lo + per);
    int64_t mine = 0;
#pragma unroll 4
    for (int c = c_lo; c < c_hi; ++c) {
        const KameraChunk ch = r.chunks[c];
        const int32_t bad = check_chunk(ch, c, r, false);
        if (bad) {
            if (blockIdx.x == 0)
                raise_err(r.err, bad);
        } else {
            mine += (ch.len + kTileM - 1) / kTileM;
        }
    }
    sh.part[tid] = mine;
    __syncthreads();
    if (tid == 0) {
        int64_t run = 0;
        for (int i = 0; i < kThreads; ++i) {
            const int64_t v = sh.part[i];
            sh.part[i] = run;
            run += v;
        }
        const int64_t TC = run;
        const int64_t T = TC * r.L * p.Z;
        const int64_t b0 = T * blockIdx.x / gridDim.x, b1 = T * (blockIdx.x + 1) / gridDim.x;
        sh.count = (int32_t)(b1 - b0);
        const int64_t LB = TC * p.Z;   // tiles of one layer
        sh.start_lz = LB ? (int32_t)(b0 / LB) * p.Z : 0;   // layer of the first tile (segment added below)
        sh.start_rem = (int32_t)(LB ? b0 % LB : 0);         // its offset inside the layer
        sh.start_c = 0;
        sh.start_t = 0;
    }
    __syncthreads();
    if (sh.count > 0) {
        const int64_t rem = sh.start_rem;
        const int64_t lo = (int64_t)p.Z * sh.part[tid];   // a chunk holds Z * (its tiles) of a layer
        if (rem >= lo && rem < lo + (int64_t)p.Z * mine) {   // exactly one thread owns the starting tile
            int64_t acc = lo;
            for (int c = c_lo; c < c_hi; ++c) {
                const KameraChunk ch = r.chunks[c];
                const int nt = chunk_tiles(ch, c, r);
                if (rem < acc + (int64_t)p.Z * nt) {
                    const int64_t o = rem - acc;
                    sh.start_lz += (int32_t)(o / nt);
                    sh.start_t = (int32_t)(o % nt);
                    sh.start_c = c;
                    break;
                }
                acc += (int64_t)p.Z * nt;
            }
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&sh.tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const int count = sh.count;
    const uint32_t tmem = sh.tmem_base;

    Cursor cur;
    cur.lz = sh.start_lz;
    cur.c = sh.start_c;
    cur.t = sh.start_t;
    if (count > 0)
        cur.load(p);

    const uint32_t ubase = base + G::kUOff, vbase = base + G::kVOff;

    if (warp < kEpiWarp0) {
    ptx::setmaxnreg_dec<kRegsLow>();
    if (warp == 0 && count > 0 && !p.withhold) {
        // ------------------------------------------------------ producer
        int issued = 0, pu = 0;
        uint32_t upar = 0, uload = 0;   // per U buffer: phase parity of its TMA loads; last use was a TMA load
        for (int i = 0; i < count; ++i, cur.next(p)) {
            const int s = i % G::S, rnd = i / G::S;
            if (!warp_wait(ptx::smem_addr(&sh.empty[s]), (rnd & 1) ^ 1, abort_flag, r.err, p.wait_ns))
                break;
            const int l = cur.lz / p.Z, z = cur.lz - l * p.Z;
            const Seg sg = segment(p, z);
            const KameraChunk& ch = cur.ch;
            const int tok0 = cur.t * kTileM;
            const int ntok = min(kTileM, ch.len - tok0);
            const bool rot = sg.rot && chunk_turns(r.rope, ch, cur.c);
            if (rot && sh.stage_tag[s] != cur.c) {   // cos/sin table in the epilogue's operand order
                float* tab = reinterpret_cast<float*>(gbase + s * kStageBytes + kTabOff);
                const bool half_pairs = r.rope.pairing == KAMERA_ROPE_ROTATE_HALF;
                for (int f = lane; f < r.rope.n_freq; f += 32) {
                    float c_, s_;
                    phase_cos_sin(freq_delta(r.rope, ch, cur.c, f), r.rope.inv_freq[f], c_, s_);
                    if (half_pairs) {
                        tab[f] = c_;
                        tab[64 + f] = s_;
                        tab[128 + f] = -s_;
                    } else {
                        tab[2 * f] = c_;
                        tab[2 * f + 1] = c_;
                        tab[128 + 2 * f] = -s_;
                        tab[128 + 2 * f + 1] = s_;
                    }
                }
                __syncwarp();
                if (lane == 0)
                    sh.stage_tag[s] = cur.c;
            }
            if (ch.rank > 0) {   // U tile of a mapped chunk: one or two swizzled boxes into the U ring
                const int u = pu % G::D;
                if (u_mapped<MC>(sh.umask, cur.c, ch.rank)) {
                    if (!warp_wait(ptx::smem_addr(&sh.uempty[u]), ((pu / G::D) & 1) ^ 1, abort_flag, r.err, p.wait_ns))
                        break;
                    if (lane == 0) {
                        const int nbox = ch.rank > 64 ? 2 : 1;
                        const uint32_t ufull = ptx::smem_addr(&sh.ufull[u]);
                        ptx::mbar_arrive_expect_tx(ufull, (uint32_t)(nbox * min(ch.rank, 64) * 2 * kTileM));
                        const CUtensorMap* map = &P.map_u[2 * cur.c + (sg.u_idx >> 1)];
                        for (int x = 0; x < nbox; ++x)
                            ptx::tma_load_3d(ubase + u * G::kUBytes + x * kAtomBytes, map, 64 * x, tok0,
                                             l * sg.FH + sg.fh, ufull);
                    }
                    upar ^= 1u << u;
                    uload |= 1u << u;
                } else {
                    uload &= ~(1u << u);
                }
                ++pu;
            }
            {   // the tile's destination slots (-1 past its last row) and its description
                const uint32_t slots = base + s * kStageBytes + kSlotOff;
                const int64_t* map = ch.dst_slot_mapping + tok0;
#pragma unroll
                for (int j = lane; j < kTileM; j += 32) {
                    if (j < ntok)
                        ptx::cp_async_small<8>(slots + 8 * j, map + j);
                    else
                        ptx::st_shared_s64(slots + 8 * j, -1);
                }
                ptx::cp_async_mbar_arrive_noinc(ptx::smem_addr(&sh.full[s]));
                if (lane == 0)
                    sh.tinfo[s] = TileInfo{l, z, ch.rank, ntok, rot ? 1 : 0};
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t full = ptx::smem_addr(&sh.full[s]);
                const uint32_t rows = base + s * kStageBytes;
                const int nx = sg.w >> 6;   // 64-column boxes
                const int y = (int)(ch.src_offset + tok0);
                if (ntok == kTileM) {
                    ptx::mbar_arrive_expect_tx(full, (uint32_t)(nx * kHalfBytes));
                    for (int x = 0; x < nx; ++x)
                        ptx::tma_load_3d(rows + x * kHalfBytes, &p.map_full[sg.array], sg.e0 + 64 * x, y, l, full);
                } else {
                    const int nb = (ntok + kTailRows - 1) / kTailRows;
                    ptx::mbar_arrive_expect_tx(full, (uint32_t)(nx * nb * kTailRows * 128));
                    for (int x = 0; x < nx; ++x)
                        for (int b = 0; b < nb; ++b)
                            ptx::tma_load_3d(rows + x * kHalfBytes + b * kTailRows * 128, &p.map_tail[sg.array],
                                             sg.e0 + 64 * x, y + b * kTailRows, l, full);
                }
            }
            __syncwarp();
            ++issued;
        }
        // no TMA load or copy may still be writing shared memory when the CTA exits
        ptx::cp_async_wait<0>();
        if (lane == 0) {
            for (int j = max(0, issued - G::S); j < issued; ++j)
                drain_bar(ptx::smem_addr(&sh.full[j % G::S]), (j / G::S) & 1);
            for (int u = 0; u < G::D; ++u)
                if ((uload >> u) & 1u)
                    drain_bar(ptx::smem_addr(&sh.ufull[u]), ((upar >> u) & 1u) ^ 1u);
        }
        __syncwarp();
    } else if (warp == 1 && count > 0) {
        // ------------------------------------------- operands + MMA
        Cursor ld = cur;   // load cursor, LA tiles ahead of the MMA cursor
        int ld_i = 0, ld_u = 0, ld_v = -1, ld_plz = -1, ld_pc = -1;
        bool stop = false;
        // operand copies of the load cursor's next tile (always one commit group)
        auto issue = [&]() {
            if (ld_i < count && !stop) {
                const int l = ld.lz / p.Z, z = ld.lz - l * p.Z;
                const Seg sg = segment(p, z);
                const KameraChunk& ch = ld.ch;
                const int m = ch.rank, mpad = (m + 15) & ~15;
                const bool new_job = ld.lz != ld_plz || ld.c != ld_pc;
                ld_plz = ld.lz;
                ld_pc = ld.c;
                if (m > 0) {
                    const int64_t lh = (int64_t)l * sg.FH + sg.fh;
                    if (new_job) {
                        ++ld_v;
                        if (!warp_wait(ptx::smem_addr(&sh.vmempty[ld_v & 1]), ((ld_v >> 1) & 1) ^ 1, abort_flag,
                                       r.err, p.wait_ns))
                            stop = true;
                        else
                            load_operand(vbase + (ld_v & 1) * G::kVBytes,
                                         patch_ptr(ch, sg.v_idx) +
                                             (lh * sg.vm_rows + sg.vm_row0) * m,
                                         sg.w, m, mpad, (uint32_t)sg.w * 128u, lane);
                    }
                    const int u = ld_u % G::D;
                    const bool by_tma = u_mapped<MC>(sh.umask, ld.c, m);   // the producer loads this U tile
                    if (!by_tma && !stop &&
                        !warp_wait(ptx::smem_addr(&sh.uempty[u]), ((ld_u / G::D) & 1) ^ 1, abort_flag, r.err, p.wait_ns))
                        stop = true;
                    if (!by_tma && !stop) {
                        const int tok0 = ld.t * kTileM;
                        load_operand(ubase + u * G::kUBytes,
                                     patch_ptr(ch, sg.u_idx) +
                                         (lh * ch.len + tok0) * m,
                                     min(kTileM, ch.len - tok0), m, mpad, kAtomBytes, lane);
                    }
                    ++ld_u;
                }
                ++ld_i;
                ld.next(p);
            }
            ptx::cp_async_commit();
        };
        for (int j = 0; j < G::LA; ++j)
            issue();
        int k = 0, vjob = -1, plz = -1, pc = -1, issued_mma = 0;
        uint32_t upar = 0;   // per U buffer: phase parity of the producer's TMA loads
        for (int i = 0; i < count && !stop; ++i) {
            ptx::cp_async_wait<G::LA - 1>();   // this tile's operand copies have landed ...
            ptx::fence_proxy_async();          // ... and are visible to the tensor cores
            __syncwarp();
            const int l = cur.lz / p.Z, z = cur.lz - l * p.Z;
            const Seg sg = segment(p, z);
            const int m = cur.ch.rank;
            const bool new_job = cur.lz != plz || cur.c != pc;
            plz = cur.lz;
            pc = cur.c;
            const int lz_now = cur.lz, c_now = cur.c;
            cur.next(p);
            const bool last_of_job = (i == count - 1) || cur.lz != lz_now || cur.c != c_now;
            if (m > 0) {
                if (new_job)
                    ++vjob;
                const bool by_tma = u_mapped<MC>(sh.umask, c_now, m);
                if (lane == 0) {
                    const int acc = k & 1, u = k % G::D;
                    bool ok = true;
                    if (by_tma) {
                        ok = wait_bar(ptx::smem_addr(&sh.ufull[u]), (upar >> u) & 1u, abort_flag, r.err, p.wait_ns);
                        upar ^= 1u << u;
                    }
                    if (!ok || !wait_bar(ptx::smem_addr(&sh.tempty[acc]), ((k >> 1) & 1) ^ 1, abort_flag, r.err, p.wait_ns)) {
                        stop = true;
                    } else {
                        ptx::tc_fence_after();
                        const uint32_t a0 = ubase + u * G::kUBytes;
                        const uint32_t b0 = vbase + (vjob & 1) * G::kVBytes;
                        const uint32_t idesc = ptx::idesc_bf16_f32(kTileM, sg.w);
                        const uint32_t d = tmem + acc * kWMax;
                        const int steps = (m + 15) >> 4;
                        for (int q = 0; q < steps; ++q) {
                            const uint32_t koff = (q & 3) * 32;
                            // A as the TMA load laid it out (rows of 2m bytes, m < 64) or in 64-rank atoms
                            const uint64_t ad = by_tma && m == 16   ? ptx::desc_k_sw32(a0)
                                                : by_tma && m == 32 ? ptx::desc_k_sw64(a0 + koff)
                                                                    : ptx::desc_k_sw128(a0 + (q >> 2) * kAtomBytes + koff);
                            const uint64_t bd = ptx::desc_k_sw128(b0 + (q >> 2) * (uint32_t)sg.w * 128u + koff);
                            ptx::umma_bf16(d, ad, bd, idesc, q > 0 ? 1u : 0u);
                        }
                        ptx::umma_commit(ptx::smem_addr(&sh.tfull[acc]));
                        ptx::umma_commit(ptx::smem_addr(&sh.uempty[k % G::D]));
                        if (last_of_job)
                            ptx::umma_commit(ptx::smem_addr(&sh.vmempty[vjob & 1]));
                        ++issued_mma;
                    }
                }
                ++k;
                stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
            }
            issue();
        }
        ptx::cp_async_wait<0>();
        if (lane == 0 && issued_mma) {   // every MMA done before TMEM is freed
            ptx::umma_commit(ptx::smem_addr(&sh.mmadone));
            drain_bar(ptx::smem_addr(&sh.mmadone), 0);
        }
        __syncwarp();
    }
    } else {
    ptx::setmaxnreg_inc<kRegsEpi>();
    if (count > 0) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;         // TMEM sub-partition of this warp
        const int hh = (warp - kEpiWarp0) >> 2;   // which share of the columns this warp owns (0..kEpiPerSub-1)
        const int tt = q * 32 + lane;   // token row of the tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        int k = 0;
        for (int i = 0; i < count; ++i) {
            const int s = i % G::S, rnd = i / G::S;
            if (!warp_wait(ptx::smem_addr(&sh.full[s]), rnd & 1, abort_flag, r.err, p.wait_ns))
                break;
            const TileInfo ti = sh.tinfo[s];   // the producer's description of the tile in this stage
            const int l = ti.l, m = ti.m, ntok = ti.ntok;
            const bool rot = ti.rot != 0;
            const Seg sg = segment(p, ti.z);
            const int acc = k & 1;
            if (m > 0) {
                if (!warp_wait(ptx::smem_addr(&sh.tfull[acc]), (k >> 1) & 1, abort_flag, r.err, p.wait_ns))
                    break;
                ptx::tc_fence_after();
            }
            const uint32_t rows_s = base + s * kStageBytes;
            const uint32_t cs_s = rows_s + kTabOff;
            int64_t slot = ptx::ld_shared_s64(rows_s + kSlotOff + 8 * tt);
            if (slot >= r.num_slots || (tt < ntok && slot < 0)) {
                raise_err(r.err, KAMERA_DEVERR_SLOT);
                slot = -1;
            }
            const bool valid = slot >= 0;
            const uint32_t tacc = tmem + lane_addr + acc * kWMax;
            const int mode = rot ? (r.rope.pairing == KAMERA_ROPE_ROTATE_HALF ? 1 : 2) : 0;
            // The row splits into P = w/16 pair-pieces and this warp owns [j0, j0+R):
            // two spans of 8R columns at a0 and b0, R rounds.  Rotate-half needs each
            // thread to hold RoPE partners, so a pair-piece is 8 columns j*8.. and the 8
            // w/2 further on; otherwise the warp's pieces form one contiguous run of the
            // row, which keeps its pool stores to whole 32-byte sectors.
            const int P = sg.w >> 4;
            const int j0 = hh * P / kEpiPerSub, R = (hh + 1) * P / kEpiPerSub - j0;
            const int a0 = mode == 1 ? 8 * j0 : 16 * j0, b0 = mode == 1 ? (sg.w >> 1) + 8 * j0 : a0 + 8 * R;
            epilogue_dispatch(mode, m > 0, rows_s, tt, a0, b0, R, tacc, cs_s, valid);
            if (m > 0) {   // accumulator free for the next MMA
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(ptx::smem_addr(&sh.tempty[acc]));
                ++k;
            }
            __syncwarp();
            // this warp's columns of its 32 rows -> pool slots, coalesced 16-byte pieces;
            // all slots, then all shared loads, then all global stores
            // 32 rows x ppr pieces; item = instruction * 32 + lane walks them row by
            // row, the pieces of a span being adjacent in the pool row
            {
                const int ppr = 2 * R;
                const uint32_t inv = (65536u + (uint32_t)ppr - 1u) / (uint32_t)ppr;   // item / ppr, exact below 512
                __nv_bfloat16* dbase = (sg.array == 0 ? r.dst_k : r.dst_v) + (int64_t)l * r.dst_ls + sg.e0;
                for (int b4 = 0; b4 < ppr; b4 += 2) {   // batches of 2 instructions (ppr is even)
                    int64_t sl[2];
                    int row[2], piece[2];
                    uint32_t v[2][4];
#pragma unroll
                    for (int it = 0; it < 2; ++it) {
                        const int item = (b4 + it) * 32 + lane;
                        row[it] = (int)(((uint32_t)item * inv) >> 16);
                        const int pi = item - row[it] * ppr;
                        piece[it] = pi < R ? (a0 >> 3) + pi : (b0 >> 3) + (pi - R);
                        sl[it] = __shfl_sync(0xffffffffu, slot, row[it]);
                    }
#pragma unroll
                    for (int it = 0; it < 2; ++it)
                        if (sl[it] >= 0)
                            ptx::lds128(piece_addr(rows_s, q * 32 + row[it], piece[it]), v[it]);
#pragma unroll
                    for (int it = 0; it < 2; ++it)
                        if (sl[it] >= 0)
                            ptx::stg128(dbase + sl[it] * r.dst_ss + piece[it] * 8, v[it]);
                }
            }
            ptx::fence_proxy_async();   // our shared-memory accesses precede the next TMA write here
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(ptx::smem_addr(&sh.empty[s]));
        }
    }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

bool umma_supported(const RowsParams& p, int family)
{
    if (p.max_rank < 1 || p.max_rank > 128 || p.num_rows < 1)
        return false;
    if (family == FAMILY_GQA) {
        if (p.d != 64 && p.d != 128)
            return false;
        return p.rope.rot_dim == 0 || (p.rope.rot_offset == 0 && p.rope.rot_dim == p.d);
    }
    if (family == FAMILY_MLA) {
        const int rope = p.d - p.kv_lora;
        if (p.kv_lora % kWMax != 0 || (rope != 64 && rope != 128))
            return false;
        return p.rope.rot_dim == 0 || (p.rope.rot_offset == 0 && p.rope.rot_dim == rope);
    }
    return false;
}

template <int KA>
static size_t smem_bytes_for()
{
    return 1024 + (size_t)Geometry<KA>::kSharedOff + sizeof(Shared);
}

size_t umma_smem_bytes(const RowsParams& p)
{
    return p.max_rank > 64 ? smem_bytes_for<2>() : smem_bytes_for<1>();
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 3-D map over a strided [L][rows][width] bf16 array: boxes of 64 columns x
// box_rows rows x 1 layer, 128-byte swizzle, out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, int64_t L, int64_t rows, int64_t width, int64_t row_stride,
              int64_t layer_stride, int box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, (cuuint64_t)L};
    const int64_t ls = L > 1 ? layer_stride : rows * row_stride;
    cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2u, (cuuint64_t)ls * 2u};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    // A box row is 128 bytes.  Promoting L2 fills to 256 bytes also brings in its
    // neighbour, which the next box of the row uses when rows start on 256-byte
    // boundaries; with rows 128 bytes off that boundary (the 1152-byte MLA row)
    // every other row's fill would drag in 128 bytes no box of the tile reads
    // (+35% DRAM reads on a DeepSeek-V2-Lite relocation), so fills stay at 128.
    const CUtensorMapL2promotion promo =
        (row_stride * 2) % 256 == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over one chunk's U factor, [L*FH][len][m] bf16 (m-contiguous):
// boxes of min(m, 64) ranks x 128 rows x 1, swizzled like the MMA operand
// (rows of 32, 64 or 128 bytes); rows past len read as zero.
bool make_u_map(CUtensorMap* m, const void* base, int64_t planes, int64_t len, int rank)
{
    auto fn = encode_fn();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || len < 1)
        return false;
    const int inner = rank < 64 ? rank : 64;
    cuuint64_t dims[3] = {(cuuint64_t)rank, (cuuint64_t)len, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)rank * 2u, (cuuint64_t)(len * rank * 2)};
    cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)kTileM, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapSwizzle sw = rank == 16   ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : rank == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_128B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KA, int MC>
cudaError_t launch_kernel(const UmmaParams& core, const KameraChunk* h_chunks, int sms, cudaStream_t stream)
{
    UmmaLaunch<MC> local;
    std::memset(&local, 0, sizeof(local));
    local.core = core;
    const RowsParams& rp = core.r;
    if (h_chunks) {
        const int64_t planes = core.family == FAMILY_GQA ? (int64_t)rp.L * rp.H : rp.L;
        const int n = rp.n_chunks < MC ? rp.n_chunks : MC;
        for (int c = 0; c < n; ++c) {
            const KameraChunk& ch = h_chunks[c];
            const int m = ch.rank;
            if ((m != 16 && m != 32 && m != 64 && m != 128) || m > rp.max_rank || ch.len < 1)
                continue;
            if (make_u_map(&local.map_u[2 * c], ch.patch_ptrs[0], planes, ch.len, m) &&
                make_u_map(&local.map_u[2 * c + 1], ch.patch_ptrs[2], planes, ch.len, m)) {
                local.u_rank[c] = m;
                local.u_len[c] = ch.len;
                local.u_base[c][0] = ch.patch_ptrs[0];
                local.u_base[c][1] = ch.patch_ptrs[2];
            }
        }
    }
    const size_t smem = smem_bytes_for<KA>();
    cudaError_t e = cudaFuncSetAttribute(relocate_patch_umma_kernel<KA, MC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    relocate_patch_umma_kernel<KA, MC><<<sms, kThreads, smem, stream>>>(local);
    return cudaGetLastError();
}

}  // namespace

bool make_rows_map(void* map, const void* base, int64_t rows, int64_t width, int64_t row_stride, int box_cols,
                   int box_rows)
{
    auto fn = encode_fn();
    if (!fn || rows < 1 || width < 1)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_stride * 2u};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_umma(const RowsParams& rp, int family, const KameraChunk* h_chunks, cudaStream_t stream)
{
    UmmaParams p;
    std::memset(&p, 0, sizeof(p));
    p.r = rp;
    p.family = family;
    p.Z = family == FAMILY_GQA ? 2 * rp.H : rp.kv_lora / kWMax + 1;
    p.wait_ns = wait_limit_ns();
    p.withhold = test_withhold_loads() ? 1 : 0;
    const int64_t width = family == FAMILY_GQA ? (int64_t)rp.H * rp.d : rp.d;
    const void* arrays[2] = {rp.src_k, family == FAMILY_GQA ? rp.src_v : rp.src_k};
    for (int a = 0; a < 2; ++a) {
        if (!make_map(&p.map_full[a], arrays[a], rp.L, rp.num_rows, width, rp.src_rs, rp.src_ls, kTileM) ||
            !make_map(&p.map_tail[a], arrays[a], rp.L, rp.num_rows, width, rp.src_rs, rp.src_ls, kTailRows))
            return cudaErrorInvalidValue;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    // a small map table for small calls keeps the launch's parameter block short
    const bool few = rp.n_chunks <= kMapChunksFew;
    if (rp.max_rank > 64)
        return few ? launch_kernel<2, kMapChunksFew>(p, h_chunks, sms, stream)
                   : launch_kernel<2, kMapChunksMany>(p, h_chunks, sms, stream);
    return few ? launch_kernel<1, kMapChunksFew>(p, h_chunks, sms, stream)
               : launch_kernel<1, kMapChunksMany>(p, h_chunks, sms, stream);
}

}  // namespace kamera
