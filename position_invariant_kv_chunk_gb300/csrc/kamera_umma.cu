// kamera_umma.cu -- tensor-core path of the Kamera operator on sm_103a.
//
// Reuse equation (gist.science technical summary, section 2):
//     KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T
// The rank-m patch U_m V_m^T of one (chunk, layer, row segment) over a tile of
// 128 tokens is a 128 x w x m contraction (w = head_dim for GQA/MHA, 128 or
// 64 for the MLA c_KV blocks / k_rope).  It runs on the 5th-generation tensor
// cores: one tcgen05.mma (M=128, N=w, K=16 per instruction, bf16 in, fp32 out)
// per 16 ranks, accumulator in TMEM.  Everything else streams:
//
//   warp 0  producer   canonical rows -> shared memory with bulk async copies
//                      (one per row, completion counted on an mbarrier); the
//                      U tile and V_m (per job) with 16-byte async copies into
//                      the 128-byte-swizzled K-major operand layout; the
//                      per-chunk cos/sin table (fp64-reduced phase).
//   warp 1  MMA        TMEM allocation; one elected lane issues the MMAs and
//                      commits them to mbarriers.
//   warps 2-5 epilogue thread = token row = TMEM lane: tcgen05.ld the patch,
//                      read the canonical row from shared memory, rotate the
//                      RoPE pairs in fp32, add, round once to bf16, write the
//                      row back in place and scatter it to its pool slot with
//                      one bulk async store.
//
// Stages: S shared-memory stages (tile data), 2 V_m buffers (job data), 2
// TMEM accumulators.  The grid is persistent (one CTA per SM); the tiles of a
// call, ordered (layer, segment, chunk, tile), are split into equal
// contiguous ranges, so consecutive tiles of a CTA share V_m.  Every wait is
// bounded in time: on expiry the CTA records KAMERA_DEVERR_TIMEOUT, drains its
// own copies and MMAs, frees TMEM and returns.
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"
#include "kamera_ptx.cuh"

namespace kamera {

namespace {

constexpr int kTileM = 128;                   // tokens per tile = UMMA M = TMEM lanes
constexpr int kWMax = 128;                    // widest segment = UMMA N
constexpr int kRowPitch = kWMax * 2 + 16;     // padded row: conflict-free row-per-thread access
constexpr int kAtomBytes = kTileM * 128;      // one 64-rank K atom of the U tile
constexpr int kThreads = 192;
constexpr int kTableBytes = kWMax / 2 * 8;    // float2 per frequency
constexpr uint32_t kTmemCols = 2 * kWMax;     // two accumulators
constexpr uint64_t kTimeoutNs = 1000000000ull;

struct UmmaParams {
    RowsParams r;
    int32_t family;
    int32_t Z;            // row segments
    int32_t KA;           // 64-rank K atoms per operand tile (1 or 2)
    int32_t S;            // shared-memory stages
    uint32_t stage_bytes;
    uint32_t vm_bytes;    // one V_m buffer
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

__device__ __forceinline__ int chunk_tiles(const KameraChunk& ch, const RowsParams& r)
{
    return check_chunk(ch, r, false) ? 0 : (ch.len + kTileM - 1) / kTileM;
}

// Walks the CTA's tiles in order; every role runs its own copy.
struct Cursor {
    int lz, c, t, ntile;
    KameraChunk ch;

    __device__ void load(const UmmaParams& p)
    {
        ch = p.r.chunks[c];
        ntile = chunk_tiles(ch, p.r);
    }
    __device__ void next(const UmmaParams& p)
    {
        if (++t < ntile)
            return;
        t = 0;
        do {
            if (++c == p.r.n_chunks) {
                c = 0;
                ++lz;
            }
            load(p);
        } while (ntile == 0);
    }
};

struct Shared {
    uint64_t full[4], empty[4], tfull[2], tempty[2], vmempty[2], mmadone;
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t start_lz, start_rem, start_c, start_t, count;
    int32_t stage_tag[4];
    int64_t part[kThreads];
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* err)
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
            if (ptx::globaltimer() - t0 > kTimeoutNs) {
                *abort_flag = 1;
                raise_err(err, KAMERA_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// time-bounded wait that ignores the abort flag (used while draining)
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer() - t0 > kTimeoutNs)
            return;
}

// Copies `rows` rows of an [*, m] bf16 factor (row stride m) into the
// 128B-swizzled K-major operand layout at `dst` (atom stride atom_bytes),
// zero-filling ranks m..mpad-1.  Lanes of one warp share the work.
__device__ __forceinline__ void load_operand(uint32_t dst, const __nv_bfloat16* src, int rows, int m, int mpad,
                                             uint32_t atom_bytes, int lane)
{
    if ((m & 7) == 0) {
        const int pr = m >> 3;               // 16-byte pieces per row
        for (int p = lane; p < rows * pr; p += 32) {
            const int r = p / pr, kc = p - r * pr;
            const uint32_t d = dst + (kc >> 3) * atom_bytes + r * 128 + ((((kc & 7) ^ (r & 7))) << 4);
            ptx::cp_async16(d, src + (size_t)r * m + kc * 8);
        }
        const int pp = (mpad - m) >> 3;
        for (int p = lane; p < rows * pp; p += 32) {
            const int r = p / pp, kc = (m >> 3) + (p - r * pp);
            ptx::st_shared_zero16(dst + (kc >> 3) * atom_bytes + r * 128 + ((((kc & 7) ^ (r & 7))) << 4));
        }
    } else {
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
        for (int p = lane; p < rows * mpad; p += 32) {
            const int r = p / mpad, k = p - r * mpad;
            const uint16_t v = k < m ? s16[(size_t)r * m + k] : (uint16_t)0;
            const int kc = k >> 3;
            ptx::st_shared_u16(dst + (kc >> 3) * atom_bytes + r * 128 + ((((kc & 7) ^ (r & 7))) << 4) + (k & 7) * 2, v);
        }
    }
}

__device__ __forceinline__ float f_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float f_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void lds128(uint32_t a, uint32_t (&v)[4])
{
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(a));
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// 16 consecutive bf16 of a shared row -> fp32
__device__ __forceinline__ void load16(uint32_t a, float* f)
{
    uint32_t v[4], u[4];
    lds128(a, v);
    lds128(a + 16, u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = f_lo(v[i]);
        f[2 * i + 1] = f_hi(v[i]);
        f[8 + 2 * i] = f_lo(u[i]);
        f[8 + 2 * i + 1] = f_hi(u[i]);
    }
}

__device__ __forceinline__ void store16(uint32_t a, const float* f)
{
    sts128(a, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    sts128(a + 16, pack_bf16x2(f[8], f[9]), pack_bf16x2(f[10], f[11]), pack_bf16x2(f[12], f[13]),
           pack_bf16x2(f[14], f[15]));
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) relocate_patch_umma_kernel(const __grid_constant__ UmmaParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled operand tiles
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t vm_base = base + p.S * p.stage_bytes;
    Shared& sh = *reinterpret_cast<Shared*>(gbase + p.S * p.stage_bytes + 2 * p.vm_bytes);
    volatile int32_t* abort_flag = &sh.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const RowsParams& r = p.r;

    // ---------------------------------------------------------- prologue
    if (tid == 0) {
        for (int i = 0; i < p.S; ++i) {
            ptx::mbar_init(ptx::smem_addr(&sh.full[i]), 2);
            ptx::mbar_init(ptx::smem_addr(&sh.empty[i]), 4);
            sh.stage_tag[i] = -1;
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_addr(&sh.tfull[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.tempty[i]), 4);
            ptx::mbar_init(ptx::smem_addr(&sh.vmempty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sh.mmadone), 1);
        sh.abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async();
    }
    // tiles per chunk: each thread sums a contiguous block of chunks
    const int n = r.n_chunks;
    const int per = (n + kThreads - 1) / kThreads;
    const int c_lo = min(n, tid * per), c_hi = min(n, c_lo + per);
    int64_t mine = 0;
#pragma unroll 4
    for (int c = c_lo; c < c_hi; ++c) {
        const KameraChunk ch = r.chunks[c];
        const int32_t bad = check_chunk(ch, r, false);
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
        sh.start_lz = TC ? (int32_t)(b0 / TC) : 0;
        sh.start_rem = (int32_t)(TC ? b0 % TC : 0);   // tile offset inside the (layer, segment) block
        sh.start_c = 0;
        sh.start_t = 0;
    }
    __syncthreads();
    if (sh.count > 0) {
        const int64_t rem = sh.start_rem;
        const int64_t lo = sh.part[tid];
        if (rem >= lo && rem < lo + mine) {   // exactly one thread owns the starting tile
            int64_t acc = lo;
            for (int c = c_lo; c < c_hi; ++c) {
                const KameraChunk ch = r.chunks[c];
                const int nt = chunk_tiles(ch, r);
                if (rem < acc + nt) {
                    sh.start_t = (int32_t)(rem - acc);
                    sh.start_c = c;
                    break;
                }
                acc += nt;
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

    const int KA = p.KA;
    if (warp == 0 && count > 0) {
        // ------------------------------------------------------ producer
        int pending = -1, issued = 0, vjobs = -1;
        int prev_lz = -1, prev_c = -1;
        for (int i = 0; i < count; ++i, cur.next(p)) {
            const int s = i % p.S, rnd = i / p.S;
            if (!wait_bar(ptx::smem_addr(&sh.empty[s]), (rnd & 1) ^ 1, abort_flag, r.err))
                break;
            const int l = cur.lz / p.Z, z = cur.lz - l * p.Z;
            const Seg sg = segment(p, z);
            const KameraChunk& ch = cur.ch;
            const int tok0 = cur.t * kTileM;
            const int ntok = min(kTileM, ch.len - tok0);
            const int m = ch.rank, mpad = (m + 15) & ~15;
            const uint32_t st = base + s * p.stage_bytes;
            const bool new_job = cur.lz != prev_lz || cur.c != prev_c;
            prev_lz = cur.lz;
            prev_c = cur.c;
            if (m > 0) {
                const int64_t lh = (int64_t)l * sg.FH + sg.fh;
                if (new_job) {
                    ++vjobs;
                    const int b = vjobs & 1;
                    if (!wait_bar(ptx::smem_addr(&sh.vmempty[b]), ((vjobs >> 1) & 1) ^ 1, abort_flag, r.err))
                        break;
                    const __nv_bfloat16* V = static_cast<const __nv_bfloat16*>(ch.patch_ptrs[sg.v_idx]);
                    load_operand(vm_base + b * p.vm_bytes, V + (lh * sg.vm_rows + sg.vm_row0) * m, sg.w, m, mpad,
                                 (uint32_t)sg.w * 128u, lane);
                }
                const __nv_bfloat16* U = static_cast<const __nv_bfloat16*>(ch.patch_ptrs[sg.u_idx]);
                load_operand(st, U + (lh * ch.len + tok0) * m, ntok, m, mpad, kAtomBytes, lane);
            }
            ptx::cp_async_commit();
            const bool rot = sg.rot && ch.delta != 0;
            if (rot && sh.stage_tag[s] != cur.c) {
                float2* cs = reinterpret_cast<float2*>(gbase + s * p.stage_bytes + KA * kAtomBytes + kTileM * kRowPitch);
                for (int f = lane; f < r.rope.n_freq; f += 32) {
                    float c_, s_;
                    phase_cos_sin(ch.delta, r.rope.inv_freq[f], c_, s_);
                    cs[f] = make_float2(c_, s_);
                }
                __syncwarp();
                if (lane == 0)
                    sh.stage_tag[s] = cur.c;
            }
            __syncwarp();
            const uint32_t full = ptx::smem_addr(&sh.full[s]);
            const uint32_t row_bytes = (uint32_t)sg.w * 2u;
            if (lane == 0)
                ptx::mbar_arrive_expect_tx(full, row_bytes * (uint32_t)ntok);
            __syncwarp();
            const __nv_bfloat16* src = (sg.array == 0 ? r.src_k : r.src_v) + (int64_t)l * r.src_ls +
                                       (ch.src_offset + tok0) * r.src_rs + sg.e0;
            const uint32_t rows_s = st + KA * kAtomBytes;
            for (int tt = lane; tt < ntok; tt += 32)
                ptx::bulk_g2s(rows_s + tt * kRowPitch, src + (int64_t)tt * r.src_rs, row_bytes, full);
            ++issued;
            if (pending >= 0) {   // operand copies of the previous tile are complete: publish them
                ptx::cp_async_wait<1>();
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(ptx::smem_addr(&sh.full[pending]));
            }
            pending = s;
        }
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async();
        __syncwarp();
        if (pending >= 0 && lane == 0)
            ptx::mbar_arrive(ptx::smem_addr(&sh.full[pending]));
        // no bulk load may still be writing shared memory when the CTA exits
        for (int j = max(0, issued - p.S); j < issued; ++j)
            drain_bar(ptx::smem_addr(&sh.full[j % p.S]), (j / p.S) & 1);
    } else if (warp == 1 && count > 0) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            int k = 0, vjobs = -1, issued_mma = 0;
            int prev_lz = -1, prev_c = -1;
            for (int i = 0; i < count; ++i) {
                const int s = i % p.S, rnd = i / p.S;
                const int l = cur.lz / p.Z, z = cur.lz - l * p.Z;
                const Seg sg = segment(p, z);
                const int m = cur.ch.rank;
                const bool new_job = cur.lz != prev_lz || cur.c != prev_c;
                prev_lz = cur.lz;
                prev_c = cur.c;
                const int lz_now = cur.lz, c_now = cur.c;
                cur.next(p);
                const bool last_of_job = (i == count - 1) || cur.lz != lz_now || cur.c != c_now;
                (void)l;
                if (m == 0)
                    continue;
                if (new_job)
                    ++vjobs;
                const int acc = k & 1;
                if (!wait_bar(ptx::smem_addr(&sh.tempty[acc]), ((k >> 1) & 1) ^ 1, abort_flag, r.err))
                    break;
                if (!wait_bar(ptx::smem_addr(&sh.full[s]), rnd & 1, abort_flag, r.err))
                    break;
                ptx::tc_fence_after();
                const uint32_t a0 = base + s * p.stage_bytes;
                const uint32_t b0 = vm_base + (vjobs & 1) * p.vm_bytes;
                const uint32_t idesc = ptx::idesc_bf16_f32(kTileM, sg.w);
                const uint32_t d = tmem + acc * kWMax;
                const int steps = (m + 15) >> 4;
                for (int q = 0; q < steps; ++q) {
                    const uint32_t koff = (q & 3) * 32;
                    const uint64_t ad = ptx::desc_k_sw128(a0 + (q >> 2) * kAtomBytes + koff);
                    const uint64_t bd = ptx::desc_k_sw128(b0 + (q >> 2) * (uint32_t)sg.w * 128u + koff);
                    ptx::umma_bf16(d, ad, bd, idesc, q > 0 ? 1u : 0u);
                }
                ptx::umma_commit(ptx::smem_addr(&sh.tfull[acc]));
                if (last_of_job)
                    ptx::umma_commit(ptx::smem_addr(&sh.vmempty[vjobs & 1]));
                ++k;
                ++issued_mma;
            }
            if (issued_mma) {   // every MMA done before TMEM is freed
                ptx::umma_commit(ptx::smem_addr(&sh.mmadone));
                drain_bar(ptx::smem_addr(&sh.mmadone), 0);
            }
        }
        __syncwarp();
    } else if (warp >= 2 && count > 0) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM sub-partition of this warp
        const int tt = q * 32 + lane;           // token row of the tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        int k = 0;
        for (int i = 0; i < count; ++i, cur.next(p)) {
            const int s = i % p.S, rnd = i / p.S;
            if (!wait_bar(ptx::smem_addr(&sh.full[s]), rnd & 1, abort_flag, r.err))
                break;
            const int l = cur.lz / p.Z, z = cur.lz - l * p.Z;
            const Seg sg = segment(p, z);
            const KameraChunk& ch = cur.ch;
            const int tok0 = cur.t * kTileM;
            const int ntok = min(kTileM, ch.len - tok0);
            const int m = ch.rank;
            const bool rot = sg.rot && ch.delta != 0;
            const int acc = k & 1;
            if (m > 0) {
                if (!wait_bar(ptx::smem_addr(&sh.tfull[acc]), (k >> 1) & 1, abort_flag, r.err))
                    break;
                ptx::tc_fence_after();
            }
            bool valid = tt < ntok;
            int64_t slot = 0;
            if (valid) {
                slot = ch.dst_slot_mapping[tok0 + tt];
                if (slot < 0 || slot >= r.num_slots) {
                    raise_err(r.err, KAMERA_DEVERR_SLOT);
                    valid = false;
                }
            }
            const uint32_t row = base + s * p.stage_bytes + KA * kAtomBytes + tt * kRowPitch;
            const float2* cs =
                reinterpret_cast<const float2*>(gbase + s * p.stage_bytes + KA * kAtomBytes + kTileM * kRowPitch);
            const uint32_t tacc = tmem + lane_addr + acc * kWMax;
            if (m > 0 || rot) {
                if (rot && r.rope.pairing == KAMERA_ROPE_ROTATE_HALF) {
                    const int half = sg.w >> 1;
                    for (int cb = 0; cb < half; cb += 16) {
                        uint32_t pa[16], pb[16];
                        if (m > 0)
                            ptx::tmem_ld16x2(tacc + cb, tacc + cb + half, pa, pb);
                        if (valid) {
                            float xa[16], xb[16];
                            load16(row + cb * 2, xa);
                            load16(row + (cb + half) * 2, xb);
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 t = cs[cb + e];
                                float oa = fmaf(xa[e], t.x, -(xb[e] * t.y));
                                float ob = fmaf(xb[e], t.x, xa[e] * t.y);
                                if (m > 0) {
                                    oa += __uint_as_float(pa[e]);
                                    ob += __uint_as_float(pb[e]);
                                }
                                xa[e] = oa;
                                xb[e] = ob;
                            }
                            store16(row + cb * 2, xa);
                            store16(row + (cb + half) * 2, xb);
                        }
                    }
                } else {
                    for (int cb = 0; cb < sg.w; cb += 32) {
                        uint32_t pa[16], pb[16];
                        if (m > 0)
                            ptx::tmem_ld16x2(tacc + cb, tacc + cb + 16, pa, pb);
                        if (valid) {
                            float xa[16], xb[16];
                            load16(row + cb * 2, xa);
                            load16(row + (cb + 16) * 2, xb);
                            if (rot) {   // interleaved pairs (2i, 2i+1), frequency cb/2 + i
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float2 t = cs[cb / 2 + e];
                                    const float a = xa[2 * e], b = xa[2 * e + 1];
                                    xa[2 * e] = fmaf(a, t.x, -(b * t.y));
                                    xa[2 * e + 1] = fmaf(b, t.x, a * t.y);
                                    const float2 u = cs[cb / 2 + 8 + e];
                                    const float c2 = xb[2 * e], d2 = xb[2 * e + 1];
                                    xb[2 * e] = fmaf(c2, u.x, -(d2 * u.y));
                                    xb[2 * e + 1] = fmaf(d2, u.x, c2 * u.y);
                                }
                            }
                            if (m > 0) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    xa[e] += __uint_as_float(pa[e]);
                                    xb[e] += __uint_as_float(pb[e]);
                                }
                            }
                            store16(row + cb * 2, xa);
                            store16(row + (cb + 16) * 2, xb);
                        }
                    }
                }
            }
            if (m > 0) {   // accumulator free for the next MMA
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(ptx::smem_addr(&sh.tempty[acc]));
                ++k;
            }
            if (valid) {
                ptx::fence_proxy_async();
                __nv_bfloat16* dst = (sg.array == 0 ? r.dst_k : r.dst_v) + (int64_t)l * r.dst_ls + slot * r.dst_ss + sg.e0;
                ptx::bulk_s2g(dst, row, (uint32_t)sg.w * 2u);
                ptx::bulk_commit();
            }
            ptx::bulk_wait_read_all();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(ptx::smem_addr(&sh.empty[s]));
        }
        ptx::bulk_wait_all();
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
    if (p.max_rank < 1 || p.max_rank > 128)
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

size_t umma_smem_bytes(const RowsParams& p)
{
    const int KA = (p.max_rank + 63) / 64;
    const int S = KA == 1 ? 3 : 2;
    const uint32_t stage = ((uint32_t)(KA * kAtomBytes + kTileM * kRowPitch + kTableBytes) + 1023u) & ~1023u;
    const uint32_t vm = (uint32_t)KA * kWMax * 128u;
    return 1024 + (size_t)S * stage + 2 * (size_t)vm + sizeof(Shared);
}

cudaError_t launch_umma(const RowsParams& rp, int family, cudaStream_t stream)
{
    UmmaParams p;
    p.r = rp;
    p.family = family;
    p.Z = family == FAMILY_GQA ? 2 * rp.H : rp.kv_lora / kWMax + 1;
    p.KA = (rp.max_rank + 63) / 64;
    p.S = p.KA == 1 ? 3 : 2;
    p.stage_bytes = ((uint32_t)(p.KA * kAtomBytes + kTileM * kRowPitch + kTableBytes) + 1023u) & ~1023u;
    p.vm_bytes = (uint32_t)p.KA * kWMax * 128u;
    const size_t smem = umma_smem_bytes(rp);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(relocate_patch_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    relocate_patch_umma_kernel<<<sms, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kamera
