// kamera_simt.cu -- CUDA-core (SIMT) path of the Kamera operator on sm_103a.
//
// Reuse equation (gist.science technical summary, section 2):
//     KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T
// One CTA owns (chunk, token tile, layer, row segment).  A row segment is one
// GQA head of K or of V, one 128-wide block of MLA c_KV, the MLA k_rope block,
// or one head of the in-place slide (section 3.2).  Threads stream 16-byte
// vectors: a rotary "pair unit" is two vectors whose elements are RoPE
// partners (rotate-half: x_i and x_{i+r/2}; interleaved: adjacent elements of
// one vector), a plain unit is one vector.  The patch sum_k U[t,k] V_m[e,k] is
// formed with fp32 FMAs from tiles staged in shared memory.  Every output
// element is rounded once to bf16 (RNE).  Pure copies (delta = 0 or no
// rotation, and rank 0) move raw bits.
//
// This path serves the rotation-only cases (slide, rank-0 relocation) at
// streaming bandwidth and is the general fallback for ranks and shapes the
// tensor-core path does not take.
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"

namespace kamera {

namespace {

struct Segment {
    int32_t array;      // 0 = K (or the MLA row), 1 = V
    int32_t e0;         // first element of the segment inside the row
    int32_t w;          // elements in the segment
    int32_t rot_off;    // rotary range inside the segment (relative); rot_dim 0 = none
    int32_t rot_dim;
    int32_t u_idx;      // patch_ptrs index of U and of V_m
    int32_t v_idx;
    int32_t fh;         // factor head index and head count ([L][FH][...])
    int32_t FH;
    int32_t vm_row0;    // first V_m row of this segment
    int32_t vm_rows;    // V_m rows per (layer, head)
};

__device__ __forceinline__ Segment decode_segment(const RowsParams& p, int family, int z)
{
    Segment s;
    if (family == FAMILY_GQA) {
        const int kv = z & 1, h = z >> 1;
        s.array = kv;
        s.e0 = h * p.d;
        s.w = p.d;
        s.rot_off = p.rope.rot_offset;
        s.rot_dim = kv == 0 ? p.rope.rot_dim : 0;
        s.u_idx = 2 * kv;
        s.v_idx = 2 * kv + 1;
        s.fh = h;
        s.FH = p.H;
        s.vm_row0 = 0;
        s.vm_rows = p.d;
    } else if (family == FAMILY_MLA) {
        const int nb = (p.kv_lora + 127) / 128;
        s.array = 0;
        s.fh = 0;
        s.FH = 1;
        if (z < nb) {
            s.e0 = 128 * z;
            s.w = min(128, p.kv_lora - 128 * z);
            s.rot_off = 0;
            s.rot_dim = 0;
            s.u_idx = 0;
            s.v_idx = 1;
            s.vm_row0 = 128 * z;
            s.vm_rows = p.kv_lora;
        } else {
            s.e0 = p.kv_lora;
            s.w = p.d - p.kv_lora;
            s.rot_off = p.rope.rot_offset;
            s.rot_dim = p.rope.rot_dim;
            s.u_idx = 2;
            s.v_idx = 3;
            s.vm_row0 = 0;
            s.vm_rows = p.d - p.kv_lora;
        }
    } else {  // FAMILY_SLIDE
        s.array = 0;
        s.e0 = z * p.d;
        s.w = p.d;
        s.rot_off = p.rope.rot_offset;
        s.rot_dim = p.rope.rot_dim;
        s.u_idx = s.v_idx = 0;
        s.fh = 0;
        s.FH = 1;
        s.vm_row0 = 0;
        s.vm_rows = 0;
    }
    return s;
}

// Adds the patch to 8 consecutive segment elements starting at e (relative).
__device__ __forceinline__ void add_patch8(float* f, const float* __restrict__ us,
                                           const float* __restrict__ vs, int w, int m, int e)
{
#pragma unroll 4
    for (int k = 0; k < m; ++k) {
        const float u = us[k];
        const float4 a = *reinterpret_cast<const float4*>(vs + k * w + e);
        const float4 b = *reinterpret_cast<const float4*>(vs + k * w + e + 4);
        f[0] = fmaf(u, a.x, f[0]);
        f[1] = fmaf(u, a.y, f[1]);
        f[2] = fmaf(u, a.z, f[2]);
        f[3] = fmaf(u, a.w, f[3]);
        f[4] = fmaf(u, b.x, f[4]);
        f[5] = fmaf(u, b.y, f[5]);
        f[6] = fmaf(u, b.z, f[6]);
        f[7] = fmaf(u, b.w, f[7]);
    }
}

}  // namespace

// grid: x = chunk * tiles_per_chunk + tile, y = layer, z = segment
template <int kFamily>
__global__ void __launch_bounds__(256) rows_simt_kernel(const __grid_constant__ RowsParams p, int tile_tokens)
{
    extern __shared__ __align__(16) float smem[];
    const int chunk = blockIdx.x / p.tiles_per_chunk;
    const int tile = blockIdx.x % p.tiles_per_chunk;
    const int l = blockIdx.y;
    const KameraChunk ch = p.chunks[chunk];
    const bool in_place = kFamily == FAMILY_SLIDE;

    const int32_t bad = check_chunk(ch, chunk, p, in_place);
    if (bad) {
        if (tile == 0 && l == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            raise_err(p.err, bad);
        return;
    }
    const int t0 = tile * tile_tokens;
    if (t0 >= ch.len)
        return;
    const int ntok = min(tile_tokens, ch.len - t0);
    const Segment sg = decode_segment(p, kFamily, blockIdx.z);
    const int m = ch.rank;
    const bool rotate = sg.rot_dim > 0 && chunk_turns(p.rope, ch, chunk);
    const int half = sg.rot_dim / 2;

    // shared memory: cos/sin table, V_m^T (fp32 [m][w]), U tile (fp32 [ntok][m])
    float2* cs = reinterpret_cast<float2*>(smem);
    float* vs = smem + 2 * ((KAMERA_MAX_ROT_DIM / 2 + 1) & ~1);
    float* us = vs + (size_t)p.max_rank * sg.w;

    if (rotate)
        for (int i = threadIdx.x; i < half; i += blockDim.x) {
            float c, s;
            phase_cos_sin(freq_delta(p.rope, ch, chunk, i), p.rope.inv_freq[i], c, s);
            cs[i] = make_float2(c, s);
        }
    if (m > 0) {
        const __nv_bfloat16* U = patch_ptr(ch, sg.u_idx);
        const __nv_bfloat16* V = patch_ptr(ch, sg.v_idx);
        const int64_t lh = (int64_t)l * sg.FH + sg.fh;
        const __nv_bfloat16* vrow = V + (lh * sg.vm_rows + sg.vm_row0) * m;
        for (int i = threadIdx.x; i < sg.w * m; i += blockDim.x) {
            const int e = i / m, k = i - e * m;
            vs[k * sg.w + e] = __bfloat162float(vrow[i]);
        }
        const __nv_bfloat16* urow = U + (lh * ch.len + t0) * m;
        for (int i = threadIdx.x; i < ntok * m; i += blockDim.x)
            us[i] = __bfloat162float(urow[i]);
    }
    __syncthreads();

    // units of this segment: rotary units first, then plain 8-element blocks
    const int n_rot = rotate ? (p.rope.pairing == KAMERA_ROPE_ROTATE_HALF ? sg.rot_dim / 16 : sg.rot_dim / 8) : 0;
    const int n_plain = rotate ? (sg.w - sg.rot_dim) / 8 : sg.w / 8;
    const int nunits = n_rot + n_plain;
    const int rb0 = sg.rot_off / 8, rb1 = (sg.rot_off + sg.rot_dim) / 8;

    __nv_bfloat16* dst_base = sg.array == 0 ? p.dst_k : p.dst_v;
    const __nv_bfloat16* src_base = in_place ? dst_base : (sg.array == 0 ? p.src_k : p.src_v);
    const int64_t* slots = ch.dst_slot_mapping;

    for (int it = threadIdx.x; it < ntok * nunits; it += blockDim.x) {
        const int jj = it / nunits;
        const int u = it - jj * nunits;
        const int j = t0 + jj;
        const int64_t slot = slots[j];
        if (slot < 0 || slot >= p.num_slots) {
            raise_err(p.err, KAMERA_DEVERR_SLOT);
            continue;
        }
        __nv_bfloat16* drow = dst_base + (int64_t)l * p.dst_ls + slot * p.dst_ss + sg.e0;
        const __nv_bfloat16* srow = in_place ? drow : src_base + (int64_t)l * p.src_ls + (ch.src_offset + j) * p.src_rs + sg.e0;
        const float* urow = us + jj * m;

        if (u < n_rot) {
            if (p.rope.pairing == KAMERA_ROPE_ROTATE_HALF) {
                const int ea = sg.rot_off + 8 * u, eb = ea + half;
                const uint4 va = *reinterpret_cast<const uint4*>(srow + ea);
                const uint4 vb = *reinterpret_cast<const uint4*>(srow + eb);
                float a[8], b[8], oa[8], ob[8];
                unpack8(va, a);
                unpack8(vb, b);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 t = cs[8 * u + i];
                    oa[i] = fmaf(a[i], t.x, -(b[i] * t.y));
                    ob[i] = fmaf(b[i], t.x, a[i] * t.y);
                }
                if (m > 0) {
                    add_patch8(oa, urow, vs, sg.w, m, ea);
                    add_patch8(ob, urow, vs, sg.w, m, eb);
                }
                *reinterpret_cast<uint4*>(drow + ea) = pack8(oa);
                *reinterpret_cast<uint4*>(drow + eb) = pack8(ob);
            } else {
                const int ea = sg.rot_off + 8 * u;
                const uint4 va = *reinterpret_cast<const uint4*>(srow + ea);
                float a[8], o[8];
                unpack8(va, a);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 t = cs[4 * u + i];
                    o[2 * i] = fmaf(a[2 * i], t.x, -(a[2 * i + 1] * t.y));
                    o[2 * i + 1] = fmaf(a[2 * i + 1], t.x, a[2 * i] * t.y);
                }
                if (m > 0)
                    add_patch8(o, urow, vs, sg.w, m, ea);
                *reinterpret_cast<uint4*>(drow + ea) = pack8(o);
            }
        } else {
            int blk = u - n_rot;
            if (rotate && blk >= rb0)
                blk += rb1 - rb0;
            const int e = 8 * blk;
            const uint4 v = *reinterpret_cast<const uint4*>(srow + e);
            if (m == 0) {
                if (!in_place)
                    *reinterpret_cast<uint4*>(drow + e) = v;
            } else {
                float f[8];
                unpack8(v, f);
                add_patch8(f, urow, vs, sg.w, m, e);
                *reinterpret_cast<uint4*>(drow + e) = pack8(f);
            }
        }
    }
}

size_t simt_smem_bytes(const RowsParams& p, int family, int tile_tokens)
{
    int wmax = p.d;
    if (family == FAMILY_MLA)
        wmax = p.kv_lora < 128 ? p.kv_lora : 128;
    if (family == FAMILY_MLA && p.d - p.kv_lora > wmax)
        wmax = p.d - p.kv_lora;
    const size_t table = sizeof(float) * 2 * ((KAMERA_MAX_ROT_DIM / 2 + 1) & ~1);
    if (family == FAMILY_SLIDE)
        return table;
    return table + sizeof(float) * (size_t)p.max_rank * (wmax + tile_tokens);
}

int simt_segments(const RowsParams& p, int family)
{
    if (family == FAMILY_GQA)
        return 2 * p.H;
    if (family == FAMILY_MLA)
        return (p.kv_lora + 127) / 128 + 1;
    return p.H;
}

// Threads per CTA.  A CTA's time is a chain of dependent loads (descriptor,
// factors, slots, rows), so when the grid is many waves deep the CTAs resident
// at once set the rate: 64-thread CTAs let 32 share an SM where 256-thread CTAs
// let 8 (4096 one-tile chunks: 244 us with 256 threads, 203 with 128, 187 with
// 64).  A grid that fits one wave of 256-thread CTAs keeps them, so each CTA's
// items are spread over the most threads (one tiny chunk: 10 us with 256
// threads, 17 with 64).
static int simt_threads(int64_t blocks)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1)
        return 256;
    return blocks <= 8ll * sms ? 256 : blocks <= 16ll * sms ? 128 : 64;
}

cudaError_t launch_simt(const RowsParams& p, int family, cudaStream_t stream)
{
    const int tile_tokens = 64;
    RowsParams q = p;
    q.tiles_per_chunk = (p.max_len + tile_tokens - 1) / tile_tokens;
    const size_t smem = simt_smem_bytes(q, family, tile_tokens);
    const dim3 grid((unsigned)((int64_t)p.n_chunks * q.tiles_per_chunk), (unsigned)p.L,
                    (unsigned)simt_segments(q, family));
    const int threads = simt_threads((int64_t)grid.x * grid.y * grid.z);
    cudaError_t e = cudaSuccess;
    switch (family) {
    case FAMILY_GQA:
        e = cudaFuncSetAttribute(rows_simt_kernel<FAMILY_GQA>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            rows_simt_kernel<FAMILY_GQA><<<grid, threads, smem, stream>>>(q, tile_tokens);
        break;
    case FAMILY_MLA:
        e = cudaFuncSetAttribute(rows_simt_kernel<FAMILY_MLA>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            rows_simt_kernel<FAMILY_MLA><<<grid, threads, smem, stream>>>(q, tile_tokens);
        break;
    default:
        e = cudaFuncSetAttribute(rows_simt_kernel<FAMILY_SLIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            rows_simt_kernel<FAMILY_SLIDE><<<grid, threads, smem, stream>>>(q, tile_tokens);
        break;
    }
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace kamera
