// kamera_slide.cu -- sliding-window survival in place on sm_103a.
//
// Survivors of an eviction move by the RoPE phase shift alone (gist.science
// technical summary, section 3.2): for every chunk c, layer l, head h and
// token j < len,
//     K[l][slot_j][h][rot range] = bf16( R(delta_c) K[l][slot_j][h][rot range] )
// and nothing else of the row changes (no patch, V untouched).
//
// One CTA owns (chunk, 128-token tile, group of layers).  It forms the chunk's
// cos/sin table once (phase in fp64, reduced modulo 2 pi) and stages the
// tile's slots in shared memory.  A token row holds H * units_per_head rotary
// units -- a rotate-half unit is a pair of 16-byte vectors whose elements are
// RoPE partners (x_i..x_{i+7} and x_{i+r/2}..), an interleaved unit one
// vector of four adjacent pairs -- and every thread owns one fixed unit, so its
// cos/sin values sit in registers for the whole CTA while rows stream
// through, four per thread in flight.  Elements outside the rotary range are
// neither read nor written; delta == 0 writes nothing (the row is unchanged).
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"

namespace kamera {

namespace {

constexpr int kSlideThreads = 256;
constexpr int kSlideTile = 128;   // tokens per CTA
constexpr int kSlideUnroll = 4;   // rows per thread in flight

template <bool HALF>
__global__ void __launch_bounds__(kSlideThreads) slide_kernel(const __grid_constant__ RowsParams p, int tiles_per_chunk,
                                                              int layers_per_cta, int units_per_head)
{
    __shared__ float2 cs[KAMERA_MAX_ROT_DIM / 2];
    __shared__ int64_t slots[kSlideTile];
    const int chunk = blockIdx.x / tiles_per_chunk, tile = blockIdx.x - chunk * tiles_per_chunk;
    const KameraChunk ch = p.chunks[chunk];
    const int32_t bad = check_chunk(ch, chunk, p, true);
    if (bad) {
        if (tile == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            raise_err(p.err, bad);
        return;
    }
    const int t0 = tile * kSlideTile;
    if (t0 >= ch.len || !chunk_turns(p.rope, ch, chunk))
        return;
    const int ntok = min(kSlideTile, ch.len - t0);
    for (int f = threadIdx.x; f < p.rope.n_freq; f += kSlideThreads) {
        float c, s;
        phase_cos_sin(freq_delta(p.rope, ch, chunk, f), p.rope.inv_freq[f], c, s);
        cs[f] = make_float2(c, s);
    }
    for (int j = threadIdx.x; j < ntok; j += kSlideThreads) {
        int64_t s = ch.dst_slot_mapping[t0 + j];
        if (s < 0 || s >= p.num_slots) {
            if (blockIdx.y == 0)
                raise_err(p.err, KAMERA_DEVERR_SLOT);
            s = -1;
        }
        slots[j] = s;
    }
    __syncthreads();

    // this thread's unit: head h, unit i of the head, first row r0 of each pass
    const int nu = p.H * units_per_head;   // divides kSlideThreads (checked on the host)
    const int rpp = kSlideThreads / nu;
    const int u = threadIdx.x % nu, r0 = threadIdx.x / nu;
    const int h = u / units_per_head, i = u - h * units_per_head;
    const int ea = h * p.d + p.rope.rot_offset + 8 * i;   // element offsets inside the row
    const int eb = ea + p.rope.rot_dim / 2;
    constexpr int NF = HALF ? 8 : 4;                       // frequencies of the unit
    float c[NF], s[NF];
#pragma unroll
    for (int k = 0; k < NF; ++k) {
        const float2 t = cs[NF * i + k];
        c[k] = t.x;
        s[k] = t.y;
    }

    const int l_end = min(p.L, (int)(blockIdx.y + 1) * layers_per_cta);
    for (int l = blockIdx.y * layers_per_cta; l < l_end; ++l) {
        __nv_bfloat16* base = p.dst_k + (int64_t)l * p.dst_ls;
        for (int jb = r0; jb < ntok; jb += rpp * kSlideUnroll) {
            uint4 va[kSlideUnroll], vb[kSlideUnroll];
            __nv_bfloat16* row[kSlideUnroll];
#pragma unroll
            for (int k = 0; k < kSlideUnroll; ++k) {
                const int j = jb + k * rpp;
                const int64_t sl = j < ntok ? slots[j] : -1;
                row[k] = sl >= 0 ? base + sl * p.dst_ss : nullptr;
                if (row[k]) {
                    va[k] = *reinterpret_cast<const uint4*>(row[k] + ea);
                    if constexpr (HALF)
                        vb[k] = *reinterpret_cast<const uint4*>(row[k] + eb);
                }
            }
#pragma unroll
            for (int k = 0; k < kSlideUnroll; ++k) {
                if (!row[k])
                    continue;
                float a[8], o[8];
                unpack8(va[k], a);
                if constexpr (HALF) {
                    float b[8], ob[8];
                    unpack8(vb[k], b);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        o[e] = fmaf(a[e], c[e], -(b[e] * s[e]));
                        ob[e] = fmaf(b[e], c[e], a[e] * s[e]);
                    }
                    *reinterpret_cast<uint4*>(row[k] + eb) = pack8(ob);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o[2 * e] = fmaf(a[2 * e], c[e], -(a[2 * e + 1] * s[e]));
                        o[2 * e + 1] = fmaf(a[2 * e + 1], c[e], a[2 * e] * s[e]);
                    }
                }
                *reinterpret_cast<uint4*>(row[k] + ea) = pack8(o);
            }
        }
    }
}

int slide_units_per_head(const RowsParams& p)
{
    if (p.rope.pairing == KAMERA_ROPE_ROTATE_HALF)
        return p.rope.rot_dim % 16 == 0 ? p.rope.rot_dim / 16 : 0;
    return p.rope.rot_dim % 8 == 0 ? p.rope.rot_dim / 8 : 0;
}

}  // namespace

bool slide_supported(const RowsParams& p)
{
    const int uph = slide_units_per_head(p);
    if (uph <= 0 || p.rope.rot_offset % 8 != 0 || p.rope.rot_offset + p.rope.rot_dim > p.d)
        return false;
    const int nu = p.H * uph;
    return nu <= kSlideThreads && kSlideThreads % nu == 0;
}

cudaError_t launch_slide(const RowsParams& p, cudaStream_t stream)
{
    const int tiles = (p.max_len + kSlideTile - 1) / kSlideTile;
    const int64_t tile_rows = (int64_t)p.n_chunks * tiles;
    // enough CTAs to fill the GPU several times over, each with a few layers
    int lg = (int)((tile_rows * p.L) / 4096);
    lg = lg < 1 ? 1 : (lg > 8 ? 8 : lg);
    if (lg > p.L)
        lg = p.L;
    const dim3 grid((unsigned)tile_rows, (unsigned)((p.L + lg - 1) / lg));
    const int uph = slide_units_per_head(p);
    if (p.rope.pairing == KAMERA_ROPE_ROTATE_HALF)
        slide_kernel<true><<<grid, kSlideThreads, 0, stream>>>(p, tiles, lg, uph);
    else
        slide_kernel<false><<<grid, kSlideThreads, 0, stream>>>(p, tiles, lg, uph);
    return cudaGetLastError();
}

}  // namespace kamera
