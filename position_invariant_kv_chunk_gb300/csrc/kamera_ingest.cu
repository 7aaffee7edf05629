// kamera_ingest.cu -- canonical ingest on sm_103a: the inverse of relocation.
//
// A chunk that lives in the paged KV cache at positions s..s+len-1 is read
// back from its slots and turned into the position-free canonical frame of
// the store (gist.science technical summary, section 2, "Canonical KV": the
// chunk as if it started at position 0):
//     Kstore[l][row_c + j][h] = bf16( R(delta_c) K[l][slot_j][h] ),  delta_c = -s_c
//     Vstore[l][row_c + j][h] = V[l][slot_j][h]                       (bit copy)
// MLA rows: c_KV copied, k_rope turned.  Elements outside the rotary range
// are copied; delta == 0 copies the whole row bit for bit.
//
// One CTA owns (chunk, 128-token tile, group of layers): it stages the
// tile's slots and the chunk's cos/sin table (phase in fp64) in shared
// memory, then streams the rows through a short list of passes built on the
// host, each a set of 16-byte units repeated per head: a rotate-half pair
// of vectors whose elements are RoPE partners, an interleaved vector (four
// adjacent pairs), or a plain vector copy.  Each pass is its own launch of
// the kernel specialised for its kind, so every launch stays lean enough to
// keep four rows per thread in flight.  When a pass's units per row divide
// the block, every thread owns one fixed unit (its cos/sin values in
// registers) and walks the rows four at a time; otherwise the threads stride
// over (row, unit) items.
#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_internal.h"

namespace kamera {

namespace {

constexpr int kIngestThreads = 256;
constexpr int kIngestTile = 128;   // tokens per CTA
constexpr int kIngestUnroll = 4;   // rows per thread in flight (fixed mapping)

// A unit's vectors of one row: loaded, then turned (or not) and stored.
template <int KIND>
__device__ __forceinline__ void unit_load(const __nv_bfloat16* src, int e, int half, uint4& va, uint4& vb)
{
    va = *reinterpret_cast<const uint4*>(src + e);
    if constexpr (KIND == INGEST_ROT_HALF)
        vb = *reinterpret_cast<const uint4*>(src + e + half);
}

template <int KIND>
__device__ __forceinline__ void unit_store(__nv_bfloat16* dst, int e, int half, const uint4& va, const uint4& vb,
                                           const float (&c)[8], const float (&s)[8], bool turn)
{
    if (KIND == INGEST_COPY || !turn) {   // delta 0: the unit's vectors are copied bit for bit
        *reinterpret_cast<uint4*>(dst + e) = va;
        if constexpr (KIND == INGEST_ROT_HALF)
            *reinterpret_cast<uint4*>(dst + e + half) = vb;
    } else if constexpr (KIND == INGEST_ROT_HALF) {
        float a[8], b[8], oa[8], ob[8];
        unpack8(va, a);
        unpack8(vb, b);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            oa[k] = fmaf(a[k], c[k], -(b[k] * s[k]));
            ob[k] = fmaf(b[k], c[k], a[k] * s[k]);
        }
        *reinterpret_cast<uint4*>(dst + e) = pack8(oa);
        *reinterpret_cast<uint4*>(dst + e + half) = pack8(ob);
    } else {   // interleaved: (x_2k, x_2k+1) pairs inside the vector, frequencies in c[0..3]
        float a[8], o[8];
        unpack8(va, a);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            o[2 * k] = fmaf(a[2 * k], c[k], -(a[2 * k + 1] * s[k]));
            o[2 * k + 1] = fmaf(a[2 * k + 1], c[k], a[2 * k] * s[k]);
        }
        *reinterpret_cast<uint4*>(dst + e) = pack8(o);
    }
}

template <int KIND>
__device__ __forceinline__ void ingest_pass(const IngestParams& p, const IngestPass& ps, const float2* cs,
                                            const int64_t* slots, int l, int64_t row0, int ntok, bool turn)
{
    const int nu = p.H * ps.per_head;
    const __nv_bfloat16* src = p.src[ps.array] + (int64_t)l * p.src_ls;
    __nv_bfloat16* dst = p.dst[ps.array] + (int64_t)l * p.dst_ls + row0 * p.dst_rs;
    constexpr int NF = KIND == INGEST_ROT_HALF ? 8 : 4;
    auto unit_setup = [&](int u, int& e, float (&c)[8], float (&s)[8]) {
        const int h = u / ps.per_head, i = u - h * ps.per_head;
        e = h * p.d + ps.off + 8 * i;
        if (KIND != INGEST_COPY && turn) {
#pragma unroll
            for (int k = 0; k < NF; ++k) {
                const float2 t = cs[ps.f_off + NF * i + k];
                c[k] = t.x;
                s[k] = t.y;
            }
        }
    };
    float c[8], s[8];
    if (kIngestThreads % nu == 0) {   // a fixed unit per thread
        const int rpp = kIngestThreads / nu;
        const int u = threadIdx.x % nu, r0 = threadIdx.x / nu;
        int e;
        unit_setup(u, e, c, s);
        for (int jb = r0; jb < ntok; jb += rpp * kIngestUnroll) {
            uint4 va[kIngestUnroll], vb[kIngestUnroll];
            bool ok[kIngestUnroll];
#pragma unroll
            for (int k = 0; k < kIngestUnroll; ++k) {   // every row's loads first ...
                const int j = jb + k * rpp;
                ok[k] = j < ntok && slots[j] >= 0;
                if (ok[k])
                    unit_load<KIND>(src + slots[j] * p.src_ss, e, ps.half, va[k], vb[k]);
            }
#pragma unroll
            for (int k = 0; k < kIngestUnroll; ++k)      // ... then the arithmetic and the stores
                if (ok[k])
                    unit_store<KIND>(dst + (int64_t)(jb + k * rpp) * p.dst_rs, e, ps.half, va[k], vb[k], c, s, turn);
        }
    } else {                          // (row, unit) items strided over the block
        for (int item = threadIdx.x; item < ntok * nu; item += kIngestThreads) {
            const int j = item / nu, u = item - j * nu;
            if (slots[j] < 0)
                continue;
            int e;
            uint4 va, vb;
            unit_setup(u, e, c, s);
            unit_load<KIND>(src + slots[j] * p.src_ss, e, ps.half, va, vb);
            unit_store<KIND>(dst + (int64_t)j * p.dst_rs, e, ps.half, va, vb, c, s, turn);
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(kIngestThreads, 2) ingest_kernel(const __grid_constant__ IngestParams p, int pass,
                                                                int tiles_per_chunk, int layers_per_cta)
{
    __shared__ float2 cs[KAMERA_MAX_ROT_DIM / 2];
    __shared__ int64_t slots[kIngestTile];
    const int chunk = blockIdx.x / tiles_per_chunk, tile = blockIdx.x - chunk * tiles_per_chunk;
    const KameraChunk ch = p.chunks[chunk];
    int32_t bad = check_axis_delta(p.rope, chunk);
    if (ch.len < 0 || ch.rank != 0 || ch.delta > KAMERA_MAX_ABS_DELTA || ch.delta < -KAMERA_MAX_ABS_DELTA ||
        (ch.len > 0 && (ch.dst_slot_mapping == nullptr || (reinterpret_cast<uintptr_t>(ch.dst_slot_mapping) & 15))))
        bad |= KAMERA_DEVERR_DESCRIPTOR;
    if (ch.src_offset < 0 || ch.src_offset + (int64_t)ch.len > p.num_rows)
        bad |= KAMERA_DEVERR_SOURCE;
    if (ch.len > p.max_len)
        bad |= KAMERA_DEVERR_LEN;
    if (bad) {
        if (tile == 0 && blockIdx.y == 0 && threadIdx.x == 0 && pass == 0)
            raise_err(p.err, bad);
        return;
    }
    const int t0 = tile * kIngestTile;
    if (t0 >= ch.len)
        return;
    const int ntok = min(kIngestTile, ch.len - t0);
    const bool turn = chunk_turns(p.rope, ch, chunk);
    if (KIND != INGEST_COPY && turn)
        for (int f = threadIdx.x; f < p.rope.n_freq; f += kIngestThreads) {
            float c, s;
            phase_cos_sin(freq_delta(p.rope, ch, chunk, f), p.rope.inv_freq[f], c, s);
            cs[f] = make_float2(c, s);
        }
    for (int j = threadIdx.x; j < ntok; j += kIngestThreads) {
        int64_t sl = ch.dst_slot_mapping[t0 + j];
        if (sl < 0 || sl >= p.num_slots) {
            if (blockIdx.y == 0 && pass == 0)
                raise_err(p.err, KAMERA_DEVERR_SLOT);
            sl = -1;
        }
        slots[j] = sl;
    }
    __syncthreads();
    const int64_t row0 = ch.src_offset + t0;
    const int l_end = min(p.L, (int)(blockIdx.y + 1) * layers_per_cta);
    for (int l = blockIdx.y * layers_per_cta; l < l_end; ++l) {
        ingest_pass<KIND>(p, p.pass[pass], cs, slots, l, row0, ntok, turn);
    }
}

}  // namespace

// Passes of one row, per head: the vectors before the rotary range, the rotary
// units, the vectors after it (array 0); the whole value row (array 1).
int ingest_passes(const RowsParams& rp, bool values, IngestPass* out)
{
    int n = 0;
    const int d = rp.d, r = rp.rope.rot_dim, o = rp.rope.rot_offset;
    const bool half = rp.rope.pairing == KAMERA_ROPE_ROTATE_HALF;
    if (o % 8 || r % (half ? 16 : 8) || o + r > d || d % 8)
        return -1;
    auto add = [&](int array, int kind, int off, int per_head, int half, int f_off) {
        if (per_head > 0)
            out[n++] = IngestPass{array, kind, off, per_head, half, f_off};
    };
    add(0, INGEST_COPY, 0, o / 8, 0, 0);
    if (r > 0) {
        if (half)
            add(0, INGEST_ROT_HALF, o, r / 16, r / 2, 0);
        else
            add(0, INGEST_ROT_IL, o, r / 8, 0, 0);
    }
    add(0, INGEST_COPY, o + r, (d - o - r) / 8, 0, 0);
    if (values)
        add(1, INGEST_COPY, 0, d / 8, 0, 0);
    return n;
}

cudaError_t launch_ingest(const IngestParams& p, cudaStream_t stream)
{
    const int tiles = (p.max_len + kIngestTile - 1) / kIngestTile;
    const int64_t tile_rows = (int64_t)p.n_chunks * tiles;
    int lg = (int)((tile_rows * p.L) / 4096);
    lg = lg < 1 ? 1 : (lg > 8 ? 8 : lg);
    if (lg > p.L)
        lg = p.L;
    const dim3 grid((unsigned)tile_rows, (unsigned)((p.L + lg - 1) / lg));
    for (int q = 0; q < p.n_pass; ++q) {
        switch (p.pass[q].kind) {
        case INGEST_ROT_HALF: ingest_kernel<INGEST_ROT_HALF><<<grid, kIngestThreads, 0, stream>>>(p, q, tiles, lg); break;
        case INGEST_ROT_IL: ingest_kernel<INGEST_ROT_IL><<<grid, kIngestThreads, 0, stream>>>(p, q, tiles, lg); break;
        default: ingest_kernel<INGEST_COPY><<<grid, kIngestThreads, 0, stream>>>(p, q, tiles, lg); break;
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace kamera
