// kamera_common.cuh -- device helpers shared by the Kamera kernels (sm_103a).
//
// The operator (Kamera, gist.science technical summary section 2, reuse
// equation) is  KV^(B|A) = R(delta) KV(B|empty) + U_m V_m^T.  This header holds
// the pieces every kernel needs: the launch parameter blocks, bf16 packing,
// the fp64-formed RoPE phase, descriptor checks and device error reporting.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kamera.h"

namespace kamera {

// ------------------------------------------------------------ parameters --
struct RopeParams {
    int32_t rot_dim;       // rotated components (0 = none)
    int32_t rot_offset;    // first rotated component inside the row segment
    int32_t pairing;       // KAMERA_ROPE_*
    int32_t n_freq;        // rot_dim / 2
    double inv_freq[KAMERA_MAX_ROT_DIM / 2];
    const int64_t* axis_delta;              // multi-axis RoPE: [n_chunks][n_axes], else null
    int32_t n_axes;                         // 0: every frequency turns by the chunk's delta
    uint8_t axis[KAMERA_MAX_ROT_DIM / 2];   // frequency f follows axis[f] (n_axes > 0)
};

// A family-neutral description of one call: token rows are read from `src`
// (the canonical store; the pool itself for the in-place slide) and written to
// `dst` at the chunk's slots.  Each kernel cuts a row into segments (GQA: one
// head of K or V; MLA: 128-wide c_KV blocks, then k_rope; slide: one head).
struct RowsParams {
    // destination (pool), element (l, s, e) at dst[l*dst_ls + s*dst_ss + e]
    __nv_bfloat16* dst_k;
    __nv_bfloat16* dst_v;           // GQA values (NULL for MLA / slide)
    int64_t num_slots;
    int64_t dst_ls, dst_ss;
    // source (store), element (l, r, e) at src[l*src_ls + r*src_rs + e]
    const __nv_bfloat16* src_k;
    const __nv_bfloat16* src_v;
    int64_t num_rows;               // rows in the store (ignored in place)
    int64_t src_ls, src_rs;
    int32_t L;
    int32_t H;                      // GQA heads (1 for MLA)
    int32_t d;                      // GQA head_dim; MLA row width
    int32_t kv_lora;                // MLA c_KV width (0 for GQA)
    const KameraChunk* chunks;
    int32_t n_chunks;
    int32_t max_len;
    int32_t max_rank;
    int32_t tiles_per_chunk;
    int32_t* err;
    RopeParams rope;
};

// Canonical ingest (kamera_ingest.cu): a pass is a set of 16-byte units of a
// row, repeated per head (head h's unit i starts at element h*d + off + 8*i).
enum IngestKind { INGEST_COPY = 0, INGEST_ROT_HALF = 1, INGEST_ROT_IL = 2 };

struct IngestPass {
    int32_t array;      // 0: K (or the MLA row), 1: V
    int32_t kind;       // IngestKind
    int32_t off;        // first element of head 0's unit 0
    int32_t per_head;   // units per head
    int32_t half;       // rotate-half: distance in elements to the partner vector
    int32_t f_off;      // rotary units: first frequency of unit 0
};

struct IngestParams {
    const __nv_bfloat16* src[2];   // pool arrays (K | V, or the MLA row), read at the slots
    __nv_bfloat16* dst[2];         // store arrays, written at rows src_offset..
    int64_t src_ls, src_ss;        // pool layer and slot strides (elements)
    int64_t dst_ls, dst_rs;        // store layer and row strides
    int64_t num_slots, num_rows;
    int32_t L, H, d;               // layers; heads of a row and their stride (elements)
    int32_t n_pass;
    IngestPass pass[6];
    const KameraChunk* chunks;
    int32_t n_chunks, max_len;
    int32_t* err;
    RopeParams rope;
};

// Patch formation: blocks (o, i) of a deficit, block index o * n_inner + i.
struct PatchFormParams {
    const __nv_bfloat16* x;        // deficit, block (o, i) at x + o * outer_stride + i * inner_stride
    int64_t n_inner, outer_stride, inner_stride, row_stride, term_stride;   // elements
    int32_t n_terms;               // deficits averaged per block (orbit patch), >= 1
    int32_t rows, cols, m;
    __nv_bfloat16* u;              // [blocks][rows][m]
    __nv_bfloat16* v;              // [blocks][cols][m]
    float* sigma;                  // [blocks][m] or null
    int32_t* err;
    uint64_t wait_ns;              // bound of each MMA completion wait (wait_limit_ns())
    int32_t cluster;               // wide blocks: CTAs of a cluster sharing one block's rows
};

// Decode attention over reused chunks: one layer's canonical store, sequences
// of chunks, one query token per sequence.
struct AttendParams {
    const __nv_bfloat16* k;        // canonical keys / values of one layer: rows of H x d,
    const __nv_bfloat16* v;        // row_stride elements apart
    int64_t row_stride, num_rows;
    int32_t H, d, G, layer;        // KV heads, head dim, query heads per KV head, factor layer
    const KameraChunk* chunks;
    const int32_t* seq_start;      // [n_seqs + 1]: sequence s = chunks seq_start[s] .. seq_start[s+1]-1
    int32_t n_seqs, n_chunks;
    const __nv_bfloat16* q;        // [n_seqs][H * G][d]
    __nv_bfloat16* out;            // [n_seqs][H * G][d]
    float scale;
    int32_t max_len, max_rank;
    int32_t cluster;               // CTAs per (sequence, KV head), 1..8
    int32_t* err;
    RopeParams rope;
};

// MLA decode attention over reused chunks: one layer's latent store (rows of
// c_KV (kv_lora) then k_rope (rope_dim)), absorbed queries (the latent part
// then the rope part), one query token per sequence and query head.
struct MlaAttendParams {
    const __nv_bfloat16* kv;       // [num_rows] rows of kv_lora + rope_dim, row_stride elements apart
    int64_t row_stride, num_rows;
    int32_t kv_lora, rope_dim, Hq, layer;
    const KameraChunk* chunks;     // factors Uc [L][len][m], Vc [L][kv_lora][m], Ur [L][len][m], Vr [L][rope_dim][m]
    const int32_t* seq_start;      // [n_seqs + 1]
    int32_t n_seqs, n_chunks;
    const __nv_bfloat16* q;        // [n_seqs][Hq][kv_lora + rope_dim]
    __nv_bfloat16* out;            // [n_seqs][Hq][kv_lora]
    float scale;
    int32_t max_len, max_rank;
    int32_t cluster;               // CTAs per sequence, 1..8
    int32_t* err;
    RopeParams rope;               // rot_offset relative to k_rope
};

// Prefill attention over reused chunks: T new query tokens per sequence, each
// attending over the reuse equation's rows of the sequence's chunks (which all
// precede the new tokens, so no mask applies among them).
struct PrefillParams {
    const __nv_bfloat16* k;        // canonical keys / values of one layer: rows of H x d,
    const __nv_bfloat16* v;        // row_stride elements apart
    int64_t row_stride, num_rows;
    int32_t H, d, G, layer;        // KV heads, head dim, query heads per KV head, factor layer
    const KameraChunk* chunks;
    const int32_t* seq_start;      // [n_seqs + 1]
    int32_t n_seqs, n_chunks;
    int32_t T;                     // query tokens per sequence
    int32_t blocks;                // 128-row blocks of one (sequence, KV head)'s T x G query rows
    const __nv_bfloat16* q;        // [n_seqs][T][H * G][d]
    __nv_bfloat16* out;            // [n_seqs][T][H * G][d]
    float* lse;                    // [n_seqs][T][H * G] (natural log), or NULL
    float scale;
    int32_t max_len, max_rank;
    int32_t* err;
    RopeParams rope;
};

// ------------------------------------------------------------------ bf16 --
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2, each rounded to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f)
{
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float* f)
{
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    return v;
}

// ----------------------------------------------------------------- phase --
// cos/sin of phi = delta * theta.  The product is formed in fp64 (exact to
// ~1 ulp of phi) and reduced to [-pi, pi] with a two-term Cody-Waite split of
// 2*pi (Cody & Waite, "Software Manual for the Elementary Functions", 1980):
// hi = fp64(2*pi), lo = 2*pi - hi.  With |k| < 2^31 the two fused steps leave
// an error of a few fp64 ulps of pi, so the only fp32 rounding is that of the
// reduced angle (<= 2^-24 * pi) and of sincosf itself.
__device__ __forceinline__ void phase_cos_sin(int64_t delta, double theta, float& c, float& s)
{
    const double kTwoPiHi = 6.283185307179586232;     // 0x401921FB54442D18
    const double kTwoPiLo = 2.4492935982947064e-16;   // 2*pi - kTwoPiHi
    const double kInvTwoPi = 0.15915494309189535;
    const double phi = (double)delta * theta;
    const double k = rint(phi * kInvTwoPi);
    double red = fma(-k, kTwoPiHi, phi);
    red = fma(-k, kTwoPiLo, red);
    sincosf((float)red, &s, &c);
}

// Multi-axis RoPE: frequency f of chunk c turns by that chunk's move along the
// axis f follows; without axes, by the descriptor's delta.
__device__ __forceinline__ int64_t freq_delta(const RopeParams& r, const KameraChunk& ch, int c, int f)
{
    return r.n_axes == 0 ? ch.delta : r.axis_delta[(int64_t)c * r.n_axes + r.axis[f]];
}

// Whether chunk c turns at all (a chunk that does not is copied bit for bit).
__device__ __forceinline__ bool chunk_turns(const RopeParams& r, const KameraChunk& ch, int c)
{
    if (r.n_axes == 0)
        return ch.delta != 0;
    bool any = false;
    for (int a = 0; a < r.n_axes; ++a)
        any |= r.axis_delta[(int64_t)c * r.n_axes + a] != 0;
    return any;
}

// KAMERA_DEVERR_DESCRIPTOR when one of chunk c's axis moves is out of range.
__device__ __forceinline__ int32_t check_axis_delta(const RopeParams& r, int c)
{
    int32_t bits = 0;
    for (int a = 0; a < r.n_axes; ++a) {
        const int64_t v = r.axis_delta[(int64_t)c * r.n_axes + a];
        if (v > KAMERA_MAX_ABS_DELTA || v < -KAMERA_MAX_ABS_DELTA)
            bits |= KAMERA_DEVERR_DESCRIPTOR;
    }
    return bits;
}

// patch_ptrs[i] without dynamic indexing (keeps a descriptor in registers)
__device__ __forceinline__ const __nv_bfloat16* patch_ptr(const KameraChunk& ch, int i)
{
    const void* v = i == 0 ? ch.patch_ptrs[0] : i == 1 ? ch.patch_ptrs[1] : i == 2 ? ch.patch_ptrs[2] : ch.patch_ptrs[3];
    return static_cast<const __nv_bfloat16*>(v);
}

// ---------------------------------------------------------------- errors --
__device__ __forceinline__ void raise_err(int32_t* err, int32_t bits)
{
    if (err)
        atomicOr(err, bits);
}

// Checks one descriptor against the call; returns 0 when the chunk may run,
// else the KAMERA_DEVERR_* bits (the chunk is then skipped whole).
// in_place: the slide (src_offset ignored, rank must be 0).
__device__ __forceinline__ int32_t check_chunk(const KameraChunk& ch, int c, const RowsParams& p, bool in_place)
{
    int32_t bits = check_axis_delta(p.rope, c);
    if (ch.len < 0 || ch.rank < 0 || ch.delta > KAMERA_MAX_ABS_DELTA || ch.delta < -KAMERA_MAX_ABS_DELTA)
        bits |= KAMERA_DEVERR_DESCRIPTOR;
    if (ch.len > 0 && (ch.dst_slot_mapping == nullptr || (reinterpret_cast<uintptr_t>(ch.dst_slot_mapping) & 15)))
        bits |= KAMERA_DEVERR_DESCRIPTOR;
    if (in_place) {
        if (ch.rank != 0)
            bits |= KAMERA_DEVERR_DESCRIPTOR;
    } else {
        if (ch.src_offset < 0 || ch.len < 0 || ch.src_offset + (int64_t)ch.len > p.num_rows)
            bits |= KAMERA_DEVERR_SOURCE;
        if (ch.rank > 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(ch.patch_ptrs[i]);
                if (a == 0 || (a & 15))
                    bits |= KAMERA_DEVERR_DESCRIPTOR;
            }
        } else if (ch.rank == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (ch.patch_ptrs[i] != nullptr)
                    bits |= KAMERA_DEVERR_DESCRIPTOR;
        }
    }
    if (ch.len > p.max_len)
        bits |= KAMERA_DEVERR_LEN;
    if (ch.rank > p.max_rank)
        bits |= KAMERA_DEVERR_RANK;
    return bits;
}

}  // namespace kamera
