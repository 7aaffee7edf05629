/*
 * kamera_oracle.c -- plain, slow, fp64 CPU oracle of the Kamera reuse operator.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg are the only code allowed to load
 * this library.  The CUDA product path never calls it; the two share no code,
 * header, table or constant generator.
 *
 * Source of the definition: "Kamera: Unified Position-Invariant Multimodal KV
 * Cache for Training-Free Reuse" as summarised on gist.science (paper
 * 2606.23581), Technical Summary section 2 ("Methodology: The Kamera
 * Operator"), the reuse equation
 *
 *     KV^(B|A) = R(delta) . KV(B|empty) + U_m V_m^T
 *
 * with R(delta) the exact RoPE phase shift of the keys by delta positions
 * ("an exact algebraic operation, not a forward pass") and U_m V_m^T the rank-m
 * conditioning patch added to K and V.  Section 2 "Unified Architecture
 * Support" gives the per-family rule (GQA/MHA: the whole key is relocated and
 * both K and V are patched; MLA: only the 64-dim k_rope is relocated, c_KV is
 * reused byte for byte, both channels are patched).  Section 3.2 (sliding-
 * window survival) gives the rotation-only relocation of survivors.
 *
 * Everything is computed in fp64 and rounded ONCE, directly from fp64 to bf16
 * with round-to-nearest-even (no fp32 intermediate, which would double-round).
 * Readings of points the pages leave open:
 *   - the patch is added after the rotation, in the target frame (the
 *     equation as printed);
 *   - theta_i = base^(-2i/r) for i < r/2 (standard RoPE; the pages give none);
 *   - delta moves a chunk later when positive: RoPE(x, p + delta) =
 *     R(delta) RoPE(x, p);
 *   - R(0) is the identity and an empty patch adds nothing, so delta = 0 with
 *     m = 0 reproduces the stored bits exactly (including -0.0);
 *   - pairing ROTATE_HALF pairs (o+i, o+i+r/2); INTERLEAVED pairs
 *     (o+2i, o+2i+1); in both, pair i turns by delta*theta_i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PAIRING_ROTATE_HALF 0
#define ORACLE_PAIRING_INTERLEAVED 1

/* ---------------------------------------------------------------- bf16 --- */

/* Exact widening of a bf16 bit pattern: the top 16 bits of an IEEE binary32. */
double kamera_oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round an fp64 value to the nearest bf16 (8 exponent bits, 7 stored mantissa
 * bits), ties to even, in one step.  Finite |x| lies in a binade whose bf16
 * spacing is q = 2^(e-7) (e = floor(log2|x|), clamped to the subnormal
 * spacing 2^-133); |x|/q is then exact in fp64, rint() rounds it half-to-even
 * in the default rounding mode, and the result times q is a bf16 value,
 * hence exactly representable in binary32 whose top half is the answer.
 */
uint16_t kamera_oracle_bf16_rne(double x)
{
    if (isnan(x))
        return (uint16_t)0x7FC0;
    const uint16_t sign = signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    if (a == 0.0)
        return sign;
    int E;
    (void)frexp(a, &E);            /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;                 /* floor(log2 a) */
    if (e < -126)
        e = -126;                  /* subnormal range keeps spacing 2^-133 */
    double q = ldexp(1.0, e - 7);
    double n = rint(a / q);        /* half to even */
    double v = n * q;
    if (v >= ldexp(1.0, 128))      /* beyond the largest finite bf16 */
        return (uint16_t)(sign | 0x7F80);
    float f = (float)v;            /* exact: v is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void kamera_oracle_bf16_rne_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kamera_oracle_bf16_rne(x[i]);
}

void kamera_oracle_bf16_to_f64_array(const uint16_t* x, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kamera_oracle_bf16_to_f64(x[i]);
}

/* ---------------------------------------------------------------- RoPE --- */

/* theta_i = base^(-2i/r), i = 0 .. r/2-1 (standard rotary frequencies). */
void kamera_oracle_inv_freq(double base, int rot_dim, double* out)
{
    for (int i = 0; i < rot_dim / 2; ++i)
        out[i] = pow(base, -2.0 * (double)i / (double)rot_dim);
}

/* Indices of the two components that pair i of the rotary range turns. */
static void pair_index(int i, int rot_dim, int rot_offset, int pairing, int* a, int* b)
{
    if (pairing == ORACLE_PAIRING_INTERLEAVED) {
        *a = rot_offset + 2 * i;
        *b = rot_offset + 2 * i + 1;
    } else {
        *a = rot_offset + i;
        *b = rot_offset + i + rot_dim / 2;
    }
}

/*
 * R(delta) applied in place to one row x[0..width): every pair (x_a, x_b) of
 * the rotary range turns by phi_i = delta*theta_i,
 *     x_a' = x_a cos(phi_i) - x_b sin(phi_i)
 *     x_b' = x_b cos(phi_i) + x_a sin(phi_i)
 * i.e. (x_a + i x_b) * exp(i phi_i).  Components outside the rotary range are
 * left alone.  delta = 0 is the identity, applied as such.
 * If scale is non-NULL it receives, per component, the sum of the magnitudes
 * of the terms that made it (|x_a cos| + |x_b sin|, or |x| when untouched).
 */
void kamera_oracle_rotate(double* x, int width, int64_t delta, const double* inv_freq,
                          int rot_dim, int rot_offset, int pairing, double* scale)
{
    if (scale)
        for (int c = 0; c < width; ++c)
            scale[c] = fabs(x[c]);
    if (delta == 0)
        return;
    for (int i = 0; i < rot_dim / 2; ++i) {
        int a, b;
        pair_index(i, rot_dim, rot_offset, pairing, &a, &b);
        double phi = (double)delta * inv_freq[i];
        double c = cos(phi), s = sin(phi);
        double xa = x[a], xb = x[b];
        x[a] = xa * c - xb * s;
        x[b] = xb * c + xa * s;
        if (scale) {
            scale[a] = fabs(xa * c) + fabs(xb * s);
            scale[b] = fabs(xb * c) + fabs(xa * s);
        }
    }
}

/*
 * One output row of the operator: y = R(delta) x + sum_r u[r] * vm[c][r].
 *   x       : width bf16 values (the canonical row)
 *   rotate  : 0 for value rows and c_KV (never rotated), 1 for key rows
 *   u       : m bf16 values, this token's row of U_m          (NULL iff m == 0)
 *   vm      : width x m bf16 values, V_m row-major, c-major   (NULL iff m == 0)
 * Outputs (each optional): bf16 bits, the fp64 value before rounding, and the
 * per-component magnitude scale (rotation terms plus sum |u_r vm_cr|).
 */
void kamera_oracle_row(const uint16_t* x, int width, int rotate, int64_t delta,
                       const double* inv_freq, int rot_dim, int rot_offset, int pairing,
                       const uint16_t* u, const uint16_t* vm, int m,
                       uint16_t* out_bf16, double* out_f64, double* out_scale)
{
    double* y = (double*)malloc(sizeof(double) * (size_t)width);
    double* sc = (double*)malloc(sizeof(double) * (size_t)width);
    for (int c = 0; c < width; ++c)
        y[c] = kamera_oracle_bf16_to_f64(x[c]);
    if (rotate)
        kamera_oracle_rotate(y, width, delta, inv_freq, rot_dim, rot_offset, pairing, sc);
    else
        for (int c = 0; c < width; ++c)
            sc[c] = fabs(y[c]);
    if (m > 0) {
        for (int c = 0; c < width; ++c) {
            double acc = 0.0, mag = 0.0;
            for (int r = 0; r < m; ++r) {
                double p = kamera_oracle_bf16_to_f64(u[r]) *
                           kamera_oracle_bf16_to_f64(vm[(size_t)c * m + r]);
                acc += p;
                mag += fabs(p);
            }
            y[c] += acc;
            sc[c] += mag;
        }
    }
    for (int c = 0; c < width; ++c) {
        if (out_bf16)
            out_bf16[c] = kamera_oracle_bf16_rne(y[c]);
        if (out_f64)
            out_f64[c] = y[c];
        if (out_scale)
            out_scale[c] = sc[c];
    }
    free(y);
    free(sc);
}

/* ------------------------------------------------------ whole problems --- */

/*
 * Chunk list, one entry per chunk (all host arrays of n_chunks entries):
 *   src_offset[c], len[c]  : canonical rows [src_offset, src_offset+len) of the store
 *   delta[c]               : RoPE phase shift in positions
 *   rank[c]                : patch rank m (0 = no patch)
 *   p0[c] .. p3[c]         : patch factor pointers (see each problem)
 *   slots[c]               : len[c] pool slot indices
 * Returns 0, or -1 (writing nothing further) when an index is out of range.
 */

static int check_chunk(int64_t src_offset, int32_t len, int64_t n_store_rows,
                       const int64_t* slots, int64_t n_slots)
{
    if (len < 0 || src_offset < 0 || src_offset + len > n_store_rows)
        return -1;
    for (int32_t j = 0; j < len; ++j)
        if (slots[j] < 0 || slots[j] >= n_slots)
            return -1;
    return 0;
}

/*
 * GQA / MHA relocate + patch + scatter.  Store and pool rows are H heads of d
 * elements; element (l, row, h, i) lives at base[l*layer_stride + row*row_stride
 * + h*d + i].  Patch factors per chunk, layer and head:
 *   Uk = p0, Vk = p1, Uv = p2, Vv = p3;  U: [L][H][len][m],  V_m: [L][H][d][m].
 * Keys: R(delta) over the rotary range, plus Uk Vk^T.  Values: plus Uv Vv^T.
 * Optional scale outputs have the pool's shape and strides.
 */
int kamera_oracle_gqa(int L, int H, int d,
                      const uint16_t* store_k, const uint16_t* store_v, int64_t n_store_rows,
                      int64_t store_layer_stride, int64_t store_row_stride,
                      uint16_t* pool_k, uint16_t* pool_v, int64_t n_slots,
                      int64_t pool_layer_stride, int64_t pool_row_stride,
                      const double* inv_freq, int rot_dim, int rot_offset, int pairing,
                      int n_chunks, const int64_t* src_offset, const int32_t* len,
                      const int64_t* delta, const int32_t* rank,
                      const uint16_t* const* p0, const uint16_t* const* p1,
                      const uint16_t* const* p2, const uint16_t* const* p3,
                      const int64_t* const* slots,
                      double* scale_k, double* scale_v)
{
    for (int c = 0; c < n_chunks; ++c)
        if (check_chunk(src_offset[c], len[c], n_store_rows, slots[c], n_slots))
            return -1;
    for (int c = 0; c < n_chunks; ++c) {
        const int32_t T = len[c];
        const int m = rank[c];
        const int64_t work = (int64_t)L * T;
#pragma omp parallel for schedule(static)
        for (int64_t w = 0; w < work; ++w) {
            const int l = (int)(w / T);
            const int32_t j = (int32_t)(w % T);
            const int64_t src = src_offset[c] + j;
            const int64_t dst = slots[c][j];
            for (int h = 0; h < H; ++h) {
                const int64_t so = l * store_layer_stride + src * store_row_stride + (int64_t)h * d;
                const int64_t po = l * pool_layer_stride + dst * pool_row_stride + (int64_t)h * d;
                const uint16_t *uk = NULL, *vk = NULL, *uv = NULL, *vv = NULL;
                if (m > 0) {
                    const int64_t lh = (int64_t)l * H + h;
                    uk = p0[c] + (lh * T + j) * m;
                    vk = p1[c] + lh * (int64_t)d * m;
                    uv = p2[c] + (lh * T + j) * m;
                    vv = p3[c] + lh * (int64_t)d * m;
                }
                kamera_oracle_row(store_k + so, d, 1, delta[c], inv_freq, rot_dim, rot_offset,
                                  pairing, uk, vk, m, pool_k + po, NULL,
                                  scale_k ? scale_k + po : NULL);
                kamera_oracle_row(store_v + so, d, 0, 0, inv_freq, rot_dim, rot_offset,
                                  pairing, uv, vv, m, pool_v + po, NULL,
                                  scale_v ? scale_v + po : NULL);
            }
        }
    }
    return 0;
}

/*
 * MLA relocate + patch + scatter.  A row is c_KV (kv_lora elements) followed
 * by k_rope (rope_dim elements); element (l, row, i) at
 * base[l*layer_stride + row*row_stride + i].  The rotary range is k_rope,
 * i.e. offset kv_lora, width rope_dim, turned by R(delta).  c_KV is never
 * rotated.  Patch factors per chunk and layer:
 *   Uc = p0 [L][len][m], Vc = p1 [L][kv_lora][m], Ur = p2 [L][len][m], Vr = p3 [L][rope_dim][m].
 */
int kamera_oracle_mla(int L, int kv_lora, int rope_dim,
                      const uint16_t* store, int64_t n_store_rows,
                      int64_t store_layer_stride, int64_t store_row_stride,
                      uint16_t* pool, int64_t n_slots,
                      int64_t pool_layer_stride, int64_t pool_row_stride,
                      const double* inv_freq, int pairing,
                      int n_chunks, const int64_t* src_offset, const int32_t* len,
                      const int64_t* delta, const int32_t* rank,
                      const uint16_t* const* p0, const uint16_t* const* p1,
                      const uint16_t* const* p2, const uint16_t* const* p3,
                      const int64_t* const* slots, double* scale)
{
    for (int c = 0; c < n_chunks; ++c)
        if (check_chunk(src_offset[c], len[c], n_store_rows, slots[c], n_slots))
            return -1;
    for (int c = 0; c < n_chunks; ++c) {
        const int32_t T = len[c];
        const int m = rank[c];
        const int64_t work = (int64_t)L * T;
#pragma omp parallel for schedule(static)
        for (int64_t w = 0; w < work; ++w) {
            const int l = (int)(w / T);
            const int32_t j = (int32_t)(w % T);
            const int64_t so = l * store_layer_stride + (src_offset[c] + j) * store_row_stride;
            const int64_t po = l * pool_layer_stride + slots[c][j] * pool_row_stride;
            const uint16_t *uc = NULL, *vc = NULL, *ur = NULL, *vr = NULL;
            if (m > 0) {
                uc = p0[c] + ((int64_t)l * T + j) * m;
                vc = p1[c] + (int64_t)l * kv_lora * m;
                ur = p2[c] + ((int64_t)l * T + j) * m;
                vr = p3[c] + (int64_t)l * rope_dim * m;
            }
            kamera_oracle_row(store + so, kv_lora, 0, 0, inv_freq, 0, 0, pairing, uc, vc, m,
                              pool + po, NULL, scale ? scale + po : NULL);
            kamera_oracle_row(store + so + kv_lora, rope_dim, 1, delta[c], inv_freq, rope_dim, 0,
                              pairing, ur, vr, m, pool + po + kv_lora, NULL,
                              scale ? scale + po + kv_lora : NULL);
        }
    }
    return 0;
}

/*
 * Sliding-window survival, in place (technical summary section 3.2): every
 * surviving key row at slot s is replaced by R(delta) of itself; no patch,
 * values untouched.  Rows are H heads of d elements as in the GQA layout; the
 * rotary range (rot_offset, rot_dim) is taken inside each head, which also
 * covers MLA's k_rope with H = 1, d = row width, rot_offset = c_KV width.
 */
int kamera_oracle_slide(int L, int H, int d, uint16_t* pool_k, int64_t n_slots,
                        int64_t pool_layer_stride, int64_t pool_row_stride,
                        const double* inv_freq, int rot_dim, int rot_offset, int pairing,
                        int n_chunks, const int32_t* len, const int64_t* delta,
                        const int64_t* const* slots, double* scale_k)
{
    if (d > 4096)
        return -1;
    for (int c = 0; c < n_chunks; ++c) {
        if (len[c] < 0)
            return -1;
        for (int32_t j = 0; j < len[c]; ++j)
            if (slots[c][j] < 0 || slots[c][j] >= n_slots)
                return -1;
    }
    for (int c = 0; c < n_chunks; ++c) {
        const int32_t T = len[c];
        const int64_t work = (int64_t)L * T;
#pragma omp parallel for schedule(static)
        for (int64_t w = 0; w < work; ++w) {
            const int l = (int)(w / T);
            const int32_t j = (int32_t)(w % T);
            for (int h = 0; h < H; ++h) {
                const int64_t po = l * pool_layer_stride + slots[c][j] * pool_row_stride + (int64_t)h * d;
                uint16_t row[4096];
                memcpy(row, pool_k + po, sizeof(uint16_t) * (size_t)d);
                kamera_oracle_row(row, d, 1, delta[c], inv_freq, rot_dim, rot_offset, pairing,
                                  NULL, NULL, 0, pool_k + po, NULL,
                                  scale_k ? scale_k + po : NULL);
            }
        }
    }
    return 0;
}

/* Canonical ingest, the inverse of relocation: a chunk that sits in the live
 * paged cache at positions s..s+len-1 is read back from its slots and turned
 * to the position-free canonical frame (its first token at position 0) by
 * R(-s).  With delta_c = -s_c, for every chunk c, layer l, head h, token j:
 *   store_k[l][row_c + j][h] = bf16( R(delta_c) pool_k[l][slot_j][h] )
 *   store_v[l][row_c + j][h] = pool_v[l][slot_j][h]          (when pool_v)
 * (Canonical KV: gist.science technical summary, section 2; R(delta) as in
 * kamera_oracle_rotate, so delta = 0 copies the row bit for bit.)  MLA rows
 * are H = 1 segments of d = kv_lora + rope elements with the rotary range at
 * rot_offset = kv_lora: c_KV is copied, k_rope turned.  Returns -1 on an
 * out-of-range slot or store row. */
int kamera_oracle_ingest(int L, int H, int d,
                         const uint16_t* pool_k, const uint16_t* pool_v, int64_t n_slots,
                         int64_t pool_layer_stride, int64_t pool_row_stride,
                         uint16_t* store_k, uint16_t* store_v, int64_t n_store_rows,
                         int64_t store_layer_stride, int64_t store_row_stride,
                         const double* inv_freq, int rot_dim, int rot_offset, int pairing,
                         int n_chunks, const int64_t* dst_row, const int32_t* len, const int64_t* delta,
                         const int64_t* const* slots, double* scale_k)
{
    for (int c = 0; c < n_chunks; ++c) {
        if (len[c] < 0 || dst_row[c] < 0 || dst_row[c] + len[c] > n_store_rows)
            return -1;
        for (int32_t j = 0; j < len[c]; ++j)
            if (slots[c][j] < 0 || slots[c][j] >= n_slots)
                return -1;
    }
    for (int c = 0; c < n_chunks; ++c) {
        const int32_t T = len[c];
        const int64_t work = (int64_t)L * T;
#pragma omp parallel for schedule(static)
        for (int64_t w = 0; w < work; ++w) {
            const int l = (int)(w / T);
            const int32_t j = (int32_t)(w % T);
            const int64_t po = l * pool_layer_stride + slots[c][j] * pool_row_stride;
            const int64_t so = l * store_layer_stride + (dst_row[c] + j) * store_row_stride;
            for (int h = 0; h < H; ++h) {
                kamera_oracle_row(pool_k + po + (int64_t)h * d, d, 1, delta[c], inv_freq, rot_dim, rot_offset,
                                  pairing, NULL, NULL, 0, store_k + so + (int64_t)h * d, NULL,
                                  scale_k ? scale_k + so + (int64_t)h * d : NULL);
                if (pool_v)
                    memcpy(store_v + so + (int64_t)h * d, pool_v + po + (int64_t)h * d, sizeof(uint16_t) * (size_t)d);
            }
        }
    }
    return 0;
}

/* Threads the OpenMP runtime would use (1 when built without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int kamera_oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int kamera_oracle_num_threads(void) { return 1; }
#endif
