/*
 * kamera.h -- C ABI of the GB300 (sm_103a) Kamera reuse operator.
 *
 * The operator is the reuse equation of "Kamera: Unified Position-Invariant
 * Multimodal KV Cache for Training-Free Reuse" (gist.science technical summary,
 * section 2, "Methodology: The Kamera Operator"):
 *
 *     KV^(B|A) = R(delta) . KV(B|empty) + U_m V_m^T
 *
 * A chunk B was prefilled once with no antecedent and stored position-free
 * (the canonical store, section 2 "Canonical KV").  To reuse it at a new
 * position its keys are turned by the exact RoPE phase shift R(delta) ("an
 * exact algebraic operation, not a forward pass"), the rank-m conditioning
 * patch U_m V_m^T (section 2 "Rank-m Conditioning Patch") is added to keys and
 * values, and the rows are written into a paged KV pool at the slots the
 * caller chose.  Section 2 "Unified Architecture Support" fixes the
 * per-family rule, one entry point each:
 *
 *   kamera_relocate_patch      GQA and MHA: the whole key (the rotary range of
 *                              each head) is re-rotated; K and V are patched.
 *   kamera_mla_relocate_patch  MLA: only the 64-dim decoupled k_rope is
 *                              re-rotated; c_KV is reused byte for byte; both
 *                              channels are patched.
 *   kamera_slide_inplace       Sliding-window survival (technical summary
 *                              section 3.2): survivors relocate by rotation
 *                              only, no patch, in place in the pool.
 *
 * Reorder (section 3.1, one orbit patch for every ordering) and recall
 * (section 3.3, rehydration of an evicted chunk) are batches of chunk
 * descriptors for kamera_relocate_patch: each chunk carries its own delta,
 * rank, factors and target slots.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Element type: bf16 (IEEE binary32 truncated to its top 16 bits) for all
 *    K/V rows and patch factors.  Arithmetic is fp32; every output element is
 *    rounded once to bf16, round-to-nearest-even.  A key row with delta == 0
 *    and rank == 0, a value row with rank == 0 and the MLA c_KV block with
 *    rank == 0 are copied bit for bit.
 *  - RoPE: pair i (i < rot_dim/2) of the rotary range turns by
 *    phi_i = delta * theta_i, theta_i = base^(-2i/rot_dim) (or the override
 *    table):  x_a' = x_a cos phi - x_b sin phi,  x_b' = x_b cos phi + x_a sin phi.
 *    ROTATE_HALF pairs (o+i, o+i+rot_dim/2); INTERLEAVED pairs (o+2i, o+2i+1),
 *    o = rot_offset.  delta > 0 moves a chunk later: RoPE(x, p + delta) =
 *    R(delta) RoPE(x, p).  The phase is formed and reduced modulo 2 pi in fp64.
 *  - The patch is added after the rotation, in the target frame, as the
 *    equation is printed.  A caller holding a canonical-frame patch passes
 *    R(delta) applied to the columns of V_m instead (R(delta)(K + U V^T) =
 *    R(delta) K + U (R(delta) V)^T).
 *  - Memory: every pointer in the structs below, and every pointer inside the
 *    chunk descriptors, is caller-owned device memory (except the RoPE
 *    override table, which is host memory read during the call).  The library
 *    allocates nothing, keeps no state between calls (apart from a cache of
 *    the device's answers to cluster-occupancy queries, per kernel and
 *    device), never synchronises, and is safe to call from several host
 *    threads.  Work is enqueued on `stream`
 *    (a cudaStream_t of the current device; NULL = legacy default stream).
 *  - Synchronous status: the return value (KAMERA_OK or a KAMERA_ERR_* code).
 *    On any error nothing is enqueued.  n_chunks == 0 or max_len == 0 is a
 *    successful no-op.
 *  - Asynchronous status: violations only visible on the device (a slot
 *    outside the pool, a source range outside the store, a malformed
 *    descriptor, a chunk longer than max_len or of higher rank than max_rank)
 *    OR a KAMERA_DEVERR_* bit into *d_err (device int32, may be NULL to
 *    ignore) and skip the offending row or chunk; nothing outside the
 *    targeted slots is ever written.  The caller clears *d_err.
 *  - Preconditions (undefined results when violated; kamera_validate_chunks
 *    checks them on a host copy): slots are distinct within one call; the
 *    store and the pool do not overlap.
 */
#ifndef KAMERA_H
#define KAMERA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st* */

#define KAMERA_ABI_VERSION 9

/* Limits of this library. */
#define KAMERA_MAX_RANK 128          /* largest patch rank m */
#define KAMERA_MAX_ROT_DIM 256       /* largest rotary width (128 frequencies) */
#define KAMERA_MAX_ROW_ELEMS 4096    /* largest head_dim (GQA) / row width (MLA) */
#define KAMERA_MAX_ABS_DELTA 2147483647LL /* |delta| bound (positions are int32) */

/* Synchronous status codes. */
enum {
    KAMERA_OK = 0,
    KAMERA_ERR_INVALID_ARGUMENT = 1, /* NULL pointer, negative count or size, bad stride */
    KAMERA_ERR_MISALIGNED = 2,       /* a base pointer or stride is not 16-byte aligned */
    KAMERA_ERR_UNSUPPORTED = 3,      /* a shape or RoPE layout the library does not handle */
    KAMERA_ERR_CUDA = 4              /* a CUDA launch or attribute call failed */
};

/* Bits OR-ed into *d_err by the device. */
enum {
    KAMERA_DEVERR_SLOT = 1,        /* a slot outside [0, num_slots): that row skipped */
    KAMERA_DEVERR_SOURCE = 2,      /* src_offset < 0 or src_offset + len > store rows: chunk skipped */
    KAMERA_DEVERR_DESCRIPTOR = 4,  /* len < 0, rank < 0, |delta| too large, a NULL or
                                      misaligned factor or slot map: chunk skipped */
    KAMERA_DEVERR_LEN = 8,         /* len > max_len: chunk skipped */
    KAMERA_DEVERR_RANK = 16,       /* rank > max_rank: chunk skipped */
    KAMERA_DEVERR_TIMEOUT = 32     /* an internal pipeline wait gave up: results incomplete
                                      (every wait of the tensor-core kernels is bounded by
                                      1 s; the environment variable KAMERA_WAIT_LIMIT_NS,
                                      read at each call, overrides the bound.  Test hooks:
                                      KAMERA_TEST_WITHHOLD_LOADS=1 makes the producers of
                                      the relocation and prefill attention kernels issue
                                      no tile loads, and for patch
                                      formation a bound of 0 gives up at its first wait;
                                      the kernels then give up early, drain their own
                                      copies and MMAs, free their tensor memory and
                                      return with this bit set) */
};

/* RoPE pairings. */
enum {
    KAMERA_ROPE_ROTATE_HALF = 0,   /* (o+i, o+i+r/2): Llama/Qwen/NeoX style */
    KAMERA_ROPE_INTERLEAVED = 1    /* (o+2i, o+2i+1): original / GPT-J style */
};

/*
 * One chunk of work (64 bytes; an array of these lives in device memory).
 *   src_offset        first canonical row of the chunk in the store (ignored by
 *                     kamera_slide_inplace)
 *   len               tokens in the chunk, 0 <= len <= max_len of the call
 *   rank              patch rank m, 0 <= m <= max_rank of the call (0 = no
 *                     patch; kamera_slide_inplace requires 0)
 *   delta             RoPE phase shift in positions (target - canonical)
 *   patch_ptrs        four bf16 factor arrays, all NULL iff rank == 0, each
 *                     16-byte aligned:
 *                       GQA/MHA: Uk [L][H][len][m], Vk [L][H][head_dim][m],
 *                                Uv [L][H][len][m], Vv [L][H][head_dim][m]
 *                       MLA:     Uc [L][len][m], Vc [L][kv_lora_rank][m],
 *                                Ur [L][len][m], Vr [L][rope_dim][m]
 *                     (row-major, m contiguous; a joint 576-wide MLA factor is
 *                     the same call with Uc == Ur)
 *   dst_slot_mapping  len int64 pool slots, token j -> slot (16-byte aligned)
 */
typedef struct KameraChunk {
    int64_t src_offset;
    int32_t len;
    int32_t rank;
    int64_t delta;
    const void* patch_ptrs[4];
    const int64_t* dst_slot_mapping;
} KameraChunk;

/*
 * RoPE layout inside each head (GQA/MHA) or of the k_rope block (MLA).
 *   base               theta_i = base^(-2i/rot_dim) (ignored with an override)
 *   rot_dim            rotated components (even; 0 = no rotation); a multiple
 *                      of 16 for ROTATE_HALF and of 8 for INTERLEAVED
 *   rot_offset         first rotated component (multiple of 8); for MLA it is
 *                      relative to the start of k_rope and rot_offset + rot_dim
 *                      <= rope_dim
 *   pairing            KAMERA_ROPE_ROTATE_HALF or KAMERA_ROPE_INTERLEAVED
 *   n_axes             0: every frequency turns by the chunk's delta.
 *                      1..3: multi-axis RoPE (time, height, width), each
 *                      frequency following one axis; frequency f of chunk c
 *                      turns by d_axis_delta[c*n_axes + freq_axis[f]]; the
 *                      descriptor's delta is then not used for the phases
 *                      (it is still range-checked), and a chunk whose axis
 *                      deltas are all 0 is copied, as delta = 0 is
 *   inv_freq_override  NULL, or a host array of rot_dim/2 fp64 frequencies
 *                      (e.g. a model's scaled table), read during the call
 *   freq_axis          n_axes > 0: a host array of rot_dim/2 axis indices in
 *                      [0, n_axes) (contiguous sections, e.g. 16/24/24 of 64
 *                      frequencies, or interleaved), read during the call;
 *                      NULL with n_axes = 0
 *   d_axis_delta       n_axes > 0: a device array of n_chunks*n_axes int64
 *                      position moves, 8-byte aligned, read by the kernels
 *                      (|value| <= KAMERA_MAX_ABS_DELTA, else the chunk is
 *                      skipped with KAMERA_DEVERR_DESCRIPTOR); NULL with
 *                      n_axes = 0
 */
typedef struct KameraRope {
    double base;
    int32_t rot_dim;
    int32_t rot_offset;
    int32_t pairing;
    int32_t n_axes;
    const double* inv_freq_override;
    const uint8_t* freq_axis;
    const int64_t* d_axis_delta;
} KameraRope;

/*
 * Paged GQA/MHA pool.  Element (l, s, h, i) of K lives at
 * k[l*layer_stride + s*slot_stride + h*head_dim + i] (strides in elements,
 * multiples of 8; slot_stride >= num_kv_heads*head_dim; layer_stride >=
 * num_slots*slot_stride).  Slot s = page*P + offset for page size P: the
 * library sees slots only.  head_dim is a multiple of 8.
 */
typedef struct KameraGqaPool {
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t reserved;
    void* k;
    void* v;
    int64_t num_slots;
    int64_t layer_stride;
    int64_t slot_stride;
} KameraGqaPool;

/* Canonical GQA/MHA store (same L, H, head_dim as the pool): element
 * (l, row, h, i) of K at k[l*layer_stride + row*row_stride + h*head_dim + i]. */
typedef struct KameraGqaStore {
    const void* k;
    const void* v;
    int64_t num_rows;
    int64_t layer_stride;
    int64_t row_stride;
} KameraGqaStore;

/* Pool for the in-place slide: the K half of a GQA pool (V is never touched).
 * MLA k_rope survival uses num_kv_heads = 1, head_dim = kv_lora + rope and a
 * rotary range at rot_offset = kv_lora. */
typedef struct KameraSlidePool {
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t reserved;
    void* k;
    int64_t num_slots;
    int64_t layer_stride;
    int64_t slot_stride;
} KameraSlidePool;

/*
 * Paged MLA pool: one row per (layer, slot) = c_KV (kv_lora_rank elements)
 * followed by k_rope (rope_dim elements); element (l, s, i) at
 * kv[l*layer_stride + s*slot_stride + i].  kv_lora_rank and rope_dim are
 * multiples of 16.
 */
typedef struct KameraMlaPool {
    int32_t num_layers;
    int32_t kv_lora_rank;
    int32_t rope_dim;
    int32_t reserved;
    void* kv;
    int64_t num_slots;
    int64_t layer_stride;
    int64_t slot_stride;
} KameraMlaPool;

/* Canonical MLA store: element (l, row, i) at kv[l*layer_stride + row*row_stride + i]. */
typedef struct KameraMlaStore {
    const void* kv;
    int64_t num_rows;
    int64_t layer_stride;
    int64_t row_stride;
} KameraMlaStore;

/*
 * GQA/MHA relocate + patch + paged scatter (reuse equation; recall and
 * reorder batches).  For every chunk c, layer l, head h, token j < len:
 *   K[l][slot_j][h] = bf16( R(delta_c) Kstore[l][src_c+j][h] + Uk[l][h][j] Vk[l][h]^T )
 *   V[l][slot_j][h] = bf16(            Vstore[l][src_c+j][h] + Uv[l][h][j] Vv[l][h]^T )
 *   pool, store, rope   host structs (read during the call)
 *   d_chunks            device array of n_chunks descriptors
 *   h_chunks            NULL, or a host copy of the same n_chunks descriptors,
 *                       read during the call.  It lets the library describe
 *                       each chunk's U factors to the tensor-memory-access
 *                       engine, which then moves the U tiles of chunks of rank
 *                       16, 32, 64 or 128 (the first 104 chunks of a call)
 *                       without the copy work of a warp.  Results are the same
 *                       with or without it.  The device checks each such chunk
 *                       against its device descriptor (rank, len and the two U
 *                       addresses): a chunk whose host copy differs takes the
 *                       copy path (the result follows d_chunks) and the call
 *                       ORs KAMERA_DEVERR_DESCRIPTOR into *d_err.
 *   max_len, max_rank   upper bounds of len and rank over the chunks (size the
 *                       launch; larger chunks are skipped with a d_err bit)
 *   d_err               device int32 or NULL
 * Returns KAMERA_OK or a KAMERA_ERR_* code (nothing enqueued on error).
 */
int kamera_relocate_patch(const KameraGqaPool* pool, const KameraGqaStore* store,
                          const KameraRope* rope, const KameraChunk* d_chunks,
                          const KameraChunk* h_chunks, int32_t n_chunks, int32_t max_len,
                          int32_t max_rank, int32_t* d_err, struct CUstream_st* stream);

/*
 * Sliding-window survival in place (technical summary section 3.2): for every
 * chunk c, layer l, head h, token j < len:
 *   K[l][slot_j][h] = bf16( R(delta_c) K[l][slot_j][h] )
 * src_offset is ignored and rank must be 0 (else KAMERA_DEVERR_DESCRIPTOR).
 * V is never read or written.
 */
int kamera_slide_inplace(const KameraSlidePool* pool, const KameraRope* rope,
                         const KameraChunk* d_chunks, int32_t n_chunks, int32_t max_len,
                         int32_t* d_err, struct CUstream_st* stream);

/*
 * MLA relocate + patch + paged scatter (section 2, MLA rule): for every chunk
 * c, layer l, token j < len, with row = c_KV | k_rope:
 *   c_KV'   = bf16( c_KV + Uc[l][j] Vc[l]^T )                (bit copy when rank == 0)
 *   k_rope' = bf16( R(delta_c) k_rope + Ur[l][j] Vr[l]^T )
 * rope->rot_offset/rot_dim are relative to k_rope (usually 0 / rope_dim).
 * Arguments as for kamera_relocate_patch (h_chunks: NULL or a host copy of
 * d_chunks, whose Uc and Ur tiles it lets the copy engine move).
 */
int kamera_mla_relocate_patch(const KameraMlaPool* pool, const KameraMlaStore* store,
                              const KameraRope* rope, const KameraChunk* d_chunks,
                              const KameraChunk* h_chunks, int32_t n_chunks, int32_t max_len,
                              int32_t max_rank, int32_t* d_err, struct CUstream_st* stream);

/* Canonical stores written by the ingest calls (layouts as KameraGqaStore and
 * KameraMlaStore, writable). */
typedef struct KameraGqaStoreOut {
    void* k;
    void* v;
    int64_t num_rows;
    int64_t layer_stride;
    int64_t row_stride;
} KameraGqaStoreOut;

typedef struct KameraMlaStoreOut {
    void* kv;
    int64_t num_rows;
    int64_t layer_stride;
    int64_t row_stride;
} KameraMlaStoreOut;

/*
 * Canonical ingest, the inverse of relocation (technical summary section 2,
 * "Canonical KV": a chunk's KV as if it had no antecedent and started at
 * position 0).  A chunk that sits in the live paged cache at positions
 * s_c..s_c+len-1 is gathered from its slots and turned to that frame:
 *   Kstore[l][row_c + j][h] = bf16( R(delta_c) K[l][slot_j][h] ),  delta_c = -s_c
 *   Vstore[l][row_c + j][h] = V[l][slot_j][h]                       (bit copy)
 * Descriptor fields: src_offset = row_c, the first store row written; len;
 * delta; rank must be 0 and patch_ptrs NULL (else KAMERA_DEVERR_DESCRIPTOR);
 * dst_slot_mapping = the pool slots READ (outside [0, num_slots):
 * KAMERA_DEVERR_SLOT, that row skipped); row_c + len beyond the store:
 * KAMERA_DEVERR_SOURCE.  Elements outside the rotary range are copied, and
 * delta == 0 copies every row bit for bit.  Store rows of different chunks
 * must not overlap, and pool and store must not overlap.
 *   pool, store, rope   host structs (read during the call); store is written
 *   d_chunks, n_chunks  device descriptors; max_len bounds len (larger: KAMERA_DEVERR_LEN)
 *   d_err               device int32 or NULL
 * Returns KAMERA_OK or a KAMERA_ERR_* code (nothing enqueued on error).
 */
int kamera_ingest_canonical(const KameraGqaPool* pool, const KameraGqaStoreOut* store,
                            const KameraRope* rope, const KameraChunk* d_chunks, int32_t n_chunks,
                            int32_t max_len, int32_t* d_err, struct CUstream_st* stream);

/*
 * MLA canonical ingest: row = c_KV | k_rope; c_KV is copied bit for bit and
 * k_rope turned by R(delta_c) (rope->rot_offset/rot_dim relative to k_rope, as
 * for kamera_mla_relocate_patch).  Arguments as for kamera_ingest_canonical.
 */
int kamera_mla_ingest_canonical(const KameraMlaPool* pool, const KameraMlaStoreOut* store,
                                const KameraRope* rope, const KameraChunk* d_chunks, int32_t n_chunks,
                                int32_t max_len, int32_t* d_err, struct CUstream_st* stream);

/*
 * Host-side check of a HOST copy of a descriptor array (dst_slot_mapping
 * pointers must point to host memory here; patch pointers are only tested
 * for NULL-ness and 16-byte alignment).  Checks every device-side condition
 * plus the preconditions: slots distinct across the whole array and in
 * [0, num_slots); source ranges inside [0, num_store_rows) (skipped when
 * num_store_rows < 0, as for the slide); len <= max_len; rank <= max_rank.
 * Returns KAMERA_OK, or KAMERA_ERR_INVALID_ARGUMENT with *bad_chunk (if
 * non-NULL) set to the first offending chunk index and *bad_bits to the
 * KAMERA_DEVERR_* bits it would raise (KAMERA_DEVERR_SLOT also for a duplicate).
 */
int kamera_validate_chunks(const KameraChunk* h_chunks, int32_t n_chunks, int64_t num_store_rows,
                           int64_t num_slots, int32_t max_len, int32_t max_rank,
                           int32_t* bad_chunk, int32_t* bad_bits);

/* Static description of a status code (never NULL). */
const char* kamera_status_string(int status);

/*
 * One deficit tensor for kamera_form_patch: blocks (o, i), o < n_outer,
 * i < n_inner, each a rows x cols bf16 matrix (row-major, row_stride apart)
 * at x + o * outer_stride + i * inner_stride; with n_terms > 1 the block is
 * the mean of n_terms such matrices, term_stride apart (the orbit patch).
 * Strides in elements, multiples of 8; x 16-byte aligned.  A [L][len][H][d]
 * deficit is n_outer = L, n_inner = H, outer_stride = len*H*d,
 * inner_stride = d, row_stride = H*d.
 */
typedef struct KameraDeficit {
    const void* x;
    int64_t n_outer, n_inner;
    int64_t outer_stride, inner_stride, row_stride, term_stride;
    int32_t n_terms;
    int32_t rows, cols;
    int32_t reserved;   /* 0 */
} KameraDeficit;

/*
 * Patch formation, the one-time step before reuse (technical summary
 * section 2, "Rank-m Conditioning Patch": the patch is the top-m part of an
 * SVD of Delta = KV(B|A) - KV(B|empty); section 3.1: the orbit patch is the
 * same from the deficit averaged over orderings).  For every block X it
 * writes the best rank-m approximation U V^T of X (Eckart-Young):
 *     X = W diag(sigma) Z^T (sigma descending),  V = Z[:, :m],  U = X V = W[:, :m] diag(sigma[:m])
 * i.e. the singular values sit in U and V has orthonormal columns.  Method,
 * in fp32: Gram matrix X^T X, Householder tridiagonalisation, bisection for
 * the m largest eigenvalues, inverse iteration and Gram-Schmidt for their
 * eigenvectors, U = X V.  Each column's sign is the one the solve reaches
 * (singular vectors are unique up to sign, and within equal singular values
 * only their span is); directions whose squared singular value lies below
 * ~1e-6 of the largest are resolved as a span, not one by one.
 *   u      bf16 [n_outer*n_inner][rows][m] (written; block index o*n_inner + i:
 *          the Uk/Uv or Ur layout of KameraChunk for a [L][H] block grid)
 *   v      bf16 [n_outer*n_inner][cols][m] (written; the Vk/Vv or Vr layout)
 *   sigma  fp32 [n_outer*n_inner][m] singular values (written), or NULL
 * Supported: cols % 8 == 0 and 8 <= cols <= 128 with 1 <= m <= cols (head_dim
 * up to 128, MLA k_rope), or 128 < cols <= 576 with 1 <= m <= 32 (the MLA
 * c_KV block, or the whole 576-wide latent row c_KV | k_rope as one joint
 * block); rows >= 1, n_outer*n_inner < 2^31.  Blocks wider than 128
 * columns take subspace iteration on X^T X (three products of a basis of
 * k = min(48, m + 16 rounded up to 16) columns) and a Rayleigh-Ritz step:
 * exact to fp32 rounding when sigma_{k+1} is well below sigma_m (a deficit
 * whose energy sits in fewer than k directions), near-optimal otherwise; in
 * that case sigma holds the Ritz values ||X v_r|| of the returned directions
 * (what U = X V carries), which approach the singular values as the gap after
 * sigma_m grows and are exact only with such a gap.  u, v and sigma
 * must not overlap each other or the deficit.  Non-finite input gives
 * non-finite factors.  No block (n_outer, n_inner or rows 0) is a successful
 * no-op.  d_err: reserved for device-side errors (none is raised by this
 * entry point); may be NULL.
 */
int kamera_form_patch(const KameraDeficit* deficit, int32_t m, void* u, void* v, float* sigma,
                      int32_t* d_err, struct CUstream_st* stream);

/*
 * Decode attention over reused chunks, without the pool (the pages serve reused
 * chunks through a hook in the attention kernel: technical summary section 3,
 * "Production Deployment").  Each sequence s has one query token per query
 * head and attends, in one softmax, over the tokens of its chunks
 * d_chunks[d_seq_start[s] .. d_seq_start[s+1]-1]; the keys and values of a
 * chunk's token j are the reuse equation's rows, unrounded:
 *     K_j = R(delta) k_j + Uk[j] Vk^T,   V_j = v_j + Uv[j] Vv^T
 * (k_j, v_j: store row src_offset + j of this layer; factors as for
 * kamera_relocate_patch, read at `layer`).  out = softmax(scale q K^T) V per
 * query head; query head h reads KV head h / (num_q_heads / num_kv_heads).
 * The kernel turns the query by -delta once per chunk and folds the patch into
 * Vk^T q and Vv (sum_j p_j Uv[j]), so it reads only the store rows and the U
 * rows.  fp32 sums of bf16 products (hi + lo pairs for non-bf16 values), one
 * bf16 rounding of the output; a sequence with no token gets zeros.
 *   kv      the canonical store of ONE layer: k, v bf16 [num_rows][num_kv_heads]
 *           [head_dim], rows row_stride elements apart (16-byte aligned,
 *           row_stride a multiple of 8); layer = the factors' layer index
 *   query   q bf16 [n_seqs][num_q_heads][head_dim] (RoPE already applied at the
 *           query's position), out bf16 of the same shape (written), scale
 *   d_seq_start  device int32 [n_seqs + 1], non-decreasing, in [0, n_chunks]
 *   dst_slot_mapping of the descriptors is not read; ranks <= max_rank <= 64.
 * Supported: head_dim 64 or 128, num_q_heads / num_kv_heads in 1..8.
 *   d_workspace, workspace_bytes  NULL / 0, or device scratch of at least
 *           kamera_attend_workspace_bytes(n_seqs, num_kv_heads, head_dim) bytes,
 *           16-byte aligned, disjoint from the call's arrays; owned by the
 *           caller, overwritten by the call (calls that overlap on the GPU must
 *           not share one).  With it the call may spread every (sequence, KV
 *           head)'s tiles over all SMs, each CTA leaving a partial softmax
 *           state per unit it touches in the workspace, and merge them in a
 *           second launch on the same stream; without it the units' tiles are
 *           split only within clusters of at most 8 CTAs (the same results to
 *           fp32 rounding order).  A workspace that is too small, misaligned or
 *           overlapping: INVALID_ARGUMENT / MISALIGNED.
 * Device errors (the chunk is skipped): SOURCE, DESCRIPTOR (also a malformed
 * d_seq_start: the sequence is skipped), LEN, RANK; TIMEOUT if a tile's copy
 * wait runs past its bound (outputs of the call then undefined).  Host error
 * UNSUPPORTED also for num_rows > 2^31 - 1 (tile rows are addressed by 32-bit
 * coordinates).
 */
typedef struct KameraAttnKV {
    const void* k;
    const void* v;
    int64_t num_rows;
    int64_t row_stride;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t layer;
    int32_t reserved;   /* 0 */
} KameraAttnKV;

typedef struct KameraAttnQuery {
    const void* q;
    void* out;
    int32_t n_seqs;
    int32_t num_q_heads;
    float scale;
    int32_t reserved;   /* 0 */
} KameraAttnQuery;

int kamera_attend_reused(const KameraAttnKV* kv, const KameraAttnQuery* query, const KameraRope* rope,
                         const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                         int32_t max_len, int32_t max_rank, void* d_workspace, size_t workspace_bytes,
                         int32_t* d_err, struct CUstream_st* stream);

/* Workspace bytes kamera_attend_reused may use for this batch on the current
 * device ((SM count + n_seqs * num_kv_heads - 1) partial states of
 * 4 (32 + 16 head_dim) bytes); 0 for an unsupported head_dim or empty batch,
 * or when the device cannot be queried. */
size_t kamera_attend_workspace_bytes(int32_t n_seqs, int32_t num_kv_heads, int32_t head_dim);

/*
 * MLA decode attention over reused chunks (absorbed form), without the pool.
 * The rows of chunk c's token j are the MLA reuse rows, unrounded:
 *     c'_j  = c_j + Uc[j] Vc^T           (latent, kv_lora_rank wide)
 *     kr'_j = R(delta) kr_j + Ur[j] Vr^T  (k_rope, rope_dim wide)
 * (c_j | kr_j: store row src_offset + j; factors as for
 * kamera_mla_relocate_patch, read at `layer`).  Query head h of sequence s
 * holds q_lat (the no-position query taken through the key up-projection,
 * kv_lora_rank wide) then q_rope (rope_dim wide, RoPE applied at the query's
 * position); out_h = softmax_j(scale (q_lat . c'_j + q_rope . kr'_j)) c'_j, the
 * latent output the caller takes through the value up-projection.  All query
 * heads share the one latent row.  fp32 accumulation on bf16 operands (values
 * that are not bf16 enter as a hi + lo pair), one bf16 rounding of the output;
 * a sequence with no token gets zeros.
 *   kv      the canonical MLA store of ONE layer: bf16 [num_rows][kv_lora_rank +
 *           rope_dim], rows row_stride elements apart (16-byte aligned, row_stride
 *           a multiple of 8); layer = the factors' layer index
 *   query   q bf16 [n_seqs][num_q_heads][kv_lora_rank + rope_dim], out bf16
 *           [n_seqs][num_q_heads][kv_lora_rank] (written), scale; q and out
 *           16-byte aligned
 *   rope    rot_offset / rot_dim relative to k_rope
 *   d_seq_start, descriptors: as for kamera_attend_reused; ranks even.
 * Supported: kv_lora_rank 512, rope_dim 64 (DeepSeek-V2/V3), num_q_heads 1..128
 * (served in groups of 16: each group beyond the first is one more pass over the
 * rows), max_rank <= 32.  d_workspace, workspace_bytes: as for
 * kamera_attend_reused, sized by kamera_mla_attend_workspace_bytes (the units
 * are (sequence, group of 16 query heads)).  Device errors (the chunk is
 * skipped): SOURCE, DESCRIPTOR (also an odd rank, or a malformed d_seq_start:
 * the sequence is skipped), LEN, RANK; TIMEOUT as for kamera_attend_reused.
 * Host error UNSUPPORTED also for num_rows > 2^31 - 1.
 */
typedef struct KameraAttnMlaKV {
    const void* kv;
    int64_t num_rows;
    int64_t row_stride;
    int32_t kv_lora_rank;
    int32_t rope_dim;
    int32_t layer;
    int32_t reserved;   /* 0 */
} KameraAttnMlaKV;

int kamera_mla_attend_reused(const KameraAttnMlaKV* kv, const KameraAttnQuery* query, const KameraRope* rope,
                             const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                             int32_t max_len, int32_t max_rank, void* d_workspace, size_t workspace_bytes,
                             int32_t* d_err, struct CUstream_st* stream);

/* Workspace bytes kamera_mla_attend_reused may use for this batch on the
 * current device ((SM count + n_seqs * ceil(num_q_heads / 16) - 1) partial
 * states of 4 (32 + 16 * 512) bytes); 0 for an empty batch or when the device
 * cannot be queried. */
size_t kamera_mla_attend_workspace_bytes(int32_t n_seqs, int32_t num_q_heads);

/*
 * Prefill attention over reused chunks, without the pool (technical summary
 * section 3, "Production Deployment": the attention-kernel hook; the rows are
 * section 2's reuse equation).  Each sequence s brings q_tokens new query
 * tokens; every one of them attends, in one softmax and with no mask, over the
 * tokens of the sequence's chunks d_chunks[d_seq_start[s] .. d_seq_start[s+1]-1]
 * (they precede the new tokens), whose keys and values are, unrounded,
 *     K_j = R(delta) k_j + Uk[j] Vk^T,   V_j = v_j + Uv[j] Vv^T
 * as for kamera_attend_reused.  out = softmax(scale q K^T) V per query token
 * and head, and lse = log sum_j exp(scale q . K_j) (natural log), so a caller
 * merges this softmax with the one over the new tokens themselves:
 * out = (e^lse1 out1 + e^lse2 out2) / (e^lse1 + e^lse2).  fp32 accumulation of
 * bf16 products on the tensor cores (hi + lo bf16 pairs for the turned query,
 * V_k^T q and the softmax weights), one bf16 rounding of the output; a
 * sequence with no token gets zeros and lse = -infinity.
 *   kv      as for kamera_attend_reused (one layer's canonical store, layer =
 *           the factors' layer index)
 *   query   q bf16 [n_seqs][q_tokens][num_q_heads][head_dim] (RoPE already
 *           applied at each token's position, 16-byte aligned), out bf16 of the
 *           same shape (written, 16-byte aligned), lse float
 *           [n_seqs][q_tokens][num_q_heads] (written) or NULL, scale
 *   d_seq_start, descriptors: as for kamera_attend_reused.
 * Supported: head_dim 64 or 128, num_q_heads a multiple of num_kv_heads,
 * ranks <= max_rank <= 64.  Device errors (the chunk is skipped): SOURCE,
 * DESCRIPTOR (also a malformed d_seq_start: the sequence is skipped), LEN,
 * RANK; TIMEOUT if a pipeline wait runs past its bound (outputs of the call
 * then undefined).  Host errors: INVALID_ARGUMENT (also out overlapping q, the
 * store or lse), MISALIGNED, UNSUPPORTED (also num_rows > 2^31 - 1 or more
 * than 2^31 - 1 blocks of 128 query rows).
 */
typedef struct KameraPrefillQuery {
    const void* q;
    void* out;
    float* lse;
    int32_t n_seqs;
    int32_t q_tokens;
    int32_t num_q_heads;
    float scale;
} KameraPrefillQuery;

int kamera_prefill_attend_reused(const KameraAttnKV* kv, const KameraPrefillQuery* query, const KameraRope* rope,
                                 const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                                 int32_t max_len, int32_t max_rank, int32_t* d_err, struct CUstream_st* stream);

/*
 * kamera_attend_reused for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is an interface of this library only.
 * A plug-in whose host process gives all device memory to its own caching
 * allocator (with no hook to borrow from it), or a serving loop that must not
 * call cudaMalloc once it runs (the call can synchronise the device), has no
 * workspace to pass.  This entry point takes the same arguments as
 * kamera_attend_reused without d_workspace / workspace_bytes, and uses as the
 * workspace a fixed 4 MiB scratch array that the library keeps in device
 * memory on every GPU that loads it, for the life of the process; it calls no
 * allocating routine.  The caller still provides every input and the output.
 *   - Limit: the batch must fit the scratch, kamera_attend_workspace_bytes(
 *     n_seqs, num_kv_heads, head_dim) <= 4 MiB (for head_dim 128 on a 148-SM
 *     GB300: n_seqs * num_kv_heads <= 357); a larger batch returns
 *     KAMERA_ERR_UNSUPPORTED and nothing is launched.
 *   - The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call on a device shares the one scratch and leaves its partial
 *     states in it; nothing in it has to start at zero (each call writes every
 *     slot it reads), but calls that can overlap on the GPU (on different
 *     streams without an ordering between them) race on it.
 * Other arguments, results and errors: as for kamera_attend_reused.
 */
int kamera_attend_reused_static(const KameraAttnKV* kv, const KameraAttnQuery* query, const KameraRope* rope,
                                const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                                int32_t max_len, int32_t max_rank, int32_t* d_err, struct CUstream_st* stream);

/* KAMERA_ABI_VERSION of the loaded library. */
int kamera_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KAMERA_H */
