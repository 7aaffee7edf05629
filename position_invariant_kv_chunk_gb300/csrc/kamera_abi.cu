// kamera_abi.cu -- host side of the Kamera C ABI (include/kamera.h):
// argument validation, RoPE frequency tables, kernel selection and launch.
//
// Nothing here allocates device memory or synchronises; every error is
// reported before anything is enqueued.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <utility>
#include <vector>

#include "kamera.h"
#include "kamera_common.cuh"
#include "kamera_internal.h"

using namespace kamera;

namespace kamera {

uint64_t wait_limit_ns()
{
    const char* v = std::getenv("KAMERA_WAIT_LIMIT_NS");
    if (!v || !*v)
        return 1000000000ull;
    char* end = nullptr;
    const unsigned long long n = std::strtoull(v, &end, 10);
    return (end && *end == '\0') ? (uint64_t)n : 1000000000ull;
}

bool test_withhold_loads()
{
    const char* v = std::getenv("KAMERA_TEST_WITHHOLD_LOADS");
    return v && v[0] == '1' && v[1] == '\0';
}

int cluster_fit(const void* kernel, int block_threads, int smem_bytes, int cl)
{
    struct Entry {
        const void* kernel;
        int dev, block, bytes, cl, fit;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    {
        std::lock_guard<std::mutex> g(mu);
        for (const Entry& e : cache)
            if (e.kernel == kernel && e.dev == dev && e.block == block_threads && e.bytes == smem_bytes && e.cl == cl)
                return e.fit;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cl);
    cfg.blockDim = dim3((unsigned)block_threads);
    cfg.dynamicSmemBytes = (size_t)smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int fit = 0;
    if (cudaOccupancyMaxActiveClusters(&fit, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;   // not cached: a later call asks again
    }
    std::lock_guard<std::mutex> g(mu);
    cache.push_back(Entry{kernel, dev, block_threads, smem_bytes, cl, fit});
    return fit;
}

}  // namespace kamera

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte range [lo, hi) spanned by a strided [L][rows][width] bf16 array.
std::pair<uintptr_t, uintptr_t> span(const void* base, int64_t L, int64_t ls, int64_t rows, int64_t rs,
                                     int64_t width)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(base);
    if (L <= 0 || rows <= 0)
        return {lo, lo};
    const int64_t last = (L - 1) * ls + (rows - 1) * rs + width;
    return {lo, lo + static_cast<uintptr_t>(last) * 2u};
}

bool overlap(std::pair<uintptr_t, uintptr_t> a, std::pair<uintptr_t, uintptr_t> b)
{
    return a.first < b.second && b.first < a.second;
}

// RoPE: theta_i = base^(-2i/rot_dim) (standard rotary frequencies) or the
// caller's table.  `width` is the extent the rotary range must fit in.
int fill_rope(const KameraRope* r, int width, RopeParams* out)
{
    if (!r || r->n_axes < 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (r->n_axes > 3)
        return KAMERA_ERR_UNSUPPORTED;
    if (r->n_axes == 0 ? (r->freq_axis || r->d_axis_delta)
                       : (!r->freq_axis || !r->d_axis_delta || (reinterpret_cast<uintptr_t>(r->d_axis_delta) & 7)))
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (r->rot_dim < 0 || (r->rot_dim & 1) || r->rot_offset < 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (r->rot_dim > KAMERA_MAX_ROT_DIM)
        return KAMERA_ERR_UNSUPPORTED;
    if ((int64_t)r->rot_offset + r->rot_dim > width)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (r->pairing != KAMERA_ROPE_ROTATE_HALF && r->pairing != KAMERA_ROPE_INTERLEAVED)
        return KAMERA_ERR_UNSUPPORTED;
    if (r->rot_dim > 0) {
        if (r->pairing == KAMERA_ROPE_ROTATE_HALF && (r->rot_dim % 16))
            return KAMERA_ERR_UNSUPPORTED;
        if (r->pairing == KAMERA_ROPE_INTERLEAVED && (r->rot_dim % 8))
            return KAMERA_ERR_UNSUPPORTED;
        if (r->rot_offset % 8)
            return KAMERA_ERR_UNSUPPORTED;
    }
    std::memset(out, 0, sizeof(*out));
    out->rot_dim = r->rot_dim;
    out->rot_offset = r->rot_offset;
    out->pairing = r->pairing;
    out->n_freq = r->rot_dim / 2;
    for (int i = 0; i < out->n_freq; ++i) {
        double t;
        if (r->inv_freq_override) {
            t = r->inv_freq_override[i];
        } else {
            if (!(r->base > 0.0) || !std::isfinite(r->base))
                return KAMERA_ERR_INVALID_ARGUMENT;
            t = std::pow(r->base, -2.0 * (double)i / (double)r->rot_dim);
        }
        if (!std::isfinite(t))
            return KAMERA_ERR_INVALID_ARGUMENT;
        out->inv_freq[i] = t;
        if (r->n_axes > 0) {
            if (r->freq_axis[i] >= r->n_axes)
                return KAMERA_ERR_INVALID_ARGUMENT;
            out->axis[i] = r->freq_axis[i];
        }
    }
    out->n_axes = r->n_axes;
    out->axis_delta = r->d_axis_delta;
    return KAMERA_OK;
}

int check_call(const KameraChunk* d_chunks, int32_t n_chunks, int32_t max_len, int32_t max_rank,
               bool* noop)
{
    *noop = false;
    if (n_chunks < 0 || max_len < 0 || max_rank < 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (max_rank > KAMERA_MAX_RANK)
        return KAMERA_ERR_UNSUPPORTED;
    if (n_chunks == 0 || max_len == 0) {
        *noop = true;
        return KAMERA_OK;
    }
    if (!d_chunks)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(d_chunks) & 7u)
        return KAMERA_ERR_MISALIGNED;
    return KAMERA_OK;
}

int check_strided(const void* base, int64_t L, int64_t ls, int64_t rows, int64_t rs, int64_t width,
                  bool need_rows)
{
    if (!base)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (!aligned16(base) || (ls & 7) || (rs & 7))
        return KAMERA_ERR_MISALIGNED;
    if (rows < 0 || (need_rows && rows < 1) || rs < width || ls < 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (L > 1 && ls < rows * rs)
        return KAMERA_ERR_INVALID_ARGUMENT;
    return KAMERA_OK;
}

// Kernel choice: the tensor-core path whenever the call carries patches and
// its shape fits (head_dim 64/128, whole-head rotary; MLA c_KV in 128-blocks
// and a 64/128 k_rope), except for short chunks with tiny ranks; the slide
// kernel for the in-place rotation when its rotary units tile a block; the
// CUDA-core path otherwise.  Chunks of at most 128 tokens with ranks <= 8 go to
// the CUDA-core path: its independent CTAs (8 FMAs an element for the patch)
// beat the tensor-core pipeline, whose fixed cost per tile dominates one-tile
// jobs (4096 chunks of 128 tokens, rank 4: 244 against 428 us; rank 8: 333
// against 354 us; rank 16, or rank 8 on 1296-token chunks, favours the tensor
// cores).  KAMERA_PATH=simt in the environment pins the CUDA-core path,
// KAMERA_PATH=umma the tensor-core path wherever it applies (testing both on
// one input).
int launch(const RowsParams& p, int family, const KameraChunk* h_chunks, cudaStream_t stream)
{
    const char* force = std::getenv("KAMERA_PATH");
    const bool want_simt = force && std::strcmp(force, "simt") == 0;
    const bool want_umma = force && std::strcmp(force, "umma") == 0;
    const bool tc_ok = family != FAMILY_SLIDE && umma_supported(p, family) && umma_smem_bytes(p) <= 227u * 1024u;
    const int64_t tiles = (p.max_len + 63) / 64;
    const bool simt_ok = simt_smem_bytes(p, family, 64) <= 227u * 1024u &&
                         (int64_t)p.n_chunks * tiles <= 0x7FFFFFFFll && p.L <= 65535;
    const bool short_small = p.max_rank <= 8 && p.max_len <= 128;
    const bool use_tc = !want_simt && tc_ok && (want_umma || !(short_small && simt_ok));
    if (use_tc)
        return launch_umma(p, family, h_chunks, stream) == cudaSuccess ? KAMERA_OK : KAMERA_ERR_CUDA;
    if (!want_simt && family == FAMILY_SLIDE && p.L <= 65535 && slide_supported(p))
        return launch_slide(p, stream) == cudaSuccess ? KAMERA_OK : KAMERA_ERR_CUDA;
    if (!simt_ok)
        return KAMERA_ERR_UNSUPPORTED;
    return launch_simt(p, family, stream) == cudaSuccess ? KAMERA_OK : KAMERA_ERR_CUDA;
}

// Workspace of the attention split path on the current device: one slot per
// (CTA, unit) pair the split can make, CTAs resident at once (<= the SM count)
// + units - 1, of attend_slot_bytes(dout) each; 0 if the device is unknown.
size_t attend_workspace_for(int64_t units, int dout)
{
    int dev = 0, sms = 0;
    if (units < 1 || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return 0;
    return (size_t)(sms + units - 1) * attend_slot_bytes(dout);
}

// The caller's workspace: NULL (the cluster path) or 16-byte aligned, at least
// `need` bytes, and disjoint from the call's arrays.
int check_workspace(const void* ws, size_t bytes, size_t need, std::initializer_list<std::pair<uintptr_t, uintptr_t>> arrays)
{
    if (!ws)
        return KAMERA_OK;
    if (!aligned16(ws))
        return KAMERA_ERR_MISALIGNED;
    if (need == 0 || bytes < need)
        return KAMERA_ERR_INVALID_ARGUMENT;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ws);
    for (const auto& a : arrays)
        if (overlap({lo, lo + bytes}, a))
            return KAMERA_ERR_INVALID_ARGUMENT;
    return KAMERA_OK;
}

}  // namespace

extern "C" {

int kamera_abi_version(void) { return KAMERA_ABI_VERSION; }

const char* kamera_status_string(int status)
{
    switch (status) {
    case KAMERA_OK: return "ok";
    case KAMERA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KAMERA_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case KAMERA_ERR_UNSUPPORTED: return "shape or RoPE layout not supported by this library";
    case KAMERA_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
    }
}

int kamera_relocate_patch(const KameraGqaPool* pool, const KameraGqaStore* store, const KameraRope* rope,
                          const KameraChunk* d_chunks, const KameraChunk* h_chunks, int32_t n_chunks,
                          int32_t max_len, int32_t max_rank, int32_t* d_err, struct CUstream_st* stream)
{
    if (!pool || !store || !rope)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (pool->num_layers < 1 || pool->num_kv_heads < 1 || pool->head_dim < 8 || pool->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if ((pool->head_dim % 8) || pool->head_dim > KAMERA_MAX_ROW_ELEMS)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t L = pool->num_layers, W = (int64_t)pool->num_kv_heads * pool->head_dim;
    int rc;
    if ((rc = check_strided(pool->k, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    if ((rc = check_strided(pool->v, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    if ((rc = check_strided(store->k, L, store->layer_stride, store->num_rows, store->row_stride, W, false)))
        return rc;
    if ((rc = check_strided(store->v, L, store->layer_stride, store->num_rows, store->row_stride, W, false)))
        return rc;
    const auto pk = span(pool->k, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W);
    const auto pv = span(pool->v, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W);
    const auto sk = span(store->k, L, store->layer_stride, store->num_rows, store->row_stride, W);
    const auto sv = span(store->v, L, store->layer_stride, store->num_rows, store->row_stride, W);
    if (overlap(pk, pv) || overlap(pk, sk) || overlap(pk, sv) || overlap(pv, sk) || overlap(pv, sv))
        return KAMERA_ERR_INVALID_ARGUMENT;
    bool noop;
    if ((rc = check_call(d_chunks, n_chunks, max_len, max_rank, &noop)) || noop)
        return rc;
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, pool->head_dim, &p.rope)))
        return rc;
    p.dst_k = static_cast<__nv_bfloat16*>(pool->k);
    p.dst_v = static_cast<__nv_bfloat16*>(pool->v);
    p.num_slots = pool->num_slots;
    p.dst_ls = pool->layer_stride;
    p.dst_ss = pool->slot_stride;
    p.src_k = static_cast<const __nv_bfloat16*>(store->k);
    p.src_v = static_cast<const __nv_bfloat16*>(store->v);
    p.num_rows = store->num_rows;
    p.src_ls = store->layer_stride;
    p.src_rs = store->row_stride;
    p.L = pool->num_layers;
    p.H = pool->num_kv_heads;
    p.d = pool->head_dim;
    p.kv_lora = 0;
    p.chunks = d_chunks;
    p.n_chunks = n_chunks;
    p.max_len = max_len;
    p.max_rank = max_rank;
    p.err = d_err;
    return launch(p, FAMILY_GQA, h_chunks, reinterpret_cast<cudaStream_t>(stream));
}

int kamera_slide_inplace(const KameraSlidePool* pool, const KameraRope* rope, const KameraChunk* d_chunks,
                         int32_t n_chunks, int32_t max_len, int32_t* d_err, struct CUstream_st* stream)
{
    if (!pool || !rope)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (pool->num_layers < 1 || pool->num_kv_heads < 1 || pool->head_dim < 8 || pool->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if ((pool->head_dim % 8) || pool->head_dim > KAMERA_MAX_ROW_ELEMS)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t L = pool->num_layers, W = (int64_t)pool->num_kv_heads * pool->head_dim;
    int rc;
    if ((rc = check_strided(pool->k, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    bool noop;
    if ((rc = check_call(d_chunks, n_chunks, max_len, 0, &noop)) || noop)
        return rc;
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, pool->head_dim, &p.rope)))
        return rc;
    p.dst_k = static_cast<__nv_bfloat16*>(pool->k);
    p.num_slots = pool->num_slots;
    p.dst_ls = pool->layer_stride;
    p.dst_ss = pool->slot_stride;
    p.L = pool->num_layers;
    p.H = pool->num_kv_heads;
    p.d = pool->head_dim;
    p.chunks = d_chunks;
    p.n_chunks = n_chunks;
    p.max_len = max_len;
    p.max_rank = 0;
    p.err = d_err;
    return launch(p, FAMILY_SLIDE, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int kamera_mla_relocate_patch(const KameraMlaPool* pool, const KameraMlaStore* store, const KameraRope* rope,
                              const KameraChunk* d_chunks, const KameraChunk* h_chunks, int32_t n_chunks,
                              int32_t max_len, int32_t max_rank, int32_t* d_err, struct CUstream_st* stream)
{
    if (!pool || !store || !rope)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (pool->num_layers < 1 || pool->kv_lora_rank < 0 || pool->rope_dim < 0 || pool->reserved != 0 ||
        pool->kv_lora_rank + pool->rope_dim < 16)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if ((pool->kv_lora_rank % 16) || (pool->rope_dim % 16) ||
        pool->kv_lora_rank + pool->rope_dim > KAMERA_MAX_ROW_ELEMS || pool->rope_dim > KAMERA_MAX_ROT_DIM)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t L = pool->num_layers, W = (int64_t)pool->kv_lora_rank + pool->rope_dim;
    int rc;
    if ((rc = check_strided(pool->kv, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    if ((rc = check_strided(store->kv, L, store->layer_stride, store->num_rows, store->row_stride, W, false)))
        return rc;
    if (overlap(span(pool->kv, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W),
                span(store->kv, L, store->layer_stride, store->num_rows, store->row_stride, W)))
        return KAMERA_ERR_INVALID_ARGUMENT;
    bool noop;
    if ((rc = check_call(d_chunks, n_chunks, max_len, max_rank, &noop)) || noop)
        return rc;
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, pool->rope_dim, &p.rope)))
        return rc;
    p.dst_k = static_cast<__nv_bfloat16*>(pool->kv);
    p.num_slots = pool->num_slots;
    p.dst_ls = pool->layer_stride;
    p.dst_ss = pool->slot_stride;
    p.src_k = static_cast<const __nv_bfloat16*>(store->kv);
    p.num_rows = store->num_rows;
    p.src_ls = store->layer_stride;
    p.src_rs = store->row_stride;
    p.L = pool->num_layers;
    p.H = 1;
    p.d = (int32_t)W;
    p.kv_lora = pool->kv_lora_rank;
    p.chunks = d_chunks;
    p.n_chunks = n_chunks;
    p.max_len = max_len;
    p.max_rank = max_rank;
    p.err = d_err;
    return launch(p, FAMILY_MLA, h_chunks, reinterpret_cast<cudaStream_t>(stream));
}

static int ingest_launch(const RowsParams& rp, bool values, const void* pk, const void* pv, void* sk, void* sv,
                         int64_t src_ls, int64_t src_ss, int64_t num_rows, int64_t dst_ls, int64_t dst_rs,
                         cudaStream_t stream)
{
    IngestParams ip;
    std::memset(&ip, 0, sizeof(ip));
    const int np = ingest_passes(rp, values, ip.pass);
    if (np <= 0)
        return KAMERA_ERR_UNSUPPORTED;
    ip.n_pass = np;
    ip.src[0] = static_cast<const __nv_bfloat16*>(pk);
    ip.src[1] = static_cast<const __nv_bfloat16*>(pv);
    ip.dst[0] = static_cast<__nv_bfloat16*>(sk);
    ip.dst[1] = static_cast<__nv_bfloat16*>(sv);
    ip.src_ls = src_ls;
    ip.src_ss = src_ss;
    ip.dst_ls = dst_ls;
    ip.dst_rs = dst_rs;
    ip.num_slots = rp.num_slots;
    ip.num_rows = num_rows;
    ip.L = rp.L;
    ip.H = rp.H;
    ip.d = rp.d;
    ip.chunks = rp.chunks;
    ip.n_chunks = rp.n_chunks;
    ip.max_len = rp.max_len;
    ip.err = rp.err;
    ip.rope = rp.rope;
    const int64_t tiles = (rp.max_len + 127) / 128;
    if ((int64_t)rp.n_chunks * tiles > 0x7FFFFFFFll || rp.L > 65535)
        return KAMERA_ERR_UNSUPPORTED;
    return launch_ingest(ip, stream) == cudaSuccess ? KAMERA_OK : KAMERA_ERR_CUDA;
}

int kamera_ingest_canonical(const KameraGqaPool* pool, const KameraGqaStoreOut* store, const KameraRope* rope,
                            const KameraChunk* d_chunks, int32_t n_chunks, int32_t max_len, int32_t* d_err,
                            struct CUstream_st* stream)
{
    if (!pool || !store || !rope)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (pool->num_layers < 1 || pool->num_kv_heads < 1 || pool->head_dim < 8 || pool->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if ((pool->head_dim % 8) || pool->head_dim > KAMERA_MAX_ROW_ELEMS)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t L = pool->num_layers, W = (int64_t)pool->num_kv_heads * pool->head_dim;
    int rc;
    if ((rc = check_strided(pool->k, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    if ((rc = check_strided(pool->v, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    if ((rc = check_strided(store->k, L, store->layer_stride, store->num_rows, store->row_stride, W, false)))
        return rc;
    if ((rc = check_strided(store->v, L, store->layer_stride, store->num_rows, store->row_stride, W, false)))
        return rc;
    const auto pk = span(pool->k, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W);
    const auto pv = span(pool->v, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W);
    const auto sk = span(store->k, L, store->layer_stride, store->num_rows, store->row_stride, W);
    const auto sv = span(store->v, L, store->layer_stride, store->num_rows, store->row_stride, W);
    if (overlap(sk, sv) || overlap(pk, sk) || overlap(pk, sv) || overlap(pv, sk) || overlap(pv, sv))
        return KAMERA_ERR_INVALID_ARGUMENT;
    bool noop;
    if ((rc = check_call(d_chunks, n_chunks, max_len, 0, &noop)) || noop)
        return rc;
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, pool->head_dim, &p.rope)))
        return rc;
    p.num_slots = pool->num_slots;
    p.L = pool->num_layers;
    p.H = pool->num_kv_heads;
    p.d = pool->head_dim;
    p.chunks = d_chunks;
    p.n_chunks = n_chunks;
    p.max_len = max_len;
    p.err = d_err;
    return ingest_launch(p, true, pool->k, pool->v, store->k, store->v, pool->layer_stride, pool->slot_stride,
                         store->num_rows, store->layer_stride, store->row_stride,
                         reinterpret_cast<cudaStream_t>(stream));
}

int kamera_mla_ingest_canonical(const KameraMlaPool* pool, const KameraMlaStoreOut* store, const KameraRope* rope,
                                const KameraChunk* d_chunks, int32_t n_chunks, int32_t max_len, int32_t* d_err,
                                struct CUstream_st* stream)
{
    if (!pool || !store || !rope)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (pool->num_layers < 1 || pool->kv_lora_rank < 0 || pool->rope_dim < 0 || pool->reserved != 0 ||
        pool->kv_lora_rank + pool->rope_dim < 16)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if ((pool->kv_lora_rank % 16) || (pool->rope_dim % 16) ||
        pool->kv_lora_rank + pool->rope_dim > KAMERA_MAX_ROW_ELEMS || pool->rope_dim > KAMERA_MAX_ROT_DIM)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t L = pool->num_layers, W = (int64_t)pool->kv_lora_rank + pool->rope_dim;
    int rc;
    if ((rc = check_strided(pool->kv, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W, true)))
        return rc;
    if ((rc = check_strided(store->kv, L, store->layer_stride, store->num_rows, store->row_stride, W, false)))
        return rc;
    if (overlap(span(pool->kv, L, pool->layer_stride, pool->num_slots, pool->slot_stride, W),
                span(store->kv, L, store->layer_stride, store->num_rows, store->row_stride, W)))
        return KAMERA_ERR_INVALID_ARGUMENT;
    bool noop;
    if ((rc = check_call(d_chunks, n_chunks, max_len, 0, &noop)) || noop)
        return rc;
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, pool->rope_dim, &p.rope)))
        return rc;
    p.rope.rot_offset += pool->kv_lora_rank;   // relative to k_rope in the ABI, to the row here
    p.num_slots = pool->num_slots;
    p.L = pool->num_layers;
    p.H = 1;
    p.d = (int32_t)W;
    p.chunks = d_chunks;
    p.n_chunks = n_chunks;
    p.max_len = max_len;
    p.err = d_err;
    return ingest_launch(p, false, pool->kv, nullptr, store->kv, nullptr, pool->layer_stride, pool->slot_stride,
                         store->num_rows, store->layer_stride, store->row_stride,
                         reinterpret_cast<cudaStream_t>(stream));
}

int kamera_validate_chunks(const KameraChunk* h_chunks, int32_t n_chunks, int64_t num_store_rows, int64_t num_slots,
                           int32_t max_len, int32_t max_rank, int32_t* bad_chunk, int32_t* bad_bits)
{
    if (bad_chunk)
        *bad_chunk = -1;
    if (bad_bits)
        *bad_bits = 0;
    if (n_chunks < 0 || (n_chunks > 0 && !h_chunks))
        return KAMERA_ERR_INVALID_ARGUMENT;
    auto fail = [&](int32_t c, int32_t bits) {
        if (bad_chunk)
            *bad_chunk = c;
        if (bad_bits)
            *bad_bits = bits;
        return KAMERA_ERR_INVALID_ARGUMENT;
    };
    std::vector<std::pair<int64_t, int32_t>> all;
    for (int32_t c = 0; c < n_chunks; ++c) {
        const KameraChunk& ch = h_chunks[c];
        int32_t bits = 0;
        if (ch.len < 0 || ch.rank < 0 || ch.delta > KAMERA_MAX_ABS_DELTA || ch.delta < -KAMERA_MAX_ABS_DELTA)
            bits |= KAMERA_DEVERR_DESCRIPTOR;
        if (ch.len > 0 && (!ch.dst_slot_mapping || !aligned16(ch.dst_slot_mapping)))
            bits |= KAMERA_DEVERR_DESCRIPTOR;
        for (int i = 0; i < 4; ++i) {
            const bool null = ch.patch_ptrs[i] == nullptr;
            if ((ch.rank > 0 && (null || !aligned16(ch.patch_ptrs[i]))) || (ch.rank == 0 && !null))
                bits |= KAMERA_DEVERR_DESCRIPTOR;
        }
        if (num_store_rows >= 0 && (ch.src_offset < 0 || ch.src_offset + (int64_t)ch.len > num_store_rows))
            bits |= KAMERA_DEVERR_SOURCE;
        if (ch.len > max_len)
            bits |= KAMERA_DEVERR_LEN;
        if (ch.rank > max_rank)
            bits |= KAMERA_DEVERR_RANK;
        if (!bits && ch.len > 0) {
            for (int32_t j = 0; j < ch.len; ++j) {
                const int64_t s = ch.dst_slot_mapping[j];
                if (s < 0 || s >= num_slots) {
                    bits |= KAMERA_DEVERR_SLOT;
                    break;
                }
                all.emplace_back(s, c);
            }
        }
        if (bits)
            return fail(c, bits);
    }
    std::sort(all.begin(), all.end());
    for (size_t i = 1; i < all.size(); ++i)
        if (all[i].first == all[i - 1].first)
            return fail(std::max(all[i].second, all[i - 1].second), KAMERA_DEVERR_SLOT);
    return KAMERA_OK;
}


int kamera_form_patch(const KameraDeficit* df, int32_t m, void* u, void* v, float* sigma, int32_t* d_err,
                      struct CUstream_st* stream)
{
    if (!df || df->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (df->n_outer < 0 || df->n_inner < 0 || df->n_terms < 1 || df->rows < 0 || df->cols < 1 || m < 1)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (df->n_outer == 0 || df->n_inner == 0 || df->rows == 0)
        return KAMERA_OK;   // no block: nothing to form
    if (!df->x || !u || !v)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (df->outer_stride < 0 || df->inner_stride < 0 || df->row_stride < df->cols || df->term_stride < 0 ||
        (df->n_terms > 1 && df->term_stride == 0))
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (!patch_form_supported(df->cols, m))
        return KAMERA_ERR_UNSUPPORTED;
    if (!aligned16(df->x) || !aligned16(u) || !aligned16(v) || (sigma && !aligned16(sigma)) ||
        (df->outer_stride | df->inner_stride | df->row_stride | df->term_stride) % 8)
        return KAMERA_ERR_MISALIGNED;
    if (df->n_outer > 0 && df->n_inner > 0x7FFFFFFFll / df->n_outer)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t nb = df->n_outer * df->n_inner;
    const int64_t last = (df->n_outer - 1) * df->outer_stride + (df->n_inner - 1) * df->inner_stride +
                         (int64_t)(df->n_terms - 1) * df->term_stride + (int64_t)(df->rows - 1) * df->row_stride +
                         df->cols;
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(df->x);
    const std::pair<uintptr_t, uintptr_t> xs{x0, x0 + (uintptr_t)last * 2u};
    const uintptr_t u0 = reinterpret_cast<uintptr_t>(u), v0 = reinterpret_cast<uintptr_t>(v);
    const std::pair<uintptr_t, uintptr_t> us{u0, u0 + (uintptr_t)(nb * df->rows * m) * 2u};
    const std::pair<uintptr_t, uintptr_t> vs{v0, v0 + (uintptr_t)(nb * df->cols * m) * 2u};
    if (overlap(xs, us) || overlap(xs, vs) || overlap(us, vs))
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (sigma) {
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(sigma);
        const std::pair<uintptr_t, uintptr_t> ss{s0, s0 + (uintptr_t)(nb * m) * 4u};
        if (overlap(ss, xs) || overlap(ss, us) || overlap(ss, vs))
            return KAMERA_ERR_INVALID_ARGUMENT;
    }
    PatchFormParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = static_cast<const __nv_bfloat16*>(df->x);
    p.n_inner = df->n_inner;
    p.outer_stride = df->outer_stride;
    p.inner_stride = df->inner_stride;
    p.row_stride = df->row_stride;
    p.term_stride = df->term_stride;
    p.n_terms = df->n_terms;
    p.rows = df->rows;
    p.cols = df->cols;
    p.m = m;
    p.u = static_cast<__nv_bfloat16*>(u);
    p.v = static_cast<__nv_bfloat16*>(v);
    p.sigma = sigma;
    p.err = d_err;
    p.wait_ns = wait_limit_ns();
    return launch_patch_form(p, nb, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KAMERA_OK
                                                                                          : KAMERA_ERR_CUDA;
}

size_t kamera_attend_workspace_bytes(int32_t n_seqs, int32_t num_kv_heads, int32_t head_dim)
{
    if (n_seqs < 1 || num_kv_heads < 1 || (head_dim != 64 && head_dim != 128))
        return 0;
    return attend_workspace_for((int64_t)n_seqs * num_kv_heads, head_dim);
}

size_t kamera_mla_attend_workspace_bytes(int32_t n_seqs, int32_t num_q_heads)
{
    if (n_seqs < 1 || num_q_heads < 1)
        return 0;
    return attend_workspace_for((int64_t)n_seqs * ((num_q_heads + 15) / 16), 512);
}

int kamera_attend_reused(const KameraAttnKV* kv, const KameraAttnQuery* query, const KameraRope* rope,
                         const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                         int32_t max_len, int32_t max_rank, void* d_workspace, size_t workspace_bytes,
                         int32_t* d_err, struct CUstream_st* stream)
{
    if (!kv || !query || !rope || kv->reserved != 0 || query->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (query->n_seqs < 0 || n_chunks < 0 || max_len < 0 || max_rank < 0 || kv->num_rows < 0 || kv->layer < 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (kv->num_kv_heads < 1 || kv->head_dim < 8 || query->num_q_heads < 1 ||
        query->num_q_heads % kv->num_kv_heads != 0 || !(query->scale == query->scale))
        return KAMERA_ERR_INVALID_ARGUMENT;
    const int G = query->num_q_heads / kv->num_kv_heads;
    if (!attend_supported(kv->head_dim, G, max_rank) || kv->num_kv_heads > 65535 ||
        query->n_seqs > 0x7FFFFFFF || kv->num_rows > 0x7FFFFFFF)
        return KAMERA_ERR_UNSUPPORTED;
    if (query->n_seqs == 0)
        return KAMERA_OK;
    if (!kv->k || !kv->v || !query->q || !query->out || !d_seq_start || (n_chunks > 0 && !d_chunks))
        return KAMERA_ERR_INVALID_ARGUMENT;
    const int64_t W = (int64_t)kv->num_kv_heads * kv->head_dim;
    if (kv->row_stride < W)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (!aligned16(kv->k) || !aligned16(kv->v) || !aligned16(d_chunks) || kv->row_stride % 8)
        return KAMERA_ERR_MISALIGNED;
    const auto ks = span(kv->k, 1, 0, kv->num_rows, kv->row_stride, W);
    const auto vs = span(kv->v, 1, 0, kv->num_rows, kv->row_stride, W);
    const int64_t qn = (int64_t)query->n_seqs * query->num_q_heads * kv->head_dim;
    const auto os = span(query->out, 1, 0, 1, 0, qn);
    const auto qs = span(query->q, 1, 0, 1, 0, qn);
    if (overlap(os, ks) || overlap(os, vs) || overlap(os, qs))
        return KAMERA_ERR_INVALID_ARGUMENT;
    int rc = check_workspace(d_workspace, workspace_bytes,
                             attend_workspace_for((int64_t)query->n_seqs * kv->num_kv_heads, kv->head_dim),
                             {ks, vs, qs, os});
    if (rc)
        return rc;
    AttendParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, kv->head_dim, &p.rope)))
        return rc;
    p.k = static_cast<const __nv_bfloat16*>(kv->k);
    p.v = static_cast<const __nv_bfloat16*>(kv->v);
    p.row_stride = kv->row_stride;
    p.num_rows = kv->num_rows;
    p.H = kv->num_kv_heads;
    p.d = kv->head_dim;
    p.G = G;
    p.layer = kv->layer;
    p.chunks = d_chunks;
    p.seq_start = d_seq_start;
    p.n_seqs = query->n_seqs;
    p.n_chunks = n_chunks;
    p.q = static_cast<const __nv_bfloat16*>(query->q);
    p.out = static_cast<__nv_bfloat16*>(query->out);
    p.scale = query->scale;
    p.max_len = max_len;
    p.max_rank = max_rank;
    p.err = d_err;
    p.cluster = attend_cluster((int64_t)query->n_seqs * kv->num_kv_heads);   // the launch may pick up to 8
    if ((int64_t)query->n_seqs * 8 > 0x7FFFFFFF)
        return KAMERA_ERR_UNSUPPORTED;
    return launch_attend(p, d_workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KAMERA_OK
               : KAMERA_ERR_CUDA;
}

int kamera_prefill_attend_reused(const KameraAttnKV* kv, const KameraPrefillQuery* query, const KameraRope* rope,
                                 const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                                 int32_t max_len, int32_t max_rank, int32_t* d_err, struct CUstream_st* stream)
{
    if (!kv || !query || !rope || kv->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (query->n_seqs < 0 || query->q_tokens < 0 || n_chunks < 0 || max_len < 0 || max_rank < 0 ||
        kv->num_rows < 0 || kv->layer < 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (kv->num_kv_heads < 1 || kv->head_dim < 8 || query->num_q_heads < 1 ||
        query->num_q_heads % kv->num_kv_heads != 0 || !(query->scale == query->scale))
        return KAMERA_ERR_INVALID_ARGUMENT;
    const int G = query->num_q_heads / kv->num_kv_heads;
    if (!prefill_supported(kv->head_dim, max_rank) || kv->num_rows > 0x7FFFFFFF)
        return KAMERA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)query->q_tokens * G;   // query rows of one (sequence, KV head)
    const int64_t blocks = (rows + 127) / 128;
    if (rows > 0x7FFFFFFF || (int64_t)query->n_seqs * kv->num_kv_heads * blocks > 0x7FFFFFFF)
        return KAMERA_ERR_UNSUPPORTED;
    if (query->n_seqs == 0 || query->q_tokens == 0)
        return KAMERA_OK;
    if (!kv->k || !kv->v || !query->q || !query->out || !d_seq_start || (n_chunks > 0 && !d_chunks))
        return KAMERA_ERR_INVALID_ARGUMENT;
    const int64_t W = (int64_t)kv->num_kv_heads * kv->head_dim;
    if (kv->row_stride < W)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (!aligned16(kv->k) || !aligned16(kv->v) || !aligned16(d_chunks) || kv->row_stride % 8 ||
        !aligned16(query->q) || !aligned16(query->out) || (reinterpret_cast<uintptr_t>(query->lse) & 3))
        return KAMERA_ERR_MISALIGNED;
    const auto ks = span(kv->k, 1, 0, kv->num_rows, kv->row_stride, W);
    const auto vs = span(kv->v, 1, 0, kv->num_rows, kv->row_stride, W);
    const int64_t qn = (int64_t)query->n_seqs * query->q_tokens * query->num_q_heads;
    const auto os = span(query->out, 1, 0, 1, 0, qn * kv->head_dim);
    const auto qs = span(query->q, 1, 0, 1, 0, qn * kv->head_dim);
    if (overlap(os, ks) || overlap(os, vs) || overlap(os, qs))
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (query->lse) {
        const auto ls = span(query->lse, 1, 0, 1, 0, 2 * qn);   // fp32: two bf16 widths each
        if (overlap(ls, ks) || overlap(ls, vs) || overlap(ls, qs) || overlap(ls, os))
            return KAMERA_ERR_INVALID_ARGUMENT;
    }
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    int rc = fill_rope(rope, kv->head_dim, &p.rope);
    if (rc)
        return rc;
    p.k = static_cast<const __nv_bfloat16*>(kv->k);
    p.v = static_cast<const __nv_bfloat16*>(kv->v);
    p.row_stride = kv->row_stride;
    p.num_rows = kv->num_rows;
    p.H = kv->num_kv_heads;
    p.d = kv->head_dim;
    p.G = G;
    p.layer = kv->layer;
    p.chunks = d_chunks;
    p.seq_start = d_seq_start;
    p.n_seqs = query->n_seqs;
    p.n_chunks = n_chunks;
    p.T = query->q_tokens;
    p.blocks = (int32_t)blocks;
    p.q = static_cast<const __nv_bfloat16*>(query->q);
    p.out = static_cast<__nv_bfloat16*>(query->out);
    p.lse = query->lse;
    p.scale = query->scale;
    p.max_len = max_len;
    p.max_rank = max_rank;
    p.err = d_err;
    return launch_prefill(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KAMERA_OK : KAMERA_ERR_CUDA;
}

int kamera_mla_attend_reused(const KameraAttnMlaKV* kv, const KameraAttnQuery* query, const KameraRope* rope,
                             const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                             int32_t max_len, int32_t max_rank, void* d_workspace, size_t workspace_bytes,
                             int32_t* d_err, struct CUstream_st* stream)
{
    if (!kv || !query || !rope || kv->reserved != 0 || query->reserved != 0)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (query->n_seqs < 0 || n_chunks < 0 || max_len < 0 || max_rank < 0 || kv->num_rows < 0 || kv->layer < 0 ||
        kv->kv_lora_rank < 1 || kv->rope_dim < 0 || query->num_q_heads < 1 || !(query->scale == query->scale))
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (!mla_attend_supported(kv->kv_lora_rank, kv->rope_dim, query->num_q_heads, max_rank) ||
        query->n_seqs > 0x7FFFFFFF / 8 || kv->num_rows > 0x7FFFFFFF)
        return KAMERA_ERR_UNSUPPORTED;
    if (query->n_seqs == 0)
        return KAMERA_OK;
    if (!kv->kv || !query->q || !query->out || !d_seq_start || (n_chunks > 0 && !d_chunks))
        return KAMERA_ERR_INVALID_ARGUMENT;
    const int64_t W = (int64_t)kv->kv_lora_rank + kv->rope_dim;
    if (kv->row_stride < W)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (!aligned16(kv->kv) || !aligned16(d_chunks) || kv->row_stride % 8 || !aligned16(query->q) ||
        !aligned16(query->out))
        return KAMERA_ERR_MISALIGNED;
    const auto ks = span(kv->kv, 1, 0, kv->num_rows, kv->row_stride, W);
    const auto qs = span(query->q, 1, 0, 1, 0, (int64_t)query->n_seqs * query->num_q_heads * W);
    const auto os = span(query->out, 1, 0, 1, 0, (int64_t)query->n_seqs * query->num_q_heads * kv->kv_lora_rank);
    if (overlap(os, ks) || overlap(os, qs))
        return KAMERA_ERR_INVALID_ARGUMENT;
    int rc = check_workspace(
        d_workspace, workspace_bytes,
        attend_workspace_for((int64_t)query->n_seqs * ((query->num_q_heads + 15) / 16), kv->kv_lora_rank), {ks, qs, os});
    if (rc)
        return rc;
    MlaAttendParams p;
    std::memset(&p, 0, sizeof(p));
    if ((rc = fill_rope(rope, kv->rope_dim, &p.rope)))
        return rc;
    p.kv = static_cast<const __nv_bfloat16*>(kv->kv);
    p.row_stride = kv->row_stride;
    p.num_rows = kv->num_rows;
    p.kv_lora = kv->kv_lora_rank;
    p.rope_dim = kv->rope_dim;
    p.Hq = query->num_q_heads;
    p.layer = kv->layer;
    p.chunks = d_chunks;
    p.seq_start = d_seq_start;
    p.n_seqs = query->n_seqs;
    p.n_chunks = n_chunks;
    p.q = static_cast<const __nv_bfloat16*>(query->q);
    p.out = static_cast<__nv_bfloat16*>(query->out);
    p.scale = query->scale;
    p.max_len = max_len;
    p.max_rank = max_rank;
    p.err = d_err;
    return launch_mla_attend(p, d_workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KAMERA_OK
               : KAMERA_ERR_CUDA;
}

}  // extern "C"
