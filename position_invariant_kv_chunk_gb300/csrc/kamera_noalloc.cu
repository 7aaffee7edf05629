// kamera_noalloc.cu -- decode attention over reused chunks for callers that
// cannot allocate device memory.
//
// kamera_attend_reused spreads a small batch over every SM only when the
// caller hands it a workspace for the partial softmax states.  Some callers
// have no way to get one: a plug-in whose host process hands all device memory
// to its own caching allocator and offers no hook to borrow from it, or a
// serving loop that must not call cudaMalloc once it runs (cudaMalloc can
// synchronise the device and stall every stream).  For them this file keeps
// one fixed scratch array in the library's own device memory and passes it to
// the ordinary entry point as its workspace; the caller still passes its
// inputs and outputs.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "kamera.h"

namespace {

// The shared scratch: 4 MiB on every GPU that loads the library, held until
// the process exits.  With head_dim 128 a partial state takes 8320 bytes, so
// a call fits while (SM count + n_seqs * num_kv_heads - 1) <= 504.
constexpr size_t kScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_attend_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];   // device address of g_attend_scratch, per device (set once)

// The scratch array's device address on the current device, looked up on the
// first call that runs on that device.  NULL if the lookup fails.
void* scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attend_scratch) != cudaSuccess)
            return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

int kamera_attend_reused_static(const KameraAttnKV* kv, const KameraAttnQuery* query, const KameraRope* rope,
                                const KameraChunk* d_chunks, const int32_t* d_seq_start, int32_t n_chunks,
                                int32_t max_len, int32_t max_rank, int32_t* d_err, struct CUstream_st* stream)
{
    if (!kv || !query)
        return KAMERA_ERR_INVALID_ARGUMENT;
    if (query->n_seqs > 0 && kv->num_kv_heads > 0 &&
        kamera_attend_workspace_bytes(query->n_seqs, kv->num_kv_heads, kv->head_dim) > kScratchBytes)
        return KAMERA_ERR_UNSUPPORTED;   // the batch needs more partial states than the scratch holds
    void* scratch = scratch_on_current_device();
    if (!scratch)
        return KAMERA_ERR_CUDA;
    return kamera_attend_reused(kv, query, rope, d_chunks, d_seq_start, n_chunks, max_len, max_rank, scratch,
                                kScratchBytes, d_err, stream);
}

}  // extern "C"
