// kamera_internal.h -- declarations shared by the Kamera translation units
// (host launchers; not part of the public C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kamera.h"

namespace kamera {

enum Family { FAMILY_GQA = 0, FAMILY_MLA = 1, FAMILY_SLIDE = 2 };

struct RowsParams;

// Bound, in ns, of the pipeline waits of the tensor-core kernels: 1 s, or the
// value of the environment variable KAMERA_WAIT_LIMIT_NS when it is set (a
// test hook: a short bound makes the kernels give up early and report
// KAMERA_DEVERR_TIMEOUT).  Read on the host at each launch.
uint64_t wait_limit_ns();

// Test hook: KAMERA_TEST_WITHHOLD_LOADS=1 in the environment makes the
// producers of the relocation and prefill attention kernels issue no loads,
// so their first pipeline waits run out after the bound above (read on the
// host at each launch).
bool test_withhold_loads();

// CUDA-core streaming path (any rank within the shared-memory budget).
cudaError_t launch_simt(const RowsParams& p, int family, cudaStream_t stream);
size_t simt_smem_bytes(const RowsParams& p, int family, int tile_tokens);

// Sliding-window survival (in place, rotation only): one fixed rotary unit
// per thread; shapes whose units per row divide the block (else the CUDA-core path).
bool slide_supported(const RowsParams& p);
cudaError_t launch_slide(const RowsParams& p, cudaStream_t stream);

// Canonical ingest: the passes of a row (returns their count, -1 if the rotary
// layout does not split into 16-byte units) and the launch.
struct IngestPass;
struct IngestParams;
struct PatchFormParams;
struct AttendParams;
struct PrefillParams;
int ingest_passes(const RowsParams& rp, bool values, IngestPass* out);
cudaError_t launch_ingest(const IngestParams& p, cudaStream_t stream);

// Patch formation: whether a block shape is handled; one CTA per block.
bool patch_form_supported(int cols, int m);
cudaError_t launch_patch_form(const PatchFormParams& p, int64_t n_blocks, cudaStream_t stream);

// Clusters of `cl` CTAs (block_threads threads, smem_bytes of dynamic shared
// memory) of `kernel` that fit on the current device at once, from
// cudaOccupancyMaxActiveClusters; 0 if the query fails.  The answer depends
// only on these arguments and the device, so it is cached (thread-safe).
int cluster_fit(const void* kernel, int block_threads, int smem_bytes, int cl);

// Decode attention over reused chunks: shapes handled; one CTA per (sequence, KV head).
// With a workspace (ws non-NULL, ws_bytes of it) a call may take the split
// path: partial softmax states per (CTA, unit) in the workspace, then a merge
// launch; the workspace needs (CTAs resident at once + units - 1) slots of
// attend_slot_bytes(output width) bytes.
bool attend_supported(int head_dim, int G, int max_rank);
int attend_cluster(int64_t units);
cudaError_t launch_attend(const AttendParams& p, void* ws, size_t ws_bytes, cudaStream_t stream);
bool mla_attend_supported(int kv_lora, int rope_dim, int num_q_heads, int max_rank);
cudaError_t launch_mla_attend(const MlaAttendParams& p, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t attend_slot_bytes(int dout);
cudaError_t launch_attend_merge(const float* ws, int64_t units, int64_t ctas, int dout, int groups, int Hq,
                                int rows, __nv_bfloat16* out, cudaStream_t stream);

// Prefill attention over reused chunks (tensor cores): shapes handled; one CTA
// per 128 query rows of a (sequence, KV head).
bool prefill_supported(int head_dim, int max_rank);
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);

// 2-D tensor map (a CUtensorMap, 64-byte aligned, at `map`) over a bf16 array
// of `rows` rows of `width` elements, row_stride elements apart: boxes of
// box_cols x box_rows, 128-byte swizzle, rows past the end read as zero.
// False if the driver has no encoder or refuses the shape.
bool make_rows_map(void* map, const void* base, int64_t rows, int64_t width, int64_t row_stride, int box_cols,
                   int box_rows);

// Tensor-core path (tcgen05 MMA for the rank-m patch; relocation with rank > 0).
bool umma_supported(const RowsParams& p, int family);
size_t umma_smem_bytes(const RowsParams& p);
// h_chunks: NULL or a host copy of the descriptors (U tiles then move by TMA).
cudaError_t launch_umma(const RowsParams& p, int family, const KameraChunk* h_chunks, cudaStream_t stream);

}  // namespace kamera
