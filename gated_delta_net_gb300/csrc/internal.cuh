// internal.cuh -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "gdn_tree.h"

namespace gdn {

constexpr int kMaxNodes = 256;
constexpr int kMaxWords = kMaxNodes / 32;

__device__ __forceinline__ float load_f(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_f(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_f(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ void flag(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------
// launchers (one per translation unit); each returns a cudaError_t
// ---------------------------------------------------------------------------
cudaError_t launch_build_desc(const int32_t *parent, const int32_t *node_offsets, int batch,
                              int max_nodes, uint32_t *anc_mask, int mask_words,
                              int32_t *depth, int32_t *dev_status, cudaStream_t stream);

cudaError_t launch_verify_simt(const gdn_verify_args &a, cudaStream_t stream);
cudaError_t launch_relabel(const int32_t *parent_in, const int32_t *node_offsets, int batch, int total,
                           int max_nodes, int32_t *order, int32_t *rank, int32_t *parent_out,
                           int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_grow(const int32_t *node_offsets, int batch, int total, int width, int max_depth, int max_children,
                        const int32_t *n_children, const float *draws, int32_t *parent, float *score, int32_t *n_nodes,
                        int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_gather_rows(const void *src, void *dst, const int32_t *index, const int32_t *node_offsets,
                               int batch, int total, int64_t row_bytes, int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_verify_branches(const gdn_verify_args &a, cudaStream_t stream);
cudaError_t launch_commit_simt(const gdn_commit_args &a, cudaStream_t stream);

// TMA-staged commit for d_k = d_v = 128 and accepted paths of at most 16 nodes
bool commit_fast_supported(const gdn_commit_args &a);
cudaError_t launch_commit_fast(const gdn_commit_args &a, cudaStream_t stream);

// tensor-core commit for bf16 k/v, d_k = d_v = 128 and paths of at most 16 nodes
bool commit_tc_supported(const gdn_commit_args &a);
cudaError_t launch_commit_tc(const gdn_commit_args &a, cudaStream_t stream);

// the same kernel writing the states at selected nodes
bool states_tc_supported(const gdn_states_args &a);
cudaError_t launch_states_tc(const gdn_states_args &a, cudaStream_t stream);

// driver entry point for TMA descriptors (nullptr when the driver lacks it)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// streaming multiprocessors on the current device (1 if the query fails)
int sm_count();

// Poll limit of the wait probe (0 = off), set by gdn_test_set_wait_probe.
int wait_probe_polls();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device,
// once per (kernel, device, size): `have` remembers the largest size set so far
// per device.  Launches after the first make no attribute call, so they can be
// captured into a CUDA graph.
template <typename Kernel>
cudaError_t ensure_smem(Kernel kern, int bytes, int (&have)[16]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 16 && bytes <= have[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 16) have[dev] = bytes;
    return e;
}

// tcgen05/TMA fast path; after_commit launches it as the programmatic dependent
// of the commit launched just before it in the stream
bool verify_tc_supported(const gdn_verify_args &a);
cudaError_t launch_verify_tc(const gdn_verify_args &a, cudaStream_t stream, bool after_commit);

// the same for trees of 129 to 256 nodes (two node tiles per request)
bool verify_wide_supported(const gdn_verify_args &a);
cudaError_t launch_verify_wide(const gdn_verify_args &a, cudaStream_t stream, bool after_commit);

}  // namespace gdn
