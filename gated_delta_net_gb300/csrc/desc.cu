// desc.cu -- tree descriptor: ancestor bitmask rows and depths.
//
// "Trees from Marginals" (gist.science Technical Summary, section 3, Solution):
// the tree is sorted topologically and the interaction matrices are restricted
// to ancestor relationships.  Bit j of row i is set iff j is on i's
// root-to-node path (i included); depth counts the nodes on that path.
#include "internal.cuh"

namespace gdn {
namespace {

// One block per request, one thread per node.  Each thread walks its parent
// chain in shared memory; the walk is at most max_nodes steps because every
// valid step strictly decreases the node id.
__global__ void __launch_bounds__(kMaxNodes)
build_desc_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ offsets,
                  int max_nodes, uint32_t *__restrict__ anc_mask, int mask_words,
                  int32_t *__restrict__ depth, int32_t *dev_status) {
    __shared__ int32_t par[kMaxNodes];
    const int b = blockIdx.x;
    const int lo = offsets[b];
    const int n = offsets[b + 1] - lo;
    if (n <= 0) return;
    if (n > max_nodes) {
        if (threadIdx.x == 0) flag(dev_status, GDN_DEV_TOO_MANY);
        return;
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) par[i] = parent[lo + i];
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        uint32_t row[kMaxWords];
#pragma unroll
        for (int w = 0; w < kMaxWords; ++w) row[w] = 0u;
        int d = 0;
        bool ok = true;
        for (int j = i; j >= 0;) {
            const uint32_t bit = 1u << (j & 31);
#pragma unroll
            for (int w = 0; w < kMaxWords; ++w)
                if ((j >> 5) == w) row[w] |= bit;
            ++d;
            const int p = par[j];
            if (p < -1 || p >= j) { ok = false; break; }
            j = p;
        }
        if (!ok) {
            flag(dev_status, GDN_DEV_BAD_TREE);
            d = 0;
#pragma unroll
            for (int w = 0; w < kMaxWords; ++w) row[w] = 0u;
        }
        uint32_t *dst = anc_mask + (int64_t)(lo + i) * mask_words;
#pragma unroll
        for (int w = 0; w < kMaxWords; ++w)
            if (w < mask_words) dst[w] = row[w];
        depth[lo + i] = d;
    }
}

}  // namespace

cudaError_t launch_build_desc(const int32_t *parent, const int32_t *node_offsets, int batch,
                              int max_nodes, uint32_t *anc_mask, int mask_words,
                              int32_t *depth, int32_t *dev_status, cudaStream_t stream) {
    const int threads = max_nodes <= 32 ? 32 : (max_nodes <= 128 ? 128 : kMaxNodes);
    build_desc_kernel<<<batch, threads, 0, stream>>>(parent, node_offsets, max_nodes, anc_mask,
                                                     mask_words, depth, dev_status);
    return cudaGetLastError();
}

}  // namespace gdn
