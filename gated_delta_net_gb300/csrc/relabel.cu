// relabel.cu -- topological relabelling of draft trees (integer work, bit-exact).
//
// "Trees from Marginals" (gist.science Technical Summary, section 3, Solution,
// bullet 1) verifies a tree in topological order.  A tree given in any other
// order is relabelled by (depth, old id): parents are one level shallower
// than their children, so they always come first, and the order is unique.
//
// One block per request, one thread per node (at most 256):
//   depth by pointer jumping: after r rounds a node has summed the lengths of
//   2^r path segments, so 8 rounds reach the root from any of 256 nodes; a node
//   whose pointer is still not past a root lies on or below a cycle;
//   rank_i = #{ j : (depth_j, j) < (depth_i, i) }, a count over the block.
#include <algorithm>

#include "internal.cuh"

namespace gdn {
namespace {

constexpr int kT = kMaxNodes;  // 256 threads: one per node

__global__ void __launch_bounds__(kT)
relabel_kernel(const int32_t *__restrict__ parent_in, const int32_t *__restrict__ offsets, int total,
               int max_nodes, int32_t *__restrict__ order, int32_t *__restrict__ rank,
               int32_t *__restrict__ parent_out, int32_t *status) {
    __shared__ int jmp[2][kT], len[2][kT], dep[kT], rnk[kT];
    __shared__ int s_bad;
    const int b = blockIdx.x, i = threadIdx.x;
    const int lo = offsets[b];
    const int n = offsets[b + 1] - lo;
    if (n == 0) return;
    if (n < 0 || n > max_nodes || lo < 0 || lo + n > total) {
        if (i == 0) flag(status, n > max_nodes ? GDN_DEV_TOO_MANY : GDN_DEV_BAD_DESC);
        return;
    }
    if (i == 0) s_bad = 0;
    __syncthreads();
    int p = -1;
    if (i < n) {
        p = parent_in[lo + i];
        if (p < -1 || p >= n || p == i) atomicOr(&s_bad, 1);
    }
    jmp[0][i] = i < n ? p : -1;
    len[0][i] = 1;
    __syncthreads();
    if (s_bad) {
        if (i == 0) flag(status, GDN_DEV_BAD_TREE);
        return;
    }
    int cur = 0;
#pragma unroll 1
    for (int r = 0; r < 8; ++r) {
        int j = jmp[cur][i], l = len[cur][i];
        if (j >= 0) {
            l += len[cur][j];
            j = jmp[cur][j];
        }
        jmp[cur ^ 1][i] = j;
        len[cur ^ 1][i] = l;
        __syncthreads();
        cur ^= 1;
    }
    if (i < n && jmp[cur][i] >= 0) atomicOr(&s_bad, 1);  // never reached a root: a cycle
    dep[i] = i < n ? len[cur][i] : 0x7fffffff;
    __syncthreads();
    if (s_bad) {
        if (i == 0) flag(status, GDN_DEV_BAD_TREE);
        return;
    }
    if (i < n) {
        const int di = dep[i];
        int r = 0;
        for (int j = 0; j < n; ++j) {
            const int dj = dep[j];
            r += (dj < di) | ((dj == di) & (j < i));
        }
        rnk[i] = r;
        rank[lo + i] = r;
        order[lo + r] = i;
    }
    __syncthreads();
    if (i < n) parent_out[lo + rnk[i]] = p < 0 ? -1 : rnk[p];
}

// dst row lo + j = src row lo + index[lo + j] (request-local index).  Block
// (x, b) serves request b: its threads stride over the request's rows x 16-byte
// chunks, four independent copies in flight per thread.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, const int32_t *__restrict__ index,
                   const int32_t *__restrict__ offsets, int total, int64_t chunks, int32_t *status) {
    const int b = blockIdx.y;
    const int lo = offsets[b], n = offsets[b + 1] - lo;
    if (n <= 0 || lo < 0 || lo + n > total) return;
    const int64_t work = (int64_t)n * chunks;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e0 < work; e0 += 4 * step) {
        uint4 v[4];
        int64_t to[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t e = e0 + u * step;
            to[u] = -1;
            if (e < work) {
                const int r = (int)(e / chunks);
                const int64_t c = e - (int64_t)r * chunks;
                const int j = __ldg(index + lo + r);
                if (j < 0 || j >= n) {
                    if (c == 0) flag(status, GDN_DEV_BAD_DESC);
                } else {
                    v[u] = __ldg(src + (int64_t)(lo + j) * chunks + c);
                    to[u] = (int64_t)(lo + r) * chunks + c;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (to[u] >= 0) dst[to[u]] = v[u];
    }
}

}  // namespace

cudaError_t launch_gather_rows(const void *src, void *dst, const int32_t *index, const int32_t *node_offsets,
                               int batch, int total, int64_t row_bytes, int32_t *dev_status, cudaStream_t stream) {
    if (batch > 65535) return cudaErrorInvalidValue;
    const int64_t chunks = row_bytes / 16;
    // about four blocks per SM over the whole batch, at least one per request
    const int per = std::max(1, std::min(256, (4 * sm_count() + batch - 1) / batch));
    gather_rows_kernel<<<dim3((unsigned)per, (unsigned)batch), 256, 0, stream>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), index, node_offsets, total, chunks, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_relabel(const int32_t *parent_in, const int32_t *node_offsets, int batch, int total,
                           int max_nodes, int32_t *order, int32_t *rank, int32_t *parent_out,
                           int32_t *dev_status, cudaStream_t stream) {
    relabel_kernel<<<batch, kT, 0, stream>>>(parent_in, node_offsets, total, max_nodes, order, rank, parent_out,
                                             dev_status);
    return cudaGetLastError();
}

}  // namespace gdn
