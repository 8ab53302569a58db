// grow.cu -- draft-tree construction by top-w best-first expansion (sm_103a).
//
// "Trees from Marginals" (gist.science Technical Summary, Methodology, section 2
// "Tree Construction") modifies DySpec's best-first search: the top-w nodes of
// the candidate heap are expanded together.  Node 0 is the root (score 0,
// depth 1); ids follow creation order; the frontier is every node not yet
// expanded whose depth is below max_depth.  One step takes the w best frontier
// nodes (score descending, then id ascending) and expands them in that order:
// node p gets children j < c_p with score_p - e_pj * (j + 1), until the
// request's capacity is reached.
//
// One block per request, one thread per node slot (capacity <= 256).  Per step
// each frontier node counts the frontier nodes ahead of it (its rank); the w
// best write their child counts by rank, an exclusive sum over ranks gives
// each one's first child id, and the children are written.  Scores use one
// rounded multiply and one rounded subtract, the float32 definition.
#include "internal.cuh"

namespace gdn {
namespace {

constexpr int kT = kMaxNodes;

__global__ void __launch_bounds__(kT)
grow_kernel(const int32_t *__restrict__ offsets, int total, int width, int max_depth, int max_children,
            const int32_t *__restrict__ n_children, const float *__restrict__ draws, int32_t *__restrict__ parent,
            float *__restrict__ score, int32_t *__restrict__ n_nodes, int32_t *status) {
    __shared__ float sc[kT];
    __shared__ int par[kT], dep[kT], expd[kT], cnt[kT];
    __shared__ int s_created;
    const int b = blockIdx.x, t = threadIdx.x;
    const int lo = offsets[b];
    const int cap = offsets[b + 1] - lo;
    if (cap == 0) {
        if (t == 0) n_nodes[b] = 0;
        return;
    }
    if (cap < 0 || cap > kT || lo < 0 || lo + cap > total) {
        if (t == 0) flag(status, cap > kT ? GDN_DEV_TOO_MANY : GDN_DEV_BAD_DESC);
        return;
    }
    if (t == 0) {
        par[0] = -1;
        dep[0] = 1;
        sc[0] = 0.f;
        expd[0] = 0;
        s_created = 1;
    }
    __syncthreads();
    // every step creates a node or expands one, so 2 * capacity steps suffice
#pragma unroll 1
    for (int step = 0; step < 2 * kT; ++step) {
        const int created = s_created;
        if (created >= cap) break;  // block-uniform
        const bool front = t < created && !expd[t] && dep[t] < max_depth;
        int r = 0;
        if (front) {
            const float st = sc[t];
            for (int j = 0; j < created; ++j) {
                const float sj = sc[j];
                r += (!expd[j] && dep[j] < max_depth) & ((sj > st) | ((sj == st) & (j < t)));
            }
        }
        const int nf = __syncthreads_count(front);  // every rank is computed
        if (nf == 0) break;                         // block-uniform: the frontier is empty
        const bool chosen = front && r < width;
        int c = 0;
        if (chosen) {
            c = min(max(n_children[lo + t], 0), max_children);
            cnt[r] = c;
        }
        __syncthreads();
        if (chosen) {
            expd[t] = 1;
            int base = created;
            for (int q = 0; q < r; ++q) base += cnt[q];
            const float sp = sc[t];
            const int dp = dep[t];
            for (int j = 0; j < c; ++j) {
                const int id = base + j;
                if (id >= cap) break;
                const float e = draws[(int64_t)(lo + t) * max_children + j];
                par[id] = t;
                dep[id] = dp + 1;
                expd[id] = 0;
                sc[id] = __fsub_rn(sp, __fmul_rn(e, (float)(j + 1)));
            }
        }
        __syncthreads();
        if (t == 0) {
            int made = 0;
            for (int q = 0; q < min(width, nf); ++q) made += cnt[q];
            s_created = min(cap, created + made);
        }
        __syncthreads();
    }
    const int created = s_created;
    if (t < cap) {
        parent[lo + t] = t < created ? par[t] : -1;
        score[lo + t] = t < created ? sc[t] : -INFINITY;
    }
    if (t == 0) n_nodes[b] = created;
}

}  // namespace

cudaError_t launch_grow(const int32_t *node_offsets, int batch, int total, int width, int max_depth, int max_children,
                        const int32_t *n_children, const float *draws, int32_t *parent, float *score, int32_t *n_nodes,
                        int32_t *dev_status, cudaStream_t stream) {
    grow_kernel<<<batch, kT, 0, stream>>>(node_offsets, total, width, max_depth, max_children, n_children, draws,
                                          parent, score, n_nodes, dev_status);
    return cudaGetLastError();
}

}  // namespace gdn
