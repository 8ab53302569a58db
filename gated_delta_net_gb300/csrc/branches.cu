// branches.cu -- per-branch recurrent verification (the measurement baseline).
//
// "Trees from Marginals" (gist.science Experimental Results, Verification
// Efficiency) compares the fused tree kernel with per-branch recurrent
// verification.  This kernel is that baseline, written for this GPU: one block
// per (d_v slab, value head, request, leaf) carries the slab of the state in
// registers and applies the gated delta rule
//     S <- exp(g) * S * (I - beta k k^T) + beta v k^T,   o = scale * S q
// token by token down the leaf's root-to-leaf path, writing each node's output.
// Every leaf re-reads S0 and re-walks shared prefixes; nodes on several paths
// get identical values from each (the same operations in the same order).
#include "internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;

struct BranchParams {
    int hk_n, hv_n, dv, max_nodes;
    float scale;
    const int32_t *offsets, *parent;
    const void *q, *k, *v;
    const float *g, *beta, *S0;
    void *o;
    int32_t *status;
};

// SW state rows per block, TPR = 256 / SW threads per row, EPT = DK / TPR
// consecutive state columns per thread.
template <typename Tin, typename Tout, int DK, int SW>
__global__ void __launch_bounds__(kThreads)
verify_branches_kernel(BranchParams p) {
    constexpr int TPR = kThreads / SW;
    constexpr int EPT = DK / TPR;
    static_assert(EPT >= 1 && TPR <= 32 && (32 % TPR) == 0, "bad split");
    __shared__ int par[kMaxNodes];
    __shared__ int path[kMaxNodes];
    __shared__ int s_len;

    const int nslab = p.dv / SW;
    const int slab = blockIdx.x % nslab, h = blockIdx.y;
    const int bl = blockIdx.x / nslab;
    const int b = bl / p.max_nodes, leaf = bl % p.max_nodes;
    const int tid = threadIdx.x;
    const int lo = p.offsets[b];
    const int n = p.offsets[b + 1] - lo;
    if (leaf >= n) return;
    if (n > p.max_nodes) {
        if (tid == 0 && leaf == 0) flag(p.status, GDN_DEV_TOO_MANY);
        return;
    }
    bool has_child = false, bad = false;
    for (int i = tid; i < n; i += kThreads) {
        const int pi = p.parent[lo + i];
        par[i] = pi;
        has_child |= (pi == leaf);
        bad |= (pi < -1 || pi >= i);
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0 && leaf == 0) flag(p.status, GDN_DEV_BAD_TREE);
        return;
    }
    if (__syncthreads_or(has_child)) return;
    if (tid == 0) {
        int len = 0;
        for (int j = leaf; j >= 0; j = par[j]) ++len;
        int pos = len;
        for (int j = leaf; j >= 0; j = par[j]) path[--pos] = j;
        s_len = len;
    }
    __syncthreads();

    const int c = tid / TPR, part = tid % TPR, m0 = part * EPT;
    const int hk = h / (p.hv_n / p.hk_n);
    const Tin *qp = static_cast<const Tin *>(p.q);
    const Tin *kp = static_cast<const Tin *>(p.k);
    const Tin *vp = static_cast<const Tin *>(p.v);
    Tout *op = static_cast<Tout *>(p.o);
    const int row = slab * SW + c;
    float S[EPT];
    const float *src = p.S0 + (((int64_t)b * p.hv_n + h) * p.dv + row) * DK + m0;
#pragma unroll
    for (int e = 0; e < EPT; ++e) S[e] = src[e];

    const int len = s_len;
    for (int s = 0; s < len; ++s) {
        const int64_t t = lo + path[s];
        const int64_t krow = (t * p.hk_n + hk) * DK + m0;
        float kk[EPT], qq[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            kk[e] = load_f(kp, krow + e);
            qq[e] = load_f(qp, krow + e);
        }
        float sk = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) sk = fmaf(S[e], kk[e], sk);
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) sk += __shfl_xor_sync(0xffffffffu, sk, off);
        const float alpha = expf(p.g[t * p.hv_n + h]);
        const float beta = p.beta[t * p.hv_n + h];
        const float bv = beta * load_f(vp, (t * p.hv_n + h) * p.dv + row);
        float so = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            S[e] = alpha * (S[e] - beta * sk * kk[e]) + bv * kk[e];
            so = fmaf(S[e], qq[e], so);
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) so += __shfl_xor_sync(0xffffffffu, so, off);
        if (part == 0) store_f(op, (t * p.hv_n + h) * p.dv + row, p.scale * so);
    }
}

template <typename Tin, typename Tout, int SW>
cudaError_t launch_sw(const BranchParams &p, int dk, int batch, cudaStream_t stream) {
    dim3 grid((unsigned)(p.dv / SW) * (unsigned)batch * (unsigned)p.max_nodes, p.hv_n);
    switch (dk) {
        case 16: verify_branches_kernel<Tin, Tout, 16, SW><<<grid, kThreads, 0, stream>>>(p); break;
        case 32: verify_branches_kernel<Tin, Tout, 32, SW><<<grid, kThreads, 0, stream>>>(p); break;
        case 64: verify_branches_kernel<Tin, Tout, 64, SW><<<grid, kThreads, 0, stream>>>(p); break;
        case 128: verify_branches_kernel<Tin, Tout, 128, SW><<<grid, kThreads, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_io(const BranchParams &p, int dk, int batch, cudaStream_t stream) {
    return p.dv < 32 ? launch_sw<Tin, Tout, 16>(p, dk, batch, stream)
                     : launch_sw<Tin, Tout, 32>(p, dk, batch, stream);
}

}  // namespace

cudaError_t launch_verify_branches(const gdn_verify_args &a, cudaStream_t stream) {
    if ((int64_t)a.batch * a.max_nodes * (a.d_v < 32 ? 1 : a.d_v / 32) > 2147483647LL) return cudaErrorInvalidConfiguration;
    BranchParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.dv = a.d_v; p.max_nodes = a.max_nodes;
    p.scale = a.scale;
    p.offsets = a.node_offsets; p.parent = a.parent;
    p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.o = a.o; p.status = a.dev_status;
    const bool in_bf = a.qkv_dtype == GDN_BF16, out_bf = a.out_dtype == GDN_BF16;
    if (in_bf && out_bf) return launch_io<__nv_bfloat16, __nv_bfloat16>(p, a.d_k, a.batch, stream);
    if (in_bf) return launch_io<__nv_bfloat16, float>(p, a.d_k, a.batch, stream);
    if (out_bf) return launch_io<float, __nv_bfloat16>(p, a.d_k, a.batch, stream);
    return launch_io<float, float>(p, a.d_k, a.batch, stream);
}

}  // namespace gdn
