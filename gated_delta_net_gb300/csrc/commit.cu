// commit.cu -- delayed state commit along the accepted path, in chunked form.
//
// "Trees from Marginals" (gist.science Technical Summary, section 3, Solution,
// last bullet): the recurrent state is committed in the next decoding
// iteration, once the accepted branch is known, so nothing is ever rolled back.
// For the accepted path p_1..p_L the state after the path is
//     S_new = exp(gamma_L) S0 + sum_t exp(gamma_L - gamma_t) u_t k_t^T,
// where gamma_t sums g over p_1..p_t and u solves the verification system of
// the same section restricted to the path (a chain):
//     u_t = beta_t (v_t - exp(gamma_t) S0 k_t)
//           - sum_{s<t} beta_t exp(gamma_t - gamma_s) (k_t . k_s) u_s.
//
// One block per (d_v slab of 32 state rows, value head, request).  The block
// reads its S0 slab into shared memory before writing anything, and blocks
// own disjoint slabs, so S_new may alias S0.
#include "internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kKChunk = 32;  // path keys staged per round of the state update

struct CommitParams {
    int hk_n, hv_n, dv, max_nodes, sw;
    const int32_t *offsets, *parent, *poff, *pidx;
    const void *k, *v;
    const float *g, *beta, *S0;
    float *S_new;
    int32_t *status;
};

struct CommitSmem {
    int s0, u, gam, bet, coef, kc, kq;  // float offsets
    int pn;                             // int offset after floats
    int floats, ints;
};

__host__ __device__ inline CommitSmem commit_layout(int nm, int sw, int dk) {
    CommitSmem L;
    int f = 0;
    L.s0 = f;   f += sw * (dk + 1);
    L.u = f;    f += nm * sw;
    L.gam = f;  f += nm;
    L.bet = f;  f += nm;
    L.coef = f; f += nm;
    L.kc = f;   f += kKChunk * dk;
    L.kq = f;   f += kWarps * dk;
    L.floats = f;
    L.pn = 0;
    L.ints = nm;
    return L;
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreads)
commit_simt_kernel(CommitParams p) {
    constexpr int EPL = (DK + 31) / 32;
    extern __shared__ float smem[];
    const int nm = p.max_nodes, SW = p.sw;
    const CommitSmem L = commit_layout(nm, SW, DK);
    float *S0s = smem + L.s0, *U = smem + L.u, *gam = smem + L.gam, *bet = smem + L.bet;
    float *coef = smem + L.coef, *Kc = smem + L.kc;
    int *pn = reinterpret_cast<int *>(smem + L.floats) + L.pn;

    const int nslab = p.dv / p.sw;
    const int slab = blockIdx.x % nslab, b = blockIdx.x / nslab, h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = p.offsets[b];
    const int n = p.offsets[b + 1] - lo;
    const int pa = p.poff[b];
    const int len = p.poff[b + 1] - pa;
    const int hk = h / (p.hv_n / p.hk_n);
    const Tin *kp = static_cast<const Tin *>(p.k);
    const Tin *vp = static_cast<const Tin *>(p.v);
    const int64_t sbase = ((int64_t)b * p.hv_n + h) * p.dv * DK + (int64_t)slab * SW * DK;
    const float *s0src = p.S0 + sbase;
    float *sdst = p.S_new + sbase;

    if (n > nm) {
        if (tid == 0) flag(p.status, GDN_DEV_TOO_MANY);
        return;
    }
    // a path visits distinct nodes of its own request, root first
    bool bad = len < 0 || len > n;
    if (!bad) {
        for (int t = tid; t < len; t += kThreads) {
            const int node = p.pidx[pa + t];
            const int expect = t == 0 ? -1 : p.pidx[pa + t - 1];
            if (node < 0 || node >= n || p.parent[lo + node] != expect) bad = true;
        }
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) flag(p.status, GDN_DEV_BAD_PATH);
        return;
    }
    for (int e = tid; e < SW * DK; e += kThreads) {
        const int c = e / DK, m = e - c * DK;
        S0s[c * (DK + 1) + m] = s0src[e];
    }
    for (int t = tid; t < len; t += kThreads) {
        const int node = p.pidx[pa + t];
        pn[t] = node;
        bet[t] = p.beta[(int64_t)(lo + node) * p.hv_n + h];
        gam[t] = p.g[(int64_t)(lo + node) * p.hv_n + h];  // prefix-summed below
    }
    __syncthreads();
    if (len == 0) {
        if (sdst != s0src)
            for (int e = tid; e < SW * DK; e += kThreads) sdst[e] = S0s[(e / DK) * (DK + 1) + e % DK];
        return;
    }
    if (tid == 0)
        for (int t = 1; t < len; ++t) gam[t] += gam[t - 1];
    __syncthreads();

    // right-hand side r_t = beta_t (v_t - e^{gamma_t} S0 k_t) for the slab's rows
    float *kqw = smem + L.kq + warp * DK;
    for (int t = warp; t < len; t += kWarps) {
        const int64_t krow = ((int64_t)(lo + pn[t]) * p.hk_n + hk) * DK;
        for (int m = lane; m < DK; m += 32) kqw[m] = load_f(kp, krow + m);
        __syncwarp();
        if (lane < SW) {
            float w = 0.f;
            const float *srow = S0s + lane * (DK + 1);
#pragma unroll 8
            for (int m = 0; m < DK; ++m) w = fmaf(srow[m], kqw[m], w);
            const float vt = load_f(vp, ((int64_t)(lo + pn[t]) * p.hv_n + h) * p.dv + slab * SW + lane);
            U[t * SW + lane] = bet[t] * (vt - expf(gam[t]) * w);
        }
        __syncwarp();
    }
    __syncthreads();

    // chain forward substitution, one path position at a time
    for (int t = 1; t < len; ++t) {
        const int64_t trow = ((int64_t)(lo + pn[t]) * p.hk_n + hk) * DK;
        float kt[EPL];
#pragma unroll
        for (int r = 0; r < EPL; ++r) {
            const int m = lane + 32 * r;
            kt[r] = m < DK ? load_f(kp, trow + m) : 0.f;
        }
        for (int s = warp; s < t; s += kWarps) {
            const int64_t srow = ((int64_t)(lo + pn[s]) * p.hk_n + hk) * DK;
            float d = 0.f;
#pragma unroll
            for (int r = 0; r < EPL; ++r) {
                const int m = lane + 32 * r;
                d = fmaf(kt[r], m < DK ? load_f(kp, srow + m) : 0.f, d);
            }
            d = warp_sum(d);
            if (lane == 0) coef[s] = bet[t] * expf(gam[t] - gam[s]) * d;
        }
        __syncthreads();
        if (tid < SW) {
            float acc = U[t * SW + tid];
            for (int s = 0; s < t; ++s) acc -= coef[s] * U[s * SW + tid];
            U[t * SW + tid] = acc;
        }
        __syncthreads();
    }

    // S_new = e^{gamma_L} S0 + sum_t e^{gamma_L - gamma_t} u_t k_t^T
    const float gL = gam[len - 1];
    for (int t = tid; t < len; t += kThreads) coef[t] = expf(gL - gam[t]);
    const float eL = expf(gL);
    constexpr int kPer = (32 * DK + kThreads - 1) / kThreads;  // elements per thread (SW <= 32)
    float acc[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int e = tid + r * kThreads;
        acc[r] = e < SW * DK ? eL * S0s[(e / DK) * (DK + 1) + e % DK] : 0.f;
    }
    for (int t0 = 0; t0 < len; t0 += kKChunk) {
        const int tn = min(kKChunk, len - t0);
        __syncthreads();
        for (int e = tid; e < tn * DK; e += kThreads) {
            const int t = e / DK, m = e - t * DK;
            Kc[e] = load_f(kp, ((int64_t)(lo + pn[t0 + t]) * p.hk_n + hk) * DK + m);
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const int e = tid + r * kThreads;
            if (e < SW * DK) {
                const int c = e / DK, m = e - c * DK;
                float a = acc[r];
                for (int t = 0; t < tn; ++t) a = fmaf(coef[t0 + t] * U[(t0 + t) * SW + c], Kc[t * DK + m], a);
                acc[r] = a;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int e = tid + r * kThreads;
        if (e < SW * DK) sdst[e] = acc[r];
    }
}

template <typename Tin, int DK>
cudaError_t launch_typed(const CommitParams &p, int batch, cudaStream_t stream) {
    const CommitSmem L = commit_layout(p.max_nodes, p.sw, DK);
    const size_t bytes = sizeof(float) * (size_t)L.floats + sizeof(int) * (size_t)L.ints;
    auto kern = commit_simt_kernel<Tin, DK>;
    static int have[16];  // one per template instance
    cudaError_t e = ensure_smem(kern, (int)bytes, have);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.dv / p.sw) * (unsigned)batch, p.hv_n);
    kern<<<grid, kThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dk(const CommitParams &p, int dk, int batch, cudaStream_t stream) {
    switch (dk) {
        case 16: return launch_typed<Tin, 16>(p, batch, stream);
        case 32: return launch_typed<Tin, 32>(p, batch, stream);
        case 64: return launch_typed<Tin, 64>(p, batch, stream);
        case 128: return launch_typed<Tin, 128>(p, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_commit_simt(const gdn_commit_args &a, cudaStream_t stream) {
    CommitParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.dv = a.d_v; p.max_nodes = a.max_nodes;
    p.sw = a.d_v < 32 ? a.d_v : 32;
    p.offsets = a.node_offsets; p.parent = a.parent; p.poff = a.path_offsets; p.pidx = a.path_idx;
    p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.S_new = a.S_new; p.status = a.dev_status;
    if (a.qkv_dtype == GDN_BF16) return launch_dk<__nv_bfloat16>(p, a.d_k, a.batch, stream);
    return launch_dk<float>(p, a.d_k, a.batch, stream);
}

}  // namespace gdn
