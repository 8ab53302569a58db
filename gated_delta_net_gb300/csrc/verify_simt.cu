// verify_simt.cu -- general tree verification kernel (any dtype, any d, any depth).
//
// "Trees from Marginals" (gist.science Technical Summary, section 3
// "Rollback-Free Tree Verification for GDN"): the outputs of every node of a
// topologically sorted draft tree come from one triangular solve,
//     (I + X) U = beta * (V - exp(gamma) * K S0^T),
//     O = scale * (exp(gamma) * Q S0^T + Y U),
// where X and Y only couple a node to its ancestors.  Because row i of X has
// non-zeros only on i's strict ancestors, the solve runs level by level: all
// nodes at one depth are independent once the shallower levels are done.
//
// One block per (d_v slab of 32 columns, value head, request); 8 warps.
//   phase 0: tree metadata, gamma (sum of g along each path), depth buckets;
//   phase 1: per node, W = S0 k, Z = S0 q for the slab, R = beta (v - e^gamma W);
//   phase 2: per depth level, per node (one warp): dot products with each
//            ancestor's key, forward substitution for u_i, then o_i.
// For small trees (max_nodes x path bound <= kRawMax) the coefficients of every
// (node, ancestor) pair, beta_i e^(gamma_i - gamma_a) k_i.k_a and
// e^(gamma_i - gamma_a) q_i.k_a, and each node's path are made first, by all warps
// at once (phase 1b), so that the level-ordered phase 2 only combines them: a
// chain, one node per level, then no longer runs its dot products one level at a
// time.
// Only a node's ancestors are ever read, so a non-finite input on one branch
// cannot reach another branch's outputs.  Everything accumulates in fp32.
#include <algorithm>

#include "internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRawMax = 4096;  // entries of each raw dot-product table [nodes][path length]

struct SimtParams {
    int hk_n, hv_n, dv, max_nodes, sw;
    int md;  // > 0: phase 1b on, rows of md entries (path length bound); 0: off
    float scale;
    const int32_t *offsets, *parent, *depth;
    const void *q, *k, *v;
    const float *g, *beta, *S0;
    void *o;
    int32_t *status;
};

struct SmemLayout {
    int s0, ub, zb, gam, gl, bet, kq, rk, rq, self, pth;  // float offsets (pth: int entries)
    int par, dep, order, cnt, start;   // int offsets (after the floats)
    int floats, ints;
};

__host__ __device__ inline SmemLayout smem_layout(int nm, int sw, int dk, int md) {
    SmemLayout L;
    int f = 0;
    L.s0 = f;  f += sw * (dk + 1);
    L.ub = f;  f += nm * sw;
    L.zb = f;  f += nm * sw;
    L.gam = f; f += nm;
    L.gl = f;  f += nm;
    L.bet = f; f += nm;
    L.kq = f;  f += kWarps * 2 * dk;
    L.rk = f;  f += nm * md;
    L.rq = f;  f += nm * md;
    L.self = f; f += md > 0 ? nm : 0;
    L.pth = f; f += nm * md;
    L.floats = f;
    int i = 0;
    L.par = i;   i += nm;
    L.dep = i;   i += nm;
    L.order = i; i += nm;
    L.cnt = i;   i += nm + 2;
    L.start = i; i += nm + 2;
    L.ints = i;
    return L;
}

template <typename Tin, typename Tout, int DK>
__global__ void __launch_bounds__(kThreads)
verify_simt_kernel(SimtParams p) {
    constexpr int EPL = (DK + 31) / 32;  // key elements per lane
    extern __shared__ float smem[];
    const int nm = p.max_nodes, SW = p.sw;
    const SmemLayout L = smem_layout(nm, SW, DK, p.md);
    float *S0s = smem + L.s0, *Ub = smem + L.ub, *Zb = smem + L.zb;
    float *RK = smem + L.rk, *RQ = smem + L.rq, *SELF = smem + L.self;  // phase 1b tables
    int *PTH = reinterpret_cast<int *>(smem + L.pth);
    const int MD = p.md;
    float *gam = smem + L.gam, *gl = smem + L.gl, *bet = smem + L.bet;
    int *ism = reinterpret_cast<int *>(smem + L.floats);
    int *par = ism + L.par, *dep = ism + L.dep, *order = ism + L.order;
    int *cnt = ism + L.cnt, *start = ism + L.start;
    __shared__ int s_maxd;

    const int nslab = p.dv / p.sw;
    const int slab = blockIdx.x % nslab, b = blockIdx.x / nslab, h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = p.offsets[b];
    const int n = p.offsets[b + 1] - lo;
    if (n <= 0) return;
    if (n > nm) {
        if (tid == 0) flag(p.status, GDN_DEV_TOO_MANY);
        return;
    }
    const int hk = h / (p.hv_n / p.hk_n);
    const Tin *qp = static_cast<const Tin *>(p.q);
    const Tin *kp = static_cast<const Tin *>(p.k);
    const Tin *vp = static_cast<const Tin *>(p.v);
    Tout *op = static_cast<Tout *>(p.o);

    // ---- phase 0: metadata ------------------------------------------------
    if (tid == 0) s_maxd = 0;
    for (int i = tid; i < nm + 2; i += kThreads) cnt[i] = 0;
    for (int i = tid; i < n; i += kThreads) {
        par[i] = p.parent[lo + i];
        dep[i] = p.depth[lo + i];
        gl[i] = p.g[(int64_t)(lo + i) * p.hv_n + h];
        bet[i] = p.beta[(int64_t)(lo + i) * p.hv_n + h];
    }
    const float *s0src = p.S0 + ((int64_t)b * p.hv_n + h) * p.dv * DK + (int64_t)slab * SW * DK;
    for (int e = tid; e < SW * DK; e += kThreads) {
        const int c = e / DK, m = e - c * DK;
        S0s[c * (DK + 1) + m] = s0src[e];
    }
    __syncthreads();
    bool bad_tree = false, bad_desc = false;
    for (int i = tid; i < n; i += kThreads) {
        const int pi = par[i];
        if (pi < -1 || pi >= i) bad_tree = true;
        else if (dep[i] != (pi < 0 ? 1 : dep[pi] + 1)) bad_desc = true;
    }
    if (__syncthreads_or(bad_tree)) {
        if (tid == 0) flag(p.status, GDN_DEV_BAD_TREE);
        return;
    }
    if (__syncthreads_or(bad_desc)) {
        if (tid == 0) flag(p.status, GDN_DEV_BAD_DESC);
        return;
    }
    for (int i = tid; i < n; i += kThreads) {
        float acc = 0.f;
        for (int j = i; j >= 0; j = par[j]) acc += gl[j];
        gam[i] = acc;
        atomicAdd(&cnt[dep[i]], 1);
        atomicMax(&s_maxd, dep[i]);
    }
    __syncthreads();
    const int maxd = s_maxd;
    if (tid == 0) {
        int run = 0;
        for (int d = 0; d <= maxd + 1; ++d) {
            start[d] = run;
            run += (d <= maxd) ? cnt[d] : 0;
        }
    }
    __syncthreads();
    for (int i = tid; i < nm + 2; i += kThreads) cnt[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
        const int d = dep[i];
        order[start[d] + atomicAdd(&cnt[d], 1)] = i;
    }

    // ---- phase 1: S0 read-out and right-hand side -------------------------
    float *kqw = smem + L.kq + warp * 2 * DK;
    // each warp's next node's k and q rows are requested while it works on the current one
    float kn[EPL], qn[EPL];
    auto kq_load = [&](int i) {
        const int64_t krow = ((int64_t)(lo + i) * p.hk_n + hk) * DK;
#pragma unroll
        for (int r = 0; r < EPL; ++r) {
            const int m = lane + 32 * r;
            kn[r] = (i < n && m < DK) ? load_f(kp, krow + m) : 0.f;
            qn[r] = (i < n && m < DK) ? load_f(qp, krow + m) : 0.f;
        }
    };
    kq_load(warp);
    for (int i = warp; i < n; i += kWarps) {
#pragma unroll
        for (int r = 0; r < EPL; ++r) {
            const int m = lane + 32 * r;
            if (m < DK) {
                kqw[m] = kn[r];
                kqw[DK + m] = qn[r];
            }
        }
        kq_load(i + kWarps);
        __syncwarp();
        if (lane < SW) {
            const float vi = load_f(vp, ((int64_t)(lo + i) * p.hv_n + h) * p.dv + slab * SW + lane);
            float w = 0.f, z = 0.f;
            const float *srow = S0s + lane * (DK + 1);
#pragma unroll 8
            for (int m = 0; m < DK; ++m) {
                w = fmaf(srow[m], kqw[m], w);
                z = fmaf(srow[m], kqw[DK + m], z);
            }
            Ub[i * SW + lane] = bet[i] * (vi - expf(gam[i]) * w);
            Zb[i * SW + lane] = z;
        }
        __syncwarp();
    }
    __syncthreads();

    // ---- phase 1b: pair coefficients of every (node, ancestor) pair --------
    // for the strict ancestors a of i, at l = dep(a) - 1:
    //   RK[i][l] = beta_i e^(gamma_i - gamma_a) k_i.k_a,  RQ[i][l] = e^(gamma_i - gamma_a) q_i.k_a,
    //   PTH[i][l] = a;  SELF[i] = q_i.k_i.  The rows hold MD >= the tree's depth entries.
    const bool raw = MD > 0 && maxd <= MD;
    if (raw) {
        for (int i = warp; i < n; i += kWarps) {
            const int64_t krow = ((int64_t)(lo + i) * p.hk_n + hk) * DK;
            float kr[EPL], qr[EPL];
#pragma unroll
            for (int r = 0; r < EPL; ++r) {
                const int m = lane + 32 * r;
                kr[r] = m < DK ? load_f(kp, krow + m) : 0.f;
                qr[r] = m < DK ? load_f(qp, krow + m) : 0.f;
            }
            float self = 0.f;
#pragma unroll
            for (int r = 0; r < EPL; ++r) self = fmaf(qr[r], kr[r], self);
            self = warp_sum(self);
            if (lane == 0) SELF[i] = self;
            // ancestors four at a time: their key rows are requested together
            constexpr int kBatch = 4;
            for (int j = par[i]; j >= 0;) {
                int js[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    js[u] = j;
                    if (j >= 0) j = par[j];
                }
                float kj[kBatch][EPL];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int64_t jrow = ((int64_t)(lo + max(js[u], 0)) * p.hk_n + hk) * DK;
#pragma unroll
                    for (int r = 0; r < EPL; ++r) {
                        const int m = lane + 32 * r;
                        kj[u][r] = (js[u] >= 0 && m < DK) ? load_f(kp, jrow + m) : 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (js[u] < 0) break;  // warp-uniform
                    float pk = 0.f, pq = 0.f;
#pragma unroll
                    for (int r = 0; r < EPL; ++r) {
                        pk = fmaf(kr[r], kj[u][r], pk);
                        pq = fmaf(qr[r], kj[u][r], pq);
                    }
                    pk = warp_sum(pk);
                    pq = warp_sum(pq);
                    if (lane == 0) {
                        const int ja = js[u], l = dep[ja] - 1;
                        const float dec = expf(gam[i] - gam[ja]);
                        RK[i * MD + l] = bet[i] * dec * pk;
                        RQ[i * MD + l] = dec * pq;
                        PTH[i * MD + l] = ja;
                    }
                }
            }
        }
        __syncthreads();
    }

    // ---- phase 2: level-ordered forward substitution and outputs ----------
    for (int d = 1; d <= maxd; ++d) {
        for (int idx = start[d] + warp; idx < start[d + 1]; idx += kWarps) {
            const int i = order[idx];
            if (raw) {
                // the pair coefficients are in the tables: combine along the path,
                // from the parent up
                const float gi = gam[i];
                float acc_u = lane < SW ? Ub[i * SW + lane] : 0.f;
                float acc_o = 0.f;
                const int *pi_row = PTH + i * MD;
                const float *rk = RK + i * MD, *rq = RQ + i * MD;
                for (int l = dep[i] - 2; l >= 0; --l) {
                    const int j = pi_row[l];
                    const float uj = lane < SW ? Ub[j * SW + lane] : 0.f;
                    acc_u -= rk[l] * uj;
                    acc_o += rq[l] * uj;
                }
                if (lane < SW) {
                    Ub[i * SW + lane] = acc_u;
                    const float o = p.scale * (expf(gi) * Zb[i * SW + lane] + acc_o + SELF[i] * acc_u);
                    store_f(op, ((int64_t)(lo + i) * p.hv_n + h) * p.dv + slab * SW + lane, o);
                }
                continue;
            }
            const int64_t krow = ((int64_t)(lo + i) * p.hk_n + hk) * DK;
            float kr[EPL], qr[EPL];
#pragma unroll
            for (int r = 0; r < EPL; ++r) {
                const int m = lane + 32 * r;
                kr[r] = m < DK ? load_f(kp, krow + m) : 0.f;
                qr[r] = m < DK ? load_f(qp, krow + m) : 0.f;
            }
            const float gi = gam[i], bi = bet[i];
            float acc_u = lane < SW ? Ub[i * SW + lane] : 0.f;
            float acc_o = 0.f;
            // ancestors from the parent up, four at a time: their key rows are
            // requested together, so a path costs one memory latency per four
            // ancestors (the accumulation order is unchanged)
            constexpr int kBatch = 4;
            for (int j = par[i]; j >= 0;) {
                int js[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    js[u] = j;
                    if (j >= 0) j = par[j];
                }
                float kj[kBatch][EPL];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int64_t jrow = ((int64_t)(lo + max(js[u], 0)) * p.hk_n + hk) * DK;
#pragma unroll
                    for (int r = 0; r < EPL; ++r) {
                        const int m = lane + 32 * r;
                        kj[u][r] = (js[u] >= 0 && m < DK) ? load_f(kp, jrow + m) : 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int ja = js[u];
                    if (ja < 0) break;  // warp-uniform
                    float pk = 0.f, pq = 0.f;
#pragma unroll
                    for (int r = 0; r < EPL; ++r) {
                        pk = fmaf(kr[r], kj[u][r], pk);
                        pq = fmaf(qr[r], kj[u][r], pq);
                    }
                    pk = warp_sum(pk);
                    pq = warp_sum(pq);
                    const float dec = expf(gi - gam[ja]);
                    const float uj = lane < SW ? Ub[ja * SW + lane] : 0.f;
                    acc_u -= bi * dec * pk * uj;
                    acc_o += dec * pq * uj;
                }
            }
            float self = 0.f;
#pragma unroll
            for (int r = 0; r < EPL; ++r) self = fmaf(qr[r], kr[r], self);
            self = warp_sum(self);
            if (lane < SW) {
                Ub[i * SW + lane] = acc_u;
                const float o = p.scale * (expf(gi) * Zb[i * SW + lane] + acc_o + self * acc_u);
                store_f(op, ((int64_t)(lo + i) * p.hv_n + h) * p.dv + slab * SW + lane, o);
            }
        }
        __syncthreads();
    }
}

template <typename Tin, typename Tout, int DK>
cudaError_t launch_typed(const SimtParams &p, int batch, cudaStream_t stream) {
    const SmemLayout L = smem_layout(p.max_nodes, p.sw, DK, p.md);
    const size_t bytes = sizeof(float) * (size_t)L.floats + sizeof(int) * (size_t)L.ints;
    auto kern = verify_simt_kernel<Tin, Tout, DK>;
    static int have[16];  // one per template instance
    cudaError_t e = ensure_smem(kern, (int)bytes, have);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.dv / p.sw) * (unsigned)batch, p.hv_n);
    kern<<<grid, kThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_dk(const SimtParams &p, int dk, int batch, cudaStream_t stream) {
    switch (dk) {
        case 16: return launch_typed<Tin, Tout, 16>(p, batch, stream);
        case 32: return launch_typed<Tin, Tout, 32>(p, batch, stream);
        case 64: return launch_typed<Tin, Tout, 64>(p, batch, stream);
        case 128: return launch_typed<Tin, Tout, 128>(p, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_verify_simt(const gdn_verify_args &a, cudaStream_t stream) {
    SimtParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.dv = a.d_v; p.max_nodes = a.max_nodes;
    p.sw = a.d_v < 32 ? a.d_v : 32;
    // phase 1b for small trees: path length bound = the declared depth, else the node count
    const int md = a.max_depth > 0 ? std::min(a.max_depth, a.max_nodes) : a.max_nodes;
    p.md = (int64_t)a.max_nodes * md <= kRawMax ? md : 0;
    p.scale = a.scale;
    p.offsets = a.node_offsets; p.parent = a.parent; p.depth = a.depth;
    p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.o = a.o; p.status = a.dev_status;
    const bool in_bf = a.qkv_dtype == GDN_BF16, out_bf = a.out_dtype == GDN_BF16;
    if (in_bf && out_bf) return launch_dk<__nv_bfloat16, __nv_bfloat16>(p, a.d_k, a.batch, stream);
    if (in_bf) return launch_dk<__nv_bfloat16, float>(p, a.d_k, a.batch, stream);
    if (out_bf) return launch_dk<float, __nv_bfloat16>(p, a.d_k, a.batch, stream);
    return launch_dk<float, float>(p, a.d_k, a.batch, stream);
}

}  // namespace gdn
