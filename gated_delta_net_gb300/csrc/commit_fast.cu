// commit_fast.cu -- delayed state commit for d_k = d_v = 128 and accepted paths of
// at most 16 nodes (sm_103a).
//
// "Trees from Marginals" (gist.science Technical Summary, section 3, Solution,
// last bullet): the state is committed in the next iteration along the accepted
// branch only.  For the accepted path p_1..p_L (gamma_t = sum of g over p_1..p_t)
//     u_t = beta_t (v_t - e^gamma_t S0 k_t) - sum_{s<t} beta_t e^(gamma_t - gamma_s) (k_t . k_s) u_s
//     S_new = e^gamma_L S0 + sum_t e^(gamma_L - gamma_t) u_t k_t^T
// which equals running the gated delta rule along the path.
//
// One block per (request, value head).  The 64 KB fp32 state tile arrives by
// TMA (128-byte swizzle, four 32-column boxes), each thread keeps a 2-row x
// 32-column register tile of it, and S_new leaves through the same shared
// memory by TMA store; the tile is read before anything is written, so S_new
// may alias S0.  All arithmetic is fp32: per row, W_t = S0 k_t (reduced over the
// four column quarters with shuffles), the chain solve for u, then the rank-L
// update.  The path's keys and values are staged in shared memory.
#include "internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kT = 256;
constexpr int kD = 128;
constexpr int kMaxPath = 16;
constexpr int kKPad = 36;  // floats per key quarter (32 + 4): quarters land on distinct banks

struct FastCommitParams {
    int hk_n, hv_n, total;
    const int32_t *offsets, *parent, *poff, *pidx;
    const void *k, *v;
    const float *g, *beta;
    int32_t *status;
};

struct alignas(16) CommitShared {
    float tile[kD * kD];                  // state tile, 4 x [128 rows][32 floats], 128B swizzle
    float kp[kMaxPath][4][kKPad];         // path keys by column quarter
    float vp[kMaxPath][kD];               // path values
    float coef[kMaxPath][kMaxPath];       // beta_t e^(gamma_t - gamma_s) (k_t . k_s), s < t
    float bet[kMaxPath], egam[kMaxPath], fdec[kMaxPath], gam[kMaxPath];
    int pn[kMaxPath];
    uint64_t bar;
    int bad;
};

// Offset (in floats) of element (row, col) of the state tile: column quarter
// q = col / 32 is a [128][32] box whose 16-byte chunks are permuted by row mod 8.
__device__ __forceinline__ int tile_index(int row, int col) {
    return (col >> 5) * (kD * 32) + row * 32 + ((((col & 31) >> 2) ^ (row & 7)) << 2) + (col & 3);
}

template <typename Tin>
__global__ void __launch_bounds__(kT, 2)
commit_fast_kernel(const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmSN,
                   FastCommitParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    CommitShared &sh = *reinterpret_cast<CommitShared *>(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hv = blockIdx.x % p.hv_n, b = blockIdx.x / p.hv_n;
    const int hk = hv / (p.hv_n / p.hk_n);
    const int lo = p.offsets[b];
    const int n = p.offsets[b + 1] - lo;
    const int pa = p.poff[b];
    const int L = p.poff[b + 1] - pa;
    const int tile_row = blockIdx.x * kD;  // first row of this (request, head) in the [B*Hv*128][128] view
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (tid == 0) flag(p.status, GDN_DEV_INTERNAL);
        return;
    }
    if (L < 0 || L > kMaxPath || L > n || lo < 0 || lo + n > p.total) {
        if (tid == 0) flag(p.status, L > kMaxPath && L <= n ? GDN_DEV_TOO_DEEP : GDN_DEV_BAD_PATH);
        return;
    }
    if (tid == 0) {
        mbar_init(&sh.bar, 1);
        fence_mbar_init();
        sh.bad = 0;
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&sh.bar, kD * kD * 4);
        for (int q = 0; q < 4; ++q) tma_load_2d(sh.tile + q * kD * 32, &tmS0, &sh.bar, q * 32, tile_row);
    }

    // path: validation, keys, values, gates
    if (tid < L) {
        const int node = p.pidx[pa + tid];
        const int expect = tid == 0 ? -1 : p.pidx[pa + tid - 1];
        if (node < 0 || node >= n || p.parent[lo + node] != expect) atomicOr(&sh.bad, 1);
        sh.pn[tid] = node;
    }
    __syncthreads();
    const bool bad = sh.bad != 0;
    if (!bad) {
        const Tin *kp = static_cast<const Tin *>(p.k);
        const Tin *vp = static_cast<const Tin *>(p.v);
        for (int e = tid; e < L * kD; e += kT) {
            const int t = e >> 7, m = e & (kD - 1);
            const int64_t node = lo + sh.pn[t];
            sh.kp[t][m >> 5][m & 31] = load_f(kp, (node * p.hk_n + hk) * kD + m);
            sh.vp[t][m] = load_f(vp, (node * p.hv_n + hv) * kD + m);
        }
        if (tid < L) {
            const int64_t node = lo + sh.pn[tid];
            sh.gam[tid] = p.g[node * p.hv_n + hv];
            sh.bet[tid] = p.beta[node * p.hv_n + hv];
        }
    }
    __syncthreads();
    if (tid == 0 && !bad) {
        float acc = 0.f;
        for (int t = 0; t < L; ++t) {
            acc += sh.gam[t];
            sh.gam[t] = acc;
            sh.egam[t] = expf(acc);
        }
        for (int t = 0; t < L; ++t) sh.fdec[t] = expf(acc - sh.gam[t]);
    }
    __syncthreads();
    // chain coefficients: one warp per (t, s) pair
    if (!bad) {
        for (int pr = warp; pr < L * (L - 1) / 2; pr += kT / 32) {
            int t = 1, base = 0;
            while (base + t <= pr) { base += t; ++t; }
            const int s = pr - base;
            float d = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) d = fmaf(sh.kp[t][r][lane], sh.kp[s][r][lane], d);
            d = warp_sum(d);
            if (lane == 0) sh.coef[t][s] = sh.bet[t] * expf(sh.gam[t] - sh.gam[s]) * d;
        }
    }
    bool ok = mbar_wait(&sh.bar, 0);
    __syncthreads();
    if (bad) {
        if (tid == 0) flag(p.status, GDN_DEV_BAD_PATH);
        return;
    }

    // register tile: rows r0 = 16 warp + rr and r0 + 8, columns 32 q .. 32 q + 31
    const int q = lane & 3, rr = lane >> 2;
    const int rows[2] = {warp * 16 + rr, warp * 16 + 8 + rr};
    float s[2][32];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 x = *reinterpret_cast<const float4 *>(sh.tile + tile_index(rows[h], q * 32 + c * 4));
            s[h][c * 4 + 0] = x.x; s[h][c * 4 + 1] = x.y; s[h][c * 4 + 2] = x.z; s[h][c * 4 + 3] = x.w;
        }

    // W_t = S0 k_t per row; then the chain solve in place: w -> u -> e^(gamma_L - gamma_t) u
    float w[2][kMaxPath];
#pragma unroll
    for (int t = 0; t < kMaxPath; ++t) {
        float a0 = 0.f, a1 = 0.f;
        if (t < L) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 kv = *reinterpret_cast<const float4 *>(&sh.kp[t][q][c * 4]);
                a0 = fmaf(s[0][c * 4 + 0], kv.x, a0); a0 = fmaf(s[0][c * 4 + 1], kv.y, a0);
                a0 = fmaf(s[0][c * 4 + 2], kv.z, a0); a0 = fmaf(s[0][c * 4 + 3], kv.w, a0);
                a1 = fmaf(s[1][c * 4 + 0], kv.x, a1); a1 = fmaf(s[1][c * 4 + 1], kv.y, a1);
                a1 = fmaf(s[1][c * 4 + 2], kv.z, a1); a1 = fmaf(s[1][c * 4 + 3], kv.w, a1);
            }
        }
        a0 += __shfl_xor_sync(0xffffffffu, a0, 1);
        a0 += __shfl_xor_sync(0xffffffffu, a0, 2);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
        w[0][t] = a0;
        w[1][t] = a1;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int t = 0; t < kMaxPath; ++t) {
            if (t < L) {
                float u = sh.bet[t] * (sh.vp[t][rows[h]] - sh.egam[t] * w[h][t]);
#pragma unroll
                for (int sidx = 0; sidx < t; ++sidx) u = fmaf(-sh.coef[t][sidx], w[h][sidx], u);
                w[h][t] = u;
            }
        }
#pragma unroll
        for (int t = 0; t < kMaxPath; ++t) w[h][t] = t < L ? w[h][t] * sh.fdec[t] : 0.f;
    }

    // S_new = e^gamma_L S0 + sum_t (e^(gamma_L - gamma_t) u_t) k_t^T, back into the tile
    const float eL = L > 0 ? sh.egam[L - 1] : 1.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float o0[4], o1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o0[e] = eL * s[0][c * 4 + e];
            o1[e] = eL * s[1][c * 4 + e];
        }
#pragma unroll
        for (int t = 0; t < kMaxPath; ++t) {
            if (t < L) {
                const float4 kv = *reinterpret_cast<const float4 *>(&sh.kp[t][q][c * 4]);
                o0[0] = fmaf(w[0][t], kv.x, o0[0]); o0[1] = fmaf(w[0][t], kv.y, o0[1]);
                o0[2] = fmaf(w[0][t], kv.z, o0[2]); o0[3] = fmaf(w[0][t], kv.w, o0[3]);
                o1[0] = fmaf(w[1][t], kv.x, o1[0]); o1[1] = fmaf(w[1][t], kv.y, o1[1]);
                o1[2] = fmaf(w[1][t], kv.z, o1[2]); o1[3] = fmaf(w[1][t], kv.w, o1[3]);
            }
        }
        *reinterpret_cast<float4 *>(sh.tile + tile_index(rows[0], q * 32 + c * 4)) = make_float4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<float4 *>(sh.tile + tile_index(rows[1], q * 32 + c * 4)) = make_float4(o1[0], o1[1], o1[2], o1[3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        for (int qq = 0; qq < 4; ++qq) tma_store_2d(&tmSN, sh.tile + qq * kD * 32, qq * 32, tile_row);
        bulk_commit();
        bulk_wait_read();
    }
    if (!ok && tid == 0) flag(p.status, GDN_DEV_TIMEOUT);
}

// fp32 [rows][128] viewed as a 2-D tensor; boxes of 32 columns x 128 rows, 128-byte swizzle
bool encode_state(CUtensorMap *map, const float *base, int64_t rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)kD};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool commit_fast_supported(const gdn_commit_args &a) {
    return a.d_k == kD && a.d_v == kD && a.max_path >= 1 && a.max_path <= kMaxPath && aligned16(a.S0) &&
           aligned16(a.S_new) && (int64_t)a.batch * a.n_v_heads * kD <= 2147483647LL &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_commit_fast(const gdn_commit_args &a, cudaStream_t stream) {
    const int64_t rows = (int64_t)a.batch * a.n_v_heads * kD;
    CUtensorMap tmS0, tmSN;
    if (!encode_state(&tmS0, a.S0, rows) || !encode_state(&tmSN, a.S_new, rows)) return cudaErrorInvalidValue;
    FastCommitParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.total = a.total_nodes;
    p.offsets = a.node_offsets; p.parent = a.parent; p.poff = a.path_offsets; p.pidx = a.path_idx;
    p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta; p.status = a.dev_status;
    const size_t bytes = sizeof(CommitShared);
    const dim3 grid((unsigned)a.batch * (unsigned)a.n_v_heads);
    cudaError_t e;
    if (a.qkv_dtype == GDN_BF16) {
        static int have[16];
        e = ensure_smem(commit_fast_kernel<__nv_bfloat16>, (int)bytes, have);
        if (e != cudaSuccess) return e;
        commit_fast_kernel<__nv_bfloat16><<<grid, kT, bytes, stream>>>(tmS0, tmSN, p);
    } else {
        static int have[16];
        e = ensure_smem(commit_fast_kernel<float>, (int)bytes, have);
        if (e != cudaSuccess) return e;
        commit_fast_kernel<float><<<grid, kT, bytes, stream>>>(tmS0, tmSN, p);
    }
    return cudaGetLastError();
}

}  // namespace gdn
