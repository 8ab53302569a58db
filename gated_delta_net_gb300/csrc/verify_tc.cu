// verify_tc.cu -- tcgen05/TMA tree verification for bf16 tokens, d_k = d_v = 128,
// trees of at most 128 nodes and depth at most 16 (sm_103a).
//
// Computes, for one (request, value head) per thread block, the masked
// triangular solve of "Trees from Marginals" (gist.science Technical Summary,
// section 3 "Rollback-Free Tree Verification for GDN"):
//     X = strict-ancestor mask * beta_i * D_ij * (K K^T),  Y = ancestor mask * D_ij * (Q K^T)
//     (I + X) U = R = beta * (V - e^gamma * K S0^T)
//     O = scale * (e^gamma * Q S0^T + Y U)
// with D_ij = exp(gamma_i - gamma_j), gamma the sum of g along each path.
// Because only ancestors interact and paths are at most 16 long, each node's
// row of P = Y (I + X)^-1 has at most 16 non-zeros and is found by a 16-step
// back substitution along the node's own path; then O = e^gamma Z + P R.
//
// Dense contractions run on the tensor cores (kind::f16, fp32 accumulate):
//   Gram   : K [K;Q]^T           A = K tile, B = [K;Q] tile (TMA, 128B swizzle)
//   S0 part: S0 [K;Q]^T = [W^T | Z^T]  the fp32 state enters as bf16 hi + lo
//            (S0 = hi + lo to ~2^-17 relative), so K S0^T and Q S0^T keep the
//            state's precision; the block converts it through a 2-slot ring.
//   Output : Z^T + R^T (e^-gamma' P)^T accumulated onto Z^T in tensor memory
//            (gamma' = max(gamma, -80) keeps e^-gamma' finite), then scaled by
//            e^gamma' per node in the epilogue.
// Tensor memory: 256 columns (Gram, then [W^T | Z^T]), so two blocks share an SM.
// The K|Q tile space is reused: V lands in its first k-block once the MMAs that
// read it are done, then R^T, then P, then the staged output.
// A node whose right-hand side row turns non-finite has that row replaced by
// zero in the output product and its subtree's outputs set to NaN, so
// non-finite values never leave their own branch.
#include <cudaTypedefs.h>

#include "internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kT = 256;           // threads per block
constexpr int kN = 128;           // tile rows: nodes (max_nodes <= 128)
constexpr int kD = 128;           // d_k = d_v
constexpr int kMaxDepth = 16;
constexpr int kSlots = 2;         // S0 conversion ring
constexpr int kChunks = kD / 16;  // one MMA k-step of S0 per chunk
constexpr float kGammaFloor = -80.f;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int OFF_KQ = 0;         // [2 k-blocks][256 rows (K then Q)][128 B], 128B swizzle
constexpr int OFF_LO = 0;         // first half of the K|Q space: V, then P
constexpr int OFF_HI = 32768;     // second half: R^T, then the staged output
constexpr int OFF_S0 = 65536;                           // kSlots x (hi 4 KB + lo 4 KB)
constexpr int OFF_X = OFF_S0 + kSlots * 8192;           // float [128][16]
constexpr int OFF_Y = OFF_X + kN * kMaxDepth * 4;       // float [128][16]
constexpr int OFF_MASK = OFF_Y + kN * kMaxDepth * 4;    // uint32 [128][4]
constexpr int OFF_PATH = OFF_MASK + kN * 4 * 4;         // uint8 [128][16]
constexpr int OFF_F = OFF_PATH + kN * kMaxDepth;        // float graw, gam, egt, eg, bet [128]
constexpr int OFF_I = OFF_F + 5 * kN * 4;               // int dep, par [128]; uint8 pflag [128]
constexpr int OFF_MISC = OFF_I + 2 * kN * 4 + kN;       // tmem slot, poison[4], err
constexpr int OFF_BAR = (OFF_MISC + 64 + 7) & ~7;
constexpr int kBars = 5 + 2 * kSlots;                   // kq, gram, s0, out, v, fill[], free[]
constexpr int kSmemBytes = OFF_BAR + kBars * 8 + 1024;  // + alignment slack

struct TcParams {
    int hk_n, hv_n, words, total;
    float scale;
    const int32_t *offsets, *parent, *depth;
    const uint32_t *mask;
    const float *g, *beta, *S0;
    void *o;
    int32_t *status;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Byte offset of element (row, k) in a K-major, 128-byte-swizzled bf16 tile of
// `rows` rows: k-blocks of 64 elements, rows of 128 bytes, 16-byte chunks
// permuted by (row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows) {
    return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                      (k & 7) * 2);
}

// Core-matrix ("interleaved", no swizzle) K-major offset of the 16-byte group
// (row, kh) of a 128-row x 16-column chunk: 8-row x 16-byte core matrices,
// K-adjacent core matrices 128 bytes apart, 8-row groups 256 bytes apart.
__device__ __forceinline__ uint32_t core_offset(int row, int kh) {
    return (uint32_t)((row >> 3) * 256 + kh * 128 + (row & 7) * 16);
}

template <typename Tout>
__global__ void __launch_bounds__(kT, 2)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmV, TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    float *Xs = reinterpret_cast<float *>(sm + OFF_X);
    float *Ys = reinterpret_cast<float *>(sm + OFF_Y);
    uint32_t *msk = reinterpret_cast<uint32_t *>(sm + OFF_MASK);
    uint8_t *path = sm + OFF_PATH;
    float *graw = reinterpret_cast<float *>(sm + OFF_F);
    float *gam = graw + kN, *egt = graw + 2 * kN, *eg = graw + 3 * kN, *bet = graw + 4 * kN;
    int *dep = reinterpret_cast<int *>(sm + OFF_I), *par = dep + kN;
    uint8_t *pflag = reinterpret_cast<uint8_t *>(par + kN);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    uint32_t *poison = tslot + 1;
    int *s_err = reinterpret_cast<int *>(tslot + 5);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_kq = bars, *bar_gram = bars + 1, *bar_s0 = bars + 2, *bar_out = bars + 3;
    uint64_t *bar_v = bars + 4, *bar_fill = bars + 5, *bar_free = bars + 5 + kSlots;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
    const int hv = blockIdx.x % p.hv_n, b = blockIdx.x / p.hv_n;
    const int hk = hv / (p.hv_n / p.hk_n);
    const int lo = p.offsets[b];
    const int n = p.offsets[b + 1] - lo;
    if (n <= 0) return;
    if (n > kN || lo < 0 || lo + n > p.total) {
        if (tid == 0) flag(p.status, n > kN ? GDN_DEV_TOO_MANY : GDN_DEV_BAD_DESC);
        return;
    }

    // ---- set-up: barriers, tensor memory, TMA of the K and Q tiles --------
    if (tid == 0) {
        mbar_init(bar_kq, 1);
        mbar_init(bar_gram, 1);
        mbar_init(bar_s0, 1);
        mbar_init(bar_out, 1);
        mbar_init(bar_v, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&bar_fill[s], kT);
            mbar_init(&bar_free[s], 1);
        }
        fence_mbar_init();
        *s_err = 0;
    }
    if (tid < 4) poison[tid] = 0u;
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    const int nbox = (n + 31) >> 5;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_kq, (uint32_t)(2 * 2 * nbox * 4096));
        for (int kb = 0; kb < 2; ++kb)
            for (int r = 0; r < nbox; ++r) {
                tma_load_3d(sm + OFF_KQ + kb * 32768 + r * 4096, &tmK, bar_kq, kb * 64, hk, lo + 32 * r);
                tma_load_3d(sm + OFF_KQ + kb * 32768 + (128 + 32 * r) * 128, &tmQ, bar_kq, kb * 64, hk,
                            lo + 32 * r);
            }
    }

    // ---- S0 prefetch: thread -> (row m, half kh); chunk c = columns [16c, 16c+16)
    const float *S0t = p.S0 + ((int64_t)b * p.hv_n + hv) * (kD * kD);
    const int m_row = tid >> 1, m_half = tid & 1;
    const float *s0row = S0t + m_row * kD + m_half * 8;
    float4 s0r[4][2];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        s0r[c][0] = __ldg(reinterpret_cast<const float4 *>(s0row + 16 * c));
        s0r[c][1] = __ldg(reinterpret_cast<const float4 *>(s0row + 16 * c + 4));
    }

    // ---- tree metadata (thread i = node i) ---------------------------------
    if (tid < kN) {
        const int i = tid;
        if (i < n) {
            par[i] = p.parent[lo + i];
            dep[i] = p.depth[lo + i];
#pragma unroll
            for (int w = 0; w < 4; ++w)
                msk[i * 4 + w] = w < p.words ? p.mask[(int64_t)(lo + i) * p.words + w] : 0u;
            graw[i] = p.g[(int64_t)(lo + i) * p.hv_n + hv];
            bet[i] = p.beta[(int64_t)(lo + i) * p.hv_n + hv];
        } else {
            par[i] = -1;
            dep[i] = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) msk[i * 4 + w] = 0u;
            graw[i] = 0.f;
            bet[i] = 0.f;
        }
        pflag[i] = 0;
    }
    __syncthreads();
    if (tid < n) {
        const int i = tid, pi = par[i];
        int e = 0;
        if (pi < -1 || pi >= i) {
            e = GDN_DEV_BAD_TREE;
        } else {
            const int want = pi < 0 ? 1 : dep[pi] + 1;
            bool same = dep[i] == want;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t expect = (pi < 0 ? 0u : msk[pi * 4 + w]) | ((i >> 5) == w ? 1u << (i & 31) : 0u);
                same = same && msk[i * 4 + w] == expect;
            }
            if (!same) e = GDN_DEV_BAD_DESC;
            else if (dep[i] > kMaxDepth) e = GDN_DEV_TOO_DEEP;
        }
        if (e) atomicOr(s_err, e);
    }
    __syncthreads();
    if (*s_err) {
        if (tid == 0) {
            flag(p.status, *s_err);
            mbar_wait(bar_kq, 0);  // no TMA may land after the block exits
        }
        __syncthreads();
        tc_fence_before();
        if (warp == 0) tmem_dealloc(tmem, 256);
        return;
    }

    // ---- paths (the set bits of each mask row, root first) and gamma -------
    const int myd = tid < n ? dep[tid] : 0;
    if (tid < n) {
        const int i = tid;
        float acc = 0.f;
        int l = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t word = msk[i * 4 + w];
            while (word) {
                const int j = w * 32 + __ffs(word) - 1;
                word &= word - 1;
                path[i * kMaxDepth + l++] = (uint8_t)j;
                acc += graw[j];
            }
        }
        gam[i] = acc;
        egt[i] = expf(acc);
        eg[i] = expf(fmaxf(acc, kGammaFloor));
    } else if (tid < kN) {
        gam[tid] = 0.f;
        egt[tid] = 0.f;
        eg[tid] = 1.f;
    }

    // ---- S0 chunks 0, 1 -> ring slots (bf16 hi + lo, core-matrix layout) ---
    auto convert = [&](int c, const float4 (&x)[2]) {
        uint8_t *slot = sm + OFF_S0 + (c % kSlots) * 8192;
        const float f[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
        float h[8], l[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            h[e] = __bfloat162float(__float2bfloat16_rn(f[e]));
            l[e] = f[e] - h[e];
        }
        const uint4 hv4 = make_uint4(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]), pack_bf16(h[4], h[5]),
                                     pack_bf16(h[6], h[7]));
        const uint4 lv4 = make_uint4(pack_bf16(l[0], l[1]), pack_bf16(l[2], l[3]), pack_bf16(l[4], l[5]),
                                     pack_bf16(l[6], l[7]));
        const uint32_t off = core_offset(m_row, m_half);
        *reinterpret_cast<uint4 *>(slot + off) = hv4;
        *reinterpret_cast<uint4 *>(slot + 4096 + off) = lv4;
        fence_proxy_async_smem();
        mbar_arrive(&bar_fill[c % kSlots]);
    };
    auto reload = [&](int c) {  // chunk c into the registers chunk c - 4 just vacated
        s0r[c & 3][0] = __ldg(reinterpret_cast<const float4 *>(s0row + 16 * c));
        s0r[c & 3][1] = __ldg(reinterpret_cast<const float4 *>(s0row + 16 * c + 4));
    };
    convert(0, s0r[0]);
    reload(4);
    convert(1, s0r[1]);
    reload(5);

    const uint32_t id_n256 = idesc_bf16_f32(128, 256), id_n128 = idesc_bf16_f32(128, 128);
    bool ok = true;

    // ---- Gram: K [K;Q]^T -> tensor memory columns [0, 256) -----------------
    if (tid == 0) {
        ok = mbar_wait(bar_kq, 0);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a = smem_u32(sm + OFF_KQ + (ks >> 2) * 32768 + (ks & 3) * 32);
            const uint64_t d = smem_desc(a, 16, 1024, 2);
            mma_bf16(tmem, d, d, id_n256, ks > 0);
        }
        mma_commit(bar_gram);
    }
    __syncthreads();  // gam[] complete for every node

    // this row's decay factors D_i,path[l] = exp(gamma_i - gamma_path[l])
    float dec[kMaxDepth];
#pragma unroll
    for (int l = 0; l < kMaxDepth; ++l)
        dec[l] = (tid < n && l < myd) ? expf(gam[tid] - gam[path[tid * kMaxDepth + l]]) : 0.f;

    ok = mbar_wait(bar_gram, 0) && ok;
    tc_fence_after();

    // scatter: lane a holds k_a.k_i (cols 0..127) and k_a.q_i (cols 128..255);
    // node a writes its entries into the rows of its descendants i.  The bits
    // "a is an ancestor of i" for the 32 columns of a chunk are transposed from
    // the mask rows with one ballot per lane.
    {
        const int a = quad * 32 + lane;
        const bool kpart = warp < 4;
        const int da = a < n ? dep[a] : 0;
        float *dst = kpart ? Xs : Ys;
        for (int cc = quad; cc < 4; ++cc) {
            float v[32];
            tmem_ld32(tmem + lane_base + (kpart ? 0 : 128) + cc * 32, v);
            const uint32_t wc = msk[(cc * 32 + lane) * 4 + quad];
            uint32_t dm = 0u;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const uint32_t bx = __ballot_sync(0xffffffffu, (wc >> x) & 1u);
                if (lane == x) dm = bx;
            }
            if (!kpart || cc != quad) {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if ((dm >> c) & 1u) dst[(cc * 32 + c) * kMaxDepth + da - 1] = v[c];
            } else {
                dm &= ~(1u << lane);  // X is strictly lower: skip the diagonal
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if ((dm >> c) & 1u) dst[(cc * 32 + c) * kMaxDepth + da - 1] = v[c];
            }
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- S0 part, chunks 0 and 1 --------------------------------------------
    auto issue_s0 = [&](int c) {
        const int s = c % kSlots;
        const bool w = mbar_wait(&bar_fill[s], (uint32_t)((c / kSlots) & 1));
        tc_fence_after();
        const uint64_t bdesc = smem_desc(smem_u32(sm + OFF_KQ + (c >> 2) * 32768 + (c & 3) * 32), 16, 1024, 2);
        const uint32_t slot = smem_u32(sm + OFF_S0 + s * 8192);
        mma_bf16(tmem, smem_desc(slot, 128, 256, 0), bdesc, id_n256, c > 0);
        mma_bf16(tmem, smem_desc(slot + 4096, 128, 256, 0), bdesc, id_n256, true);
        mma_commit(&bar_free[s]);
        return w;
    };
    if (tid == 0) {
        tc_fence_after();
        ok = issue_s0(0) && ok;
        ok = issue_s0(1) && ok;
    }

    // ---- X, Y scaling and P = Y (I + X)^-1 along each path -------------------
    // Row i of P has non-zeros only on i's path; it overwrites row i of Ys.
    if (tid < n) {
        const int i = tid;
        const float bi = bet[i];
#pragma unroll
        for (int l = 0; l < kMaxDepth; ++l)
            if (l < myd - 1) Xs[i * kMaxDepth + l] *= bi * dec[l];
    }
    __syncthreads();
    if (tid < n) {
        const int i = tid;
        float P[kMaxDepth];
#pragma unroll
        for (int l = 0; l < kMaxDepth; ++l) P[l] = l < myd ? dec[l] * Ys[i * kMaxDepth + l] : 0.f;
#pragma unroll
        for (int a = kMaxDepth - 1; a >= 1; --a) {
            if (a < myd) {
                const float pa = P[a];
                const float *xr = Xs + path[i * kMaxDepth + a] * kMaxDepth;
#pragma unroll
                for (int l = 0; l < a; ++l) P[l] = fmaf(-pa, xr[l], P[l]);
            }
        }
        const float inv = 1.f / eg[i];
#pragma unroll
        for (int l = 0; l < kMaxDepth; ++l) Ys[i * kMaxDepth + l] = P[l] * inv;
    }

    // ---- S0 chunks 2..7 through the ring; V lands once k-steps 0..3 are done
#pragma unroll
    for (int c = 2; c < kChunks; ++c) {
        const int s = c % kSlots;
        ok = mbar_wait(&bar_free[s], (uint32_t)(((c / kSlots) - 1) & 1)) && ok;
        if (c == 5 && tid == 0) {  // MMA of chunk 3 complete: the first k-block of K|Q is free
            mbar_arrive_expect_tx(bar_v, (uint32_t)(2 * nbox * 4096));
            for (int h = 0; h < 2; ++h)
                for (int r = 0; r < nbox; ++r)
                    tma_load_3d(sm + OFF_LO + h * 16384 + r * 4096, &tmV, bar_v, h * 64, hv, lo + 32 * r);
        }
        convert(c, s0r[c & 3]);
        if (c + 4 < kChunks) reload(c + 4);
        if (tid == 0) ok = issue_s0(c) && ok;
    }
    if (tid == 0) mma_commit(bar_s0);

    ok = mbar_wait(bar_s0, 0) && ok;
    ok = mbar_wait(bar_v, 0) && ok;
    tc_fence_after();

    // ---- R^T (bf16, K-major 128B swizzle) from W^T and V, poison non-finite rows
    const int nn = quad * 32 + lane;
    const int jbase = warp < 4 ? 0 : 64;
    {
        const __nv_bfloat16 *vs = reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_LO) + (nn >> 6) * 8192 + (nn & 63);
#pragma unroll
        for (int jc = 0; jc < 2; ++jc) {
            float w[32];
            tmem_ld32(tmem + lane_base + jbase + jc * 32, w);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int j = jbase + jc * 32 + c;
                float x = 0.f;
                if (j < n) {
                    x = bet[j] * (__bfloat162float(vs[j * 64]) - egt[j] * w[c]);
                    if (!isfinite(x)) {
                        atomicOr(&poison[j >> 5], 1u << (j & 31));
                        x = 0.f;
                    }
                }
                w[c] = x;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j0 = jbase + jc * 32 + q * 8;
                const uint4 val = make_uint4(pack_bf16(w[q * 8 + 0], w[q * 8 + 1]), pack_bf16(w[q * 8 + 2], w[q * 8 + 3]),
                                             pack_bf16(w[q * 8 + 4], w[q * 8 + 5]), pack_bf16(w[q * 8 + 6], w[q * 8 + 7]));
                *reinterpret_cast<uint4 *>(sm + OFF_HI + sw128_offset(nn, j0, kN)) = val;
            }
        }
    }
    fence_proxy_async_smem();
    __syncthreads();  // R^T written; V no longer read

    // ---- P rows (B operand, K-major 128B swizzle): zero row, then its path ---
    if (tid < kN) {
        const int i = tid;
        uint8_t *prow = sm + OFF_LO;
#pragma unroll
        for (int q = 0; q < 16; ++q)
            *reinterpret_cast<uint4 *>(prow + sw128_offset(i, q * 8, kN)) = make_uint4(0u, 0u, 0u, 0u);
        if (i < n) {
            bool hit = false;
#pragma unroll
            for (int w = 0; w < 4; ++w) hit |= (msk[i * 4 + w] & poison[w]) != 0u;
            pflag[i] = hit ? 1 : 0;
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l)
                if (l < myd)
                    *reinterpret_cast<__nv_bfloat16 *>(prow + sw128_offset(i, path[i * kMaxDepth + l], kN)) =
                        __float2bfloat16_rn(Ys[i * kMaxDepth + l]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- output: Z^T += R^T (e^-gamma' P)^T ---------------------------------
    if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = smem_desc(smem_u32(sm + OFF_HI + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
            const uint64_t bd = smem_desc(smem_u32(sm + OFF_LO + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
            mma_bf16(tmem + 128, ad, bd, id_n128, true);
        }
        mma_commit(bar_out);
    }
    ok = mbar_wait(bar_out, 0) && ok;
    tc_fence_after();

    // ---- epilogue: o[i][n] = scale * e^gamma'_i * acc[n][i], staged through
    // shared memory (rows of 128 outputs, 16-byte chunks xor-permuted by row)
    // for 16-byte global stores
    constexpr int kRowBytes = kD * (int)sizeof(Tout);
    uint8_t *stage = sm + OFF_KQ;
#pragma unroll
    for (int ic = 0; ic < 2; ++ic) {
        float z[32];
        tmem_ld32(tmem + lane_base + 128 + jbase + ic * 32, z);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int i = jbase + ic * 32 + c;
            const float val = pflag[i] ? __int_as_float(0x7fc00000) : p.scale * eg[i] * z[c];
            const int byte = nn * (int)sizeof(Tout);
            Tout *dst = reinterpret_cast<Tout *>(stage + i * kRowBytes + ((((byte >> 4) ^ (i & 7))) << 4) + (byte & 15));
            store_f(dst, 0, val);
        }
    }
    tc_fence_before();
    __syncthreads();
    {
        const int i = tid >> 1, half = tid & 1;
        if (i < n) {
            uint8_t *gdst = static_cast<uint8_t *>(p.o) + ((int64_t)(lo + i) * p.hv_n + hv) * kRowBytes;
#pragma unroll
            for (int q = 0; q < kRowBytes / 32; ++q) {
                const int chunk = half * (kRowBytes / 32) + q;
                const uint4 val = *reinterpret_cast<const uint4 *>(stage + i * kRowBytes + ((chunk ^ (i & 7)) << 4));
                *reinterpret_cast<uint4 *>(gdst + chunk * 16) = val;
            }
        }
    }
    if (!ok) flag(p.status, GDN_DEV_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [T][H][128] bf16 viewed as a 3-D tensor (d, head, token); boxes of 64 x 1 x 32.
bool encode_tokens(CUtensorMap *map, const void *base, int heads, int total, bool swizzle) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
    cuuint32_t box[3] = {64, 1, 32};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool verify_tc_supported(const gdn_verify_args &a) {
    return a.qkv_dtype == GDN_BF16 && a.d_k == kD && a.d_v == kD && a.max_nodes <= kN &&
           a.max_depth >= 1 && a.max_depth <= kMaxDepth && a.total_nodes > 0 && aligned16(a.q) &&
           aligned16(a.k) && aligned16(a.v) && aligned16(a.S0) && aligned16(a.o) && get_encoder() != nullptr;
}

cudaError_t launch_verify_tc(const gdn_verify_args &a, cudaStream_t stream) {
    CUtensorMap tmK, tmQ, tmV;
    if (!encode_tokens(&tmK, a.k, a.n_k_heads, a.total_nodes, true) ||
        !encode_tokens(&tmQ, a.q, a.n_k_heads, a.total_nodes, true) ||
        !encode_tokens(&tmV, a.v, a.n_v_heads, a.total_nodes, false))
        return cudaErrorInvalidValue;
    TcParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.words = a.mask_words < 4 ? a.mask_words : 4;
    p.total = a.total_nodes; p.scale = a.scale;
    p.offsets = a.node_offsets; p.parent = a.parent; p.depth = a.depth; p.mask = a.anc_mask;
    p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.o = a.o; p.status = a.dev_status;
    const dim3 grid((unsigned)a.batch * (unsigned)a.n_v_heads);
    cudaError_t e;
    if (a.out_dtype == GDN_BF16) {
        e = cudaFuncSetAttribute(verify_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e != cudaSuccess) return e;
        verify_tc_kernel<__nv_bfloat16><<<grid, kT, kSmemBytes, stream>>>(tmK, tmQ, tmV, p);
    } else {
        e = cudaFuncSetAttribute(verify_tc_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        verify_tc_kernel<float><<<grid, kT, kSmemBytes, stream>>>(tmK, tmQ, tmV, p);
    }
    return cudaGetLastError();
}

}  // namespace gdn
