// verify_tc.cu -- tcgen05/TMA tree verification for bf16 tokens, d_k = d_v = 128,
// trees of at most 128 nodes and depth at most 16 (sm_103a).
//
// Computes, for each (request, value head) work item, the masked triangular
// solve of "Trees from Marginals" (gist.science Technical Summary,
// section 3 "Rollback-Free Tree Verification for GDN"):
//     X = strict-ancestor mask * beta_i * D_ij * (K K^T),  Y = ancestor mask * D_ij * (Q K^T)
//     (I + X) U = R = beta * (V - e^gamma * K S0^T)
//     O = scale * (e^gamma * Q S0^T + Y U)
// with D_ij = exp(gamma_i - gamma_j), gamma the sum of g along each path.
// Because only ancestors interact and paths are at most 16 long, each node's
// row of P = Y (I + X)^-1 has at most 16 non-zeros and is found by a 16-step
// back substitution along the node's own path; then O = e^gamma Z + P R.
//
// Dense contractions run on the tensor cores (kind::f16, fp32 accumulate);
// tensor-memory lane = tree node throughout:
//   Gram   : K [K;Q]^T                A = K tile, B = [K;Q] tile (TMA, 128B swizzle)
//   S0 part: W = K S0^T, Z = Q S0^T   B = S0 rounded to bf16 like the tokens
//   Output : Z += (e^-gamma' P) R     A = P rows, B = R rows (MN-major);
//            gamma' = max(gamma, -80) keeps e^-gamma' finite; the epilogue scales
//            row i by e^gamma'_i, so O = e^gamma' Z + P R.
// Tensor memory: 256 columns (Gram, then [W | Z]), so two blocks share an SM.
//
// Warp roles, handing off through mbarriers rather than block-wide barriers:
//   warps 0-3 ("tree"):  node metadata, paths, gamma; scatter of the Gram into
//                        per-node ancestor rows (X and Y); X scaling; P; P rows.
//   warps 4-7 ("state"): S0 conversion; right-hand side R rows; epilogue.
//   thread 128 issues the TMA copies and the S0 and output MMAs, thread 0 the Gram.
// The grid is persistent (two blocks per SM); a block walks its (request, value
// head) items.  The next item's tree metadata is built during the current
// item's right-hand side and epilogue, its K/Q tiles load once the output MMA
// has consumed P and R, and its S0 conversion follows the epilogue (whose
// staged rows occupy the S0 space), overlapping its own Gram and scatters.
// Every mbarrier completes once per item, so waits use the item's parity.
// A node whose right-hand side row turns non-finite has that row replaced by
// zero in the output product and its subtree's outputs set to NaN, so
// non-finite values never leave their own branch.
// Launched as the dependent of a commit that writes the state (programmatic
// dependent launch), the kernel starts on the SMs the commit frees: only the
// state warps' first state read waits for the commit grid to finish.
#include <cuda_fp16.h>

#include <algorithm>
#include "internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kT = 256;           // threads per block
constexpr int kN = 128;           // tile rows: nodes (max_nodes <= 128)
constexpr int kD = 128;           // d_k = d_v
constexpr int kMaxDepth = 16;
constexpr float kGammaFloor = -80.f;

// shared-memory layout (bytes from the dynamic base, which is 1024-aligned)
constexpr int OFF_KQ = 0;                               // [2 k-blocks][256 rows (K, Q)][128 B]
constexpr int OFF_RB = 0;                               // reuse: R [j][n], MN-major B operand
constexpr int OFF_PA = 32768;                           // reuse: e^-gamma' P [i][j], A operand
constexpr int OFF_S0 = 65536;                           // S0 bf16 [2 k-blocks][128 rows][128 B]
constexpr int OFF_X = OFF_S0 + 32768;                   // half [128][16] raw k.k, then X
constexpr int OFF_Y = OFF_X + kN * kMaxDepth * 2;       // half [128][16] raw k.q
constexpr int OFF_MASK = OFF_Y + kN * kMaxDepth * 2;    // uint32 [128][4] ancestor, then descendant bits
constexpr int OFF_PATH = OFF_MASK + kN * 4 * 4;         // uint8 [128][16]
constexpr int OFF_F = OFF_PATH + kN * kMaxDepth;        // float graw, gam, egt, eg, bet [128]
constexpr int OFF_I = OFF_F + 5 * kN * 4;               // int dep, par [128]
constexpr int OFF_MISC = OFF_I + 2 * kN * 4;            // tmem slot, poisoned-node sets[2][4], errors[2]
constexpr int OFF_BAR = OFF_MISC + 64;
constexpr int kBars = 12;
constexpr int kSmemBytes = OFF_BAR + kBars * 8;

// mbarrier indices
enum { B_KQ, B_GRAM, B_DESC, B_TFREE, B_S0IN, B_S0, B_R, B_P, B_OUT, B_V, B_META, B_ZFREE };

struct TcParams {
    int hk_n, hv_n, words, total, items;
    float scale;
    const int32_t *offsets, *parent, *depth;
    const uint32_t *mask;
    const float *g, *beta, *S0;
    void *o;
    int32_t *status;
};

// one (request, value head) work item
struct Item {
    int idx, b, hv, hk, lo, n;
};

__device__ __forceinline__ bool item_ok(int lo, int n, int total) {
    return n > 0 && n <= kN && lo >= 0 && lo + n <= total;
}

__device__ __forceinline__ void set_item(const TcParams &p, int idx, int lo, int n, Item &it) {
    it.idx = idx;
    it.b = idx / p.hv_n;
    it.hv = idx % p.hv_n;
    it.hk = it.hv / (p.hv_n / p.hk_n);
    it.lo = lo;
    it.n = n;
}

// The first item at or after idx (stride `step`) whose request is non-empty and
// well placed; requests that are too large or reach past the node count are
// flagged (when `report`) and passed over.
__device__ bool find_item(const TcParams &p, int idx, int step, bool report, Item &it) {
    for (; idx < p.items; idx += step) {
        const int b = idx / p.hv_n;
        const int lo = __ldg(p.offsets + b);
        const int n = __ldg(p.offsets + b + 1) - lo;
        if (n == 0) continue;
        if (!item_ok(lo, n, p.total)) {
            if (report) flag(p.status, n > kN ? GDN_DEV_TOO_MANY : GDN_DEV_BAD_DESC);
            continue;
        }
        set_item(p, idx, lo, n, it);
        return true;
    }
    return false;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// element l (0..15) of 16 halves packed in two 16-byte words
__device__ __forceinline__ float half_at(const uint4 (&w)[2], int l) {
    const uint4 &v = w[l >> 3];
    const int k = (l & 7) >> 1;
    const uint32_t word = k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
    return __half2float(__ushort_as_half((unsigned short)((l & 1) ? (word >> 16) : (word & 0xFFFFu))));
}

__device__ __forceinline__ uint32_t pack_half(float a, float b) {
    return (uint32_t)__half_as_ushort(__float2half_rn(a)) | ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
}

// Byte offset of element (row, k) in a 128-row, 128-byte-swizzled bf16 tile:
// column blocks of 64 elements (16 KB apart), rows of 128 bytes, 16-byte
// chunks permuted by (row mod 8).  Used K-major (row = M/N index, k = K index)
// and, for R, MN-major (row = K index j, k = N index n).
__device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
    return (uint32_t)((k >> 6) * 16384 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <typename Tout>
__global__ void __launch_bounds__(kT, 2)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, TcParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __half *Xs = reinterpret_cast<__half *>(sm + OFF_X);
    __half *Ys = reinterpret_cast<__half *>(sm + OFF_Y);
    uint32_t *msk = reinterpret_cast<uint32_t *>(sm + OFF_MASK);  // ancestor rows, then descendant rows
    uint8_t *path = sm + OFF_PATH;
    float *graw = reinterpret_cast<float *>(sm + OFF_F);
    float *gam = graw + kN, *egt = graw + 2 * kN, *eg = graw + 3 * kN, *bet = graw + 4 * kN;
    int *dep = reinterpret_cast<int *>(sm + OFF_I), *par = dep + kN;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    uint32_t *pset = tslot + 1;                           // [parity][4]: nodes whose output is poisoned
    int *s_err = reinterpret_cast<int *>(tslot + 9);      // [parity]: descriptor errors of the item
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
    const bool tree = warp < 4;
    const int row = quad * 32 + lane;  // tensor-memory lane of this thread = a tree node
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const bool issuer = tid == 128;
    // a block that leaves early still waits for a preceding grid, so that this
    // grid never completes before the grid it depends on
    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0) flag(p.status, GDN_DEV_INTERNAL);
        griddep_wait();
        return;
    }
    Item cur;
    if (!find_item(p, blockIdx.x, gridDim.x, tid == 0, cur)) {
        griddep_wait();
        return;
    }

    // ---- set-up, once per block ---------------------------------------------
    if (tid == 0) {
        for (int k = 0; k < kBars; ++k) {
            const bool one = k == B_KQ || k == B_GRAM || k == B_S0 || k == B_OUT || k == B_V;
            mbar_init(&bar[k], k == B_TFREE ? 256u : one ? 1u : 128u);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;

    // K and Q tiles of an item (boxes of 32 nodes x 64 features, both k-blocks)
    auto issue_kq = [&](const Item &it) {
        const int nb = (it.n + 31) >> 5;
        mbar_arrive_expect_tx(&bar[B_KQ], (uint32_t)(2 * 2 * nb * 4096));
        for (int kb = 0; kb < 2; ++kb)
            for (int r = 0; r < nb; ++r) {
                tma_load_3d(sm + OFF_KQ + kb * 32768 + r * 4096, &tmK, &bar[B_KQ], kb * 64, it.hk, it.lo + 32 * r);
                tma_load_3d(sm + OFF_KQ + kb * 32768 + (128 + 32 * r) * 128, &tmQ, &bar[B_KQ], kb * 64, it.hk,
                            it.lo + 32 * r);
            }
    };

    // Tree warps: an item's node metadata, validation, paths, gamma and
    // descendant rows into shared memory, then arrive on B_DESC.
    auto tree_meta = [&](const Item &it, int pp) {
        const int i = tid;
        int pi = -1, di = 0;
        uint32_t mw[4] = {0u, 0u, 0u, 0u};
        float gr = 0.f, br = 0.f;
        if (i < it.n) {
            const int64_t gi = it.lo + i;
            pi = __ldg(p.parent + gi);
            di = __ldg(p.depth + gi);
#pragma unroll
            for (int w = 0; w < 4; ++w) mw[w] = w < p.words ? __ldg(p.mask + gi * p.words + w) : 0u;
            gr = __ldg(p.g + gi * p.hv_n + it.hv);
            br = __ldg(p.beta + gi * p.hv_n + it.hv);
        }
        named_sync(1, 128);  // the previous item's tree data is no longer read
        par[i] = pi;
        dep[i] = di;
#pragma unroll
        for (int w = 0; w < 4; ++w) msk[i * 4 + w] = mw[w];
        graw[i] = gr;
        bet[i] = br;
        // raw ancestor rows start at zero (entries past a node's depth stay zero)
        reinterpret_cast<uint4 *>(Xs + i * kMaxDepth)[0] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(Xs + i * kMaxDepth)[1] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(Ys + i * kMaxDepth)[0] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(Ys + i * kMaxDepth)[1] = make_uint4(0u, 0u, 0u, 0u);
        if (i < 4) pset[pp * 4 + i] = 0u;
        if (i == 0) s_err[pp] = 0;
        named_sync(1, 128);
        // validation: parent in [-1, i), depth and mask row consistent with the parent's
        if (i < it.n) {
            int e = 0;
            if (pi < -1 || pi >= i) {
                e = GDN_DEV_BAD_TREE;
            } else {
                const int want = pi < 0 ? 1 : dep[pi] + 1;
                bool same = di == want;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t expect = (pi < 0 ? 0u : msk[pi * 4 + w]) | ((i >> 5) == w ? 1u << (i & 31) : 0u);
                    same = same && mw[w] == expect;
                }
                if (!same) e = GDN_DEV_BAD_DESC;
                else if (di > kMaxDepth) e = GDN_DEV_TOO_DEEP;
            }
            if (e) atomicOr(&s_err[pp], e);
        }
        // paths (the set bits of each mask row, root first; at most kMaxDepth
        // entries even for a malformed row) and gamma
        if (i < it.n) {
            float acc = 0.f;
            int l = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t word = mw[w];
                while (word && l < kMaxDepth) {
                    const int j = w * 32 + __ffs(word) - 1;
                    word &= word - 1;
                    path[i * kMaxDepth + l++] = (uint8_t)j;
                    acc += graw[j];
                }
            }
            gam[i] = acc;
            egt[i] = expf(acc);
            eg[i] = expf(fmaxf(acc, kGammaFloor));
        } else {
            gam[i] = 0.f;
            egt[i] = 0.f;
            eg[i] = 1.f;
        }
        // mask rows become descendant rows: bit i of row a iff a is on i's path.
        // Tree warp w owns word w of every row: the transpose of the 32 x 32 bit
        // block (its nodes i) x (word c of their ancestor rows), by five rounds of
        // shuffles (block transpose of Hacker's Delight, section 7-3, on
        // bit-reversed words so that bit c stands for column c); zero for c > w.
        uint32_t mine[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c > quad) break;  // warp-uniform
            uint32_t x = __brev(mw[c]);
            uint32_t m = 0x0000FFFFu;
#pragma unroll
            for (int j = 16; j != 0; j >>= 1, m ^= (m << j)) {
                const uint32_t other = __shfl_xor_sync(0xffffffffu, x, j);
                x = (lane & j) ? x ^ (((other ^ (x >> j)) & m) << j) : x ^ ((x ^ (other >> j)) & m);
            }
            mine[c] = __brev(x);
        }
        named_sync(1, 128);  // every ancestor row has been read by the validation
#pragma unroll
        for (int c = 0; c < 4; ++c) msk[(c * 32 + lane) * 4 + quad] = mine[c];
        if (i == 0 && s_err[pp]) flag(p.status, s_err[pp]);
        named_sync(1, 128);
        mbar_arrive(&bar[B_DESC]);
    };

    // State warps: S0 rows 32 sw .. 32 sw + 31 as bf16 (B operand, K-major,
    // 128-byte swizzle), eight rows per batch, double-buffered; lane l holds
    // columns 4l .. 4l + 3 (coalesced row reads).  Arrives on B_S0IN.
    const int sw = warp - 4;
    auto state_s0 = [&](const Item &it) {
        const float *s0t = p.S0 + ((int64_t)it.b * p.hv_n + it.hv) * (kD * kD);
        float4 s0a[8], s0b[8];
        auto s0_load = [&](float4 (&dst)[8], int batch) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
                dst[r] = __ldg(reinterpret_cast<const float4 *>(s0t + (sw * 32 + batch * 8 + r) * kD) + lane);
        };
        auto s0_put = [&](const float4 (&src)[8], int batch) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
                *reinterpret_cast<uint2 *>(sm + OFF_S0 + sw128_offset(sw * 32 + batch * 8 + r, 4 * lane)) =
                    make_uint2(pack_bf16(src[r].x, src[r].y), pack_bf16(src[r].z, src[r].w));
        };
        s0_load(s0a, 0);
        s0_load(s0b, 1);
        s0_put(s0a, 0);
        s0_load(s0a, 2);
        s0_put(s0b, 1);
        s0_load(s0b, 3);
        s0_put(s0a, 2);
        s0_put(s0b, 3);
        fence_proxy_async_smem();
        mbar_arrive(&bar[B_S0IN]);
    };

    // scatter of one half of the Gram: lane a holds k_a.k_i (cols 0..127) or
    // k_a.q_i (cols 128..255) and writes them into the ancestor rows of its
    // descendants i (the descendant bits of a come from its mask row).
    auto scatter = [&](int col0, __half *dst, bool strict) {
        const int a = row;
        const int da = a < cur.n ? min(max(dep[a], 1), kMaxDepth) : 1;
#pragma unroll 1
        for (int cc = quad; cc < 4; ++cc) {
            uint32_t dm = msk[a * 4 + cc];
            if (strict && cc == quad) dm &= ~(1u << lane);  // X is strictly lower
            if (!__any_sync(0xffffffffu, dm != 0u)) continue;
            uint32_t v[32];
            tmem_ld32_nowait(tmem + lane_base + col0 + cc * 32, v);
            tmem_wait_ld_into(v);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if ((dm >> c) & 1u) dst[(cc * 32 + c) * kMaxDepth + da - 1] = __float2half_rn(__uint_as_float(v[c]));
        }
    };

    // ---- the first item's operands -------------------------------------------
    if (issuer) issue_kq(cur);
    if (tree) {
        tree_meta(cur, 0);
    } else {
        griddep_wait();  // S0 may be the output of the preceding grid (a commit)
        state_s0(cur);
    }

    const uint32_t id_n256 = idesc_bf16_f32(128, 256), id_n128 = idesc_bf16_f32(128, 128);
    for (int it = 0;; ++it) {
        const int ph = it & 1;
        const int n = cur.n, nb = (n + 31) >> 5;
        // the next item: its offsets are read now, used near the end of this one
        const int cand = cur.idx + gridDim.x;
        int c_lo = 0, c_hi = 0;
        if (cand < p.items) {
            c_lo = __ldg(p.offsets + cand / p.hv_n);
            c_hi = __ldg(p.offsets + cand / p.hv_n + 1);
        }
        if (issuer) {
            // L2 hints: the next item's S0 tile and this item's V tile
            if (cand < p.items) prefetch_l2(p.S0 + (int64_t)cand * (kD * kD), kD * kD * 4);
            for (int h = 0; h < 2; ++h)
                for (int r = 0; r < nb; ++r) tma_prefetch_3d(&tmV, h * 64, cur.hv, cur.lo + 32 * r);
        }
        auto next = [&](Item &nx) -> bool {
            if (cand >= p.items) return false;
            if (item_ok(c_lo, c_hi - c_lo, p.total)) {
                set_item(p, cand, c_lo, c_hi - c_lo, nx);
                return true;
            }
            return find_item(p, cand, gridDim.x, tid == 0, nx);
        };

        if (tree) {
            // ===================== tree warps ==================================
            const int i = tid;
            const int myd = i < n ? min(dep[i], kMaxDepth) : 0;
            if (i == 0) {
                // Gram: K [K;Q]^T -> columns [0, 256), once the tiles have landed
                // and the previous item's Z has been read out
                if (it > 0) ok = mbar_wait(&bar[B_ZFREE], ph ^ 1) && ok;
                ok = mbar_wait(&bar[B_KQ], ph) && ok;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = smem_desc(smem_u32(sm + OFF_KQ + (ks >> 2) * 32768 + (ks & 3) * 32), 16, 1024, 2);
                    mma_bf16(tmem, d, d, id_n256, ks > 0);
                }
                mma_commit(&bar[B_GRAM]);
            }
            const uint4 pr = *reinterpret_cast<const uint4 *>(path + i * kMaxDepth);
            const uint32_t pw[4] = {pr.x, pr.y, pr.z, pr.w};
            int node_at[kMaxDepth];
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l) node_at[l] = l < myd ? (int)((pw[l >> 2] >> (8 * (l & 3))) & 0x7Fu) : i;

            // strict part of the Gram -> raw X rows, full part -> raw Y rows; the
            // state warps meanwhile convert this item's S0
            ok = mbar_wait(&bar[B_GRAM], ph) && ok;
            tc_fence_after();
            scatter(0, Xs, true);
            scatter(128, Ys, false);
            tc_fence_before();
            mbar_arrive(&bar[B_TFREE]);

            // decay factors, X scaling, then P = Y (I + X)^-1 along the path
            float dec[kMaxDepth];  // exp(gamma_i - gamma_path[l]); zero past the depth
            const float gi = gam[i];
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l) dec[l] = l < myd ? expf(gi - gam[node_at[l]]) : 0.f;
            ok = mbar_wait(&bar[B_TFREE], ph) && ok;  // every X and Y entry is in
            {
                const float bi = bet[i];
                uint4 xw[2];
                xw[0] = reinterpret_cast<const uint4 *>(Xs + i * kMaxDepth)[0];
                xw[1] = reinterpret_cast<const uint4 *>(Xs + i * kMaxDepth)[1];
                float xs[kMaxDepth];
#pragma unroll
                for (int l = 0; l < kMaxDepth; ++l) xs[l] = half_at(xw, l) * bi * dec[l];
                reinterpret_cast<uint4 *>(Xs + i * kMaxDepth)[0] =
                    make_uint4(pack_half(xs[0], xs[1]), pack_half(xs[2], xs[3]), pack_half(xs[4], xs[5]), pack_half(xs[6], xs[7]));
                reinterpret_cast<uint4 *>(Xs + i * kMaxDepth)[1] =
                    make_uint4(pack_half(xs[8], xs[9]), pack_half(xs[10], xs[11]), pack_half(xs[12], xs[13]), pack_half(xs[14], xs[15]));
            }
            named_sync(1, 128);
            float P[kMaxDepth];
            {
                uint4 yw[2];
                yw[0] = reinterpret_cast<const uint4 *>(Ys + i * kMaxDepth)[0];
                yw[1] = reinterpret_cast<const uint4 *>(Ys + i * kMaxDepth)[1];
#pragma unroll
                for (int l = 0; l < kMaxDepth; ++l) P[l] = dec[l] * half_at(yw, l);
            }
#pragma unroll
            for (int a = kMaxDepth - 1; a >= 1; --a) {
                // entries past the depth are zero, so a short path costs no branches
                uint4 xw[2];
                xw[0] = reinterpret_cast<const uint4 *>(Xs + node_at[a] * kMaxDepth)[0];
                xw[1] = reinterpret_cast<const uint4 *>(Xs + node_at[a] * kMaxDepth)[1];
                const float pa = a < myd ? P[a] : 0.f;
#pragma unroll
                for (int l = 0; l < a; ++l) P[l] = fmaf(-pa, half_at(xw, l), P[l]);
            }
            const float inv = 1.f / eg[i];

            // P rows (A operand, K-major) once the K|Q space is free
            ok = mbar_wait(&bar[B_S0], ph) && ok;
            uint8_t *prow = sm + OFF_PA;
#pragma unroll
            for (int q = 0; q < 16; ++q)
                *reinterpret_cast<uint4 *>(prow + sw128_offset(i, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l)
                if (l < myd)
                    *reinterpret_cast<__nv_bfloat16 *>(prow + sw128_offset(i, node_at[l])) = __float2bfloat16_rn(P[l] * inv);
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_P]);

            // the next item's tree data, once the state warps hold this item's
            Item nx;
            if (!next(nx)) break;
            ok = mbar_wait(&bar[B_META], ph) && ok;
            tree_meta(nx, ph ^ 1);
            cur = nx;
        } else {
            // ===================== state warps =================================
            ok = mbar_wait(&bar[B_DESC], ph) && ok;
            mbar_arrive(&bar[B_TFREE]);  // the tree warps read the Gram out

            if (issuer) {
                // S0 part: W = K S0^T (cols 0..127), Z = Q S0^T (cols 128..255)
                ok = mbar_wait(&bar[B_S0IN], ph) && ok;
                ok = mbar_wait(&bar[B_TFREE], ph) && ok;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kq = smem_u32(sm + OFF_KQ + (ks >> 2) * 32768 + (ks & 3) * 32);
                    const uint64_t bs = smem_desc(smem_u32(sm + OFF_S0 + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
                    mma_bf16(tmem, smem_desc(kq, 16, 1024, 2), bs, id_n128, ks > 0);
                    mma_bf16(tmem + 128, smem_desc(kq + 16384, 16, 1024, 2), bs, id_n128, ks > 0);
                }
                mma_commit(&bar[B_S0]);
                // V tile into the S0 space once those MMAs are done
                ok = mbar_wait(&bar[B_S0], ph) && ok;
                mbar_arrive_expect_tx(&bar[B_V], (uint32_t)(2 * nb * 4096));
                for (int h = 0; h < 2; ++h)
                    for (int r = 0; r < nb; ++r)
                        tma_load_3d(sm + OFF_S0 + h * 16384 + r * 4096, &tmV, &bar[B_V], h * 64, cur.hv, cur.lo + 32 * r);
            }

            // this item's per-row data into registers; the tree warps may then
            // overwrite it with the next item's
            const int j = row;
            const float bj = bet[j], bej = bj * egt[j];
            const float f_out = p.scale * eg[j];
            uint32_t desc_row[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) desc_row[w] = msk[j * 4 + w];
            const bool item_good = s_err[ph] == 0;
            const bool store = item_good && j < n;
            mbar_arrive(&bar[B_META]);

            // right-hand side rows R[j][n] = beta_j v[j][n] - beta_j e^gamma_j W[j][n] (MN-major B).
            // A row with a non-finite entry is stored as zero (its subtree's outputs are
            // set to NaN), and so is every row past the tree.
            ok = mbar_wait(&bar[B_V], ph) && ok;
            tc_fence_after();
            float chk = 0.f;  // 0 * x: stays zero while every entry is finite
            auto r_chunk = [&](const uint32_t (&w)[32], int cc) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int n0 = cc * 32 + q * 8;
                    const uint4 vv = *reinterpret_cast<const uint4 *>(sm + OFF_S0 + sw128_offset(j, n0));
                    const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                    float r[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float vj = (e & 1) ? bf16_hi(vw[e >> 1]) : bf16_lo(vw[e >> 1]);
                        r[e] = fmaf(-bej, __uint_as_float(w[q * 8 + e]), bj * vj);
                        chk = fmaf(0.f, r[e], chk);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_RB + sw128_offset(j, n0)) =
                        make_uint4(pack_bf16(r[0], r[1]), pack_bf16(r[2], r[3]), pack_bf16(r[4], r[5]), pack_bf16(r[6], r[7]));
                }
            };
            {
                // W columns 32 at a time, the next load in flight while one is used
                uint32_t wa[32], wb[32];
                tmem_ld32_nowait(tmem + lane_base, wa);
                tmem_wait_ld_into(wa);
                tmem_ld32_nowait(tmem + lane_base + 32, wb);
                r_chunk(wa, 0);
                tmem_wait_ld_into(wb);
                tmem_ld32_nowait(tmem + lane_base + 64, wa);
                r_chunk(wb, 1);
                tmem_wait_ld_into(wa);
                tmem_ld32_nowait(tmem + lane_base + 96, wb);
                r_chunk(wa, 2);
                tmem_wait_ld_into(wb);
                r_chunk(wb, 3);
            }
            const bool bad = chk != 0.f;
            if (bad || j >= n) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<uint4 *>(sm + OFF_RB + sw128_offset(j, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (bad && j < n) {  // the row and every node below it
#pragma unroll
                for (int w = 0; w < 4; ++w) atomicOr(&pset[ph * 4 + w], desc_row[w]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_R]);

            Item nx;
            const bool more = next(nx);
            // output: Z += (e^-gamma' P) R
            if (issuer) {
                ok = mbar_wait(&bar[B_R], ph) && ok;
                ok = mbar_wait(&bar[B_P], ph) && ok;
                tc_fence_after();
                const uint32_t id_out = id_n128 | (1u << 16);  // B (R) is MN-major
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t ad = smem_desc(smem_u32(sm + OFF_PA + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
                    const uint64_t bd = smem_desc(smem_u32(sm + OFF_RB + ks * 2048), 16384, 1024, 2);
                    mma_bf16(tmem + 128, ad, bd, id_out, true);
                }
                mma_commit(&bar[B_OUT]);
            }
            ok = mbar_wait(&bar[B_OUT], ph) && ok;  // also: every R row (and V read) is done
            tc_fence_after();
            if (issuer && more) issue_kq(nx);       // the K|Q space is free again

            // epilogue: o[i][n] = scale * e^gamma'_i * Z[i][n], NaN for a poisoned row.
            // bf16 rows of whole 32-node boxes are staged in the S0 space (free once
            // every R row is built) in the 128-byte-swizzled box layout and leave by
            // TMA; rows of a ragged last box, and fp32 rows, are stored directly.
            const int i = row;
            const bool hit = (pset[ph * 4 + (i >> 5)] >> (i & 31)) & 1u;
            const float f = hit ? __int_as_float(0x7fc00000) : f_out;  // NaN * z is NaN
            const int nfull = n & ~31;
            const bool staged = sizeof(Tout) == 2 && i < nfull;
            Tout *orow = static_cast<Tout *>(p.o) + ((int64_t)(cur.lo + i) * p.hv_n + cur.hv) * kD;
            auto o_chunk = [&](const uint32_t (&zr)[32], int cc) {
                float z[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) z[e] = f * __uint_as_float(zr[e]);
                if (!store) return;
                if constexpr (sizeof(Tout) == 2) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w = make_uint4(pack_bf16(z[q * 8 + 0], z[q * 8 + 1]), pack_bf16(z[q * 8 + 2], z[q * 8 + 3]),
                                                   pack_bf16(z[q * 8 + 4], z[q * 8 + 5]), pack_bf16(z[q * 8 + 6], z[q * 8 + 7]));
                        if (staged)
                            *reinterpret_cast<uint4 *>(sm + OFF_S0 + sw128_offset(i, cc * 32 + q * 8)) = w;
                        else
                            reinterpret_cast<uint4 *>(orow + cc * 32)[q] = w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        reinterpret_cast<float4 *>(orow + cc * 32)[q] =
                            make_float4(z[q * 4 + 0], z[q * 4 + 1], z[q * 4 + 2], z[q * 4 + 3]);
                }
            };
            {
                uint32_t za[32], zb[32];
                tmem_ld32_nowait(tmem + lane_base + 128, za);
                tmem_wait_ld_into(za);
                tmem_ld32_nowait(tmem + lane_base + 160, zb);
                o_chunk(za, 0);
                tmem_wait_ld_into(zb);
                tmem_ld32_nowait(tmem + lane_base + 192, za);
                o_chunk(zb, 1);
                tmem_wait_ld_into(za);
                tmem_ld32_nowait(tmem + lane_base + 224, zb);
                o_chunk(za, 2);
                tmem_wait_ld_into(zb);
                o_chunk(zb, 3);
            }
            tc_fence_before();
            mbar_arrive(&bar[B_ZFREE]);
            if constexpr (sizeof(Tout) == 2) {
                fence_proxy_async_smem();  // staged rows are visible to the TMA engine
                named_sync(2, 128);
                if (issuer && item_good && nfull > 0) {
                    for (int h = 0; h < 2; ++h)
                        for (int r = 0; r < (nfull >> 5); ++r)
                            tma_store_3d(&tmO, sm + OFF_S0 + h * 16384 + r * 4096, h * 64, cur.hv, cur.lo + 32 * r);
                    bulk_commit();
                    bulk_wait_read();
                }
                named_sync(2, 128);  // the S0 space may be written again
            }
            if (!more) break;
            state_s0(nx);
            cur = nx;
        }
    }
    if (!ok) flag(p.status, GDN_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// [T][H][128] bf16 viewed as a 3-D tensor (d, head, token); boxes of 64 x 1 x 32,
// 128-byte swizzle.
bool encode_tokens(CUtensorMap *map, const void *base, int heads, int total) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
    cuuint32_t box[3] = {64, 1, 32};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool verify_tc_supported(const gdn_verify_args &a) {
    return a.qkv_dtype == GDN_BF16 && a.d_k == kD && a.d_v == kD && a.max_nodes <= kN &&
           a.max_depth >= 1 && a.max_depth <= kMaxDepth && a.total_nodes > 0 && aligned16(a.q) &&
           aligned16(a.k) && aligned16(a.v) && aligned16(a.S0) && aligned16(a.o) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_verify_tc(const gdn_verify_args &a, cudaStream_t stream, bool after_commit) {
    CUtensorMap tmK, tmQ, tmV, tmO;
    if (!encode_tokens(&tmK, a.k, a.n_k_heads, a.total_nodes) ||
        !encode_tokens(&tmQ, a.q, a.n_k_heads, a.total_nodes) ||
        !encode_tokens(&tmV, a.v, a.n_v_heads, a.total_nodes))
        return cudaErrorInvalidValue;
    // bf16 outputs leave through TMA stores of the same box shape as V
    if (a.out_dtype == GDN_BF16) {
        if (!encode_tokens(&tmO, a.o, a.n_v_heads, a.total_nodes)) return cudaErrorInvalidValue;
    } else {
        tmO = tmV;  // unused by the fp32-output kernel
    }
    TcParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.words = a.mask_words < 4 ? a.mask_words : 4;
    p.total = a.total_nodes; p.items = a.batch * a.n_v_heads; p.scale = a.scale;
    p.offsets = a.node_offsets; p.parent = a.parent; p.depth = a.depth; p.mask = a.anc_mask;
    p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.o = a.o; p.status = a.dev_status;
    static int have_bf16[16], have_f32[16];
    auto kern = a.out_dtype == GDN_BF16 ? verify_tc_kernel<__nv_bfloat16> : verify_tc_kernel<float>;
    cudaError_t e = ensure_smem(kern, kSmemBytes, a.out_dtype == GDN_BF16 ? have_bf16 : have_f32);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    // persistent: two blocks per SM (tensor memory and shared memory allow two)
    cfg.gridDim = dim3((unsigned)std::min(p.items, 2 * sm_count()));
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    // after a commit of the state in the same stream, the launch may begin while
    // the commit drains (programmatic dependent launch; the kernel waits for it
    // before its first state read)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = after_commit ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tmK, tmQ, tmV, tmO, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace gdn
