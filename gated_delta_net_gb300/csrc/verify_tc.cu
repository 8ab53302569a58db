// verify_tc.cu -- tcgen05/TMA tree verification for bf16 tokens, d_k = d_v = 128,
// trees of at most 128 nodes and depth at most 16 (sm_103a).
//
// Computes, for each (request, value head), the masked triangular solve of
// "Trees from Marginals" (gist.science Technical Summary, section 3
// "Rollback-Free Tree Verification for GDN"):
//     X = strict-ancestor mask * beta_i * D_ij * (K K^T),  Y = ancestor mask * D_ij * (Q K^T)
//     (I + X) U = R = beta * (V - e^gamma * K S0^T)
//     O = scale * (e^gamma * Q S0^T + Y U)
// with D_ij = exp(gamma_i - gamma_j), gamma the sum of g along each path.
// Because only ancestors interact and paths are at most 16 long, each node's
// row of P = Y (I + X)^-1 has at most 16 non-zeros and is found by a 16-step
// back substitution along the node's own path; then O = e^gamma Z + P R.
// Writing P[l] = D_{i,path(l)} P'[l], the decays cancel inside the substitution:
//     P'[l] = (q_i . k_l) - sum_{a > l} P'[a] beta_a (k_a . k_l)
// so the raw dot products (kept in fp32) serve every value head of a key head.
//
// Work unit: (request, key head, pair of value heads).  The two value heads of
// a unit share the K and Q tiles, the Gram K [K;Q]^T, its scatter into raw
// per-node ancestor rows, and the request's tree data; one block per SM walks a
// contiguous run of units.
//
// Dense contractions run on the tensor cores (kind::f16, fp32 accumulate);
// tensor-memory lane = tree node throughout.  Tensor memory is 512 columns in
// two halves of 256; the u-th unit of a block (parity u % 2) puts its Gram in
// half u % 2, value head A's [W | Z] in half 1 - u % 2 and value head B's
// [W | Z] in half u % 2 once the Gram has been read out:
//   Gram   : K [K;Q]^T                A = K tile, B = [K;Q] tile (TMA, 128B swizzle)
//   S0 part: W = K S0^T, Z = Q S0^T   B = S0 rounded to bf16 like the tokens
//   Output : Z += (e^-gamma' P) R     A = P rows, B = R rows (MN-major);
//            gamma' = max(gamma, -80) keeps e^-gamma' finite; the epilogue scales
//            row i by e^gamma'_i, so O = e^gamma' Z + P R.
//
// Warp roles (512 threads), handing off through mbarriers:
//   warps 0-3   tree:   the Gram (thread 0) and its scatter into raw X and Y rows;
//                       P rows of head B.
//   warps 4-7   state A, warps 8-11 state B: per value head, the S0 and output
//                       MMAs (its thread 0), the right-hand side R (written over V),
//                       the epilogue (staged over R, stored by TMA), then the next
//                       unit's V by TMA; head B's thread 0 also loads the next
//                       unit's K/Q tiles once both output MMAs have read the P rows.
//   warps 12-15 aux:    P rows of head A; the next unit's node data (paths, gamma,
//                       descriptor checks, descendant rows); the next unit's S0 of
//                       both heads as bf16; the first K/Q tiles.
// The P rows of both heads go to the K/Q space once the Gram and the S0 MMAs
// have read it, so that each head's S0 space is free for the next unit as soon
// as its S0 MMA is done.
// Every mbarrier completes once per unit, so waits use the unit's parity.
// A node whose right-hand side row turns non-finite has that row replaced by
// zero in the output product and its subtree's outputs set to NaN, so
// non-finite values never leave their own branch.
// Launched as the dependent of a commit that writes the state (programmatic
// dependent launch), only the state warps' first state read waits for the
// commit grid to finish.
#include <cuda_fp16.h>

#include <algorithm>
#include "internal.cuh"
#include "sm100.cuh"
#include "tc_tiles.cuh"

namespace gdn {
namespace {

using namespace sm100;
using namespace tiles;

constexpr int kT = 512;           // threads per block
constexpr int kN = 128;           // tile rows: nodes (max_nodes <= 128)
constexpr int kMaxDepth = 16;
constexpr float kGammaFloor = -80.f;
// Row stride (floats) of the raw X and Y rows: 16 entries padded to 20, so that a
// warp's 16-byte reads of 32 different rows spread over all banks.
constexpr int kXS = 20;

// shared-memory layout (bytes from the dynamic base, which is 1024-aligned)
constexpr int OFF_KQ = 0;                               // [2 k-blocks][256 rows (K, Q)][128 B], then P rows of both heads
constexpr int OFF_S = 65536;                            // [2 heads] S0 bf16 [2 k-blocks][128][128 B]
constexpr int OFF_V = OFF_S + 2 * 32768;                // [2 heads] V tile, then R over it, then staged outputs
constexpr int OFF_X = OFF_V + 2 * 32768;                // float [128][kXS] raw k.k
constexpr int OFF_Y = OFF_X + kN * kXS * 4;             // float [128][kXS] raw q.k
constexpr int OFF_MASK = OFF_Y + kN * kXS * 4;          // uint32 [128][4] ancestor, then descendant bits
constexpr int OFF_PATH = OFF_MASK + kN * 4 * 4;         // uint8 [128][16]
constexpr int OFF_F = OFF_PATH + kN * kMaxDepth;        // [2 heads] float graw, gam, egt, eg, bet [128]
constexpr int OFF_I = OFF_F + 2 * 5 * kN * 4;           // int dep, par [128]
constexpr int OFF_MISC = OFF_I + 2 * kN * 4;            // tmem slot; pset[2][2][4]; err[2]
constexpr int OFF_BAR = OFF_MISC + 128;
constexpr int kBars = 24;
constexpr int kSmemBytes = OFF_BAR + kBars * 8;

// mbarrier indices; the 0/1 variants are per value head of the unit (A, B)
enum {
    B_KQ, B_GRAM, B_SCAT, B_DESC,
    B_S0IN0, B_S0IN1, B_S00, B_S01, B_V0, B_V1, B_R0, B_R1, B_P0, B_P1,
    B_OUT0, B_OUT1, B_ZF0, B_ZF1, B_META0, B_META1, B_META2,
    B_PROBE  // never arrived on; the wait probe's bounded wait
};
static_assert(B_PROBE < kBars, "barrier count");

// arrival counts: 1 for TMA/commit-completed barriers, 128 for one warp group
__device__ __forceinline__ uint32_t bar_count(int k) {
    switch (k) {
        case B_KQ: case B_GRAM: case B_S00: case B_S01: case B_V0: case B_V1:
        case B_OUT0: case B_OUT1: case B_PROBE:
            return 1u;
        default:
            return 128u;
    }
}

struct TcParams {
    int hk_n, hv_n, words, stride, total, units, group, npair;
    int probe;  // > 0: thread 0 makes one wait of `probe` polls on B_PROBE (test hook)
    float scale;
    const int32_t *offsets, *parent, *depth;
    const uint32_t *mask;
    const float *g, *beta, *S0;
    void *o;
    int32_t *status;
};

// one (request, key head, value-head pair) unit: value heads hv0 and hv0 + 1;
// a key head's group with an odd number of value heads left has only hv0
// (has2 false: head B repeats hv0 and stores nothing)
struct Unit {
    int idx, b, hk, lo, n, hv0;
    bool has2, meta;
};

__device__ __forceinline__ int hv_of(const Unit &u, int g) { return u.hv0 + (g != 0 && u.has2 ? 1 : 0); }

__device__ __forceinline__ bool unit_ok(int lo, int n, int total) {
    return n > 0 && n <= kN && lo >= 0 && lo + n <= total;
}

__device__ __forceinline__ void set_unit(const TcParams &p, int idx, int lo, int n, Unit &u) {
    u.idx = idx;
    const int j = idx % p.npair, bh = idx / p.npair;
    u.b = bh / p.hk_n;
    u.hk = bh % p.hk_n;
    u.hv0 = u.hk * p.group + 2 * j;
    u.has2 = 2 * j + 1 < p.group;
    u.lo = lo;
    u.n = n;
    u.meta = true;
}

// The first unit in [idx, end) whose request is non-empty and well placed;
// requests that are too large or reach past the node count are flagged (when
// `report`) and passed over.
__device__ bool find_unit(const TcParams &p, int idx, int end, bool report, Unit &u) {
    for (; idx < end; ++idx) {
        const int b = idx / (p.npair * p.hk_n);
        const int lo = __ldg(p.offsets + b);
        const int n = __ldg(p.offsets + b + 1) - lo;
        if (n == 0) continue;
        if (!unit_ok(lo, n, p.total)) {
            if (report) flag(p.status, n > kN ? GDN_DEV_TOO_MANY : GDN_DEV_BAD_DESC);
            continue;
        }
        set_unit(p, idx, lo, n, u);
        return true;
    }
    return false;
}

// Node i's path within the current request: node_at[l] for l < myd (root first),
// i itself past the depth (so every index stays in the tile).
__device__ __forceinline__ int load_path(const uint8_t *path, const int *dep, int i, int n, int (&node_at)[kMaxDepth]) {
    const int myd = i < n ? min(max(dep[i], 0), kMaxDepth) : 0;
    const uint4 pr = *reinterpret_cast<const uint4 *>(path + i * kMaxDepth);
    const uint32_t pw[4] = {pr.x, pr.y, pr.z, pr.w};
#pragma unroll
    for (int l = 0; l < kMaxDepth; ++l) node_at[l] = l < myd ? (int)((pw[l >> 2] >> (8 * (l & 3))) & 0x7Fu) : i;
    return myd;
}

// Row i of P for one value head along i's path (fh: its per-node floats graw,
// gam, egt, eg, bet), from the raw rows X (k.k, strict ancestors) and Y (q.k),
// scaled by e^-gamma'_i for the output MMA; zero past the depth.
__device__ __forceinline__ void p_solve(const float *Xf, const float *Yf, const float *fh, int i, int myd,
                                        const int (&node_at)[kMaxDepth], float (&P)[kMaxDepth]) {
    const float *gm = fh + kN, *bt = fh + 4 * kN;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 y = reinterpret_cast<const float4 *>(Yf + i * kXS)[q];
        P[4 * q] = y.x; P[4 * q + 1] = y.y; P[4 * q + 2] = y.z; P[4 * q + 3] = y.w;
    }
#pragma unroll
    for (int a = kMaxDepth - 1; a >= 1; --a) {
        // entries past the depth are zero, so a short path costs no branches
        const float4 *xr = reinterpret_cast<const float4 *>(Xf + node_at[a] * kXS);
        const float ca = a < myd ? P[a] * bt[node_at[a]] : 0.f;
#pragma unroll
        for (int q = 0; q < (a + 3) / 4; ++q) {
            const float4 v = xr[q];
            if (4 * q + 0 < a) P[4 * q + 0] = fmaf(-ca, v.x, P[4 * q + 0]);
            if (4 * q + 1 < a) P[4 * q + 1] = fmaf(-ca, v.y, P[4 * q + 1]);
            if (4 * q + 2 < a) P[4 * q + 2] = fmaf(-ca, v.z, P[4 * q + 2]);
            if (4 * q + 3 < a) P[4 * q + 3] = fmaf(-ca, v.w, P[4 * q + 3]);
        }
    }
    const float gi = gm[i], inv = 1.f / fh[3 * kN + i];
#pragma unroll
    for (int l = 0; l < kMaxDepth; ++l) P[l] = l < myd ? P[l] * (expf(gi - gm[node_at[l]]) * inv) : 0.f;
}

// Row i of P as the bf16 A operand of the output MMA (K-major, 128-byte swizzle) at prow.
__device__ __forceinline__ void p_write(uint8_t *prow, int i, int myd, const int (&node_at)[kMaxDepth],
                                        const float (&P)[kMaxDepth]) {
#pragma unroll
    for (int q = 0; q < 16; ++q) *reinterpret_cast<uint4 *>(prow + sw128_offset(i, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int l = 0; l < kMaxDepth; ++l)
        if (l < myd) *reinterpret_cast<__nv_bfloat16 *>(prow + sw128_offset(i, node_at[l])) = __float2bfloat16_rn(P[l]);
}

template <typename Tout>
__global__ void __launch_bounds__(kT, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, TcParams p) {
    extern __shared__ __align__(1024) uint8_t sm[];
    float *Xs = reinterpret_cast<float *>(sm + OFF_X);
    float *Ys = reinterpret_cast<float *>(sm + OFF_Y);
    uint32_t *msk = reinterpret_cast<uint32_t *>(sm + OFF_MASK);  // ancestor rows, then descendant rows
    uint8_t *path = sm + OFF_PATH;
    // per value head g: graw, gam, egt (e^gamma), eg (e^gamma'), bet, 128 floats each
    float *fhead = reinterpret_cast<float *>(sm + OFF_F);
    int *dep = reinterpret_cast<int *>(sm + OFF_I), *par = dep + kN;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    uint32_t *pset = tslot + 1;                           // [parity][head][4]: nodes whose output is poisoned
    int *s_err = reinterpret_cast<int *>(tslot + 17);     // [parity]: descriptor errors of the request
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
    const int role = warp >> 2;        // 0 tree, 1 state A, 2 state B, 3 aux
    const int row = quad * 32 + lane;  // tensor-memory lane of this thread = a tree node
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    // a block that leaves early still waits for a preceding grid, so that this
    // grid never completes before the grid it depends on
    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0) flag(p.status, GDN_DEV_INTERNAL);
        griddep_wait();
        return;
    }
    // the tensor maps' descriptors, ahead of their first use
    if (tid == 0) {
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmO);
    }
    const int unit_end = (int)(((int64_t)(blockIdx.x + 1) * p.units) / gridDim.x);
    Unit cur;
    if (!find_unit(p, (int)(((int64_t)blockIdx.x * p.units) / gridDim.x), unit_end, tid == 0, cur)) {
        griddep_wait();
        return;
    }

    // ---- set-up, once per block ---------------------------------------------
    if (tid == 0) {
        for (int k = 0; k < kBars; ++k) mbar_init(&bar[k], bar_count(k));
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;
    // test hook: a bounded wait on a barrier that nothing arrives on runs out,
    // and the block records GDN_DEV_TIMEOUT at exit; nothing else changes
    if (p.probe > 0 && tid == 0) ok = mbar_wait(&bar[B_PROBE], 0, (uint32_t)p.probe);

    // the unit after `c` in this block's run (false at the end of the run)
    auto next_unit = [&](const Unit &c, Unit &nx) -> bool {
        if (!find_unit(p, c.idx + 1, unit_end, tid == 0, nx)) return false;
        nx.meta = nx.b != c.b;
        return true;
    };

    // K and Q tiles of a unit (boxes of 32 nodes x 64 features, both k-blocks)
    auto issue_kq = [&](const Unit &u) {
        const int nb = (u.n + 31) >> 5;
        mbar_arrive_expect_tx(&bar[B_KQ], (uint32_t)(2 * 2 * nb * 4096));
        for (int kb = 0; kb < 2; ++kb)
            for (int r = 0; r < nb; ++r) {
                tma_load_3d(sm + OFF_KQ + kb * 32768 + r * 4096, &tmK, &bar[B_KQ], kb * 64, u.hk, u.lo + 32 * r);
                tma_load_3d(sm + OFF_KQ + kb * 32768 + (128 + 32 * r) * 128, &tmQ, &bar[B_KQ], kb * 64, u.hk,
                            u.lo + 32 * r);
            }
    };
    // V tile of value head g into its buffer
    auto issue_v = [&](const Unit &u, int g) {
        const int nb = (u.n + 31) >> 5;
        mbar_arrive_expect_tx(&bar[B_V0 + g], (uint32_t)(2 * nb * 4096));
        for (int h = 0; h < 2; ++h)
            for (int r = 0; r < nb; ++r)
                tma_load_3d(sm + OFF_V + g * 32768 + h * 16384 + r * 4096, &tmV, &bar[B_V0 + g], h * 64, hv_of(u, g),
                            u.lo + 32 * r);
    };

    const uint32_t id_n256 = idesc_bf16_f32(128, 256), id_n128 = idesc_bf16_f32(128, 128);

    // S0 of value head g of unit u as bf16 (B operand, K-major, 128-byte
    // swizzle) into head g's S space by one warp group; eight rows per batch,
    // double-buffered; lane l holds columns 4l .. 4l + 3 (coalesced row reads).
    auto convert = [&](const Unit &u, int g) {
        const int sw = quad;  // rows 32 sw .. 32 sw + 31 of the state tile
        const float *s0t = p.S0 + ((int64_t)u.b * p.hv_n + hv_of(u, g)) * (kD * kD);
        uint8_t *dst = sm + OFF_S + g * 32768;
        float4 s0a[8], s0b[8];
        auto s0_load = [&](float4 (&d)[8], int batch) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
                d[r] = __ldg(reinterpret_cast<const float4 *>(s0t + (sw * 32 + batch * 8 + r) * kD) + lane);
        };
        auto s0_put = [&](const float4 (&src)[8], int batch) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
                *reinterpret_cast<uint2 *>(dst + sw128_offset(sw * 32 + batch * 8 + r, 4 * lane)) =
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
        mbar_arrive(&bar[B_S0IN0 + g]);
    };

    if (role == 0) {
        // ======================= tree warps ===================================
        const int i = tid;
        // Scatter of the Gram (tensor-memory columns from `gram`): lane a holds
        // k_a.k_i (cols 0..127) and k_a.q_i (cols 128..255) and writes them into
        // the ancestor rows of its descendants i (the descendant bits of a come
        // from its mask row): X rows (strict descendants) and Y rows (a included).
        auto scatter = [&](uint32_t gram) {
            const int a = row;
            const int da = a < cur.n ? min(max(dep[a], 1), kMaxDepth) : 1;
#pragma unroll 1
            for (int cc = quad; cc < 4; ++cc) {
                const uint32_t dm = msk[a * 4 + cc];
                if (!__any_sync(0xffffffffu, dm != 0u)) continue;
                uint32_t v[32];
                tmem_ld32_nowait(gram + lane_base + cc * 32, v);
                tmem_wait_ld_into(v);
                const uint32_t dx = cc == quad ? dm & ~(1u << lane) : dm;  // X is strictly lower
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if ((dx >> c) & 1u) Xs[(cc * 32 + c) * kXS + da - 1] = __uint_as_float(v[c]);
                tmem_ld32_nowait(gram + lane_base + 128 + cc * 32, v);
                tmem_wait_ld_into(v);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if ((dm >> c) & 1u) Ys[(cc * 32 + c) * kXS + da - 1] = __uint_as_float(v[c]);
            }
        };

        // the first unit's K and Q: a tree-warp thread issues them, since the first
        // TMA loads of a launch take long to issue and the aux warps meanwhile
        // build the first unit's tree data and state tiles
        if (tid == 32) issue_kq(cur);
        for (int it = 0;; ++it) {
            const int ph = it & 1;
            const uint32_t gram = tmem + (uint32_t)(ph * 256);
            ok = mbar_wait(&bar[B_DESC], ph) && ok;  // this unit's tree data
            if (i == 0) {
                // Gram: K [K;Q]^T -> half ph, once the tiles have landed and head A
                // of the previous unit (which held that half) has read its Z out
                if (it > 0) ok = mbar_wait(&bar[B_ZF0], ph ^ 1) && ok;
                ok = mbar_wait(&bar[B_KQ], ph) && ok;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = smem_desc(smem_u32(sm + OFF_KQ + (ks >> 2) * 32768 + (ks & 3) * 32), 16, 1024, 2);
                    mma_bf16(gram, d, d, id_n256, ks > 0);
                }
                mma_commit(&bar[B_GRAM]);
            }
            Unit nx;
            const bool more = next_unit(cur, nx);
            int node_at[kMaxDepth];
            const int myd = load_path(path, dep, i, cur.n, node_at);
            ok = mbar_wait(&bar[B_GRAM], ph) && ok;
            tc_fence_after();
            scatter(gram);
            tc_fence_before();
            mbar_arrive(&bar[B_SCAT]);
            ok = mbar_wait(&bar[B_SCAT], ph) && ok;  // every X and Y entry is in
            float P[kMaxDepth];
            p_solve(Xs, Ys, fhead + 5 * kN, i, myd, node_at, P);
            mbar_arrive(&bar[B_META2]);  // this unit's tree data is no longer read here
            // P rows of head B into the K/Q space, free once the Gram and both S0
            // MMAs (head B's is the last) have read it
            ok = mbar_wait(&bar[B_S01], ph) && ok;
            p_write(sm + OFF_KQ + 32768, i, myd, node_at, P);
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_P1]);
            if (!more) break;
            // the next unit's head-B state tile, into head B's S space, free since
            // its S0 MMA (the aux warps convert head A's)
            if (it == 0) griddep_wait();  // S0 may be the output of the preceding grid
            convert(nx, 1);
            cur = nx;
        }
    } else if (role <= 2) {
        // ======================= state warps (value head g) ==================
        const int g = role - 1;
        const bool issuer = (tid & 127) == 0;
        const int j = row;
        const float *fb = fhead + g * 5 * kN;
        uint8_t *sbuf = sm + OFF_S + g * 32768, *vbuf = sm + OFF_V + g * 32768;
        uint8_t *pbuf = sm + OFF_KQ + g * 32768;  // this head's P rows
        if (issuer) issue_v(cur, g);
        for (int it = 0;; ++it) {
            const int ph = it & 1;
            const int n = cur.n;
            // head A's [W | Z] in half 1 - ph, head B's in half ph (after the Gram)
            const uint32_t wz = tmem + (uint32_t)((g == 0 ? ph ^ 1 : ph) * 256);
            Unit nx;
            const bool more = next_unit(cur, nx);
            // this unit's per-row data into registers; the tree warps may then
            // overwrite it with the next unit's
            ok = mbar_wait(&bar[B_DESC], ph) && ok;
            const float bj = fb[4 * kN + j], bej = bj * fb[2 * kN + j];
            const float f_out = p.scale * fb[3 * kN + j];
            uint32_t desc_row[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) desc_row[w] = msk[j * 4 + w];
            const bool item_good = s_err[ph] == 0 && (g == 0 || cur.has2);
            const bool store = item_good && j < n;
            mbar_arrive(&bar[B_META0 + g]);

            if (issuer) {
                // S0 part: W = K S0^T (cols 0..127), Z = Q S0^T (cols 128..255)
                ok = mbar_wait(&bar[B_KQ], ph) && ok;
                ok = mbar_wait(&bar[B_S0IN0 + g], ph) && ok;
                if (g == 0) {
                    if (it > 0) ok = mbar_wait(&bar[B_ZF1], ph ^ 1) && ok;  // head B of the previous unit
                } else {
                    ok = mbar_wait(&bar[B_SCAT], ph) && ok;  // the Gram has been read out
                    // after head A's S0 MMA: head B's unit then cannot finish
                    // before head A has waited for head B's previous one
                    ok = mbar_wait(&bar[B_S00], ph) && ok;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kq = smem_u32(sm + OFF_KQ + (ks >> 2) * 32768 + (ks & 3) * 32);
                    const uint64_t bs = smem_desc(smem_u32(sbuf + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
                    mma_bf16(wz, smem_desc(kq, 16, 1024, 2), bs, id_n128, ks > 0);
                    mma_bf16(wz + 128, smem_desc(kq + 16384, 16, 1024, 2), bs, id_n128, ks > 0);
                }
                mma_commit(&bar[B_S00 + g]);
            }

            // right-hand side rows R[j][n] = beta_j v[j][n] - beta_j e^gamma_j W[j][n],
            // written over V (same MN-major B layout).  A row with a non-finite entry
            // is stored as zero (its subtree's outputs are set to NaN), and so is
            // every row past the tree.
            ok = mbar_wait(&bar[B_S00 + g], ph) && ok;
            ok = mbar_wait(&bar[B_V0 + g], ph) && ok;
            tc_fence_after();
            float chk = 0.f;  // 0 * x: stays zero while every entry is finite
            auto r_chunk = [&](const uint32_t (&w)[32], int cc) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int n0 = cc * 32 + q * 8;
                    uint4 *at = reinterpret_cast<uint4 *>(vbuf + sw128_offset(j, n0));
                    const uint4 vv = *at;
                    const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                    float r[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float vj = (e & 1) ? bf16_hi(vw[e >> 1]) : bf16_lo(vw[e >> 1]);
                        r[e] = fmaf(-bej, __uint_as_float(w[q * 8 + e]), bj * vj);
                        chk = fmaf(0.f, r[e], chk);
                    }
                    *at = make_uint4(pack_bf16(r[0], r[1]), pack_bf16(r[2], r[3]), pack_bf16(r[4], r[5]), pack_bf16(r[6], r[7]));
                }
            };
            {
                // W columns 32 at a time, the next load in flight while one is used
                uint32_t wa[32], wb[32];
                tmem_ld32_nowait(wz + lane_base, wa);
                tmem_wait_ld_into(wa);
#pragma unroll 1
                for (int cc = 0; cc < 4; cc += 2) {
                    tmem_ld32_nowait(wz + lane_base + (cc + 1) * 32, wb);
                    r_chunk(wa, cc);
                    tmem_wait_ld_into(wb);
                    if (cc < 2) tmem_ld32_nowait(wz + lane_base + (cc + 2) * 32, wa);
                    r_chunk(wb, cc + 1);
                    if (cc < 2) tmem_wait_ld_into(wa);
                }
            }
            const bool bad = chk != 0.f;
            if (bad || j >= n) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<uint4 *>(vbuf + sw128_offset(j, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (bad && j < n) {  // the row and every node below it
#pragma unroll
                for (int w = 0; w < 4; ++w) atomicOr(&pset[(ph * 2 + g) * 4 + w], desc_row[w]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_R0 + g]);

            // output: Z += (e^-gamma' P) R
            if (issuer) {
                ok = mbar_wait(&bar[B_R0 + g], ph) && ok;
                ok = mbar_wait(&bar[B_P0 + g], ph) && ok;
                tc_fence_after();
                const uint32_t id_out = id_n128 | (1u << 16);  // B (R) is MN-major
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t ad = smem_desc(smem_u32(pbuf + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
                    const uint64_t bd = smem_desc(smem_u32(vbuf + ks * 2048), 16384, 1024, 2);
                    mma_bf16(wz + 128, ad, bd, id_out, true);
                }
                mma_commit(&bar[B_OUT0 + g]);
                if (g == 1 && more) {
                    // the next unit's K/Q tiles once both output MMAs have read the P rows
                    ok = mbar_wait(&bar[B_OUT1], ph) && ok;
                    ok = mbar_wait(&bar[B_OUT0], ph) && ok;
                    issue_kq(nx);
                }
            }
            ok = mbar_wait(&bar[B_OUT0 + g], ph) && ok;  // also: every R row is consumed
            tc_fence_after();

            // epilogue: o[i][n] = scale * e^gamma'_i * Z[i][n], NaN for a poisoned row.
            // bf16 rows of whole 32-node boxes are staged over R in the
            // 128-byte-swizzled box layout and leave by TMA; rows of a ragged last
            // box, and fp32 rows, are stored directly.
            const int i = row;
            const bool hit = (pset[(ph * 2 + g) * 4 + (i >> 5)] >> (i & 31)) & 1u;
            const float f = hit ? __int_as_float(0x7fc00000) : f_out;  // NaN * z is NaN
            const int nfull = n & ~31;
            const bool staged = sizeof(Tout) == 2 && i < nfull;
            Tout *orow = static_cast<Tout *>(p.o) + ((int64_t)(cur.lo + i) * p.hv_n + hv_of(cur, g)) * kD;
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
                            *reinterpret_cast<uint4 *>(vbuf + sw128_offset(i, cc * 32 + q * 8)) = w;
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
                tmem_ld32_nowait(wz + lane_base + 128, za);
                tmem_wait_ld_into(za);
#pragma unroll 1
                for (int cc = 0; cc < 4; cc += 2) {
                    tmem_ld32_nowait(wz + lane_base + 128 + (cc + 1) * 32, zb);
                    o_chunk(za, cc);
                    tmem_wait_ld_into(zb);
                    if (cc < 2) tmem_ld32_nowait(wz + lane_base + 128 + (cc + 2) * 32, za);
                    o_chunk(zb, cc + 1);
                    if (cc < 2) tmem_wait_ld_into(za);
                }
            }
            tc_fence_before();
            mbar_arrive(&bar[B_ZF0 + g]);
            // staged rows are visible to the TMA engine; every thread of the group
            // is done with its V/R row before the buffer is reloaded
            fence_proxy_async_smem();
            named_sync(2 + g, 128);
            if (sizeof(Tout) == 2 && issuer && item_good && nfull > 0) {
                for (int h = 0; h < 2; ++h)
                    for (int r = 0; r < (nfull >> 5); ++r)
                        tma_store_3d(&tmO, vbuf + h * 16384 + r * 4096, h * 64, hv_of(cur, g), cur.lo + 32 * r);
                bulk_commit();
                bulk_wait_read();
            }
            if (!more) break;
            if (issuer) issue_v(nx, g);  // the buffer is free again
            cur = nx;
        }
    } else {
        // ======================= aux warps ====================================
        const int i = tid & 127;
        // g and beta of both value heads of a unit at node i (loaded a unit ahead)
        auto load_gb = [&](const Unit &u, float (&gb)[4]) {
            gb[0] = gb[1] = gb[2] = gb[3] = 0.f;
            if (i < u.n) {
                const int64_t gi = u.lo + i;
                gb[0] = __ldg(p.g + gi * p.hv_n + u.hv0);
                gb[1] = __ldg(p.beta + gi * p.hv_n + u.hv0);
                gb[2] = __ldg(p.g + gi * p.hv_n + hv_of(u, 1));
                gb[3] = __ldg(p.beta + gi * p.hv_n + hv_of(u, 1));
            }
        };
        // Per-head node data of a unit: g, beta and the decay sums along the
        // paths (which `full` rebuilds, with the descriptor checks and the
        // descendant rows, when the request changes).  Arrives on B_DESC.
        auto meta = [&](const Unit &u, int pp, bool full, const float (&gb)[4]) {
            int pi = -1, di = 0;
            uint32_t mw[4] = {0u, 0u, 0u, 0u};
            bool tail_zero = true;  // words past the fourth (rows of a wider descriptor) are empty
            if (full && i < u.n) {
                const int64_t gi = u.lo + i;
                pi = __ldg(p.parent + gi);
                di = __ldg(p.depth + gi);
#pragma unroll
                for (int w = 0; w < 4; ++w) mw[w] = w < p.words ? __ldg(p.mask + gi * p.stride + w) : 0u;
                for (int w = 4; w < p.stride; ++w) tail_zero = tail_zero && __ldg(p.mask + gi * p.stride + w) == 0u;
            }
            named_sync(4, 128);  // the previous unit's node data is no longer read
            fhead[i] = gb[0];
            fhead[4 * kN + i] = gb[1];
            fhead[5 * kN + i] = gb[2];
            fhead[9 * kN + i] = gb[3];
            if (i < 8) pset[pp * 8 + i] = 0u;
            if (full) {
                par[i] = pi;
                dep[i] = di;
#pragma unroll
                for (int w = 0; w < 4; ++w) msk[i * 4 + w] = mw[w];
                // raw ancestor rows start at zero (entries past a node's depth stay zero)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    reinterpret_cast<float4 *>(Xs + i * kXS)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    reinterpret_cast<float4 *>(Ys + i * kXS)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (i == 0) s_err[pp] = 0;
            } else if (i == 0) {
                s_err[pp] = s_err[pp ^ 1];  // same request
            }
            named_sync(4, 128);
            if (full && i < u.n) {
                // validation: parent in [-1, i), depth and mask row consistent with the parent's
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
                    if (!same || !tail_zero) e = GDN_DEV_BAD_DESC;
                    else if (di > kMaxDepth) e = GDN_DEV_TOO_DEEP;
                }
                if (e) atomicOr(&s_err[pp], e);
                // path: the set bits of the mask row, root first; at most kMaxDepth
                // entries even for a malformed row
                int l = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t word = mw[w];
                    while (word && l < kMaxDepth) {
                        const int j = w * 32 + __ffs(word) - 1;
                        word &= word - 1;
                        path[i * kMaxDepth + l++] = (uint8_t)j;
                    }
                }
            }
            // gamma of both heads along the path (its length is the depth, clamped;
            // a malformed row's outputs are not stored)
            {
                int node_at[kMaxDepth];
                const int d = load_path(path, dep, i, u.n, node_at);
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int l = 0; l < kMaxDepth; ++l) {
                    const float a0 = fhead[node_at[l]], a1 = fhead[5 * kN + node_at[l]];
                    acc0 += l < d ? a0 : 0.f;
                    acc1 += l < d ? a1 : 0.f;
                }
                const bool in = i < u.n;
                fhead[kN + i] = acc0;
                fhead[2 * kN + i] = in ? expf(acc0) : 0.f;
                fhead[3 * kN + i] = in ? expf(fmaxf(acc0, kGammaFloor)) : 1.f;
                fhead[6 * kN + i] = acc1;
                fhead[7 * kN + i] = in ? expf(acc1) : 0.f;
                fhead[8 * kN + i] = in ? expf(fmaxf(acc1, kGammaFloor)) : 1.f;
            }
            if (full) {
                // mask rows become descendant rows: bit i of row a iff a is on i's
                // path.  Tree warp w owns word w of every row: the transpose of the
                // 32 x 32 bit block (its nodes i) x (word c of their ancestor rows),
                // by five rounds of shuffles (block transpose of Hacker's Delight,
                // section 7-3, on bit-reversed words so that bit c stands for
                // column c); zero for c > w.
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
                named_sync(4, 128);  // every ancestor row has been read by the validation
#pragma unroll
                for (int c = 0; c < 4; ++c) msk[(c * 32 + lane) * 4 + quad] = mine[c];
                if (i == 0 && s_err[pp]) flag(p.status, s_err[pp]);
            }
            named_sync(4, 128);
            mbar_arrive(&bar[B_DESC]);
        };
        float gb[4];
        load_gb(cur, gb);
        meta(cur, 0, true, gb);
        griddep_wait();  // S0 may be the output of the preceding grid (a commit)
#pragma unroll 1
        for (int g = 0; g < 2; ++g) convert(cur, g);
        for (int it = 0;; ++it) {
            const int ph = it & 1;
            Unit nx;
            const bool more = next_unit(cur, nx);
            if (more) load_gb(nx, gb);  // the next unit's g and beta, in flight during this one
            // P rows of head A into its S space, free once its S0 MMA is done
            int node_at[kMaxDepth];
            const int myd = load_path(path, dep, i, cur.n, node_at);
            ok = mbar_wait(&bar[B_SCAT], ph) && ok;  // every X and Y entry is in
            float P[kMaxDepth];
            p_solve(Xs, Ys, fhead, i, myd, node_at, P);
            ok = mbar_wait(&bar[B_S01], ph) && ok;  // after both S0 MMAs: the K/Q space is free
            p_write(sm + OFF_KQ, i, myd, node_at, P);
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_P0]);
            if (!more) break;
            // the next unit's tree data, once the tree and state warps hold this unit's
            ok = mbar_wait(&bar[B_META0], ph) && ok;
            ok = mbar_wait(&bar[B_META1], ph) && ok;
            ok = mbar_wait(&bar[B_META2], ph) && ok;
            meta(nx, ph ^ 1, nx.meta, gb);
            // the next unit's head-A state tile (the tree warps convert head B's)
            convert(nx, 0);
            cur = nx;
        }
    }
    if (!ok) flag(p.status, GDN_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

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
    // rows of mask_words words, of which a tree of at most 128 nodes uses the first four
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.words = a.mask_words < 4 ? a.mask_words : 4;
    p.stride = a.mask_words; p.probe = wait_probe_polls();
    p.group = a.n_v_heads / a.n_k_heads; p.npair = (p.group + 1) / 2;
    p.total = a.total_nodes; p.units = a.batch * a.n_k_heads * p.npair; p.scale = a.scale;
    p.offsets = a.node_offsets; p.parent = a.parent; p.depth = a.depth; p.mask = a.anc_mask;
    p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.o = a.o; p.status = a.dev_status;
    static int have_bf16[16], have_f32[16];
    auto kern = a.out_dtype == GDN_BF16 ? verify_tc_kernel<__nv_bfloat16> : verify_tc_kernel<float>;
    cudaError_t e = ensure_smem(kern, kSmemBytes, a.out_dtype == GDN_BF16 ? have_bf16 : have_f32);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    // persistent: one block per SM (it takes all 512 tensor-memory columns)
    cfg.gridDim = dim3((unsigned)std::min(p.units, sm_count()));
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
