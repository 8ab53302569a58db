// verify_wide.cu -- tcgen05/TMA tree verification for trees of up to 256 nodes:
// bf16 tokens, d_k = d_v = 128, depth at most 16 (sm_103a).
//
// The same computation as verify_tc.cu ("Trees from Marginals", gist.science
// Technical Summary, section 3 "Rollback-Free Tree Verification for GDN"):
//     (I + X) U = R = beta * (V - e^gamma * K S0^T),   O = scale * (e^gamma * Q S0^T + Y U)
// with X, Y the ancestor-masked, decay-weighted K K^T and Q K^T.  Row i of
// P = Y (I + X)^-1 is found by the decay-free back substitution along i's path
//     P'[l] = (q_i . k_l) - sum_{a > l} P'[a] beta_a (k_a . k_l),   P[l] = e^(gamma_i - gamma_l) P'[l]
// and O = e^gamma Z + P R with Z = Q S0^T.
//
// The nodes form two tiles of 128 (T1 = nodes 0..127, T2 = 128..255; the tensor
// memory lane is the node within its tile).  Because the tree is sorted
// topologically, a node of T1 has its ancestors in T1, so P is block-lower-
// triangular: O_T1 = e^gamma Z_T1 + P11 R_T1 and O_T2 = e^gamma Z_T2 + P21 R_T1 + P22 R_T2.
//
// One block of 256 threads per SM walks a contiguous range of (request, value
// head) items; thread t is node t.  Per item, in order:
//   1. node data (paths, gamma, descriptor checks, descendant rows; kept while
//      the request stays); K and Q arrive by TMA, S0 is already bf16.
//   2. Gram of the ancestors in T1: K_T1 [K;Q]^T (N = 256 + 256, all 512 tensor-
//      memory columns), scattered into raw X and Y rows of every descendant; then
//      Z = Q S0^T and the Gram of the ancestors in T2, K_T2 [K_T2;Q_T2]^T, which
//      frees the Q space for V; the second scatter; W = K S0^T.  The raw rows hold
//      no value-head data, so the next value head of the same key head keeps them
//      and skips the Grams (its K and Q come again, from L2).
//   3. P rows into the K and S0 spaces (P11 | P21 | P22); R over V; Z_T1 += P11
//      R_T1, Z_T2 += P21 R_T1 + P22 R_T2.
//   4. The next item's fp32 state tile by bulk copy into the K space (free once
//      the output products are done) while the epilogue runs, staged over R and
//      stored by TMA; then the state tile to bf16, and the next K and Q loads.
// Every mbarrier completes once per item (the Gram's once per Gram); every wait
// is bounded, and a timeout sets GDN_DEV_TIMEOUT.  A non-finite right-hand side
// row is replaced by zero in the output products and its subtree's outputs are
// set to NaN.
#include <algorithm>

#include "internal.cuh"
#include "sm100.cuh"
#include "tc_tiles.cuh"

namespace gdn {
namespace {

using namespace sm100;
using namespace tiles;

constexpr float kGammaFloor = -80.f;

// Block shape and shared-memory layout (bytes from the dynamic base, which is
// 1024-aligned) for NT node tiles of 128 and paths of at most MAXD nodes:
// NT = 2, MAXD = 16 for trees of up to 256 nodes; NT = 1, MAXD = 32 or 64 for
// trees of up to 128 nodes deeper than the one-tile kernel of verify_tc.cu takes.
// Where the next item's fp32 state tile waits for its conversion to bf16:
enum StageMode {
    kStageK,       // in the K space, once the output products are done (two tiles)
    kStageOwn,     // in a 64 KB region of its own, loading during the whole item
    kStageDirect,  // nowhere: converted straight from global memory (paths of up to
                   // 64 nodes leave no room for a staging region)
};
template <int NT, int MAXD>
struct Cfg {
    static constexpr int kT = 128 * NT;     // threads per block = node slots
    static constexpr int kNW = 128 * NT;    // nodes
    static constexpr int kMaxDepth = MAXD;
    static constexpr int kXS = MAXD + 4;    // row stride (floats) of the raw X and Y rows
    static constexpr int kWords = 4 * NT;   // mask words per node
    static constexpr int kKB = kNW * 128;   // bytes of one 64-column k-block of K or Q
    // K [2 k-blocks][kNW rows][128 B]; then P11 (+0) and P21 (+32 KB)
    static constexpr int OFF_K = 0;
    // Q [2 k-blocks][kNW rows][128 B]; then V|R|outputs of T1 (+0) and T2 (+32 KB)
    static constexpr int OFF_Q = 2 * kKB;
    // S0 bf16 [2 k-blocks][128][128 B]; then P22
    static constexpr int OFF_S0 = 4 * kKB;
    static constexpr StageMode kStage = NT == 2 ? kStageK : MAXD <= 32 ? kStageOwn : kStageDirect;
    static constexpr int OFF_STG = kStage == kStageOwn ? OFF_S0 + 32768 : OFF_K;  // fp32 staging (unused when direct)
    static constexpr int OFF_X = kStage == kStageOwn ? OFF_STG + 65536 : OFF_S0 + 32768;  // float [kNW][kXS] raw k.k of strict ancestors
    static constexpr int OFF_Y = OFF_X + kNW * kXS * 4;            // float [kNW][kXS] raw q.k of ancestors
    static constexpr int OFF_MASK = OFF_Y + kNW * kXS * 4;         // uint32 [kNW][kWords] ancestor, then descendant rows
    static constexpr int OFF_PATH = OFF_MASK + kNW * kWords * 4;   // uint8 [kNW][MAXD]
    static constexpr int OFF_F = OFF_PATH + kNW * MAXD;            // float [2 items][graw, gam, egt, eg, bet][kNW]
    static constexpr int OFF_I = OFF_F + 2 * 5 * kNW * 4;          // int dep, par [kNW]
    static constexpr int OFF_MISC = OFF_I + 2 * kNW * 4;           // tmem slot; pset[8]; err
    static constexpr int OFF_BAR = OFF_MISC + 64;
    static constexpr int kSmemBytes = OFF_BAR + 11 * 8;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(MAXD % 16 == 0, "path rows are read 16 bytes at a time");
};
// K, Q arrived; first Gram done, scattered; Q products done (the Q space is
// free); second scatter; W done (the K and S0 spaces are free); V arrived;
// output products done; next state tile arrived; wait probe
enum { W_K, W_Q, W_G1, W_SC1, W_G2, W_SC2, W_S0M, W_V, W_OUT, W_S0F, W_PROBE, W_BARS };
static_assert(W_BARS == 11, "barrier count in Cfg");

struct WideParams {
    int hk_n, hv_n, words, stride, total, items;
    int probe;  // > 0: thread 0 makes one wait of `probe` polls on W_PROBE (test hook)
    float scale;
    const int32_t *offsets, *parent, *depth;
    const uint32_t *mask;
    const float *g, *beta, *S0;
    void *o;
    int32_t *status;
};

struct Item {
    int idx, b, hv, hk, lo, n;
};

// The first item in [idx, end) whose request is non-empty and well placed;
// others are flagged (when `report`) and passed over.
__device__ bool find_item(const WideParams &p, int idx, int end, int max_n, bool report, Item &it) {
    for (; idx < end; ++idx) {
        const int b = idx / p.hv_n;
        const int lo = __ldg(p.offsets + b);
        const int n = __ldg(p.offsets + b + 1) - lo;
        if (n == 0) continue;
        if (n > max_n || lo < 0 || lo + n > p.total) {
            if (report) flag(p.status, n > max_n ? GDN_DEV_TOO_MANY : GDN_DEV_BAD_DESC);
            continue;
        }
        it.idx = idx;
        it.b = b;
        it.hv = idx % p.hv_n;
        it.hk = it.hv / (p.hv_n / p.hk_n);
        it.lo = lo;
        it.n = n;
        return true;
    }
    return false;
}

// Thread 0: the item's fp32 state tile (64 KB, contiguous) into `dst`.
__device__ __forceinline__ void issue_state(const WideParams &p, const Item &it, uint8_t *dst, uint64_t *bar) {
    const uint8_t *src = reinterpret_cast<const uint8_t *>(p.S0 + ((int64_t)it.b * p.hv_n + it.hv) * (kD * kD));
    mbar_arrive_expect_tx(bar, 65536u);
    for (int c = 0; c < 4; ++c) bulk_load(dst + c * 16384, src + c * 16384, 16384u, bar);
}

// Thread 0: the item's K or Q rows (boxes of 32 nodes, both 64-column halves,
// k-blocks `kb_bytes` apart).
__device__ __forceinline__ void issue_tokens(const CUtensorMap *map, const Item &it, uint8_t *dst, uint64_t *bar,
                                             int kb_bytes) {
    const int nb = (it.n + 31) >> 5;
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * nb * 4096));
    for (int kb = 0; kb < 2; ++kb)
        for (int r = 0; r < nb; ++r) tma_load_3d(dst + kb * kb_bytes + r * 4096, map, bar, kb * 64, it.hk, it.lo + 32 * r);
}

template <typename Tout, int NT, int MAXD>
__global__ void __launch_bounds__(128 * NT, 1)
verify_wide_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, WideParams p) {
    using C = Cfg<NT, MAXD>;
    constexpr int kT = C::kT, kNW = C::kNW, kMaxDepth = C::kMaxDepth, kXS = C::kXS, kWords = C::kWords, kKB = C::kKB;
    constexpr int OFF_K = C::OFF_K, OFF_Q = C::OFF_Q, OFF_S0 = C::OFF_S0, OFF_STG = C::OFF_STG, OFF_X = C::OFF_X,
                  OFF_Y = C::OFF_Y, OFF_MASK = C::OFF_MASK, OFF_PATH = C::OFF_PATH, OFF_F = C::OFF_F, OFF_I = C::OFF_I,
                  OFF_MISC = C::OFF_MISC, OFF_BAR = C::OFF_BAR;
    extern __shared__ __align__(1024) uint8_t sm[];
    float *Xs = reinterpret_cast<float *>(sm + OFF_X);
    float *Ys = reinterpret_cast<float *>(sm + OFF_Y);
    uint32_t *msk = reinterpret_cast<uint32_t *>(sm + OFF_MASK);
    uint8_t *path = sm + OFF_PATH;
    float *fbase = reinterpret_cast<float *>(sm + OFF_F);
    int *dep = reinterpret_cast<int *>(sm + OFF_I), *par = dep + kNW;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    uint32_t *pset = tslot + 1;                       // [8]: nodes whose output is poisoned
    int *s_err = reinterpret_cast<int *>(tslot + 9);  // descriptor errors of the item
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, grp = warp >> 2;
    const int i = tid;                 // node
    const int rr = i & 127;            // row of the node in its tile = tensor-memory lane
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0) flag(p.status, GDN_DEV_INTERNAL);
        return;
    }
    // a contiguous range of items per block, so that the value heads of one key
    // head follow each other and share the tree data, the Gram and its scatter
    const int end = (int)(((int64_t)(blockIdx.x + 1) * p.items) / gridDim.x);
    Item cur;
    if (!find_item(p, (int)(((int64_t)blockIdx.x * p.items) / gridDim.x), end, kNW, tid == 0, cur)) {
        griddep_wait();  // the block ends after the preceding grid, like the others
        return;
    }

    if (tid == 0) {
        for (int k = 0; k < W_BARS; ++k) mbar_init(&bar[k], k == W_SC1 || k == W_SC2 ? (uint32_t)kT : 1u);
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
    if (p.probe > 0 && tid == 0) ok = mbar_wait(&bar[W_PROBE], 0, (uint32_t)p.probe);
    griddep_wait();  // S0 may be the output of a preceding grid

    const uint32_t id_nw = idesc_bf16_f32(128, kNW), id_n128 = idesc_bf16_f32(128, 128);
    const uint32_t id_out = id_n128 | (1u << 16);  // B (R) is MN-major

    // The fp32 state tile in the staging space (or global memory) to bf16 in the S0 space (B
    // operand, K-major, 128-byte swizzle): rows 16 warp .. 16 warp + 15, and 64
    // rows further on too with one tile's four warps; lane l holds columns
    // 4l .. 4l + 3;
    // then, with two tiles, the K space takes the item's keys.
    int sph = 0;
    auto convert_state = [&](const Item &it) {
        const float4 *src;
        if constexpr (C::kStage == kStageDirect) {
            src = reinterpret_cast<const float4 *>(p.S0 + ((int64_t)it.b * p.hv_n + it.hv) * (kD * kD));
        } else {
            ok = mbar_wait(&bar[W_S0F], sph) && ok;
            sph ^= 1;
            src = reinterpret_cast<const float4 *>(sm + OFF_STG);
        }
#pragma unroll
        for (int r0 = warp * 16; r0 < kD; r0 += kT / 2) {  // 16 rows per warp and pass
            float4 sa[8], sb[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                sa[r] = src[(r0 + r) * 32 + lane];
                sb[r] = src[(r0 + 8 + r) * 32 + lane];
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                *reinterpret_cast<uint2 *>(sm + OFF_S0 + sw128_offset(r0 + r, 4 * lane)) =
                    make_uint2(pack_bf16(sa[r].x, sa[r].y), pack_bf16(sa[r].z, sa[r].w));
                *reinterpret_cast<uint2 *>(sm + OFF_S0 + sw128_offset(r0 + 8 + r, 4 * lane)) =
                    make_uint2(pack_bf16(sb[r].x, sb[r].y), pack_bf16(sb[r].z, sb[r].w));
            }
        }
        fence_proxy_async_smem();  // the bf16 tile is read, the staging space written, by the async proxy
        __syncthreads();
        if (tid == 0 && C::kStage == kStageK) issue_tokens(&tmK, it, sm + OFF_K, &bar[W_K], kKB);
    };
    if (tid == 0) {
        if (C::kStage != kStageDirect) issue_state(p, cur, sm + OFF_STG, &bar[W_S0F]);
        issue_tokens(&tmQ, cur, sm + OFF_Q, &bar[W_Q], kKB);
        if (C::kStage != kStageK) issue_tokens(&tmK, cur, sm + OFF_K, &bar[W_K], kKB);
    }
    convert_state(cur);
    // the item after the current one is looked up one item ahead, off the critical path
    Item nx;
    bool more = find_item(p, cur.idx + 1, end, kNW, tid == 0, nx);

    int prev_b = -1, prev_hk = -1, gph = 0;
    for (int it = 0;; ++it) {
        const int ph = it & 1;
        const int n = cur.n, nb = (n + 31) >> 5;
        const bool two = NT == 2 && n > 128;  // block-uniform: the second tile has nodes
        const bool same_req = cur.b == prev_b;               // tree data kept
        const bool same_kh = same_req && cur.hk == prev_hk;  // raw X and Y rows kept too
        prev_b = cur.b;
        prev_hk = cur.hk;
        // per-head node data (g, beta, decay sums) of this item, and of the next one
        // when it is another value head of the same request (made during this item)
        float *graw = fbase + ph * 5 * kNW;
        float *gam = graw + kNW, *egt = graw + 2 * kNW, *eg = graw + 3 * kNW, *bet = graw + 4 * kNW;
        float *graw_n = fbase + (ph ^ 1) * 5 * kNW;
        const bool pre_next = more && nx.b == cur.b;
        // with a staging region of its own, the next state tile loads during the whole item
        if (C::kStage == kStageOwn && tid == 0 && more) issue_state(p, nx, sm + OFF_STG, &bar[W_S0F]);
        float gr_n = 0.f, br_n = 0.f;  // in flight during the item
        if (pre_next && i < n) {
            gr_n = __ldg(p.g + (int64_t)(nx.lo + i) * p.hv_n + nx.hv);
            br_n = __ldg(p.beta + (int64_t)(nx.lo + i) * p.hv_n + nx.hv);
        }
        // ---- 1. node data -------------------------------------------------------
        int pi = -1, di = 0;
        uint32_t mw[kWords];
#pragma unroll
        for (int w = 0; w < kWords; ++w) mw[w] = 0u;
        float gr = 0.f, br = 0.f;
        if (i < n && !same_req) {
            const int64_t gi = cur.lo + i;
            pi = __ldg(p.parent + gi);
            di = __ldg(p.depth + gi);
#pragma unroll
            for (int w = 0; w < kWords; ++w) mw[w] = w < p.words ? __ldg(p.mask + gi * p.stride + w) : 0u;
            gr = __ldg(p.g + gi * p.hv_n + cur.hv);
            br = __ldg(p.beta + gi * p.hv_n + cur.hv);
        }
        if (!same_req) {
            par[i] = pi;
            dep[i] = di;
#pragma unroll
            for (int w = 0; w < kWords; ++w) msk[i * kWords + w] = mw[w];
            if (i == 0) *s_err = 0;
        }
        if (!same_kh) {
#pragma unroll
            for (int q = 0; q < kXS / 4; ++q) {
                reinterpret_cast<float4 *>(Xs + i * kXS)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(Ys + i * kXS)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (!same_req) {
            graw[i] = gr;
            bet[i] = br;
        }
        if (i < 8) pset[i] = 0u;
        __syncthreads();
        // validation: parent in [-1, i), depth and mask row consistent with the parent's
        if (i < n && !same_req) {
            int e = 0;
            if (pi < -1 || pi >= i) {
                e = GDN_DEV_BAD_TREE;
            } else {
                const int want = pi < 0 ? 1 : dep[pi] + 1;
                bool same = di == want;
#pragma unroll
                for (int w = 0; w < kWords; ++w) {
                    const uint32_t expect = (pi < 0 ? 0u : msk[pi * kWords + w]) | ((i >> 5) == w ? 1u << (i & 31) : 0u);
                    same = same && mw[w] == expect;
                }
                if (!same) e = GDN_DEV_BAD_DESC;
                else if (di > kMaxDepth) e = GDN_DEV_TOO_DEEP;
            }
            if (e) atomicOr(s_err, e);
            // path: the set bits of the mask row, root first; at most kMaxDepth
            // entries even for a malformed row
            int l = 0;
#pragma unroll
            for (int w = 0; w < kWords; ++w) {
                uint32_t word = mw[w];
                while (word && l < kMaxDepth) {
                    const int j = w * 32 + __ffs(word) - 1;
                    word &= word - 1;
                    path[i * kMaxDepth + l++] = (uint8_t)j;
                }
            }
        }
        // node i's path (i itself past the depth, so every index stays in range)
        const int myd = i < n ? min(max(dep[i], 0), kMaxDepth) : 0;
        int node_at[kMaxDepth];
#pragma unroll
        for (int h = 0; h < kMaxDepth / 16; ++h) {
            const uint4 pr = reinterpret_cast<const uint4 *>(path + i * kMaxDepth)[h];
            const uint32_t pw[4] = {pr.x, pr.y, pr.z, pr.w};
#pragma unroll
            for (int l = 16 * h; l < 16 * h + 16; ++l)
                node_at[l] = l < myd ? (int)((pw[(l >> 2) & 3] >> (8 * (l & 3))) & 0xFFu) : i;
        }
        // decay sums along the path (made by the previous item for the same request)
        auto decay_sums = [&](float *f) {
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l) acc += l < myd ? f[node_at[l]] : 0.f;
            f[kNW + i] = acc;
            f[2 * kNW + i] = i < n ? expf(acc) : 0.f;
            f[3 * kNW + i] = i < n ? expf(fmaxf(acc, kGammaFloor)) : 1.f;
        };
        if (!same_req) decay_sums(graw);
        // mask rows become descendant rows: bit i of row a iff a is on i's path.
        // Warp w owns word w of every row: the transpose of the 32 x 32 bit block
        // (its nodes i) x (word c of their ancestor rows), by five rounds of
        // shuffles (block transpose of Hacker's Delight, section 7-3, on bit-
        // reversed words so that bit c stands for column c); zero for c > w.
        if (!same_req) {  // block-uniform
            uint32_t mine[kWords];
#pragma unroll
            for (int c = 0; c < kWords; ++c) {
                mine[c] = 0u;
                if (c > warp) continue;  // warp-uniform
                uint32_t x = __brev(mw[c]);
                uint32_t m = 0x0000FFFFu;
#pragma unroll
                for (int j = 16; j != 0; j >>= 1, m ^= (m << j)) {
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, x, j);
                    x = (lane & j) ? x ^ (((other ^ (x >> j)) & m) << j) : x ^ ((x ^ (other >> j)) & m);
                }
                mine[c] = __brev(x);
            }
            __syncthreads();  // every ancestor row has been read by the validation
#pragma unroll
            for (int c = 0; c < kWords; ++c) msk[(c * 32 + lane) * kWords + warp] = mine[c];
            __syncthreads();
        }
        const bool item_good = *s_err == 0;
        if (i == 0 && !item_good && !same_req) flag(p.status, *s_err);

        // ---- 2. Grams, scatters and the state products -----------------------------
        // lane a holds k_a.k_j and k_a.q_j and writes them into the raw ancestor
        // rows of its descendants j (X strict, Y inclusive); the warps of both
        // groups share a lane quarter and take alternate 32-column chunks
        // (tensor-memory column of node chunk cc: (cc - org) * 32 from kk and kq)
        auto scatter = [&](int a, int cc0, int org, uint32_t kk, uint32_t kq) {
            const int da = a < n ? min(max(dep[a], 1), kMaxDepth) : 1;
#pragma unroll 1
            for (int cc = cc0 + grp; cc < kWords; cc += NT) {
                const uint32_t dm = msk[a * kWords + cc];
                if (!__any_sync(0xffffffffu, dm != 0u)) continue;
                uint32_t v[32];
                tmem_ld32_nowait(kk + lane_base + (uint32_t)((cc - org) * 32), v);
                tmem_wait_ld_into(v);
                const uint32_t dx = cc == cc0 ? dm & ~(1u << lane) : dm;  // X is strictly lower
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if ((dx >> c) & 1u) Xs[(cc * 32 + c) * kXS + da - 1] = __uint_as_float(v[c]);
                tmem_ld32_nowait(kq + lane_base + (uint32_t)((cc - org) * 32), v);
                tmem_wait_ld_into(v);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if ((dm >> c) & 1u) Ys[(cc * 32 + c) * kXS + da - 1] = __uint_as_float(v[c]);
            }
        };
        // k-step ks of a 128-row operand at `base` (two 16 KB k-blocks per 128 rows)
        auto kdesc = [&](int off, int ks) {
            return smem_desc(smem_u32(sm + off + (ks >> 2) * kKB + (ks & 3) * 32), 16, 1024, 2);
        };
        auto sdesc = [&](int ks) {  // S0 bf16: 128 rows, k-blocks of 16 KB
            return smem_desc(smem_u32(sm + OFF_S0 + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
        };
        // Z_t = Q_t S0^T into columns 256 + 128 t
        auto issue_z = [&]() {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                mma_bf16(tmem + 256, kdesc(OFF_Q, ks), sdesc(ks), id_n128, ks > 0);
                if (two) mma_bf16(tmem + 384, kdesc(OFF_Q + 16384, ks), sdesc(ks), id_n128, ks > 0);
            }
        };
        // W_t = K_t S0^T into columns 128 t
        auto issue_w = [&]() {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                mma_bf16(tmem, kdesc(OFF_K, ks), sdesc(ks), id_n128, ks > 0);
                if (two) mma_bf16(tmem + 128, kdesc(OFF_K + 16384, ks), sdesc(ks), id_n128, ks > 0);
            }
        };
        // V of both tiles into the Q space, once the Q products are done
        auto issue_v = [&]() {
            ok = mbar_wait(&bar[W_G2], ph) && ok;
            const int nb1 = min(nb, 4), nb2 = nb - nb1;
            mbar_arrive_expect_tx(&bar[W_V], (uint32_t)(2 * nb * 4096));
            for (int h = 0; h < 2; ++h) {
                for (int r = 0; r < nb1; ++r)
                    tma_load_3d(sm + OFF_Q + h * 16384 + r * 4096, &tmV, &bar[W_V], h * 64, cur.hv, cur.lo + 32 * r);
                for (int r = 0; r < nb2; ++r)
                    tma_load_3d(sm + OFF_Q + 32768 + h * 16384 + r * 4096, &tmV, &bar[W_V], h * 64, cur.hv,
                                cur.lo + 128 + 32 * r);
            }
        };
        if (!same_kh) {  // block-uniform
            if (tid == 0) {
                ok = mbar_wait(&bar[W_K], ph) && ok;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = kdesc(OFF_K, ks);
                    // K_T1 K^T (N = kNW: the B operand spans every tile's rows)
                    mma_bf16(tmem, a, a, id_nw, ks > 0);
                }
                ok = mbar_wait(&bar[W_Q], ph) && ok;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)  // K_T1 Q^T
                    mma_bf16(tmem + 256, kdesc(OFF_K, ks), kdesc(OFF_Q, ks), id_nw, ks > 0);
                mma_commit(&bar[W_G1]);
            }
            ok = mbar_wait(&bar[W_G1], gph) && ok;
            tc_fence_after();
            // ancestors in T1: lanes quad * 32 + lane, chunks quad .. 7 of all 256 columns
            scatter(quad * 32 + lane, quad, 0, tmem, tmem + 256);
            tc_fence_before();
            mbar_arrive(&bar[W_SC1]);
            if (tid == 0) {
                ok = mbar_wait(&bar[W_SC1], gph) && ok;  // the first Gram has been read out
                tc_fence_after();
                issue_z();
                if (two) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t a = kdesc(OFF_K + 16384, ks);
                        mma_bf16(tmem, a, a, id_n128, ks > 0);                                 // K_T2 K_T2^T
                        mma_bf16(tmem + 128, a, kdesc(OFF_Q + 16384, ks), id_n128, ks > 0);   // K_T2 Q_T2^T
                    }
                }
                mma_commit(&bar[W_G2]);
                issue_v();
            }
            ok = mbar_wait(&bar[W_G2], ph) && ok;
            ok = mbar_wait(&bar[W_SC1], gph) && ok;  // every T1 ancestor's entries are in
            if (two) {
                tc_fence_after();
                // ancestors in T2: lanes 128 + quad * 32 + lane, chunks 4 + quad .. 7
                scatter(128 + quad * 32 + lane, 4 + quad, 4, tmem, tmem + 128);
            }
            tc_fence_before();
            mbar_arrive(&bar[W_SC2]);
            ok = mbar_wait(&bar[W_SC2], gph) && ok;  // every X and Y entry is in, the Gram columns are free
            gph ^= 1;
            if (tid == 0) {
                tc_fence_after();
                issue_w();
                mma_commit(&bar[W_S0M]);
            }
        } else if (tid == 0) {
            ok = mbar_wait(&bar[W_K], ph) && ok;
            ok = mbar_wait(&bar[W_Q], ph) && ok;
            tc_fence_after();
            issue_z();
            mma_commit(&bar[W_G2]);
            issue_w();
            mma_commit(&bar[W_S0M]);
            issue_v();
        }

        // ---- 3. P rows, right-hand side, output products ----------------------
        float P[kMaxDepth];
        {
#pragma unroll
            for (int q = 0; q < kMaxDepth / 4; ++q) {
                const float4 y = reinterpret_cast<const float4 *>(Ys + i * kXS)[q];
                P[4 * q] = y.x; P[4 * q + 1] = y.y; P[4 * q + 2] = y.z; P[4 * q + 3] = y.w;
            }
#pragma unroll
            for (int a = kMaxDepth - 1; a >= 1; --a) {
                // entries past the depth are zero, so a short path costs no branches
                const float4 *xr = reinterpret_cast<const float4 *>(Xs + node_at[a] * kXS);
                const float ca = a < myd ? P[a] * bet[node_at[a]] : 0.f;
#pragma unroll
                for (int q = 0; q < (a + 3) / 4; ++q) {
                    const float4 v = xr[q];
                    if (4 * q + 0 < a) P[4 * q + 0] = fmaf(-ca, v.x, P[4 * q + 0]);
                    if (4 * q + 1 < a) P[4 * q + 1] = fmaf(-ca, v.y, P[4 * q + 1]);
                    if (4 * q + 2 < a) P[4 * q + 2] = fmaf(-ca, v.z, P[4 * q + 2]);
                    if (4 * q + 3 < a) P[4 * q + 3] = fmaf(-ca, v.w, P[4 * q + 3]);
                }
            }
            const float gi = gam[i], inv = 1.f / eg[i];
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l) P[l] = l < myd ? P[l] * (expf(gi - gam[node_at[l]]) * inv) : 0.f;
        }
        if (pre_next) {
            graw_n[i] = gr_n;
            graw_n[4 * kNW + i] = br_n;
        }
        Item nn;
        const bool more_n = more && find_item(p, nx.idx + 1, end, kNW, tid == 0, nn);
        // P rows (A operands, K-major) once W is done with the K and S0 spaces
        ok = mbar_wait(&bar[W_S0M], ph) && ok;
        {
            uint8_t *pa = sm + (i < 128 ? OFF_K : OFF_K + 32768);  // P11 row i or P21 row i - 128
            uint8_t *pb = sm + OFF_S0;                             // P22 row i - 128
            if (i < 128 || two) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<uint4 *>(pa + sw128_offset(rr, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (i >= 128 && two) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<uint4 *>(pb + sw128_offset(rr, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int l = 0; l < kMaxDepth; ++l)
                if (l < myd) {
                    const int j = node_at[l];
                    uint8_t *dst = j < 128 ? pa : pb;
                    *reinterpret_cast<__nv_bfloat16 *>(dst + sw128_offset(rr, j & 127)) = __float2bfloat16_rn(P[l]);
                }
        }
        // R[j][n] = beta_j v[j][n] - beta_j e^gamma_j W[j][n] over V (same MN-major
        // layout); a row with a non-finite entry, and every row past the tree, is zero
        const int tile = i >> 7;
        uint8_t *vbuf = sm + OFF_Q + tile * 32768;
        const uint32_t wcol = tmem + (uint32_t)(tile * 128);
        const uint32_t zcol = tmem + 256 + (uint32_t)(tile * 128);
        const bool live = tile == 0 || two;  // the thread's tile takes part
        ok = mbar_wait(&bar[W_V], ph) && ok;
        tc_fence_after();
        if (live) {
            const float bj = bet[i], bej = bj * egt[i];
            float chk = 0.f;  // 0 * x: stays zero while every entry is finite
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t w[32];
                tmem_ld32_nowait(wcol + lane_base + cc * 32, w);
                tmem_wait_ld_into(w);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int n0 = cc * 32 + q * 8;
                    uint4 *at = reinterpret_cast<uint4 *>(vbuf + sw128_offset(rr, n0));
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
            }
            const bool bad = chk != 0.f;
            if (bad || i >= n) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    *reinterpret_cast<uint4 *>(vbuf + sw128_offset(rr, q * 8)) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (bad && i < n) {  // the row and every node below it
#pragma unroll
                for (int w = 0; w < kWords; ++w) atomicOr(&pset[w], msk[i * kWords + w]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            // Z_T1 += P11 R_T1; Z_T2 += P21 R_T1 + P22 R_T2
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t asub = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint64_t r1 = smem_desc(smem_u32(sm + OFF_Q + ks * 2048), 16384, 1024, 2);
                mma_bf16(tmem + 256, smem_desc(smem_u32(sm + OFF_K + asub), 16, 1024, 2), r1, id_out, true);
                if (two) {
                    const uint64_t r2 = smem_desc(smem_u32(sm + OFF_Q + 32768 + ks * 2048), 16384, 1024, 2);
                    mma_bf16(tmem + 384, smem_desc(smem_u32(sm + OFF_K + 32768 + asub), 16, 1024, 2), r1, id_out, true);
                    mma_bf16(tmem + 384, smem_desc(smem_u32(sm + OFF_S0 + asub), 16, 1024, 2), r2, id_out, true);
                }
            }
            mma_commit(&bar[W_OUT]);
        }
        if (pre_next) decay_sums(graw_n);  // the next item's g of every node is in
        if (tid == 0) {
            ok = mbar_wait(&bar[W_OUT], ph) && ok;
            // the K space is free: the next item's state tile (two tiles) or its
            // keys (one tile), during the epilogue
            if (more && C::kStage == kStageK) issue_state(p, nx, sm + OFF_STG, &bar[W_S0F]);
            if (more && C::kStage != kStageK) issue_tokens(&tmK, nx, sm + OFF_K, &bar[W_K], kKB);
        }
        ok = mbar_wait(&bar[W_OUT], ph) && ok;
        tc_fence_after();

        // ---- 4. epilogue ------------------------------------------------------
        // o[i][n] = scale * e^gamma'_i * Z[i][n], NaN for a poisoned row.  bf16 rows
        // of whole 32-node boxes are staged over R in the box layout and leave by
        // TMA; rows of a ragged last box, and fp32 rows, are stored directly.
        const int nt = tile == 0 ? min(n, 128) : max(n - 128, 0);  // rows of this tile
        const int nfull = nt & ~31;
        if (live) {
            const bool hit = (pset[i >> 5] >> (i & 31)) & 1u;
            const float f = hit ? __int_as_float(0x7fc00000) : p.scale * eg[i];  // NaN * z is NaN
            const bool store = item_good && i < n;
            const bool staged = sizeof(Tout) == 2 && rr < nfull;
            Tout *orow = static_cast<Tout *>(p.o) + ((int64_t)(cur.lo + i) * p.hv_n + cur.hv) * kD;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t zr[32];
                tmem_ld32_nowait(zcol + lane_base + cc * 32, zr);
                tmem_wait_ld_into(zr);
                float z[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) z[e] = f * __uint_as_float(zr[e]);
                if (!store) continue;
                if constexpr (sizeof(Tout) == 2) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w = make_uint4(pack_bf16(z[q * 8 + 0], z[q * 8 + 1]), pack_bf16(z[q * 8 + 2], z[q * 8 + 3]),
                                                   pack_bf16(z[q * 8 + 4], z[q * 8 + 5]), pack_bf16(z[q * 8 + 6], z[q * 8 + 7]));
                        if (staged)
                            *reinterpret_cast<uint4 *>(vbuf + sw128_offset(rr, cc * 32 + q * 8)) = w;
                        else
                            reinterpret_cast<uint4 *>(orow + cc * 32)[q] = w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        reinterpret_cast<float4 *>(orow + cc * 32)[q] =
                            make_float4(z[q * 4 + 0], z[q * 4 + 1], z[q * 4 + 2], z[q * 4 + 3]);
                }
            }
        }
        // each warp stores its own box of 32 staged rows (both 64-column halves)
        // as soon as it is written
        if (sizeof(Tout) == 2 && item_good && live && 32 * quad < nfull) {  // warp-uniform
            fence_proxy_async_smem();  // staged rows are visible to the TMA engine
            __syncwarp();
            if (lane == 0) {
                for (int h = 0; h < 2; ++h)
                    tma_store_3d(&tmO, vbuf + h * 16384 + quad * 4096, h * 64, cur.hv, cur.lo + tile * 128 + 32 * quad);
                bulk_commit();
                bulk_wait_read();  // the Q space may be loaded again
            }
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && more) issue_tokens(&tmQ, nx, sm + OFF_Q, &bar[W_Q], kKB);
        if (!more) break;
        convert_state(nx);  // its leading wait orders every thread after the epilogue
        cur = nx;
        nx = nn;
        more = more_n;
    }
    if (!ok) flag(p.status, GDN_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// One launch shape: NT node tiles, paths of at most MAXD nodes.
template <int NT, int MAXD>
cudaError_t launch_shape(const gdn_verify_args &a, cudaStream_t stream, bool after_commit, const CUtensorMap &tmK,
                         const CUtensorMap &tmQ, const CUtensorMap &tmV, const CUtensorMap &tmO, WideParams p) {
    using C = Cfg<NT, MAXD>;
    p.words = a.mask_words < C::kWords ? a.mask_words : C::kWords;
    static int have_bf16[16], have_f32[16];
    auto kern = a.out_dtype == GDN_BF16 ? verify_wide_kernel<__nv_bfloat16, NT, MAXD> : verify_wide_kernel<float, NT, MAXD>;
    cudaError_t e = ensure_smem(kern, C::kSmemBytes, a.out_dtype == GDN_BF16 ? have_bf16 : have_f32);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    // persistent: one block per SM (it takes all 512 tensor-memory columns)
    cfg.gridDim = dim3((unsigned)std::min(p.items, sm_count()));
    cfg.blockDim = dim3(C::kT);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    // after a commit of the state in the same stream, the launch may begin while
    // the commit drains (the kernel waits for it before its first state read)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = after_commit ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tmK, tmQ, tmV, tmO, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Two tiles (paths of up to 16 nodes) for trees of 129 to 256 nodes; one tile
// with paths of up to 32 or 64 nodes for smaller trees.
bool verify_wide_supported(const gdn_verify_args &a) {
    const bool shape = a.max_nodes > 128 ? a.max_nodes <= 256 && a.max_depth <= 16 : a.max_depth <= 64;
    return a.qkv_dtype == GDN_BF16 && a.d_k == kD && a.d_v == kD && shape && a.max_depth >= 1 &&
           a.total_nodes > 0 && tiles::aligned16(a.q) && tiles::aligned16(a.k) && tiles::aligned16(a.v) &&
           tiles::aligned16(a.S0) && tiles::aligned16(a.o) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_verify_wide(const gdn_verify_args &a, cudaStream_t stream, bool after_commit) {
    CUtensorMap tmK, tmQ, tmV, tmO;
    if (!encode_tokens(&tmK, a.k, a.n_k_heads, a.total_nodes) ||
        !encode_tokens(&tmQ, a.q, a.n_k_heads, a.total_nodes) ||
        !encode_tokens(&tmV, a.v, a.n_v_heads, a.total_nodes))
        return cudaErrorInvalidValue;
    if (a.out_dtype == GDN_BF16) {
        if (!encode_tokens(&tmO, a.o, a.n_v_heads, a.total_nodes)) return cudaErrorInvalidValue;
    } else {
        tmO = tmV;  // unused by the fp32-output kernel
    }
    WideParams p;
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.words = 0;
    p.stride = a.mask_words; p.probe = wait_probe_polls();
    p.total = a.total_nodes; p.items = a.batch * a.n_v_heads; p.scale = a.scale;
    p.offsets = a.node_offsets; p.parent = a.parent; p.depth = a.depth; p.mask = a.anc_mask;
    p.g = a.g; p.beta = a.beta; p.S0 = a.S0;
    p.o = a.o; p.status = a.dev_status;
    if (a.max_nodes > 128) return launch_shape<2, 16>(a, stream, after_commit, tmK, tmQ, tmV, tmO, p);
    if (a.max_depth <= 32) return launch_shape<1, 32>(a, stream, after_commit, tmK, tmQ, tmV, tmO, p);
    return launch_shape<1, 64>(a, stream, after_commit, tmK, tmQ, tmV, tmO, p);
}

}  // namespace gdn
