// commit_tc.cu -- delayed state commit on the tensor cores: bf16 k/v, d_k = d_v = 128,
// accepted paths of at most 32 nodes (sm_103a).
//
// "Trees from Marginals" (gist.science Technical Summary, section 3, Solution,
// last bullet): the state is committed in the next iteration along the accepted
// branch only.  For the accepted path p_1..p_L (gamma_t = sum of g over p_1..p_t)
//     u_t = beta_t (v_t - e^gamma_t S0 k_t) - sum_{s<t} beta_t e^(gamma_t - gamma_s) (k_t . k_s) u_s
//     S_new = e^gamma_L S0 + sum_t e^(gamma_L - gamma_t) u_t k_t^T
// which equals running the gated delta rule along the path.
//
// The same kernel, instantiated for selected nodes, gives the state at any
// chosen node (the path is the node's ancestor-mask row, root first), so that
// a later commit of one of them needs no recompute.
//
// Persistent blocks (two per SM) walk the (request, value head) items.  The
// next item's path data (keys, values, g, beta, node ids and their checks) is
// prepared into a second buffer while thread 0 waits for the current state
// tile's store, and the next tile is requested into L2.
// The contractions run on tcgen05 with fp32 accumulation, with a side as wide as
// the longest path (P = 16, or 32 for longer paths):
//     G  = K K^T       the path keys' Gram, for the chain coefficients
//     W  = S0 K^T      M = 128 state rows, N = P path keys, K = 128
//     U  = A K         M = 128 state rows, N = 128 columns, K = P path keys
// where A[row][t] = e^(gamma_L - gamma_t) u_t[row].  The fp32 operands S0 and
// A enter as bf16 hi + lo pairs (x = hi + lo to ~2^-17 relative) and the keys
// are exact in bf16, so the products keep fp32 accuracy.  The chain solve for
// u runs per state row in registers.  The state tile moves by TMA both ways and
// is fully read before it is overwritten, so S_new may alias S0.
#include <algorithm>

#include "internal.cuh"
#include "sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kT = 256;
constexpr int kD = 128;
// Shared memory (bytes from a 1024-aligned base) for paths of at most P nodes.
// Path data is double-buffered for P = 16 (one item's is prepared while the
// previous item's state tile is stored); for P = 32 one buffer keeps two
// blocks per SM (an item's path data is only prepared once the previous item's
// products are done, so one buffer serves as well).
template <int P>
struct CommitCfg {
    static constexpr int kMaxPath = P;
    static constexpr int kBufs = P == 16 ? 2 : 1;
    static constexpr int kKeyBytes = P * kD * 2;        // bf16 path keys [P][128], 128B swizzle (2 column blocks)
    static constexpr int kABytes = kD * P * 2;          // A hi or lo: bf16 [128][P] core-matrix layout
    static constexpr int OFF_TILE = 0;                  // fp32 state tile (TMA, 4 x [128][32], 128B swizzle); also
                                                        // S0 hi | lo as bf16 K-major tiles ([2][128][128 B] each)
    static constexpr int OFF_KEYS = 65536;              // [kBufs] path keys
    static constexpr int OFF_A = OFF_KEYS + kBufs * kKeyBytes;  // A hi | lo
    static constexpr int OFF_VP = OFF_A + 2 * kABytes;  // [kBufs] fp32 path values [P][128]
    static constexpr int OFF_COEF = OFF_VP + kBufs * P * kD * 4;  // fp32 [P][P]
    static constexpr int OFF_SCAL = OFF_COEF + P * P * 4;       // [kBufs] bet, egam, fdec, gam [P]; pn [P]
    static constexpr int kScal = 5 * P;                         // floats per buffer
    static constexpr int OFF_MISC = OFF_SCAL + kBufs * kScal * 4;  // tmem slot, bad path flags [2]
    static constexpr int OFF_BAR = OFF_MISC + 16;
    static constexpr int kSmemBytes = OFF_BAR + 5 * 8;  // barriers: tile, W, U, probe (never arrived on), Gram
    static_assert(2 * kSmemBytes + 2048 <= 233472, "two blocks per SM");
};

struct TcCommitParams {
    int hk_n, hv_n, total, items, batch, words;
    int probe;  // > 0: thread 0 makes one wait of `probe` polls on the probe barrier (test hook)
    const float *S0;
    const int32_t *offsets, *parent, *poff, *pidx;
    const int32_t *sel_req, *sel_node;  // selected nodes (state mode)
    const uint32_t *mask;               // ancestor-mask rows (state mode)
    const __nv_bfloat16 *k, *v;
    const float *g, *beta;
    int32_t *status;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// fp32 state tile written by TMA: column quarter q = col / 32 is a [128][32] box
// whose 16-byte chunks are permuted by row mod 8 (offset in floats).
__device__ __forceinline__ int tile_index(int row, int col) {
    return (col >> 5) * (kD * 32) + row * 32 + ((((col & 31) >> 2) ^ (row & 7)) << 2) + (col & 3);
}

// bf16 K-major 128B-swizzled tile with `rows` rows (byte offset).
__device__ __forceinline__ uint32_t sw128(int row, int k, int rows) {
    return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2);
}

// The t-th set bit (0-based, ascending) of a multi-word mask row, or -1.
__device__ __forceinline__ int nth_bit(const uint32_t (&m)[kMaxWords], int words, int t) {
#pragma unroll
    for (int w = 0; w < kMaxWords; ++w) {
        if (w >= words) break;
        const int c = __popc(m[w]);
        if (t < c) {
            uint32_t x = m[w];
            for (int k = 0; k < t; ++k) x &= x - 1;
            return w * 32 + __ffs(x) - 1;
        }
        t -= c;
    }
    return -1;
}

// kSel = false: item (request, value head) commits the request's accepted path
// into S_new.  kSel = true: item (selection s, value head) writes the state at
// node sel_node[s] of request sel_req[s] into row block s of S_sel.  Paths of at
// most P nodes.
template <bool kSel, int P>
__global__ void __launch_bounds__(kT, 2)
commit_tc_kernel(const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmSN,
                 TcCommitParams p) {
    using C = CommitCfg<P>;
    constexpr int kMaxPath = C::kMaxPath, kScal = C::kScal;
    constexpr int OFF_TILE = C::OFF_TILE, OFF_KEYS = C::OFF_KEYS, OFF_A = C::OFF_A, OFF_VP = C::OFF_VP,
                  OFF_COEF = C::OFF_COEF, OFF_SCAL = C::OFF_SCAL, OFF_MISC = C::OFF_MISC, OFF_BAR = C::OFF_BAR;
    extern __shared__ __align__(1024) uint8_t sm[];
    float *tile = reinterpret_cast<float *>(sm + OFF_TILE);
    float *coef = reinterpret_cast<float *>(sm + OFF_COEF);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    int *s_bad = reinterpret_cast<int *>(sm + OFF_MISC + 4);     // [2], by path-data buffer
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);  // tile, W, U

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0) flag(p.status, GDN_DEV_INTERNAL);
        return;
    }
    if ((int)blockIdx.x >= p.items) return;
    const int row = quad * 32 + lane, half = warp >> 2;  // tensor-memory lane = state row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    if (tid == 0) {
        for (int k = 0; k < 5; ++k) mbar_init(&bar[k], 1);
        fence_mbar_init();
        s_bad[0] = s_bad[1] = 0;
    }
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // A verification launched as this grid's programmatic dependent may now take
    // the SMs as this grid's blocks finish (it waits for this grid before reading
    // state).  The trigger follows this block's tensor-memory allocation, so a
    // dependent block can never hold columns that a block of this grid still
    // waits for.
    griddep_launch_dependents();
    bool ok = true;
    // test hook: a bounded wait on a barrier that nothing arrives on runs out,
    // and the block records GDN_DEV_TIMEOUT at exit; nothing else changes
    if (p.probe > 0 && tid == 0) ok = mbar_wait(&bar[3], 0, (uint32_t)p.probe);
    uint32_t ph_tile = 0, ph_mma = 0, ph_gram = 0;  // completed phases of the tile and MMA barriers
    int it = 0;                        // items committed by this block (path-data buffer = it & 1)

    struct Itm {
        int b, hv, hk, lo, n, pa, L, sel;
    };
    // An item's parameters; false, with the status bit to raise, for one that is skipped.
    auto params = [&](int idx, Itm &q, uint32_t (&mrow)[kMaxWords], int &err) -> bool {
        q.hv = idx % p.hv_n;
        const int grp = idx / p.hv_n;
        q.hk = q.hv / (p.hv_n / p.hk_n);
        q.b = kSel ? __ldg(p.sel_req + grp) : grp;
        err = 0;
        if (kSel && (q.b < 0 || q.b >= p.batch)) {
            err = GDN_DEV_BAD_PATH;
            return false;
        }
        q.lo = __ldg(p.offsets + q.b);
        q.n = __ldg(p.offsets + q.b + 1) - q.lo;
        q.pa = 0;
        q.sel = -1;
        if constexpr (kSel) {
            // the selected node's path: the set bits of its ancestor-mask row
            q.sel = __ldg(p.sel_node + grp);
            if (q.sel < 0 || q.sel >= q.n || q.lo < 0 || q.lo + q.n > p.total) {
                err = GDN_DEV_BAD_PATH;
                return false;
            }
            q.L = 0;
#pragma unroll
            for (int w = 0; w < kMaxWords; ++w) {
                mrow[w] = w < p.words ? __ldg(p.mask + (int64_t)(q.lo + q.sel) * p.words + w) : 0u;
                q.L += __popc(mrow[w]);
            }
            if (q.L > kMaxPath) {
                err = GDN_DEV_TOO_DEEP;
                return false;
            }
        } else {
            q.pa = __ldg(p.poff + q.b);
            q.L = __ldg(p.poff + q.b + 1) - q.pa;
            if (q.L < 0 || q.L > kMaxPath || q.L > q.n || q.lo < 0 || q.lo + q.n > p.total) {
                err = q.L > kMaxPath && q.L <= q.n ? GDN_DEV_TOO_DEEP : GDN_DEV_BAD_PATH;
                return false;
            }
        }
        return true;
    };
    // An item's path data into buffer `buf` (whose bad flag reads zero): the path
    // checked root first along parent -> child edges (and, for a selected node,
    // ending at it), node ids, keys (bf16, 16-byte pieces, rows past L zero),
    // values (fp32), raw g and beta.
    auto prep = [&](const Itm &q, const uint32_t (&mrow)[kMaxWords], int buf, int pb) {
        float *bet = reinterpret_cast<float *>(sm + OFF_SCAL) + buf * kScal, *gam = bet + 3 * kMaxPath;
        int *pn = reinterpret_cast<int *>(bet + 4 * kMaxPath);
        float *vp = reinterpret_cast<float *>(sm + OFF_VP) + buf * (kMaxPath * kD);
        uint8_t *keys = sm + OFF_KEYS + buf * C::kKeyBytes;
        auto node_at = [&](int t) -> int {
            if constexpr (kSel) return nth_bit(mrow, p.words, t);
            else return __ldg(p.pidx + q.pa + t);
        };
        if (kSel && q.L == 0 && tid == 0) atomicOr(s_bad + pb, 1);
        if (tid < q.L) {
            const int node = node_at(tid);
            const int expect = tid == 0 ? -1 : node_at(tid - 1);
            pn[tid] = node;
            const bool in = node >= 0 && node < q.n;
            if (!in || __ldg(p.parent + q.lo + node) != expect || (kSel && tid == q.L - 1 && node != q.sel))
                atomicOr(s_bad + pb, 1);
            if (in) {
                gam[tid] = __ldg(p.g + (int64_t)(q.lo + node) * p.hv_n + q.hv);
                bet[tid] = __ldg(p.beta + (int64_t)(q.lo + node) * p.hv_n + q.hv);
            }
        }
        const int c = tid & 15;
#pragma unroll
        for (int t = tid >> 4; t < kMaxPath; t += kT / 16) {
            uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = make_uint4(0u, 0u, 0u, 0u);
            if (t < q.L) {
                const int node = node_at(t);
                if (node >= 0 && node < q.n) {
                    const int64_t gnode = q.lo + node;
                    kv = __ldg(reinterpret_cast<const uint4 *>(p.k + (gnode * p.hk_n + q.hk) * kD) + c);
                    vv = __ldg(reinterpret_cast<const uint4 *>(p.v + (gnode * p.hv_n + q.hv) * kD) + c);
                }
            }
            *reinterpret_cast<uint4 *>(keys + sw128(t, c * 8, kMaxPath)) = kv;
            const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
            float *vrow = vp + t * kD + c * 8;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                vrow[2 * e] = __uint_as_float(w[e] << 16);
                vrow[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
        fence_proxy_async_smem();  // the keys are also a tensor-core operand
    };

    int prepped = -1;  // the item whose path data is already in its buffer
    for (int idx = blockIdx.x; idx < p.items; idx += gridDim.x) {
        Itm q;
        uint32_t mrow[kMaxWords];
        int err;
        if (!params(idx, q, mrow, err)) {
            if (tid == 0) flag(p.status, err);
            continue;
        }
        const int L = q.L, buf = C::kBufs == 2 ? (it & 1) : 0, pb = it & 1;  // data buffer; bad-flag slot
        const int row_in = (q.b * p.hv_n + q.hv) * kD, tile_row = idx * kD;
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar[0], kD * kD * 4);
            for (int qq = 0; qq < 4; ++qq) tma_load_2d(tile + qq * kD * 32, &tmS0, &bar[0], qq * 32, row_in);
            const int nx = idx + (int)gridDim.x;  // the next item's state tile, into L2
            if (nx < p.items) {
                const int nb = kSel ? __ldg(p.sel_req + nx / p.hv_n) : nx / p.hv_n;
                if (nb >= 0 && nb < p.batch)
                    prefetch_l2(p.S0 + ((int64_t)nb * p.hv_n + nx % p.hv_n) * (kD * kD), kD * kD * 4);
            }
        }
        if (prepped != idx) prep(q, mrow, buf, pb);
        __syncthreads();
        const bool bad = s_bad[pb] != 0;
        if (tid == 0) s_bad[pb ^ 1] = 0;  // the next item's flag starts clear
        float *bet = reinterpret_cast<float *>(sm + OFF_SCAL) + buf * kScal, *egam = bet + kMaxPath,
              *fdec = bet + 2 * kMaxPath, *gam = bet + 3 * kMaxPath;
        const float *vp = reinterpret_cast<const float *>(sm + OFF_VP) + buf * (kMaxPath * kD);
        uint8_t *keys = sm + OFF_KEYS + buf * C::kKeyBytes;
        if (tid == 0 && !bad) {
            float acc = 0.f;
            for (int t = 0; t < L; ++t) {
                acc += gam[t];
                gam[t] = acc;
                egam[t] = expf(acc);
            }
            for (int t = 0; t < L; ++t) fdec[t] = expf(acc - gam[t]);
        }
        __syncthreads();
        // chain coefficients beta_t e^(gamma_t - gamma_s) (k_t . k_s): the Gram K K^T of the
        // path keys on the tensor cores (M = 128, of which rows past L read other shared
        // memory and are ignored; N = P; into the P columns next to W), then lane t of
        // warp 0 scales row t
        if (!bad && L > 1) {
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, kMaxPath);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = smem_desc(smem_u32(keys + (ks >> 2) * (kMaxPath * 128) + (ks & 3) * 32), 16, 1024, 2);
                    mma_bf16(tmem + kMaxPath, d, d, id, ks > 0);
                }
                mma_commit(&bar[4]);
            }
            if (warp == 0) {
                ok = mbar_wait(&bar[4], ph_gram & 1) && ok;
                tc_fence_after();
                uint32_t gv[32];  // columns past P are not read
                tmem_ld32_nowait(tmem + kMaxPath, gv);
                tmem_wait_ld_into(gv);
                if (lane < L) {
                    const float bt = bet[lane], gt = gam[lane];
#pragma unroll
                    for (int s_ = 0; s_ < kMaxPath - 1; ++s_)
                        if (s_ < lane) coef[lane * kMaxPath + s_] = bt * expf(gt - gam[s_]) * __uint_as_float(gv[s_]);
                }
                tc_fence_before();
            }
            ++ph_gram;
        }

        // the state tile: row, columns 64 half .. 64 half + 63 into registers
        ok = mbar_wait(&bar[0], ph_tile & 1) && ok;
        ++ph_tile;
        float s[64];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float4 x = *reinterpret_cast<const float4 *>(tile + tile_index(row, half * 64 + c * 4));
            s[c * 4 + 0] = x.x; s[c * 4 + 1] = x.y; s[c * 4 + 2] = x.z; s[c * 4 + 3] = x.w;
        }
        __syncthreads();  // every thread holds its part; the tile space becomes S0 hi | lo
        if (!bad) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float hi[8], lw[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    hi[e] = __bfloat162float(__float2bfloat16_rn(s[c * 8 + e]));
                    lw[e] = s[c * 8 + e] - hi[e];
                }
                const uint32_t off = sw128(row, half * 64 + c * 8, kD);
                *reinterpret_cast<uint4 *>(sm + OFF_TILE + off) =
                    make_uint4(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]), pack_bf16(hi[4], hi[5]), pack_bf16(hi[6], hi[7]));
                *reinterpret_cast<uint4 *>(sm + OFF_TILE + 32768 + off) =
                    make_uint4(pack_bf16(lw[0], lw[1]), pack_bf16(lw[2], lw[3]), pack_bf16(lw[4], lw[5]), pack_bf16(lw[6], lw[7]));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        if (!bad) {
            // W = S0 K^T (hi + lo) -> tensor-memory columns [0, P)
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, kMaxPath);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ad = smem_desc(smem_u32(sm + OFF_TILE + part * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32), 16, 1024, 2);
                        const uint64_t bd = smem_desc(smem_u32(keys + (ks >> 2) * (kMaxPath * 128) + (ks & 3) * 32), 16, 1024, 2);
                        mma_bf16(tmem, ad, bd, id, part > 0 || ks > 0);
                    }
                mma_commit(&bar[1]);
            }
            ok = mbar_wait(&bar[1], ph_mma & 1) && ok;
            tc_fence_after();
            // chain solve for this row: u_t, then A[row][t] = e^(gamma_L - gamma_t) u_t
            uint32_t wr[kMaxPath];
            if constexpr (kMaxPath == 16) {
                tmem_ld16_nowait(tmem + lane_base, wr);
                tmem_wait_ld();
            } else {
                tmem_ld32_nowait(tmem + lane_base, wr);
                tmem_wait_ld_into(wr);
            }
            float a[kMaxPath];
#pragma unroll
            for (int t = 0; t < kMaxPath; ++t) {
                float u = 0.f;
                if (t < L) {
                    u = bet[t] * (vp[t * kD + row] - egam[t] * __uint_as_float(wr[t]));
#pragma unroll
                    for (int si = 0; si < t; ++si) u = fmaf(-coef[t * kMaxPath + si], a[si], u);
                }
                a[t] = u;
            }
#pragma unroll
            for (int t = 0; t < kMaxPath; ++t) a[t] = t < L ? a[t] * fdec[t] : 0.f;
            // A hi (half 0) or lo (half 1), core-matrix layout: 8 rows x 8 keys per 128 bytes
            float part[kMaxPath];
#pragma unroll
            for (int t = 0; t < kMaxPath; ++t) {
                const float h = __bfloat162float(__float2bfloat16_rn(a[t]));
                part[t] = half == 0 ? h : a[t] - h;
            }
            uint8_t *abase = sm + OFF_A + half * C::kABytes + (row >> 3) * (kMaxPath * 16) + (row & 7) * 16;
#pragma unroll
            for (int kh = 0; kh < kMaxPath / 8; ++kh)
                *reinterpret_cast<uint4 *>(abase + kh * 128) =
                    make_uint4(pack_bf16(part[kh * 8 + 0], part[kh * 8 + 1]), pack_bf16(part[kh * 8 + 2], part[kh * 8 + 3]),
                               pack_bf16(part[kh * 8 + 4], part[kh * 8 + 5]), pack_bf16(part[kh * 8 + 6], part[kh * 8 + 7]));
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            // U = A K (hi + lo) -> columns [128, 256); K is the same key tile read
            // MN-major, 16 path keys per MMA
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16_f32(128, 128) | (1u << 16);
#pragma unroll
                for (int ks = 0; ks < kMaxPath / 16; ++ks) {
                    const uint64_t bd = smem_desc(smem_u32(keys + ks * 2048), kMaxPath * 128, 1024, 2);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
                        mma_bf16(tmem + 128, smem_desc(smem_u32(sm + OFF_A + part * C::kABytes + ks * 256), 128, kMaxPath * 16, 0),
                                 bd, id, part > 0 || ks > 0);
                }
                mma_commit(&bar[2]);
            }
            ok = mbar_wait(&bar[2], ph_mma & 1) && ok;
            ++ph_mma;
            tc_fence_after();
            // S_new = e^gamma_L S0 + U, back into the tile in the TMA layout
            const float eL = L > 0 ? egam[L - 1] : 1.f;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t ur[32];
                tmem_ld32_nowait(tmem + lane_base + 128 + half * 64 + cc * 32, ur);
                tmem_wait_ld_into(ur);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int col = half * 64 + cc * 32 + c * 4;
                    float4 o;
                    o.x = fmaf(eL, s[cc * 32 + c * 4 + 0], __uint_as_float(ur[c * 4 + 0]));
                    o.y = fmaf(eL, s[cc * 32 + c * 4 + 1], __uint_as_float(ur[c * 4 + 1]));
                    o.z = fmaf(eL, s[cc * 32 + c * 4 + 2], __uint_as_float(ur[c * 4 + 2]));
                    o.w = fmaf(eL, s[cc * 32 + c * 4 + 3], __uint_as_float(ur[c * 4 + 3]));
                    *reinterpret_cast<float4 *>(tile + tile_index(row, col)) = o;
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            if (bad) {
                flag(p.status, kSel ? GDN_DEV_BAD_DESC : GDN_DEV_BAD_PATH);
            } else {
                for (int qq = 0; qq < 4; ++qq) tma_store_2d(&tmSN, tile + qq * kD * 32, qq * 32, tile_row);
                bulk_commit();
                bulk_wait_read();  // the tile space is free for the next item's load
            }
        }
        // the next item's path data, into the other buffer, while the store above
        // reads the tile out
        const int nidx = idx + (int)gridDim.x;
        if (nidx < p.items) {
            Itm nq;
            uint32_t nm[kMaxWords];
            int nerr;
            if (params(nidx, nq, nm, nerr)) {
                prep(nq, nm, C::kBufs == 2 ? (buf ^ 1) : 0, pb ^ 1);
                prepped = nidx;
            }
        }
        ++it;
    }
    if (!ok) flag(p.status, GDN_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
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

bool commit_tc_supported(const gdn_commit_args &a) {
    return a.qkv_dtype == GDN_BF16 && a.d_k == kD && a.d_v == kD && a.max_path >= 1 && a.max_path <= 32 &&
           aligned16(a.S0) && aligned16(a.S_new) && aligned16(a.k) && aligned16(a.v) &&
           (int64_t)a.batch * a.n_v_heads * kD <= 2147483647LL && tensor_map_encoder() != nullptr;
}

cudaError_t launch_commit_tc(const gdn_commit_args &a, cudaStream_t stream) {
    const int64_t rows = (int64_t)a.batch * a.n_v_heads * kD;
    CUtensorMap tmS0, tmSN;
    if (!encode_state(&tmS0, a.S0, rows) || !encode_state(&tmSN, a.S_new, rows)) return cudaErrorInvalidValue;
    TcCommitParams p = {};
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.total = a.total_nodes; p.items = a.batch * a.n_v_heads;
    p.batch = a.batch; p.S0 = a.S0;
    p.offsets = a.node_offsets; p.parent = a.parent; p.poff = a.path_offsets; p.pidx = a.path_idx;
    p.k = static_cast<const __nv_bfloat16 *>(a.k); p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.g = a.g; p.beta = a.beta; p.status = a.dev_status; p.probe = wait_probe_polls();
    // persistent: two blocks per SM; paths of up to 16 nodes, or up to 32
    const unsigned grid = (unsigned)std::min(p.items, 2 * sm_count());
    if (a.max_path <= 16) {
        static int have[16];
        cudaError_t e = ensure_smem(commit_tc_kernel<false, 16>, CommitCfg<16>::kSmemBytes, have);
        if (e != cudaSuccess) return e;
        commit_tc_kernel<false, 16><<<grid, kT, CommitCfg<16>::kSmemBytes, stream>>>(tmS0, tmSN, p);
    } else {
        static int have[16];
        cudaError_t e = ensure_smem(commit_tc_kernel<false, 32>, CommitCfg<32>::kSmemBytes, have);
        if (e != cudaSuccess) return e;
        commit_tc_kernel<false, 32><<<grid, kT, CommitCfg<32>::kSmemBytes, stream>>>(tmS0, tmSN, p);
    }
    return cudaGetLastError();
}

bool states_tc_supported(const gdn_states_args &a) {
    return a.qkv_dtype == GDN_BF16 && a.d_k == kD && a.d_v == kD && aligned16(a.S0) && aligned16(a.S_sel) &&
           aligned16(a.k) && aligned16(a.v) && (int64_t)a.batch * a.n_v_heads * kD <= 2147483647LL &&
           (int64_t)a.n_sel * a.n_v_heads * kD <= 2147483647LL && tensor_map_encoder() != nullptr;
}

cudaError_t launch_states_tc(const gdn_states_args &a, cudaStream_t stream) {
    CUtensorMap tmS0, tmSN;
    if (!encode_state(&tmS0, a.S0, (int64_t)a.batch * a.n_v_heads * kD) ||
        !encode_state(&tmSN, a.S_sel, (int64_t)a.n_sel * a.n_v_heads * kD))
        return cudaErrorInvalidValue;
    TcCommitParams p = {};
    p.hk_n = a.n_k_heads; p.hv_n = a.n_v_heads; p.total = a.total_nodes; p.items = a.n_sel * a.n_v_heads;
    p.batch = a.batch; p.words = a.mask_words; p.S0 = a.S0;
    p.offsets = a.node_offsets; p.parent = a.parent; p.sel_req = a.sel_request; p.sel_node = a.sel_node;
    p.mask = a.anc_mask;
    p.k = static_cast<const __nv_bfloat16 *>(a.k); p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.g = a.g; p.beta = a.beta; p.status = a.dev_status;
    static int have[16];
    cudaError_t e = ensure_smem(commit_tc_kernel<true, 16>, CommitCfg<16>::kSmemBytes, have);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)std::min(p.items, 2 * sm_count());
    commit_tc_kernel<true, 16><<<grid, kT, CommitCfg<16>::kSmemBytes, stream>>>(tmS0, tmSN, p);
    return cudaGetLastError();
}

}  // namespace gdn
