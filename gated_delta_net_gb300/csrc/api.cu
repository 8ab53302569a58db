// api.cu -- host side of the C ABI: argument checks, kernel choice, error text.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "internal.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool supported_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool valid_dtype(int t) { return t == GDN_F32 || t == GDN_BF16; }

int check_common(int batch, int hk, int hv, int dk, int dv, int max_nodes) {
    if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (hk < 1 || hv < 1) return fail(GDN_ERR_INVALID_ARG, "head counts must be >= 1");
    if (hv % hk) return fail(GDN_ERR_INVALID_ARG, "n_v_heads %d not a multiple of n_k_heads %d", hv, hk);
    if (!supported_dim(dk) || !supported_dim(dv))
        return fail(GDN_ERR_UNSUPPORTED, "d_k=%d d_v=%d: supported sizes are 16, 32, 64, 128", dk, dv);
    if (max_nodes < 1) return fail(GDN_ERR_INVALID_ARG, "max_nodes %d < 1", max_nodes);
    if (max_nodes > gdn::kMaxNodes)
        return fail(GDN_ERR_UNSUPPORTED, "max_nodes %d > %d", max_nodes, gdn::kMaxNodes);
    return GDN_OK;
}

int check_verify(const gdn_verify_args *a) {
    if (!a) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
    int st = check_common(a->batch, a->n_k_heads, a->n_v_heads, a->d_k, a->d_v, a->max_nodes);
    if (st) return st;
    if (!valid_dtype(a->qkv_dtype) || !valid_dtype(a->out_dtype))
        return fail(GDN_ERR_UNSUPPORTED, "unknown dtype (qkv %d, out %d)", a->qkv_dtype, a->out_dtype);
    if (a->max_depth < 0) return fail(GDN_ERR_INVALID_ARG, "max_depth %d < 0", a->max_depth);
    if (a->total_nodes < 0) return fail(GDN_ERR_INVALID_ARG, "total_nodes %d < 0", a->total_nodes);
    if (!std::isfinite(a->scale)) return fail(GDN_ERR_INVALID_ARG, "scale is not finite");
    if (a->batch == 0) return GDN_OK;
    if (!a->node_offsets || !a->q || !a->k || !a->v || !a->g || !a->beta || !a->S0 || !a->parent ||
        !a->anc_mask || !a->depth || !a->o)
        return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    if (a->mask_words < (a->max_nodes + 31) / 32 || a->mask_words > gdn::kMaxWords)
        return fail(GDN_ERR_INVALID_ARG, "mask_words %d must be in [%d, %d]", a->mask_words,
                    (a->max_nodes + 31) / 32, gdn::kMaxWords);
    return GDN_OK;
}

int check_commit(const gdn_commit_args *a) {
    if (!a) return fail(GDN_ERR_INVALID_ARG, "commit args are NULL");
    int st = check_common(a->batch, a->n_k_heads, a->n_v_heads, a->d_k, a->d_v, a->max_nodes);
    if (st) return st;
    if (!valid_dtype(a->qkv_dtype)) return fail(GDN_ERR_UNSUPPORTED, "unknown dtype %d", a->qkv_dtype);
    if (a->total_nodes < 0) return fail(GDN_ERR_INVALID_ARG, "total_nodes %d < 0", a->total_nodes);
    if (a->max_path < 0) return fail(GDN_ERR_INVALID_ARG, "max_path %d < 0", a->max_path);
    if (a->batch == 0) return GDN_OK;
    if (!a->node_offsets || !a->k || !a->v || !a->g || !a->beta || !a->S0 || !a->parent ||
        !a->path_offsets || !a->path_idx || !a->S_new)
        return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    return GDN_OK;
}

cudaError_t launch_commit_any(const gdn_commit_args &a, cudaStream_t stream) {
    return gdn::commit_tc_supported(a)     ? gdn::launch_commit_tc(a, stream)
           : gdn::commit_fast_supported(a) ? gdn::launch_commit_fast(a, stream)
                                           : gdn::launch_commit_simt(a, stream);
}

// the verification; after_commit: the preceding launch in the stream commits its state
cudaError_t launch_verify_any(const gdn_verify_args &a, cudaStream_t stream, bool after_commit) {
    if (gdn::verify_tc_supported(a)) return gdn::launch_verify_tc(a, stream, after_commit);
    if (gdn::verify_wide_supported(a)) return gdn::launch_verify_wide(a, stream, after_commit);
    return gdn::launch_verify_simt(a, stream);
}

}  // namespace

namespace gdn {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

int sm_count() {
    // cached per device: a process may launch on devices of different sizes
    static std::atomic<int> count[16];
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 16 && (c = count[dev].load(std::memory_order_relaxed)) > 0) return c;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1) return 1;
    if (dev >= 0 && dev < 16) count[dev].store(c, std::memory_order_relaxed);
    return c;
}

namespace {
std::atomic<int> g_probe{0};
}

int wait_probe_polls() { return g_probe.load(std::memory_order_relaxed); }

}  // namespace gdn

extern "C" {

const char *gdn_last_error(void) { return g_err; }

int gdn_tree_version(void) { return 200; }

void gdn_test_set_wait_probe(int32_t polls) { gdn::g_probe.store(polls > 0 ? polls : 0); }

int gdn_tree_build_desc(const int32_t *parent, const int32_t *node_offsets, int32_t batch,
                        int32_t max_nodes, uint32_t *anc_mask, int32_t mask_words,
                        int32_t *depth, int32_t *dev_status, void *stream) {
    g_err[0] = 0;
    if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (max_nodes < 1) return fail(GDN_ERR_INVALID_ARG, "max_nodes %d < 1", max_nodes);
    if (max_nodes > gdn::kMaxNodes)
        return fail(GDN_ERR_UNSUPPORTED, "max_nodes %d > %d", max_nodes, gdn::kMaxNodes);
    if (mask_words < (max_nodes + 31) / 32 || mask_words > gdn::kMaxWords)
        return fail(GDN_ERR_INVALID_ARG, "mask_words %d must be in [%d, %d]", mask_words,
                    (max_nodes + 31) / 32, gdn::kMaxWords);
    if (batch == 0) return GDN_OK;
    if (!parent || !node_offsets || !anc_mask || !depth)
        return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    cudaError_t e = gdn::launch_build_desc(parent, node_offsets, batch, max_nodes, anc_mask,
                                           mask_words, depth, dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "build_desc launch");
}

int gdn_tree_grow(const int32_t *node_offsets, int32_t batch, int32_t total_nodes, int32_t width, int32_t max_depth,
                  int32_t max_children, const int32_t *n_children, const float *draws, int32_t *parent, float *score,
                  int32_t *n_nodes, int32_t *dev_status, void *stream) {
    g_err[0] = 0;
    if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (total_nodes < 0) return fail(GDN_ERR_INVALID_ARG, "total_nodes %d < 0", total_nodes);
    if (width < 1) return fail(GDN_ERR_INVALID_ARG, "width %d < 1", width);
    if (max_depth < 1) return fail(GDN_ERR_INVALID_ARG, "max_depth %d < 1", max_depth);
    if (max_children < 1 || max_children > 64)
        return fail(GDN_ERR_INVALID_ARG, "max_children %d outside [1, 64]", max_children);
    if (batch == 0) return GDN_OK;
    if (!node_offsets || !n_children || !draws || !parent || !score || !n_nodes)
        return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    cudaError_t e = gdn::launch_grow(node_offsets, batch, total_nodes, width, max_depth, max_children, n_children,
                                     draws, parent, score, n_nodes, dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "grow launch");
}

int gdn_tree_relabel(const int32_t *parent_in, const int32_t *node_offsets, int32_t batch, int32_t total_nodes,
                     int32_t max_nodes, int32_t *order, int32_t *rank, int32_t *parent_out, int32_t *dev_status,
                     void *stream) {
    g_err[0] = 0;
    if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (total_nodes < 0) return fail(GDN_ERR_INVALID_ARG, "total_nodes %d < 0", total_nodes);
    if (max_nodes < 1) return fail(GDN_ERR_INVALID_ARG, "max_nodes %d < 1", max_nodes);
    if (max_nodes > gdn::kMaxNodes)
        return fail(GDN_ERR_UNSUPPORTED, "max_nodes %d > %d", max_nodes, gdn::kMaxNodes);
    if (batch == 0 || total_nodes == 0) return GDN_OK;
    if (!parent_in || !node_offsets || !order || !rank || !parent_out)
        return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    cudaError_t e = gdn::launch_relabel(parent_in, node_offsets, batch, total_nodes, max_nodes, order, rank,
                                        parent_out, dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "relabel launch");
}

int gdn_gather_rows(const void *src, void *dst, const int32_t *index, const int32_t *node_offsets, int32_t batch,
                    int32_t total_nodes, int64_t row_bytes, int32_t *dev_status, void *stream) {
    g_err[0] = 0;
    if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch %d < 0", batch);
    if (total_nodes < 0) return fail(GDN_ERR_INVALID_ARG, "total_nodes %d < 0", total_nodes);
    if (batch > 65535) return fail(GDN_ERR_UNSUPPORTED, "batch %d > 65535", batch);
    if (row_bytes <= 0 || row_bytes % 16)
        return fail(GDN_ERR_INVALID_ARG, "row_bytes %lld must be a positive multiple of 16", (long long)row_bytes);
    if (batch == 0 || total_nodes == 0) return GDN_OK;
    if (!src || !dst || !index || !node_offsets) return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15)
        return fail(GDN_ERR_INVALID_ARG, "src and dst must be 16-byte aligned");
    const char *s = static_cast<const char *>(src), *d = static_cast<const char *>(dst);
    const int64_t span = (int64_t)total_nodes * row_bytes;
    if (s < d + span && d < s + span) return fail(GDN_ERR_INVALID_ARG, "dst overlaps src");
    cudaError_t e = gdn::launch_gather_rows(src, dst, index, node_offsets, batch, total_nodes, row_bytes,
                                            dev_status, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gather launch");
}

int gdn_tree_verify(const gdn_verify_args *a, void *stream) {
    g_err[0] = 0;
    int st = check_verify(a);
    if (st || a->batch == 0) return st;
    cudaError_t e = launch_verify_any(*a, (cudaStream_t)stream, false);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "verify launch");
}

int gdn_tree_verify_branches(const gdn_verify_args *a, void *stream) {
    g_err[0] = 0;
    int st = check_verify(a);
    if (st || a->batch == 0) return st;
    cudaError_t e = gdn::launch_verify_branches(*a, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "verify_branches launch");
}

int gdn_tree_commit(const gdn_commit_args *a, void *stream) {
    g_err[0] = 0;
    int st = check_commit(a);
    if (st || a->batch == 0) return st;
    cudaError_t e = launch_commit_any(*a, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "commit launch");
}

int gdn_tree_commit_verify(const gdn_commit_args *c, const gdn_verify_args *v, void *stream) {
    g_err[0] = 0;
    int st = check_commit(c);
    if (st) return st;
    if (!v) return fail(GDN_ERR_INVALID_ARG, "verify args are NULL");
    gdn_verify_args vv = *v;
    vv.S0 = c->S_new;  // the new tree is verified from the committed state
    st = check_verify(&vv);
    if (st) return st;
    if (c->batch != v->batch || c->n_k_heads != v->n_k_heads || c->n_v_heads != v->n_v_heads ||
        c->d_k != v->d_k || c->d_v != v->d_v)
        return fail(GDN_ERR_INVALID_ARG, "commit and verify shapes differ");
    if (v->batch == 0) return GDN_OK;
    cudaError_t e = launch_commit_any(*c, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    e = launch_verify_any(vv, (cudaStream_t)stream, true);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "verify launch");
}

int gdn_tree_states(const gdn_states_args *a, void *stream) {
    g_err[0] = 0;
    if (!a) return fail(GDN_ERR_INVALID_ARG, "args is NULL");
    int st = check_common(a->batch, a->n_k_heads, a->n_v_heads, a->d_k, a->d_v, a->max_nodes);
    if (st) return st;
    if (!valid_dtype(a->qkv_dtype)) return fail(GDN_ERR_UNSUPPORTED, "unknown dtype %d", a->qkv_dtype);
    if (a->total_nodes < 0) return fail(GDN_ERR_INVALID_ARG, "total_nodes %d < 0", a->total_nodes);
    if (a->n_sel < 0) return fail(GDN_ERR_INVALID_ARG, "n_sel %d < 0", a->n_sel);
    if (a->batch == 0 || a->n_sel == 0) return GDN_OK;
    if (!a->node_offsets || !a->k || !a->v || !a->g || !a->beta || !a->S0 || !a->parent || !a->anc_mask ||
        !a->sel_request || !a->sel_node || !a->S_sel)
        return fail(GDN_ERR_INVALID_ARG, "a required pointer is NULL");
    if (a->mask_words < (a->max_nodes + 31) / 32 || a->mask_words > gdn::kMaxWords)
        return fail(GDN_ERR_INVALID_ARG, "mask_words %d must be in [%d, %d]", a->mask_words,
                    (a->max_nodes + 31) / 32, gdn::kMaxWords);
    if (!gdn::states_tc_supported(*a))
        return fail(GDN_ERR_UNSUPPORTED, "states: bf16 k/v with d_k = d_v = 128 and 16-byte aligned tensors only");
    cudaError_t e = gdn::launch_states_tc(*a, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "states launch");
}

}  // extern "C"
