/*
 * gdn_tree.h -- C ABI of the GB300 (sm_103a) library for rollback-free
 * verification of a speculative proposal tree through one Gated Delta Net layer.
 *
 * The operation, from "Trees from Marginals: Autoregressive drafting with
 * factorized priors" (gist.science Technical Summary, section 3 "Rollback-Free
 * Tree Verification for GDN"):
 *   - a GDN layer advances its state with the gated delta rule (Challenge bullet);
 *     this library keeps the state as S[d_v][d_k] and applies, per token t,
 *         S_t = exp(g_t) * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *         o_t = scale * S_t q_t
 *     (the page writes the transpose; outputs are identical);
 *   - a draft tree, topologically sorted, is verified in one pass: every node's
 *     output equals the rule run along that node's root-to-node path from the
 *     committed state S0, computed through ancestor-masked interaction matrices
 *     and one triangular solve (Solution bullets 1-3);
 *   - S0 is never written by verification; the state is committed in the next
 *     iteration along the accepted branch only (Solution bullet 4).
 *
 * Conventions shared by every entry point
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     keeps no pointer after a call returns and allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream.
 *   - The return value is a gdn_status.  Argument, shape, support and launch
 *     errors are detected on the host and returned before anything is launched
 *     (GDN_ERR_CUDA: a launch failed).  gdn_last_error() then gives a message
 *     (thread-local, valid until the next call on the same thread).
 *   - Data-dependent problems found on the device (a malformed tree, a bad path,
 *     a request larger than max_nodes, a tree deeper than the bound a kernel
 *     needs) are OR-ed into *dev_status as GDN_DEV_* bits; the kernel skips the
 *     affected request and never traps.  The caller zeroes *dev_status before
 *     the call and reads it after synchronising the stream.
 *   - Requests: node_offsets[B+1] (int32, ascending, node_offsets[0] = 0)
 *     splits the T = node_offsets[B] tree nodes into B requests (the caller
 *     also passes T as total_nodes; a request reaching past it sets
 *     GDN_DEV_BAD_DESC and is skipped); node ids in
 *     parent[] and path_idx[] are request-local.  parent[i] = -1 marks a root
 *     (a child of S0; forests are allowed); otherwise 0 <= parent[i] < i.
 *   - Layouts (row-major, contiguous):
 *       q, k   [T][Hk][d_k]      (dtype qkv_dtype)
 *       v      [T][Hv][d_v]      (dtype qkv_dtype)
 *       g      [T][Hv]  float32  log-decay, alpha = exp(g)
 *       beta   [T][Hv]  float32
 *       S0, S_new [B][Hv][d_v][d_k] float32
 *       o      [T][Hv][d_v]      (dtype out_dtype)
 *     Value head h reads key head h / (Hv / Hk) (Hv a multiple of Hk).
 *   - Supported: d_k, d_v in {16, 32, 64, 128}; 1 <= max_nodes <= 256.
 */
#ifndef GDN_TREE_H_
#define GDN_TREE_H_

#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent sizes */
    GDN_ERR_UNSUPPORTED = 2,   /* a size or dtype outside the supported set */
    GDN_ERR_INVALID_TREE = 3,  /* reserved for host-side tree checks */
    GDN_ERR_INVALID_PATH = 4,  /* reserved for host-side path checks */
    GDN_ERR_CUDA = 5,          /* a CUDA launch or attribute call failed */
    GDN_ERR_DEVICE = 6         /* reserved: raised by wrappers that read dev_status */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* bits OR-ed into *dev_status */
#define GDN_DEV_BAD_TREE      1   /* parent[i] outside [-1, i) */
#define GDN_DEV_BAD_PATH      2   /* path not root-first or not parent->child */
#define GDN_DEV_TOO_MANY      4   /* a request has more than max_nodes nodes */
#define GDN_DEV_TOO_DEEP      8   /* a tree is deeper than the declared max_depth */
#define GDN_DEV_TIMEOUT      16   /* a bounded wait inside a kernel ran out */
#define GDN_DEV_BAD_DESC     32   /* anc_mask/depth disagree with parent[] */
#define GDN_DEV_INTERNAL     64   /* a launch invariant of a kernel did not hold */

/*
 * gdn_tree_build_desc -- tree descriptor ("interaction matrices representing
 * ancestor relationships", same section, Solution bullet 2; topological order,
 * bullet 1).
 *   anc_mask [T][mask_words] uint32: bit j of row i (request-local ids) is set
 *            iff node j lies on i's root-to-node path, i included.
 *   depth    [T] int32: number of nodes on that path (a root has depth 1).
 *   mask_words >= ceil(max_nodes / 32), at most 8.
 * Integer work, bit-exact.  A node whose walk meets a parent outside [-1, i)
 * gets a zero row and depth 0, and GDN_DEV_BAD_TREE is set.
 */
GDN_API int gdn_tree_build_desc(const int32_t *parent, const int32_t *node_offsets, int32_t batch,
                        int32_t max_nodes, uint32_t *anc_mask, int32_t mask_words,
                        int32_t *depth, int32_t *dev_status, void *stream);

/*
 * gdn_tree_grow -- draft-tree construction ("Methodology", section 2 "Tree
 * Construction": DySpec's best-first search, modified to expand the top-w
 * nodes of the candidate heap together).  Per request, node 0 is the root
 * (score 0, depth 1) and ids follow creation order.  One step takes the w best
 * frontier nodes -- not yet expanded, depth < max_depth -- by score descending,
 * then id ascending, and expands them in that order: node p gets children
 * j = 0 .. c_p - 1 scored score_p - e_pj * (j + 1) (float32 multiply, then
 * subtract), until the request's capacity is reached or the frontier is empty.
 * The random draws are inputs:
 *   node_offsets [B+1]: the capacity N_b of each request (<= 256 nodes);
 *   n_children [T] int32: c_p for node p of its request (row lo + p), used if p
 *              is expanded, clipped to [0, max_children];
 *   draws [T][max_children] float32: e_pj >= 0, finite (a NaN gives an
 *              unspecified tree);
 *   parent [T] int32 (request-local; -1 for the root and for rows past the
 *              built tree), score [T] float32 (-inf past the tree), n_nodes [B].
 * The tree is topologically ordered and ready for gdn_tree_build_desc.
 * 1 <= width, 1 <= max_depth, 1 <= max_children <= 64.  Integer results and
 * scores are bit-exact against the float32 definition.
 */
GDN_API int gdn_tree_grow(const int32_t *node_offsets, int32_t batch, int32_t total_nodes, int32_t width,
                          int32_t max_depth, int32_t max_children, const int32_t *n_children,
                          const float *draws, int32_t *parent, float *score, int32_t *n_nodes,
                          int32_t *dev_status, void *stream);

/*
 * gdn_tree_relabel -- topological order for a tree given in any order (same
 * section, Solution bullet 1: the tree is processed parent before child).
 * Per request, nodes are sorted by (depth, old id), which is unique:
 *   parent_in  [T] int32: request-local parent ids in any labelling (-1 = root;
 *              forests allowed).
 *   order      [T] int32: order[lo + j] = old id of the node placed j-th.
 *   rank       [T] int32: rank[lo + i] = new id of old node i.
 *   parent_out [T] int32: parents in new ids; parent_out[lo + j] < j.
 * Integer work, bit-exact.  total_nodes = T.  A request whose parents do not
 * form a forest (a parent outside [-1, n), a self-parent, a cycle) sets
 * GDN_DEV_BAD_TREE and its rows of the three outputs are left untouched.
 * max_nodes <= 256.  Token rows are then gathered by `order` (e.g. with
 * gdn_gather_rows) before gdn_tree_build_desc.
 */
GDN_API int gdn_tree_relabel(const int32_t *parent_in, const int32_t *node_offsets, int32_t batch,
                             int32_t total_nodes, int32_t max_nodes, int32_t *order, int32_t *rank,
                             int32_t *parent_out, int32_t *dev_status, void *stream);

/*
 * gdn_gather_rows -- permute rows within each request: dst row lo + j = src
 * row lo + index[lo + j], index request-local (no counterpart in the pages: the
 * data movement that goes with gdn_tree_relabel).  With index = order it puts
 * token rows (q, k, v, g, beta) into the new order; with index = rank it maps
 * outputs in the new order back to the old labels.
 *   src, dst  [T] rows of row_bytes bytes each (row_bytes > 0, a multiple of
 *             16; both pointers 16-byte aligned; dst must not overlap src).
 * An index outside [0, n) sets GDN_DEV_BAD_DESC and leaves that dst row
 * untouched.  batch <= 65535.
 */
GDN_API int gdn_gather_rows(const void *src, void *dst, const int32_t *index, const int32_t *node_offsets,
                            int32_t batch, int32_t total_nodes, int64_t row_bytes, int32_t *dev_status,
                            void *stream);

typedef struct {
    int32_t batch, n_k_heads, n_v_heads, d_k, d_v;
    int32_t total_nodes;   /* T = node_offsets[batch]: rows of q, k, v, g, beta, o */
    int32_t max_nodes;     /* upper bound on any request's node count (<= 256) */
    int32_t max_depth;     /* caller's bound on tree depth, or 0 if unknown */
    float scale;           /* output scale (1.0 for the plain rule) */
    int32_t qkv_dtype;     /* gdn_dtype of q, k, v */
    int32_t out_dtype;     /* gdn_dtype of o */
    const int32_t *node_offsets;
    const void *q, *k, *v;
    const float *g, *beta, *S0;
    const int32_t *parent;
    const uint32_t *anc_mask;  /* from gdn_tree_build_desc */
    int32_t mask_words;
    const int32_t *depth;      /* from gdn_tree_build_desc */
    void *o;
    int32_t *dev_status;
} gdn_verify_args;

/*
 * gdn_tree_verify -- every node's output, computed as the masked triangular
 * solve of the same section (Solution bullets 2-3): with gamma_i the sum of g
 * over i's path, D_ij = exp(gamma_i - gamma_j) on ancestors j of i,
 *     X = strict-ancestor mask * beta_i * D * (K K^T)
 *     Y = ancestor mask * D * (Q K^T)
 *     (I + X) U = beta * (V - exp(gamma) * K S0^T)
 *     O = scale * (exp(gamma) * Q S0^T + Y U)
 * S0 is read, never written.  Nodes off a node's path never affect its output.
 * Fast paths: bf16 q/k/v with d_k = d_v = 128 run a tcgen05/TMA kernel when
 * the declared max_depth is 1..16 (max_nodes <= 128: one node tile per
 * request, two value heads at a time; 128 < max_nodes <= 256: two node tiles)
 * or 17..64 with max_nodes <= 128 (one tile, one value head at a time).  A
 * tree deeper than the declared max_depth sets GDN_DEV_TOO_DEEP and its
 * request is skipped.  Every other case runs the general kernel, which
 * accepts any depth.
 * q and k need no normalisation on any path (the fast paths keep the raw
 * products k_i.k_j and q_i.k_j in fp32); non-finite inputs propagate to the
 * outputs of the nodes below them only.
 */
GDN_API int gdn_tree_verify(const gdn_verify_args *args, void *stream);

/*
 * gdn_tree_verify_branches -- the per-branch recurrent verification the pages
 * compare against ("Experimental Results", Verification Efficiency): one
 * thread block per (request, value head, root-to-leaf path, d_v slab) runs the
 * gated delta rule sequentially along its path from S0 and writes the outputs
 * of the nodes on it.  Same arguments and results as gdn_tree_verify (up to
 * rounding); anc_mask/depth are not read.  Used as the measurement baseline.
 */
GDN_API int gdn_tree_verify_branches(const gdn_verify_args *args, void *stream);

typedef struct {
    int32_t batch, n_k_heads, n_v_heads, d_k, d_v;
    int32_t total_nodes;   /* T = node_offsets[batch]: rows of k, v, g, beta */
    int32_t max_nodes;     /* upper bound on any request's node count (<= 256) */
    int32_t max_path;      /* caller's bound on accepted-path length, or 0 if unknown */
    int32_t qkv_dtype;     /* gdn_dtype of k, v */
    const int32_t *node_offsets;
    const void *k, *v;
    const float *g, *beta, *S0;
    const int32_t *parent;
    const int32_t *path_offsets;  /* [B+1] */
    const int32_t *path_idx;      /* accepted path per request, request-local ids, root first */
    float *S_new;                 /* [B][Hv][d_v][d_k]; may equal S0 (in-place commit) */
    int32_t *dev_status;
} gdn_commit_args;

/*
 * gdn_tree_commit -- the delayed commit (same section, Solution bullet 4): the
 * new state after the accepted path p_1..p_L, in chunked form:
 *     u = chain solve of the path (the verify system restricted to the path)
 *     S_new = exp(gamma_L) S0 + sum_t exp(gamma_L - gamma_t) u_t k_t^T
 * equal to running the rule along the path.  L = 0 leaves S0 (copied when
 * S_new != S0).  A path that does not start at a root or does not follow
 * parent -> child edges sets GDN_DEV_BAD_PATH and leaves that request's S_new
 * unwritten.  Everything accumulates in fp32.
 * Fast paths for d_k = d_v = 128: bf16 k/v with 1 <= max_path <= 32 run a
 * persistent tcgen05 kernel (two blocks per SM walking the (request, value
 * head) items, the state tile moved by TMA both ways); fp32 k/v (and bf16
 * k/v the tensor-core kernel does not take) with 1 <= max_path <= 16 run one
 * block per item with the tile moved by TMA.  A path longer than the declared
 * max_path sets GDN_DEV_TOO_DEEP and its request is skipped.  Every other case
 * runs the general kernel.
 */
GDN_API int gdn_tree_commit(const gdn_commit_args *args, void *stream);

/*
 * gdn_tree_commit_verify -- the delayed commit followed by the next
 * verification (same section, Solution bullet 4: the state is committed in the
 * next decoding iteration).  commit->S0 is committed along the previous tree's
 * accepted path (commit's tree, tokens and path) into commit->S_new, and the
 * new tree (verify's) is verified from commit->S_new; verify->S0 is not read.
 *   Results equal gdn_tree_commit then gdn_tree_verify on the same stream.
 *   The two launches overlap: the verification is launched as the commit's
 *   programmatic dependent, its blocks start on the SMs the commit releases,
 *   and each waits for the whole commit before its first state read.
 *   commit->S_new may equal commit->S0 (in place); it must not overlap any
 *   other input of the verification.  Shapes of both calls must agree (batch,
 *   heads, d_k, d_v); any shapes that both gdn_tree_commit and
 *   gdn_tree_verify accept are accepted.
 *   A bad path sets GDN_DEV_BAD_PATH (GDN_DEV_TOO_DEEP past the commit kernel's
 *   limit) and leaves that request's S_new unwritten; its new outputs are then
 *   computed from whatever S_new held and must be discarded.
 */
GDN_API int gdn_tree_commit_verify(const gdn_commit_args *commit, const gdn_verify_args *verify,
                                   void *stream);

typedef struct {
    int32_t batch, n_k_heads, n_v_heads, d_k, d_v;
    int32_t total_nodes;   /* T = node_offsets[batch]: rows of k, v, g, beta */
    int32_t max_nodes;     /* upper bound on any request's node count (<= 256) */
    int32_t qkv_dtype;     /* gdn_dtype of k, v */
    const int32_t *node_offsets;
    const void *k, *v;
    const float *g, *beta, *S0;
    const int32_t *parent;
    const uint32_t *anc_mask;     /* from gdn_tree_build_desc */
    int32_t mask_words;
    int32_t n_sel;                /* number of selected nodes */
    const int32_t *sel_request;   /* [n_sel] request of each selected node */
    const int32_t *sel_node;      /* [n_sel] request-local node id */
    float *S_sel;                 /* [n_sel][Hv][d_v][d_k]: the state at each selected node */
    int32_t *dev_status;
} gdn_states_args;

/*
 * gdn_tree_states -- the state S_i at chosen nodes i: the commit of i's own
 * root-to-node path (same section, Solution bullet 4, applied to a node that
 * is not yet accepted), so that committing one of them later needs no
 * recompute (a commit applied to a node that is not yet accepted; the pages
 * describe only the commit of the accepted path).  A node's path is read from its
 * anc_mask row (root first) and checked against parent[]; a row that does not
 * follow parent -> child edges to the node sets GDN_DEV_BAD_DESC, a selection
 * outside its request sets GDN_DEV_BAD_PATH, a path longer than 16 sets
 * GDN_DEV_TOO_DEEP, and that selection's S_sel block is left unwritten.
 * Supported: bf16 k/v with d_k = d_v = 128 (else GDN_ERR_UNSUPPORTED); fp32
 * accumulation throughout, same numerics as gdn_tree_commit's fast path.
 */
GDN_API int gdn_tree_states(const gdn_states_args *args, void *stream);

/* Message for the last non-OK return on this thread ("" if none). */
GDN_API const char *gdn_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
GDN_API int gdn_tree_version(void);

/*
 * gdn_test_set_wait_probe -- test hook for the kernels' bounded waits (no
 * counterpart in the pages).  With polls > 0, every later launch of the
 * tensor-core verify and commit kernels makes one extra wait, of `polls` polls,
 * on an mbarrier that nothing arrives on.  The wait runs out, the kernel sets
 * GDN_DEV_TIMEOUT in *dev_status and otherwise computes and returns as usual.
 * polls <= 0 (the default) turns the hook off.  Process-wide; not for
 * production use.
 */
GDN_API void gdn_test_set_wait_probe(int32_t polls);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TREE_H_ */
