/*
 * tgdn.h — C ABI of the rollback-free GDN tree-verification library (libtgdn.so).
 *
 * One decode step of tree speculative decoding on a hybrid model with Gated
 * DeltaNet (GDN) layers, as described in "Trees from Marginals: Autoregressive
 * drafting with factorized priors" (Technisches Resümee, Methodik 3,
 * "Rollback-freie Baumverifizierung für GDN"):
 *
 *   tgdn_tree_prep  sort the draft tree topologically and build its ancestor
 *                   relation (Methodik 3: "Der Baum wird topologisch sortiert").
 *   tgdn_verify     every node's output from the committed state S0 in one
 *                   pass: Gram tiles, a masked triangular solve (I + X) U = R
 *                   and the output phase, without updating the state
 *                   (Methodik 3: interaction matrices X and Y; the system
 *                   (I+X)U = beta V; Implementierung: Gram matrix, tiled
 *                   forward substitution, output phase).
 *   tgdn_accept     greedy acceptance: the longest root path whose draft
 *                   tokens all equal the verifier's tokens (mean acceptance
 *                   length, Experimentelle Ergebnisse).
 *   tgdn_commit     the accepted node's state, written from the same factors
 *                   U once the accepted branch is known; no rollback and no
 *                   replay (Methodik 3, deferred state commitment).
 *
 * The recurrence is the GDN update eq. (Methodik 3, "Herausforderung"):
 *   S_n = a_n (I - b_n k_n k_n^T) S_parent(n) + b_n k_n v_n^T,  a_n = exp(g_n),
 * with S a d_k x d_v matrix stored row-major (row = key index), and the output
 * of node n is o_n = S_n^T q_n.  The root of each tree is a real token whose
 * parent state is S0.  q and k are used exactly as given (no normalisation,
 * no 1/sqrt(d) scaling).  v-head h reads query/key head h / (H_v / H_qk).
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless stated otherwise.  The
 *     caller owns and allocates every buffer, workspace included; the library
 *     never allocates device memory and keeps no state between calls.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and returns after enqueueing its kernels.
 *   - Host-side argument checks run before any launch and return a negative
 *     tgdn_status; nothing is enqueued in that case.  Errors that only the
 *     device can see (a malformed tree, an expired bounded wait) are written
 *     to the per-sequence status word and never trap.
 *   - Row ranges: sequence b owns node rows cu_nodes[b] .. cu_nodes[b+1]-1 of
 *     every [T]-leading array; parent[] holds LOCAL indices (0 .. N_b-1,
 *     -1 for the root).
 */
#ifndef TGDN_H_
#define TGDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* An opaque CUDA stream handle, layout-compatible with cudaStream_t. */
typedef struct CUstream_st* tgdn_stream_t;

/* Return codes of every call. */
typedef enum {
  TGDN_OK = 0,
  TGDN_EINVAL = -1,       /* null pointer, negative size, inconsistent dims */
  TGDN_ETOOBIG = -3,      /* a bound above the library's limits (see below) */
  TGDN_ECUDA = -4,        /* a CUDA launch or driver call failed */
  TGDN_EUNSUPPORTED = -5  /* a valid combination this build does not run */
} tgdn_status;

/* Per-sequence status words written by tgdn_tree_prep (values 1-5 and 7) and
 * by the other calls (value 6).  tgdn_tree_prep checks the row range first
 * (value 7), then the values 1-5 in this order; the first failing check wins. */
typedef enum {
  TGDN_SEQ_OK = 0,
  TGDN_SEQ_TOO_BIG = 1,     /* N_b > n_max */
  TGDN_SEQ_BAD_PARENT = 2,  /* some parent < -1, >= N_b, or equal to the node */
  TGDN_SEQ_ROOTS = 3,       /* N_b > 0 and not exactly one root */
  TGDN_SEQ_CYCLE = 4,       /* some node never reaches the root */
  TGDN_SEQ_TOO_DEEP = 5,    /* some depth > depth_max */
  TGDN_SEQ_TIMEOUT = 6,     /* a bounded device wait expired; outputs of the
                               sequence are unspecified */
  TGDN_SEQ_BAD_RANGE = 7    /* cu_nodes[b] < 0, cu_nodes[b+1] < cu_nodes[b] or
                               cu_nodes[b+1] > T: no call reads or writes any row
                               of the sequence (only status[b] is written) */
} tgdn_seq_status;

/* Element type of q, k, v and o.  g, b, S0, the state and the workspace are
 * always fp32. */
typedef enum { TGDN_F32 = 0, TGDN_BF16 = 1 } tgdn_dtype;

/* Library limits. */
#define TGDN_MAX_NODES 256  /* n_max bound: nodes per tree, root included */
#define TGDN_MAX_DEPTH 64   /* depth_max bound: edges on the longest root path */
#define TGDN_MAX_HEAD_DIM 128

/* A batch of draft trees and the metadata tgdn_tree_prep derives from it.
 *   B          number of sequences (>= 0)
 *   T          total rows of every [T]-leading array (host copy): tree prep
 *              gives a sequence whose row range leaves [0, T) the status
 *              TGDN_SEQ_BAD_RANGE, so a bad cu_nodes never makes a call touch
 *              rows outside the arrays
 *   n_max      caller's bound on nodes per sequence, 1 .. TGDN_MAX_NODES
 *   depth_max  caller's bound on depth, 0 .. TGDN_MAX_DEPTH
 *   words      64-bit words per ancestor mask, must equal ceil(n_max / 64)
 *   cu_nodes   [B+1] int32, non-decreasing row offsets, cu_nodes[0] = 0
 *   parent     [T] int32, local parent index, -1 for the root
 * Written by tgdn_tree_prep, read by the other calls:
 *   depth      [T] int32, edges from the node to the root
 *   order      [T] int32, order[cu_nodes[b] + p] = local index of the node at
 *              topological position p (stable sort by (depth, index))
 *   pos        [T] int32, inverse of order: pos[cu_nodes[b] + n] = p
 *   anc        [T][words] uint64, row cu_nodes[b] + pos(n) has bit pos(s) set
 *              for every s on the root path of n, n included
 *   status     [B] int32, tgdn_seq_status
 * For a sequence whose status is not TGDN_SEQ_OK, depth/order/pos are -1 and
 * anc rows are 0, except under TGDN_SEQ_BAD_RANGE, where none of its rows is
 * written.  Every other call skips a sequence whose status is not TGDN_SEQ_OK
 * (zero outputs, state kept) and never touches the rows of one with
 * TGDN_SEQ_BAD_RANGE. */
typedef struct {
  int32_t B, T, n_max, depth_max, words;
  const int32_t* cu_nodes;
  const int32_t* parent;
  int32_t* depth;
  int32_t* order;
  int32_t* pos;
  uint64_t* anc;
  int32_t* status;
} tgdn_tree;

/* Head geometry of one GDN layer.  H_v must be a multiple of H_qk;
 * 1 <= d_k, d_v <= TGDN_MAX_HEAD_DIM; io is a tgdn_dtype. */
typedef struct {
  int32_t H_qk, H_v, d_k, d_v;
  int32_t io;
} tgdn_dims;

/* Topological sort and ancestor masks for every sequence (Methodik 3: "Der
 * Baum wird topologisch sortiert"; ancestor relations behind X and Y).
 * Validates each tree and writes depth, order, pos, anc and status.
 * Returns TGDN_OK, TGDN_EINVAL (null pointer, B < 0, words mismatch) or
 * TGDN_ETOOBIG (n_max or depth_max above the limits). */
int tgdn_tree_prep(const tgdn_tree* tree, tgdn_stream_t stream);

/* Bytes of the workspace tgdn_verify writes and tgdn_commit reads for this
 * tree and geometry: the factors U [T][H_v][d_v] fp32 followed, at the next
 * 256-byte boundary, by the path-cumulative log-gates G [T][H_v] fp32.
 * Returns 0 for invalid arguments. */
size_t tgdn_verify_workspace_bytes(const tgdn_tree* tree, const tgdn_dims* dims);

/* Single-pass verification of every node (Methodik 3 and Implementierung:
 * Gram matrix, tiled forward substitution, output phase).  With
 * G_n = sum of g over the root path of n (n included):
 *   X_ns = b_n exp(G_n - G_s) k_n.k_s   for s a strict ancestor of n,
 *   Y_ns =     exp(G_n - G_s) q_n.k_s   for s an ancestor of n or n itself,
 *   (I + X) U = diag(b) (V - diag(exp(G)) K S0)         (one row per node),
 *   O = diag(exp(G)) Q S0 + Y U,
 * which equals replaying the recurrence along every root path.
 *   q, k  [T][H_qk][d_k]   io dtype
 *   v     [T][H_v][d_v]    io dtype
 *   g, b  [T][H_v]         fp32; g is the log-gate (<= 0), b the write strength
 *   S0    [B][H_v][d_k][d_v] fp32, read only
 *   o     [T][H_v][d_v]    io dtype, written
 *   ws    tgdn_verify_workspace_bytes() bytes, 256-byte aligned, written
 * tgdn_tree_prep must have run on `tree` (same stream or ordered before).
 * A sequence with a bad status gets zero outputs and zero workspace rows.
 * bf16 io with d_k = d_v = 128 and depth_max <= 30 runs on tensor-core kernels
 * (sequences of at most 64 nodes: two items per SM in flight; 65-129 nodes: one
 * item at a time); every other valid case runs the fp32 SIMT kernel.
 * Returns TGDN_OK, TGDN_EINVAL, TGDN_ETOOBIG or TGDN_ECUDA. */
int tgdn_verify(const tgdn_tree* tree, const tgdn_dims* dims, const void* q, const void* k,
                const void* v, const float* g, const float* b, const float* S0, void* o,
                void* ws, tgdn_stream_t stream);

/* Per-branch recurrent verification, the method the pages measure the fused
 * kernel against ("Trees from Marginals", Experimentelle Ergebnisse: the fused
 * kernel versus per-branch recurrent verification at tree size 128).  Every
 * root-to-leaf branch is walked token by token with the GDN update eq. from
 * S0, recomputing shared prefixes; every node's output is written (nodes on
 * several branches get the same value again).  Same arguments and outputs as
 * tgdn_verify, without the workspace (no factors are produced, so nothing can
 * be committed from it).  tgdn_tree_prep must have run on `tree`.
 * Returns TGDN_OK, TGDN_EINVAL, TGDN_ETOOBIG or TGDN_ECUDA. */
int tgdn_verify_recurrent(const tgdn_tree* tree, const tgdn_dims* dims, const void* q,
                          const void* k, const void* v, const float* g, const float* b,
                          const float* S0, void* o, tgdn_stream_t stream);

/* Draft-tree construction by top-w parallel best-first expansion (Methodik 2,
 * "Baumerstellung": the w best candidates are taken from the candidate heap
 * and expanded together, so B nodes take about B / w sequential steps).
 * For each sequence b, slot 0 is the root (root_token[b], score 0, depth 0).
 * Each round takes the min(w, budget - size) best candidates (fewer if none
 * are left), gives them the next slots in order of priority, then, unless the
 * tree is full, expands them: the node in slot i offers its K continuations
 * child_token[b][i][r] with priority score[i] + child_logp[b][i][r] (one fp32
 * addition; the path log-probability), except beyond depth_max.  Ties go to
 * the smaller id i * K + r.  Row i of the tables is the drafter's output for
 * the node in slot i (rows of slots the tree never reaches are not read).
 *   root_token  [B] int32
 *   child_logp  [B][budget][K] fp32, finite
 *   child_token [B][budget][K] int32
 *   parent, token, depth [B][budget] int32 out: parent slot (-1 for the root),
 *               token, depth; -1 in the slots past n_nodes[b]
 *   score       [B][budget] fp32 out: path log-probability (0 past n_nodes[b])
 *   n_nodes     [B] int32 out: tree size (budget unless candidates ran out)
 *   rounds      [B] int32 out: rounds that took at least one candidate
 * Parents precede children, so parent[b][0:n_nodes[b]] is a tree tgdn_tree_prep
 * takes as is.  1 <= budget <= TGDN_MAX_NODES, 1 <= K <= TGDN_BUILD_MAX_K,
 * w >= 1, 0 <= depth_max <= TGDN_MAX_DEPTH.
 * Returns TGDN_OK, TGDN_EINVAL, TGDN_ETOOBIG or TGDN_ECUDA. */
#define TGDN_BUILD_MAX_K 16
int tgdn_tree_build(int32_t B, int32_t budget, int32_t K, int32_t w, int32_t depth_max,
                    const int32_t* root_token, const float* child_logp,
                    const int32_t* child_token, int32_t* parent, int32_t* token, float* score,
                    int32_t* depth, int32_t* n_nodes, int32_t* rounds, tgdn_stream_t stream);

/* Ancestor-masked tree attention for the verifier's attention layers
 * (Problemstellung: tree verification in attention layers uses attention
 * masks).  Node n of sequence b attends to the sequence's cached context
 * (positions 0 .. prefix_len[b] - 1) and to the tree nodes on its own root
 * path, itself included:
 *   o[n][h] = softmax_j(scale * q[n][h] . k_j) v_j   over those keys j,
 * query head h reading key/value head h / (H_q / H_kv).  bf16 tensors:
 *   q       [T][H_q][d]        k_tree, v_tree [T][H_kv][d]  (the tree's own keys)
 *   k_cache, v_cache [B][P_max][H_kv][d]  (cached context; may be NULL if P_max is 0)
 *   prefix_len [B] int32 (device; clamped to [0, P_max])
 *   o       [T][H_q][d] bf16, written
 *   ws      optional workspace of tgdn_tree_attention_workspace_bytes() bytes
 *           (NULL, or fewer bytes: no split): with it the cached context of each
 *           (sequence, key/value head, 128 query rows) is split over several CTAs
 *           and the parts merged, which keeps every SM busy on small batches
 * tgdn_tree_prep must have run on `tree`; sequences with a bad status get zero
 * outputs.  Tensor-core kernel: d = 128, H_q / H_kv in {1, 2, 4, 8, 16},
 * n_max <= 128; other shapes return TGDN_EUNSUPPORTED.  scale must be positive
 * and finite (TGDN_EINVAL otherwise).  All pointers 16-byte aligned.  Returns
 * TGDN_OK, TGDN_EINVAL, TGDN_ETOOBIG, TGDN_EUNSUPPORTED or TGDN_ECUDA. */
int tgdn_tree_attention(const tgdn_tree* tree, int32_t H_q, int32_t H_kv, int32_t d,
                        const void* q, const void* k_tree, const void* v_tree,
                        const void* k_cache, const void* v_cache, const int32_t* prefix_len,
                        int32_t P_max, float scale, void* o, void* ws, size_t ws_bytes,
                        tgdn_stream_t stream);

/* Workspace bytes that let tgdn_tree_attention split the cached context for this
 * tree and shape on the current device (0: no split would be used, or invalid
 * arguments). */
size_t tgdn_tree_attention_workspace_bytes(const tgdn_tree* tree, int32_t H_q, int32_t H_kv,
                                           int32_t d, int32_t P_max);

/* Greedy acceptance (Experimentelle Ergebnisse, mean acceptance length).  The
 * root is always accepted; a non-root node is accepted when it and every
 * non-root node on its root path satisfy target_ids == draft_ids.  The
 * accepted node is the deepest accepted node, ties going to the smallest
 * topological position.
 *   draft_ids, target_ids [T] int32 (target_ids[n]: the verifier's token for
 *                                     node n's position)
 *   accept_node [B] int32: local index, -1 for an empty or invalid tree
 *   accept_len  [B] int32: depth + 1 (root counted), 0 if none
 *   path        [B][depth_max + 1] int32: local indices root first, -1 padded
 * Returns TGDN_OK, TGDN_EINVAL or TGDN_ECUDA. */
int tgdn_accept(const tgdn_tree* tree, const int32_t* draft_ids, const int32_t* target_ids,
                int32_t* accept_node, int32_t* accept_len, int32_t* path,
                tgdn_stream_t stream);

/* Deferred, rollback-free state commitment (Methodik 3, last bullet): with
 * n* = accept_node[b] and P its root path,
 *   S_out = exp(G_n*) S_in + sum_{s in P} exp(G_n* - G_s) k_s u_s^T
 * using the U and G that tgdn_verify left in `ws` for the same tree and the
 * same S_in.  S_in, S_out [B][H_v][d_k][d_v] fp32; S_out may equal S_in (in
 * place); otherwise the two must not overlap.  Sequences with n* < 0 or a
 * bad status keep S_in.  k is the same [T][H_qk][d_k] tensor given to verify.
 * Returns TGDN_OK, TGDN_EINVAL or TGDN_ECUDA. */
int tgdn_commit(const tgdn_tree* tree, const tgdn_dims* dims, const int32_t* accept_node,
                const void* k, const void* ws, const float* S_in, float* S_out,
                tgdn_stream_t stream);

/* One decode step with the previous step's commit deferred into it
 * (Methodik 3, last bullet: the state is committed in the next decoding
 * iteration, once the accepted branch is known).  Equivalent to
 *   tgdn_commit(prev_tree, dims, prev_accept_node, prev_k, prev_ws, S, S);
 *   tgdn_verify(tree, dims, q, k, v, g, b, S, o, ws);
 * but, on the tensor-core path, each state block is read once, updated in
 * registers, written back once and verified from the same registers, so the
 * state crosses HBM once per direction per step instead of three times.
 *   S              [B][H_v][d_k][d_v] fp32: on entry the state the previous
 *                  step verified from; on return the committed state (the S0
 *                  of this step's verification)
 *   prev_tree      the previous step's tree (same B, prep'd, unchanged since)
 *   prev_accept_node, prev_path  the previous step's tgdn_accept outputs
 *                  ([B] and [B][prev_tree->depth_max + 1])
 *   prev_k         the previous step's k
 *   prev_ws        the previous step's verify workspace; it must not overlap
 *                  ws (alternate two workspaces step after step)
 * Other arguments as tgdn_verify.  Sequences whose previous tree was empty or
 * invalid keep their state.  The tensor-core path needs what tgdn_verify's
 * needs plus prev_tree->depth_max <= 30; other cases run the two passes.
 * The last step of a decode still needs its own tgdn_commit.
 * Returns TGDN_OK, TGDN_EINVAL, TGDN_ETOOBIG or TGDN_ECUDA. */
int tgdn_verify_fused(const tgdn_tree* tree, const tgdn_dims* dims, const void* q,
                      const void* k, const void* v, const float* g, const float* b, float* S,
                      void* o, void* ws, const tgdn_tree* prev_tree,
                      const int32_t* prev_accept_node, const int32_t* prev_path,
                      const void* prev_k, const void* prev_ws, tgdn_stream_t stream);

/* Verification for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this call; it exists for integrators.  Some
 * callers of this library cannot call cudaMalloc: a plugin inside a serving
 * engine that has reserved all device memory for its own pools and hands its
 * extensions only input and output buffers, or code on a latency-critical
 * path that must not take cudaMalloc's implicit device synchronisation.
 * tgdn_verify_noalloc computes exactly what tgdn_verify computes (same
 * arguments minus the workspace) and keeps the factors U and G in a
 * library-owned device array of TGDN_NOALLOC_SCRATCH_BYTES instead of a
 * caller workspace.  That array is a file-scope static: every GPU that loads
 * the library holds it until the process exits.
 *   - Sizes: tgdn_verify_workspace_bytes(tree, dims) must not exceed
 *     TGDN_NOALLOC_SCRATCH_BYTES, otherwise TGDN_ETOOBIG is returned and
 *     nothing is enqueued.
 *   - Device: every call looks up the array's device address
 *     (cudaGetSymbolAddress) in the calling thread's current context, so the stream
 *     must belong to that context's device.  The first call on a device may load
 *     the library's device code (which holds the array); make it before any
 *     stream capture.
 *   - Sharing: every call on a device uses the same array and leaves its
 *     contents behind.  Calls whose kernels overlap on the GPU (different
 *     streams without ordering) race on it; order them on one stream.
 *   - The factors stay inside the library, so tgdn_commit cannot use them:
 *     a caller that commits uses tgdn_verify with its own workspace.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Returns TGDN_OK, TGDN_EINVAL, TGDN_ETOOBIG or TGDN_ECUDA. */
#define TGDN_NOALLOC_SCRATCH_BYTES (20u * 1024u * 1024u)
int tgdn_verify_noalloc(const tgdn_tree* tree, const tgdn_dims* dims, const void* q,
                        const void* k, const void* v, const float* g, const float* b,
                        const float* S0, void* o, tgdn_stream_t stream);

/* Test hook for the bounded device waits; the paper has no counterpart and it is
 * not meant for production use.  Every device wait of the library gives up after
 * 2 s, marks the affected sequences TGDN_SEQ_TIMEOUT and lets the kernel return
 * (nothing traps or hangs).  From the next launch on, the tensor-core verification
 * kernel for trees of at most 64 nodes (tgdn_verify, tgdn_verify_fused,
 * tgdn_verify_noalloc) uses wait_limit_ns instead (0: the 2 s default), and when
 * withhold_item >= 0 its producer warps never issue the first tensor-core product of
 * work item withhold_item (sequence withhold_item / H_v, value head
 * withhold_item % H_v), so that the consumer's wait for it expires: the CTA that owns
 * that item stops,
 * reports every item it owns as TGDN_SEQ_TIMEOUT, waits for its own copies and
 * products to finish and returns; other CTAs are unaffected.  Process-wide, not
 * thread-safe with concurrent launches; tgdn_debug_set_wait_hooks(0, -1) restores
 * the defaults.  Returns TGDN_OK, or TGDN_EINVAL for wait_limit_ns above 2 s or
 * withhold_item < -1. */
int tgdn_debug_set_wait_hooks(uint64_t wait_limit_ns, int32_t withhold_item);

/* Static, human-readable text for a tgdn_status value. */
const char* tgdn_status_string(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int tgdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TGDN_H_ */
