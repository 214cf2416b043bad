// tgdn_kernels.h — internal launchers behind the C ABI (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tgdn.h"

namespace tgdn {

// Streaming multiprocessors of the current device (cached per device; safe to call
// from several host threads).  1 if the device cannot be queried.
int device_sm_count();

// Workspace layout shared by verify (writer) and commit (reader).
struct WsLayout {
  size_t u_off, g_off, bytes;
};
inline WsLayout ws_layout(const tgdn_tree& t, const tgdn_dims& d) {
  WsLayout w;
  w.u_off = 0;
  const size_t u_bytes = (size_t)t.T * d.H_v * d.d_v * sizeof(float);
  w.g_off = (u_bytes + 255) / 256 * 256;
  w.bytes = w.g_off + (size_t)t.T * d.H_v * sizeof(float);
  return w;
}

cudaError_t launch_tree_prep(const tgdn_tree& t, cudaStream_t s);
cudaError_t launch_accept(const tgdn_tree& t, const int32_t* draft, const int32_t* target,
                          int32_t* accept_node, int32_t* accept_len, int32_t* path,
                          cudaStream_t s);

// fp32 SIMT verify: any valid geometry (d_k, d_v <= 128, n_max <= 256, depth_max <= 64).
// only_n > 0: just the valid sequences of only_n nodes whose root is not node 0.
cudaError_t launch_verify_simt(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                               const void* k, const void* v, const float* g, const float* b,
                               const float* S0, void* o, float* U, float* G, cudaStream_t s,
                               int only_n = 0);

// The previous decode step's commit, folded into this step's verify: the
// accepted root path of every sequence and the factors of that step.
// path == nullptr means there is nothing to commit.
struct PendingCommit {
  const int32_t* cu;      // previous tree: cu_nodes [B + 1]
  const int32_t* status;  // previous tree: status [B]
  const int32_t* path;    // [B][path_len] accepted root path, root first, -1 padded
  int path_len;           // previous depth_max + 1
  const void* k;          // previous keys [T'][H_qk][d_k] (bf16)
  const float* U;         // previous factors [T'][H_v][d_v]
  const float* G;         // previous path-cumulative log-gates [T'][H_v]
};

// Tensor-core verify: bf16 io, d_k = d_v = 128, n_max <= 64, depth_max <= 30; with
// small_only the node bound is per sequence (larger sequences are passed over).
bool verify_tc_supported(const tgdn_tree& t, const tgdn_dims& d, const void* q, const void* k,
                         const void* v, const float* S0, const void* o, bool small_only = false);
// Tensor-core verify for larger trees: bf16 io, d_k = d_v = 128, n_max <= 129,
// depth_max <= 30; one item per SM at a time, sparse second step on CUDA cores.
// A 129-node tree is taken when its root is node 0 (the root is folded into the
// state); otherwise it is left for launch_verify_simt(..., only_n = 129).
constexpr int kTc128FoldNodes = 129;
bool verify_tc128_supported(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                            const void* k, const void* v, const float* S0, const void* o);
// big_only: sequences of at most 64 nodes are passed over (the 64-node kernel's).
cudaError_t launch_verify_tc128(const tgdn_tree& t, const tgdn_dims& d, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const void* q, const void* k,
                                const void* v, const float* g,
                                const float* b, const float* S0, void* o, float* U, float* G,
                                bool big_only, cudaStream_t s);
// Tensor maps of the verify outputs for TMA stores (128-byte swizzle): the factors
// U [T][H_v][128] fp32 with boxes {32, 1, 64} and {32, 1, 8}, the outputs o
// [T][H_v][128] bf16 with boxes {64, 1, 64} and {64, 1, 8}.
struct OutMaps {
  CUtensorMap u64, u8, o64, o8;
};
bool encode_out_maps(OutMaps* m, float* U, void* o, int T, int H_v);
// Test hooks of the bounded device waits (tgdn_debug_set_wait_hooks): a shorter wait
// limit (0: the default) and a work item whose hand-over the 64-node kernel's producer
// withholds (-1: none).
struct WaitHooks {
  uint64_t wait_ns;
  int hold_item;
};
WaitHooks wait_hooks();
// Whether the tensor-core verify can also apply a pending commit of `prev`.
bool pending_commit_tc_supported(const tgdn_tree& prev, const void* prev_k);
// With cm.path set, S is first updated in place by the pending commit and the
// committed state is verified; otherwise S is only read.  small_only (no pending
// commit): only the sequences of at most 64 nodes are verified, the rest untouched.
cudaError_t launch_verify_tc(const tgdn_tree& t, const tgdn_dims& d, const CUtensorMap& qmap,
                             const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const OutMaps& om, const float* g, const float* b, float* S,
                             void* o, float* U, float* G, const PendingCommit& cm,
                             bool small_only, cudaStream_t s);

// Per-branch recurrent verification (every root-to-leaf path replayed from S0).
cudaError_t launch_verify_recurrent(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                                    const void* k, const void* v, const float* g,
                                    const float* b, const float* S0, void* o, cudaStream_t s);

// Top-w best-first draft-tree construction, one warp per sequence.
size_t tree_build_smem_bytes(int budget, int K);
cudaError_t launch_tree_build(int B, int budget, int K, int w, int depth_max,
                              const int32_t* root_token, const float* child_logp,
                              const int32_t* child_token, int32_t* parent, int32_t* token,
                              float* score, int32_t* depth, int32_t* n_nodes, int32_t* rounds,
                              cudaStream_t s);

// Ancestor-masked tree attention (bf16, d = 128), one CTA per (sequence, key/value
// head, 128 query rows).  Tensor maps: q [T][H_q][128] with box {64, G, 128 / G};
// k_tree, v_tree [T][H_kv][128] and k_cache, v_cache [B * P_max][H_kv][128] with
// box {64, 1, 64}; all 128-byte swizzled.
// With a workspace of tree_attn_workspace_bytes() (0: no split for this shape) the
// cached context is split over several CTAs and merged by a second kernel.
bool tree_attn_supported(const tgdn_tree& t, int H_q, int H_kv, int d);
size_t tree_attn_workspace_bytes(const tgdn_tree& t, int H_q, int H_kv, int P_max);
cudaError_t launch_tree_attn(const tgdn_tree& t, int H_q, int H_kv, int P_max, float scale,
                             const CUtensorMap& qmap, const CUtensorMap& ktmap,
                             const CUtensorMap& vtmap, const CUtensorMap& kcmap,
                             const CUtensorMap& vcmap, const int32_t* prefix_len, void* o,
                             void* ws, size_t ws_bytes, cudaStream_t s);

cudaError_t launch_commit(const tgdn_tree& t, const tgdn_dims& d, const int32_t* accept_node,
                          const void* k, const float* U, const float* G, const float* S_in,
                          float* S_out, cudaStream_t s);

}  // namespace tgdn
