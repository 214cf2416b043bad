// tgdn_api.cu — the C ABI (include/tgdn.h): host-side argument checks,
// kernel selection and TMA descriptor encoding.  No call allocates memory.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace {

using tgdn::WsLayout;

// An NVTX range around each call of the C ABI (a no-op unless a profiler listens), so
// that a timeline shows which library call enqueued which kernels.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
};

int check_tree(const tgdn_tree* t) {
  if (!t) return TGDN_EINVAL;
  if (t->B < 0 || t->T < 0 || t->n_max < 1 || t->depth_max < 0) return TGDN_EINVAL;
  if (t->n_max > TGDN_MAX_NODES || t->depth_max > TGDN_MAX_DEPTH) return TGDN_ETOOBIG;
  if (t->words != (t->n_max + 63) / 64) return TGDN_EINVAL;
  if (t->B > 0 && (!t->cu_nodes || !t->status)) return TGDN_EINVAL;
  if (t->T > 0 && (!t->parent || !t->depth || !t->order || !t->pos || !t->anc))
    return TGDN_EINVAL;
  return TGDN_OK;
}

int check_dims(const tgdn_dims* d) {
  if (!d) return TGDN_EINVAL;
  if (d->H_qk < 1 || d->H_v < 1 || d->H_v % d->H_qk != 0) return TGDN_EINVAL;
  if (d->d_k < 1 || d->d_v < 1) return TGDN_EINVAL;
  if (d->d_k > TGDN_MAX_HEAD_DIM || d->d_v > TGDN_MAX_HEAD_DIM) return TGDN_ETOOBIG;
  if (d->io != TGDN_F32 && d->io != TGDN_BF16) return TGDN_EINVAL;
  return TGDN_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? TGDN_OK : TGDN_ECUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// q or k [T][H_qk][128] bf16 as a 3-D tensor; box = 64 elements x 1 head x 64 rows,
// 128-byte swizzle (the tcgen05 K-major SWIZZLE_128B operand layout).
bool encode_qk_map(CUtensorMap* map, const void* base, int T, int H_qk) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)H_qk, (cuuint64_t)T};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H_qk * 128 * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows][H][128] bf16 tensor as a 3-D TMA map with box {64, box_h, box_rows},
// 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, const void* base, long rows, int H, int box_h,
                     int box_rows) {
  auto fn = encode_fn();
  if (!fn || rows < 1) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace tgdn {

namespace {
std::atomic<unsigned long long> g_hook_wait_ns{0};
std::atomic<int> g_hook_item{-1};
}  // namespace

WaitHooks wait_hooks() { return WaitHooks{g_hook_wait_ns.load(), g_hook_item.load()}; }

int device_sm_count() {
  constexpr int kDevices = 64;
  static std::atomic<int> cache[kDevices];  // 0: not looked up yet
  int dev = 0, c = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kDevices) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1)
    return 1;
  if (dev >= 0 && dev < kDevices) cache[dev].store(c, std::memory_order_relaxed);
  return c;
}

bool encode_out_maps(OutMaps* m, float* U, void* o, int T, int H_v) {
  auto fn = encode_fn();
  if (!fn || T < 1) return false;
  const cuuint64_t dims[3] = {128, (cuuint64_t)H_v, (cuuint64_t)T};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint64_t su[2] = {128 * 4, (cuuint64_t)H_v * 128 * 4};
  const cuuint64_t so[2] = {128 * 2, (cuuint64_t)H_v * 128 * 2};
  auto enc = [&](CUtensorMap* map, CUtensorMapDataType ty, void* base, const cuuint64_t* str,
                 cuuint32_t inner, cuuint32_t rows) {
    const cuuint32_t box[3] = {inner, 1, rows};
    return fn(map, ty, 3, base, dims, str, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  return enc(&m->u64, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, U, su, 32, 64) &&
         enc(&m->u8, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, U, su, 32, 8) &&
         enc(&m->o64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o, so, 64, 64) &&
         enc(&m->o8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o, so, 64, 8);
}

}  // namespace tgdn

extern "C" {

int tgdn_version(void) { return 100; }

int tgdn_debug_set_wait_hooks(uint64_t wait_limit_ns, int32_t withhold_item) {
  if (wait_limit_ns > tgdn::kWaitLimitNs || withhold_item < -1) return TGDN_EINVAL;
  tgdn::g_hook_wait_ns.store(wait_limit_ns);
  tgdn::g_hook_item.store(withhold_item);
  return TGDN_OK;
}

const char* tgdn_status_string(int code) {
  switch (code) {
    case TGDN_OK: return "ok";
    case TGDN_EINVAL: return "invalid argument";
    case TGDN_ETOOBIG: return "size above the library limits";
    case TGDN_ECUDA: return "CUDA launch or driver error";
    case TGDN_EUNSUPPORTED: return "unsupported configuration";
    default: return "unknown status";
  }
}

int tgdn_tree_prep(const tgdn_tree* tree, tgdn_stream_t stream) {
  CallRange range_("tgdn_tree_prep");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  return from_cuda(tgdn::launch_tree_prep(*tree, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tgdn_verify_workspace_bytes(const tgdn_tree* tree, const tgdn_dims* dims) {
  if (check_tree(tree) != TGDN_OK || check_dims(dims) != TGDN_OK) return 0;
  return tgdn::ws_layout(*tree, *dims).bytes;
}

int tgdn_verify(const tgdn_tree* tree, const tgdn_dims* dims, const void* q, const void* k,
                const void* v, const float* g, const float* b, const float* S0, void* o,
                void* ws, tgdn_stream_t stream) {
  CallRange range_("tgdn_verify");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  rc = check_dims(dims);
  if (rc != TGDN_OK) return rc;
  const tgdn_tree& t = *tree;
  const tgdn_dims& d = *dims;
  if (t.T > 0 && (!q || !k || !v || !g || !b || !o || !ws)) return TGDN_EINVAL;
  if (t.B > 0 && !S0) return TGDN_EINVAL;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return TGDN_EINVAL;
  if (t.B == 0 || t.T == 0) return TGDN_OK;
  const WsLayout L = tgdn::ws_layout(t, d);
  float* U = reinterpret_cast<float*>(static_cast<char*>(ws) + L.u_off);
  float* G = reinterpret_cast<float*>(static_cast<char*>(ws) + L.g_off);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (tgdn::verify_tc_supported(t, d, q, k, v, S0, o)) {
    CUtensorMap qmap, kmap, vmap;
    tgdn::OutMaps om;
    if (!encode_qk_map(&qmap, q, t.T, d.H_qk) || !encode_qk_map(&kmap, k, t.T, d.H_qk) ||
        !encode_rows_map(&vmap, v, t.T, d.H_v, 1, 64) ||
        !tgdn::encode_out_maps(&om, U, o, t.T, d.H_v))
      return TGDN_ECUDA;  // the driver could not describe q/k/v/U/o for TMA
    const tgdn::PendingCommit none{};
    return from_cuda(tgdn::launch_verify_tc(t, d, qmap, kmap, vmap, om, g, b,
                                            const_cast<float*>(S0), o, U, G, none, false, s));
  }
  if (tgdn::verify_tc128_supported(t, d, q, k, v, S0, o)) {
    CUtensorMap qmap, kmap, vmap;
    tgdn::OutMaps om;
    if (!encode_qk_map(&qmap, q, t.T, d.H_qk) || !encode_qk_map(&kmap, k, t.T, d.H_qk) ||
        !encode_rows_map(&vmap, v, t.T, d.H_v, 1, 64) ||
        !tgdn::encode_out_maps(&om, U, o, t.T, d.H_v))
      return TGDN_ECUDA;
    // sequences of at most 64 nodes on the 64-node kernel (two items in flight per SM),
    // the larger ones on the 128-node kernel; each kernel passes over the other's
    const tgdn::PendingCommit none{};
    rc = from_cuda(tgdn::launch_verify_tc(t, d, qmap, kmap, vmap, om, g, b,
                                          const_cast<float*>(S0), o, U, G, none, true, s));
    if (rc != TGDN_OK) return rc;
    rc = from_cuda(
        tgdn::launch_verify_tc128(t, d, qmap, kmap, q, k, v, g, b, S0, o, U, G, true, s));
    if (rc != TGDN_OK || t.n_max < tgdn::kTc128FoldNodes) return rc;
    // 129-node trees whose root is not node 0 (the rest of the batch is done)
    return from_cuda(tgdn::launch_verify_simt(t, d, q, k, v, g, b, S0, o, U, G, s,
                                              tgdn::kTc128FoldNodes));
  }
  return from_cuda(tgdn::launch_verify_simt(t, d, q, k, v, g, b, S0, o, U, G, s));
}

int tgdn_verify_fused(const tgdn_tree* tree, const tgdn_dims* dims, const void* q,
                      const void* k, const void* v, const float* g, const float* b, float* S,
                      void* o, void* ws, const tgdn_tree* prev_tree,
                      const int32_t* prev_accept_node, const int32_t* prev_path,
                      const void* prev_k, const void* prev_ws, tgdn_stream_t stream) {
  CallRange range_("tgdn_verify_fused");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  rc = check_tree(prev_tree);
  if (rc != TGDN_OK) return rc;
  rc = check_dims(dims);
  if (rc != TGDN_OK) return rc;
  const tgdn_tree& t = *tree;
  const tgdn_tree& pt = *prev_tree;
  const tgdn_dims& d = *dims;
  if (pt.B != t.B) return TGDN_EINVAL;  // the same sequences, step after step
  if (t.T > 0 && (!q || !k || !v || !g || !b || !o || !ws)) return TGDN_EINVAL;
  if (t.B > 0 && (!S || !prev_accept_node || !prev_path)) return TGDN_EINVAL;
  if (pt.T > 0 && (!prev_k || !prev_ws)) return TGDN_EINVAL;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0 ||
      reinterpret_cast<uintptr_t>(prev_ws) % 256 != 0)
    return TGDN_EINVAL;
  if (t.B == 0) return TGDN_OK;
  const WsLayout L = tgdn::ws_layout(t, d);
  const WsLayout PL = tgdn::ws_layout(pt, d);
  if (t.T > 0 && pt.T > 0) {  // this step's factors must not overwrite the pending ones
    const char* a = static_cast<const char*>(ws);
    const char* c = static_cast<const char*>(prev_ws);
    if (a < c + PL.bytes && c < a + L.bytes) return TGDN_EINVAL;
  }
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float* pU = pt.T > 0 ? reinterpret_cast<const float*>(
                                   static_cast<const char*>(prev_ws) + PL.u_off)
                             : nullptr;
  const float* pG = pt.T > 0 ? reinterpret_cast<const float*>(
                                   static_cast<const char*>(prev_ws) + PL.g_off)
                             : nullptr;
  if (t.T > 0 && pt.T > 0 && tgdn::verify_tc_supported(t, d, q, k, v, S, o) &&
      tgdn::pending_commit_tc_supported(pt, prev_k)) {
    float* U = reinterpret_cast<float*>(static_cast<char*>(ws) + L.u_off);
    float* G = reinterpret_cast<float*>(static_cast<char*>(ws) + L.g_off);
    CUtensorMap qmap, kmap, vmap;
    tgdn::OutMaps om;
    if (!encode_qk_map(&qmap, q, t.T, d.H_qk) || !encode_qk_map(&kmap, k, t.T, d.H_qk) ||
        !encode_rows_map(&vmap, v, t.T, d.H_v, 1, 64) ||
        !tgdn::encode_out_maps(&om, U, o, t.T, d.H_v))
      return TGDN_ECUDA;
    const tgdn::PendingCommit cm{pt.cu_nodes, pt.status, prev_path, pt.depth_max + 1,
                                 prev_k,      pU,        pG};
    return from_cuda(
        tgdn::launch_verify_tc(t, d, qmap, kmap, vmap, om, g, b, S, o, U, G, cm, false, s));
  }
  // any other case: the commit as its own pass, then the verify
  if (pt.T > 0) {
    rc = from_cuda(tgdn::launch_commit(pt, d, prev_accept_node, prev_k, pU, pG, S, S, s));
    if (rc != TGDN_OK) return rc;
  }
  return tgdn_verify(tree, dims, q, k, v, g, b, S, o, ws, stream);
}

int tgdn_verify_recurrent(const tgdn_tree* tree, const tgdn_dims* dims, const void* q,
                          const void* k, const void* v, const float* g, const float* b,
                          const float* S0, void* o, tgdn_stream_t stream) {
  CallRange range_("tgdn_verify_recurrent");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  rc = check_dims(dims);
  if (rc != TGDN_OK) return rc;
  const tgdn_tree& t = *tree;
  if (t.T > 0 && (!q || !k || !v || !g || !b || !o)) return TGDN_EINVAL;
  if (t.B > 0 && !S0) return TGDN_EINVAL;
  if (t.B == 0 || t.T == 0) return TGDN_OK;
  return from_cuda(tgdn::launch_verify_recurrent(t, *dims, q, k, v, g, b, S0, o,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int tgdn_tree_build(int32_t B, int32_t budget, int32_t K, int32_t w, int32_t depth_max,
                    const int32_t* root_token, const float* child_logp,
                    const int32_t* child_token, int32_t* parent, int32_t* token, float* score,
                    int32_t* depth, int32_t* n_nodes, int32_t* rounds, tgdn_stream_t stream) {
  CallRange range_("tgdn_tree_build");
  if (B < 0 || budget < 1 || K < 1 || w < 1 || depth_max < 0) return TGDN_EINVAL;
  if (budget > TGDN_MAX_NODES || K > TGDN_BUILD_MAX_K || depth_max > TGDN_MAX_DEPTH)
    return TGDN_ETOOBIG;
  if (B == 0) return TGDN_OK;
  if (!root_token || !child_logp || !child_token || !parent || !token || !score || !depth ||
      !n_nodes || !rounds)
    return TGDN_EINVAL;
  return from_cuda(tgdn::launch_tree_build(B, budget, K, w, depth_max, root_token, child_logp,
                                           child_token, parent, token, score, depth, n_nodes,
                                           rounds, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tgdn_tree_attention_workspace_bytes(const tgdn_tree* tree, int32_t H_q, int32_t H_kv,
                                           int32_t d, int32_t P_max) {
  if (check_tree(tree) != TGDN_OK || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || P_max < 0)
    return 0;
  if (!tgdn::tree_attn_supported(*tree, H_q, H_kv, d)) return 0;
  return tgdn::tree_attn_workspace_bytes(*tree, H_q, H_kv, P_max);
}

int tgdn_tree_attention(const tgdn_tree* tree, int32_t H_q, int32_t H_kv, int32_t d,
                        const void* q, const void* k_tree, const void* v_tree,
                        const void* k_cache, const void* v_cache, const int32_t* prefix_len,
                        int32_t P_max, float scale, void* o, void* ws, size_t ws_bytes,
                        tgdn_stream_t stream) {
  CallRange range_("tgdn_tree_attention");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  const tgdn_tree& t = *tree;
  if (H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || d < 1 || P_max < 0) return TGDN_EINVAL;
  if (!(scale > 0.f && isfinite(scale))) return TGDN_EINVAL;  // positive and finite
  if (!tgdn::tree_attn_supported(t, H_q, H_kv, d)) return TGDN_EUNSUPPORTED;
  if (t.B > 0 && (!prefix_len || (P_max > 0 && (!k_cache || !v_cache)))) return TGDN_EINVAL;
  if (t.T > 0 && (!q || !k_tree || !v_tree || !o)) return TGDN_EINVAL;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; };
  if (!al16(q) || !al16(k_tree) || !al16(v_tree) || !al16(k_cache) || !al16(v_cache) ||
      !al16(o) || !al16(ws))
    return TGDN_EINVAL;
  if (t.B == 0 || t.T == 0) return TGDN_OK;
  const int G = H_q / H_kv;
  CUtensorMap qm, ktm, vtm, kcm, vcm;
  // with no cached context the cache maps are never read; describe the tree instead
  const void* kc = P_max > 0 ? k_cache : k_tree;
  const void* vc = P_max > 0 ? v_cache : v_tree;
  const long crows = P_max > 0 ? (long)t.B * P_max : t.T;
  if (!encode_rows_map(&qm, q, t.T, H_q, G, 128 / G) ||
      !encode_rows_map(&ktm, k_tree, t.T, H_kv, 1, 128) ||
      !encode_rows_map(&vtm, v_tree, t.T, H_kv, 1, 128) ||
      !encode_rows_map(&kcm, kc, crows, H_kv, 1, 128) ||
      !encode_rows_map(&vcm, vc, crows, H_kv, 1, 128))
    return TGDN_ECUDA;
  return from_cuda(tgdn::launch_tree_attn(t, H_q, H_kv, P_max, scale, qm, ktm, vtm, kcm, vcm,
                                          prefix_len, o, ws, ws ? ws_bytes : 0,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int tgdn_accept(const tgdn_tree* tree, const int32_t* draft_ids, const int32_t* target_ids,
                int32_t* accept_node, int32_t* accept_len, int32_t* path,
                tgdn_stream_t stream) {
  CallRange range_("tgdn_accept");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  if (tree->B > 0 && (!accept_node || !accept_len || !path)) return TGDN_EINVAL;
  if (tree->T > 0 && (!draft_ids || !target_ids)) return TGDN_EINVAL;
  return from_cuda(tgdn::launch_accept(*tree, draft_ids, target_ids, accept_node, accept_len,
                                       path, reinterpret_cast<cudaStream_t>(stream)));
}

int tgdn_commit(const tgdn_tree* tree, const tgdn_dims* dims, const int32_t* accept_node,
                const void* k, const void* ws, const float* S_in, float* S_out,
                tgdn_stream_t stream) {
  CallRange range_("tgdn_commit");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  rc = check_dims(dims);
  if (rc != TGDN_OK) return rc;
  const tgdn_tree& t = *tree;
  const tgdn_dims& d = *dims;
  if (t.B > 0 && (!accept_node || !S_in || !S_out)) return TGDN_EINVAL;
  if (t.T > 0 && (!k || !ws)) return TGDN_EINVAL;
  if (t.B == 0) return TGDN_OK;
  if (S_in != S_out) {  // distinct buffers must not overlap
    const size_t bytes = (size_t)t.B * d.H_v * d.d_k * d.d_v * sizeof(float);
    const char* a = reinterpret_cast<const char*>(S_in);
    const char* c = reinterpret_cast<const char*>(S_out);
    if (a < c + bytes && c < a + bytes) return TGDN_EINVAL;
  }
  const WsLayout L = tgdn::ws_layout(t, d);
  const float* U = reinterpret_cast<const float*>(static_cast<const char*>(ws) + L.u_off);
  const float* G = reinterpret_cast<const float*>(static_cast<const char*>(ws) + L.g_off);
  return from_cuda(tgdn::launch_commit(t, d, accept_node, k, U, G, S_in, S_out,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// tgdn_verify_noalloc: the same verification with the factors kept in a
// library-owned device array, for callers that cannot allocate.
// ---------------------------------------------------------------------------
namespace {

// One array per device that loads the library, alive until the process exits.
// In host code this name is only a host-side stand-in: the device address is
// looked up with cudaGetSymbolAddress (below) and passed to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TGDN_NOALLOC_SCRATCH_BYTES];

// Device address of the array in the current context.  It is looked up on every
// call (cheap once the library's device code is loaded): an address cached per
// device would go stale after cudaDeviceReset or under another context.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return TGDN_ECUDA;
  *out = p;
  return TGDN_OK;
}

}  // namespace

extern "C" int tgdn_verify_noalloc(const tgdn_tree* tree, const tgdn_dims* dims, const void* q,
                                   const void* k, const void* v, const float* g,
                                   const float* b, const float* S0, void* o,
                                   tgdn_stream_t stream) {
  CallRange range_("tgdn_verify_noalloc");
  int rc = check_tree(tree);
  if (rc != TGDN_OK) return rc;
  rc = check_dims(dims);
  if (rc != TGDN_OK) return rc;
  if (tgdn::ws_layout(*tree, *dims).bytes > TGDN_NOALLOC_SCRATCH_BYTES) return TGDN_ETOOBIG;
  void* ws = nullptr;
  rc = noalloc_scratch(&ws);
  if (rc != TGDN_OK) return rc;
  // Every row of U and G that the launch covers is written by it, so the
  // contents left by an earlier call need no clearing.
  return tgdn_verify(tree, dims, q, k, v, g, b, S0, o, ws, stream);
}
