// tree.cu — tree metadata and greedy acceptance kernels.
//
// tree_prep: topological sort of each draft tree and its ancestor relation
//   ("Trees from Marginals", Technisches Resümee, Methodik 3: "Der Baum wird
//   topologisch sortiert"; the interaction matrices X and Y encode ancestor
//   relations).  One warp per sequence; N <= 256 nodes live in shared memory.
// accept: greedy longest accepted root path (mean acceptance length,
//   Experimentelle Ergebnisse).  One warp per sequence.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kTreeWarps = 4;
constexpr unsigned kFull = 0xffffffffu;

__global__ void __launch_bounds__(kTreeWarps * 32)
tree_prep_kernel(int B, int T, const int32_t* __restrict__ cu, const int32_t* __restrict__ parent,
                 int n_max, int depth_max, int words, int32_t* __restrict__ depth,
                 int32_t* __restrict__ order, int32_t* __restrict__ pos,
                 uint64_t* __restrict__ anc, int32_t* __restrict__ status) {
  __shared__ int s_par[kTreeWarps][TGDN_MAX_NODES];
  __shared__ int s_dep[kTreeWarps][TGDN_MAX_NODES];
  __shared__ int s_pos[kTreeWarps][TGDN_MAX_NODES];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kTreeWarps + warp;
  if (b >= B) return;
  int* par = s_par[warp];
  int* dep = s_dep[warp];
  int* ps = s_pos[warp];
  const int lo = cu[b], hi = cu[b + 1];
  // A row range outside [0, T) is reported and nothing of the sequence is touched.
  if (lo < 0 || hi < lo || hi > T) {
    if (lane == 0) status[b] = TGDN_SEQ_BAD_RANGE;
    return;
  }
  const int N = hi - lo;

  int st = TGDN_SEQ_OK;
  if (N > n_max) st = TGDN_SEQ_TOO_BIG;
  if (st == TGDN_SEQ_OK) {
    bool bad = false;
    int roots = 0;
    for (int i = lane; i < N; i += 32) {
      const int p = parent[lo + i];
      par[i] = p;
      bad |= (p < -1) || (p >= N) || (p == i);
      roots += (p == -1);
    }
    if (__any_sync(kFull, bad)) {
      st = TGDN_SEQ_BAD_PARENT;
    } else {
      for (int o = 16; o > 0; o >>= 1) roots += __shfl_xor_sync(kFull, roots, o);
      if (N > 0 && roots != 1) st = TGDN_SEQ_ROOTS;
    }
  }
  __syncwarp();
  if (st == TGDN_SEQ_OK) {
    bool cyc = false, deep = false;
    for (int i = lane; i < N; i += 32) {
      int j = i, h = 0;
      while (par[j] != -1 && h <= N) {  // at most N + 1 hops
        j = par[j];
        ++h;
      }
      if (par[j] != -1) {
        cyc = true;
      } else {
        dep[i] = h;
        deep |= h > depth_max;
      }
    }
    if (__any_sync(kFull, cyc))
      st = TGDN_SEQ_CYCLE;
    else if (__any_sync(kFull, deep))
      st = TGDN_SEQ_TOO_DEEP;
  }
  __syncwarp();
  if (lane == 0) status[b] = st;
  if (st != TGDN_SEQ_OK) {
    for (int i = lane; i < N; i += 32) {
      depth[lo + i] = -1;
      order[lo + i] = -1;
      pos[lo + i] = -1;
      for (int w = 0; w < words; ++w) anc[(size_t)(lo + i) * words + w] = 0;
    }
    return;
  }
  // Stable topological order: position = number of nodes with a smaller (depth, index).
  for (int i = lane; i < N; i += 32) {
    const int di = dep[i];
    int p = 0;
    for (int m = 0; m < N; ++m) {
      const int dm = dep[m];
      p += (dm < di) || (dm == di && m < i);
    }
    ps[i] = p;
    pos[lo + i] = p;
    order[lo + p] = i;
    depth[lo + i] = di;
  }
  __syncwarp();
  // Ancestor-or-self mask of node i, stored at row pos(i), bits pos(s).
  for (int i = lane; i < N; i += 32) {
    uint64_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    for (int j = i, h = 0; j != -1 && h <= depth_max; j = par[j], ++h) {
      const int p = ps[j];
      const uint64_t bit = 1ull << (p & 63);
      switch (p >> 6) {
        case 0: m0 |= bit; break;
        case 1: m1 |= bit; break;
        case 2: m2 |= bit; break;
        default: m3 |= bit; break;
      }
    }
    uint64_t* row = anc + (size_t)(lo + ps[i]) * words;
    row[0] = m0;
    if (words > 1) row[1] = m1;
    if (words > 2) row[2] = m2;
    if (words > 3) row[3] = m3;
  }
}

__global__ void __launch_bounds__(kTreeWarps * 32)
accept_kernel(int B, const int32_t* __restrict__ cu, const int32_t* __restrict__ parent,
              const int32_t* __restrict__ depth, const int32_t* __restrict__ status,
              int depth_max, const int32_t* __restrict__ draft,
              const int32_t* __restrict__ target, int32_t* __restrict__ accept_node,
              int32_t* __restrict__ accept_len, int32_t* __restrict__ path) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kTreeWarps + warp;
  if (b >= B) return;
  const int lo = cu[b], N = cu[b + 1] - lo;
  int32_t* prow = path + (size_t)b * (depth_max + 1);
  for (int j = lane; j <= depth_max; j += 32) prow[j] = -1;
  if (status[b] != TGDN_SEQ_OK || N == 0) {
    if (lane == 0) {
      accept_node[b] = -1;
      accept_len[b] = 0;
    }
    return;
  }
  // Key = depth * 2^16 + (2^16 - 1 - index): the max is the deepest accepted
  // node with the smallest index (= smallest topological position) at that depth.
  int best = -1;
  for (int i = lane; i < N; i += 32) {
    bool ok = true;
    for (int j = i, h = 0; h <= depth_max; ++h) {
      const int p = parent[lo + j];
      if (p == -1) break;  // the root is always accepted
      if (target[lo + j] != draft[lo + j]) {
        ok = false;
        break;
      }
      j = p;
    }
    if (ok) best = max(best, (depth[lo + i] << 16) | (0xFFFF - i));
  }
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(kFull, best, o));
  __syncwarp();
  if (lane == 0) {
    const int n = 0xFFFF - (best & 0xFFFF);
    const int d = best >> 16;
    accept_node[b] = n;
    accept_len[b] = d + 1;
    for (int j = n, h = d; h >= 0 && j != -1; --h) {
      prow[h] = j;
      j = parent[lo + j];
    }
  }
}

cudaError_t launch_tree_prep(const tgdn_tree& t, cudaStream_t s) {
  if (t.B == 0) return cudaSuccess;
  const int grid = (t.B + kTreeWarps - 1) / kTreeWarps;
  tree_prep_kernel<<<grid, kTreeWarps * 32, 0, s>>>(t.B, t.T, t.cu_nodes, t.parent, t.n_max,
                                                    t.depth_max, t.words, t.depth, t.order,
                                                    t.pos, t.anc, t.status);
  return cudaGetLastError();
}

cudaError_t launch_accept(const tgdn_tree& t, const int32_t* draft, const int32_t* target,
                          int32_t* accept_node, int32_t* accept_len, int32_t* path,
                          cudaStream_t s) {
  if (t.B == 0) return cudaSuccess;
  const int grid = (t.B + kTreeWarps - 1) / kTreeWarps;
  accept_kernel<<<grid, kTreeWarps * 32, 0, s>>>(t.B, t.cu_nodes, t.parent, t.depth, t.status,
                                                 t.depth_max, draft, target, accept_node,
                                                 accept_len, path);
  return cudaGetLastError();
}

}  // namespace tgdn
