// tree_build.cu — draft-tree construction by top-w parallel best-first expansion.
//
// "Trees from Marginals" (Technisches Resümee, Methodik 2 "Baumerstellung"):
// rather than expanding one best candidate at a time, the w best candidates are
// taken from the candidate heap together and expanded together, so a tree of B
// nodes is built in about B / w sequential steps.  A candidate's priority is
// its path log-probability (parent score + the drafter's log-probability of the
// continuation, one fp32 addition); ties go to the smaller candidate id
// (parent slot * K + rank).  Row i of the child table holds the drafter's top-K
// continuations of the node in tree slot i.
//
// One warp per sequence (sequences are independent).  The candidate pool lives
// in shared memory as 64-bit keys (order-preserving score bits, then the
// complemented id), appended as nodes are expanded, so the largest key is the
// best candidate.  Lane l owns the pool positions p = l (mod 32) and keeps the
// best key among them in a register; taking the best candidate is a warp
// maximum over the 32 lane bests, after which the warp rescans the owner's
// positions together.  Pool capacity: B * K keys (every node is expanded at
// most once).  The tree itself is kept in shared memory while it grows and is
// written out once at the end, so taking a candidate touches no global memory.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr unsigned kAll = 0xffffffffu;

// Order-preserving map of an fp32 score to 32 bits (larger score, larger key),
// with the candidate id below it (smaller id, larger key).  Finite scores never
// give the key 0, which marks a taken or missing candidate.
__device__ __forceinline__ uint64_t cand_key(float s, uint32_t id) {
  const uint32_t u = __float_as_uint(s);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | (0xFFFFFFFFu - id);
}
__device__ __forceinline__ float key_score(uint64_t key) {
  const uint32_t ord = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ uint32_t key_id(uint64_t key) {
  return 0xFFFFFFFFu - static_cast<uint32_t>(key);
}
// Warp maximum of a 64-bit key: the high words first, then the low words of the
// lanes that hold the highest high word (two warp reductions).
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x) {
  const uint32_t hi = static_cast<uint32_t>(x >> 32);
  const uint32_t mh = __reduce_max_sync(kAll, hi);
  const uint32_t ml = __reduce_max_sync(kAll, hi == mh ? static_cast<uint32_t>(x) : 0u);
  return (static_cast<uint64_t>(mh) << 32) | ml;
}

__global__ void __launch_bounds__(32)
tree_build_kernel(int B, int budget, int K, int w, int depth_max,
                  const int32_t* __restrict__ root_token, const float* __restrict__ child_logp,
                  const int32_t* __restrict__ child_token, int32_t* __restrict__ parent,
                  int32_t* __restrict__ token, float* __restrict__ score,
                  int32_t* __restrict__ depth, int32_t* __restrict__ n_nodes,
                  int32_t* __restrict__ rounds) {
  extern __shared__ __align__(16) uint8_t bsm[];
  uint64_t* pool = reinterpret_cast<uint64_t*>(bsm);                      // [budget * K]
  float* nscore = reinterpret_cast<float*>(pool + (size_t)budget * K);    // [budget]
  int* ndepth = reinterpret_cast<int*>(nscore + budget);                  // [budget]
  int* nid = ndepth + budget;  // [budget] candidate id (parent slot * K + rank); -1: root
  float* lps = reinterpret_cast<float*>(nid + budget);  // [budget * K] the drafter's log-probs
  const int b = blockIdx.x;
  const int lane = threadIdx.x;
  if (b >= B) return;
  const size_t obase = (size_t)b * budget;
  const float* lp = child_logp + obase * K;
  const int32_t* tk = child_token + obase * K;

  if (lane == 0) {
    nscore[0] = 0.f;
    ndepth[0] = 0;
    nid[0] = -1;
  }
  // the whole child table once (coalesced), so no round waits on global memory
  for (int e = lane; e < budget * K; e += 32) lps[e] = lp[e];
  __syncwarp();

  int count = 0;           // pool positions used (same in every lane)
  uint64_t best = 0;       // best key among this lane's positions
  int best_pos = -1;
  // Offer the children of slots [s0, s1) (the candidates their expansion produces).
  auto expand = [&](int s0, int s1) {
    const int total = (s1 - s0) * K;
    for (int e = lane; e < total; e += 32) {
      const int node = s0 + e / K, r = e % K;
      uint64_t key = 0;
      if (ndepth[node] + 1 <= depth_max)
        key = cand_key(__fadd_rn(nscore[node], lps[node * K + r]),
                       static_cast<uint32_t>(node * K + r));
      pool[count + e] = key;
    }
    __syncwarp();
    const int first = count + ((lane - count) % 32 + 32) % 32;  // first owned new position
    for (int p = first; p < count + total; p += 32) {
      const uint64_t k = pool[p];
      if (k > best) {
        best = k;
        best_pos = p;
      }
    }
    count += total;
  };

  expand(0, 1);
  int n = 1, nr = 0;
  while (n < budget) {
    const int take = min(w, budget - n);
    int got = 0;
    for (int t = 0; t < take; ++t) {
      const uint64_t key = warp_max_u64(best);
      if (key == 0) break;  // the pool is empty (warp-uniform)
      const int winner = __ffs(__ballot_sync(kAll, best == key)) - 1;
      const int pos = __shfl_sync(kAll, best_pos, winner);
      if (lane == winner) pool[pos] = 0;
      __syncwarp();
      // the winner's next best: its positions winner + 32 m, scanned by the whole warp
      uint64_t loc = 0;
      int loc_pos = -1;
      for (int p = winner + 32 * lane; p < count; p += 32 * 32) {
        const uint64_t k = pool[p];
        if (k > loc) {
          loc = k;
          loc_pos = p;
        }
      }
      const uint64_t nk = warp_max_u64(loc);
      const unsigned who = __ballot_sync(kAll, nk != 0 && loc == nk);
      const int npos = __shfl_sync(kAll, loc_pos, who ? __ffs(who) - 1 : 0);
      if (lane == winner) {
        best = nk;
        best_pos = nk != 0 ? npos : -1;
      }
      if (lane == 0) {  // the candidate becomes tree slot n
        const int id = static_cast<int>(key_id(key));
        nscore[n] = key_score(key);
        ndepth[n] = ndepth[id / K] + 1;
        nid[n] = id;
      }
      ++n;
      ++got;
    }
    if (got == 0) break;
    ++nr;
    __syncwarp();
    if (n < budget) expand(n - got, n);
  }
  __syncwarp();
  for (int i = lane; i < budget; i += 32) {  // slots past the tree stay padded
    const bool live = i < n;
    const int id = live ? nid[i] : -1;
    parent[obase + i] = id >= 0 ? id / K : -1;
    token[obase + i] = !live ? -1 : (id >= 0 ? tk[id] : root_token[b]);
    score[obase + i] = live ? nscore[i] : 0.f;
    depth[obase + i] = live ? ndepth[i] : -1;
  }
  if (lane == 0) {
    n_nodes[b] = n;
    rounds[b] = nr;
  }
}

size_t tree_build_smem_bytes(int budget, int K) {
  return (size_t)budget * K * (sizeof(uint64_t) + sizeof(float)) +
         (size_t)budget * (sizeof(float) + 2 * sizeof(int));
}

cudaError_t launch_tree_build(int B, int budget, int K, int w, int depth_max,
                              const int32_t* root_token, const float* child_logp,
                              const int32_t* child_token, int32_t* parent, int32_t* token,
                              float* score, int32_t* depth, int32_t* n_nodes, int32_t* rounds,
                              cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const size_t smem = tree_build_smem_bytes(budget, K);
  cudaError_t e = cudaFuncSetAttribute(tree_build_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tree_build_kernel<<<B, 32, smem, s>>>(B, budget, K, w, depth_max, root_token, child_logp,
                                        child_token, parent, token, score, depth, n_nodes,
                                        rounds);
  return cudaGetLastError();
}

}  // namespace tgdn
