// commit.cu — deferred, rollback-free state commitment.
//
// "Trees from Marginals" (Technisches Resümee, Methodik 3, last bullet): the
// state is committed once the accepted branch is known, so nothing has to be
// rolled back.  The accepted node's state follows from the same factors U that
// verification produced: with n* the accepted node and P its root path,
//   S_new = e^{G_n*} S0 + sum_{s in P} e^{G_n* - G_s} k_s u_s^T,
// a rank-|P| update of the d_k x d_v fp32 state (|P| <= depth_max + 1).
//
// The kernel streams the state once (read S_in, write S_out; in place is
// allowed): one CTA per (sequence, v-head, 32 state rows), 256 threads, each
// thread a 4-row x 4-column register tile, so every warp instruction moves one
// contiguous 512-byte state row.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kCommitThreads = 256;
constexpr int kCommitRows = 32;  // state rows per CTA

template <typename T>
__global__ void __launch_bounds__(kCommitThreads)
commit_kernel(int H_qk, int H_v, int dk, int dv, int depth_max, const int32_t* __restrict__ cu,
              const int32_t* __restrict__ parent, const int32_t* __restrict__ depth,
              const int32_t* __restrict__ status, const int32_t* __restrict__ accept_node,
              const T* __restrict__ k, const float* __restrict__ Uws,
              const float* __restrict__ Gws, const float* S_in, float* S_out, int vec) {
  extern __shared__ __align__(16) float csm[];
  const int DM1 = depth_max + 1;
  float* ck = csm;                          // [DM1][kCommitRows]  e^{G*-G_s} k_s[row]
  float* us = csm + DM1 * kCommitRows;      // [DM1][dv]           u_s
  __shared__ int s_path[TGDN_MAX_DEPTH + 1];
  __shared__ int s_len;
  __shared__ float s_decay;

  const int rblocks = (dk + kCommitRows - 1) / kCommitRows;
  const int rb = blockIdx.x % rblocks;
  const int h = (blockIdx.x / rblocks) % H_v;
  const int bi = blockIdx.x / (rblocks * H_v);
  const int qh = h / (H_v / H_qk);
  const int r0 = rb * kCommitRows;
  const int nrows = min(kCommitRows, dk - r0);
  const int tid = threadIdx.x;
  const int lo = cu[bi], N = cu[bi + 1] - lo;
  const size_t sbase = ((size_t)bi * H_v + h) * dk * dv + (size_t)r0 * dv;

  if (tid == 0) {
    const int n = accept_node[bi];
    int len = 0;
    if (status[bi] == TGDN_SEQ_OK && n >= 0 && n < N) {
      const int dn = depth[lo + n];
      if (dn >= 0 && dn <= depth_max) {
        int j = n, d = dn;
        for (; d >= 0 && j >= 0 && j < N; --d) {
          s_path[d] = j;
          j = parent[lo + j];
        }
        if (d == -1 && j == -1) len = dn + 1;  // the path reached the root at depth 0
      }
    }
    s_len = len;
    s_decay = len ? __expf(Gws[(size_t)(lo + n) * H_v + h]) : 1.f;
  }
  __syncthreads();
  const int L = s_len;
  if (L == 0) {  // nothing accepted: the state is kept
    if (S_out != S_in)
      for (int e = tid; e < nrows * dv; e += kCommitThreads)
        S_out[sbase + e] = S_in[sbase + e];
    return;
  }
  const float Gstar = Gws[(size_t)(lo + s_path[L - 1]) * H_v + h];
  for (int e = tid; e < L * kCommitRows; e += kCommitThreads) {
    const int l = e / kCommitRows, i = e % kCommitRows;
    const int s = s_path[l];
    const float c = __expf(Gstar - Gws[(size_t)(lo + s) * H_v + h]);
    ck[e] = (i < nrows) ? c * Io<T>::load(k + ((size_t)(lo + s) * H_qk + qh) * dk + r0 + i) : 0.f;
  }
  for (int e = tid; e < L * dv; e += kCommitThreads) {
    const int l = e / dv, j = e % dv;
    us[e] = Uws[((size_t)(lo + s_path[l]) * H_v + h) * dv + j];
  }
  __syncthreads();
  const float decay = s_decay;

  if (vec) {
    // 4x4 register tiles: column group cg, rows rg*4 .. rg*4+3
    const int ncg = dv >> 2;
    const int tiles = ((nrows + 3) >> 2) * ncg;
    for (int t = tid; t < tiles; t += kCommitThreads) {
      const int cg = t % ncg, rg = t / ncg;
      float4 acc[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = rg * 4 + r;
        acc[r] = (i < nrows) ? *reinterpret_cast<const float4*>(S_in + sbase + (size_t)i * dv + cg * 4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        acc[r].x *= decay;
        acc[r].y *= decay;
        acc[r].z *= decay;
        acc[r].w *= decay;
      }
      for (int l = 0; l < L; ++l) {
        const float4 u = *reinterpret_cast<const float4*>(us + l * dv + cg * 4);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float kv = ck[l * kCommitRows + rg * 4 + r];
          acc[r].x = fmaf(kv, u.x, acc[r].x);
          acc[r].y = fmaf(kv, u.y, acc[r].y);
          acc[r].z = fmaf(kv, u.z, acc[r].z);
          acc[r].w = fmaf(kv, u.w, acc[r].w);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = rg * 4 + r;
        if (i < nrows) *reinterpret_cast<float4*>(S_out + sbase + (size_t)i * dv + cg * 4) = acc[r];
      }
    }
  } else {
    for (int e = tid; e < nrows * dv; e += kCommitThreads) {
      const int i = e / dv, j = e % dv;
      float acc = decay * S_in[sbase + e];
      for (int l = 0; l < L; ++l) acc = fmaf(ck[l * kCommitRows + i], us[l * dv + j], acc);
      S_out[sbase + e] = acc;
    }
  }
}

template <typename T>
static cudaError_t launch_commit_t(const tgdn_tree& t, const tgdn_dims& d,
                                   const int32_t* accept_node, const void* k, const float* U,
                                   const float* G, const float* S_in, float* S_out,
                                   cudaStream_t s) {
  const int rblocks = (d.d_k + kCommitRows - 1) / kCommitRows;
  const long grid = (long)t.B * d.H_v * rblocks;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)(t.depth_max + 1) * (kCommitRows + d.d_v) * sizeof(float);
  const auto kern = commit_kernel<T>;
  const int vec = (d.d_v % 4 == 0) && (reinterpret_cast<uintptr_t>(S_in) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(S_out) % 16 == 0);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, kCommitThreads, smem, s>>>(d.H_qk, d.H_v, d.d_k, d.d_v, t.depth_max,
                                                     t.cu_nodes, t.parent, t.depth, t.status,
                                                     accept_node, static_cast<const T*>(k), U, G,
                                                     S_in, S_out, vec);
  return cudaGetLastError();
}

cudaError_t launch_commit(const tgdn_tree& t, const tgdn_dims& d, const int32_t* accept_node,
                          const void* k, const float* U, const float* G, const float* S_in,
                          float* S_out, cudaStream_t s) {
  if (d.io == TGDN_BF16)
    return launch_commit_t<__nv_bfloat16>(t, d, accept_node, k, U, G, S_in, S_out, s);
  return launch_commit_t<float>(t, d, accept_node, k, U, G, S_in, S_out, s);
}

}  // namespace tgdn
