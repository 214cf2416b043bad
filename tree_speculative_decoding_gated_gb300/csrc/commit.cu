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
// allowed).  One CTA per (sequence, v-head, 64 state rows), 256 threads, each
// thread two 4-row x 4-column register tiles, so every warp instruction moves
// one contiguous 512-byte state row.  The state loads are issued first; the
// accepted path is read meanwhile from the ancestor mask written by tree prep
// (one thread per candidate bit, no pointer chasing).
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kCommitThreads = 256;
constexpr int kCommitRows = 64;  // state rows per CTA
constexpr int kCommitTiles = 2;  // 4x4 tiles per thread on the vector path (d_v = 128)

template <typename T>
__global__ void __launch_bounds__(kCommitThreads)
commit_kernel(int H_qk, int H_v, int dk, int dv, int depth_max, int words,
              const int32_t* __restrict__ cu, const int32_t* __restrict__ depth,
              const int32_t* __restrict__ order, const int32_t* __restrict__ pos,
              const uint64_t* __restrict__ anc, const int32_t* __restrict__ status,
              const int32_t* __restrict__ accept_node, const T* __restrict__ k,
              const float* __restrict__ Uws, const float* __restrict__ Gws, const float* S_in,
              float* S_out, int vec128) {
  extern __shared__ __align__(16) float csm[];
  const int DM1 = depth_max + 1;
  float* ck = csm;                          // [DM1][kCommitRows]  e^{G*-G_s} k_s[row]
  float* us = csm + DM1 * kCommitRows;      // [DM1][dv]           u_s
  __shared__ int s_path[TGDN_MAX_DEPTH + 1];
  __shared__ uint64_t s_mask[TGDN_MAX_NODES / 64];
  __shared__ int s_len;
  __shared__ int s_ok;

  const int rblocks = (dk + kCommitRows - 1) / kCommitRows;
  const int rb = blockIdx.x % rblocks;
  const int h = (blockIdx.x / rblocks) % H_v;
  const int bi = blockIdx.x / (rblocks * H_v);
  const int qh = h / (H_v / H_qk);
  const int r0 = rb * kCommitRows;
  const int nrows = min(kCommitRows, dk - r0);
  const int tid = threadIdx.x;
  const size_t sbase = ((size_t)bi * H_v + h) * dk * dv + (size_t)r0 * dv;

  // ---- state loads first (vector path: d_v = 128, all 64 rows present)
  const int cg = tid & 31, rg0 = tid >> 5;  // column group, first row group
  float4 acc[kCommitTiles][4];
  if (vec128) {
#pragma unroll
    for (int t = 0; t < kCommitTiles; ++t)
#pragma unroll
      for (int r = 0; r < 4; ++r)
        acc[t][r] = *reinterpret_cast<const float4*>(
            S_in + sbase + (size_t)((rg0 + 8 * t) * 4 + r) * dv + cg * 4);
  }

  // ---- the accepted path from tree prep's ancestor mask
  const int lo = cu[bi], N = cu[bi + 1] - lo;
  const int n = accept_node[bi];
  if (tid == 0) {
    s_ok = status[bi] == TGDN_SEQ_OK && n >= 0 && n < N;
    s_len = 0;
  }
  __syncthreads();
  int p = -1, dn = -1;
  if (s_ok) {
    p = pos[lo + n];
    dn = depth[lo + n];
    if (p < 0 || p >= N || dn < 0 || dn > depth_max) p = -1;
  }
  if (p >= 0 && tid < words) s_mask[tid] = anc[(size_t)(lo + p) * words + tid];
  __syncthreads();
  if (p >= 0 && tid < N) {
    const uint64_t w = s_mask[tid >> 6];
    if ((w >> (tid & 63)) & 1ull) {
      int rank = __popcll(w & ((1ull << (tid & 63)) - 1ull));
      for (int j = 0; j < (tid >> 6); ++j) rank += __popcll(s_mask[j]);
      if (rank <= dn) s_path[rank] = order[lo + tid];
      if (rank == dn) s_len = dn + 1;  // the deepest set bit is n* itself
    }
  }
  __syncthreads();
  const int L = s_len;

  if (L == 0) {  // nothing accepted: the state is kept
    if (S_out != S_in) {
      if (vec128) {
#pragma unroll
        for (int t = 0; t < kCommitTiles; ++t)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(S_out + sbase + (size_t)((rg0 + 8 * t) * 4 + r) * dv +
                                       cg * 4) = acc[t][r];
      } else {
        for (int e = tid; e < nrows * dv; e += kCommitThreads) S_out[sbase + e] = S_in[sbase + e];
      }
    }
    return;
  }
  const float Gstar = Gws[(size_t)(lo + n) * H_v + h];
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
  const float decay = __expf(Gstar);

  if (vec128) {
#pragma unroll
    for (int t = 0; t < kCommitTiles; ++t) {
      const int rg = rg0 + 8 * t;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        acc[t][r].x *= decay;
        acc[t][r].y *= decay;
        acc[t][r].z *= decay;
        acc[t][r].w *= decay;
      }
      for (int l = 0; l < L; ++l) {
        const float4 u = *reinterpret_cast<const float4*>(us + l * dv + cg * 4);
        const float4 kv = *reinterpret_cast<const float4*>(ck + l * kCommitRows + rg * 4);
        const float kr[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          acc[t][r].x = fmaf(kr[r], u.x, acc[t][r].x);
          acc[t][r].y = fmaf(kr[r], u.y, acc[t][r].y);
          acc[t][r].z = fmaf(kr[r], u.z, acc[t][r].z);
          acc[t][r].w = fmaf(kr[r], u.w, acc[t][r].w);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4*>(S_out + sbase + (size_t)(rg * 4 + r) * dv + cg * 4) =
            acc[t][r];
    }
  } else {
    for (int e = tid; e < nrows * dv; e += kCommitThreads) {
      const int i = e / dv, j = e % dv;
      float a = decay * S_in[sbase + e];
      for (int l = 0; l < L; ++l) a = fmaf(ck[l * kCommitRows + i], us[l * dv + j], a);
      S_out[sbase + e] = a;
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
  // vector path: 128 value columns, whole 64-row blocks, 16-byte aligned states
  const int vec128 = (d.d_v == 128) && (d.d_k % kCommitRows == 0) &&
                     (reinterpret_cast<uintptr_t>(S_in) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(S_out) % 16 == 0);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, kCommitThreads, smem, s>>>(
      d.H_qk, d.H_v, d.d_k, d.d_v, t.depth_max, t.words, t.cu_nodes, t.depth, t.order, t.pos,
      t.anc, t.status, accept_node, static_cast<const T*>(k), U, G, S_in, S_out, vec128);
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
