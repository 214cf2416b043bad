// commit.cu — deferred, rollback-free state commitment.
//
// "Trees from Marginals" (Technisches Resümee, Methodik 3, last bullet): the
// state is committed once the accepted branch is known, so nothing has to be
// rolled back.  The accepted node's state follows from the same factors U that
// verification produced: with n* the accepted node and P its root path,
//   S_new = e^{G_n*} S0 + sum_{s in P} e^{G_n* - G_s} k_s u_s^T,
// a rank-|P| update of the d_k x d_v fp32 state (|P| <= depth_max + 1).
//
// The state is streamed once (read S_in, write S_out; in place is allowed).
// Two kernels:
//   commit128_kernel (d_v = 128, d_k a multiple of 64, 16-byte aligned states):
//     one CTA of 128 threads per (sequence, v-head, 64 state rows).  The 32 KiB
//     block arrives by one bulk copy issued at entry, so it is in flight while
//     the accepted path is found (ancestor mask of n*, then the path nodes' u
//     rows and k values); each thread then updates a 16-row x 4-column tile and
//     writes it back with one coalesced 512-byte row per warp instruction.
//   commit_kernel (any other shape): one CTA of 256 threads per (sequence,
//     v-head, 64 state rows), element-wise.
// Both read the accepted path from the ancestor mask written by tree prep (one
// thread per candidate bit, no pointer chasing).
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

// ----------------------------------------------------------------- shared steps
// The accepted path of sequence bi: s_path[0..L-1] (root first) from the ancestor
// mask of n* (positions whose bit is set, ranked by position), L = depth(n*) + 1,
// or L = 0 when nothing is committed.  s_ord holds order[lo + q] for q < N.
// Called by every thread of the CTA (it contains barriers).
__device__ __forceinline__ int accepted_path(int nthreads, int tid, int N, int p, int dn,
                                             const uint64_t* s_mask, const int* s_ord,
                                             int* s_path, int* s_len) {
  if (tid == 0) *s_len = 0;
  __syncthreads();
  if (p >= 0) {
    for (int q = tid; q < N; q += nthreads) {
      const uint64_t w = s_mask[q >> 6];
      if ((w >> (q & 63)) & 1ull) {
        int rank = __popcll(w & ((1ull << (q & 63)) - 1ull));
        for (int j = 0; j < (q >> 6); ++j) rank += __popcll(s_mask[j]);
        if (rank <= dn) s_path[rank] = s_ord[q];
        if (rank == dn) *s_len = dn + 1;  // the deepest set bit is n* itself
      }
    }
  }
  __syncthreads();
  return *s_len;
}

// ----------------------------------------------------------------- any shape
constexpr int kCommitThreads = 256;
constexpr int kCommitRows = 64;  // state rows per CTA

template <typename T>
__global__ void __launch_bounds__(kCommitThreads)
commit_kernel(int H_qk, int H_v, int dk, int dv, int depth_max, int words,
              const int32_t* __restrict__ cu, const int32_t* __restrict__ depth,
              const int32_t* __restrict__ order, const int32_t* __restrict__ pos,
              const uint64_t* __restrict__ anc, const int32_t* __restrict__ status,
              const int32_t* __restrict__ accept_node, const T* __restrict__ k,
              const float* __restrict__ Uws, const float* __restrict__ Gws, const float* S_in,
              float* S_out) {
  extern __shared__ __align__(16) float csm[];
  const int DM1 = depth_max + 1;
  float* ck = csm;                          // [DM1][kCommitRows]  e^{G*-G_s} k_s[row]
  float* us = csm + DM1 * kCommitRows;      // [DM1][dv]           u_s
  __shared__ int s_path[TGDN_MAX_DEPTH + 1];
  __shared__ int s_ord[TGDN_MAX_NODES];
  __shared__ uint64_t s_mask[TGDN_MAX_NODES / 64];
  __shared__ int s_len;

  const int rblocks = (dk + kCommitRows - 1) / kCommitRows;
  const int rb = blockIdx.x % rblocks;
  const int h = (blockIdx.x / rblocks) % H_v;
  const int bi = blockIdx.x / (rblocks * H_v);
  const int qh = h / (H_v / H_qk);
  const int r0 = rb * kCommitRows;
  const int nrows = min(kCommitRows, dk - r0);
  const int tid = threadIdx.x;
  const size_t sbase = ((size_t)bi * H_v + h) * dk * dv + (size_t)r0 * dv;

  const int lo = cu[bi], N = cu[bi + 1] - lo;
  const int n = accept_node[bi];
  const bool ok = status[bi] == TGDN_SEQ_OK && n >= 0 && n < N;
  int p = -1, dn = -1;
  if (ok) {
    p = pos[lo + n];
    dn = depth[lo + n];
    if (p < 0 || p >= N || dn < 0 || dn > depth_max) p = -1;
  }
  if (ok)
    for (int q = tid; q < N; q += kCommitThreads) s_ord[q] = order[lo + q];
  if (p >= 0 && tid < words) s_mask[tid] = anc[(size_t)(lo + p) * words + tid];
  const int L = accepted_path(kCommitThreads, tid, N, p, dn, s_mask, s_ord, s_path, &s_len);

  if (L == 0) {  // nothing accepted: the state is kept
    if (S_out != S_in)
      for (int e = tid; e < nrows * dv; e += kCommitThreads) S_out[sbase + e] = S_in[sbase + e];
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
  for (int e = tid; e < nrows * dv; e += kCommitThreads) {
    const int i = e / dv, j = e % dv;
    float a = decay * S_in[sbase + e];
    for (int l = 0; l < L; ++l) a = fmaf(ck[l * kCommitRows + i], us[l * dv + j], a);
    S_out[sbase + e] = a;
  }
}

// ----------------------------------------------------------------- d_v = 128
constexpr int kC128Threads = 128;
constexpr int kC128Rows = 64;                       // state rows per CTA
constexpr uint32_t kC128Bytes = kC128Rows * 128 * 4;  // one state block, 32 KiB

template <typename T>
__global__ void __launch_bounds__(kC128Threads, 4)
commit128_kernel(int H_qk, int H_v, int dk, int depth_max, int n_max, int words,
                 const int32_t* __restrict__ cu, const int32_t* __restrict__ depth,
                 const int32_t* __restrict__ order, const int32_t* __restrict__ pos,
                 const uint64_t* __restrict__ anc, int32_t* __restrict__ status,
                 const int32_t* __restrict__ accept_node, const T* __restrict__ k,
                 const float* __restrict__ Uws, const float* __restrict__ Gws,
                 const float* S_in, float* S_out) {
  extern __shared__ __align__(128) float c128[];
  const int DM1 = depth_max + 1;
  float* st = c128;                       // [64][128] the state block (bulk copy)
  float* ck = st + kC128Rows * 128;       // [DM1][64]  e^{G*-G_s} k_s[row]
  float* us = ck + DM1 * kC128Rows;       // [DM1][128] u_s
  // sized by the launch's n_max (so that more CTAs fit an SM for small trees)
  uint64_t* s_anc = reinterpret_cast<uint64_t*>(us + DM1 * 128);  // [position][word]
  int* s_ord = reinterpret_cast<int*>(s_anc + (size_t)n_max * words);
  float* s_G = reinterpret_cast<float*>(s_ord + n_max);
  __shared__ uint64_t bar;
  __shared__ int s_path[TGDN_MAX_DEPTH + 1];
  __shared__ float s_c[TGDN_MAX_DEPTH + 1];
  __shared__ uint64_t s_mask[TGDN_MAX_NODES / 64];
  __shared__ int s_len;

  const int rblocks = dk / kC128Rows;
  const int rb = blockIdx.x % rblocks;
  const int h = (blockIdx.x / rblocks) % H_v;
  const int bi = blockIdx.x / (rblocks * H_v);
  const int qh = h / (H_v / H_qk);
  const int r0 = rb * kC128Rows;
  const int tid = threadIdx.x;
  const size_t sbase = ((size_t)bi * H_v + h) * dk * 128 + (size_t)r0 * 128;

  // the state block goes out first; it lands while the path is found
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, kC128Bytes);
    bulk_load(st, S_in + sbase, kC128Bytes, &bar);
  }
  // Dependent loads in two rounds before the path's factors: the sequence's bounds
  // and accepted node; then its position and depth together with the topological
  // order, every node's G and every position's ancestor mask (n*'s is picked after).
  const int lo = cu[bi], N = cu[bi + 1] - lo;
  const int n = accept_node[bi];
  const bool ok = status[bi] == TGDN_SEQ_OK && n >= 0 && n < N;
  int p = -1, dn = -1;
  if (ok) {
    p = pos[lo + n];
    dn = depth[lo + n];
    for (int q = tid; q < N; q += kC128Threads) {
      s_ord[q] = order[lo + q];
      s_G[q] = Gws[(size_t)(lo + q) * H_v + h];
    }
    for (int e = tid; e < N * words; e += kC128Threads) s_anc[e] = anc[(size_t)lo * words + e];
    if (p < 0 || p >= N || dn < 0 || dn > depth_max) p = -1;
  }
  __syncthreads();
  if (p >= 0 && tid < words) s_mask[tid] = s_anc[p * words + tid];
  const int L = accepted_path(kC128Threads, tid, N, p, dn, s_mask, s_ord, s_path, &s_len);

  float Gstar = 0.f;
  if (L > 0) {
    Gstar = s_G[n];
    if (tid < L) s_c[tid] = __expf(Gstar - s_G[s_path[tid]]);
    __syncthreads();
    // the path nodes' k values of these 64 rows (scaled) and u rows
    for (int e = tid; e < L * kC128Rows; e += kC128Threads) {
      const int l = e / kC128Rows, i = e % kC128Rows;
      ck[e] = s_c[l] * Io<T>::load(k + ((size_t)(lo + s_path[l]) * H_qk + qh) * dk + r0 + i);
    }
    for (int e = tid; e < L * 32; e += kC128Threads) {
      const int l = e >> 5, j4 = e & 31;
      reinterpret_cast<float4*>(us)[e] = reinterpret_cast<const float4*>(
          Uws + ((size_t)(lo + s_path[l]) * H_v + h) * 128)[j4];
    }
  }
  // the state block has landed (a bounded wait: past the limit the sequence is
  // reported as timed out and nothing is written)
  const bool landed = mbar_wait(&bar, 0);
  __syncthreads();
  if (!landed) {
    if (tid == 0) atomicCAS(&status[bi], TGDN_SEQ_OK, TGDN_SEQ_TIMEOUT);
    return;
  }
  if (L == 0 && S_out == S_in) return;  // nothing accepted: the state is kept

  // thread: columns 4 cg .. 4 cg + 3 of rows 16 rg .. 16 rg + 15; a warp reads and
  // writes whole 512-byte rows
  const int cg = tid & 31, rg = tid >> 5;
  const float decay = L > 0 ? __expf(Gstar) : 1.f;
  float4 acc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float4 x = reinterpret_cast<const float4*>(st + (rg * 16 + r) * 128)[cg];
    acc[r] = make_float4(decay * x.x, decay * x.y, decay * x.z, decay * x.w);
  }
  for (int l = 0; l < L; ++l) {
    const float4 u = reinterpret_cast<const float4*>(us + l * 128)[cg];
    const float4* kk = reinterpret_cast<const float4*>(ck + l * kC128Rows + rg * 16);
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
      const float4 kv = kk[r4];
      const float kr[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float4& a = acc[r4 * 4 + r];
        a.x = fmaf(kr[r], u.x, a.x);
        a.y = fmaf(kr[r], u.y, a.y);
        a.z = fmaf(kr[r], u.z, a.z);
        a.w = fmaf(kr[r], u.w, a.w);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 16; ++r)
    reinterpret_cast<float4*>(S_out + sbase + (size_t)(rg * 16 + r) * 128)[cg] = acc[r];
}

template <typename T>
static cudaError_t launch_commit_t(const tgdn_tree& t, const tgdn_dims& d,
                                   const int32_t* accept_node, const void* k, const float* U,
                                   const float* G, const float* S_in, float* S_out,
                                   cudaStream_t s) {
  // the bulk-copy kernel: 128 value columns, whole 64-row blocks, 16-byte aligned states
  const bool b128 = d.d_v == 128 && d.d_k % kC128Rows == 0 &&
                    reinterpret_cast<uintptr_t>(S_in) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(S_out) % 16 == 0;
  if (b128) {
    const long grid = (long)t.B * d.H_v * (d.d_k / kC128Rows);
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    const size_t smem = kC128Bytes + (size_t)(t.depth_max + 1) * (kC128Rows + 128) * sizeof(float) +
                        (size_t)t.n_max * t.words * sizeof(uint64_t) +
                        (size_t)t.n_max * (sizeof(int) + sizeof(float));
    const auto kern = commit128_kernel<T>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kC128Threads, smem, s>>>(
        d.H_qk, d.H_v, d.d_k, t.depth_max, t.n_max, t.words, t.cu_nodes, t.depth, t.order, t.pos,
        t.anc, t.status, accept_node, static_cast<const T*>(k), U, G, S_in, S_out);
    return cudaGetLastError();
  }
  const int rblocks = (d.d_k + kCommitRows - 1) / kCommitRows;
  const long grid = (long)t.B * d.H_v * rblocks;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)(t.depth_max + 1) * (kCommitRows + d.d_v) * sizeof(float);
  const auto kern = commit_kernel<T>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, kCommitThreads, smem, s>>>(
      d.H_qk, d.H_v, d.d_k, d.d_v, t.depth_max, t.words, t.cu_nodes, t.depth, t.order, t.pos,
      t.anc, t.status, accept_node, static_cast<const T*>(k), U, G, S_in, S_out);
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
