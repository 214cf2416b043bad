// verify_recurrent.cu — per-branch recurrent verification (the comparison point).
//
// "Trees from Marginals" (Experimentelle Ergebnisse) measures its fused tree
// kernel against per-branch recurrent verification: every branch of the tree
// is walked with the GDN recurrence from the committed state, token by token,
// as ordinary sequential decoding would, so shared prefixes are recomputed
// once per branch.  This kernel is that method, written as a reasonable GPU
// program: one CTA per (sequence, v-head, 32 value columns) keeps its
// 128 x 32 fp32 state slice in registers and, for every leaf, restarts from
// S0 and applies the GDN update eq.
//   S <- a (S - b k (k^T S)) + b k v^T,   o = S^T q
// along the leaf's root path, writing the output of every node it passes (a
// node on several branches is written with the same value each time).
// Same inputs and outputs as tgdn_verify (no workspace); bf16 or fp32 io.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kRecThreads = 128;   // 4 warps x 32 columns
constexpr int kRecCols = 32;       // value columns per CTA
constexpr int kRecRowsPerThread = 32;  // d_k = 128 rows split over the 4 warps

template <typename T>
__global__ void __launch_bounds__(kRecThreads)
verify_recurrent_kernel(int n_max, int depth_max, int H_qk, int H_v, int dk, int dv,
                        const int32_t* __restrict__ cu, const int32_t* __restrict__ parent,
                        const int32_t* __restrict__ depth, const int32_t* __restrict__ status,
                        const T* __restrict__ q, const T* __restrict__ k,
                        const T* __restrict__ v, const float* __restrict__ g,
                        const float* __restrict__ bta, const float* __restrict__ S0,
                        T* __restrict__ o) {
  __shared__ float s_k[TGDN_MAX_HEAD_DIM];
  __shared__ float s_q[TGDN_MAX_HEAD_DIM];
  __shared__ float s_part[2][4][kRecCols];
  __shared__ int s_path[TGDN_MAX_DEPTH + 1];
  __shared__ int s_is_parent[TGDN_MAX_NODES];
  __shared__ int s_len;

  const int nsl = (dv + kRecCols - 1) / kRecCols;
  const int c = blockIdx.x % nsl;
  const int h = (blockIdx.x / nsl) % H_v;
  const int bi = blockIdx.x / (nsl * H_v);
  const int qh = h / (H_v / H_qk);
  const int c0 = c * kRecCols;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = lane;                  // value column (within the slice)
  const bool jlive = c0 + j < dv;
  const int i0 = warp * kRecRowsPerThread;  // first key row of this thread
  const int lo = cu[bi], N = cu[bi + 1] - lo;
  const int st = status[bi];
  if (N <= 0 || st == TGDN_SEQ_BAD_RANGE) return;  // (a bad row range is never touched)
  const size_t orow_stride = (size_t)H_v * dv;
  T* obase = o + ((size_t)lo * H_v + h) * dv + c0;

  if (st != TGDN_SEQ_OK || N > n_max) {
    for (int e = tid; e < N * kRecCols; e += kRecThreads) {
      const int n = e / kRecCols, jj = e % kRecCols;
      if (c0 + jj < dv) Io<T>::store(obase + n * orow_stride + jj, 0.f);
    }
    return;
  }
  for (int n = tid; n < N; n += kRecThreads) s_is_parent[n] = 0;
  __syncthreads();
  for (int n = tid; n < N; n += kRecThreads) {
    const int p = parent[lo + n];
    if (p >= 0 && p < N) s_is_parent[p] = 1;
  }
  __syncthreads();

  const float* S0h = S0 + ((size_t)bi * H_v + h) * dk * dv + c0;
  float S[kRecRowsPerThread];
  for (int leaf = 0; leaf < N; ++leaf) {
    if (s_is_parent[leaf]) continue;  // only leaves start a branch
    if (tid == 0) {
      const int d = depth[lo + leaf];
      int len = 0;
      if (d >= 0 && d <= depth_max) {
        int n = leaf, dd = d;
        for (; dd >= 0 && n >= 0 && n < N; --dd) {
          s_path[dd] = n;
          n = parent[lo + n];
        }
        if (dd == -1 && n == -1) len = d + 1;
      }
      s_len = len;
    }
    __syncthreads();
    const int L = s_len;
#pragma unroll
    for (int r = 0; r < kRecRowsPerThread; ++r) {
      const int i = i0 + r;
      S[r] = (jlive && i < dk) ? __ldg(S0h + (size_t)i * dv + j) : 0.f;
    }
    for (int step = 0; step < L; ++step) {
      const int n = s_path[step];
      const size_t row = (size_t)(lo + n);
      for (int i = tid; i < dk; i += kRecThreads) {
        s_k[i] = Io<T>::load(k + (row * H_qk + qh) * dk + i);
        s_q[i] = Io<T>::load(q + (row * H_qk + qh) * dk + i);
      }
      const float a = __expf(g[row * H_v + h]);
      const float bb = bta[row * H_v + h];
      const float vj = jlive ? Io<T>::load(v + (row * H_v + h) * dv + c0 + j) : 0.f;
      __syncthreads();
      // w_j = sum_i k_i S_ij  (partial over this warp's rows, then across warps)
      float w = 0.f;
#pragma unroll
      for (int r = 0; r < kRecRowsPerThread; ++r)
        if (i0 + r < dk) w = fmaf(s_k[i0 + r], S[r], w);
      s_part[0][warp][j] = w;
      __syncthreads();
      w = s_part[0][0][j] + s_part[0][1][j] + s_part[0][2][j] + s_part[0][3][j];
      // S <- a (S - b k w^T) + b k v^T, then o_j = sum_i q_i S_ij
      float oj = 0.f;
#pragma unroll
      for (int r = 0; r < kRecRowsPerThread; ++r) {
        if (i0 + r < dk) {
          const float ki = s_k[i0 + r];
          S[r] = a * (S[r] - bb * ki * w) + bb * ki * vj;
          oj = fmaf(s_q[i0 + r], S[r], oj);
        }
      }
      s_part[1][warp][j] = oj;
      __syncthreads();
      if (warp == 0 && jlive)
        Io<T>::store(obase + n * orow_stride + j,
                     s_part[1][0][j] + s_part[1][1][j] + s_part[1][2][j] + s_part[1][3][j]);
    }
    __syncthreads();
  }
}

template <typename T>
static cudaError_t launch_rec_t(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                                const void* k, const void* v, const float* g, const float* b,
                                const float* S0, void* o, cudaStream_t s) {
  const int nsl = (d.d_v + kRecCols - 1) / kRecCols;
  const long grid = (long)t.B * d.H_v * nsl;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  verify_recurrent_kernel<T><<<(unsigned)grid, kRecThreads, 0, s>>>(
      t.n_max, t.depth_max, d.H_qk, d.H_v, d.d_k, d.d_v, t.cu_nodes, t.parent, t.depth, t.status,
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g, b, S0,
      static_cast<T*>(o));
  return cudaGetLastError();
}

cudaError_t launch_verify_recurrent(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                                    const void* k, const void* v, const float* g,
                                    const float* b, const float* S0, void* o, cudaStream_t s) {
  if (d.io == TGDN_BF16) return launch_rec_t<__nv_bfloat16>(t, d, q, k, v, g, b, S0, o, s);
  return launch_rec_t<float>(t, d, q, k, v, g, b, S0, o, s);
}

}  // namespace tgdn
