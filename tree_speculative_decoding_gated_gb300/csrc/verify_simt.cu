// verify_simt.cu — fp32 SIMT tree verification for any supported geometry.
//
// Implements the single-pass verification of "Trees from Marginals"
// (Technisches Resümee, Methodik 3 and Implementierung) with plain fp32 CUDA
// cores: path-cumulative log-gates G, the ancestor-masked Gram entries X and Y
// (only ancestor pairs are formed), the right-hand side
// R = diag(b)(V - diag(e^G) K S0), the level-by-level forward substitution of
// (I + X) U = R over the topological order, and the output phase
// O = diag(e^G) Q S0 + Y U.  One CTA per (sequence, v-head, 32 value columns):
// value columns are independent, only the Gram entries are shared.
//
// This is the exact-precision path (fp32 io, the 16x16 toy head) and the
// general path for shapes the tensor-core kernels do not take.  In complement
// mode (only_n > 0) it verifies just the valid sequences of only_n nodes whose
// root is not node 0: the ones the 128-node tensor-core kernel leaves to it.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kSimtThreads = 256;
constexpr int kSimtCols = 32;

struct SimtShape {
  int n_max, dm1, dk;
  // byte offsets in dynamic shared memory
  size_t s0, u, xs, ys, g, bb, gg, par, dep, ord, lvl, anc, total;
};

__host__ __device__ inline SimtShape simt_shape(int n_max, int depth_max, int dk) {
  SimtShape s;
  s.n_max = n_max;
  s.dm1 = depth_max + 1;
  s.dk = dk;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 15) / 16 * 16;
    return at;
  };
  s.s0 = take((size_t)dk * kSimtCols * 4);
  s.u = take((size_t)n_max * kSimtCols * 4);
  s.xs = take((size_t)n_max * s.dm1 * 4);
  s.ys = take((size_t)n_max * s.dm1 * 4);
  s.g = take((size_t)n_max * 4);
  s.bb = take((size_t)n_max * 4);
  s.gg = take((size_t)n_max * 4);
  s.par = take((size_t)n_max * 4);
  s.dep = take((size_t)n_max * 4);
  s.ord = take((size_t)n_max * 4);
  s.lvl = take((size_t)(s.dm1 + 1) * 4);
  s.anc = take((size_t)n_max * s.dm1);
  s.total = o;
  return s;
}

template <typename T>
__global__ void __launch_bounds__(kSimtThreads)
verify_simt_kernel(int n_max, int depth_max, int H_qk, int H_v, int dk, int dv,
                   const int32_t* __restrict__ cu, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ depth, const int32_t* __restrict__ order,
                   const int32_t* __restrict__ status, const T* __restrict__ q,
                   const T* __restrict__ k, const T* __restrict__ v,
                   const float* __restrict__ g, const float* __restrict__ bta,
                   const float* __restrict__ S0, T* __restrict__ o, float* __restrict__ Uws,
                   float* __restrict__ Gws, int only_n) {
  extern __shared__ __align__(16) uint8_t smem[];
  const SimtShape sh = simt_shape(n_max, depth_max, dk);
  float* S0s = reinterpret_cast<float*>(smem + sh.s0);
  float* U = reinterpret_cast<float*>(smem + sh.u);
  float* XS = reinterpret_cast<float*>(smem + sh.xs);
  float* YS = reinterpret_cast<float*>(smem + sh.ys);
  float* G = reinterpret_cast<float*>(smem + sh.g);
  float* bb = reinterpret_cast<float*>(smem + sh.bb);
  float* gg = reinterpret_cast<float*>(smem + sh.gg);
  int* par = reinterpret_cast<int*>(smem + sh.par);
  int* dep = reinterpret_cast<int*>(smem + sh.dep);
  int* ord = reinterpret_cast<int*>(smem + sh.ord);
  int* lvl = reinterpret_cast<int*>(smem + sh.lvl);
  uint8_t* anc_at = smem + sh.anc;
  const int DM1 = sh.dm1;

  const int nsl = (dv + kSimtCols - 1) / kSimtCols;
  const int tid = threadIdx.x;
  __shared__ int s_bad;
  // one (sequence, v-head, 32 value columns) item
  auto run = [&](const int item) {
    const int c = item % nsl;
    const int h = (item / nsl) % H_v;
    const int bi = item / (nsl * H_v);
    const int qh = h / (H_v / H_qk);
    const int c0 = c * kSimtCols;
    const int ncol = min(kSimtCols, dv - c0);
    const int lo = cu[bi], N = cu[bi + 1] - lo;
    const int st = status[bi];
    if (N <= 0 || st == TGDN_SEQ_BAD_RANGE) return;  // (a bad row range is never touched)
    if (tid == 0) s_bad = (st != TGDN_SEQ_OK) || (N > n_max);
    __syncthreads();

    auto orow = [&](int n) { return ((size_t)(lo + n) * H_v + h) * dv + c0; };
    auto zero_rows = [&]() {
      for (int it = tid; it < N * kSimtCols; it += kSimtThreads) {
        const int n = it / kSimtCols, j = it % kSimtCols;
        if (j >= ncol) continue;
        Io<T>::store(o + orow(n) + j, 0.f);
        Uws[orow(n) + j] = 0.f;
      }
      if (c == 0)
        for (int n = tid; n < N; n += kSimtThreads) Gws[(size_t)(lo + n) * H_v + h] = 0.f;
    };
    if (s_bad) {
      zero_rows();
      return;
    }

    // --- stage the tree, the gates and the S0 column slice (metadata that is
    // inconsistent with a prepared tree marks the sequence bad instead of
    // indexing out of bounds)
    for (int n = tid; n < N; n += kSimtThreads) {
      const int p = parent[lo + n], dd = depth[lo + n], od = order[lo + n];
      par[n] = p;
      dep[n] = dd;
      ord[n] = od;
      if (p < -1 || p >= N || dd < 0 || dd > depth_max || od < 0 || od >= N) s_bad = 1;
      gg[n] = g[(size_t)(lo + n) * H_v + h];
      bb[n] = bta[(size_t)(lo + n) * H_v + h];
    }
    const float* S0h = S0 + ((size_t)bi * H_v + h) * dk * dv;
    for (int it = tid; it < dk * kSimtCols; it += kSimtThreads) {
      const int i = it / kSimtCols, j = it % kSimtCols;
      S0s[it] = (j < ncol) ? __ldg(S0h + (size_t)i * dv + c0 + j) : 0.f;
    }
    __syncthreads();

    if (s_bad) {
      zero_rows();
      return;
    }
    // --- root paths (ancestor at each depth) and path-cumulative log-gates
    for (int n = tid; n < N; n += kSimtThreads) {
      int s = n;
      for (int d = dep[n]; d >= 0; --d) {
        if (s < 0) {
          s_bad = 1;
          break;
        }
        anc_at[n * DM1 + d] = static_cast<uint8_t>(s);
        s = par[s];
      }
      if (s != -1) {
        s_bad = 1;
        continue;
      }
      float acc = 0.f;
      for (int d = 0; d <= dep[n]; ++d) acc += gg[anc_at[n * DM1 + d]];
      G[n] = acc;
    }
    if (tid == 0) {
      int cur = 0;
      for (int p = 0; p < N; ++p) {
        const int d = dep[ord[p]];
        while (cur <= d) lvl[cur++] = p;
      }
      while (cur <= DM1) lvl[cur++] = N;
    }
    __syncthreads();
    if (s_bad) {
      zero_rows();
      return;
    }

    // --- ancestor-masked Gram entries: X (strict ancestors, x b_n) and Y (ancestors + self).
    // One warp per (node, ancestor) pair: the lanes split d_k, so the three rows are read
    // with coalesced loads, and a warp sum finishes each dot product.
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int it = warp; it < N * DM1; it += kSimtThreads / 32) {
        const int n = it / DM1, d = it % DM1;
        if (d > dep[n]) continue;
        const int s = anc_at[it];
        const T* kn = k + ((size_t)(lo + n) * H_qk + qh) * dk;
        const T* qn = q + ((size_t)(lo + n) * H_qk + qh) * dk;
        const T* ks = k + ((size_t)(lo + s) * H_qk + qh) * dk;
        float kk = 0.f, qk = 0.f;
        for (int i = lane; i < dk; i += 32) {
          const float kv = Io<T>::load(ks + i);
          kk = fmaf(Io<T>::load(kn + i), kv, kk);
          qk = fmaf(Io<T>::load(qn + i), kv, qk);
        }
  #pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          kk += __shfl_xor_sync(0xffffffffu, kk, off);
          qk += __shfl_xor_sync(0xffffffffu, qk, off);
        }
        if (lane == 0) {
          const float e = expf(G[n] - G[s]);
          YS[it] = e * qk;
          XS[it] = (d < dep[n]) ? bb[n] * e * kk : 0.f;
        }
      }
    }
    // --- right-hand side R = diag(b) (V - diag(e^G) K S0), stored in U
    for (int it = tid; it < N * kSimtCols; it += kSimtThreads) {
      const int n = it / kSimtCols, j = it % kSimtCols;
      const T* kn = k + ((size_t)(lo + n) * H_qk + qh) * dk;
      float ks = 0.f;
      for (int i = 0; i < dk; ++i) ks = fmaf(Io<T>::load(kn + i), S0s[i * kSimtCols + j], ks);
      const float vj = (j < ncol) ? Io<T>::load(v + orow(n) + j) : 0.f;
      U[it] = bb[n] * (vj - expf(G[n]) * ks);
    }
    __syncthreads();

    // --- forward substitution (I + X) U = R, one depth level at a time
    int maxdep = 0;
    while (maxdep + 1 < DM1 && lvl[maxdep + 1] < N) ++maxdep;
    for (int d = 1; d <= maxdep; ++d) {
      const int p0 = lvl[d], cnt = lvl[d + 1] - lvl[d];
      for (int it = tid; it < cnt * kSimtCols; it += kSimtThreads) {
        const int n = ord[p0 + it / kSimtCols], j = it % kSimtCols;
        float acc = U[n * kSimtCols + j];
        for (int dd = 0; dd < d; ++dd)
          acc = fmaf(-XS[n * DM1 + dd], U[anc_at[n * DM1 + dd] * kSimtCols + j], acc);
        U[n * kSimtCols + j] = acc;
      }
      __syncthreads();
    }

    // --- output phase O = diag(e^G) Q S0 + Y U, and the workspace rows
    for (int it = tid; it < N * kSimtCols; it += kSimtThreads) {
      const int n = it / kSimtCols, j = it % kSimtCols;
      if (j >= ncol) continue;
      const T* qn = q + ((size_t)(lo + n) * H_qk + qh) * dk;
      float qs = 0.f;
      for (int i = 0; i < dk; ++i) qs = fmaf(Io<T>::load(qn + i), S0s[i * kSimtCols + j], qs);
      float acc = expf(G[n]) * qs;
      for (int dd = 0; dd <= dep[n]; ++dd)
        acc = fmaf(YS[n * DM1 + dd], U[anc_at[n * DM1 + dd] * kSimtCols + j], acc);
      Io<T>::store(o + orow(n) + j, acc);
      Uws[orow(n) + j] = U[it];
    }
    if (c == 0)
      for (int n = tid; n < N; n += kSimtThreads) Gws[(size_t)(lo + n) * H_v + h] = G[n];
  };
  if (only_n > 0) {
    // complement mode: one CTA per (sequence, v-head).  It leaves at once unless
    // its sequence is one the 128-node kernel leaves (only_n nodes, valid, root not
    // node 0), and then verifies the column slices in turn; so a batch with no such
    // sequence costs one short wave instead of a CTA per column slice.
    const int bi = blockIdx.x / H_v;
    const int lo = cu[bi], N = cu[bi + 1] - lo;
    if (!(N == only_n && status[bi] == TGDN_SEQ_OK && depth[lo] != 0)) return;
    for (int c = 0; c < nsl; ++c) {
      if (c > 0) __syncthreads();  // the previous slice is done with shared memory
      run(blockIdx.x * nsl + c);
    }
  } else {
    run(blockIdx.x);
  }
}

template <typename T>
static cudaError_t launch_simt_t(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                                 const void* k, const void* v, const float* g, const float* b,
                                 const float* S0, void* o, float* U, float* G, int only_n,
                                 cudaStream_t s) {
  const SimtShape sh = simt_shape(t.n_max, t.depth_max, d.d_k);
  const auto kern = verify_simt_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sh.total);
  if (e != cudaSuccess) return e;
  const int nsl = (d.d_v + kSimtCols - 1) / kSimtCols;
  const long grid = (long)t.B * d.H_v * (only_n > 0 ? 1 : nsl);
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)grid, kSimtThreads, sh.total, s>>>(
      t.n_max, t.depth_max, d.H_qk, d.H_v, d.d_k, d.d_v, t.cu_nodes, t.parent, t.depth, t.order,
      t.status, static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g,
      b, S0, static_cast<T*>(o), U, G, only_n);
  return cudaGetLastError();
}

cudaError_t launch_verify_simt(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                               const void* k, const void* v, const float* g, const float* b,
                               const float* S0, void* o, float* U, float* G, cudaStream_t s,
                               int only_n) {
  if (d.io == TGDN_BF16)
    return launch_simt_t<__nv_bfloat16>(t, d, q, k, v, g, b, S0, o, U, G, only_n, s);
  return launch_simt_t<float>(t, d, q, k, v, g, b, S0, o, U, G, only_n, s);
}

}  // namespace tgdn
