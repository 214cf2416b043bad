// verify_tc.cu — tensor-core tree verification (bf16 io, d_k = d_v = 128, sm_103a).
//
// Single-pass verification of a draft tree through one GDN layer, following
// "Trees from Marginals" (Technisches Resümee, Methodik 3 and Implementierung:
// Gram matrix, forward substitution and output phase in one kernel).  With G
// the path-cumulative log-gate and A(n) / A*(n) the strict / inclusive
// ancestors of n,
//   X_ns = b_n e^{G_n-G_s} k_n.k_s  (s in A(n)),  Y_ns = e^{G_n-G_s} q_n.k_s  (s in A*(n))
//   (I + X) U = R = diag(b) (V - diag(e^G) K S0),   O = diag(e^G) Q S0 + Y U.
// Because X only links a node to its own ancestors, T = (I + X)^{-1} and
// W = Y T keep that sparsity, and row n of either depends only on the root
// path of n: it is the solution of a (depth+1)-sized unit triangular system.
// So U = T R and O = diag(e^G) Q S0 + W R.
//
// One CTA per (sequence, v-head, 64 value columns); 128 threads; the tree has
// at most 64 nodes and depth at most 30.
//   1. TMA brings the key and query rows of the CTA's q/k head into shared
//      memory as one 128 x 128 bf16 operand A = [K; Q] (128-byte swizzle).
//      All threads stream the fp32 state slice S0[:, c0:c0+64] from HBM and
//      split it into bf16 hi + lo operands (products keep ~16 mantissa bits).
//   2. tcgen05.mma into TMEM (fp32):  D[:, 0:64] = A S0_hi + A S0_lo,
//      D[:, 64:128] = A K^T.  Lane n < 64 holds k_n S0 and k_n.K; lane 64 + n
//      holds q_n S0 and q_n.K.
//   3. Every lane writes its Gram row to shared memory; key lanes form
//      R = diag(b)(V - e^G K S0) as a bf16 hi + lo operand.
//   4. Thread of key lane n solves its root path's system for row n of T,
//      thread of query lane n for row n of W (back substitution over at most
//      depth + 1 entries); the rows become a 128 x 64 bf16 hi + lo operand
//      [T; W] (zero off the path).
//   5. tcgen05.mma: D[:, 64:128] = [T; W] R (three bf16 products for hi/lo).
//      Key lanes read U rows, query lanes read W R and add e^G Q S0.  U and G
//      go to the workspace for tgdn_commit; O is stored as bf16.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kTcThreads = 128;
constexpr int kTcNodes = 64;   // nodes per tree on this kernel
constexpr int kTcDK = 128;
constexpr int kTcDV = 128;
constexpr int kTcCols = 64;    // value columns per CTA
constexpr int kTcDepth = 30;   // depth bound on this kernel
constexpr int kTcPath = kTcDepth + 1;  // entries of a root path (odd: conflict-free stride)
constexpr uint32_t kTmemCols = 128;

// Shared-memory map (bytes from a 1024-byte aligned base).  Operands of the
// first product are dead once it completes and their space is reused.
constexpr int kOffA = 0;        // [K;Q] operand: [2 d_k halves][128 rows][128 B]
constexpr int kOffS0hi = 32768; // S0 operand, MN-major: [16 k-groups][8 rows][128 B]
constexpr int kOffS0lo = 49152;
constexpr int kOffGR = 0;       // after product 1: Gram rows, [128 lanes][64] fp32
constexpr int kOffRhi = 32768;  // R operand, MN-major: [8 node groups][8 rows][128 B]
constexpr int kOffRlo = 40960;
constexpr int kOffRS = 49152;   // per-thread path solutions, [128][kTcPath] fp32
constexpr int kOffA2hi = 0;     // after the path solves: [T; W] operand, K-major
constexpr int kOffA2lo = 16384;
constexpr int kOperandBytes = 65536;
static_assert(kOffRS + kTcThreads * kTcPath * 4 <= kOperandBytes, "path scratch fits");

struct TcMeta {
  uint64_t tma_bar;
  uint64_t mma_bar;
  uint32_t tmem_slot;
  int bad;
  int tma_ok;
  int mma_issued;
  int dep[kTcNodes];
  int pos[kTcNodes];
  int ord[kTcNodes];
  float G[kTcNodes];
  float bb[kTcNodes];
  float gg[kTcNodes];
  uint8_t anc_at[kTcNodes][kTcPath + 1];
};
constexpr int kOffMeta = kOperandBytes;
constexpr int kTcSmemBytes = kOffMeta + (int)sizeof(TcMeta) + 1024;  // + alignment slack

// 16-byte chunk swizzle used by every 128-byte-row operand (matches the TMA
// and tcgen05 SWIZZLE_128B layout for 1024-byte aligned 8-row atoms).
__device__ __forceinline__ int swz(int row, int chunk) { return chunk ^ (row & 7); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// x ~= hi + lo with hi = bf16(x), lo = bf16(x - hi), for 8 consecutive values.
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  float h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
  hi = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                  pack_bf16x2(h[6], h[7]));
  lo = make_uint4(pack_bf16x2(x[0] - h[0], x[1] - h[1]), pack_bf16x2(x[2] - h[2], x[3] - h[3]),
                  pack_bf16x2(x[4] - h[4], x[5] - h[5]), pack_bf16x2(x[6] - h[6], x[7] - h[7]));
}

// Byte offset of 16-byte chunk `chunk` of 128-byte row `row` in an operand made
// of 1024-byte, 8-row swizzle atoms stacked along the row index.
__device__ __forceinline__ int atom_off(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + (swz(row, chunk) << 4);
}

__global__ void __launch_bounds__(kTcThreads)
verify_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 int H_qk, int H_v, int depth_max, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ depth, const int32_t* __restrict__ order,
                 const int32_t* __restrict__ pos, const uint64_t* __restrict__ anc,
                 int32_t* __restrict__ status, const __nv_bfloat16* __restrict__ v,
                 const float* __restrict__ g, const float* __restrict__ bta,
                 const float* __restrict__ S0, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ Uws, float* __restrict__ Gws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcMeta& m = *reinterpret_cast<TcMeta*>(smem + kOffMeta);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int nsl = kTcDV / kTcCols;
  const int c = blockIdx.x % nsl;
  const int h = (blockIdx.x / nsl) % H_v;
  const int bi = blockIdx.x / (nsl * H_v);
  const int qh = h / (H_v / H_qk);
  const int c0 = c * kTcCols;
  const int lo = cu[bi], N = cu[bi + 1] - lo;
  if (N <= 0) return;

  auto zero_rows = [&]() {
    for (int it = tid; it < N * (kTcCols / 4); it += kTcThreads) {
      const int n = it >> 4, ch = it & 15;
      const size_t row = ((size_t)(lo + n) * H_v + h) * kTcDV + c0 + ch * 4;
      *reinterpret_cast<uint2*>(o + row) = make_uint2(0u, 0u);
      *reinterpret_cast<float4*>(Uws + row) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (c == 0)
      for (int n = tid; n < N; n += kTcThreads) Gws[(size_t)(lo + n) * H_v + h] = 0.f;
  };

  if (tid == 0) m.bad = (status[bi] != TGDN_SEQ_OK) || (N > kTcNodes);
  __syncthreads();
  if (m.bad) {  // nothing issued yet: no copies in flight, no TMEM held
    zero_rows();
    return;
  }

  // ---- 1. operand staging
  if (tid == 0) {
    mbar_init(&m.tma_bar, 1);
    mbar_init(&m.mma_bar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&qmap);
    mbar_arrive_expect_tx(&m.tma_bar, 4 * 64 * 128);
    // box = 64 d_k elements x 1 head x 64 node rows, 128-byte swizzled rows
    tma_load_3d(smem + kOffA + 0, &kmap, &m.tma_bar, 0, qh, lo);
    tma_load_3d(smem + kOffA + 8192, &qmap, &m.tma_bar, 0, qh, lo);
    tma_load_3d(smem + kOffA + 16384, &kmap, &m.tma_bar, 64, qh, lo);
    tma_load_3d(smem + kOffA + 24576, &qmap, &m.tma_bar, 64, qh, lo);
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(&m.tmem_slot, kTmemCols);

  const float* s0src = S0 + ((size_t)bi * H_v + h) * kTcDK * kTcDV + c0;
  const int r0 = tid >> 4, q4 = tid & 15;  // 8 state rows x 16 float4 per pass
  float4 sbuf[16];
#pragma unroll
  for (int p = 0; p < 16; ++p)
    sbuf[p] = __ldg(reinterpret_cast<const float4*>(s0src + (size_t)(r0 + 8 * p) * kTcDV) + q4);

  uint64_t my_anc = 0;
  if (tid < N) {
    const int dd = depth[lo + tid], ps = pos[lo + tid], od = order[lo + tid];
    m.dep[tid] = dd;
    m.pos[tid] = ps;
    m.ord[tid] = od;
    if (dd < 0 || dd > depth_max || dd > kTcDepth || ps < 0 || ps >= N || od < 0 || od >= N)
      m.bad = 1;
    else
      my_anc = anc[lo + ps];  // one 64-bit word: n_max <= 64
    m.gg[tid] = g[(size_t)(lo + tid) * H_v + h];
    m.bb[tid] = bta[(size_t)(lo + tid) * H_v + h];
  }

#pragma unroll
  for (int p = 0; p < 16; ++p) {  // S0 -> bf16 hi/lo, MN-major (row = d_k index)
    const int kr = r0 + 8 * p;
    const float4 x = sbuf[p];
    const float h0 = __bfloat162float(__float2bfloat16_rn(x.x));
    const float h1 = __bfloat162float(__float2bfloat16_rn(x.y));
    const float h2 = __bfloat162float(__float2bfloat16_rn(x.z));
    const float h3 = __bfloat162float(__float2bfloat16_rn(x.w));
    const int off = atom_off(kr, q4 >> 1) + (q4 & 1) * 8;
    *reinterpret_cast<uint2*>(smem + kOffS0hi + off) =
        make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
    *reinterpret_cast<uint2*>(smem + kOffS0lo + off) =
        make_uint2(pack_bf16x2(x.x - h0, x.y - h1), pack_bf16x2(x.z - h2, x.w - h3));
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = m.tmem_slot;

  // ---- root path of every node from its ancestor mask (bits = topological
  // positions, ascending = root first) and its path-cumulative log-gate
  if (tid < N && !m.bad) {
    const int dn = m.dep[tid];
    uint64_t mk = my_anc;
    bool ok = __popcll(mk) == dn + 1 && ((mk >> m.pos[tid]) & 1ull);
    float acc = 0.f;
    for (int i = 0; ok && i <= dn; ++i) {
      const int b = __ffsll(static_cast<long long>(mk)) - 1;
      mk &= mk - 1;
      if (b >= N) {
        ok = false;
        break;
      }
      const int s = m.ord[b];
      ok = m.dep[s] == i;
      m.anc_at[tid][i] = static_cast<uint8_t>(s);
      acc += m.gg[s];
    }
    if (!ok || m.anc_at[tid][dn] != tid) m.bad = 1;
    m.G[tid] = acc;
  }
  __syncthreads();

  // ---- 2. first product (one thread).  The key/query copies are always
  // waited for, so no copy is left in flight on any exit path.
  if (tid == 0) {
    m.tma_ok = mbar_wait(&m.tma_bar, 0);
    m.mma_issued = 0;
    if (m.tma_ok && !m.bad) {
      tc_fence_after_sync();
      const uint32_t sA = smem_addr(smem + kOffA);
      const uint32_t sHi = smem_addr(smem + kOffS0hi);
      const uint32_t sLo = smem_addr(smem + kOffS0lo);
      constexpr uint32_t id_s0 = idesc_bf16_f32(128, kTcCols, 0, 1);
      constexpr uint32_t id_gram = idesc_bf16_f32(128, kTcNodes, 0, 0);
#pragma unroll
      for (int s = 0; s < kTcDK / 16; ++s) {
        const uint32_t a_off = (s >> 2) * 16384 + (s & 3) * 32;
        const uint64_t ad = smem_desc(sA + a_off, 16, 1024, kSwizzle128B);
        const uint64_t hd = smem_desc(sHi + s * 2048, 1024, 1024, kSwizzle128B);
        const uint64_t ld = smem_desc(sLo + s * 2048, 1024, 1024, kSwizzle128B);
        umma_bf16(tmem, ad, hd, id_s0, s > 0);
        umma_bf16(tmem, ad, ld, id_s0, 1);
        umma_bf16(tmem + kTcCols, ad, ad, id_gram, s > 0);  // B = the key rows of A
      }
      umma_commit(&m.mma_bar);
      m.mma_issued = 1;
    }
  }
  __syncthreads();
  bool mma_ok = false;
  if (m.mma_issued) mma_ok = !__syncthreads_or(!mbar_wait(&m.mma_bar, 0));
  tc_fence_after_sync();

  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const bool key_row = warp < 2;
  const int n = key_row ? tid : tid - 64;  // this thread's node
  const bool live = n < N;

  // ---- 3. Gram rows to shared memory; R = diag(b)(V - e^G K S0) as bf16 hi/lo
  if (mma_ok) {
    float* GR = reinterpret_cast<float*>(smem + kOffGR);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float r[32];
      tmem_ld32(tmem + lane_base + kTcCols + half * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<float4*>(GR + tid * 64 + swz(tid, half * 8 + ch) * 4) =
            make_float4(r[ch * 4], r[ch * 4 + 1], r[ch * 4 + 2], r[ch * 4 + 3]);
    }
    if (key_row) {
      const float eG = live ? __expf(m.G[n]) : 0.f;
      const float bn = live ? m.bb[n] : 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 vv[4] = {};
        if (live) {
          const uint4* vp = reinterpret_cast<const uint4*>(
              v + ((size_t)(lo + n) * H_v + h) * kTcDV + c0 + half * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) vv[i] = __ldg(vp + i);
        }
        float r[32];
        tmem_ld32(tmem + lane_base + half * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {  // 8 columns per 16-byte bf16 chunk
          const __nv_bfloat162* vb = reinterpret_cast<const __nv_bfloat162*>(&vv[ch]);
          float x[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 vf = __bfloat1622float2(vb[i]);
            x[2 * i] = live ? bn * (vf.x - eG * r[ch * 8 + 2 * i]) : 0.f;
            x[2 * i + 1] = live ? bn * (vf.y - eG * r[ch * 8 + 2 * i + 1]) : 0.f;
          }
          uint4 hi, lw;
          split8(x, hi, lw);  // rows of R beyond the tree are exact zeros
          const int off = atom_off(n, half * 4 + ch);
          *reinterpret_cast<uint4*>(smem + kOffRhi + off) = hi;
          *reinterpret_cast<uint4*>(smem + kOffRlo + off) = lw;
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();

  // ---- 4. one row of T (key lanes) or W (query lanes) per thread, by back
  // substitution on the root path P = (p_0 = root, ..., p_d = n):
  //   r (I + X_P) = y,  X_P[i][j] = b_{p_i} e^{G_{p_i} - G_{p_j}} k_{p_i}.k_{p_j} (i > j),
  //   y = e_d for T;  y_j = e^{G_n - G_{p_j}} q_n.k_{p_j} for W.
  // Every exponent is <= 0 (G only decreases down a path), so nothing overflows.
  float* RS = reinterpret_cast<float*>(smem + kOffRS) + tid * kTcPath;
  const uint8_t* P = m.anc_at[live ? n : 0];
  const int dn = (mma_ok && live) ? m.dep[n] : -1;
  if (dn >= 0) {
    const float* GR = reinterpret_cast<const float*>(smem + kOffGR);
    const float Gn = m.G[n];
    for (int j = dn; j >= 0; --j) {
      const int pj = P[j];
      const float Gj = m.G[pj];
      const int cj = pj >> 2, wj = pj & 3;
      float y;
      if (key_row)
        y = (j == dn) ? 1.f : 0.f;
      else
        y = __expf(Gn - Gj) * GR[tid * 64 + swz(tid, cj) * 4 + wj];
      float acc = 0.f;
      for (int i = j + 1; i <= dn; ++i) {
        const int pi = P[i];
        const float x = m.bb[pi] * __expf(m.G[pi] - Gj) * GR[pi * 64 + swz(pi, cj) * 4 + wj];
        acc = fmaf(RS[i], x, acc);
      }
      RS[j] = y - acc;
    }
  }
  __syncthreads();  // the Gram rows are no longer read: their space becomes [T; W]

  // [T; W] row `tid` as a bf16 hi/lo K-major operand: zero, then the path entries
  {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      *reinterpret_cast<uint4*>(smem + kOffA2hi + atom_off(tid, ch)) = zero;
      *reinterpret_cast<uint4*>(smem + kOffA2lo + atom_off(tid, ch)) = zero;
    }
    for (int j = 0; j <= dn; ++j) {
      const int t = P[j];
      const float r = RS[j];
      const __nv_bfloat16 hi = __float2bfloat16_rn(r);
      const __nv_bfloat16 lw = __float2bfloat16_rn(r - __bfloat162float(hi));
      const int off = atom_off(tid, t >> 3) + (t & 7) * 2;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2hi + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2lo + off) = lw;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  // ---- 5. second product: D[:, 64:128] = [T; W] R  (hi.hi + hi.lo + lo.hi)
  if (tid == 0 && mma_ok) {
    const uint32_t sA2hi = smem_addr(smem + kOffA2hi);
    const uint32_t sA2lo = smem_addr(smem + kOffA2lo);
    const uint32_t sRhi = smem_addr(smem + kOffRhi);
    const uint32_t sRlo = smem_addr(smem + kOffRlo);
    constexpr uint32_t id_r = idesc_bf16_f32(128, kTcCols, 0, 1);
#pragma unroll
    for (int s = 0; s < kTcNodes / 16; ++s) {
      const uint64_t ah = smem_desc(sA2hi + s * 32, 16, 1024, kSwizzle128B);
      const uint64_t al = smem_desc(sA2lo + s * 32, 16, 1024, kSwizzle128B);
      const uint64_t bh = smem_desc(sRhi + s * 2048, 1024, 1024, kSwizzle128B);
      const uint64_t bl = smem_desc(sRlo + s * 2048, 1024, 1024, kSwizzle128B);
      umma_bf16(tmem + kTcCols, ah, bh, id_r, s > 0);
      umma_bf16(tmem + kTcCols, ah, bl, id_r, 1);
      umma_bf16(tmem + kTcCols, al, bh, id_r, 1);
    }
    umma_commit(&m.mma_bar);
  }
  bool mma2_ok = false;
  if (mma_ok) mma2_ok = !__syncthreads_or(!mbar_wait(&m.mma_bar, 1));
  tc_fence_after_sync();

  // ---- 6. key lanes: U rows to the workspace; query lanes: O = e^G Q S0 + W R
  if (mma2_ok) {
    if (key_row) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float r[32];
        tmem_ld32(tmem + lane_base + kTcCols + half * 32, r);
        tmem_ld_wait();
        if (live) {
          float4* dst = reinterpret_cast<float4*>(
              Uws + ((size_t)(lo + n) * H_v + h) * kTcDV + c0 + half * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
        }
      }
      if (live && c == 0) Gws[(size_t)(lo + n) * H_v + h] = m.G[n];
    } else {
      const float eG = live ? __expf(m.G[n]) : 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float a[32], w[32];
        tmem_ld32(tmem + lane_base + half * 32, a);
        tmem_ld32(tmem + lane_base + kTcCols + half * 32, w);
        tmem_ld_wait();
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(
              o + ((size_t)(lo + n) * H_v + h) * kTcDV + c0 + half * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* aa = a + 8 * i;
            const float* ww = w + 8 * i;
            dst[i] = make_uint4(pack_bf16x2(fmaf(eG, aa[0], ww[0]), fmaf(eG, aa[1], ww[1])),
                                pack_bf16x2(fmaf(eG, aa[2], ww[2]), fmaf(eG, aa[3], ww[3])),
                                pack_bf16x2(fmaf(eG, aa[4], ww[4]), fmaf(eG, aa[5], ww[5])),
                                pack_bf16x2(fmaf(eG, aa[6], ww[6]), fmaf(eG, aa[7], ww[7])));
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (!mma2_ok) {
    if (m.bad) {
      zero_rows();
    } else if (tid == 0) {  // a bounded wait expired: report it, leave the outputs alone
      status[bi] = TGDN_SEQ_TIMEOUT;
    }
  }
}

bool verify_tc_supported(const tgdn_tree& t, const tgdn_dims& d, const void* q, const void* k,
                         const void* v, const float* S0, const void* o) {
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
  return d.io == TGDN_BF16 && d.d_k == kTcDK && d.d_v == kTcDV && t.n_max <= kTcNodes &&
         t.depth_max <= kTcDepth && al(q, 16) && al(k, 16) && al(v, 16) && al(S0, 16) &&
         al(o, 16);
}

cudaError_t launch_verify_tc(const tgdn_tree& t, const tgdn_dims& d, const CUtensorMap& qmap,
                             const CUtensorMap& kmap, const void* v, const float* g,
                             const float* b, const float* S0, void* o, float* U, float* G,
                             cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (e != cudaSuccess) return e;
  const long grid = (long)t.B * d.H_v * (kTcDV / kTcCols);
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  verify_tc_kernel<<<(unsigned)grid, kTcThreads, kTcSmemBytes, s>>>(
      qmap, kmap, d.H_qk, d.H_v, t.depth_max, t.cu_nodes, t.depth, t.order, t.pos, t.anc,
      t.status, static_cast<const __nv_bfloat16*>(v), g, b, S0, static_cast<__nv_bfloat16*>(o),
      U, G);
  return cudaGetLastError();
}

}  // namespace tgdn
