// verify_tc.cu — tensor-core tree verification (bf16 io, d_k = d_v = 128, sm_103a).
//
// Single-pass verification of a draft tree through one GDN layer, following
// "Trees from Marginals" (Technisches Resümee, Methodik 3 and Implementierung:
// Gram matrix, tiled forward substitution and output phase in one kernel).
// With G the path-cumulative log-gate,
//   X_ns = b_n e^{G_n-G_s} k_n.k_s  (s strict ancestor of n)
//   Y_ns =     e^{G_n-G_s} q_n.k_s  (s ancestor of n or n itself)
//   (I + X) U = diag(b) (V - diag(e^G) K S0),   O = diag(e^G) Q S0 + Y U.
//
// One CTA per (sequence, v-head, 64 value columns); 128 threads.
//   1. TMA brings the tree's key and query rows of the CTA's q/k head into
//      shared memory as one 128 x 128 bf16 operand A = [K; Q] (rows 0-63 keys,
//      64-127 queries, 128-byte swizzle).  Meanwhile all threads stream the
//      fp32 state slice S0[:, c0:c0+64] from HBM and split it into two bf16
//      operands hi + lo (hi = bf16(S0), lo = bf16(S0 - hi)), so the products
//      with S0 keep about 16 mantissa bits.
//   2. One thread issues tcgen05.mma into TMEM (fp32 accumulators):
//        D[:,  0: 64] = A . S0_hi + A . S0_lo   (K S0 rows and Q S0 rows)
//        D[:, 64:128] = A . K^T                 (K K^T rows and Q K^T rows)
//   3. Each thread reads its TMEM lane (one node's key or query row) and forms
//      R = diag(b)(V - e^G K S0), e^G Q S0 and the ancestor-masked, gated
//      X and Y entries; the operand buffers are dead by then and are reused.
//   4. Forward substitution of (I + X) U = R one depth level at a time (nodes
//      of one depth never depend on each other), then the output phase.  U and
//      G go to the workspace for tgdn_commit.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kTcThreads = 128;
constexpr int kTcNodes = 64;   // nodes per tree on this kernel
constexpr int kTcDK = 128;
constexpr int kTcDV = 128;
constexpr int kTcCols = 64;    // value columns per CTA
constexpr int kTcDepth = 32;   // depth bound on this kernel
constexpr int kTcDM1 = kTcDepth + 1;
constexpr uint32_t kTmemCols = 128;

// Shared-memory map (bytes from a 1024-byte aligned base).
constexpr int kOffA = 0;           // [2 d_k halves][128 rows][128 B], swizzled
constexpr int kOffBhi = 32768;     // [16 k-groups][8 rows][128 B], swizzled, MN-major
constexpr int kOffBlo = 49152;
constexpr int kOperandBytes = 65536;
// after the MMAs complete the operand area is reused:
constexpr int kOffU = 0;           // [64 nodes][16 chunks x 16 B] fp32, chunk ^= row & 7
constexpr int kOffEQ = 16384;      // e^G Q S0 rows, same layout
constexpr int kOffXS = 32768;      // [64][33] fp32
constexpr int kOffYS = kOffXS + kTcNodes * kTcDM1 * 4;
static_assert(kOffYS + kTcNodes * kTcDM1 * 4 <= kOperandBytes, "scratch fits the operands");
// persistent metadata
constexpr int kOffMeta = kOperandBytes;
struct TcMeta {
  uint64_t tma_bar;
  uint64_t mma_bar;
  uint64_t strict[kTcNodes];   // strict-ancestor mask by local index
  uint32_t tmem_slot;
  int bad;
  int tma_ok;
  int mma_issued;
  int par[kTcNodes];
  int dep[kTcNodes];
  int ord[kTcNodes];
  int lvl[kTcDM1 + 1];
  float G[kTcNodes];
  float bb[kTcNodes];
  float gg[kTcNodes];
  uint8_t anc_at[kTcNodes][kTcDM1];
};
constexpr int kTcSmemBytes = kOffMeta + (int)sizeof(TcMeta) + 1024;  // + alignment slack

__device__ __forceinline__ int swz(int row, int chunk) { return chunk ^ (row & 7); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

__global__ void __launch_bounds__(kTcThreads)
verify_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 int H_qk, int H_v, int depth_max, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ parent, const int32_t* __restrict__ depth,
                 const int32_t* __restrict__ order, int32_t* __restrict__ status,
                 const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
                 const float* __restrict__ bta, const float* __restrict__ S0,
                 __nv_bfloat16* __restrict__ o, float* __restrict__ Uws,
                 float* __restrict__ Gws) {
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

  // ---- 1. operand staging: TMA for [K; Q], register path for S0 hi/lo
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

  for (int n = tid; n < N; n += kTcThreads) {
    const int p = parent[lo + n], dd = depth[lo + n], od = order[lo + n];
    m.par[n] = p;
    m.dep[n] = dd;
    m.ord[n] = od;
    if (p < -1 || p >= N || dd < 0 || dd > depth_max || dd > kTcDepth || od < 0 || od >= N)
      m.bad = 1;
    m.gg[n] = g[(size_t)(lo + n) * H_v + h];
    m.bb[n] = bta[(size_t)(lo + n) * H_v + h];
  }

  {  // S0[:, c0:c0+64] -> bf16 hi/lo, MN-major with 128-byte swizzle
    const float* src = S0 + ((size_t)bi * H_v + h) * kTcDK * kTcDV + c0;
    const int r0 = tid >> 4, q4 = tid & 15;  // 8 rows x 16 float4 per pass
    float4 buf[16];
#pragma unroll
    for (int p = 0; p < 16; ++p)
      buf[p] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(r0 + 8 * p) * kTcDV) + q4);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const int kr = r0 + 8 * p;  // d_k row
      const float4 x = buf[p];
      const float h0 = __bfloat162float(__float2bfloat16_rn(x.x));
      const float h1 = __bfloat162float(__float2bfloat16_rn(x.y));
      const float h2 = __bfloat162float(__float2bfloat16_rn(x.z));
      const float h3 = __bfloat162float(__float2bfloat16_rn(x.w));
      const uint2 hi = make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
      const uint2 lw =
          make_uint2(pack_bf16x2(x.x - h0, x.y - h1), pack_bf16x2(x.z - h2, x.w - h3));
      const int off = (kr >> 3) * 1024 + (kr & 7) * 128 + (swz(kr, q4 >> 1) << 4) + (q4 & 1) * 8;
      *reinterpret_cast<uint2*>(smem + kOffBhi + off) = hi;
      *reinterpret_cast<uint2*>(smem + kOffBlo + off) = lw;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = m.tmem_slot;

  // ---- root paths, path-cumulative log-gates and depth levels
  if (!m.bad) {
    for (int n = tid; n < N; n += kTcThreads) {
      int s = n;
      uint64_t strict = 0;
      const int dn = m.dep[n];
      for (int d = dn; d >= 0 && s >= 0; --d) {
        m.anc_at[n][d] = static_cast<uint8_t>(s);
        if (d < dn) strict |= 1ull << s;
        s = m.par[s];
      }
      if (s != -1) {  // the depth disagrees with the parent chain
        m.bad = 1;
        continue;
      }
      float acc = 0.f;
      for (int d = 0; d <= dn; ++d) acc += m.gg[m.anc_at[n][d]];
      m.G[n] = acc;
      m.strict[n] = strict;
    }
    if (tid == 32) {
      int cur = 0;
      for (int p = 0; p < N; ++p) {
        const int d = m.dep[m.ord[p]];
        while (cur <= d) m.lvl[cur++] = p;
      }
      while (cur <= kTcDM1) m.lvl[cur++] = N;
    }
  }
  __syncthreads();

  // ---- 2. MMA issue (one thread).  The key/query copies are always waited
  // for, so no copy is left in flight on any exit path.
  if (tid == 0) {
    m.tma_ok = mbar_wait(&m.tma_bar, 0);
    m.mma_issued = 0;
    if (m.tma_ok && !m.bad) {
      tc_fence_after_sync();
      const uint32_t sA = smem_addr(smem + kOffA);
      const uint32_t sHi = smem_addr(smem + kOffBhi);
      const uint32_t sLo = smem_addr(smem + kOffBlo);
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

  // ---- 3. TMEM -> per-node rows (one TMEM lane per thread; warps 0-1 hold
  // key rows, warps 2-3 query rows).  The operand area is dead and reused.
  if (mma_ok) {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const bool key_row = warp < 2;
    const int n = key_row ? tid : tid - 64;
    const bool live = n < N;
    float* U = reinterpret_cast<float*>(smem + kOffU);
    float* EQ = reinterpret_cast<float*>(smem + kOffEQ);
    float* XS = reinterpret_cast<float*>(smem + kOffXS);
    float* YS = reinterpret_cast<float*>(smem + kOffYS);
    const float Gn = live ? m.G[n] : 0.f;
    const float eG = __expf(Gn);
    const float bn = live ? m.bb[n] : 0.f;
    const uint64_t strict = live ? m.strict[n] : 0ull;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float r[32];
      uint4 vv[4];
      if (key_row && live) {
        const uint4* vp = reinterpret_cast<const uint4*>(
            v + ((size_t)(lo + n) * H_v + h) * kTcDV + c0 + half * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) vv[i] = __ldg(vp + i);
      }
      tmem_ld32(tmem + lane_base + half * 32, r);
      tmem_ld_wait();
      if (live) {
        float* dst = key_row ? U : EQ;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float4 w;
          if (key_row) {
            const __nv_bfloat162* vb = reinterpret_cast<const __nv_bfloat162*>(&vv[ch >> 1]);
            const float2 v01 = __bfloat1622float2(vb[(ch & 1) * 2 + 0]);
            const float2 v23 = __bfloat1622float2(vb[(ch & 1) * 2 + 1]);
            w.x = bn * (v01.x - eG * r[ch * 4 + 0]);
            w.y = bn * (v01.y - eG * r[ch * 4 + 1]);
            w.z = bn * (v23.x - eG * r[ch * 4 + 2]);
            w.w = bn * (v23.y - eG * r[ch * 4 + 3]);
          } else {
            w = make_float4(eG * r[ch * 4 + 0], eG * r[ch * 4 + 1], eG * r[ch * 4 + 2],
                            eG * r[ch * 4 + 3]);
          }
          const int gch = half * 8 + ch;
          *reinterpret_cast<float4*>(dst + n * 64 + swz(n, gch) * 4) = w;
        }
      }
    }
    // Gram row: key rows give X (strict ancestors), query rows give Y (ancestors + self)
    const uint64_t mask = key_row ? strict : (strict | (live ? 1ull << n : 0ull));
    const float scale = key_row ? bn : 1.f;
    float* dst = key_row ? XS : YS;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float r[32];
      tmem_ld32(tmem + lane_base + kTcCols + half * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int s = half * 32 + i;
        if ((mask >> s) & 1ull) dst[n * kTcDM1 + m.dep[s]] = scale * __expf(Gn - m.G[s]) * r[i];
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (!mma_ok) {
    if (!m.bad) {  // a bounded wait expired: report it, leave the outputs alone
      if (tid == 0) status[bi] = TGDN_SEQ_TIMEOUT;
    } else {
      zero_rows();
    }
    return;
  }

  // ---- 4. forward substitution over depth levels, then the output phase
  float* U = reinterpret_cast<float*>(smem + kOffU);
  const float* EQ = reinterpret_cast<const float*>(smem + kOffEQ);
  const float* XS = reinterpret_cast<const float*>(smem + kOffXS);
  const float* YS = reinterpret_cast<const float*>(smem + kOffYS);
  int maxdep = 0;
  while (maxdep + 1 <= kTcDepth && m.lvl[maxdep + 1] < N) ++maxdep;
  for (int d = 1; d <= maxdep; ++d) {
    const int p0 = m.lvl[d], cnt = m.lvl[d + 1] - p0;
    for (int it = tid; it < cnt * 16; it += kTcThreads) {
      const int n = m.ord[p0 + (it >> 4)], ch = it & 15;
      float4 acc = *reinterpret_cast<const float4*>(U + n * 64 + swz(n, ch) * 4);
      for (int dd = 0; dd < d; ++dd) {
        const int s = m.anc_at[n][dd];
        const float x = XS[n * kTcDM1 + dd];
        const float4 us = *reinterpret_cast<const float4*>(U + s * 64 + swz(s, ch) * 4);
        acc.x = fmaf(-x, us.x, acc.x);
        acc.y = fmaf(-x, us.y, acc.y);
        acc.z = fmaf(-x, us.z, acc.z);
        acc.w = fmaf(-x, us.w, acc.w);
      }
      *reinterpret_cast<float4*>(U + n * 64 + swz(n, ch) * 4) = acc;
    }
    __syncthreads();
  }
  for (int it = tid; it < N * 16; it += kTcThreads) {
    const int n = it >> 4, ch = it & 15;
    float4 acc = *reinterpret_cast<const float4*>(EQ + n * 64 + swz(n, ch) * 4);
    const int dn = m.dep[n];
    for (int dd = 0; dd <= dn; ++dd) {
      const int s = m.anc_at[n][dd];
      const float y = YS[n * kTcDM1 + dd];
      const float4 us = *reinterpret_cast<const float4*>(U + s * 64 + swz(s, ch) * 4);
      acc.x = fmaf(y, us.x, acc.x);
      acc.y = fmaf(y, us.y, acc.y);
      acc.z = fmaf(y, us.z, acc.z);
      acc.w = fmaf(y, us.w, acc.w);
    }
    const size_t row = ((size_t)(lo + n) * H_v + h) * kTcDV + c0 + ch * 4;
    *reinterpret_cast<uint2*>(o + row) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    *reinterpret_cast<float4*>(Uws + row) =
        *reinterpret_cast<const float4*>(U + n * 64 + swz(n, ch) * 4);
  }
  if (c == 0)
    for (int n = tid; n < N; n += kTcThreads) Gws[(size_t)(lo + n) * H_v + h] = m.G[n];
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
      qmap, kmap, d.H_qk, d.H_v, t.depth_max, t.cu_nodes, t.parent, t.depth, t.order, t.status,
      static_cast<const __nv_bfloat16*>(v), g, b, S0, static_cast<__nv_bfloat16*>(o), U, G);
  return cudaGetLastError();
}

}  // namespace tgdn
