// verify_tc128.cu — tensor-core tree verification for trees of 65 to 128 nodes
// (bf16 io, d_k = d_v = 128, depth <= 30, sm_103a).
//
// Same method as verify_tc.cu ("Trees from Marginals", Technisches Resümee,
// Methodik 3 and Implementierung): with G the path-cumulative log-gate,
//   (I + X) U = R = diag(b)(V - diag(e^G) K S0),   O = diag(e^G) Q S0 + Y U,
// solved as T = (I + X)^{-1}, W = Y T row by row along each node's root path.
// For trees this large the dense contractions fill the whole TMEM in one go:
//   D[:,   0:128] = K S0      D[:, 128:256] = Q S0      (S0 as bf16 hi + lo)
//   D[:, 256:384] = K K^T     D[:, 384:512] = Q K^T     (lanes = node index)
// so an SM holds one item (sequence, v-head) at a time.  The second step is
// sparse: a row of T or W has at most depth + 1 nonzeros, so U = T R and
// W R are formed on the CUDA cores from an fp32 R in shared memory (the same
// algebra as verify_tc.cu's second product, with R unrounded).
// A tree of 129 nodes whose root is node 0 (a root and 128 draft tokens) is
// taken by folding the root into the state first: S_r = a_r S0 + k_r u_r^T with
// u_r = b_r (v_r - a_r S0^T k_r), o_r = S_r^T q_r, after which the other 128
// nodes form a forest verified from S_r with gates summed below the root.  The
// same tree with its root elsewhere is left untouched for the SIMT kernel,
// launched after this one (verify_simt_kernel's complement mode).
// Persistent CTAs of 512 threads; every wait is bounded (TGDN_SEQ_TIMEOUT on
// expiry).  In a launch that also runs the 64-node kernel, up to 2048 sequences, each
// CTA lists the sequences above 64 nodes and numbers its items over them.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kT8Threads = 512;
constexpr int kT8Nodes = 128;
constexpr int kT8D = 128;
constexpr int kT8Depth = 30;
constexpr int kT8Path = kT8Depth + 1;

// Shared memory (bytes from a 1024-byte aligned base).  Phase 1 (operands of
// the tensor-core product), then phase 2 overlays once that product is done.
constexpr int kO8AK = 0;          // K rows [2 d halves][128 rows][128 B]          32 KiB
constexpr int kO8AQ = 32768;      // Q rows                                          32 KiB
constexpr int kO8S0hi = 65536;    // S0 [2 col atoms][16 k-groups][8][128 B]        32 KiB
constexpr int kO8S0lo = 98304;
constexpr int kO8KKf = 0;         // phase 2a: full K K^T rows [128][128] fp32      64 KiB
constexpr int kO8QKf = 65536;     //           full Q K^T rows                       64 KiB
constexpr int kO8R = 0;           // phase 2b: R [128 nodes][128 cols] fp32         64 KiB
constexpr int kO8Tc = 65536;      //           T coefficients [128][kT8Path] fp32
constexpr int kO8Wc = 65536 + 16384;         // W coefficients
constexpr int kO8SS = 65536 + 32768;         // solve scratch [256][kT8Path] fp32
constexpr int kO8GK = 131072;     // K K^T along each node's path [128][kT8Path]
constexpr int kO8GQ = 131072 + 16384;        // Q K^T along each node's path
constexpr int kO8Meta = 131072 + 32768;


struct T8Meta {
  uint64_t tma_bar, mma_bar;
  uint32_t tmem_slot;
  int abort, tma_n, mma_n;
  int dep[kT8Nodes];
  int ord[kT8Nodes];   // topological position -> node
  float gg[kT8Nodes];
  float bb[kT8Nodes];
  float G[kT8Nodes];
  uint8_t anc_at[kT8Path + 1][kT8Nodes];  // [depth][node]: ancestor of node at that depth
  // Mixed launches: the sequences above 64 nodes in order (items are numbered over them,
  // so that no CTA steps over the 64-node kernel's items).
  int n_big;
  float g_root;  // the folded root's gate, for the path gates written at the end of an item
  int16_t big_seq[2048];
};
constexpr int kT8MaxList = 2048;
constexpr int kT8SmemBytes = kO8Meta + (int)sizeof(T8Meta) + 1024;
static_assert(kT8SmemBytes <= 227 * 1024, "fits one CTA per SM");
static_assert(kO8SS + 256 * kT8Path * 4 <= kO8GK, "solve scratch fits");

__device__ __forceinline__ int t8_atom_off(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
}
// fp32 [row][128] with the 16-byte chunks of each row rotated by the row, so that
// 32 consecutive rows touch 32 different bank groups at the same column.
__device__ __forceinline__ int f_idx(int row, int col) {
  return row * 128 + ((((col >> 2) ^ (row & 31))) << 2) + (col & 3);
}
// This thread's part of one item's state: rows r0 + 16 r, float4 column sq.
__device__ __forceinline__ void load_state_rows(float4 (&sr)[8], const float* src, int r0,
                                                int sq) {
#pragma unroll
  for (int r = 0; r < 8; ++r)
    sr[r] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(r0 + 16 * r) * kT8D) + sq);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

__global__ void __launch_bounds__(kT8Threads, 1)
verify_tc128_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap, int n_items, int H_qk, int H_v,
                    int depth_max, int words, const int32_t* __restrict__ cu,
                    const int32_t* __restrict__ depth, const int32_t* __restrict__ order,
                    const int32_t* __restrict__ pos, const uint64_t* __restrict__ anc,
                    int32_t* __restrict__ status, const __nv_bfloat16* __restrict__ q,
                    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                    const float* __restrict__ g, const float* __restrict__ bta,
                    const float* __restrict__ S0, __nv_bfloat16* __restrict__ o,
                    float* __restrict__ Uws, float* __restrict__ Gws, int big_only) {
  extern __shared__ uint8_t t8_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(t8_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  T8Meta& M = *reinterpret_cast<T8Meta*>(smem + kO8Meta);
  volatile int* abort = &M.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((int)blockIdx.x >= n_items) return;
  const int grp = H_v / H_qk;

  if (tid == 0) {
    mbar_init(&M.tma_bar, 1);
    mbar_init(&M.mma_bar, 1);
    fence_mbar_init();
    M.abort = 0;
    M.tma_n = 0;
    M.mma_n = 0;
  }
  if (warp == 0) tmem_alloc(&M.tmem_slot, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = M.tmem_slot;
  // In a launch that also runs the 64-node kernel, list the sequences above 64 nodes
  // (warp 0, a ballot per 32 sequences) and number the items over them.
  const bool compact = big_only && n_items / H_v <= kT8MaxList;
  int n_it = n_items;
  if (compact) {
    if (warp == 0) {
      const int B = n_items / H_v;
      int base = 0;
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int bq = b0 + lane;
        const bool big = bq < B && cu[bq + 1] - cu[bq] > 64;
        const unsigned m = __ballot_sync(0xffffffffu, big);
        if (big) M.big_seq[base + __popc(m & ((1u << lane) - 1u))] = static_cast<int16_t>(bq);
        base += __popc(m);
      }
      if (lane == 0) M.n_big = base;
    }
    __syncthreads();
    n_it = M.n_big * H_v;
    if ((int)blockIdx.x >= n_it) {
      if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
      }
      return;
    }
  }
  auto seq_of = [&](int it) { return compact ? (int)M.big_seq[it / H_v] : it / H_v; };
  auto state_of = [&](int it) {
    return S0 + ((size_t)seq_of(it) * H_v + it % H_v) * (size_t)(kT8D * kT8D);
  };
  const int lq = warp & 3;                       // TMEM lane quarter of this warp
  const uint32_t lane_base = static_cast<uint32_t>(lq * 32) << 16;
  const int my_row = lq * 32 + lane;             // node index of this thread's TMEM lane
  const int cg = warp >> 2;                      // column group (32 columns) 0..3
  float* KKf = reinterpret_cast<float*>(smem + kO8KKf);
  float* QKf = reinterpret_cast<float*>(smem + kO8QKf);
  float* Rf = reinterpret_cast<float*>(smem + kO8R);
  float* Tc = reinterpret_cast<float*>(smem + kO8Tc);
  float* Wc = reinterpret_cast<float*>(smem + kO8Wc);
  float* SSb = reinterpret_cast<float*>(smem + kO8SS);
  float* GK = reinterpret_cast<float*>(smem + kO8GK);
  float* GQ = reinterpret_cast<float*>(smem + kO8GQ);

  // The sequence bounds and status two items ahead and the root depth one item
  // ahead in registers (raw values: nothing waits for them before they are
  // used), and the next item's state, V rows and tree metadata pulled into L2
  // while the current item is being worked on (16-byte aligned ranges).
  const int sq = tid & 31, r0 = tid >> 5;
  int nx_lo = 0, nx_hi = 0, nx_st = 0, nx_d0 = 0;  // the next item
  int nb_lo = 0, nb_hi = 0, nb_st = 0;             // the item after it
  float4 sr[8];
  auto load_bounds = [&](int it) {
    if (it < n_it) {
      const int b2 = seq_of(it);
      nb_lo = cu[b2];
      nb_hi = cu[b2 + 1];
      nb_st = status[b2];
    }
  };
  auto advance = [&](int it) {  // it: the next item; its bounds are in nb_*
    nx_lo = nb_lo;
    nx_hi = nb_hi;
    nx_st = nb_st;
    nx_d0 = 0;
    // (an item this launch passes over, a sequence of at most 64 nodes when the
    // 64-node kernel takes those, is not pulled into L2)
    if (it < n_it && nx_st == TGDN_SEQ_OK && nx_hi > nx_lo &&
        !(big_only && nx_hi - nx_lo <= 64)) {
      nx_d0 = depth[nx_lo];
      if (tid == 0) prefetch_l2(state_of(it), kT8D * kT8D * 4);
      if (tid < nx_hi - nx_lo && tid <= kT8Nodes)
        prefetch_l2(v + ((size_t)(nx_lo + tid) * H_v + it % H_v) * kT8D, kT8D * 2);
      if (tid >= 32 && tid < 35) {
        const int32_t* arr = tid == 32 ? depth : tid == 33 ? pos : order;
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(arr + nx_lo) & ~(uintptr_t)15;
        const uintptr_t a1 = reinterpret_cast<uintptr_t>(arr + nx_hi) & ~(uintptr_t)15;
        if (a1 > a0) prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
      }
      if (tid == 35) {  // the ancestor masks (16-byte aligned range inside the array)
        const uintptr_t a0 =
            reinterpret_cast<uintptr_t>(anc + (size_t)nx_lo * words) & ~(uintptr_t)15;
        const uintptr_t a1 =
            reinterpret_cast<uintptr_t>(anc + (size_t)nx_hi * words) & ~(uintptr_t)15;
        if (a1 > a0) prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
      }
    }
  };
#define T8_PREFETCH(it)              \
  advance(it);                       \
  load_bounds((it) + (int)gridDim.x);
  load_bounds((int)blockIdx.x);
  T8_PREFETCH((int)blockIdx.x)

  for (int item = blockIdx.x; item < n_it; item += gridDim.x) {
    const int h = item % H_v, qh = h / grp;
    const int lo = nx_lo, N = nx_hi - nx_lo;
    const int st = nx_st;
    const bool st_ok = st == TGDN_SEQ_OK;
    const int d0 = nx_d0;
    // the next item's bounds and L2 prefetches go out now and land during this item
    T8_PREFETCH(item + (int)gridDim.x)
    if (N <= 0) continue;  // uniform over the CTA
    if (st == TGDN_SEQ_BAD_RANGE) continue;  // rows outside the arrays: untouched
    if (big_only && N <= 64) continue;  // the 64-node kernel's sequence
    const int fold = (st_ok && N == kT8Nodes + 1 && d0 == 0) ? 1 : 0;
    if (st_ok && N == kT8Nodes + 1 && !fold) continue;  // root elsewhere: the SIMT kernel's
    const int Nf = N - fold;                             // nodes on the tensor cores
    const size_t obase0 = (size_t)lo * H_v + h;          // row of node 0
    const size_t obase = obase0 + (size_t)fold * H_v;    // row of the first tensor-core node
    bool ok = st_ok && Nf <= kT8Nodes;
    const bool tma_issued = ok;

    // ---- K and Q rows of the item by TMA (rows lo .. lo + 127; rows past the tree unused)
    if (ok && tid == 0) {
      mbar_arrive_expect_tx(&M.tma_bar, 8 * 8192);
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int rb = 0; rb < 2; ++rb) {
          tma_load_3d(smem + kO8AK + half * 16384 + rb * 8192, &kmap, &M.tma_bar, half * 64, qh,
                      lo + fold + rb * 64);
          tma_load_3d(smem + kO8AQ + half * 16384 + rb * 8192, &qmap, &M.tma_bar, half * 64, qh,
                      lo + fold + rb * 64);
        }
      M.tma_n += 1;
    }
    // the item's state rows and this thread's V slice, ahead of their use
    load_state_rows(sr, state_of(item), r0, sq);
    uint4 vreg[4];  // this thread's V row slice (32 columns), for R after the product
    if (ok && my_row < Nf) {
      const uint4* vp =
          reinterpret_cast<const uint4*>(v + (obase + (size_t)my_row * H_v) * kT8D + cg * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) vreg[i] = __ldg(vp + i);
    }
    // ---- metadata, root paths and path-cumulative gates (one thread per node)
    // (with a folded root, node nd = tid + 1 is tensor-core node tid; depths and
    // topological positions drop by one: the root is position 0)
    uint64_t mk3[3] = {0ull, 0ull, 0ull};  // this node's ancestor mask words
    if (ok && tid < Nf) {
      const int nd = tid + fold;
      const int dn = depth[lo + nd] - fold, pn = pos[lo + nd] - fold;
      const int od = order[lo + tid + fold] - fold;
      const bool v_ok = dn >= 0 && dn <= depth_max && dn <= kT8Depth && pn >= 0 && pn < Nf &&
                        od >= 0 && od < Nf;
      M.dep[tid] = v_ok ? dn : 0;
      M.ord[tid] = v_ok ? od : 0;
      M.gg[tid] = g[(size_t)(lo + nd) * H_v + h];
      M.bb[tid] = bta[(size_t)(lo + nd) * H_v + h];
      if (v_ok) {  // the mask is read before the barrier, used after it
        const uint64_t* am = anc + (size_t)(lo + pn + fold) * words;
#pragma unroll
        for (int w = 0; w < 3; ++w)
          if (w < words) mk3[w] = am[w];
      }
      if (!v_ok) ok = false;
    }
    ok = __syncthreads_and(ok) != 0;
    // ---- S0 -> bf16 hi + lo operand (thread: rows (tid >> 5) + 16 r, float4 column tid & 31)
    {
      if (fold) {  // the root's own step: S_r = a_r S0 + k_r u_r^T, o_r = S_r^T q_r
        float* part = reinterpret_cast<float*>(smem + kO8GK);  // [16][128] partial sums
        float* kr = part + 16 * kT8D;
        float* qr = kr + kT8D;
        float* ur = qr + kT8D;
        const float gr = g[obase0];
        const float ar = __expf(gr), br = bta[obase0];
        if (tid == 0) M.g_root = gr;
        if (tid < kT8D) {
          kr[tid] = __bfloat162float(k[((size_t)lo * H_qk + qh) * kT8D + tid]);
          qr[tid] = __bfloat162float(q[((size_t)lo * H_qk + qh) * kT8D + tid]);
        }
        __syncthreads();
        float4 pw = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float kv = kr[r0 + 16 * r];
          pw.x = fmaf(kv, sr[r].x, pw.x);
          pw.y = fmaf(kv, sr[r].y, pw.y);
          pw.z = fmaf(kv, sr[r].z, pw.z);
          pw.w = fmaf(kv, sr[r].w, pw.w);
        }
        reinterpret_cast<float4*>(part + r0 * kT8D)[sq] = pw;
        __syncthreads();
        if (tid < kT8D) {
          float w = 0.f;
          for (int i = 0; i < 16; ++i) w += part[i * kT8D + tid];
          const float u = br * (__bfloat162float(v[obase0 * kT8D + tid]) - ar * w);
          ur[tid] = u;
          Uws[obase0 * kT8D + tid] = u;
        }
        __syncthreads();
        const float4 u4 = reinterpret_cast<const float4*>(ur)[sq];
        float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float kv = kr[r0 + 16 * r], qv = qr[r0 + 16 * r];
          sr[r].x = fmaf(kv, u4.x, ar * sr[r].x);
          sr[r].y = fmaf(kv, u4.y, ar * sr[r].y);
          sr[r].z = fmaf(kv, u4.z, ar * sr[r].z);
          sr[r].w = fmaf(kv, u4.w, ar * sr[r].w);
          po.x = fmaf(qv, sr[r].x, po.x);
          po.y = fmaf(qv, sr[r].y, po.y);
          po.z = fmaf(qv, sr[r].z, po.z);
          po.w = fmaf(qv, sr[r].w, po.w);
        }
        reinterpret_cast<float4*>(part + r0 * kT8D)[sq] = po;
        __syncthreads();
        if (tid < kT8D) {
          float acc = 0.f;
          for (int i = 0; i < 16; ++i) acc += part[i * kT8D + tid];
          o[obase0 * kT8D + tid] = __float2bfloat16_rn(acc);
          if (tid == 0) Gws[obase0] = gr;
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int kr = r0 + 16 * r;
        const float4 x = sr[r];
        const float h0 = __bfloat162float(__float2bfloat16_rn(x.x));
        const float h1 = __bfloat162float(__float2bfloat16_rn(x.y));
        const float h2 = __bfloat162float(__float2bfloat16_rn(x.z));
        const float h3 = __bfloat162float(__float2bfloat16_rn(x.w));
        const int off = (sq >> 4) * 16384 + t8_atom_off(kr, (sq & 15) >> 1) + (sq & 1) * 8;
        *reinterpret_cast<uint2*>(smem + kO8S0hi + off) = make_uint2(pack2(h0, h1), pack2(h2, h3));
        *reinterpret_cast<uint2*>(smem + kO8S0lo + off) =
            make_uint2(pack2(x.x - h0, x.y - h1), pack2(x.z - h2, x.w - h3));
      }
    }
    fence_proxy_async_smem();
    __syncthreads();  // the S0 operand is complete
    // ---- the tensor-core product, issued by the last thread (it has no node)
    // while the node threads build their root paths
    bool step_ok = true;
    const bool product = ok;  // (uniform) metadata valid: copy issued, product goes out
    if (tid == kT8Threads - 1 && product) {
      step_ok = mbar_wait_suspend(&M.tma_bar, (M.tma_n - 1) & 1, abort);
      if (step_ok) {
        tc_fence_after_sync();
        const uint32_t sK = smem_addr(smem + kO8AK), sQ = smem_addr(smem + kO8AQ);
        const uint32_t sHi = smem_addr(smem + kO8S0hi), sLo = smem_addr(smem + kO8S0lo);
        constexpr uint32_t id_s0 = idesc_bf16_f32(128, 128, 0, 1);
        constexpr uint32_t id_g = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
        for (int s = 0; s < kT8D / 16; ++s) {
          const uint32_t ko = (s >> 2) * 16384 + (s & 3) * 32;
          const uint64_t ak = smem_desc(sK + ko, 16, 1024, kSwizzle128B);
          const uint64_t aq = smem_desc(sQ + ko, 16, 1024, kSwizzle128B);
          // MN-major S0: value-column atoms 16 KiB apart, 8-row k groups 1 KiB apart
          const uint64_t hd = smem_desc(sHi + s * 2048, 16384, 1024, kSwizzle128B);
          const uint64_t ld = smem_desc(sLo + s * 2048, 16384, 1024, kSwizzle128B);
          umma_bf16(tmem, ak, hd, id_s0, s > 0);
          umma_bf16(tmem, ak, ld, id_s0, 1);
          umma_bf16(tmem + 128, aq, hd, id_s0, s > 0);
          umma_bf16(tmem + 128, aq, ld, id_s0, 1);
          umma_bf16(tmem + 256, ak, ak, id_g, s > 0);  // B = the key rows
          umma_bf16(tmem + 384, aq, ak, id_g, s > 0);
        }
        umma_commit(&M.mma_bar);
        M.mma_n += 1;
      }
    }
    if (ok && tid < Nf) {
      // bits of the ancestor mask are topological positions; ascending = root first
      const int dn = M.dep[tid];
      int i = 0;
      float acc = 0.f;
      bool pk = true;
#pragma unroll
      for (int w = 0; w < 3; ++w) {
        if (w >= words || !pk) break;
        uint64_t mk = mk3[w];
        while (mk && pk) {
          const int b = w * 64 + __ffsll(static_cast<long long>(mk)) - 1 - fold;
          mk &= mk - 1;
          if (b < 0) continue;  // the folded root
          if (b >= Nf || i > dn) {
            pk = false;
            break;
          }
          const int s = M.ord[b];
          pk = M.dep[s] == i;
          M.anc_at[i][tid] = static_cast<uint8_t>(s);
          acc += M.gg[s];
          ++i;
        }
      }
      if (!pk || i != dn + 1 || M.anc_at[dn][tid] != tid) ok = false;
      M.G[tid] = acc;
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {  // bad sequence: zero rows, and let an issued copy and product land before reuse
      if (tid == kT8Threads - 1 && product && step_ok)
        (void)mbar_wait_suspend(&M.mma_bar, (M.mma_n - 1) & 1, abort);
      if (tid == 0 && tma_issued) (void)mbar_wait_suspend(&M.tma_bar, (M.tma_n - 1) & 1, abort);
      for (int e = tid; e < N * (kT8D / 4); e += kT8Threads) {
        const int n = e >> 5, c4 = e & 31;
        const size_t row = (obase0 + (size_t)n * H_v) * kT8D + c4 * 4;
        *reinterpret_cast<uint2*>(o + row) = make_uint2(0u, 0u);
        *reinterpret_cast<float4*>(Uws + row) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int n = tid; n < N; n += kT8Threads) Gws[obase0 + (size_t)n * H_v] = 0.f;
      if (__syncthreads_or(*abort)) break;
      continue;
    }

    if (tid == kT8Threads - 1 && step_ok)
      step_ok = mbar_wait_suspend(&M.mma_bar, (M.mma_n - 1) & 1, abort);
    if (!__syncthreads_and(step_ok)) break;
    tc_fence_after_sync();

    // ---- Gram rows TMEM -> shared memory (full rows), then compressed to the path
    {
      const int mat = cg >> 1, half = cg & 1;     // 0: K K^T, 1: Q K^T; columns half*64..
      float* F = mat == 0 ? KKf : QKf;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float r[32];
        tmem_ld32(tmem + lane_base + 256 + mat * 128 + half * 64 + q * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const int col = half * 64 + q * 32 + c4 * 4;
          *reinterpret_cast<float4*>(F + f_idx(my_row, col)) =
              make_float4(r[c4 * 4], r[c4 * 4 + 1], r[c4 * 4 + 2], r[c4 * 4 + 3]);
        }
      }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 2 * kT8Nodes) {
      const int n = tid & 127;
      if (n < Nf) {
        const float* F = tid < kT8Nodes ? KKf : QKf;
        float* C = (tid < kT8Nodes ? GK : GQ) + n * kT8Path;
        const int dn = M.dep[n];
        for (int i = 0; i <= dn; ++i) C[i] = F[f_idx(n, M.anc_at[i][n])];
      }
    }
    __syncthreads();

    // ---- R = diag(b)(V - e^G K S0) in fp32 (thread: node my_row, 32 columns)
    {
      const bool live = my_row < Nf;
      const float eG = live ? __expf(M.G[my_row]) : 0.f;
      const float bn = live ? M.bb[my_row] : 0.f;
      float r[32];
      tmem_ld32(tmem + lane_base + cg * 32, r);
      tmem_ld_wait();
      if (live) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          const __nv_bfloat162* vb = reinterpret_cast<const __nv_bfloat162*>(&vreg[c8]);
          float x[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 vf = __bfloat1622float2(vb[i]);
            x[2 * i] = bn * (vf.x - eG * r[c8 * 8 + 2 * i]);
            x[2 * i + 1] = bn * (vf.y - eG * r[c8 * 8 + 2 * i + 1]);
          }
          const int col = cg * 32 + c8 * 8;
          *reinterpret_cast<float4*>(Rf + f_idx(my_row, col)) = make_float4(x[0], x[1], x[2], x[3]);
          *reinterpret_cast<float4*>(Rf + f_idx(my_row, col + 4)) =
              make_float4(x[4], x[5], x[6], x[7]);
        }
      }
    }

    // ---- rows of T (solver 0..127) and W (128..255) by back substitution on the
    // root path P = (p_0 = root, ..., p_d = n), with each entry rescaled to
    // rho_j = r_j e^{G_{p_j} - G_n} so that the gates leave the recurrence:
    //   rho_j = y'_j - sum_{i>j} b_{p_i} rho_i k_{p_i}.k_{p_j},
    //   y' = e_d for T,  y'_j = q_n.k_{p_j} for W;  r_j = rho_j e^{G_n - G_{p_j}}.
    // k_{p_i}.k_{p_j} is entry j of p_i's compressed row (p_j is its ancestor at depth j).
    if (tid < 2 * kT8Nodes) {
      const bool t_row = tid < kT8Nodes;
      const int spos = tid & 127;
      if (spos < Nf) {
        const int sn = M.ord[spos];
        const int dn = M.dep[sn];
        float* SS = SSb + tid * kT8Path;
        float* coef = (t_row ? Tc : Wc) + sn * kT8Path;
        const float Gn = M.G[sn];
        for (int jj = dn; jj >= 0; --jj) {
          const int pj = M.anc_at[jj][sn];
          const float y = t_row ? ((jj == dn) ? 1.f : 0.f) : GQ[sn * kT8Path + jj];
          float acc = 0.f;
#pragma unroll 4
          for (int i = jj + 1; i <= dn; ++i)
            acc = fmaf(SS[i], GK[M.anc_at[i][sn] * kT8Path + jj], acc);
          const float rho = y - acc;
          SS[jj] = rho * M.bb[pj];
          coef[jj] = rho * __expf(Gn - M.G[pj]);
        }
      }
    }
    __syncthreads();

    // ---- U = T R and O = e^G Q S0 + W R (thread: node my_row, 32 columns)
    {
      const bool live = my_row < Nf;
      float w[32];
      tmem_ld32(tmem + lane_base + 128 + cg * 32, w);
      tmem_ld_wait();
      if (live) {
        const int dn = M.dep[my_row];
        const float eG = __expf(M.G[my_row]);
        float u[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          u[c] = 0.f;
          w[c] *= eG;
        }
        for (int j = 0; j <= dn; ++j) {
          const int pj = M.anc_at[j][my_row];
          const float tj = Tc[my_row * kT8Path + j], wj = Wc[my_row * kT8Path + j];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 rr = *reinterpret_cast<const float4*>(Rf + f_idx(pj, cg * 32 + c4 * 4));
            u[c4 * 4] = fmaf(tj, rr.x, u[c4 * 4]);
            u[c4 * 4 + 1] = fmaf(tj, rr.y, u[c4 * 4 + 1]);
            u[c4 * 4 + 2] = fmaf(tj, rr.z, u[c4 * 4 + 2]);
            u[c4 * 4 + 3] = fmaf(tj, rr.w, u[c4 * 4 + 3]);
            w[c4 * 4] = fmaf(wj, rr.x, w[c4 * 4]);
            w[c4 * 4 + 1] = fmaf(wj, rr.y, w[c4 * 4 + 1]);
            w[c4 * 4 + 2] = fmaf(wj, rr.z, w[c4 * 4 + 2]);
            w[c4 * 4 + 3] = fmaf(wj, rr.w, w[c4 * 4 + 3]);
          }
        }
        const size_t row = (obase + (size_t)my_row * H_v) * kT8D + cg * 32;
        float4* ud = reinterpret_cast<float4*>(Uws + row);
        uint4* od = reinterpret_cast<uint4*>(o + row);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          ud[c4] = make_float4(u[c4 * 4], u[c4 * 4 + 1], u[c4 * 4 + 2], u[c4 * 4 + 3]);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
          od[c8] = make_uint4(pack2(w[c8 * 8], w[c8 * 8 + 1]), pack2(w[c8 * 8 + 2], w[c8 * 8 + 3]),
                              pack2(w[c8 * 8 + 4], w[c8 * 8 + 5]),
                              pack2(w[c8 * 8 + 6], w[c8 * 8 + 7]));
        if (cg == 0)  // stored from the root down (the folded root's gate included)
          Gws[obase + (size_t)my_row * H_v] = M.G[my_row] + (fold ? M.g_root : 0.f);
      }
    }
    tc_fence_before_sync();
    __syncthreads();  // TMEM and shared memory are reused by the next item
    tc_fence_after_sync();
  }

  // ---- end.  After an expired wait every item still owned by this CTA is
  // reported as timed out, and the latest copy and product are drained (bounded).
  __syncthreads();
  if (M.abort && tid == 0) {
    for (int it2 = blockIdx.x; it2 < n_it; it2 += gridDim.x)
      atomicCAS(&status[seq_of(it2)], TGDN_SEQ_OK, TGDN_SEQ_TIMEOUT);
    if (M.tma_n > 0) (void)mbar_wait(&M.tma_bar, (M.tma_n - 1) & 1);
    if (M.mma_n > 0) (void)mbar_wait(&M.mma_bar, (M.mma_n - 1) & 1);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

#undef T8_PREFETCH

bool verify_tc128_supported(const tgdn_tree& t, const tgdn_dims& d, const void* q,
                            const void* k, const void* v, const float* S0, const void* o) {
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
  return d.io == TGDN_BF16 && d.d_k == kT8D && d.d_v == kT8D && t.n_max <= kT8Nodes + 1 &&
         t.depth_max <= kT8Depth && al(q, 16) && al(k, 16) && al(v, 16) && al(S0, 16) &&
         al(o, 16);
}


cudaError_t launch_verify_tc128(const tgdn_tree& t, const tgdn_dims& d, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const void* q, const void* k,
                                const void* v, const float* g,
                                const float* b, const float* S0, void* o, float* U, float* G,
                                bool big_only, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(verify_tc128_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kT8SmemBytes);
  if (e != cudaSuccess) return e;
  const long items = (long)t.B * d.H_v;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  const int sms = device_sm_count();
  const int grid = (int)(items < sms ? items : sms);
  verify_tc128_kernel<<<grid, kT8Threads, kT8SmemBytes, s>>>(
      qmap, kmap, (int)items, d.H_qk, d.H_v, t.depth_max, t.words, t.cu_nodes, t.depth, t.order,
      t.pos, t.anc, t.status, static_cast<const __nv_bfloat16*>(q),
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), g, b, S0,
      static_cast<__nv_bfloat16*>(o), U, G, big_only ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace tgdn
