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
// path of n: it solves a (depth+1)-sized unit triangular system.  So
// U = T R and O = diag(e^G) Q S0 + W R, both tensor-core products.
//
// Persistent, warp-specialised kernel: one CTA per SM, 16 warps, looping over
// work items (sequence, v-head) that cover all 128 value columns (a contiguous
// run per CTA with a pending commit, else dealt round robin); trees have at most
// 64 nodes and depth at most 30.  Two items are in flight per SM:
//   producer warps 0-7, item j+1:
//     tree metadata (prefetched as raw values) -> root paths (reused for the
//     next head of the same sequence) and path-cumulative gates;
//     S0 (prefetched into registers; warp w holds rows 16 w .. 16 w + 15) ->
//     bf16 hi + lo operands (~16-bit products);
//     TMA of the item's key and query rows -> A = [K; Q] (128-byte swizzle);
//     the group's last thread issues tcgen05.mma into TMEM half (j+1)&1:
//        D[:, 0:128] = A (S0_hi + S0_lo),  D[:, 128:192] = A K^T
//     while the others prefetch the next item and build the paths; the
//     product's completion is awaited one item later, just before its operands
//     are overwritten.
//   consumer warps 8-15, item j:
//     Gram rows -> shared memory; V rows arrive by TMA in the R lo operand area
//     and the key-lane warps form R = diag(b)(V - e^G K S0) there in place
//     (bf16 hi/lo operand) while the query-lane warps substitute along the root
//     paths with the partial sums in registers (depth <= 16: a node's T and W
//     rows in one thread; deeper: one row per thread), writing straight into
//     the [T; W] operand;
//     tcgen05.mma: D[:, 128:256] = [T; W] R;
//     U (workspace) and O = e^G Q S0 + W R (bf16) leave through shared-memory
//     staging and bulk copies.
// The halves hand over through mbarriers: "stage 1 done" (the first product's
// completion plus the producer's metadata) and "TMEM half free".  The kernel
// is launched with programmatic stream serialization: its prologue may overlap
// the previous kernel's tail and no input is read before griddepcontrol.wait.
// In a launch above 64 nodes it takes only the sequences of at most 64 nodes
// (small_only) and passes over the others without touching them.
//
// Deferred commit folded into the next verify (Methodik 3, last bullet: the
// state is committed once the accepted branch is known, in the following
// decode iteration).  When the previous step left a commit pending, the
// producer stages that step's accepted path for the item (u_s rows, k_s rows
// and G_s by 16-byte asynchronous copies, one item ahead, into an area of
// their own) and forms
//   S = e^{G*} S_prev + sum_{s on the path} e^{G*-G_s} k_s u_s^T
// in registers, writes it back in place (the committed state) and verifies
// from it.  The state then crosses HBM once in each direction per step.  The
// commit touches neither the TMEM half nor the metadata slot of its item, so
// the producer does it before it waits for the consumer to free them.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kTcThreads = 512;
constexpr int kGroup = 256;    // threads per warp group (producer / consumer)
constexpr int kBarP = 1, kBarC = 2;  // hardware barrier ids of the two groups
constexpr int kTcNodes = 64;   // nodes per tree on this kernel
constexpr int kTcDK = 128;
constexpr int kTcDV = 128;
constexpr int kTcDepth = 30;   // depth bound on this kernel
constexpr int kTcPath = kTcDepth + 1;  // entries of a root path
constexpr int kPathBytes = 32;         // one root path: a byte per depth, zero past the node
constexpr uint32_t kTmemCols = 512;    // two halves of 256 columns
constexpr int kGramCol = 128;          // within a half: Gram rows, then [T; W] R

// Shared-memory map (bytes from a 1024-byte aligned base).
constexpr int kOffA = 0;          // [K;Q] operand: [2 d_k halves][128 rows][128 B]      32 KiB
constexpr int kOffS0hi = 32768;   // S0 operand, MN-major [2 col atoms][16 k-groups][8][128 B]
constexpr int kOffS0lo = 65536;
constexpr int kOffGR = 98304;     // Gram rows [128 lanes][64] fp32                        32 KiB
constexpr int kOffRhi = 131072;   // R operand, MN-major [2 col atoms][8 node groups][8][128 B]
constexpr int kOffRlo = 147456;
constexpr int kOffA2hi = 163840;  // [T; W] operand, K-major [16 row groups][8][128 B]     16 KiB
constexpr int kOffA2lo = 180224;
// Pending-commit staging, an area of its own so that the next item's rows are in
// flight while this item's operands are still being read:
constexpr int kOffUP = 196608;                        // u_s rows [kTcPath][128] fp32   15.5 KiB
constexpr int kOffKP = kOffUP + kTcPath * kTcDV * 4;  // k_s rows [kTcPath][128] bf16   7.75 KiB
constexpr int kOffGP = kOffKP + kTcPath * kTcDK * 2;  // 16-byte chunks holding G_s [kTcPath]
constexpr int kOffMeta = (kOffGP + kTcPath * 16 + 127) & ~127;
// Output staging after the second product (its operand areas are free then):
constexpr int kOffUst = kOffGR;     // U rows [64][528 B] fp32 (GR and the start of R hi)
constexpr int kUstRow = 528;        // 512 B + 16: rows 8 apart share banks, no more
constexpr int kOffOst = kOffA2hi;   // O rows [64][272 B] bf16 (the [T; W] operand area)
constexpr int kOstRow = 272;
static_assert(kOffUst + 64 * kUstRow <= kOffRlo, "U staging stays clear of the V rows");
static_assert(kOffOst + 64 * kOstRow <= kOffUP, "O staging stays in the [T; W] area");

struct alignas(16) ItemMeta {
  uint8_t path[kTcNodes][kPathBytes];  // [node][depth]: the node's ancestor at that depth
  int lo, N, h, good;
  int skip;  // a sequence above 64 nodes in a mixed launch: nothing to do here
  int dep[kTcNodes];
  int ord[kTcNodes];
  int pos[kTcNodes];
  float gg[kTcNodes];
  float G[kTcNodes];
  float bb[kTcNodes];
};
struct TcShared {
  uint64_t tma_bar, mma1_bar, mma2_bar, v_bar;
  uint64_t s1_done[2];    // consumer waits: first product done + metadata written
  uint64_t tmem_free[2];  // producer waits: consumer finished the item in this half
  uint32_t tmem_slot;
  int abort;
  int tma_issued;
  int v_issued;
  int mma1_issued;
  int c_L[2];             // staged path length per item parity (0: nothing to commit)
  int c_row[2][kTcPath];  // previous-step node rows of the staged path
  int c_gi[2][kTcPath];   // index of G_s within its staged 16-byte chunk
  ItemMeta meta[2];
};
constexpr int kTcSmemBytes = kOffMeta + (int)sizeof(TcShared) + 1024;  // + alignment slack
static_assert(kTcSmemBytes <= 227 * 1024, "fits one CTA per SM");

// 16-byte chunk swizzle of the 128-byte-row operands (TMA and tcgen05
// SWIZZLE_128B layout for 1024-byte aligned 8-row atoms).
__device__ __forceinline__ int swz(int row, int chunk) { return chunk ^ (row & 7); }
__device__ __forceinline__ int atom_off(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + (swz(row, chunk) << 4);
}

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

// One thread of a warp group waits on the mbarrier (suspending, bounded); the
// rest of the group parks on the group's hardware barrier, which also makes
// the outcome the same for every thread of the group.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, int bar_id,
                                           bool leader, volatile int* abort) {
  bool ok = true;
  if (leader) ok = mbar_wait_suspend(bar, parity, abort);
  return named_sync_and(bar_id, kGroup, ok);
}

// Everything the producer prefetches for one item (one node per thread < 64).
struct Prefetch {
  int lo, N, st;
  int dep, pos, ord;
  float gg, bb;
};

// v[k] for a run-time k in [0, N), N a power of two: a binary multiplexer over
// the bits of k (fixed register indices, log2 N dependent selects).
template <int N>
__device__ __forceinline__ float pick(const float (&v)[N], int k) {
  float t[N];
#pragma unroll
  for (int m = 0; m < N; ++m) t[m] = v[m];
#pragma unroll
  for (int w = N / 2, bit = 0; w >= 1; w /= 2, ++bit) {
    const bool hi = (k >> bit) & 1;
#pragma unroll
    for (int m = 0; m < w; ++m) t[m] = hi ? t[2 * m + 1] : t[2 * m];
  }
  return t[0];
}

// Byte j of the packed root path (a node index).
__device__ __forceinline__ int path_at(const uint32_t (&pw)[8], int j) {
  return static_cast<int>((pw[j >> 2] >> (8 * (j & 3))) & 0xffu);
}

// acc[j] += s * row[p_j ^ x] for j < W.  Only j < i - 1 matter at step i; the
// other entries are either the next one (taken out before) or settled ones,
// never read again, so the width only has to cover i - 1 (no per-entry test).
template <int W, int N>
__device__ __forceinline__ void path_update(float (&acc)[N], const uint32_t (&pw)[8], float s,
                                            const float* row, int x) {
  static_assert(W <= N, "width within the partial sums");
#pragma unroll
  for (int j = 0; j < W; ++j) acc[j] = fmaf(s, row[path_at(pw, j) ^ x], acc[j]);
}

// The same for the T and W rows of one node (one Gram read, two sums).
template <int W, int N>
__device__ __forceinline__ void path_update2(float (&accT)[N], float (&accW)[N],
                                             const uint32_t (&pw)[8], float sT, float sW,
                                             const float* row, int x) {
  static_assert(W <= N, "width within the partial sums");
#pragma unroll
  for (int j = 0; j < W; ++j) {
    const float gk = row[path_at(pw, j) ^ x];
    accT[j] = fmaf(sT, gk, accT[j]);
    accW[j] = fmaf(sW, gk, accW[j]);
  }
}

// One row of T (t_row) or W of the node sn at depth dn, by substitution along
// its root path P = (p_0 = root, ..., p_dn = sn):
//   r (I + X_P) = y,  X_P[i][j] = b_{p_i} e^{G_{p_i} - G_{p_j}} k_{p_i}.k_{p_j} (i > j),
//   y = e_dn for T;  y_j = e^{G_n - G_{p_j}} q_n.k_{p_j} for W.
// With phi_i = e^{G_{p_i} - G_n} >= 1 and s_i = r_i b_{p_i} phi_i:
//   r_j = y_j - (1 / phi_j) acc_j,  acc_j = sum_{i>j} s_i k_{p_i}.k_{p_j}.
// Entries are settled from the node towards the root; once s_i is known it is
// added into every acc_j (j < i) at once.  acc lives in registers; the loop
// runs from the warp's deepest row, so the step index i is the same in every
// lane.  The next entry's sum is taken out of acc before the update and only
// its own term is added, so the chain from one entry to the next is a few
// dependent operations; the Gram reads and the other updates are off it.
// (phi is capped at e^80; the capped terms are below fp32 resolution.)  r_j is
// written as bf16 hi + lo at column p_j of the [T; W] operand row.
template <int D>
__device__ __forceinline__ void solve_path_row(const ItemMeta& M, const float* GR,
                                               uint8_t* smem, int sn, int dn, int wmax,
                                               bool t_row) {
  constexpr int NA = D <= 16 ? 16 : 32;  // partial sums held (entries 0 .. NA-1)
  static_assert(D <= NA, "path fits the partial sums");
  const uint8_t* prow = M.path[sn];  // entries past the node are 0 (a valid node)
  const uint4* pr = reinterpret_cast<const uint4*>(prow);
  const uint4 pa = pr[0], pb = pr[1];
  const uint32_t pw[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
  const float Gn = M.G[sn];
  const int a2row = t_row ? sn : 64 + sn;
  const float* GRq = GR + (64 + sn) * 64;  // q_n . k_s, row 64 + sn (same swizzle phase)
  const int xq = (sn & 7) << 2;
  float acc[NA];
#pragma unroll
  for (int k = 0; k < NA; ++k) acc[k] = 0.f;
  float ai = 0.f;  // acc_i of the current step
  // Software pipeline: the path entry two steps ahead and the gate, beta and
  // query-Gram value one step ahead are loaded before they are needed.
  int pi = prow[wmax];
  int pn = wmax > 0 ? prow[wmax - 1] : 0;  // the next entry's node
  float Gi = M.G[pi], bi = M.bb[pi];
  float qi = t_row ? 0.f : GRq[pi ^ xq];
  for (int i = wmax; i >= 0; --i) {
    const int pnn = i > 1 ? prow[i - 2] : 0;
    const float Gnx = M.G[pn], bnx = M.bb[pn];
    const float qnx = t_row ? 0.f : GRq[pn ^ xq];
    // Gram row p_i: element (p_i, c) sits at p_i * 64 + (c ^ ((p_i & 7) << 2))
    const float* GRi = GR + pi * 64;
    const int xi = (pi & 7) << 2;
    const float kn = GRi[pn ^ xi];  // k_{p_i}.k_{p_{i-1}}
    const float y = t_row ? (i == dn ? 1.f : 0.f) : __expf(Gn - Gi) * qi;
    const float inv_phi = __expf(fmaxf(Gn - Gi, -80.f));
    const float f = bi * __expf(fminf(Gi - Gn, 80.f));
    const float base = pick<NA>(acc, i - 1);  // acc_{i-1} before this step's term
    const float r = y - inv_phi * ai;
    const bool own = i <= dn;
    const float s = own ? r * f : 0.f;
    if (own) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(r);
      const __nv_bfloat16 lw = __float2bfloat16_rn(r - __bfloat162float(hi));
      const int off = atom_off(a2row, pi >> 3) + (pi & 7) * 2;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2hi + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2lo + off) = lw;
    }
    const int lim = i - 1;  // entries 0 .. i-2 take their terms here
    if (lim <= 8) {
      path_update<8>(acc, pw, s, GRi, xi);
    } else if (lim <= 16) {
      path_update<16>(acc, pw, s, GRi, xi);
    } else if (lim <= 24) {
      path_update<(NA < 24 ? NA : 24)>(acc, pw, s, GRi, xi);
    } else {
      path_update<NA>(acc, pw, s, GRi, xi);
    }
    ai = fmaf(s, kn, base);
    pi = pn;
    pn = pnn;
    Gi = Gnx;
    bi = bnx;
    qi = qnx;
  }
}

// The T row and the W row of node sn together (trees of depth <= 16): one path
// walk, one Gram read per entry for both sums, the gate factors shared.
template <int D>
__device__ __forceinline__ void solve_path_pair(const ItemMeta& M, const float* GR,
                                                uint8_t* smem, int sn, int dn, int wmax) {
  static_assert(D <= 16, "paired rows keep 2 x 16 partial sums");
  constexpr int NA = 16;
  const uint8_t* prow = M.path[sn];  // entries past the node are 0 (a valid node)
  const uint4* pr = reinterpret_cast<const uint4*>(prow);
  const uint4 pa = pr[0], pb = pr[1];
  const uint32_t pw[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
  const float Gn = M.G[sn];
  const float* GRq = GR + (64 + sn) * 64;  // q_n . k_s, row 64 + sn (same swizzle phase)
  const int xq = (sn & 7) << 2;
  float accT[NA], accW[NA];
#pragma unroll
  for (int k = 0; k < NA; ++k) {
    accT[k] = 0.f;
    accW[k] = 0.f;
  }
  float aiT = 0.f, aiW = 0.f;
  int pi = prow[wmax];
  int pn = wmax > 0 ? prow[wmax - 1] : 0;
  float Gi = M.G[pi], bi = M.bb[pi], qi = GRq[pi ^ xq];
  for (int i = wmax; i >= 0; --i) {
    const int pnn = i > 1 ? prow[i - 2] : 0;
    const float Gnx = M.G[pn], bnx = M.bb[pn], qnx = GRq[pn ^ xq];
    const float* GRi = GR + pi * 64;
    const int xi = (pi & 7) << 2;
    const float kn = GRi[pn ^ xi];
    const float yW = __expf(Gn - Gi) * qi;
    const float inv_phi = __expf(fmaxf(Gn - Gi, -80.f));
    const float f = bi * __expf(fminf(Gi - Gn, 80.f));
    const float baseT = pick<NA>(accT, i - 1);
    const float baseW = pick<NA>(accW, i - 1);
    const float rT = (i == dn ? 1.f : 0.f) - inv_phi * aiT;
    const float rW = yW - inv_phi * aiW;
    const bool own = i <= dn;
    const float sT = own ? rT * f : 0.f;
    const float sW = own ? rW * f : 0.f;
    if (own) {
      const int col = (pi >> 3);
      const int sub = (pi & 7) * 2;
      const int offT = atom_off(sn, col) + sub;
      const int offW = atom_off(64 + sn, col) + sub;
      const __nv_bfloat16 hT = __float2bfloat16_rn(rT);
      const __nv_bfloat16 hW = __float2bfloat16_rn(rW);
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2hi + offT) = hT;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2lo + offT) =
          __float2bfloat16_rn(rT - __bfloat162float(hT));
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2hi + offW) = hW;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2lo + offW) =
          __float2bfloat16_rn(rW - __bfloat162float(hW));
    }
    const int lim = i - 1;
    if (lim <= 4) {
      path_update2<4>(accT, accW, pw, sT, sW, GRi, xi);
    } else if (lim <= 8) {
      path_update2<8>(accT, accW, pw, sT, sW, GRi, xi);
    } else if (lim <= 12) {
      path_update2<12>(accT, accW, pw, sT, sW, GRi, xi);
    } else {
      path_update2<16>(accT, accW, pw, sT, sW, GRi, xi);
    }
    aiT = fmaf(sT, kn, baseT);
    aiW = fmaf(sW, kn, baseW);
    pi = pn;
    pn = pnn;
    Gi = Gnx;
    bi = bnx;
    qi = qnx;
  }
}

template <int kSolveD>
__global__ void __launch_bounds__(kTcThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap,
                 int n_items, int H_qk, int H_v, int depth_max, int words, int small_only,
                 const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ depth, const int32_t* __restrict__ order,
                 const int32_t* __restrict__ pos, const uint64_t* __restrict__ anc,
                 int32_t* __restrict__ status,
                 const float* __restrict__ g, const float* __restrict__ bta, float* S,
                 __nv_bfloat16* __restrict__ o, float* __restrict__ Uws,
                 float* __restrict__ Gws, const PendingCommit cm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcShared& sh = *reinterpret_cast<TcShared*>(smem + kOffMeta);
  volatile int* abort = &sh.abort;
  const int tid = threadIdx.x, warp = tid >> 5;
  if ((int)blockIdx.x >= n_items) return;
  // Item order.  With a pending commit the producer warps are the critical path,
  // so each CTA takes a contiguous run of items: consecutive items are mostly the
  // heads of one sequence, whose root paths are then reused.  Otherwise the items
  // are dealt round robin, so that the CTAs work on neighbouring heads of the
  // same rows at the same time (better DRAM locality for the v, U and o rows).
  const bool runs = cm.path != nullptr;
  const int i_begin = runs ? (int)(((long)blockIdx.x * n_items) / gridDim.x) : (int)blockIdx.x;
  const int i_end = runs ? (int)(((long)(blockIdx.x + 1) * n_items) / gridDim.x) : n_items;
  const int i_step = runs ? 1 : (int)gridDim.x;
  const int grp = H_v / H_qk;  // v-heads per query/key head
  const bool fused = cm.path != nullptr;
  // Launched with programmatic stream serialization: everything up to
  // griddepcontrol.wait below touches no global memory (the first item's state
  // is only pulled into L2, which stays coherent), so it can overlap the tail of
  // the previous kernel in the stream.
  if (tid == 0) prefetch_l2(S + (size_t)i_begin * kTcDK * kTcDV, kTcDK * kTcDV * 4);

  if (tid == 0) {
    mbar_init(&sh.tma_bar, 1);
    mbar_init(&sh.mma1_bar, 1);
    mbar_init(&sh.mma2_bar, 1);
    mbar_init(&sh.v_bar, 1);
    mbar_init(&sh.s1_done[0], 2);
    mbar_init(&sh.s1_done[1], 2);
    mbar_init(&sh.tmem_free[0], 1);
    mbar_init(&sh.tmem_free[1], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    sh.abort = 0;
    sh.tma_issued = 0;
    sh.v_issued = 0;
    sh.mma1_issued = 0;
  }
  if (warp == 0) tmem_alloc(&sh.tmem_slot, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_slot;
  grid_dependency_wait();     // the previous kernel's writes are visible from here on
  grid_launch_dependents();   // the next kernel may start its own prologue
  if (small_only) {  // a CTA whose items all belong to the 128-node kernel leaves at once
    int mine = 0;
    if (warp == 0)
      for (int it = i_begin + (tid & 31) * i_step; it < i_end; it += 32 * i_step) {
        const int n = cu[it / H_v + 1] - cu[it / H_v];
        mine |= (n > 0 && n <= kTcNodes) ? 1 : 0;
      }
    if (!__syncthreads_or(mine)) {
      if (warp == 0) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }

  if (tid < kGroup) {
    // =================================================== producer warps 0-7
    const int p = tid;
    auto issue_kq = [&](int item, int row0) {  // thread 0 only; row0 = cu[item / H_v]
      const int qh = (item % H_v) / grp;
      mbar_arrive_expect_tx(&sh.tma_bar, 4 * 64 * 128);
      // box = 64 d_k elements x 1 head x 64 node rows, 128-byte swizzled rows
      tma_load_3d(smem + kOffA + 0, &kmap, &sh.tma_bar, 0, qh, row0);
      tma_load_3d(smem + kOffA + 8192, &qmap, &sh.tma_bar, 0, qh, row0);
      tma_load_3d(smem + kOffA + 16384, &kmap, &sh.tma_bar, 64, qh, row0);
      tma_load_3d(smem + kOffA + 24576, &qmap, &sh.tma_bar, 64, qh, row0);
      sh.tma_issued += 1;
    };
    // S0 of one item: warp w holds rows 16 w .. 16 w + 15, lane p & 31 float4
    // column p & 31 (plain loads: with a pending commit the kernel writes these
    // rows back)
    const int srow0 = (p >> 5) * 16, sq = p & 31;
    float4 sreg[16];
    auto load_s0 = [&](int item) {
      const float* src = S + (size_t)item * kTcDK * kTcDV;  // item = bi * H_v + h
#pragma unroll
      for (int r = 0; r < 16; ++r)
        sreg[r] = reinterpret_cast<const float4*>(src + (size_t)(srow0 + r) * kTcDV)[sq];
    };
    // Warp 0, two items ahead of its staging: the item's accepted path in the
    // previous tree (lane l holds entry l) and that sequence's bounds and status.
    // (Raw values only: nothing here waits for these loads; they are combined
    // when the item is published, an iteration later.)
    int c_node = -1, c_plo = 0, c_phi = 0, c_st = TGDN_SEQ_OK;
    auto load_commit_meta = [&](int it) {
      const int bi = it / H_v;
      c_plo = cm.cu[bi];
      c_phi = cm.cu[bi + 1];
      c_st = cm.status[bi];
      c_node = cm.path[(size_t)bi * cm.path_len + (p < cm.path_len ? p : cm.path_len - 1)];
    };
    // Warp 0: the item's staged path (entries after the first invalid one are
    // ignored) -> c_L[cb], c_row[cb].
    auto publish_commit = [&](int cb) {
      const bool valid = c_st == TGDN_SEQ_OK && p < cm.path_len && c_node >= 0 &&
                         c_node < c_phi - c_plo;
      const int L = __ffs(__ballot_sync(0xffffffffu, !valid)) - 1;  // path_len <= 31
      if (p == 0) sh.c_L[cb] = L;
      if (p < L) sh.c_row[cb][p] = c_plo + c_node;
    };
    // All producer threads: 16-byte asynchronous copies of the published path's
    // u_s rows, k_s rows and the chunks holding G_s (49 chunks per path node).
    auto stage_commit = [&](int it, int cb) {
      const int h = it % H_v, qh = h / grp;
      const int L = sh.c_L[cb];
      for (int e = p; e < L * 49; e += kGroup) {
        const int l = e / 49, w = e - l * 49;
        const size_t row = static_cast<size_t>(sh.c_row[cb][l]);
        if (w < 32) {
          cp_async16(smem + kOffUP + l * (kTcDV * 4) + w * 16,
                     cm.U + (row * H_v + h) * kTcDV + w * 4);
        } else if (w < 48) {
          cp_async16(smem + kOffKP + l * (kTcDK * 2) + (w - 32) * 16,
                     static_cast<const __nv_bfloat16*>(cm.k) + (row * H_qk + qh) * kTcDK +
                         (w - 32) * 8);
        } else {
          const size_t ge = row * H_v + h;  // the workspace base is 256-byte aligned
          sh.c_gi[cb][l] = static_cast<int>(ge & 3);
          cp_async16(smem + kOffGP + l * 16, cm.G + (ge & ~static_cast<size_t>(3)));
        }
      }
      cp_async_commit();
    };
    // Sequence bounds and status one item ahead of the node metadata, so that no
    // load waits on another load of the same iteration (raw bounds: the count is
    // formed when they are used).
    int q_lo = 0, q_hi = 0, q_st = 0;
    auto load_seq = [&](int item) {
      const int bi = item / H_v;
      q_lo = cu[bi];
      q_hi = cu[bi + 1];
      q_st = status[bi];
    };
    Prefetch pf;
    auto load_meta = [&](int item) {  // node metadata; the bounds come from load_seq
      const int h = item % H_v;
      pf.lo = q_lo;
      pf.N = q_hi - q_lo;
      pf.st = q_st;
      if (p < pf.N && p < kTcNodes) {
        pf.dep = depth[pf.lo + p];
        pf.pos = pos[pf.lo + p];
        pf.ord = order[pf.lo + p];
        pf.gg = g[(size_t)(pf.lo + p) * H_v + h];
        pf.bb = bta[(size_t)(pf.lo + p) * H_v + h];
      }
    };
    int item = i_begin;
    load_seq(item);
    load_meta(item);
    if (item + i_step < i_end) load_seq(item + i_step);
    if (!(small_only && pf.N > kTcNodes)) load_s0(item);
    if (fused) {
      if (p < 32) {
        load_commit_meta(item);
        publish_commit(0);
      }
      named_sync(kBarP, kGroup);
      stage_commit(item, 0);
      if (p < 32 && item + i_step < i_end) load_commit_meta(item + i_step);
    }

    int prev_bi = -1;  // sequence of the previous item when its tree was valid
    int npr = 0;       // items processed so far (passed-over items excluded): one [K;Q]
                       // copy and one first product each, in order
    for (int j = 0; item < i_end; ++j, item += i_step) {
      const int slot = j & 1;
      ItemMeta& M = sh.meta[slot];
      const int bi = item / H_v, h = item % H_v;
      const int lo = pf.lo, N = pf.N;
      const int next = item + i_step;
      if (fused) {
        // the previous step's commit: S = e^{G*} S + sum_l e^{G*-G_l} k_l u_l^T,
        // written back in place; the committed state is what gets verified
        cp_async_wait_all();
        if (p < 32 && next < i_end) publish_commit(slot ^ 1);  // the next item's path
        // thread 0: the previous first product has completed, so its operands (the
        // [K; Q] and S0 areas) are free; this item's key and query rows go out
        bool w_ok = true;
        if (p == 0) {
          if (npr > 0) w_ok = mbar_wait_suspend(&sh.mma1_bar, (npr - 1) & 1, abort);
          if (w_ok) issue_kq(item, lo);
        }
        if (!named_sync_and(kBarP, kGroup, w_ok && !*abort)) break;
        const int L = sh.c_L[slot];
        if (L > 0) {
          const float4* UP = reinterpret_cast<const float4*>(smem + kOffUP);
          const uint4* KP = reinterpret_cast<const uint4*>(smem + kOffKP);
          const float* GP = reinterpret_cast<const float*>(smem + kOffGP);
          const float Gstar = GP[(L - 1) * 4 + sh.c_gi[slot][L - 1]];
          const float decay = __expf(Gstar);
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            sreg[r].x *= decay;
            sreg[r].y *= decay;
            sreg[r].z *= decay;
            sreg[r].w *= decay;
          }
          // one path node per step; its u row, k rows and G_s are read a step ahead
          const int kq = srow0 >> 3;  // 16-byte chunk of this warp's 16 rows of k
          float4 un = UP[sq];
          uint4 kan = KP[kq], kbn = KP[kq + 1];
          float gn = GP[sh.c_gi[slot][0]];
          for (int l = 0; l < L; ++l) {
            float4 u = un;
            const uint4 ka = kan, kb = kbn;
            const float cl = __expf(Gstar - gn);
            if (l + 1 < L) {
              un = UP[(l + 1) * (kTcDV / 4) + sq];
              kan = KP[(l + 1) * (kTcDK / 8) + kq];
              kbn = KP[(l + 1) * (kTcDK / 8) + kq + 1];
              gn = GP[(l + 1) * 4 + sh.c_gi[slot][l + 1]];
            }
            u.x *= cl;
            u.y *= cl;
            u.z *= cl;
            u.w *= cl;
            // k_l at this warp's 16 rows: 32 bytes, the same for the whole warp
            const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // bf16 pair -> rows srow0 + 2 i, + 2 i + 1
              const float k0 = __uint_as_float(kw[i] << 16);
              const float k1 = __uint_as_float(kw[i] & 0xffff0000u);
              float4& a0 = sreg[2 * i];
              float4& a1 = sreg[2 * i + 1];
              a0.x = fmaf(k0, u.x, a0.x);
              a0.y = fmaf(k0, u.y, a0.y);
              a0.z = fmaf(k0, u.z, a0.z);
              a0.w = fmaf(k0, u.w, a0.w);
              a1.x = fmaf(k1, u.x, a1.x);
              a1.y = fmaf(k1, u.y, a1.y);
              a1.z = fmaf(k1, u.z, a1.z);
              a1.w = fmaf(k1, u.w, a1.w);
            }
          }
          // the committed rows, written back in place (a warp stores whole rows)
          float* dst = S + (size_t)item * kTcDK * kTcDV;
#pragma unroll
          for (int r = 0; r < 16; ++r)
            reinterpret_cast<float4*>(dst + (size_t)(srow0 + r) * kTcDV)[sq] = sreg[r];
        }
      }
      // the consumer has finished item j-2, the previous user of this half and slot
      // (every wait is agreed on by the whole group before anyone leaves the loop);
      // the commit above touches neither, so it runs while the consumer finishes
      if (j >= 2 && !group_wait(&sh.tmem_free[slot], ((j >> 1) + 1) & 1, kBarP, p == 0, abort))
        break;
      bool ok = (pf.st == TGDN_SEQ_OK) && N > 0 && N <= kTcNodes;
      // (small_only: sequences above 64 nodes belong to the 128-node kernel; their
      // items pass through without state, solve or writes)
      const bool skip = small_only && N > kTcNodes;
      uint64_t my_anc = 0;
      if (p == 0) {
        M.lo = lo;
        M.N = N;
        M.h = h;
        M.skip = skip;
      }
      if (ok && p < N) {
        const bool v_ok = pf.dep >= 0 && pf.dep <= depth_max && pf.dep <= kTcDepth &&
                          pf.pos >= 0 && pf.pos < N && pf.ord >= 0 && pf.ord < N;
        ok = v_ok;
        M.dep[p] = pf.dep;
        M.pos[p] = pf.pos;
        M.ord[p] = pf.ord;
        M.gg[p] = pf.gg;
        M.bb[p] = pf.bb;
        if (v_ok) my_anc = anc[(size_t)(lo + pf.pos) * words];  // positions < 64: word 0
      }
      // Without a pending commit the same hand-over happens here.
      bool step_ok = true;
      if (!fused && p == 0 && !skip) {
        if (npr > 0) step_ok = mbar_wait_suspend(&sh.mma1_bar, (npr - 1) & 1, abort);
        if (step_ok) issue_kq(item, lo);
      }
      // (also: every thread has finished reading this item's staged commit)
      if (!named_sync_and(kBarP, kGroup, step_ok && !*abort)) break;
      // the next item's small loads go out before the operand stores, so that they
      // wait neither behind those stores nor for their source registers
      if (next < i_end) {
        load_meta(next);
        if (next + i_step < i_end) {
          load_seq(next + i_step);
          if (fused && p < 32) load_commit_meta(next + i_step);
        }
      }
      if (fused && next < i_end) stage_commit(next, slot ^ 1);
      // S0 registers -> bf16 hi/lo operand
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (skip) break;  // (uniform)
        const int kr = srow0 + r;
        const float4 xv = sreg[r];
        const float h0 = __bfloat162float(__float2bfloat16_rn(xv.x));
        const float h1 = __bfloat162float(__float2bfloat16_rn(xv.y));
        const float h2 = __bfloat162float(__float2bfloat16_rn(xv.z));
        const float h3 = __bfloat162float(__float2bfloat16_rn(xv.w));
        const int off = (sq >> 4) * 16384 + atom_off(kr, (sq & 15) >> 1) + (sq & 1) * 8;
        *reinterpret_cast<uint2*>(smem + kOffS0hi + off) =
            make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
        *reinterpret_cast<uint2*>(smem + kOffS0lo + off) =
            make_uint2(pack_bf16x2(xv.x - h0, xv.y - h1), pack_bf16x2(xv.z - h2, xv.w - h3));
      }
      fence_proxy_async_smem();
      named_sync(kBarP, kGroup);  // the S0 operand is complete
      // First product into TMEM half `slot`, issued by the group's last thread (no
      // node of its own) while the others prefetch and build the paths; its
      // completion is awaited in the next iteration.  Items found invalid below
      // get the product too; the consumer ignores it and zero-fills.
      if (p == kGroup - 1 && skip) {
        mbar_arrive(&sh.s1_done[slot]);  // a passed-over item: no copy, no product
      } else if (p == kGroup - 1) {
        if (mbar_wait_suspend(&sh.tma_bar, npr & 1, abort)) {
          tc_fence_after_sync();
          const uint32_t tb = tmem + slot * 256;
          const uint32_t sA = smem_addr(smem + kOffA);
          const uint32_t sHi = smem_addr(smem + kOffS0hi);
          const uint32_t sLo = smem_addr(smem + kOffS0lo);
          constexpr uint32_t id_s0 = idesc_bf16_f32(128, 128, 0, 1);
          constexpr uint32_t id_gram = idesc_bf16_f32(128, kTcNodes, 0, 0);
#pragma unroll
          for (int s = 0; s < kTcDK / 16; ++s) {
            const uint64_t ad = smem_desc(sA + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024,
                                          kSwizzle128B);
            // MN-major S0: value-column atoms 16 KiB apart (leading byte offset),
            // 8-row k groups 1 KiB apart (stride byte offset)
            const uint64_t hd = smem_desc(sHi + s * 2048, 16384, 1024, kSwizzle128B);
            const uint64_t ld = smem_desc(sLo + s * 2048, 16384, 1024, kSwizzle128B);
            umma_bf16(tb, ad, hd, id_s0, s > 0);
            umma_bf16(tb, ad, ld, id_s0, 1);
            umma_bf16(tb + kGramCol, ad, ad, id_gram, s > 0);  // B = the key rows of A
          }
          umma_commit(&sh.mma1_bar);
          umma_commit(&sh.s1_done[slot]);
          sh.mma1_issued += 1;
        } else {
          mbar_arrive(&sh.s1_done[slot]);  // no product: the consumer zero-fills
        }
      }
      // the next item's state while this one is finished
      if (next < i_end && !(small_only && pf.N > kTcNodes)) load_s0(next);
      // root paths from the ancestor masks (bits = topological positions,
      // ascending = root first) and path-cumulative log-gates; the same tree as
      // the previous item (another head) reuses its paths and only sums the gates.
      // This runs while the first product is being issued, before the group has
      // agreed that every node's metadata is valid, so a node index read from
      // another thread's metadata is range-checked before it is used.
      const bool reuse = prev_bi == bi;
      if (ok && p < N && reuse) {
        const int dn = M.dep[p];
        const uint8_t* srow = sh.meta[slot ^ 1].path[p];
        const uint4* src = reinterpret_cast<const uint4*>(srow);
        uint4* dst = reinterpret_cast<uint4*>(M.path[p]);
        dst[0] = src[0];
        dst[1] = src[1];
        float acc = 0.f;
        for (int i = 0; i <= dn; ++i) acc += M.gg[srow[i]];
        M.G[p] = acc;
      } else if (ok && p < N) {
        const int dn = M.dep[p];
        uint64_t mk = my_anc;
        bool pk = __popcll(mk) == dn + 1 && ((mk >> M.pos[p]) & 1ull);
        uint8_t* prow = M.path[p];
        reinterpret_cast<uint4*>(prow)[0] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(prow)[1] = make_uint4(0u, 0u, 0u, 0u);
        float acc = 0.f;
        int last = -1;
        for (int i = 0; pk && i <= dn; ++i) {
          const int b = __ffsll(static_cast<long long>(mk)) - 1;
          mk &= mk - 1;
          if (b >= N) {
            pk = false;
            break;
          }
          const int s = M.ord[b];
          if (s < 0 || s >= N) {
            pk = false;
            break;
          }
          pk = M.dep[s] == i;
          prow[i] = static_cast<uint8_t>(s);
          acc += M.gg[s];
          last = s;
        }
        if (!pk || last != p) ok = false;
        M.G[p] = acc;
      }
      ok = named_sync_and(kBarP, kGroup, ok);
      prev_bi = ok ? bi : -1;
      if (p == 0) {
        M.good = ok;
        mbar_arrive(&sh.s1_done[slot]);  // the metadata above is written
      }
      if (!skip) ++npr;
    }
  } else {
    // =================================================== consumer warps 8-15
    const int c = tid - kGroup;
    const int cw = c >> 5;            // 0..7
    const int lq = cw & 3;            // TMEM lane quarter (warp index mod 4)
    const int chalf = cw >> 2;        // value-column half
    const uint32_t lane_base = static_cast<uint32_t>(lq * 32) << 16;
    const int lane_row = lq * 32 + (c & 31);
    const bool key_lane = lq < 2;
    const int lane_node = key_lane ? lane_row : lane_row - 64;
    // Thread 0, one item ahead: the V rows of an item go by TMA into the R lo
    // operand area (the same swizzled layout), where R is then formed in place.
    int cv_lo = 0, cv_hi = 0;  // node rows of the item whose V rows go out next
    auto load_vseq = [&](int item) {
      cv_lo = cu[item / H_v];
      cv_hi = cu[item / H_v + 1];
    };
    // a passed-over item (small_only, above 64 nodes) gets no V rows
    auto v_wanted = [&]() { return !(small_only && cv_hi - cv_lo > kTcNodes); };
    auto issue_v = [&](int item) {
      mbar_arrive_expect_tx(&sh.v_bar, 2 * 64 * 128);
      tma_load_3d(smem + kOffRlo, &vmap, &sh.v_bar, 0, item % H_v, cv_lo);
      tma_load_3d(smem + kOffRlo + 8192, &vmap, &sh.v_bar, 64, item % H_v, cv_lo);
      sh.v_issued += 1;
    };
    int item = i_begin;
    if (c == 0) {
      load_vseq(item);
      if (v_wanted()) issue_v(item);
      if (item + i_step < i_end) load_vseq(item + i_step);
    }
    uint32_t mma2_count = 0;  // second products issued so far (same in every thread)
    int nv = 0;               // V copies consumed so far (one per item not passed over)
    for (int j = 0; item < i_end; ++j, item += i_step) {
      const int slot = j & 1;
      bulk_wait_read();  // the previous item's output rows have left shared memory
      if (!group_wait(&sh.s1_done[slot], (j >> 1) & 1, kBarC, c == 0, abort)) break;
      tc_fence_after_sync();
      const ItemMeta& M = sh.meta[slot];
      const int lo = M.lo, N = M.N, h = M.h;
      const uint32_t tb = tmem + slot * 256;
      const int next = item + i_step;

      if (!M.good) {  // bad or empty sequence: zero rows (none for a passed-on item)
        const int nz = M.skip ? 0 : N;
        for (int e = c; e < nz * (kTcDV / 4); e += kGroup) {
          const int n = e >> 5, c4 = e & 31;
          const size_t row = ((size_t)(lo + n) * H_v + h) * kTcDV + c4 * 4;
          *reinterpret_cast<uint2*>(o + row) = make_uint2(0u, 0u);
          *reinterpret_cast<float4*>(Uws + row) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int n = c; n < nz; n += kGroup) Gws[(size_t)(lo + n) * H_v + h] = 0.f;
        bool v_ok = true;
        if (c == 0) {  // this item's V rows have landed: the area is free for the next
          if (!M.skip) v_ok = mbar_wait_suspend(&sh.v_bar, nv & 1, abort);
          if (v_ok && next < i_end) {
            if (v_wanted()) issue_v(next);
            if (next + i_step < i_end) load_vseq(next + i_step);
          }
        }
        if (!M.skip) ++nv;
        if (!named_sync_and(kBarC, kGroup, v_ok)) break;
        if (c == 0) mbar_arrive(&sh.tmem_free[slot]);
        continue;
      }

      // ---- Gram rows -> shared memory; [T; W] operand zeroed
      {
        float* GR = reinterpret_cast<float*>(smem + kOffGR);
        float r[32];
        tmem_ld32(tb + lane_base + kGramCol + chalf * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          *reinterpret_cast<float4*>(GR + lane_row * 64 + swz(lane_row, chalf * 8 + c4) * 4) =
              make_float4(r[c4 * 4], r[c4 * 4 + 1], r[c4 * 4 + 2], r[c4 * 4 + 3]);
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i)  // 32 KiB of [T; W] hi + lo, consecutive 16 B per thread
          *reinterpret_cast<uint4*>(smem + kOffA2hi + (i * kGroup + c) * 16) = zero;
      }
      named_sync(kBarC, kGroup);  // Gram rows stored, [T; W] operand zeroed

      // Key-lane warps form R while the query-lane warps solve for T and W (the
      // solve needs only the Gram rows and the metadata).
      // ---- R = diag(b)(V - e^G K S0) as a bf16 hi/lo operand (key lanes)
      bool v_ok = true;
      if (key_lane) {
        v_ok = mbar_wait_suspend(&sh.v_bar, nv & 1, abort);
        const bool live = lane_node < N;
        const float eG = live ? __expf(M.G[lane_node]) : 0.f;
        const float bn = live ? M.bb[lane_node] : 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // 32 value columns at a time
          float r[32];
          tmem_ld32(tb + lane_base + chalf * 64 + q * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {  // 8 columns per 16-byte bf16 chunk
            const int off = chalf * 8192 + atom_off(lane_node, q * 4 + c8);
            const uint4 vv = *reinterpret_cast<const uint4*>(smem + kOffRlo + off);
            const __nv_bfloat162* vb = reinterpret_cast<const __nv_bfloat162*>(&vv);
            float xr[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 vf = __bfloat1622float2(vb[i]);
              xr[2 * i] = live ? bn * (vf.x - eG * r[c8 * 8 + 2 * i]) : 0.f;
              xr[2 * i + 1] = live ? bn * (vf.y - eG * r[c8 * 8 + 2 * i + 1]) : 0.f;
            }
            uint4 hi, lw;
            split8(xr, hi, lw);  // rows of R beyond the tree are exact zeros
            *reinterpret_cast<uint4*>(smem + kOffRhi + off) = hi;
            *reinterpret_cast<uint4*>(smem + kOffRlo + off) = lw;
          }
        }
      }

      // ---- the rows of T and W on the query-lane warps (solve_path_pair for
      // trees of depth <= 16, else solve_path_row).  Rows are handed out in
      // topological order so that a warp sees similar depths.
      if (!key_lane) {
        const float* GR = reinterpret_cast<const float*>(smem + kOffGR);
        if constexpr (kSolveD <= 16) {
          // warps 10 and 11 (one per scheduler): a node's T and W rows per thread
          if (chalf == 0) {
            const int spos = (lq - 2) * 32 + (c & 31);
            const bool act = spos < N;
            const int sn = act ? M.ord[spos] : 0;
            const int dn = act ? M.dep[sn] : -1;
            const int wmax = __reduce_max_sync(0xffffffffu, dn);
            solve_path_pair<kSolveD>(M, GR, smem, sn, dn, wmax);
          }
        } else {
          const int sc = (lq - 2) * 64 + chalf * 32 + (c & 31);  // solver index 0..127
          const int spos = sc & 63;
          const bool act = spos < N;
          const int sn = act ? M.ord[spos] : 0;
          const int dn = act ? M.dep[sn] : -1;
          const int wmax = __reduce_max_sync(0xffffffffu, dn);
          solve_path_row<kSolveD>(M, GR, smem, sn, dn, wmax, sc < 64);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      if (!named_sync_and(kBarC, kGroup, v_ok)) break;
      tc_fence_after_sync();

      // ---- second product: D[:, 128:256] = [T; W] R  (hi.hi + hi.lo + lo.hi)
      if (c == 0) {
        const uint32_t sA2hi = smem_addr(smem + kOffA2hi);
        const uint32_t sA2lo = smem_addr(smem + kOffA2lo);
        const uint32_t sRhi = smem_addr(smem + kOffRhi);
        const uint32_t sRlo = smem_addr(smem + kOffRlo);
        constexpr uint32_t id_r = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
        for (int s = 0; s < kTcNodes / 16; ++s) {
          const uint64_t ah = smem_desc(sA2hi + s * 32, 16, 1024, kSwizzle128B);
          const uint64_t al = smem_desc(sA2lo + s * 32, 16, 1024, kSwizzle128B);
          // MN-major R: value-column atoms 8 KiB apart, 8-node groups 1 KiB apart
          const uint64_t bh = smem_desc(sRhi + s * 2048, 8192, 1024, kSwizzle128B);
          const uint64_t bl = smem_desc(sRlo + s * 2048, 8192, 1024, kSwizzle128B);
          const uint32_t d = tb + kGramCol;
          umma_bf16(d, ah, bh, id_r, s > 0);
          umma_bf16(d, ah, bl, id_r, 1);
          umma_bf16(d, al, bh, id_r, 1);
        }
        umma_commit(&sh.mma2_bar);
      }
      const bool done2 = group_wait(&sh.mma2_bar, mma2_count & 1, kBarC, c == 0, abort);
      ++mma2_count;
      if (!done2) break;
      tc_fence_after_sync();
      // the operand areas are free: the next item's V rows go out now
      ++nv;
      if (c == 0 && next < i_end) {
        if (v_wanted()) issue_v(next);
        if (next + i_step < i_end) load_vseq(next + i_step);
      }

      // ---- key lanes: U rows; query lanes: O = e^G Q S0 + W R (bf16).  Each
      // thread stages its half row in shared memory (padded rows: conflict-free)
      // and sends it to global memory with one bulk copy.
      {
        const bool live = lane_node < N;
        if (key_lane) {
          float4* stg = reinterpret_cast<float4*>(smem + kOffUst + lane_node * kUstRow + chalf * 256);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float r[32];
            tmem_ld32(tb + lane_base + kGramCol + chalf * 64 + q * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              stg[q * 8 + i] = make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
          }
          if (live) {
            fence_proxy_async_smem();
            bulk_copy_s2g(Uws + ((size_t)(lo + lane_node) * H_v + h) * kTcDV + chalf * 64, stg,
                          256);
            bulk_commit();
            if (chalf == 0) Gws[(size_t)(lo + lane_node) * H_v + h] = M.G[lane_node];
          }
        } else {
          uint4* stg = reinterpret_cast<uint4*>(smem + kOffOst + lane_node * kOstRow + chalf * 128);
          const float eG = live ? __expf(M.G[lane_node]) : 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // 16 value columns at a time
            float a[16], w[16];
            tmem_ld16(tb + lane_base + chalf * 64 + q * 16, a);
            tmem_ld16(tb + lane_base + kGramCol + chalf * 64 + q * 16, w);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float* aa = a + 8 * i;
              const float* ww = w + 8 * i;
              stg[q * 2 + i] =
                  make_uint4(pack_bf16x2(fmaf(eG, aa[0], ww[0]), fmaf(eG, aa[1], ww[1])),
                             pack_bf16x2(fmaf(eG, aa[2], ww[2]), fmaf(eG, aa[3], ww[3])),
                             pack_bf16x2(fmaf(eG, aa[4], ww[4]), fmaf(eG, aa[5], ww[5])),
                             pack_bf16x2(fmaf(eG, aa[6], ww[6]), fmaf(eG, aa[7], ww[7])));
            }
          }
          if (live) {
            fence_proxy_async_smem();
            bulk_copy_s2g(o + ((size_t)(lo + lane_node) * H_v + h) * kTcDV + chalf * 64, stg, 128);
            bulk_commit();
          }
        }
      }
      tc_fence_before_sync();
      named_sync(kBarC, kGroup);
      if (c == 0) mbar_arrive(&sh.tmem_free[slot]);  // this half is free again
    }
    bulk_wait_all();  // this thread's output rows are written
  }

  // ---- end.  After an expired wait every item still owned by this CTA is
  // reported as timed out, and the latest copies and products are drained (bounded).
  cp_async_wait_all();  // staging copies left by a loop that ended early
  __syncthreads();
  if (sh.abort && tid == 0) {
    for (int it2 = i_begin; it2 < i_end; it2 += i_step)
      atomicCAS(&status[it2 / H_v], TGDN_SEQ_OK, TGDN_SEQ_TIMEOUT);
    if (sh.tma_issued > 0) (void)mbar_wait(&sh.tma_bar, (sh.tma_issued - 1) & 1);
    if (sh.v_issued > 0) (void)mbar_wait(&sh.v_bar, (sh.v_issued - 1) & 1);
  }
  // the last first product, before TMEM and the operands are released (bounded)
  if (tid == 0 && sh.mma1_issued > 0) (void)mbar_wait(&sh.mma1_bar, (sh.mma1_issued - 1) & 1);
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool pending_commit_tc_supported(const tgdn_tree& prev, const void* prev_k) {
  return prev.depth_max + 1 <= kTcPath && (reinterpret_cast<uintptr_t>(prev_k) % 16) == 0;
}

bool verify_tc_supported(const tgdn_tree& t, const tgdn_dims& d, const void* q, const void* k,
                         const void* v, const float* S0, const void* o, bool small_only) {
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
  return d.io == TGDN_BF16 && d.d_k == kTcDK && d.d_v == kTcDV &&
         (small_only || t.n_max <= kTcNodes) && t.depth_max <= kTcDepth && al(q, 16) &&
         al(k, 16) && al(v, 16) && al(S0, 16) && al(o, 16);
}

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && c > 0)
      n = c;
    else
      return 1;
  }
  return n;
}

cudaError_t launch_verify_tc(const tgdn_tree& t, const tgdn_dims& d, const CUtensorMap& qmap,
                             const CUtensorMap& kmap, const CUtensorMap& vmap, const float* g,
                             const float* b, float* S, void* o, float* U, float* G,
                             const PendingCommit& cm, bool small_only, cudaStream_t s) {
  // the path solve keeps depth_max + 1 partial sums in registers
  auto kern = t.depth_max <= 16 ? verify_tc_kernel<16> : verify_tc_kernel<kTcDepth>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (e != cudaSuccess) return e;
  const long items = (long)t.B * d.H_v;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  const int grid = (int)(items < sms ? items : sms);
  // programmatic stream serialization: the kernel's prologue may overlap the
  // previous kernel's tail (it waits for that kernel before reading any input)
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(kTcThreads);
  lc.dynamicSmemBytes = kTcSmemBytes;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, kern, qmap, kmap, vmap, (int)items, d.H_qk, d.H_v, t.depth_max,
                         t.words, small_only ? 1 : 0, t.cu_nodes, t.depth, t.order, t.pos,
                         t.anc, t.status, g, b, S, static_cast<__nv_bfloat16*>(o), U, G, cm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tgdn
